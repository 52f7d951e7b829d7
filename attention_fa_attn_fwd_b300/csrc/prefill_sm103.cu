// FlashAttention-2-style attention forward for sm_103a (B300).
//
// Computes O = softmax(scale * Q K^T [causal]) V and the per-row natural
// log-sum-exp in one pass over K/V, so the N x N matrices S and P never
// reach HBM (FAQ page "Wie unterscheidet sich die Implementierung von
// FlashAttention-2 ...", comparison table: tiling, online softmax; interview
// notes "他人面经整理", flashattention answer part 2: kernel fusion, tiling,
// online softmax with running max m and running sum l).
//
// One CTA owns one 128-row Q tile of one (batch, head) and streams all of the
// K/V tiles it may attend (causal: up to the diagonal).  Warp roles:
//   warp 0      TMA producer: Q once, then K_j / V_j into a ring of stages
//               (the double-buffered prefetch of the FSA page, section 3.2).
//   warp 1      tcgen05 MMA issuer (one thread): S_j = Q K_j^T into TMEM,
//               O += P_j V_j with P_j read from TMEM.
//   warps 2..5  softmax: thread r owns TMEM lane / Q row r.  Online softmax in
//               base 2 with scale*log2(e) folded into one FFMA; the running
//               max is only moved when it grows by more than 8 (log2 units),
//               and O in TMEM is rescaled only then; P is written back to
//               TMEM as bf16.  At the end: O / l (deferred normalisation),
//               bf16 O through smem and a TMA store, lse = (m + log2 l) ln 2.
//
// TMEM columns: S0 [0,128) S1 [128,256) O [256,256+d) P0 [384,448) P1 [448,512).
// The mbarrier protocol and why each wait is sufficient is described next to
// each role below.  Every wait is bounded (ptx.cuh).

#include <cmath>
#include <cstdio>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {

__device__ int g_prefill_error;

namespace {

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: p <= 2^8 between rescales

template <int D>
struct Cfg {
  static constexpr int kSlabs = D / 64;          // 64-element (128-byte) column slabs
  static constexpr int kSlabBytes = 128 * 128;   // 128 rows x 128 B
  static constexpr int kTileBytes = kSlabs * kSlabBytes;
  static constexpr int kStages = (D == 128) ? 3 : 4;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kStages * kTileBytes;
  // barrier indices
  static constexpr int kBarQ = 0;
  static constexpr int kBarKF = 1;
  static constexpr int kBarKE = kBarKF + kStages;
  static constexpr int kBarVF = kBarKE + kStages;
  static constexpr int kBarVE = kBarVF + kStages;
  static constexpr int kBarSF = kBarVE + kStages;  // 2
  static constexpr int kBarPF = kBarSF + 2;        // 2: P_j written (softmax -> MMA)
  static constexpr int kBarPE = kBarPF + 2;        // 2: PV_j done (MMA -> softmax)
  static constexpr int kBarDrain = kBarPE + 2;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack for 1024-B alignment
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColO = 256;
  static constexpr uint32_t kColP = 384;
  static constexpr int kThreads = 192;
};

struct Args {
  float* lse;
  int B, H, Hkv, Nq, Nk;
  int n_qtiles;
  float c_log2;  // scale * log2(e)
  int causal;
};

template <int D>
__global__ void __launch_bounds__(192, 1)
    prefill_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_o, const Args a) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  int* err = &g_prefill_error;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Heavy (late, causal) Q tiles first; heads of one KV group adjacent.
  const int BH = a.B * a.H;
  const int bh = blockIdx.x % BH;
  const int qt = a.n_qtiles - 1 - blockIdx.x / BH;
  const int q0 = qt * 128;
  const int b = bh / a.H;
  const int h = bh % a.H;
  const int zkv = b * a.Hkv + h / (a.H / a.Hkv);
  int kv_end = a.Nk;
  if (a.causal) kv_end = min(a.Nk, q0 + 128 + (a.Nk - a.Nq));
  const bool dead = timed_out_before(err);
  const int n_tiles = (kv_end > 0 && !dead) ? (kv_end + 127) / 128 : 0;

  if (threadIdx.x == 0) {
    mbar_init(bar(C::kBarQ), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kBarKF + s), 1);
      mbar_init(bar(C::kBarKE + s), 1);
      mbar_init(bar(C::kBarVF + s), 1);
      mbar_init(bar(C::kBarVE + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::kBarSF + i), 1);
      mbar_init(bar(C::kBarPF + i), 128);
      mbar_init(bar(C::kBarPE + i), 1);
    }
    mbar_init(bar(C::kBarDrain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_o);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    // K_j goes to stage j % S once QK_{j-S} has finished reading it (K-empty,
    // committed by the MMA warp); V_j likewise once PV_{j-S} has finished.
    if (lane == 0 && n_tiles > 0) {
      int k_issued = 0, v_issued = 0;
      bool ok = true;
      mbar_arrive_expect_tx(bar(C::kBarQ), C::kTileBytes);
      for (int s = 0; s < C::kSlabs; ++s)
        tma_load_3d(sbase + C::kOffQ + s * C::kSlabBytes, &tm_q, bar(C::kBarQ), s * 64, q0, bh);
      for (int j = 0; j < n_tiles; ++j) {
        const int st = j % C::kStages;
        const uint32_t ph = (j / C::kStages) & 1;
        ok = mbar_wait(bar(C::kBarKE + st), ph ^ 1, abort_flag, err, kErrTimeoutProducer);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(C::kBarKF + st), C::kTileBytes);
        for (int s = 0; s < C::kSlabs; ++s)
          tma_load_3d(sbase + C::kOffK + st * C::kTileBytes + s * C::kSlabBytes, &tm_k,
                      bar(C::kBarKF + st), s * 64, j * 128, zkv);
        k_issued = j + 1;
        ok = mbar_wait(bar(C::kBarVE + st), ph ^ 1, abort_flag, err, kErrTimeoutProducer);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(C::kBarVF + st), C::kTileBytes);
        for (int s = 0; s < C::kSlabs; ++s)
          tma_load_3d(sbase + C::kOffV + st * C::kTileBytes + s * C::kSlabBytes, &tm_v,
                      bar(C::kBarVF + st), s * 64, j * 128, zkv);
        v_issued = j + 1;
      }
      if (!ok) {
        // Abort path: let every copy already in flight land before exit.
        const uint64_t deadline = globaltimer_ns() + kWaitTimeoutNs;
        mbar_wait_drain(bar(C::kBarQ), 0, deadline);
        for (int j = max(0, k_issued - C::kStages); j < k_issued; ++j)
          mbar_wait_drain(bar(C::kBarKF + j % C::kStages), (j / C::kStages) & 1, deadline);
        for (int j = max(0, v_issued - C::kStages); j < v_issued; ++j)
          mbar_wait_drain(bar(C::kBarVF + j % C::kStages), (j / C::kStages) & 1, deadline);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // Order: QK_0, then for each j: QK_{j+1}, PV_j.  QK_{j+1} writes S buffer
    // (j+1)&1, last read by softmax_{j-1}, which finished before PV_{j-1} was
    // issued (P-full wait).  PV_j reads P buffer j&1 and accumulates into O.
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, 0);
      constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, 1);
      bool ok = mbar_wait(bar(C::kBarQ), 0, abort_flag, err, kErrTimeoutMma);
      auto issue_qk = [&](int j) -> bool {
        const int st = j % C::kStages;
        if (!mbar_wait(bar(C::kBarKF + st), (j / C::kStages) & 1, abort_flag, err, kErrTimeoutMma))
          return false;
        tc_fence_after();
        const uint32_t d_tmem = tmem + C::kColS + (j & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kSlabBytes + (kk & 3) * 32;
          const uint64_t ad = smem_desc_sw128(sbase + C::kOffQ + off, 16, 1024);
          const uint64_t bd = smem_desc_sw128(sbase + C::kOffK + st * C::kTileBytes + off, 16, 1024);
          mma_bf16_ss(d_tmem, ad, bd, kIdescQK, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(C::kBarSF + (j & 1)));
        mma_commit(bar(C::kBarKE + st));
        return true;
      };
      auto issue_pv = [&](int j) -> bool {
        const int st = j % C::kStages;
        if (!mbar_wait(bar(C::kBarPF + (j & 1)), (j >> 1) & 1, abort_flag, err, kErrTimeoutMma))
          return false;
        if (!mbar_wait(bar(C::kBarVF + st), (j / C::kStages) & 1, abort_flag, err, kErrTimeoutMma))
          return false;
        tc_fence_after();
        const uint32_t a_tmem = tmem + C::kColP + (j & 1) * 64;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // V tile is [128 keys][D] in 64-column slabs: B operand MN-major,
          // 16 keys per MMA = 2 swizzle atoms of 8 rows (SBO 1024), next
          // 64 output columns one slab further (LBO = slab size).
          const uint64_t bd = smem_desc_sw128(sbase + C::kOffV + st * C::kTileBytes + kk * 2048,
                                              C::kSlabBytes, 1024);
          mma_bf16_ts(tmem + C::kColO, a_tmem + kk * 8, bd, kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(C::kBarVE + st));
        mma_commit(bar(C::kBarPE + (j & 1)));
        return true;
      };
      if (ok) ok = issue_qk(0);
      for (int j = 0; ok && j < n_tiles; ++j) {
        if (j + 1 < n_tiles) ok = issue_qk(j + 1);
        if (ok) ok = issue_pv(j);
      }
      if (!ok) {
        // Abort path: no MMA may be in flight when TMEM is released.
        mma_commit(bar(C::kBarDrain));
        mbar_wait_drain(bar(C::kBarDrain), 0, globaltimer_ns() + kWaitTimeoutNs);
      }
    }
  } else {
    // ---------------------------------------------------------- softmax
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (uint32_t(quarter * 32) << 16);
    const int q_row = q0 + row;
    // Last key this row may attend (bottom-right causal alignment).
    const int row_last = a.causal ? min(a.Nk - 1, q_row + (a.Nk - a.Nq)) : (a.Nk - 1);
    const float c = a.c_log2;
    float m = -INFINITY;  // reference maximum, log2 units of the scaled score
    float l = 0.f;        // running sum of 2^(s*c - m)
    bool ok = !dead;
    for (int j = 0; j < n_tiles; ++j) {
      const int buf = j & 1;
      ok = mbar_wait(bar(C::kBarSF + buf), (j >> 1) & 1, abort_flag, err, kErrTimeoutSoftmax);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t s[128];
      tmem_ld32(lane_base + C::kColS + buf * 128 + 0, s + 0);
      tmem_ld32(lane_base + C::kColS + buf * 128 + 32, s + 32);
      tmem_ld32(lane_base + C::kColS + buf * 128 + 64, s + 64);
      tmem_ld32(lane_base + C::kColS + buf * 128 + 96, s + 96);
      tmem_ld_wait();
      reg_fence<128>(s);

      const int lim = row_last - j * 128;  // columns > lim are masked
      if (lim < 127) {
#pragma unroll
        for (int cc = 0; cc < 128; ++cc)
          if (cc > lim) s[cc] = __float_as_uint(-INFINITY);
      }
      __syncwarp();
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = __uint_as_float(s[i]);
#pragma unroll
      for (int cc = 8; cc < 128; ++cc) mx[cc & 7] = fmaxf(mx[cc & 7], __uint_as_float(s[cc]));
      const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * c;
      // Move the reference only when the max grew by more than the threshold
      // (or on the first finite max).  alpha rescales l and O.
      const bool move = mt > m + kRescaleThreshold;
      float alpha = 1.f;
      if (move) {
        alpha = ex2_approx(m - mt);  // m == -inf -> 0
        m = mt;
        l *= alpha;
      }
      if (j > 0 && __any_sync(0xffffffffu, move)) {
        // O must not be in flight: wait for PV_{j-1}.
        ok = mbar_wait(bar(C::kBarPE + ((j - 1) & 1)), ((j - 1) >> 1) & 1, abort_flag, err,
                       kErrTimeoutSoftmax);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(lane_base + C::kColO + c0, o);
          tmem_ld_wait();
          reg_fence<32>(o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(lane_base + C::kColO + c0, o);
        }
        tmem_st_wait();
      }
      const float neg_m = (m == -INFINITY) ? 0.f : -m;
      float rs[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) rs[i] = 0.f;
      uint32_t pk[64];
#pragma unroll
      for (int cc = 0; cc < 128; cc += 2) {
        const float p0 = ex2_approx(fmaf(__uint_as_float(s[cc]), c, neg_m));
        const float p1 = ex2_approx(fmaf(__uint_as_float(s[cc + 1]), c, neg_m));
        rs[(cc >> 1) & 7] += p0 + p1;
        pk[cc >> 1] = pack_bf16x2(p0, p1);
      }
      l += ((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7]));
      if (j >= 2) {
        // P buffer `buf` was last read by PV_{j-2}.
        ok = mbar_wait(bar(C::kBarPE + buf), ((j - 2) >> 1) & 1, abort_flag, err,
                       kErrTimeoutSoftmax);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
      }
      __syncwarp();
      tmem_st32(lane_base + C::kColP + buf * 64, pk);
      tmem_st32(lane_base + C::kColP + buf * 64 + 32, pk + 32);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::kBarPF + buf));
    }

    // ---------------------------------------------------------- epilogue
    if (ok && n_tiles > 0) {
      ok = mbar_wait(bar(C::kBarPE + ((n_tiles - 1) & 1)), ((n_tiles - 1) >> 1) & 1, abort_flag,
                     err, kErrTimeoutEpilogue);
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
    }
    if (ok) {
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      uint8_t* stage = smem + C::kOffQ;  // Q is no longer read: every MMA is done
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        if (n_tiles > 0) {
          tmem_ld32(lane_base + C::kColO + c0, o);
          tmem_ld_wait();
          reg_fence<32>(o);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        uint32_t pw[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pw[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
        uint8_t* rowp = stage + (c0 >> 6) * C::kSlabBytes + row * 128;
        const int chunk0 = (c0 & 63) >> 3;
#pragma unroll
        for (int qd = 0; qd < 4; ++qd) {
          const int ch = (chunk0 + qd) ^ (row & 7);  // 128-byte swizzle, as the TMA store expects
          *reinterpret_cast<uint4*>(rowp + ch * 16) =
              make_uint4(pw[4 * qd], pw[4 * qd + 1], pw[4 * qd + 2], pw[4 * qd + 3]);
        }
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 128);
    if (!*abort_flag && ok) {
      if (warp == 2 && lane == 0) {
        for (int s = 0; s < C::kSlabs; ++s)
          tma_store_3d(&tm_o, sbase + C::kOffQ + s * C::kSlabBytes, s * 64, q0, bh);
        bulk_commit_group();
        bulk_wait_group_read0();
      }
      if (a.lse != nullptr && q_row < a.Nq)
        a.lse[size_t(bh) * a.Nq + q_row] = (l > 0.f) ? (m + log2f(l)) * kLn2 : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D>
cudaError_t launch(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int Hkv, int Nq, int Nk, float scale, int causal, cudaStream_t stream,
                   const char** err) {
  using C = Cfg<D>;
  CUtensorMap tq, tk, tv, to;
  const uint32_t box[3] = {64, 128, 1};
  const uint64_t dq[3] = {uint64_t(D), uint64_t(Nq), uint64_t(B) * H};
  const uint64_t sq[2] = {uint64_t(D) * 2, uint64_t(Nq) * D * 2};
  const uint64_t dk[3] = {uint64_t(D), uint64_t(Nk), uint64_t(B) * Hkv};
  const uint64_t sk[2] = {uint64_t(D) * 2, uint64_t(Nk) * D * 2};
  if (!encode_tmap_bf16(&tq, q, 3, dq, sq, box, true, err)) return cudaErrorInvalidValue;
  if (!encode_tmap_bf16(&tk, k, 3, dk, sk, box, true, err)) return cudaErrorInvalidValue;
  if (!encode_tmap_bf16(&tv, v, 3, dk, sk, box, true, err)) return cudaErrorInvalidValue;
  if (!encode_tmap_bf16(&to, o, 3, dq, sq, box, true, err)) return cudaErrorInvalidValue;
  static thread_local int configured_device[2] = {-1, -1};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device[D == 128] != dev) {
    e = cudaFuncSetAttribute(prefill_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device[D == 128] = dev;
  }
  Args a;
  a.lse = lse;
  a.B = B;
  a.H = H;
  a.Hkv = Hkv;
  a.Nq = Nq;
  a.Nk = Nk;
  a.n_qtiles = (Nq + 127) / 128;
  a.c_log2 = scale * kLog2e;
  a.causal = causal;
  const unsigned grid = unsigned(a.n_qtiles) * unsigned(B) * unsigned(H);
  prefill_fwd_kernel<D><<<grid, C::kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, to, a);
  return cudaGetLastError();
}

}  // namespace

int prefill_smem_bytes(int d) { return d == 128 ? Cfg<128>::kSmemBytes : Cfg<64>::kSmemBytes; }

cudaError_t prefill_launch(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                           int H, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                           cudaStream_t stream, const char** err) {
  if (d == 128) return launch<128>(q, k, v, o, lse, B, H, Hkv, Nq, Nk, scale, causal, stream, err);
  return launch<64>(q, k, v, o, lse, B, H, Hkv, Nq, Nk, scale, causal, stream, err);
}

int prefill_take_device_error() {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_prefill_error, sizeof(int)) != cudaSuccess) return -1;
  if (v != 0) cudaMemcpyToSymbol(g_prefill_error, &zero, sizeof(int));
  return v;
}

}  // namespace attn
