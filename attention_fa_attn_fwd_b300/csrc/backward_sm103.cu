// Attention backward pass for sm_103a (B300): dQ, dK, dV by recomputation.
//
// The forward pass keeps only O and the per-row log-sum-exp; the backward
// pass recomputes P from Q, K and that statistic instead of reading a stored
// N x N matrix (interview notes "他人面经整理", flashattention answer part 3,
// recomputation for the backward pass; FAQ page "Wie unterscheidet sich die
// Implementierung von FlashAttention-2 ...", comparison table, backward row).
// With S = scale Q K^T (masked) and P = softmax(S):
//   dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),  D_i = rowsum(dO_i o O_i),
//   dQ = scale dS K,  dK = scale dS^T Q,
// and a KV head's gradient sums over the query heads that read it (GQA).
//
// Two paths, all kernels on the caller's stream:
//   default at d = 128:  bwd_delta_kernel (D = rowsum(dO o O), and zeroes an
//                      fp32 dQ accumulator) + bwd_fused_kernel (key-
//                      stationary, all five products; dQ summed over key
//                      tiles with fp32 atomic adds, see its own comment) +
//                      bwd_dq_convert_kernel (dq = bf16(scale * acc)).
//   ATTN_BWD_DETERMINISTIC, and d = 64, no atomics (bit-reproducible):
//   bwd_delta_kernel   D into the workspace (bandwidth-bound).
//   bwd_dq_kernel      Q-stationary: a CTA owns 128 query rows of one head and
//                      streams the K/V tiles they attend: S = Q K^T and
//                      dP = dO V^T into TMEM, dS (bf16) back into TMEM,
//                      dQ += dS K accumulated in TMEM.
//   bwd_dkdv_kernel    KV-stationary: a CTA owns 128 keys of one KV head and
//                      streams, for every query head of its group, the Q/dO
//                      tiles that attend them (in half-tiles of 64 queries,
//                      each released as soon as its products are done):
//                      S^T = K Q^T and dP^T = V dO^T, P^T and dS^T (bf16)
//                      back into TMEM, dV += P^T dO and dK += dS^T Q
//                      accumulated in TMEM.
//   Splitting dQ from dK/dV recomputes S and dP once more (7 instead of 5
//   matrix products) but keeps every accumulator in TMEM.
//
// Warp roles in the two deterministic tcgen05 kernels (12 warps): warp 0 TMA
// producer, warp 1 MMA issuer (one elected lane), warps 2-3 idle, warps 4-7
// and 8-11 two compute warpgroups.  Every 128-wide score tile is split into
// two 64-wide halves, one per compute warpgroup, each with its own TMEM
// buffer (S and dP side by side, 64 columns each).  The MMA warp issues the next tile's
// products for one half while the other half's warpgroup is still computing,
// and the accumulating products (dQ, or dV and dK) of a half as soon as its
// warpgroup has written its bf16 operands, so the tensor pipe and the
// exponentials overlap.  A warpgroup writes its bf16 results over the first
// 32 columns of the 64-column block they came from.

#include <cmath>
#include <cstdio>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {

__device__ int g_backward_error[2];  // see ErrSink

namespace {

constexpr float kLog2e = 1.44269504088896340736f;

template <int D>
struct BCfg {
  static constexpr int kSlabs = D / 64;
  static constexpr int kSlabBytes = 128 * 128;             // 128 rows x 64 bf16
  static constexpr int kTileBytes = kSlabs * kSlabBytes;   // one 128-row tile
  static constexpr int kRegsLow = 80;
  static constexpr int kRegsHigh = 208;
  static constexpr uint32_t kTmemCols = 512;
};

// ---------------------------------------------------------------- helpers

// 32 lanes x 16 columns of 32-bit into tensor memory (one row per thread).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// 128-byte-swizzled row write of 32 fp32 values (scaled, rounded to bf16)
// into a 128-row staging tile laid out in 64-column slabs.
template <int D>
__device__ __forceinline__ void stage_row32(uint8_t* tile, int row, int c0, const uint32_t* v,
                                            float mul) {
  uint32_t pw[16];
#pragma unroll
  for (int e = 0; e < 16; ++e)
    pw[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
  uint8_t* rowp = tile + (c0 >> 6) * BCfg<D>::kSlabBytes + row * 128;
  const int chunk0 = (c0 & 63) >> 3;
#pragma unroll
  for (int qd = 0; qd < 4; ++qd) {
    const int ch = (chunk0 + qd) ^ (row & 7);
    *reinterpret_cast<uint4*>(rowp + ch * 16) =
        make_uint4(pw[4 * qd], pw[4 * qd + 1], pw[4 * qd + 2], pw[4 * qd + 3]);
  }
}

struct BArgs {
  const uint16_t* q;     // [B*H, Nq, D] bf16 (the dQ kernel reads its rows directly)
  const uint16_t* dout;  // [B*H, Nq, D] bf16
  const float* lse;  // [B, H, Nq] natural log, from the forward pass
  float* delta;      // [B, H, Nq] workspace: rowsum(dO o O)
  int B, H, Hkv, Nq, Nk;
  float c_log2;  // scale * log2(e)
  float scale;
  int causal;
  unsigned launch_id;     // set per kernel launch (see ErrSink)
  unsigned diag_wait_ns;  // != 0: CTA 0 of the key-stationary kernel lets one wait expire
};

// -log2-domain LSE: P = 2^(s * c_log2 + neg_lse2).  A row with no key
// (lse = -inf) gets -inf, i.e. P = 0.
__device__ __forceinline__ float neg_lse2_of(float lse) {
  return (lse == -INFINITY) ? -INFINITY : -lse * kLog2e;
}

// ================================================================ delta
// D[row] = sum_c dO[row, c] * O[row, c]; D/8 threads per row, 16-byte loads.
// If acc is given, the row's D fp32 dQ accumulator entries are zeroed too.
template <int D>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const uint16_t* __restrict__ o,
                                                        const uint16_t* __restrict__ dout,
                                                        float* __restrict__ delta, long long rows,
                                                        float* __restrict__ acc) {
  constexpr int TPR = D / 8;  // threads per row
  const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long row = t / TPR;
  const int part = int(t % TPR);
  float sum = 0.f;
  if (row < rows) {
    const uint4 a = *reinterpret_cast<const uint4*>(o + row * D + part * 8);
    const uint4 b = *reinterpret_cast<const uint4*>(dout + row * D + part * 8);
    const uint32_t av[4] = {a.x, a.y, a.z, a.w};
    const uint32_t bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      sum += __uint_as_float(av[e] << 16) * __uint_as_float(bv[e] << 16);
      sum += __uint_as_float(av[e] & 0xffff0000u) * __uint_as_float(bv[e] & 0xffff0000u);
    }
    if (acc) {
      float4* z = reinterpret_cast<float4*>(acc + row * D + part * 8);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if (row < rows && part == 0) delta[row] = sum;
}

// ================================================================ dQ
template <int D>
struct DqCfg : BCfg<D> {
  using B_ = BCfg<D>;
  // Q and dO live in TMEM (the A operand of S and dP), so shared memory holds
  // only the K and V stages.
  static constexpr int kKStages = (D == 128) ? 4 : 6;
  static constexpr int kVStages = (D == 128) ? 3 : 5;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKStages * B_::kTileBytes;
  static constexpr int kOffBar = kOffV + kVStages * B_::kTileBytes;
  static constexpr int kBarQF = 0;                  // Q, dO in TMEM (256 arrivals)
  static constexpr int kBarKF = 1;
  static constexpr int kBarKE = kBarKF + kKStages;
  static constexpr int kBarVF = kBarKE + kKStages;
  static constexpr int kBarVE = kBarVF + kVStages;
  static constexpr int kBarSF = kBarVE + kVStages;  // 2: S_h and dP_h of half h in TMEM
  static constexpr int kBarPF = kBarSF + 2;         // 2: dS_h written (256 arrivals each)
  static constexpr int kBarOF = kBarPF + 2;         // dQ complete
  static constexpr int kBarDrain = kBarOF + 1;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
  // half h: S_h at h*128 (64 columns), dP_h at h*128 + 64; dQ at 256;
  // Q and dO as bf16 pairs (D/2 columns each) after it.
  static constexpr uint32_t kColDQ = 256;
  static constexpr uint32_t kColQ = 256 + D;
  static constexpr uint32_t kColDO = kColQ + D / 2;
  static_assert(kColDO + D / 2 <= B_::kTmemCols, "TMEM budget");
};

template <int D>
__global__ void __launch_bounds__(384, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_dq, const BArgs a) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  // Copies the producer has issued (for the abort drain at the end; kept in
  // shared memory, not registers).
  volatile int* issued_state = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
  const ErrSink err{g_backward_error, a.launch_id};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Heavy (late, causal) query tiles first; heads of one KV group adjacent.
  const int BH = a.B * a.H;
  const int n_qt = (a.Nq + 127) / 128;
  const int bh = blockIdx.x % BH;
  const int q0 = (n_qt - 1 - int(blockIdx.x / BH)) * 128;
  const int b = bh / a.H, h = bh % a.H;
  const int zkv = b * a.Hkv + h / (a.H / a.Hkv);
  const bool dead = err.this_launch_timed_out();
  int kv_end = a.Nk;
  if (a.causal) kv_end = min(a.Nk, q0 + 128 + (a.Nk - a.Nq));
  const int n = (kv_end > 0 && !dead) ? (kv_end + 127) / 128 : 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kNumBars; ++i)
      mbar_init(bar(i), (i == C::kBarQF || i == C::kBarPF || i == C::kBarPF + 1) ? 256u : 1u);
    *abort_flag = 0;
    *issued_state = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_dq);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    setmaxnreg_dec<C::kRegsLow>();
    if (warp == 0 && n > 0) {
      // ------------------------------------------------------ producer
      // K_j and V_j complete on one barrier (K-full of K_j's stage, expecting
      // both tiles' bytes), so the MMA warp waits once per tile: every wait
      // costs that warp over 100 cycles even on a completed phase.
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < n; ++j) {
        const int ks = j % C::kKStages, vs = j % C::kVStages;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kBarKE + ks), ((j / C::kKStages) & 1) ^ 1,
                                               abort_flag, err, kErrTimeoutProducer));
        if (!ok) break;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kBarVE + vs), ((j / C::kVStages) & 1) ^ 1,
                                               abort_flag, err, kErrTimeoutProducer));
        if (!ok) break;
        mbar_arrive_expect_tx_elect(bar(C::kBarKF + ks), 2 * C::kTileBytes);
        for (int s = 0; s < C::kSlabs; ++s)
          tma_load_3d_elect(sbase + C::kOffK + ks * C::kTileBytes + s * C::kSlabBytes, &tm_k,
                            bar(C::kBarKF + ks), s * 64, j * 128, zkv);
        for (int s = 0; s < C::kSlabs; ++s)
          tma_load_3d_elect(sbase + C::kOffV + vs * C::kTileBytes + s * C::kSlabBytes, &tm_v,
                            bar(C::kBarKF + ks), s * 64, j * 128, zkv);
        issued = j + 1;
        if (lane == 0) *issued_state = issued;
      }
    } else if (warp == 1 && n > 0) {
      // ------------------------------------------------------ MMA issuer
      constexpr uint32_t kIdescHalf = idesc_bf16_f32(128, 64, 0);
      constexpr uint32_t kIdescDQ = idesc_bf16_f32(128, D, 1);
      const uint64_t k_desc = smem_desc_sw128(sbase + C::kOffK, 16, 1024);
      const uint64_t v_desc = smem_desc_sw128(sbase + C::kOffV, 16, 1024);
      const uint64_t kmn_desc = smem_desc_sw128(sbase + C::kOffK, C::kSlabBytes, 1024);
      // S_h = Q K_j[h]^T and dP_h = dO V_j[h]^T over keys h*64 .. h*64+63
      // (64 rows further into the K / V tile: +8 KB per slab).  A (Q, dO)
      // comes from TMEM, 16 elements = 8 columns per MMA, so shared memory
      // only supplies the 64-row B operand.
      auto issue_s_dp = [&](int h, int ks, int vs) {
        const uint64_t ko = uint64_t((ks * C::kTileBytes + h * 8192) >> 4);
        const uint64_t vo = uint64_t((vs * C::kTileBytes + h * 8192) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = uint64_t(((kk >> 2) * C::kSlabBytes + (kk & 3) * 32) >> 4);
          mma_bf16_ts(tmem + h * 128, tmem + C::kColQ + kk * 8, k_desc + ko + off, kIdescHalf,
                      kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = uint64_t(((kk >> 2) * C::kSlabBytes + (kk & 3) * 32) >> 4);
          mma_bf16_ts(tmem + h * 128 + 64, tmem + C::kColDO + kk * 8, v_desc + vo + off,
                      kIdescHalf, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(C::kBarSF + h));
      };
      // dQ += dS_h K_j[h]: A = dS_h (bf16 in TMEM), 16 keys per MMA; keys
      // 0-31 of the half at columns 0-15 of its block, keys 32-63 at 32-47.
      auto issue_dq = [&](int h, int j) -> bool {
        if (!__all_sync(0xffffffffu, mbar_wait(bar(C::kBarPF + h), j & 1, abort_flag, err,
                                               kErrTimeoutMma)))
          return false;
        tc_fence_after();
        const int ks = j % C::kKStages;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16_ts(tmem + C::kColDQ, tmem + h * 128 + (kk >> 1) * 32 + (kk & 1) * 8,
                      kmn_desc + uint64_t((ks * C::kTileBytes + (h * 64 + kk * 16) * 128) >> 4),
                      kIdescDQ, (j > 0 || h > 0 || kk > 0) ? 1u : 0u);
        if (h == 1) mma_commit(bar(C::kBarKE + ks));
        return true;
      };
      bool ok = __all_sync(0xffffffffu,
                           mbar_wait(bar(C::kBarQF), 0, abort_flag, err, kErrTimeoutMma));
      // Issue order: S/dP(j,0) [dQ(j-1,1)] S/dP(j,1) dQ(j,0), so one half's
      // products run while the other half's warpgroup computes.
      for (int j = 0; ok && j < n; ++j) {
        const int ks = j % C::kKStages, vs = j % C::kVStages;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kBarKF + ks), (j / C::kKStages) & 1,
                                               abort_flag, err, kErrTimeoutMma));
        if (!ok) break;
        tc_fence_after();
        issue_s_dp(0, ks, vs);
        if (j > 0) {
          ok = issue_dq(1, j - 1);
          if (!ok) break;
        }
        issue_s_dp(1, ks, vs);
        mma_commit(bar(C::kBarVE + vs));
        ok = issue_dq(0, j);
      }
      if (ok && n > 0) ok = issue_dq(1, n - 1);
      if (ok) {
        mma_commit(bar(C::kBarOF));
      } else {
        mma_commit(bar(C::kBarDrain));
        mbar_wait_drain(bar(C::kBarDrain), 0, globaltimer_ns() + kWaitTimeoutNs);
      }
    }
  } else {
    setmaxnreg_inc<C::kRegsHigh>();
    // -------------------------------------------------------- compute
    const int wg = (warp >> 2) - 1;   // which 32 columns of each 64-column half
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (uint32_t(quarter * 32) << 16);
    const int q_row = q0 + row;
    const int row_last = a.causal ? min(a.Nk - 1, q_row + (a.Nk - a.Nq)) : (a.Nk - 1);
    float neg_lse2 = -INFINITY, drow = 0.f;
    if (q_row < a.Nq) {
      neg_lse2 = neg_lse2_of(a.lse[size_t(bh) * a.Nq + q_row]);
      drow = a.delta[size_t(bh) * a.Nq + q_row];
    }
    if (n > 0) {
      // This thread's row of Q (first warpgroup) or dO (second) into TMEM as
      // bf16 pairs, the A operand of S and dP; rows past Nq are zero.
      const uint16_t* src = wg == 0 ? a.q : a.dout;
      const uint4* rp = reinterpret_cast<const uint4*>(src + (size_t(bh) * a.Nq + q_row) * D);
      const uint32_t col = wg == 0 ? C::kColQ : C::kColDO;
#pragma unroll
      for (int c0 = 0; c0 < D / 2; c0 += 32) {
        uint32_t w[32];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint4 x = q_row < a.Nq ? __ldg(rp + c0 / 4 + e) : make_uint4(0u, 0u, 0u, 0u);
          w[4 * e] = x.x;
          w[4 * e + 1] = x.y;
          w[4 * e + 2] = x.z;
          w[4 * e + 3] = x.w;
        }
        tmem_st32(lane_base + col + c0, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::kBarQF));
    }
    const float c = a.c_log2;
    bool ok = !dead;
    const float2 c2 = make_float2(c, c), nl2 = make_float2(neg_lse2, neg_lse2);
    const float2 nd2 = make_float2(-drow, -drow);
    // Both warpgroups take every half: this one its columns wg*32 .. wg*32+31
    // of S_h and dP_h, writing dS over the first 16 of them.
    for (int j = 0; ok && j < n; ++j) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait(bar(C::kBarSF + h), j & 1, abort_flag, err, kErrTimeoutSoftmax));
        if (!ok) break;
        tc_fence_after();
        const uint32_t col = h * 128 + wg * 32;
        uint32_t s[32], p[32];
        tmem_ld32(lane_base + col, s);
        tmem_ld32(lane_base + col + 64, p);
        tmem_ld_wait();
        reg_fence<32>(s);
        reg_fence<32>(p);
        const int lim = row_last - j * 128 - h * 64 - wg * 32;  // columns > lim are masked
        const bool masked = lim < 31;  // only tiles on the diagonal or the tail
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float2 x = __ffma2_rn(
              make_float2(__uint_as_float(s[2 * e]), __uint_as_float(s[2 * e + 1])), c2, nl2);
          x.x = ex2_approx(x.x);
          x.y = ex2_approx(x.y);
          if (masked) {
            if (2 * e > lim) x.x = 0.f;
            if (2 * e + 1 > lim) x.y = 0.f;
          }
          const float2 dp = __fadd2_rn(
              make_float2(__uint_as_float(p[2 * e]), __uint_as_float(p[2 * e + 1])), nd2);
          const float2 d = __fmul2_rn(x, dp);
          pk[e] = pack_bf16x2(d.x, d.y);
        }
        tmem_st16(lane_base + col, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::kBarPF + h));
      }
    }
    // -------------------------------------------------------- epilogue
    if (ok && n > 0) {
      ok = __all_sync(0xffffffffu,
                      mbar_wait(bar(C::kBarOF), 0, abort_flag, err, kErrTimeoutEpilogue));
      tc_fence_after();
    }
    uint8_t* stage = smem + C::kOffK;  // every K/V stage is consumed once dQ is complete
    if (ok) {
#pragma unroll
      for (int c0 = wg * (D / 2); c0 < (wg + 1) * (D / 2); c0 += 32) {
        uint32_t v[32];
        if (n > 0) {
          tmem_ld32(lane_base + C::kColDQ + c0, v);
          tmem_ld_wait();
          reg_fence<32>(v);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;
        }
        stage_row32<D>(stage, row, c0, v, a.scale);
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 256);
    if (!*abort_flag && ok && warp == 4 && lane == 0) {
      for (int s = 0; s < C::kSlabs; ++s)
        tma_store_3d(&tm_dq, sbase + C::kOffK + s * C::kSlabBytes, s * 64, q0, bh);
      bulk_commit_group();
      bulk_wait_group_read0();
    }
  }

  tc_fence_before();
  __syncthreads();
  // Abort path: every warp has stopped, so the flag is final.  Let every copy
  // this CTA issued land before its shared memory is released (also the ones
  // issued before another warp gave up).  Without an abort every copy has
  // been consumed, and nothing waits here.
  if (warp == 0 && *abort_flag) {
    const uint64_t deadline = globaltimer_ns() + kWaitTimeoutNs;
    const int issued = *issued_state;
    for (int j = max(0, issued - C::kKStages); j < issued; ++j)
      mbar_wait_drain(bar(C::kBarKF + j % C::kKStages), (j / C::kKStages) & 1, deadline);
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ================================================================ dK, dV
template <int D>
struct DkvCfg : BCfg<D> {
  using B_ = BCfg<D>;
  // Q and dO stream through half-stages of 64 queries each (one half of a
  // 128-query tile), so a half is released as soon as its products are done.
  static constexpr int kHalfSlabBytes = 64 * 128;                   // 64 rows x 128 B
  static constexpr int kHalfBytes = B_::kSlabs * kHalfSlabBytes;    // 64 rows of Q (or dO)
  static constexpr int kHS = (D == 128) ? 4 : 6;                    // half-stages
  static constexpr int kOffK = 0;
  static constexpr int kOffV = B_::kTileBytes;
  static constexpr int kOffQ = 2 * B_::kTileBytes;                  // Q half-stages
  static constexpr int kOffDO = kOffQ + kHS * kHalfBytes;           // dO half-stages
  static constexpr int kOffStat = kOffDO + kHS * kHalfBytes;        // [hs][2][64] fp32
  static constexpr int kOffBar = kOffStat + kHS * 2 * 64 * 4;
  static constexpr int kBarKVF = 0;
  static constexpr int kBarQF = 1;                  // kHS: half-stage full (32 arrivals + tx)
  static constexpr int kBarQE = kBarQF + kHS;       // kHS: half-stage free
  static constexpr int kBarSF = kBarQE + kHS;       // 2: S^T_h and dP^T_h in TMEM
  static constexpr int kBarPF = kBarSF + 2;         // 2: P^T_h, dS^T_h written (128 each)
  static constexpr int kBarOF = kBarPF + 2;         // dK, dV complete
  static constexpr int kBarDrain = kBarOF + 1;
  static constexpr int kBarDiag = kBarDrain + 1;    // never signalled (diagnostic wait)
  static constexpr int kNumBars = kBarDiag + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
  // half h: S^T_h at h*128 (64 columns), dP^T_h at h*128 + 64; dV, dK after.
  static constexpr uint32_t kColDV = 256, kColDK = 256 + D;
  static_assert(kHS * kHalfBytes >= B_::kTileBytes, "epilogue staging needs one tile");
};

template <int D>
__global__ void __launch_bounds__(384, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_dk,
                    const __grid_constant__ CUtensorMap tm_dv, const BArgs a) {
  using C = DkvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  // Copies the producer has issued (for the abort drain at the end; kept in
  // shared memory, not registers).
  volatile int* issued_state = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
  float* stat = reinterpret_cast<float*>(smem + C::kOffStat);
  const ErrSink err{g_backward_error, a.launch_id};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // CTA = (b, KV head, KV tile), KV tiles of one head adjacent so resident
  // CTAs share that group's Q / dO in L2; causal: early key tiles (the ones
  // most query tiles attend) first within a head.
  const int n_kt = (a.Nk + 127) / 128;
  const int zkv = blockIdx.x / n_kt;
  const int k0 = int(blockIdx.x % n_kt) * 128;
  const int b = zkv / a.Hkv, g = zkv % a.Hkv;
  const int G = a.H / a.Hkv;
  const int off = a.Nk - a.Nq;  // query row i sees keys j <= i + off (causal)
  const int n_qt = (a.Nq + 127) / 128;
  int qt0 = 0;
  if (a.causal) {
    const int first_row = k0 - off;  // first query row that sees key k0
    qt0 = first_row <= 0 ? 0 : first_row / 128;
  }
  const bool dead = err.this_launch_timed_out();
  const int per_head = max(0, n_qt - qt0);
  const int n_it = dead ? 0 : G * per_head;  // (query head, query tile) pairs

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kNumBars; ++i) {
      uint32_t cnt = 1;
      if (i == C::kBarPF || i == C::kBarPF + 1) cnt = 128;
      if (i >= C::kBarQF && i < C::kBarQF + C::kHS) cnt = 32;
      mbar_init(bar(i), cnt);
    }
    *abort_flag = 0;
    issued_state[0] = 0;  // Q / dO half-stages
    issued_state[1] = 0;  // the K and V tiles
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_do);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_dk);
    prefetch_tmap(&tm_dv);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    setmaxnreg_dec<C::kRegsLow>();
    if (warp == 0 && n_it > 0) {
      // ------------------------------------------------------ producer
      mbar_arrive_expect_tx_elect(bar(C::kBarKVF), 2 * C::kTileBytes);
      if (lane == 0) issued_state[1] = 1;
      for (int s = 0; s < C::kSlabs; ++s) {
        tma_load_3d_elect(sbase + C::kOffK + s * C::kSlabBytes, &tm_k, bar(C::kBarKVF), s * 64, k0,
                          zkv);
        tma_load_3d_elect(sbase + C::kOffV + s * C::kSlabBytes, &tm_v, bar(C::kBarKVF), s * 64, k0,
                          zkv);
      }
      bool ok = true;
      int issued = 0;
      // Half u = 2*it + h: queries h*64 .. h*64+63 of (query head, tile) it.
      // Failure-detection test (ATTN_BWD_DIAG_WAIT_EXPIRES): in CTA 0, a few
      // query halves in, the producer waits on a barrier nothing signals,
      // with a short limit, while copies and products of the CTA are in
      // flight; the wait expires and every warp of the CTA drains.
      const int diag_u = (a.diag_wait_ns != 0 && blockIdx.x == 0) ? min(4, 2 * n_it - 1) : -1;
      for (int u = 0; u < 2 * n_it; ++u) {
        if (u == diag_u) {
          __all_sync(0xffffffffu, mbar_wait_limit(bar(C::kBarDiag), 0, abort_flag, err,
                                                  kErrTimeoutDiag, a.diag_wait_ns));
          ok = false;
          break;
        }
        const int it = u >> 1, h = u & 1;
        const int hs = u % C::kHS;
        const int hq = b * a.H + g * G + it / per_head;  // query (b, h) row of the tensor maps
        const int r0 = (qt0 + it % per_head) * 128 + h * 64;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kBarQE + hs), ((u / C::kHS) & 1) ^ 1,
                                               abort_flag, err, kErrTimeoutProducer));
        if (!ok) break;
        // Row statistics of the 64 queries: -lse*log2(e) (-inf past Nq) and D.
        float* sp = stat + hs * 128;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int cidx = lane * 2 + e;
          const int r = r0 + cidx;
          float nl = -INFINITY, dd = 0.f;
          if (r < a.Nq) {
            nl = neg_lse2_of(a.lse[size_t(hq) * a.Nq + r]);
            dd = a.delta[size_t(hq) * a.Nq + r];
          }
          sp[cidx] = nl;
          sp[64 + cidx] = dd;
        }
        if (lane == 0)
          mbar_arrive_expect_tx(bar(C::kBarQF + hs), 2 * C::kHalfBytes);
        else
          mbar_arrive(bar(C::kBarQF + hs));
        __syncwarp();
        for (int s = 0; s < C::kSlabs; ++s) {
          tma_load_3d_elect(sbase + C::kOffQ + hs * C::kHalfBytes + s * C::kHalfSlabBytes, &tm_q,
                            bar(C::kBarQF + hs), s * 64, r0, hq);
          tma_load_3d_elect(sbase + C::kOffDO + hs * C::kHalfBytes + s * C::kHalfSlabBytes, &tm_do,
                            bar(C::kBarQF + hs), s * 64, r0, hq);
        }
        issued = u + 1;
        if (lane == 0) issued_state[0] = issued;
      }
    } else if (warp == 1 && n_it > 0) {
      // ------------------------------------------------------ MMA issuer
      constexpr uint32_t kIdescHalf = idesc_bf16_f32(128, 64, 0);
      constexpr uint32_t kIdescAcc = idesc_bf16_f32(128, D, 1);
      const uint64_t k_desc = smem_desc_sw128(sbase + C::kOffK, 16, 1024);
      const uint64_t v_desc = smem_desc_sw128(sbase + C::kOffV, 16, 1024);
      const uint64_t q_desc = smem_desc_sw128(sbase + C::kOffQ, 16, 1024);
      const uint64_t do_desc = smem_desc_sw128(sbase + C::kOffDO, 16, 1024);
      const uint64_t qmn_desc = smem_desc_sw128(sbase + C::kOffQ, C::kHalfSlabBytes, 1024);
      const uint64_t domn_desc = smem_desc_sw128(sbase + C::kOffDO, C::kHalfSlabBytes, 1024);
      // S^T_h = K Q[h]^T, dP^T_h = V dO[h]^T over the 64 queries of half u.
      auto issue_s_dp = [&](int u) -> bool {
        const int h = u & 1, hs = u % C::kHS;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(C::kBarQF + hs), (u / C::kHS) & 1, abort_flag,
                                               err, kErrTimeoutMma)))
          return false;
        tc_fence_after();
        const uint64_t so = uint64_t((hs * C::kHalfBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t ok_ = uint64_t(((kk >> 2) * C::kSlabBytes + (kk & 3) * 32) >> 4);
          const uint64_t oq = uint64_t(((kk >> 2) * C::kHalfSlabBytes + (kk & 3) * 32) >> 4);
          mma_bf16_ss(tmem + h * 128, k_desc + ok_, q_desc + so + oq, kIdescHalf,
                      kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t ok_ = uint64_t(((kk >> 2) * C::kSlabBytes + (kk & 3) * 32) >> 4);
          const uint64_t oq = uint64_t(((kk >> 2) * C::kHalfSlabBytes + (kk & 3) * 32) >> 4);
          mma_bf16_ss(tmem + h * 128 + 64, v_desc + ok_, do_desc + so + oq, kIdescHalf,
                      kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(C::kBarSF + h));
        return true;
      };
      // dV += P^T_h dO[h], dK += dS^T_h Q[h] (16 queries per MMA); frees the half-stage.
      auto issue_acc = [&](int u) -> bool {
        const int h = u & 1, hs = u % C::kHS;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(C::kBarPF + h), (u >> 1) & 1, abort_flag, err,
                                               kErrTimeoutMma)))
          return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t o16 = uint64_t((hs * C::kHalfBytes + kk * 16 * 128) >> 4);
          const uint32_t acc = (u > 0 || kk > 0) ? 1u : 0u;
          mma_bf16_ts(tmem + C::kColDV, tmem + h * 128 + kk * 8, domn_desc + o16, kIdescAcc, acc);
          mma_bf16_ts(tmem + C::kColDK, tmem + h * 128 + 64 + kk * 8, qmn_desc + o16, kIdescAcc,
                      acc);
        }
        mma_commit(bar(C::kBarQE + hs));
        return true;
      };
      bool ok = __all_sync(0xffffffffu,
                           mbar_wait(bar(C::kBarKVF), 0, abort_flag, err, kErrTimeoutMma));
      // Issue order per tile it: S/dP(it,0) [acc(it-1,1)] S/dP(it,1) acc(it,0).
      for (int it = 0; ok && it < n_it; ++it) {
        ok = issue_s_dp(2 * it);
        if (ok && it > 0) ok = issue_acc(2 * it - 1);
        if (ok) ok = issue_s_dp(2 * it + 1);
        if (ok) ok = issue_acc(2 * it);
      }
      if (ok && n_it > 0) ok = issue_acc(2 * n_it - 1);
      if (ok) {
        mma_commit(bar(C::kBarOF));
      } else {
        mma_commit(bar(C::kBarDrain));
        mbar_wait_drain(bar(C::kBarDrain), 0, globaltimer_ns() + kWaitTimeoutNs);
      }
    }
  } else {
    setmaxnreg_inc<C::kRegsHigh>();
    // -------------------------------------------------------- compute
    const int wg = (warp >> 2) - 1;  // which 64-query half of the tile
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // key within the tile
    const uint32_t lane_base = tmem + (uint32_t(quarter * 32) << 16);
    const int kj = k0 + row;
    const float c = a.c_log2;
    bool ok = !dead;
    for (int it = 0; ok && it < n_it; ++it) {
      const int u = 2 * it + wg, hs = u % C::kHS;
      const int r0 = (qt0 + it % per_head) * 128;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kBarQF + hs), (u / C::kHS) & 1,
                                             abort_flag, err, kErrTimeoutSoftmax));
      if (!ok) break;
      ok = __all_sync(0xffffffffu,
                      mbar_wait(bar(C::kBarSF + wg), it & 1, abort_flag, err, kErrTimeoutSoftmax));
      if (!ok) break;
      tc_fence_after();
      uint32_t s[64], p[64];
      tmem_ld32(lane_base + wg * 128, s);
      tmem_ld32(lane_base + wg * 128 + 32, s + 32);
      tmem_ld32(lane_base + wg * 128 + 64, p);
      tmem_ld32(lane_base + wg * 128 + 96, p + 32);
      tmem_ld_wait();
      reg_fence<64>(s);
      reg_fence<64>(p);
      const float* nl = stat + hs * 128;
      const float* dd = nl + 64;
      // Column q (query r0 + wg*64 + q) is masked if this key is past Nk or,
      // causally, if kj > query + off, i.e. q < kj - off - r0 - wg*64.
      const int lo = a.causal ? (kj - off - r0 - wg * 64) : -1;
      const bool key_ok = kj < a.Nk;
      const bool masked = !key_ok || lo > 0;  // only tiles on the diagonal or the key tail
      const float2 c2 = make_float2(c, c);
      const float2* nl2 = reinterpret_cast<const float2*>(nl);
      const float2* dd2 = reinterpret_cast<const float2*>(dd);
      uint32_t pp[32], pd[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        float2 x = __ffma2_rn(make_float2(__uint_as_float(s[2 * e]), __uint_as_float(s[2 * e + 1])),
                              c2, nl2[e]);
        x.x = ex2_approx(x.x);
        x.y = ex2_approx(x.y);
        if (masked) {
          if (!key_ok || 2 * e < lo) x.x = 0.f;
          if (!key_ok || 2 * e + 1 < lo) x.y = 0.f;
        }
        pp[e] = pack_bf16x2(x.x, x.y);
        const float2 ndd = dd2[e];
        const float2 dp = __fadd2_rn(make_float2(__uint_as_float(p[2 * e]), __uint_as_float(p[2 * e + 1])),
                                     make_float2(-ndd.x, -ndd.y));
        const float2 d = __fmul2_rn(x, dp);
        pd[e] = pack_bf16x2(d.x, d.y);
      }
      tmem_st32(lane_base + wg * 128, pp);
      tmem_st32(lane_base + wg * 128 + 64, pd);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::kBarPF + wg));
    }
    // -------------------------------------------------------- epilogue
    if (ok && n_it > 0) {
      ok = __all_sync(0xffffffffu,
                      mbar_wait(bar(C::kBarOF), 0, abort_flag, err, kErrTimeoutEpilogue));
      tc_fence_after();
    }
    // wg 0 writes dV through Q stage 0, wg 1 writes scale * dK through dO stage 0.
    uint8_t* stage = smem + (wg == 0 ? C::kOffQ : C::kOffDO);
    const uint32_t col = wg == 0 ? C::kColDV : C::kColDK;
    const float mul = wg == 0 ? 1.f : a.scale;
    if (ok) {
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t v[32];
        if (n_it > 0) {
          tmem_ld32(lane_base + col + c0, v);
          tmem_ld_wait();
          reg_fence<32>(v);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;
        }
        stage_row32<D>(stage, row, c0, v, mul);
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1 + wg, 128);
    if (!*abort_flag && ok && quarter == 0 && lane == 0) {
      const CUtensorMap* tm = wg == 0 ? &tm_dv : &tm_dk;
      const uint32_t src = sbase + (wg == 0 ? C::kOffQ : C::kOffDO);
      for (int s = 0; s < C::kSlabs; ++s)
        tma_store_3d(tm, src + s * C::kSlabBytes, s * 64, k0, zkv);
      bulk_commit_group();
      bulk_wait_group_read0();
    }
  }

  tc_fence_before();
  __syncthreads();
  // Abort path: every warp has stopped, so the flag is final.  Let every copy
  // this CTA issued land before its shared memory is released (also the ones
  // issued before another warp gave up).  Without an abort every copy has
  // been consumed, and nothing waits here.
  if (warp == 0 && *abort_flag) {
    const uint64_t deadline = globaltimer_ns() + kWaitTimeoutNs;
    const int issued = issued_state[0];
    const bool issued_kv = issued_state[1] != 0;
    if (issued_kv) mbar_wait_drain(bar(C::kBarKVF), 0, deadline);
    for (int u = max(0, issued - C::kHS); u < issued; ++u)
      mbar_wait_drain(bar(C::kBarQF + u % C::kHS), (u / C::kHS) & 1, deadline);
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ================================================================ fused (d = 128)
// One KV-stationary kernel for all five products.  A CTA owns 128 keys of
// one KV head and streams the 64-query halves of every (query head, query
// tile) that sees them, as bwd_dkdv_kernel does, and also forms this key
// tile's share of dQ:
//   dQ^T_u = K^T dS^T_u   (M = d = 128, N = 64 queries, K = 128 keys)
// from the bf16 dS^T the compute warpgroup writes to shared memory (P^T and
// dS^T also go back to TMEM, over the S^T columns they came from, as the A
// operands of dV and dK).  dQ^T lands in the half's dP^T columns of TMEM
// (free once the compute warpgroup has read them); a fourth warpgroup reads
// it out (lane = d, so a
// warp's 32 lanes cover 32 consecutive floats of one query row) and adds it
// to an fp32 dQ accumulator in the workspace with coalesced atomic adds in
// L2.  A conversion kernel then writes dq = bf16(scale * accumulator).  The
// adds from different key tiles arrive in no fixed order, so dq can differ
// between calls by fp32 rounding; dk and dv are accumulated in TMEM in a
// fixed order and are bit-reproducible.
//
// Warps: 0 TMA producer, 1-2 MMA issuers, 3 idle, 4-7 compute half 0,
// 8-11 compute half 1, 12-15 dQ drain.
struct FusedCfg : BCfg<128> {
  using B_ = BCfg<128>;
  static constexpr int kHalfSlabBytes = 64 * 128;
  static constexpr int kHalfBytes = B_::kSlabs * kHalfSlabBytes;  // 64 rows x 128 bf16
  // Q / dO half-stages: 3 and 4 measured the same on the long-context
  // workload (5.01 vs 5.04 ms); 3 leaves the layout 1 KB of alignment slack.
  static constexpr int kHS = 3;
  static constexpr int kDSBytes = 128 * 128;                      // dS^T: 128 keys x 64 q bf16
  static constexpr int kOffK = 0;
  static constexpr int kOffV = B_::kTileBytes;
  static constexpr int kOffQ = 2 * B_::kTileBytes;
  static constexpr int kOffDO = kOffQ + kHS * kHalfBytes;
  static constexpr int kOffDS = kOffDO + kHS * kHalfBytes;        // 2 dS^T tiles (one per half)
  static constexpr int kOffStat = kOffDS + 2 * kDSBytes;          // [hs][2][64] fp32
  static constexpr int kOffBar = kOffStat + kHS * 2 * 64 * 4;
  static constexpr int kBarKVF = 0;
  static constexpr int kBarQF = 1;                 // kHS (32 arrivals + tx)
  static constexpr int kBarQE = kBarQF + kHS;      // kHS
  static constexpr int kBarSF = kBarQE + kHS;      // 2: S^T_h, dP^T_h in TMEM
  static constexpr int kBarPF = kBarSF + 2;        // 2: P^T_h, dS^T_h written (128 arrivals)
  static constexpr int kBarDQF = kBarPF + 2;       // 2: dQ^T_h in TMEM
  static constexpr int kBarDQE = kBarDQF + 2;      // 2: dQ^T_h read out (128 arrivals)
  static constexpr int kBarSE = kBarDQE + 2;       // 2: dV, dK of half h done (S^T_h free)
  static constexpr int kBarOF = kBarSE + 2;        // dK, dV complete
  static constexpr int kBarDrain = kBarOF + 1;     // abort drains of the two MMA warps
  static constexpr int kBarDrain2 = kBarDrain + 1;
  static constexpr int kBarDiag = kBarDrain2 + 1;  // never signalled (diagnostic wait)
  static constexpr int kNumBars = kBarDiag + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
  // half h: S^T_h at h*128 (64 columns; P^T_h then dS^T_h as bf16 pairs over
  // its first 32 and second 32), dP^T_h at h*128 + 64 (then dQ^T_h).
  static constexpr uint32_t kColDV = 256, kColDK = 384;
  static constexpr int kRegsLow = 72, kRegsDrain = 72, kRegsHigh = 176;
  static_assert(kHS * kHalfBytes >= B_::kTileBytes, "epilogue staging needs one tile");
  static_assert(kRegsLow * 128 + kRegsDrain * 128 + kRegsHigh * 256 <= 65536, "register split");
};

__global__ void __launch_bounds__(512, 1)
    bwd_fused_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_dk,
                     const __grid_constant__ CUtensorMap tm_dv, const BArgs a, float* dq_acc) {
  using C = FusedCfg;
  constexpr int D = 128;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  // Copies the producer has issued (for the abort drain at the end; kept in
  // shared memory, not registers).
  volatile int* issued_state = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
  float* stat = reinterpret_cast<float*>(smem + C::kOffStat);
  const ErrSink err{g_backward_error, a.launch_id};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // CTA = (b, KV head, key tile); key tiles of one head adjacent (L2 reuse of
  // the group's Q / dO and of its dQ accumulator rows).
  const int n_kt = (a.Nk + 127) / 128;
  const int zkv = blockIdx.x / n_kt;
  const int k0 = int(blockIdx.x % n_kt) * 128;
  const int b = zkv / a.Hkv, g = zkv % a.Hkv;
  const int G = a.H / a.Hkv;
  const int off = a.Nk - a.Nq;
  const int n_qt = (a.Nq + 127) / 128;
  int qt0 = 0;
  if (a.causal) {
    const int first_row = k0 - off;
    qt0 = first_row <= 0 ? 0 : first_row / 128;
  }
  const bool dead = err.this_launch_timed_out();
  const int per_head = max(0, n_qt - qt0);
  const int n_it = dead ? 0 : G * per_head;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kNumBars; ++i) {
      uint32_t cnt = 1;
      if (i == C::kBarPF || i == C::kBarPF + 1 || i == C::kBarDQE || i == C::kBarDQE + 1) cnt = 128;
      if (i >= C::kBarQF && i < C::kBarQF + C::kHS) cnt = 32;
      mbar_init(bar(i), cnt);
    }
    *abort_flag = 0;
    issued_state[0] = 0;  // Q / dO half-stages
    issued_state[1] = 0;  // the K and V tiles
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_do);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_dk);
    prefetch_tmap(&tm_dv);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    setmaxnreg_dec<C::kRegsLow>();
    if (warp == 0 && n_it > 0) {
      // ------------------------------------------------------ producer
      mbar_arrive_expect_tx_elect(bar(C::kBarKVF), 2 * C::kTileBytes);
      if (lane == 0) issued_state[1] = 1;
      for (int s = 0; s < C::kSlabs; ++s) {
        tma_load_3d_elect(sbase + C::kOffK + s * C::kSlabBytes, &tm_k, bar(C::kBarKVF), s * 64, k0,
                          zkv);
        tma_load_3d_elect(sbase + C::kOffV + s * C::kSlabBytes, &tm_v, bar(C::kBarKVF), s * 64, k0,
                          zkv);
      }
      bool ok = true;
      int issued = 0;
      // The per-query statistics of half u are read from global memory one
      // half ahead, so that their latency overlaps the wait for a free stage
      // instead of delaying the copies.
      float st_nl[2], st_dd[2];  // lse and D of this lane's two queries
      auto load_stats = [&](int u) {
        const int it = u >> 1;
        const int hq = b * a.H + g * G + it / per_head;
        const int r0 = (qt0 + it % per_head) * 128 + (u & 1) * 64;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int r = r0 + lane * 2 + e;
          st_nl[e] = -INFINITY;
          st_dd[e] = 0.f;
          if (u < 2 * n_it && r < a.Nq) {
            st_nl[e] = a.lse[size_t(hq) * a.Nq + r];
            st_dd[e] = a.delta[size_t(hq) * a.Nq + r];
          }
        }
      };
      load_stats(0);
      // Failure-detection test (ATTN_BWD_DIAG_WAIT_EXPIRES): in CTA 0, a few
      // query halves in, the producer waits on a barrier nothing signals,
      // with a short limit, while copies and products of the CTA are in
      // flight; the wait expires and every warp of the CTA drains.
      const int diag_u = (a.diag_wait_ns != 0 && blockIdx.x == 0) ? min(4, 2 * n_it - 1) : -1;
      for (int u = 0; u < 2 * n_it; ++u) {
        if (u == diag_u) {
          __all_sync(0xffffffffu, mbar_wait_limit(bar(C::kBarDiag), 0, abort_flag, err,
                                                  kErrTimeoutDiag, a.diag_wait_ns));
          ok = false;
          break;
        }
        const int it = u >> 1, h = u & 1;
        const int hs = u % C::kHS;
        const int hq = b * a.H + g * G + it / per_head;
        const int r0 = (qt0 + it % per_head) * 128 + h * 64;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kBarQE + hs), ((u / C::kHS) & 1) ^ 1,
                                               abort_flag, err, kErrTimeoutProducer));
        if (!ok) break;
        float* sp = stat + hs * 128;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int cidx = lane * 2 + e;
          // lse = -inf past Nq (and on rows that see no key): P = 0 there
          sp[cidx] = neg_lse2_of(st_nl[e]);
          sp[64 + cidx] = st_dd[e];
        }
        if (lane == 0)
          mbar_arrive_expect_tx(bar(C::kBarQF + hs), 2 * C::kHalfBytes);
        else
          mbar_arrive(bar(C::kBarQF + hs));
        __syncwarp();
        for (int s = 0; s < C::kSlabs; ++s) {
          tma_load_3d_elect(sbase + C::kOffQ + hs * C::kHalfBytes + s * C::kHalfSlabBytes, &tm_q,
                            bar(C::kBarQF + hs), s * 64, r0, hq);
          tma_load_3d_elect(sbase + C::kOffDO + hs * C::kHalfBytes + s * C::kHalfSlabBytes, &tm_do,
                            bar(C::kBarQF + hs), s * 64, r0, hq);
        }
        issued = u + 1;
        if (lane == 0) issued_state[0] = issued;
        load_stats(u + 1);
      }
    } else if ((warp == 1 || warp == 2) && n_it > 0) {
      // ---------------------------------------------- MMA issuers (two warps)
      // The tcgen05 queue holds only a few MMAs, and one warp that both
      // issues and waits leaves the tensor pipe idle during every wait, even
      // on a barrier whose phase completed long before (~250 cycles each,
      // three per half, measured).  So two warps issue into the one pipe,
      // each waiting while the other's products run:
      //   warp 1: S^T(u), dP^T(u)           (waits: Q/dO loaded, S^T_h free,
      //                                      dQ^T(u-2) read out)
      //   warp 2: dV, dK (u), then dQ^T(u)  (wait: P^T, dS^T of u written)
      // What a single issuing warp got from its issue order now comes from
      // barriers: S^T(u) overwrites the P^T / dS^T of u - 2 only after
      // dV, dK(u - 2) (kBarSE); dP^T(u) overwrites dQ^T(u - 2) only after the
      // drain has read it (kBarDQE), which also means dQ^T(u - 2) is complete
      // before the compute warpgroup of u writes dS^T_h again (it waits for
      // dP^T(u)).  dV and dK are issued by warp 2 alone, in a fixed order.
      const uint64_t k_desc = smem_desc_sw128(sbase + C::kOffK, 16, 1024);
      auto wait_on = [&](int which, uint32_t parity) -> bool {
        if (!__all_sync(0xffffffffu,
                        mbar_wait(bar(which), parity, abort_flag, err, kErrTimeoutMma)))
          return false;
        tc_fence_after();
        return true;
      };
      const int n_u = 2 * n_it;
      bool ok = wait_on(C::kBarKVF, 0);
      if (warp == 1) {
        constexpr uint32_t kIdescHalf = idesc_bf16_f32(128, 64, 0);
        const uint64_t v_desc = smem_desc_sw128(sbase + C::kOffV, 16, 1024);
        const uint64_t q_desc = smem_desc_sw128(sbase + C::kOffQ, 16, 1024);
        const uint64_t do_desc = smem_desc_sw128(sbase + C::kOffDO, 16, 1024);
        for (int u = 0; ok && u < n_u; ++u) {
          const int h = u & 1, hs = u % C::kHS;
          ok = wait_on(C::kBarQF + hs, (u / C::kHS) & 1);  // Q, dO of half u loaded
          if (ok && u >= 2) ok = wait_on(C::kBarSE + h, ((u >> 1) - 1) & 1);  // dV, dK(u-2) done
          if (!ok) break;
          // S^T_h = K Q[u]^T over the 64 queries of half u: two chains of
          // four K-steps (32 bytes apart inside a 64-column slab; the second
          // chain in the next slab).
          const uint64_t qd = q_desc + uint64_t((hs * C::kHalfBytes) >> 4);
          mma4_bf16_ss<2, 2>(tmem + h * 128, k_desc, qd, kIdescHalf, 0u);
          mma4_bf16_ss<2, 2>(tmem + h * 128, k_desc + (C::kSlabBytes >> 4),
                             qd + (C::kHalfSlabBytes >> 4), kIdescHalf, 1u);
          // dP^T_h = V dO[u]^T into the half's second 64 columns, which hold
          // dQ^T of half u - 2 until the drain warpgroup has read it.
          if (u >= 2) ok = wait_on(C::kBarDQE + h, ((u >> 1) - 1) & 1);
          if (!ok) break;
          const uint64_t dd = do_desc + uint64_t((hs * C::kHalfBytes) >> 4);
          mma4_bf16_ss<2, 2>(tmem + h * 128 + 64, v_desc, dd, kIdescHalf, 0u);
          mma4_bf16_ss<2, 2>(tmem + h * 128 + 64, v_desc + (C::kSlabBytes >> 4),
                             dd + (C::kHalfSlabBytes >> 4), kIdescHalf, 1u);
          mma_commit(bar(C::kBarSF + h));
        }
        if (!ok) {
          mma_commit(bar(C::kBarDrain));
          mbar_wait_drain(bar(C::kBarDrain), 0, globaltimer_ns() + kWaitTimeoutNs);
        }
      } else {
        constexpr uint32_t kIdescAcc = idesc_bf16_f32(128, D, 1);
        constexpr uint32_t kIdescDQ = idesc_bf16_f32_amn(128, 64, 1);
        const uint64_t qmn_desc = smem_desc_sw128(sbase + C::kOffQ, C::kHalfSlabBytes, 1024);
        const uint64_t domn_desc = smem_desc_sw128(sbase + C::kOffDO, C::kHalfSlabBytes, 1024);
        // K^T as an MN-major A operand (M = d: 64-column slabs kSlabBytes
        // apart); dS^T as an MN-major B operand (N = 64 queries, one atom).
        const uint64_t kmn_desc = smem_desc_sw128(sbase + C::kOffK, C::kSlabBytes, 1024);
        const uint64_t ds_desc = smem_desc_sw128(sbase + C::kOffDS, C::kDSBytes, 1024);
        for (int u = 0; ok && u < n_u; ++u) {
          const int h = u & 1, hs = u % C::kHS;
          ok = wait_on(C::kBarPF + h, (u >> 1) & 1);  // P^T, dS^T of half u written
          if (!ok) break;
          // dV += P^T_h dO[u], dK += dS^T_h Q[u]; then the half-stage and
          // the S^T_h columns are free.  Queries 32c..32c+31 of the half
          // have P^T in columns 32c..32c+15 of S^T_h and dS^T in the next 16
          // (8 columns = 16 queries per K-step).
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t o16 = uint32_t((hs * C::kHalfBytes + kk * 16 * 128) >> 4);
            const uint32_t acc = (u > 0 || kk > 0) ? 1u : 0u;
            const uint32_t pcol = h * 128 + (kk >> 1) * 32 + (kk & 1) * 8;
            mma_bf16_ts(tmem + C::kColDV, tmem + pcol, desc_add(domn_desc, o16), kIdescAcc, acc);
            mma_bf16_ts(tmem + C::kColDK, tmem + pcol + 16, desc_add(qmn_desc, o16), kIdescAcc,
                        acc);
          }
          mma_commit(bar(C::kBarQE + hs));
          mma_commit(bar(C::kBarSE + h));
          // dQ^T_h = K^T dS^T_h (16 keys = 2048 bytes per MMA in both operands).
          const uint64_t dsd = ds_desc + uint64_t((h * C::kDSBytes) >> 4);
          mma4_bf16_ss<128, 128>(tmem + h * 128 + 64, kmn_desc, dsd, kIdescDQ, 0u);
          mma4_bf16_ss<128, 128>(tmem + h * 128 + 64, kmn_desc + 512, dsd + 512, kIdescDQ, 1u);
          mma_commit(bar(C::kBarDQF + h));
        }
        if (ok) {
          mma_commit(bar(C::kBarOF));
        } else {
          mma_commit(bar(C::kBarDrain2));
          mbar_wait_drain(bar(C::kBarDrain2), 0, globaltimer_ns() + kWaitTimeoutNs);
        }
      }
    }
  } else if (warp >= 12) {
    setmaxnreg_dec<C::kRegsDrain>();
    // -------------------------------------------------------- dQ drain
    const int quarter = warp & 3;
    const uint32_t lane_base = tmem + (uint32_t(quarter * 32) << 16);
    const int dcol = quarter * 32 + lane;
    bool ok = !dead;
    for (int u = 0; ok && u < 2 * n_it; ++u) {
      const int it = u >> 1, h = u & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kBarDQF + h), (u >> 1) & 1, abort_flag, err,
                                             kErrTimeoutEpilogue));
      if (!ok) break;
      tc_fence_after();
      uint32_t v[64];
      tmem_ld32(lane_base + h * 128 + 64, v);
      tmem_ld32(lane_base + h * 128 + 96, v + 32);
      tmem_ld_wait();
      reg_fence<64>(v);
      tc_fence_before();
      mbar_arrive(bar(C::kBarDQE + h));
      const int hq = b * a.H + g * G + it / per_head;
      const int r0 = (qt0 + it % per_head) * 128 + h * 64;
      const int nrow = min(64, a.Nq - r0);
      float* dst = dq_acc + (size_t(hq) * a.Nq + r0) * D + dcol;
#pragma unroll
      for (int j = 0; j < 64; ++j)
        if (j < nrow) atomicAdd(dst + size_t(j) * D, __uint_as_float(v[j]));
    }
  } else {
    setmaxnreg_inc<C::kRegsHigh>();
    // -------------------------------------------------------- compute
    const int wg = (warp >> 2) - 1;  // which 64-query half of the tile
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // key within the tile
    const uint32_t lane_base = tmem + (uint32_t(quarter * 32) << 16);
    const int kj = k0 + row;
    const float c = a.c_log2;
    uint8_t* ds_row = smem + C::kOffDS + wg * C::kDSBytes + row * 128;
    bool ok = !dead;
    for (int it = 0; ok && it < n_it; ++it) {
      const int u = 2 * it + wg, hs = u % C::kHS;
      const int r0 = (qt0 + it % per_head) * 128;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kBarQF + hs), (u / C::kHS) & 1,
                                             abort_flag, err, kErrTimeoutSoftmax));
      if (!ok) break;
      ok = __all_sync(0xffffffffu,
                      mbar_wait(bar(C::kBarSF + wg), it & 1, abort_flag, err, kErrTimeoutSoftmax));
      if (!ok) break;
      tc_fence_after();
      const float* nl = stat + hs * 128;
      const float* dd = nl + 64;
      const int lo = a.causal ? (kj - off - r0 - wg * 64) : -1;
      const bool key_ok = kj < a.Nk;
      const bool masked = !key_ok || lo > 0;
      const float2 c2 = make_float2(c, c);
      // Two chunks of 32 queries, each finished (P^T and dS^T to TMEM, dS^T
      // to shared memory) before the next is loaded: a third of the live
      // registers of one pass over 64, so the exponentials of several
      // columns overlap.
#pragma unroll
      for (int chk = 0; chk < 2; ++chk) {
        uint32_t s[32], p[32];
        tmem_ld32(lane_base + wg * 128 + chk * 32, s);
        tmem_ld32(lane_base + wg * 128 + 64 + chk * 32, p);
        tmem_ld_wait();
        reg_fence<32>(s);
        reg_fence<32>(p);
        uint32_t pp[16], pd[16];
#pragma unroll
        for (int el = 0; el < 16; ++el) {
          const int e = chk * 16 + el;  // pair within the half
          const float2 nlp = reinterpret_cast<const float2*>(nl)[e];
          const float2 ddp = reinterpret_cast<const float2*>(dd)[e];
          float2 x = __ffma2_rn(
              make_float2(__uint_as_float(s[2 * el]), __uint_as_float(s[2 * el + 1])), c2, nlp);
          x.x = ex2_approx(x.x);
          x.y = ex2_approx(x.y);
          if (masked) {
            if (!key_ok || 2 * e < lo) x.x = 0.f;
            if (!key_ok || 2 * e + 1 < lo) x.y = 0.f;
          }
          pp[el] = pack_bf16x2(x.x, x.y);
          const float2 dp =
              __fadd2_rn(make_float2(__uint_as_float(p[2 * el]), __uint_as_float(p[2 * el + 1])),
                         make_float2(-ddp.x, -ddp.y));
          const float2 d = __fmul2_rn(x, dp);
          pd[el] = pack_bf16x2(d.x, d.y);
        }
        // dS^T of these 32 queries (64 bytes of this key's row) into the
        // half's shared tile, 128-byte swizzled: the B operand of dQ^T.
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int ch = chk * 4 + q4;
          *reinterpret_cast<uint4*>(ds_row + ((ch ^ (row & 7)) << 4)) =
              make_uint4(pd[4 * q4], pd[4 * q4 + 1], pd[4 * q4 + 2], pd[4 * q4 + 3]);
        }
        // P^T and dS^T of these 32 queries over the 32 S^T columns this
        // chunk has just read (the other chunk's S^T stays intact).
        tmem_st16(lane_base + wg * 128 + chk * 32, pp);
        tmem_st16(lane_base + wg * 128 + chk * 32 + 16, pd);
      }
      fence_proxy_async_smem();
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::kBarPF + wg));
    }
    // -------------------------------------------------------- epilogue
    if (ok && n_it > 0) {
      ok = __all_sync(0xffffffffu,
                      mbar_wait(bar(C::kBarOF), 0, abort_flag, err, kErrTimeoutEpilogue));
      tc_fence_after();
    }
    uint8_t* stage = smem + (wg == 0 ? C::kOffQ : C::kOffDO);
    const uint32_t col = wg == 0 ? C::kColDV : C::kColDK;
    const float mul = wg == 0 ? 1.f : a.scale;
    if (ok) {
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t v[32];
        if (n_it > 0) {
          tmem_ld32(lane_base + col + c0, v);
          tmem_ld_wait();
          reg_fence<32>(v);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;
        }
        stage_row32<D>(stage, row, c0, v, mul);
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1 + wg, 128);
    if (!*abort_flag && ok && quarter == 0 && lane == 0) {
      const CUtensorMap* tm = wg == 0 ? &tm_dv : &tm_dk;
      const uint32_t src = sbase + (wg == 0 ? C::kOffQ : C::kOffDO);
      for (int s = 0; s < C::kSlabs; ++s)
        tma_store_3d(tm, src + s * C::kSlabBytes, s * 64, k0, zkv);
      bulk_commit_group();
      bulk_wait_group_read0();
    }
  }

  tc_fence_before();
  __syncthreads();
  // Abort path: every warp has stopped, so the flag is final.  Let every copy
  // this CTA issued land before its shared memory is released (also the ones
  // issued before another warp gave up).  Without an abort every copy has
  // been consumed, and nothing waits here.
  if (warp == 0 && *abort_flag) {
    const uint64_t deadline = globaltimer_ns() + kWaitTimeoutNs;
    const int issued = issued_state[0];
    const bool issued_kv = issued_state[1] != 0;
    if (issued_kv) mbar_wait_drain(bar(C::kBarKVF), 0, deadline);
    for (int u = max(0, issued - C::kHS); u < issued; ++u)
      mbar_wait_drain(bar(C::kBarQF + u % C::kHS), (u / C::kHS) & 1, deadline);
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// dq = bf16(scale * accumulator), 8 elements per thread.
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float* __restrict__ acc,
                                                             uint16_t* __restrict__ dq,
                                                             long long n8, float scale) {
  const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n8) return;
  const float4 x = reinterpret_cast<const float4*>(acc)[2 * t];
  const float4 y = reinterpret_cast<const float4*>(acc)[2 * t + 1];
  uint4 r;
  r.x = pack_bf16x2(x.x * scale, x.y * scale);
  r.y = pack_bf16x2(x.z * scale, x.w * scale);
  r.z = pack_bf16x2(y.x * scale, y.y * scale);
  r.w = pack_bf16x2(y.z * scale, y.w * scale);
  reinterpret_cast<uint4*>(dq)[t] = r;
}

// ================================================================ launch

template <typename K>
cudaError_t set_smem_once(K kernel, int bytes, int* configured) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (*configured != dev) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    *configured = dev;
  }
  return cudaSuccess;
}

template <int D>
cudaError_t launch_bwd(const void* q, const void* k, const void* v, const void* o,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                       int H, int Hkv, int Nq, int Nk, float scale, int causal, float* delta,
                       float* dq_acc, unsigned diag_wait_ns, cudaStream_t stream,
                       const char** err) {
  const uint32_t box[3] = {64, 128, 1};
  const uint64_t dq_[3] = {uint64_t(D), uint64_t(Nq), uint64_t(B) * H};
  const uint64_t sq[2] = {uint64_t(D) * 2, uint64_t(Nq) * D * 2};
  const uint64_t dk_[3] = {uint64_t(D), uint64_t(Nk), uint64_t(B) * Hkv};
  const uint64_t sk[2] = {uint64_t(D) * 2, uint64_t(Nk) * D * 2};
  const uint32_t box64[3] = {64, 64, 1};
  const bool fused = (D == 128) && dq_acc != nullptr;
  CUtensorMap tk, tv, tdq, tdk, tdv, tq64, tdo64;
  if (!encode_tmap_bf16(&tq64, q, 3, dq_, sq, box64, true, err) ||
      !encode_tmap_bf16(&tdo64, dout, 3, dq_, sq, box64, true, err) ||
      (!fused && !encode_tmap_bf16(&tdq, dq, 3, dq_, sq, box, true, err)) ||
      !encode_tmap_bf16(&tk, k, 3, dk_, sk, box, true, err) ||
      !encode_tmap_bf16(&tv, v, 3, dk_, sk, box, true, err) ||
      !encode_tmap_bf16(&tdk, dk, 3, dk_, sk, box, true, err) ||
      !encode_tmap_bf16(&tdv, dv, 3, dk_, sk, box, true, err))
    return cudaErrorInvalidValue;

  BArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.dout = static_cast<const uint16_t*>(dout);
  a.lse = lse;
  a.delta = delta;
  a.B = B;
  a.H = H;
  a.Hkv = Hkv;
  a.Nq = Nq;
  a.Nk = Nk;
  a.c_log2 = scale * kLog2e;
  a.scale = scale;
  a.causal = causal;
  a.diag_wait_ns = 0;

  const long long rows = (long long)B * H * Nq;
  const long long threads = rows * (D / 8);
  const unsigned grid_kv = unsigned(B) * Hkv * unsigned((Nk + 127) / 128);
  cudaError_t e;
  if (fused) {
    static thread_local int conf_fused = -1;
    e = set_smem_once(bwd_fused_kernel, FusedCfg::kSmemBytes, &conf_fused);
    if (e != cudaSuccess) return e;
    bwd_delta_kernel<D><<<unsigned((threads + 255) / 256), 256, 0, stream>>>(
        static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout), delta, rows, dq_acc);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    a.launch_id = next_launch_id();
    a.diag_wait_ns = diag_wait_ns;
    bwd_fused_kernel<<<grid_kv, 512, FusedCfg::kSmemBytes, stream>>>(tq64, tdo64, tk, tv, tdk, tdv,
                                                                     a, dq_acc);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long n8 = rows * D / 8;
    bwd_dq_convert_kernel<<<unsigned((n8 + 255) / 256), 256, 0, stream>>>(
        dq_acc, static_cast<uint16_t*>(dq), n8, scale);
    return cudaGetLastError();
  }
  static thread_local int conf_dq = -1, conf_dkdv = -1;
  e = set_smem_once(bwd_dq_kernel<D>, DqCfg<D>::kSmemBytes, &conf_dq);
  if (e != cudaSuccess) return e;
  e = set_smem_once(bwd_dkdv_kernel<D>, DkvCfg<D>::kSmemBytes, &conf_dkdv);
  if (e != cudaSuccess) return e;
  bwd_delta_kernel<D><<<unsigned((threads + 255) / 256), 256, 0, stream>>>(
      static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout), delta, rows, nullptr);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const unsigned grid_dq = unsigned(B) * H * unsigned((Nq + 127) / 128);
  a.launch_id = next_launch_id();
  bwd_dq_kernel<D><<<grid_dq, 384, DqCfg<D>::kSmemBytes, stream>>>(tk, tv, tdq, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  a.launch_id = next_launch_id();
  a.diag_wait_ns = diag_wait_ns;
  bwd_dkdv_kernel<D><<<grid_kv, 384, DkvCfg<D>::kSmemBytes, stream>>>(tq64, tdo64, tk, tv, tdk,
                                                                       tdv, a);
  return cudaGetLastError();
}

}  // namespace

// Workspace: D (B*H*Nq fp32, rounded up to 256 bytes), then, for the fused
// d = 128 path, the fp32 dQ accumulator [B*H*Nq, 128].
size_t backward_workspace_bytes(int B, int H, int Nq, int d, bool deterministic) {
  const size_t n = size_t(B) * H * Nq * sizeof(float);
  const size_t dsz = (n + 255) / 256 * 256;
  if (deterministic || d != 128) return dsz;
  return dsz + n * 128;
}

cudaError_t backward_launch(const void* q, const void* k, const void* v, const void* o,
                            const void* dout, const float* lse, void* dq, void* dk, void* dv,
                            int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                            bool deterministic, unsigned diag_wait_ns, void* workspace,
                            cudaStream_t stream, const char** err) {
  float* delta = static_cast<float*>(workspace);
  if (d == 128) {
    float* acc = nullptr;
    if (!deterministic) {
      const size_t n = size_t(B) * H * Nq * sizeof(float);
      acc = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + (n + 255) / 256 * 256);
    }
    return launch_bwd<128>(q, k, v, o, dout, lse, dq, dk, dv, B, H, Hkv, Nq, Nk, scale, causal,
                           delta, acc, diag_wait_ns, stream, err);
  }
  return launch_bwd<64>(q, k, v, o, dout, lse, dq, dk, dv, B, H, Hkv, Nq, Nk, scale, causal, delta,
                        nullptr, diag_wait_ns, stream, err);
}

int backward_take_device_error() {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_backward_error, sizeof(int)) != cudaSuccess) return -1;
  if (v != 0) cudaMemcpyToSymbol(g_backward_error, &zero, sizeof(int));
  return v;
}

}  // namespace attn
