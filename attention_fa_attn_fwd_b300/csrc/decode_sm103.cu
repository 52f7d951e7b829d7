// Paged-KV decode attention for sm_103a (B300): one query token per sequence
// attends every cached key of its sequence, read through a block table.
//
// PagedAttention keeps K/V in fixed blocks of 16 tokens addressed through a
// per-sequence block table, and sequences that share a prefix share its
// physical blocks (tutorial "第 3 章 进阶原理:性能模型与数值稳定性", sections
// 3.0.6-3.0.7).  Decode is bandwidth-bound ("以 Transformer 为例进行分析",
// section 三 and 3.1.1), so the design goal is HBM bytes in flight, not FLOPs.
//
// Kernel 1 (split): CTA = (split r, KV head g, sequence s); the split covers
// `bps` consecutive logical blocks.  Each of the 4 warps owns blocks
// r*bps + w, +4, ... and streams them through its own 3-stage ring: lane 0
// looks the physical id up in the block table and TMA-loads the block's K and
// V rows (2 KB boxes, 128-byte swizzle) on an mbarrier.  The G = H/Hkv query
// heads of the group share every K/V byte: S = Q K^T and O += P V are
// 16 x 16 x d products done with mma.sync (rows >= G are zero padding), the
// online softmax is the same base-2 recurrence as the prefill kernel.  The 4
// warps merge in shared memory and write one unnormalised partial
// (o, m, l) per head to the workspace.
//
// Kernel 2 (merge, a programmatic dependent launch so its start overlaps the
// split kernel's tail): per (sequence, head), combine the splits by their LSE:
// M = max m_r, L = sum 2^(m_r - M) l_r, o = sum 2^(m_r - M) o_r / L,
// lse = (M + log2 L) ln 2.  Deterministic order, no atomics.

#include <cmath>
#include <cstdio>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {

__device__ int g_decode_error[2];  // see ErrSink

namespace {

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;
constexpr int kWarps = 4;
constexpr int kRing = 3;          // stages per warp
constexpr int kBlockTokens = 16;  // PagedAttention block size

template <int D>
struct DCfg {
  static constexpr int kBoxes = D / 64;              // 64-column boxes per block per K or V
  static constexpr int kBoxBytes = kBlockTokens * 128;  // 16 rows x 128 B
  static constexpr int kKBytes = kBoxes * kBoxBytes;
  static constexpr int kStageBytes = 2 * kKBytes;     // K then V
  static constexpr int kWarpBytes = kRing * kStageBytes;
  static constexpr int kOffBar = kWarps * kWarpBytes;
  static constexpr int kSmemBytes = kOffBar + kWarps * kRing * 8 + 16 + 1024;
  static constexpr int kDT = D / 8;  // 8-column output tiles
};

struct DArgs {
  const uint16_t* q;       // [S, H, D]
  const int32_t* block_table;
  const int32_t* seq_lens;
  float* ws_o;             // [S, H, max_splits, D]
  float* ws_ml;            // [S, H, max_splits, 2]  (m, l) in log2 units
  int H, Hkv, G, num_blocks, max_blocks, bps, max_splits;
  float c_log2;
  unsigned launch_id;  // set per kernel launch (see ErrSink)
  // One split per sequence (max_splits == 1): the split kernel writes the
  // final output itself and no merge kernel runs.
  uint16_t* out_o;     // [S, H, D] bf16, or nullptr (partials + merge)
  float* out_lse;      // [S, H] or nullptr
};

__device__ __forceinline__ void mma_16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// Byte offset of (row, column) inside a [16 x 64] bf16 box written by TMA
// with 128-byte swizzle (box base 1024-byte aligned).
__device__ __forceinline__ uint32_t sw128(int row, int col) {
  return uint32_t(row * 128 + ((((col >> 3) ^ (row & 7))) << 4) + ((col & 7) << 1));
}

// kR16: G = H / Hkv > 8, so rows 8..15 of the 16-row mma tile are query heads
// too (each lane then keeps the softmax state of rows gq and gq + 8); with
// G <= 8 those rows are zero padding and their softmax is skipped.
template <int D, bool kR16>
__global__ void __launch_bounds__(128)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const DArgs a) {
  using C = DCfg<D>;
  constexpr int NR = kR16 ? 2 : 1;  // softmax rows per lane: gq (and gq + 8)
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffBar + kWarps * kRing * 8);
  const ErrSink err{g_decode_error, a.launch_id};

  // The merge kernel may be scheduled once every CTA of this grid has
  // started; it waits for this grid's completion before reading partials.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int seq_len = a.seq_lens[s];
  const int nblk = min((max(seq_len, 0) + kBlockTokens - 1) / kBlockTokens, a.max_blocks);
  const int b_lo = r * a.bps;
  if (b_lo >= nblk) {  // split past the end of this sequence: no partial
    if (a.out_o != nullptr && r == 0) {  // single-split output of an empty sequence
      for (int idx = threadIdx.x; idx < a.G * D; idx += blockDim.x)
        a.out_o[(size_t(s) * a.H + size_t(g) * a.G + idx / D) * D + idx % D] = 0;
      if (a.out_lse != nullptr && threadIdx.x < a.G)
        a.out_lse[size_t(s) * a.H + size_t(g) * a.G + threadIdx.x] = -INFINITY;
    }
    return;
  }
  if (err.this_launch_timed_out()) return;  // partial left unwritten; error already recorded
  const int b_hi = min(nblk, b_lo + a.bps);

  auto bar = [&](int w, int st) -> uint32_t { return sbase + C::kOffBar + 8u * (w * kRing + st); };
  const int gq = lane >> 2, tq = lane & 3;  // mma fragment coordinates
  const int n_mine = (b_hi - b_lo - warp + kWarps - 1) / kWarps;  // blocks of this warp
  const uint32_t wbase = sbase + warp * C::kWarpBytes;
  const int32_t* bt = a.block_table + size_t(s) * a.max_blocks;

  // Physical ids of this warp's blocks, read once (lane i holds block i).
  int my_phys = 0;
  if (lane < n_mine) {
    my_phys = bt[b_lo + warp + kWarps * lane];
    if (my_phys < 0 || my_phys >= a.num_blocks) {
      err.record(kErrDecodeBadBlock);
      my_phys = a.num_blocks;  // outside the tensor map: TMA fills zeros
    }
  }
  if (r == 0 && g == 0 && threadIdx.x == 0 && seq_len > a.max_blocks * kBlockTokens)
    err.record(kErrDecodeBadBlock);
  auto issue = [&](int i, int phys) {  // lane 0: TMA-load the i-th block of this warp
    const int st = i % kRing;
    const uint32_t dst = wbase + st * C::kStageBytes;
    const int row0 = (phys * a.Hkv + g) * kBlockTokens;
    mbar_arrive_expect_tx(bar(warp, st), C::kStageBytes);
#pragma unroll
    for (int bx = 0; bx < C::kBoxes; ++bx) {
      tma_load_3d(dst + bx * C::kBoxBytes, &tm_k, bar(warp, st), bx * 64, row0, 0);
      tma_load_3d(dst + C::kKBytes + bx * C::kBoxBytes, &tm_v, bar(warp, st), bx * 64, row0, 0);
    }
  };
  // Each warp's lane 0 initialises the warp's own ring barriers and issues
  // its first copies straight away, before the CTA-wide barrier below (which
  // only publishes the abort flag): the copies' latency overlaps the set-up
  // and the Q loads.
  if (lane == 0) {
    for (int st = 0; st < kRing; ++st) mbar_init(bar(warp, st), 1);
    fence_mbar_init();
  }
  __syncwarp();
#pragma unroll
  for (int i = 0; i < kRing; ++i) {
    const int ph = __shfl_sync(0xffffffffu, my_phys, i);
    if (lane == 0 && i < n_mine) issue(i, ph);
  }

  // Q fragments (A operand, rows = heads of this group, zero beyond G).
  uint32_t qa[D / 16][4];
  {
    const uint16_t* qrow = a.q + (size_t(s) * a.H + size_t(g) * a.G + gq) * D;
#pragma unroll
    for (int kc = 0; kc < D / 16; ++kc) {
      uint32_t lo = 0, hi = 0, lo8 = 0, hi8 = 0;
      if (gq < a.G) {
        lo = *reinterpret_cast<const uint32_t*>(qrow + kc * 16 + 2 * tq);
        hi = *reinterpret_cast<const uint32_t*>(qrow + kc * 16 + 8 + 2 * tq);
      }
      if (kR16 && gq + 8 < a.G) {
        lo8 = *reinterpret_cast<const uint32_t*>(qrow + 8 * D + kc * 16 + 2 * tq);
        hi8 = *reinterpret_cast<const uint32_t*>(qrow + 8 * D + kc * 16 + 8 + 2 * tq);
      }
      qa[kc][0] = lo;
      qa[kc][1] = lo8;  // rows 8..15 (zero padding when G <= 8)
      qa[kc][2] = hi;
      qa[kc][3] = hi8;
    }
  }
  if (threadIdx.x == 0) *abort_flag = 0;
  __syncthreads();

  float o[C::kDT][4];
#pragma unroll
  for (int i = 0; i < C::kDT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  // rows gq (and gq + 8); l is this lane's partial sum
  float m[NR], l[NR];
#pragma unroll
  for (int rr = 0; rr < NR; ++rr) m[rr] = -INFINITY, l[rr] = 0.f;

  bool ok = true;
  int consumed = 0;
  for (int i = 0; i < n_mine; ++i) {
    const int st = i % kRing;
    ok = mbar_wait(bar(warp, st), (i / kRing) & 1, abort_flag, err, kErrTimeoutSoftmax);
    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
    const int lb = b_lo + warp + kWarps * i;
    const int valid = min(kBlockTokens, seq_len - lb * kBlockTokens);
    const uint32_t kb = wbase + st * C::kStageBytes;
    const uint32_t vb = kb + C::kKBytes;
    if (valid < kBlockTokens) {
      // Slots past the sequence end may hold anything (even NaN): zero them
      // so 0-probability keys contribute exactly 0 to P V.
      uint8_t* kp = smem + (kb - sbase);
      uint8_t* vp = smem + (vb - sbase);
      for (int idx = lane; idx < C::kBoxes * kBlockTokens * 8; idx += 32) {
        const int bx = idx / (kBlockTokens * 8), rr = (idx / 8) % kBlockTokens, ch = idx % 8;
        if (rr >= valid) {
          *reinterpret_cast<uint4*>(kp + bx * C::kBoxBytes + rr * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(vp + bx * C::kBoxBytes + rr * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      __syncwarp();
    }
    // ---- S = Q K^T (16 heads-rows x 16 tokens)
    float sc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
    {
      const int tok = (lane & 7) + ((lane >> 4) << 3);
      const int csub = ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int kc = 0; kc < D / 16; ++kc) {
        const int col = kc * 16 + csub;
        uint32_t bfr[4];
        ldsm_x4(kb + (col >> 6) * C::kBoxBytes + sw128(tok, col & 63), bfr);
        mma_16816(sc[0], qa[kc], bfr[0], bfr[1]);
        mma_16816(sc[1], qa[kc], bfr[2], bfr[3]);
      }
    }
    // ---- online softmax on row gq (c0, c1 of both token tiles) and, with
    // kR16, row gq + 8 (c2, c3)
    uint32_t pa[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int rr = 0; rr < NR; ++rr) {
      float x[4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int tok = nt * 8 + 2 * tq + e;
          x[nt * 2 + e] = (tok < valid) ? sc[nt][2 * rr + e] * a.c_log2 : -INFINITY;
        }
      float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      if (mx > m[rr] + 8.0f) {  // move the reference (uniform across the row's 4 lanes)
        const float alpha = ex2_approx(m[rr] - mx);
        m[rr] = mx;
        l[rr] *= alpha;
#pragma unroll
        for (int dt = 0; dt < C::kDT; ++dt) {
          o[dt][2 * rr] *= alpha;
          o[dt][2 * rr + 1] *= alpha;
        }
      }
      const float nm = (m[rr] == -INFINITY) ? 0.f : -m[rr];
      float p[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) p[e] = ex2_approx(x[e] + nm);
      l[rr] += (p[0] + p[1]) + (p[2] + p[3]);
      pa[rr] = pack_bf16x2(p[0], p[1]);      // row gq (+8), tokens 2tq, 2tq+1
      pa[2 + rr] = pack_bf16x2(p[2], p[3]);  // row gq (+8), tokens 8+2tq, 9+2tq
    }
    // ---- O += P V
    {
      const int tok = (lane & 7) + (((lane >> 3) & 1) << 3);
      const int dsub = (lane >> 4) * 8;
#pragma unroll
      for (int dt = 0; dt < C::kDT; dt += 2) {
        const int col = dt * 8 + dsub;
        uint32_t bfr[4];
        ldsm_x4_t(vb + (col >> 6) * C::kBoxBytes + sw128(tok, col & 63), bfr);
        mma_16816(o[dt], pa, bfr[0], bfr[1]);
        mma_16816(o[dt + 1], pa, bfr[2], bfr[3]);
      }
    }
    // ---- refill this stage
    __syncwarp();
    const int nxt = i + kRing;
    const int ph = __shfl_sync(0xffffffffu, my_phys, nxt & 31);
    if (lane == 0 && nxt < n_mine) {
      fence_proxy_async_smem();
      issue(nxt, ph);
    }
    consumed = i + 1;
  }
  if (!ok && lane == 0) {
    // Abort path: let this warp's copies in flight land before smem is reused.
    const uint64_t deadline = globaltimer_ns() + kWaitTimeoutNs;
    for (int i = consumed; i < min(n_mine, consumed + kRing); ++i)
      mbar_wait_drain(bar(warp, i % kRing), (i / kRing) & 1, deadline);
  }

  // ---- merge the 4 warps' states through shared memory (stage memory reuse)
  __syncthreads();
  float* red_o = reinterpret_cast<float*>(smem);                   // [4 warps][16 rows][D]
  float* red_ml = reinterpret_cast<float*>(smem + kWarps * 16 * D * 4);  // [4][16][2]
#pragma unroll
  for (int rr = 0; rr < NR; ++rr) {
    l[rr] += __shfl_xor_sync(0xffffffffu, l[rr], 1);
    l[rr] += __shfl_xor_sync(0xffffffffu, l[rr], 2);
    if (!ok) m[rr] = -INFINITY, l[rr] = 0.f;
    const int hr = gq + 8 * rr;
    if (hr < a.G) {
#pragma unroll
      for (int dt = 0; dt < C::kDT; ++dt) {
        red_o[(warp * 16 + hr) * D + dt * 8 + 2 * tq] = o[dt][2 * rr];
        red_o[(warp * 16 + hr) * D + dt * 8 + 2 * tq + 1] = o[dt][2 * rr + 1];
      }
      if (tq == 0) {
        red_ml[(warp * 16 + hr) * 2 + 0] = m[rr];
        red_ml[(warp * 16 + hr) * 2 + 1] = l[rr];
      }
    }
  }
  __syncthreads();
  if (*abort_flag) return;
  for (int idx = threadIdx.x; idx < a.G * D; idx += blockDim.x) {
    const int hr = idx / D, dcol = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_ml[(w * 16 + hr) * 2]);
    float acc = 0.f, L = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = red_ml[(w * 16 + hr) * 2];
      const float wgt = (mw == -INFINITY) ? 0.f : ex2_approx(mw - M);
      acc += wgt * red_o[(w * 16 + hr) * D + dcol];
      L += wgt * red_ml[(w * 16 + hr) * 2 + 1];
    }
    const size_t head = size_t(s) * a.H + size_t(g) * a.G + hr;
    if (a.out_o != nullptr) {  // the only split: final normalised output
      const float inv = (L > 0.f) ? 1.f / L : 0.f;
      a.out_o[head * D + dcol] = uint16_t(pack_bf16x2(acc * inv, 0.f) & 0xffffu);
      if (dcol == 0 && a.out_lse != nullptr)
        a.out_lse[head] = (L > 0.f) ? (M + log2f(L)) * kLn2 : -INFINITY;
      continue;
    }
    a.ws_o[(head * a.max_splits + r) * D + dcol] = acc;
    if (dcol == 0) {
      a.ws_ml[(head * a.max_splits + r) * 2 + 0] = M;
      a.ws_ml[(head * a.max_splits + r) * 2 + 1] = L;
    }
  }
}

// One warp per (sequence, head).  Launched as a programmatic dependent of the
// split kernel: its CTAs may start while the split kernel's last wave runs and
// wait (griddepcontrol.wait) until every partial is written and visible.
// Lane r loads split r's (m, l), so the weights take one round trip; the
// partial outputs are then summed with independent loads.
template <int D>
__global__ void __launch_bounds__(256)
    decode_merge_kernel(const DArgs a, uint16_t* __restrict__ o, float* __restrict__ lse,
                        int num_seqs) {
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (gw >= num_seqs * a.H) return;
  const int s = gw / a.H;
  const int seq_len = a.seq_lens[s];
  const int nblk = min((max(seq_len, 0) + kBlockTokens - 1) / kBlockTokens, a.max_blocks);
  const int nsp = (nblk + a.bps - 1) / a.bps;
  const size_t head = size_t(gw);
  const float* ml = a.ws_ml + head * a.max_splits * 2;
  float M = -INFINITY;
  for (int r = lane; r < nsp; r += 32) M = fmaxf(M, ml[2 * r]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  constexpr int PER = D / 32;
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  float L = 0.f;
  for (int r0 = 0; r0 < nsp; r0 += 32) {
    // weights of splits r0 .. r0+31, one per lane
    float w_mine = 0.f;
    if (r0 + lane < nsp) {
      const float mr = ml[2 * (r0 + lane)];
      w_mine = (mr == -INFINITY) ? 0.f : ex2_approx(mr - M);
      L += w_mine * ml[2 * (r0 + lane) + 1];
    }
    const int cnt = min(32, nsp - r0);
    const float* src = a.ws_o + (head * a.max_splits + r0) * D + lane * PER;
#pragma unroll 4
    for (int r = 0; r < cnt; ++r) {
      const float w = __shfl_sync(0xffffffffu, w_mine, r);
      if constexpr (PER == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src + size_t(r) * D);
        acc[0] += w * v.x;
        acc[1] += w * v.y;
        acc[2] += w * v.z;
        acc[3] += w * v.w;
      } else {
        const float2 v = *reinterpret_cast<const float2*>(src + size_t(r) * D);
        acc[0] += w * v.x;
        acc[1] += w * v.y;
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  const float inv = (L > 0.f) ? 1.f / L : 0.f;
  uint16_t* dst = o + head * D + lane * PER;
#pragma unroll
  for (int e = 0; e < PER; e += 2) {
    const uint32_t pk = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
    *reinterpret_cast<uint32_t*>(dst + e) = pk;
  }
  if (lse != nullptr && lane == 0) lse[head] = (L > 0.f) ? (M + log2f(L)) * kLn2 : -INFINITY;
}

template <int D>
cudaError_t launch(const void* q, const void* k_cache, const void* v_cache, const int32_t* bt,
                   const int32_t* seq_lens, int S, int H, int Hkv, int num_blocks, int max_blocks,
                   float scale, void* o, float* lse, void* workspace, const DecodePlan& plan,
                   cudaStream_t stream, const char** err) {
  using C = DCfg<D>;
  CUtensorMap tk, tv;
  const uint64_t dims[3] = {uint64_t(D), uint64_t(num_blocks) * Hkv * kBlockTokens, 1};
  const uint64_t strides[2] = {uint64_t(D) * 2, uint64_t(D) * 2 * dims[1]};
  const uint32_t box[3] = {64, kBlockTokens, 1};
  if (!encode_tmap_bf16(&tk, k_cache, 3, dims, strides, box, true, err)) return cudaErrorInvalidValue;
  if (!encode_tmap_bf16(&tv, v_cache, 3, dims, strides, box, true, err)) return cudaErrorInvalidValue;
  const bool r16 = H / Hkv > 8;
  static thread_local int configured_device[2] = {-1, -1};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device[r16] != dev) {
    e = cudaFuncSetAttribute(r16 ? decode_split_kernel<D, true> : decode_split_kernel<D, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device[r16] = dev;
  }
  DArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.block_table = bt;
  a.seq_lens = seq_lens;
  a.ws_o = static_cast<float*>(workspace);
  a.ws_ml = a.ws_o + size_t(S) * H * plan.max_splits * D;
  a.H = H;
  a.Hkv = Hkv;
  a.G = H / Hkv;
  a.num_blocks = num_blocks;
  a.max_blocks = max_blocks;
  a.bps = plan.blocks_per_split;
  a.max_splits = plan.max_splits;
  a.c_log2 = scale * kLog2e;
  const bool direct = plan.max_splits == 1;
  a.out_o = direct ? static_cast<uint16_t*>(o) : nullptr;
  a.out_lse = direct ? lse : nullptr;
  dim3 grid(plan.max_splits, Hkv, S);
  a.launch_id = next_launch_id();
  if (r16)
    decode_split_kernel<D, true><<<grid, 128, C::kSmemBytes, stream>>>(tk, tv, a);
  else
    decode_split_kernel<D, false><<<grid, 128, C::kSmemBytes, stream>>>(tk, tv, a);
  e = cudaGetLastError();
  if (e != cudaSuccess || direct) return e;
  const int warps = S * H;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((warps + 7) / 8);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_merge_kernel<D>, a, static_cast<uint16_t*>(o), lse, S);
}

}  // namespace

DecodePlan decode_plan(int num_seqs, int H, int Hkv, int d, int max_blocks_per_seq) {
  // Blocks per split: 128 (2048 tokens), halved while that would give fewer
  // than two CTAs per SM for sequences of half the table's length; never
  // below 8.  Long splits win wherever the grid still covers the machine:
  // on 64 sequences x 8 KV heads, 128-block splits against 8-block ones took
  // 34.8 vs 43.0 us at 512 tokens and 53.3 vs 73.7 us at 1024 (fewer CTAs
  // to set up, fewer partials to write and merge), and equal times from
  // 2048 tokens on.  Small batches keep enough CTAs through the halving.
  // At most 128: each warp keeps the physical ids of its blocks one per lane
  // (4 warps x 32 lanes).
  int bps = kWarps * 32;
  const long long target = 2LL * 148;
  while (bps > 8) {
    const long long splits = (max_blocks_per_seq / 2 + bps - 1) / bps;
    if (splits * num_seqs * Hkv >= target) break;
    bps /= 2;
  }
  DecodePlan p;
  p.blocks_per_split = bps;
  p.max_splits = (max_blocks_per_seq + bps - 1) / bps;
  p.workspace_bytes = size_t(num_seqs) * H * p.max_splits * (size_t(d) + 2) * sizeof(float);
  return p;
}

cudaError_t decode_launch(const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_table, const int32_t* seq_lens, int num_seqs, int H,
                          int Hkv, int d, int num_blocks, int max_blocks_per_seq, float scale,
                          void* o, float* lse, void* workspace, const DecodePlan& plan,
                          cudaStream_t stream, const char** err) {
  if (d == 128)
    return launch<128>(q, k_cache, v_cache, block_table, seq_lens, num_seqs, H, Hkv, num_blocks,
                       max_blocks_per_seq, scale, o, lse, workspace, plan, stream, err);
  return launch<64>(q, k_cache, v_cache, block_table, seq_lens, num_seqs, H, Hkv, num_blocks,
                    max_blocks_per_seq, scale, o, lse, workspace, plan, stream, err);
}

int decode_take_device_error() {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_decode_error, sizeof(int)) != cudaSuccess) return -1;
  if (v != 0) cudaMemcpyToSymbol(g_decode_error, &zero, sizeof(int));
  return v;
}

}  // namespace attn
