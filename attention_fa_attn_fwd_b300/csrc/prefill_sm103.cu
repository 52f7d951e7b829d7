// FlashAttention-2-style attention forward for sm_103a (B300).
//
// Computes O = softmax(scale * Q K^T [causal]) V and the per-row natural
// log-sum-exp in one pass over K/V, so the N x N matrices S and P never
// reach HBM (FAQ page "Wie unterscheidet sich die Implementierung von
// FlashAttention-2 ...", comparison table: tiling, online softmax; interview
// notes "他人面经整理", flashattention answer part 2: kernel fusion, tiling,
// online softmax with running max m and running sum l).
//
// One CTA owns two 128-row Q tiles (Q0, Q1) of one (batch, head) and streams
// every K/V tile either may attend (causal: up to the diagonal); each K/V tile
// is read from shared memory by both Q tiles.  Warp roles (12 warps, three
// warpgroups; warpgroup 0 gives registers to the other two via setmaxnreg):
//   warp 0      TMA producer: Q0, Q1 once, then K_j / V_j into rings of stages
//               (the double-buffered prefetch of the FSA page, section 3.2).
//   warp 1      tcgen05 MMA issuer: S_i = Q_i K_j^T into TMEM, O_i += P_i V_j
//               with P_i read from TMEM.  Issue order per KV tile j:
//               PV(0,j) QK(0,j+1) PV(1,j) QK(1,j+1), so while one softmax
//               warpgroup works on tile i the tensor pipe runs the other's.
//   warps 2..3  idle.
//   warps 4..7  softmax warpgroup of Q0, warps 8..11 of Q1: thread r owns TMEM
//               lane / Q row r.  Online softmax in base 2 with scale*log2(e)
//               folded into one FFMA; the running max only moves when it
//               grows by more than 8 (log2 units) and only then is O_i
//               rescaled in TMEM; P_i is written back to TMEM as bf16 over
//               the S_i columns it came from.  At the end: O_i / l (deferred
//               normalisation), bf16 O through smem and a TMA store,
//               lse = (m + log2 l) ln 2.
//
// Paged variant (kPaged): K and V are read through a PagedAttention block
// table instead of from contiguous [B, Hkv, Nk, d] tensors (tutorial
// "第 3 章 进阶原理:性能模型与数值稳定性", section 3.0.6: the fused kernel and the
// paged cache work together).  Sequence b has kv_lens[b] cached tokens, the
// last Nq of which are the queries' own; a 128-key tile is 8 blocks of 16
// tokens, each fetched by its own 16-row TMA box into the same swizzled
// layout one 128-row box would produce.  Blocks past the sequence end are
// fetched from an out-of-range row (TMA fills zeros); cache slots past the
// end inside the last block may hold anything, so the MMA warp zeroes those V
// rows in shared memory before the first P V that reads them (K needs no
// fix-up: the mask replaces those scores).
//
// TMEM columns: S0 [0,128) S1 [128,256) O0 [256,256+d) O1 [256+d,256+2d);
// P_i occupies the first 64 columns of S_i.  tcgen05.mma operations of one
// issuing thread execute in order, so QK(i,j+1) overwriting P_i happens after
// PV(i,j) read it, and "S_i(j+1) complete" implies "PV(i,j) complete".
// Every wait is bounded (ptx.cuh).

#include <cmath>
#include <cstdio>

#include "attn_internal.h"
#include "exp2_poly.h"
#include "ptx.cuh"

namespace attn {

__device__ int g_prefill_error[2];  // see ErrSink

namespace {

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: p <= 2^8 between rescales

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

template <int D>
struct Cfg {
  static constexpr int kSlabs = D / 64;         // 64-element (128-byte) column slabs
  static constexpr int kSlabBytes = 128 * 128;  // 128 rows x 128 B
  static constexpr int kTileBytes = kSlabs * kSlabBytes;  // one 128-row Q, K or V tile
  static constexpr int kKStages = (D == 128) ? 3 : 4;
  static constexpr int kVStages = (D == 128) ? 2 : 4;
  static constexpr int kOffQ = 0;  // Q0, Q1 (reused as O0, O1 staging)
  static constexpr int kOffK = 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kVStages * kTileBytes;
  // barrier indices
  static constexpr int kBarQF = 0;                    // 2: Q_i loaded
  static constexpr int kBarKF = kBarQF + 2;           // K stage full
  static constexpr int kBarKE = kBarKF + kKStages;    // K stage free
  static constexpr int kBarVF = kBarKE + kKStages;    // V stage full
  static constexpr int kBarVE = kBarVF + kVStages;    // V stage free
  static constexpr int kBarSF = kBarVE + kVStages;    // 2: S_i ready in TMEM
  static constexpr int kBarPF = kBarSF + 2;           // 2: P_i keys 0..63 written (O_i rescaled)
  static constexpr int kBarPF2 = kBarPF + 2;          // 2: P_i keys 64..127 written
  static constexpr int kBarOF = kBarPF2 + 2;          // 2: last PV of tile i done
  static constexpr int kBarDrain = kBarOF + 2;
  static constexpr int kBarDiag = kBarDrain + 1;      // never signalled (diagnostic wait)
  static constexpr int kNumBars = kBarDiag + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack for 1024-B alignment
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;    // S_i at i * 128
  static constexpr uint32_t kColO = 256;  // O_i at 256 + i * D
  static constexpr int kThreads = 384;
  // Registers per thread: 168 at launch (64K / 384); warpgroup 0 drops to
  // 80, the two softmax warpgroups rise to 208 (128*80 + 256*208 <= 384*168).
  static constexpr int kRegsLow = 80;
  static constexpr int kRegsHigh = 208;
};

struct Args {
  float* lse;
  int B, H, Hkv, Nq, Nk;
  int n_pairs;   // ceil(Nq / 256)
  float c_log2;  // scale * log2(e)
  int causal;
  // paged variant only
  const int32_t* block_table;  // [B, max_blocks]
  const int32_t* kv_lens;      // [B]
  int max_blocks, num_blocks;
  int oob_row;                 // a pool row past the end: TMA fills zeros
  int group_major;             // CTA order (see the kernel)
  unsigned launch_id;          // set per kernel launch (see ErrSink)
  unsigned diag_wait_ns;       // != 0: CTA 0 lets one bounded wait expire (failure test)
};

constexpr int kPageTokens = 16;  // PagedAttention block size

// 2^x for a pair of values on the FMA and integer pipes, without the MUFU
// unit: x = n + f with n = round(x) (adding 1.5 * 2^23 rounds to an integer in
// the low mantissa bits), f in [-1/2, 1/2]; 2^f by the least-squares cubic of
// exp2_poly.h (relative error < 8e-5); 2^n by adding n to the exponent field.
// Exactly 0 below -126 (so -inf, the mask value, gives 0).
__device__ __forceinline__ float2 exp2_fma2(float2 x) {
  constexpr float kMagic = 12582912.f;  // 1.5 * 2^23
  x.x = fmaxf(x.x, -127.f);
  x.y = fmaxf(x.y, -127.f);
  const float2 j = __fadd2_rn(x, make_float2(kMagic, kMagic));
  const float2 n = __fadd2_rn(j, make_float2(-kMagic, -kMagic));
  const float2 f = __ffma2_rn(n, make_float2(-1.f, -1.f), x);
  float2 p = __ffma2_rn(make_float2(kExp2Poly3, kExp2Poly3), f,
                        make_float2(kExp2Poly2, kExp2Poly2));
  p = __ffma2_rn(p, f, make_float2(kExp2Poly1, kExp2Poly1));
  p = __ffma2_rn(p, f, make_float2(kExp2Poly0, kExp2Poly0));
  float rx = __int_as_float(__float_as_int(p.x) + (__float_as_int(j.x) << 23));
  float ry = __int_as_float(__float_as_int(p.y) + (__float_as_int(j.y) << 23));
  return make_float2(x.x < -126.f ? 0.f : rx, x.y < -126.f ? 0.f : ry);
}

// kPolyExp: the exponentials of columns 64..127 of every score tile use
// exp2_fma2 instead of the MUFU ex2, moving half of that work to the FMA pipe
// (an opt-in variant; the MUFU path is the default).
template <int D, bool kPaged, bool kPolyExp>
__global__ void __launch_bounds__(384, 1)
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
  // Copies the producer has issued, for the abort drain at the end (kept in
  // shared memory, not registers): [0] V tiles (each with K_{j+1} on its
  // barrier); [1] bit 0: K_0, bits 1-2: the Q tiles.
  volatile int* issued_state = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
  const ErrSink err{g_prefill_error, a.launch_id};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // The first copies read the Q and K descriptors: fetch them while the
  // rest of the set-up runs.
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
  }

  // Heavy (late, causal) tile pairs first; heads of one KV group adjacent.
  // group_major: all tile pairs of one (batch, KV head) group before the
  // next group, so the CTAs resident at once share one group's K/V in L2
  // (used when all groups' K/V would not fit in L2 together).
  const int BH = a.B * a.H;
  int bh, pair;
  if (a.group_major) {
    const int G = a.H / a.Hkv;
    const int per_group = a.n_pairs * G;
    const int grp = blockIdx.x / per_group, r = blockIdx.x % per_group;
    pair = r / G;
    bh = grp * G + r % G;
    if constexpr (kPaged) {
      // Sequences have their own lengths: take the groups of the longest
      // sequences first (ties by index), so the longest ones do not run
      // last.  Group grp is KV head grp % Hkv of the (grp / Hkv)-th longest
      // sequence; each warp ranks the lengths itself (up to 64 sequences,
      // else index order).
      if (a.B <= 64) {
        const int k = grp / a.Hkv;
        const int L0 = lane < a.B ? a.kv_lens[lane] : 0;
        const int L1 = lane + 32 < a.B ? a.kv_lens[lane + 32] : 0;
        int mine = -1;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int c = lane + 32 * t;
          const int Lc = t == 0 ? L0 : L1;
          int rank = 0;
          for (int o = 0; o < a.B; ++o) {
            const int Lo = __shfl_sync(0xffffffffu, o < 32 ? L0 : L1, o & 31);
            rank += (Lo > Lc || (Lo == Lc && o < c)) ? 1 : 0;
          }
          if (c < a.B && rank == k) mine = c;
        }
        const unsigned found = __ballot_sync(0xffffffffu, mine >= 0);
        const int seq = __shfl_sync(0xffffffffu, mine, __ffs(int(found)) - 1);
        bh = seq * a.H + (grp % a.Hkv) * G + r % G;
      }
    }
  } else {
    bh = blockIdx.x % BH;
    pair = blockIdx.x / BH;
  }
  const int q0 = (a.n_pairs - 1 - pair) * 256;
  const int b = bh / a.H;
  const int h = bh % a.H;
  const int g_kv = h / (a.H / a.Hkv);
  const int zkv = b * a.Hkv + g_kv;
  // Whether a wait of this launch already expired: loaded here, used after
  // the set-up barrier, so the load's latency overlaps the set-up.
  const unsigned timed_out_launch = reinterpret_cast<const volatile unsigned*>(err.word)[1];
  // Keys of this sequence; the paged variant reads its own length.
  int Nk = a.Nk;
  int nblk = 0;  // paged: cached blocks of this sequence
  if constexpr (kPaged) {
    Nk = a.kv_lens[b];
    if (Nk < 0 || Nk > a.max_blocks * kPageTokens) {
      if (threadIdx.x == 0 && q0 == (a.n_pairs - 1) * 256 && h == 0)
        err.record(kErrPagedBadLength);
      Nk = min(max(Nk, 0), a.max_blocks * kPageTokens);
    }
    nblk = (Nk + kPageTokens - 1) / kPageTokens;
  }
  // KV tiles each Q tile attends (0 for a tile past Nq or fully masked).
  int n_t[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r0 = q0 + i * 128;
    int kv_end = Nk;
    if (a.causal) kv_end = min(Nk, r0 + 128 + (Nk - a.Nq));
    n_t[i] = (r0 < a.Nq && kv_end > 0) ? (kv_end + 127) / 128 : 0;
  }
  int n_kv = max(n_t[0], n_t[1]);

  // Warp 0's lanes initialise one barrier each (one pass instead of a loop
  // of ~30 in one thread).
  static_assert(C::kNumBars <= 32, "one barrier per lane");
  if (warp == 0) {
    if (lane < C::kNumBars)
      mbar_init(bar(lane), (lane >= C::kBarPF && lane < C::kBarPF2 + 2) ? 128u : 1u);
    if (lane == 0) *abort_flag = 0;
    if (lane == 1) issued_state[0] = 0;
    if (lane == 2)  // the Q tiles and (contiguous K) K_0 leave early
      issued_state[1] = (n_kv > 0 && !kPaged ? 1 : 0) | (n_kv > 0 && n_t[0] > 0 ? 2 : 0) |
                        (n_kv > 0 && n_t[1] > 0 ? 4 : 0);
    fence_mbar_init();
    __syncwarp();
  }
  // The first copies (Q tiles, and K_0 when K is contiguous) leave before the
  // CTA-wide barrier below, from the thread that initialised the barriers, so
  // their latency overlaps the TMEM allocation and the rest of the set-up
  // (about 1.2 us per CTA, a large share of a short causal tile pair).
  const bool early = n_kv > 0;
  if (warp == 0) {
    __syncwarp();
    if (early) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if (n_t[i] == 0) continue;
        mbar_arrive_expect_tx_elect(bar(C::kBarQF + i), C::kTileBytes);
        for (int s = 0; s < C::kSlabs; ++s)
          tma_load_3d_elect(sbase + C::kOffQ + i * C::kTileBytes + s * C::kSlabBytes, &tm_q,
                            bar(C::kBarQF + i), s * 64, q0 + i * 128, bh);
      }
      if constexpr (!kPaged) {
        mbar_arrive_expect_tx_elect(bar(C::kBarKF), C::kTileBytes);
        for (int s = 0; s < C::kSlabs; ++s)
          tma_load_3d_elect(sbase + C::kOffK + s * C::kSlabBytes, &tm_k, bar(C::kBarKF), s * 64, 0,
                            zkv);
      }
    }
    if (lane == 0) {
      prefetch_tmap(&tm_v);
      prefetch_tmap(&tm_o);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // A wait of this launch already expired: skip the work (after the early
  // copies have landed, so none is in flight when the CTA exits).
  const bool dead = timed_out_launch == a.launch_id;
  if (dead) {
    if (warp == 0 && early) {
      const uint64_t deadline = globaltimer_ns() + kWaitTimeoutNs;
      for (int i = 0; i < 2; ++i)
        if (n_t[i] > 0) mbar_wait_drain(bar(C::kBarQF + i), 0, deadline);
      if (!kPaged) mbar_wait_drain(bar(C::kBarKF), 0, deadline);
    }
    n_t[0] = n_t[1] = 0;
    n_kv = 0;
  }

  if (warp < 4) {
    setmaxnreg_dec<C::kRegsLow>();
    if (warp == 0) {
      // -------------------------------------------------------- producer
      // The whole warp runs this loop; one elected lane issues each copy.
      // K_j goes to K stage j % KS once its previous occupant K_{j-KS} has
      // been consumed by its last QK (K-empty, committed by the MMA warp);
      // V_j likewise after the last PV of V_{j-VS}.
      if (n_kv > 0) {
        int v_issued = 0;
        bool ok = true;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (n_t[i] == 0 || early) continue;  // early: issued before the set-up barrier
          mbar_arrive_expect_tx_elect(bar(C::kBarQF + i), C::kTileBytes);
          for (int s = 0; s < C::kSlabs; ++s)
            tma_load_3d_elect(sbase + C::kOffQ + i * C::kTileBytes + s * C::kSlabBytes, &tm_q,
                              bar(C::kBarQF + i), s * 64, q0 + i * 128, bh);
        }
        // One K or V tile: a single 128-row box per slab, or (paged) lanes
        // 0..7 each fetch one 16-token block per slab at pool row `prow`.
        auto load_tile = [&](const CUtensorMap* tm, uint32_t dst, uint32_t fb, int j, int prow) {
          if constexpr (!kPaged) {
            for (int s = 0; s < C::kSlabs; ++s)
              tma_load_3d_elect(dst + s * C::kSlabBytes, tm, fb, s * 64, j * 128, zkv);
          } else {
            __syncwarp();
            if (lane < 8)
              for (int s = 0; s < C::kSlabs; ++s)
                tma_load_3d(dst + s * C::kSlabBytes + lane * (kPageTokens * 128), tm, fb, s * 64,
                            prow, 0);
          }
        };
        const int32_t* bt = nullptr;
        if constexpr (kPaged) bt = a.block_table + size_t(b) * a.max_blocks;
        // Paged: lanes 0..7 hold the physical ids of tile t's 8 blocks.  The
        // ids of tile j+2 are loaded while tile j's copies are issued, so the
        // table lookups stay off the path between a stage freeing and its
        // next copy.
        auto phys_of = [&](int t) -> int {
          int phys = -1;
          if constexpr (kPaged) {
            const int lb = t * 8 + lane;
            if (lane < 8 && t < n_kv && lb < nblk) phys = bt[lb];
          }
          return phys;
        };
        // Pool row of this lane's block (blocks past the sequence end, and
        // bad ids, read the zero-filled row past the pool).
        auto prow_from = [&](int t, int phys) -> int {
          int prow = 0;
          if constexpr (kPaged) {
            prow = a.oob_row;
            if (lane < 8 && t * 8 + lane < nblk) {
              if (phys >= 0 && phys < a.num_blocks)
                prow = (phys * a.Hkv + g_kv) * kPageTokens;
              else
                err.record(kErrPagedBadBlock);
            }
          }
          return prow;
        };
        // K_0 on K-full 0; then V_j and K_{j+1} together on V-full of V_j's
        // stage (issued back to back, so they land together): the MMA warp's
        // wait for V_j before P V also covers the Q K^T on K_{j+1} that
        // follows it, one wait per step fewer.
        bool k0_issued = early && !kPaged;  // contiguous K_0 left with the Q tiles
        int phys_next = phys_of(1);
        int prow = prow_from(0, phys_of(0));
        if (!k0_issued) {
          ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kBarKE), 1, abort_flag, err,
                                                 kErrTimeoutProducer));
          if (ok) {
            mbar_arrive_expect_tx_elect(bar(C::kBarKF), C::kTileBytes);
            load_tile(&tm_k, sbase + C::kOffK, bar(C::kBarKF), 0, prow);
            k0_issued = true;
            if (lane == 0) issued_state[1] = issued_state[1] | 1;
          }
        }
        // Failure-detection test (attn_fwd_ex with ATTN_FWD_DIAG_WAIT_EXPIRES):
        // in CTA 0, two KV steps in, the producer waits on a barrier nothing
        // signals, with a short limit, while copies and products of the CTA
        // are in flight.  The wait expires and records a timeout for this
        // launch; every warp of the CTA drains what it issued, and later CTAs
        // of the launch skip their work.  Other launches are unaffected.
        const int diag_j = (a.diag_wait_ns != 0 && blockIdx.x == 0) ? min(2, n_kv - 1) : -1;
        for (int j = 0; ok && j < n_kv; ++j) {
          if (j == diag_j) {
            __all_sync(0xffffffffu, mbar_wait_limit(bar(C::kBarDiag), 0, abort_flag, err,
                                                    kErrTimeoutDiag, a.diag_wait_ns));
            ok = false;
            break;
          }
          const int vs = j % C::kVStages;
          const bool next = j + 1 < n_kv;
          const int ks1 = (j + 1) % C::kKStages;
          const int phys_after = phys_of(j + 2);  // used one iteration later
          const int prow_next = next ? prow_from(j + 1, phys_next) : 0;
          ok = __all_sync(0xffffffffu,
                          mbar_wait(bar(C::kBarVE + vs), ((j / C::kVStages) & 1) ^ 1, abort_flag,
                                    err, kErrTimeoutProducer));
          if (!ok) break;
          if (next) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kBarKE + ks1),
                                                   (((j + 1) / C::kKStages) & 1) ^ 1, abort_flag,
                                                   err, kErrTimeoutProducer));
            if (!ok) break;
          }
          mbar_arrive_expect_tx_elect(bar(C::kBarVF + vs), (next ? 2 : 1) * C::kTileBytes);
          load_tile(&tm_v, sbase + C::kOffV + vs * C::kTileBytes, bar(C::kBarVF + vs), j, prow);
          if (next)
            load_tile(&tm_k, sbase + C::kOffK + ks1 * C::kTileBytes, bar(C::kBarVF + vs), j + 1,
                      prow_next);
          v_issued = j + 1;
          if (lane == 0) issued_state[0] = v_issued;
          prow = prow_next;
          phys_next = phys_after;
        }
      }
    } else if (warp == 1) {
      // -------------------------------------------------------- MMA issuer
      // The whole warp runs this loop; one elected lane issues each MMA.
      if (n_kv > 0) {
        constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, 0);
        constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, 1);
        // Base descriptors; per-step offsets go into the 16-byte address field.
        const uint64_t q_desc = smem_desc_sw128(sbase + C::kOffQ, 16, 1024);
        const uint64_t k_desc = smem_desc_sw128(sbase + C::kOffK, 16, 1024);
        const uint64_t v_desc = smem_desc_sw128(sbase + C::kOffV, C::kSlabBytes, 1024);
        bool ok = true;
        // S_i = Q_i K_j^T.  The last Q tile using K_j frees its stage.
        // Tile 1 skips the K-full wait when tile 0 has just waited for the
        // same stage and phase: a wait costs this warp over 100 cycles even
        // when the phase is complete, and the tensor pipe idles meanwhile.
        auto issue_qk = [&](int i, int j) -> bool {
          const int ks = j % C::kKStages;
          if (j == 0 && !__all_sync(0xffffffffu, mbar_wait(bar(C::kBarQF + i), 0, abort_flag, err,
                                                           kErrTimeoutMma)))
            return false;
          // K_j (j >= 1) landed with V_{j-1}, whose wait preceded this call.
          if (j == 0 && !(i == 1 && n_t[0] > 0) &&
              !__all_sync(0xffffffffu, mbar_wait(bar(C::kBarKF), 0, abort_flag, err,
                                                 kErrTimeoutMma)))
            return false;
          tc_fence_after();
          const uint32_t d_tmem = tmem + C::kColS + i * 128;
          const uint64_t qa = desc_add(q_desc, uint32_t((i * C::kTileBytes) >> 4));
          const uint64_t kb = desc_add(k_desc, uint32_t((ks * C::kTileBytes) >> 4));
          // 16 head dims (32 bytes, 2 address units) per MMA, four per 64-column slab.
#pragma unroll
          for (int g = 0; g < D / 64; ++g) {
            const uint32_t o = uint32_t((g * C::kSlabBytes) >> 4);
            mma4_bf16_ss<2, 2>(d_tmem, desc_add(qa, o), desc_add(kb, o), kIdescQK, g > 0 ? 1u : 0u);
          }
          mma_commit(bar(C::kBarSF + i));
          if (i == 1 || j >= n_t[1]) mma_commit(bar(C::kBarKE + ks));
          return true;
        };
        // Paged: the V tile holding the sequence's partial last block, and
        // the rows of that block past the end (garbage in the cache).
        int tail_tile = -1, tail_r0 = 0, tail_r1 = 0;
        if constexpr (kPaged) {
          if (Nk % kPageTokens != 0) {
            tail_tile = (Nk - 1) / 128;
            tail_r0 = Nk - tail_tile * 128;
            tail_r1 = min(128, nblk * kPageTokens - tail_tile * 128);
          }
        }
        // O_i += P_i V_j, P_i read from the first 64 TMEM columns of S_i.  The
        // products over keys 0..63 start as soon as that half of P is
        // written, while the softmax warpgroup still works on keys 64..127.
        auto issue_pv = [&](int i, int j) -> bool {
          const int vs = j % C::kVStages;
          if (!__all_sync(0xffffffffu, mbar_wait(bar(C::kBarPF + i), j & 1, abort_flag, err,
                                                 kErrTimeoutMma)))
            return false;
          if (!(i == 1 && j < n_t[0]) &&
              !__all_sync(0xffffffffu, mbar_wait(bar(C::kBarVF + vs), (j / C::kVStages) & 1,
                                                 abort_flag, err, kErrTimeoutMma)))
            return false;
          if constexpr (kPaged) {
            if (j == tail_tile) {
              // 0-probability keys must contribute exactly 0: clear the rows
              // past the end once, before the first MMA that reads them.
              const int nr = tail_r1 - tail_r0;
              uint8_t* vt = smem + C::kOffV + vs * C::kTileBytes;
              for (int idx = lane; idx < C::kSlabs * nr * 8; idx += 32) {
                const int sl = idx / (nr * 8), rem = idx % (nr * 8);
                *reinterpret_cast<uint4*>(vt + sl * C::kSlabBytes + (tail_r0 + rem / 8) * 128 +
                                          (rem % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
              }
              fence_proxy_async_smem();
              __syncwarp();
              tail_tile = -1;
            }
          }
          tc_fence_after();
          const uint32_t a_tmem = tmem + C::kColS + i * 128;
          const uint32_t d_tmem = tmem + C::kColO + i * D;
          // V tile is [128 keys][D] in 64-column slabs: B operand MN-major,
          // 16 keys per MMA = 2 swizzle atoms of 8 rows (SBO 1024, 2048 bytes
          // = 128 address units per MMA), next 64 output columns one slab
          // further (LBO = slab size).  P: 16 keys = 8 TMEM columns per MMA.
          const uint64_t vb = desc_add(v_desc, uint32_t((vs * C::kTileBytes) >> 4));
          mma4_bf16_ts<8, 128>(d_tmem, a_tmem, vb, kIdescPV, j > 0 ? 1u : 0u);
          if (!__all_sync(0xffffffffu, mbar_wait(bar(C::kBarPF2 + i), j & 1, abort_flag, err,
                                                 kErrTimeoutMma)))
            return false;  // the caller drains the first half's MMAs
          tc_fence_after();
          mma4_bf16_ts<8, 128>(d_tmem, a_tmem + 32, desc_add(vb, 512), kIdescPV, 1u);
          if (i == 1 || j >= n_t[1]) mma_commit(bar(C::kBarVE + vs));
          if (j == n_t[i] - 1) mma_commit(bar(C::kBarOF + i));
          return true;
        };
        if (n_t[0] > 0) ok = issue_qk(0, 0);
        if (ok && n_t[1] > 0) ok = issue_qk(1, 0);
        for (int j = 0; ok && j < n_kv; ++j) {
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            if (ok && j < n_t[i]) {
              ok = issue_pv(i, j);
              if (ok && j + 1 < n_t[i]) ok = issue_qk(i, j + 1);
            }
          }
        }
        if (!ok) {
          // Abort path: no MMA may be in flight when TMEM is released.
          mma_commit(bar(C::kBarDrain));
          mbar_wait_drain(bar(C::kBarDrain), 0, globaltimer_ns() + kWaitTimeoutNs);
        }
      }
    }
  } else {
    setmaxnreg_inc<C::kRegsHigh>();
    // ---------------------------------------------------------- softmax
    const int wg = (warp >> 2) - 1;  // Q tile of this warpgroup
    const int quarter = warp & 3;    // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (uint32_t(quarter * 32) << 16);
    const uint32_t col_s = C::kColS + wg * 128;
    const uint32_t col_o = C::kColO + wg * D;
    const int n = n_t[wg];
    const int q_row = q0 + wg * 128 + row;
    // Last key this row may attend (bottom-right causal alignment).
    const int row_last = a.causal ? min(Nk - 1, q_row + (Nk - a.Nq)) : (Nk - 1);
    const float c = a.c_log2;
    float m = -INFINITY;  // reference maximum, log2 units of the scaled score
    float l = 0.f;        // running sum of 2^(s*c - m)
    bool ok = !dead;
    for (int j = 0; j < n; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kBarSF + wg), j & 1, abort_flag, err,
                                             kErrTimeoutSoftmax));
      if (!ok) break;
      tc_fence_after();
      uint32_t s[128];
      // Each load also returns the maximum of its 32 columns (sm_103a).
      float cm[4];
      tmem_ld32_max(lane_base + col_s + 0, s + 0, cm[0]);
      tmem_ld32_max(lane_base + col_s + 32, s + 32, cm[1]);
      tmem_ld32_max(lane_base + col_s + 64, s + 64, cm[2]);
      tmem_ld32_max(lane_base + col_s + 96, s + 96, cm[3]);
      tmem_ld_wait();
      reg_fence<128>(s);
#pragma unroll
      for (int i = 0; i < 4; ++i) asm volatile("" : "+f"(cm[i]));

      const int lim = row_last - j * 128;  // columns > lim are masked
      float rmax;
      if (lim < 127) {
        // diagonal or tail tile: mask first, then the maximum of what is left
#pragma unroll
        for (int cc = 0; cc < 128; ++cc)
          if (cc > lim) s[cc] = __float_as_uint(-INFINITY);
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = __uint_as_float(s[i]);
#pragma unroll
        for (int cc = 8; cc < 120; cc += 16)
#pragma unroll
          for (int i = 0; i < 8; ++i)
            mx[i] = max3f(mx[i], __uint_as_float(s[cc + i]), __uint_as_float(s[cc + 8 + i]));
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = fmaxf(mx[i], __uint_as_float(s[120 + i]));
        rmax = max3f(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
      } else {
        rmax = fmaxf(max3f(cm[0], cm[1], cm[2]), cm[3]);
      }
      __syncwarp();
      const float mt = rmax * c;
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
        // S_i(j) complete implies PV(i, j-1) complete: O_i is not in flight.
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(lane_base + col_o + c0, o);
          tmem_ld_wait();
          reg_fence<32>(o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(lane_base + col_o + c0, o);
        }
      }
      const float neg_m = (m == -INFINITY) ? 0.f : -m;
      const float2 c2 = make_float2(c, c);
      const float2 nm2 = make_float2(neg_m, neg_m);
      float2 acc[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        if (half == 1) {
          // keys 0..63 of P are in TMEM (and O was rescaled before): let the
          // MMA warp start on them
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar(C::kBarPF + wg));
        }
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int cc = half * 64 + 2 * e;
          float2 x = __ffma2_rn(make_float2(__uint_as_float(s[cc]), __uint_as_float(s[cc + 1])),
                                c2, nm2);
          if (kPolyExp && half == 1) {
            x = exp2_fma2(x);
          } else {
            x.x = ex2_approx(x.x);
            x.y = ex2_approx(x.y);
          }
          acc[e & 3] = __fadd2_rn(acc[e & 3], x);
          pk[e] = pack_bf16x2(x.x, x.y);
        }
        // P over the S columns (S is already in registers).
        tmem_st32(lane_base + col_s + half * 32, pk);
      }
      const float2 t01 = __fadd2_rn(acc[0], acc[1]);
      const float2 t23 = __fadd2_rn(acc[2], acc[3]);
      const float2 t = __fadd2_rn(t01, t23);
      l += t.x + t.y;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::kBarPF2 + wg));
    }

    // ---------------------------------------------------------- epilogue
    if (ok && n > 0) {
      ok = __all_sync(0xffffffffu,
                      mbar_wait(bar(C::kBarOF + wg), 0, abort_flag, err, kErrTimeoutEpilogue));
      tc_fence_after();
    }
    uint8_t* stage = smem + C::kOffQ + wg * C::kTileBytes;  // Q_i is no longer read
    if (ok) {
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      // The whole O row in one round trip (all loads issued, one wait).
      uint32_t orow[D];
      if (n > 0) {
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) tmem_ld32(lane_base + col_o + c0, orow + c0);
        tmem_ld_wait();
        reg_fence<D>(orow);
      } else {
#pragma unroll
        for (int e = 0; e < D; ++e) orow[e] = 0u;
      }
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        const uint32_t* o = orow + c0;
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
    named_bar_sync(1 + wg, 128);
    if (!*abort_flag && ok) {
      if (quarter == 0 && lane == 0) {
        for (int s = 0; s < C::kSlabs; ++s)
          tma_store_3d(&tm_o, sbase + C::kOffQ + wg * C::kTileBytes + s * C::kSlabBytes, s * 64,
                       q0 + wg * 128, bh);
        bulk_commit_group();
        bulk_wait_group_read0();
      }
      if (a.lse != nullptr && q_row < a.Nq)
        a.lse[size_t(bh) * a.Nq + q_row] = (l > 0.f) ? (m + log2f(l)) * kLn2 : -INFINITY;
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
    const int v_issued = issued_state[0], first = issued_state[1];
    for (int i = 0; i < 2; ++i)
      if (first & (2 << i)) mbar_wait_drain(bar(C::kBarQF + i), 0, deadline);
    if (first & 1) mbar_wait_drain(bar(C::kBarKF), 0, deadline);
    for (int j = max(0, v_issued - C::kVStages); j < v_issued; ++j)
      mbar_wait_drain(bar(C::kBarVF + j % C::kVStages), (j / C::kVStages) & 1, deadline);
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Sets the kernel's dynamic shared memory limit once per device and variant.
template <int D, bool kPaged, bool kPolyExp>
cudaError_t configure_once() {
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(prefill_fwd_kernel<D, kPaged, kPolyExp>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  return cudaSuccess;
}

// Q and O: [B*H, Nq, D] viewed as a 3-D tensor (D, Nq, B*H), 64 x 128 boxes.
template <int D>
bool encode_q_o(CUtensorMap* tq, CUtensorMap* to, const void* q, void* o, int B, int H, int Nq,
                const char** err) {
  const uint32_t box[3] = {64, 128, 1};
  const uint64_t dq[3] = {uint64_t(D), uint64_t(Nq), uint64_t(B) * H};
  const uint64_t sq[2] = {uint64_t(D) * 2, uint64_t(Nq) * D * 2};
  return encode_tmap_bf16(tq, q, 3, dq, sq, box, true, err) &&
         encode_tmap_bf16(to, o, 3, dq, sq, box, true, err);
}

template <int D, bool kPolyExp>
cudaError_t launch(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int Hkv, int Nq, int Nk, float scale, int causal, unsigned diag_wait_ns,
                   cudaStream_t stream, const char** err) {
  using C = Cfg<D>;
  CUtensorMap tq, tk, tv, to;
  const uint32_t box[3] = {64, 128, 1};
  const uint64_t dk[3] = {uint64_t(D), uint64_t(Nk), uint64_t(B) * Hkv};
  const uint64_t sk[2] = {uint64_t(D) * 2, uint64_t(Nk) * D * 2};
  if (!encode_q_o<D>(&tq, &to, q, o, B, H, Nq, err)) return cudaErrorInvalidValue;
  if (!encode_tmap_bf16(&tk, k, 3, dk, sk, box, true, err)) return cudaErrorInvalidValue;
  if (!encode_tmap_bf16(&tv, v, 3, dk, sk, box, true, err)) return cudaErrorInvalidValue;
  cudaError_t e = configure_once<D, false, kPolyExp>();
  if (e != cudaSuccess) return e;
  Args a = {};
  a.lse = lse;
  a.B = B;
  a.H = H;
  a.Hkv = Hkv;
  a.Nq = Nq;
  a.Nk = Nk;
  a.n_pairs = (Nq + 255) / 256;
  a.c_log2 = scale * kLog2e;
  a.causal = causal;
  // Group-major order (all tile pairs of one (batch, KV head) group, heavy
  // first, before the next group) keeps the resident CTAs on one group's K/V
  // in L2.  It is needed when K + V of every group at once would thrash the
  // 126 MB L2 (above ~96 MB).  With GQA it also pays on grids of four or more
  // waves: on the long-context workload (4 query heads per KV head, 13.8
  // waves) DRAM traffic fell from 534 to 305 MB and time from 1352 to
  // 1339 us.  Without GQA a group is one head and the order only delays the
  // last heads' heaviest pairs (B1 H16 N16384 d64 causal: 625 vs 561 us), and
  // short grids keep the heads interleaved so the heaviest pairs of every
  // head start in the first wave.
  const unsigned grid = unsigned(a.n_pairs) * unsigned(B) * unsigned(H);
  a.group_major = (uint64_t(B) * Hkv * Nk * D * 4 > (96ull << 20) ||
                   (H > Hkv && grid >= 4u * 148u)) ? 1 : 0;
  a.diag_wait_ns = diag_wait_ns;
  a.launch_id = next_launch_id();
  prefill_fwd_kernel<D, false, kPolyExp><<<grid, C::kThreads, C::kSmemBytes, stream>>>(tq, tk, tv,
                                                                                     to, a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_paged(const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_table, const int32_t* kv_lens, int B, int H, int Hkv,
                         int Nq, int num_blocks, int max_blocks, float scale, int causal, void* o,
                         float* lse, cudaStream_t stream, const char** err) {
  using C = Cfg<D>;
  CUtensorMap tq, tk, tv, to;
  // The pool [num_blocks, Hkv, 16, D] as rows of D: one (block, KV head) is
  // 16 consecutive rows, fetched by one 64 x 16 box per 64-column slab.
  const uint64_t rows = uint64_t(num_blocks) * Hkv * kPageTokens;
  const uint32_t box[3] = {64, uint32_t(kPageTokens), 1};
  const uint64_t dk[3] = {uint64_t(D), rows, 1};
  const uint64_t sk[2] = {uint64_t(D) * 2, rows * D * 2};
  if (!encode_q_o<D>(&tq, &to, q, o, B, H, Nq, err)) return cudaErrorInvalidValue;
  if (!encode_tmap_bf16(&tk, k_cache, 3, dk, sk, box, true, err)) return cudaErrorInvalidValue;
  if (!encode_tmap_bf16(&tv, v_cache, 3, dk, sk, box, true, err)) return cudaErrorInvalidValue;
  cudaError_t e = configure_once<D, true, false>();
  if (e != cudaSuccess) return e;
  Args a = {};
  a.lse = lse;
  a.B = B;
  a.H = H;
  a.Hkv = Hkv;
  a.Nq = Nq;
  a.Nk = 0;
  a.n_pairs = (Nq + 255) / 256;
  a.c_log2 = scale * kLog2e;
  a.causal = causal;
  a.block_table = block_table;
  a.kv_lens = kv_lens;
  a.max_blocks = max_blocks;
  a.num_blocks = num_blocks;
  a.oob_row = int(rows);
  a.group_major = 1;  // sequences have their own caches: keep one group's in L2
  a.launch_id = next_launch_id();
  const unsigned grid = unsigned(a.n_pairs) * unsigned(B) * unsigned(H);
  prefill_fwd_kernel<D, true, false><<<grid, C::kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, to, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t prefill_launch(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                           int H, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                           bool poly_exp, unsigned diag_wait_ns, cudaStream_t stream,
                           const char** err) {
  const unsigned w = diag_wait_ns;
  if (poly_exp) {
    if (d == 128)
      return launch<128, true>(q, k, v, o, lse, B, H, Hkv, Nq, Nk, scale, causal, w, stream, err);
    return launch<64, true>(q, k, v, o, lse, B, H, Hkv, Nq, Nk, scale, causal, w, stream, err);
  }
  if (d == 128)
    return launch<128, false>(q, k, v, o, lse, B, H, Hkv, Nq, Nk, scale, causal, w, stream, err);
  return launch<64, false>(q, k, v, o, lse, B, H, Hkv, Nq, Nk, scale, causal, w, stream, err);
}

cudaError_t paged_prefill_launch(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* block_table, const int32_t* kv_lens, int B, int H,
                                 int Hkv, int Nq, int d, int num_blocks, int max_blocks,
                                 float scale, int causal, void* o, float* lse,
                                 cudaStream_t stream, const char** err) {
  if (d == 128)
    return launch_paged<128>(q, k_cache, v_cache, block_table, kv_lens, B, H, Hkv, Nq, num_blocks,
                             max_blocks, scale, causal, o, lse, stream, err);
  return launch_paged<64>(q, k_cache, v_cache, block_table, kv_lens, B, H, Hkv, Nq, num_blocks,
                          max_blocks, scale, causal, o, lse, stream, err);
}

int prefill_take_device_error() {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_prefill_error, sizeof(int)) != cudaSuccess) return -1;
  if (v != 0) cudaMemcpyToSymbol(g_prefill_error, &zero, sizeof(int));
  return v;
}

}  // namespace attn
