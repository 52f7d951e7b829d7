/*
 * attn_b300.h -- C ABI of libattn_b300.so: exact attention forward
 * (FlashAttention-2-style prefill) and paged-KV decode for NVIDIA B300
 * (sm_103a).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers to tensors are DEVICE pointers on the current CUDA device,
 *   allocated and owned by the caller; the library never frees or retains
 *   them (attn_fwd_host takes host tensors and a device workspace, see
 *   there).  The library allocates no device memory in these calls.
 * - Element types: q, k, v, o, k_cache, v_cache are bfloat16 (passed as
 *   void*), lse is float32, block_table and seq_lens are int32.
 * - Every tensor is dense and contiguous in the layout stated per call.
 * - Calls are asynchronous on `stream` (NULL = legacy default stream) and
 *   never synchronise.  Results are deterministic: identical calls give
 *   bit-identical outputs (except attn_bwd's dq at d = 128, see there).
 * - Errors: on invalid arguments nothing is launched and a non-zero status is
 *   returned; attn_last_error() then returns a human-readable message (per
 *   calling thread).  Kernels bound every internal wait (2 s); a wait that
 *   times out records a code that stays until attn_device_status() reads it,
 *   and the outputs of that one launch are undefined.  Poll
 *   attn_device_status() (it synchronises the stream) when a failed launch
 *   must be detected; a status of ATTN_OK from a call only means the launch
 *   was queued.  A timeout affects only the launch it happened in.
 *
 * Notation (source pages): Interview notes "他人面经整理", answer
 * "介绍你理解的flashattention", part 1 defines self-attention as
 * Softmax(Q K^T / sqrt(d_k)) V; part 2 gives the tiled single-pass online
 * softmax.  Tutorial "第 3 章 进阶原理:性能模型与数值稳定性", sections
 * 3.0.6-3.0.7, gives PagedAttention: KV blocks of 16 tokens behind a block
 * table, physical blocks shared by sequences with a common prefix.
 */
#ifndef ATTN_B300_H_
#define ATTN_B300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

/* Compatible with cudaStream_t (struct CUstream_st*). */
typedef struct CUstream_st* attn_stream_t;

typedef enum {
  ATTN_OK = 0,
  ATTN_EINVAL = 1,       /* bad argument: null pointer, bad size, misaligned, ... */
  ATTN_EUNSUPPORTED = 2, /* valid but not implemented here (head dim, GQA ratio, GPU) */
  ATTN_ECUDA = 3,        /* a CUDA runtime call or launch failed */
  ATTN_EDEVICE = 4       /* a kernel recorded a device-side error (attn_device_status) */
} attn_status;

/*
 * attn_fwd -- O = softmax(scale * Q K^T [+ causal mask]) V, plus per-row LSE.
 *
 * Defined by: interview notes "他人面经整理", flashattention answer, part 1
 * (the formula) and part 2 (tiling + online softmax: S and P are never
 * written to device memory).
 *
 *   q    [B, H,   Nq, d]  bf16, contiguous (row-major, d fastest)
 *   k    [B, Hkv, Nk, d]  bf16, contiguous
 *   v    [B, Hkv, Nk, d]  bf16, contiguous
 *   o    [B, H,   Nq, d]  bf16 output
 *   lse  [B, H,   Nq]     fp32 output, or NULL to skip.
 *        lse[i] = ln sum_j exp(scale * q_i . k_j) over the unmasked keys
 *        (natural log); -inf (and o row = 0) for a row with no unmasked key.
 *   scale  > 0 and finite (the definition uses 1/sqrt(d)).
 *   causal 0: every key; 1: bottom-right aligned mask, query row i attends
 *          key j iff j <= i + (Nk - Nq).
 *   GQA: query head h reads key/value head h / (H / Hkv).
 *
 * Requirements: B, H, Hkv, Nq, Nk >= 1; H % Hkv == 0; d in {64, 128}
 * (else ATTN_EUNSUPPORTED); every pointer 16-byte aligned; the device is
 * sm_103 (else ATTN_EUNSUPPORTED).  B*H*ceil(Nq/128) < 2^31.
 */
ATTN_API attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                     attn_stream_t stream);

/*
 * attn_fwd_ex -- attn_fwd with option flags (0 gives exactly attn_fwd).
 *
 *   ATTN_FWD_EXP2_FMA  half of the exponentials (columns 64..127 of every
 *       128-key tile) are computed on the FMA and integer pipes instead of the
 *       MUFU unit: 2^x = 2^round(x) * p(f) with a cubic p fitted by least
 *       squares (relative error < 8e-5; see csrc/fit_exp2_poly.py).  The FSA
 *       page ("FlashAttention systolic array" article, sections 2.1-2.3)
 *       replaces the exponential unit by a least-squares piecewise-linear
 *       exp2 to relieve the softmax bottleneck; this is the same idea on the
 *       GPU's FMA pipe.  Results differ from the default path by rounding
 *       only and stay within the same tolerances against the exact
 *       definition.
 * Unknown flag bits give ATTN_EINVAL.  Everything else as attn_fwd.
 */
#define ATTN_FWD_EXP2_FMA 1u
/*
 *   ATTN_FWD_DIAG_WAIT_EXPIRES  a failure-detection test, not for normal use
 *       (the source pages have no counterpart).  In the first CTA, two key
 *       tiles in (copies and matrix products of the CTA in flight), one
 *       bounded wait on a barrier that nothing signals expires after 1 ms;
 *       every warp of that CTA drains what it issued and exits, later CTAs of
 *       the launch skip their work.  The launch records a timeout (code
 *       0x105, read by attn_device_status) and its outputs are undefined.  It shows that an expired wait is survived and stays
 *       confined to its own launch: later calls, and calls on other streams,
 *       compute normally without attn_device_status being called in between.
 */
#define ATTN_FWD_DIAG_WAIT_EXPIRES 2u
ATTN_API attn_status attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                                 int B, int H, int Hkv, int Nq, int Nk, int d, float scale,
                                 int causal, unsigned flags, attn_stream_t stream);

/*
 * attn_fwd_host_workspace_size -- bytes of device workspace attn_fwd_host
 * needs: Q, K, V, O and LSE of the whole problem, each rounded up to 256
 * bytes.  Returns 0 for invalid sizes.  Pure host function.
 */
ATTN_API size_t attn_fwd_host_workspace_size(int B, int H, int Hkv, int Nq, int Nk, int d);

/*
 * attn_fwd_host -- attn_fwd on HOST buffers, the transfers overlapped with
 * the computation (the same operation and results as attn_fwd, bit for bit).
 *
 *   q, k, v  HOST pointers, layouts as attn_fwd (read).
 *   o, lse   HOST pointers, layouts as attn_fwd (written); lse may be NULL.
 *   workspace        DEVICE buffer of at least attn_fwd_host_workspace_size()
 *                    bytes, 256-byte aligned, owned by the caller.
 *   chunks  0 = automatic (8), else 1..16: the (batch, KV head) units are
 *           split into this many contiguous ranges (at most one per unit);
 *           range c+1 is copied to the device while range c computes and
 *           range c-1's results are copied back.
 *
 * Host buffers should be page-locked (cudaHostAlloc / pinned): then the call
 * returns without waiting and the copies overlap the kernels.  Pageable
 * buffers give the same results but the runtime may block the calling thread
 * during the copies.  The call is stream-ordered: the input copies start
 * after the work already queued on `stream`, and work queued on `stream`
 * after this call starts only after o and lse have reached host memory.  The
 * host buffers must stay valid until then.  The library creates two copy
 * streams and a few events per calling thread and device on the first call
 * and keeps them; it allocates no device memory.  The call can be captured
 * into a CUDA graph (the copy streams fork from and join back to `stream`;
 * make one call outside capture first so the copy streams exist, and use
 * pinned buffers).
 *
 * Requirements as attn_fwd (except host pointers need no alignment), plus a
 * large enough, aligned workspace (else ATTN_EINVAL).
 */
ATTN_API attn_status attn_fwd_host(const void* q, const void* k, const void* v, void* o,
                                   float* lse, int B, int H, int Hkv, int Nq, int Nk, int d,
                                   float scale, int causal, void* workspace,
                                   size_t workspace_bytes, int chunks, attn_stream_t stream);

/*
 * attn_bwd_workspace_size -- bytes of device workspace attn_bwd needs for
 * these sizes: the per-row fp32 D = rowsum(dO o O) (B*H*Nq floats, rounded
 * up to 256 bytes) and, for d = 128, an fp32 dQ accumulator of B*H*Nq*128
 * floats.  Enough for attn_bwd_ex with any flags.  Returns 0 for invalid
 * sizes.  Pure host function.
 */
ATTN_API size_t attn_bwd_workspace_size(int B, int H, int Nq, int d);

/*
 * attn_bwd -- gradients of attn_fwd: given dO = dL/dO, returns dQ, dK, dV,
 * recomputing P from Q, K and the forward pass's LSE instead of storing it.
 *
 * Defined by: interview notes "他人面经整理", flashattention answer, part 3
 * (the backward pass recomputes the attention matrix from Q, K, V and the
 * softmax statistics) and FAQ page "Wie unterscheidet sich die
 * Implementierung von FlashAttention-2 ...", comparison table (recomputation
 * in the backward pass).  With S = scale Q K^T (masked as in attn_fwd) and
 * P = softmax(S): dV = P^T dO, dP = dO V^T, D_i = rowsum(dO_i o O_i),
 * dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q; a KV head's dK, dV
 * sum over the H/Hkv query heads that read it.
 *
 *   q, o, dout, dq   [B, H,   Nq, d]  bf16 (dq output)
 *   k, v, dk, dv     [B, Hkv, Nk, d]  bf16 (dk, dv outputs)
 *   lse              [B, H,   Nq]     fp32, as written by attn_fwd (natural
 *                    log; -inf for rows with no key)
 *   o                attn_fwd's output for the same q, k, v, scale, causal
 *   workspace        >= attn_bwd_workspace_size(B, H, Nq, d) bytes, 16-byte
 *                    aligned, caller-owned; clobbered.
 * Rows with no unmasked key get dq = 0 and contribute nothing to dk, dv.
 *
 * At d = 128 one kernel computes all five products per (key tile, query
 * tile) and adds each key tile's share of dQ into the fp32 accumulator in
 * the workspace with atomic adds, whose order varies: dq can then differ
 * between identical calls in the last bits (dk and dv do not).  At d = 64,
 * and with ATTN_BWD_DETERMINISTIC (attn_bwd_ex), dQ and dK/dV come from two
 * separate kernels (S and dP computed twice), with no atomics: identical
 * calls give identical bits.
 *
 * Requirements: as attn_fwd (d in {64, 128}, H % Hkv == 0, pointers 16-byte
 * aligned, lse 4-byte aligned); dq, dk, dv must not alias the inputs.
 */
ATTN_API attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o,
                              const void* dout, const float* lse, void* dq, void* dk, void* dv,
                              int B, int H, int Hkv, int Nq, int Nk, int d, float scale,
                              int causal, void* workspace, size_t workspace_bytes,
                              attn_stream_t stream);

/*
 * attn_bwd_ex -- attn_bwd with option flags (0 gives exactly attn_bwd).
 *
 *   ATTN_BWD_DETERMINISTIC  bit-reproducible results: dQ from a
 *       query-stationary kernel and dK, dV from a key-stationary one, no
 *       atomics (the pair recomputes S and dP, seven matrix products instead
 *       of five, so it is slower).  Needs only the D part of the workspace
 *       (B*H*Nq floats rounded up to 256 bytes).
 *   ATTN_BWD_DIAG_WAIT_EXPIRES  a failure-detection test, not for normal use:
 *       in the first CTA of the key-stationary kernel, the producer warp lets
 *       one bounded wait (on a barrier nothing signals, 1 ms limit) expire a
 *       few query halves in, with copies and products of the CTA still in
 *       flight.  Every warp of that CTA then
 *       drains what it issued and exits; later CTAs of the launch skip their
 *       work.  The outputs of this call are undefined; attn_device_status
 *       reports code 0x105 once; later calls are unaffected.
 * Unknown flag bits give ATTN_EINVAL.  Everything else as attn_bwd.
 */
#define ATTN_BWD_DETERMINISTIC 1u
#define ATTN_BWD_DIAG_WAIT_EXPIRES 2u
ATTN_API attn_status attn_bwd_ex(const void* q, const void* k, const void* v, const void* o,
                                 const void* dout, const float* lse, void* dq, void* dk, void* dv,
                                 int B, int H, int Hkv, int Nq, int Nk, int d, float scale,
                                 int causal, void* workspace, size_t workspace_bytes,
                                 unsigned flags, attn_stream_t stream);

/*
 * paged_decode_workspace_size -- bytes of device workspace paged_decode needs
 * for these sizes (it holds the per-split partial results merged by LSE).
 * Returns 0 for invalid sizes.  Pure host function.
 */
ATTN_API size_t paged_decode_workspace_size(int num_seqs, int H, int Hkv, int d, int max_blocks_per_seq);

/*
 * paged_decode -- one query token per sequence attends all seq_lens[s] cached
 * keys of its sequence, read through a block table (no causal mask: every
 * cached key precedes the new token).
 *
 * Defined by: tutorial "第 3 章 进阶原理:性能模型与数值稳定性", sections
 * 3.0.6-3.0.7 (PagedAttention block table, block size 16, shared prefix
 * blocks), and the same definition as attn_fwd with Nq = 1.
 *
 *   q            [num_seqs, H, d]                      bf16
 *   k_cache      [num_blocks, Hkv, block_size, d]      bf16 (pool of physical blocks)
 *   v_cache      [num_blocks, Hkv, block_size, d]      bf16
 *   block_table  [num_seqs, max_blocks_per_seq]        int32; entry [s][i] is the
 *                physical block holding tokens 16i .. 16i+15 of sequence s.
 *                Entries past ceil(seq_lens[s]/16) are never read.  Several
 *                sequences may map the same physical block (shared prefix).
 *   seq_lens     [num_seqs]                            int32, 0 <= len <= 16*max_blocks_per_seq
 *   o            [num_seqs, H, d]                      bf16 output
 *   lse          [num_seqs, H]                         fp32 output or NULL
 *   workspace    device scratch of >= paged_decode_workspace_size(...) bytes,
 *                16-byte aligned, owned by the caller; contents need no
 *                initialisation and are clobbered.
 *
 * Cache slots past a sequence's length may hold any bits (even NaN); they do
 * not affect the result.  A block_table entry outside [0, num_blocks) is
 * read as zeros and recorded as a device error (attn_device_status).
 * A sequence of length 0 gets o = 0 and lse = -inf.
 *
 * Requirements: block_size == 16; H % Hkv == 0 and H / Hkv <= 16; d in
 * {64, 128}; num_blocks * Hkv * 16 < 2^31; pointers 16-byte aligned
 * (block_table, seq_lens and lse: 4-byte aligned).
 */
ATTN_API attn_status paged_decode(const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_table, const int32_t* seq_lens, int num_seqs, int H,
                         int Hkv, int d, int num_blocks, int max_blocks_per_seq, int block_size,
                         float scale, void* o, float* lse, void* workspace,
                         size_t workspace_bytes, attn_stream_t stream);

/*
 * paged_decode_noalloc -- paged_decode for callers that cannot allocate
 * device memory (the source pages have no counterpart of this call).
 *
 * Some callers may not call cudaMalloc: a plugin whose host framework passes
 * it only input and output buffers, or a serving process that reserves all
 * device memory for its KV pool at start-up.  This call takes the same
 * arguments as paged_decode minus the workspace, and uses a 32 MiB scratch
 * array compiled into the library instead; it allocates nothing.
 *   - Sizes whose paged_decode_workspace_size() exceeds 32 MiB are rejected
 *     with ATTN_EINVAL (use paged_decode with a caller workspace then).
 *   - The array exists on every GPU that loads the library, until exit.
 *   - All calls share it: calls whose kernels can overlap on the GPU (two
 *     streams, or two host threads on one device) race and give wrong
 *     results.  Serialise them on one stream.
 *   - The first call on each device looks the array's address up (once, with
 *     that device current); make that first call before any stream capture.
 *     The address is kept for the rest of the process: do not reset the
 *     device (cudaDeviceReset) after that first call.
 *   - The array keeps the last call's contents.  After a call whose bounded
 *     wait expired (attn_device_status reports ATTN_EDEVICE), o and lse are
 *     undefined and may hold values from an earlier call.
 */
ATTN_API attn_status paged_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                          const int32_t* block_table, const int32_t* seq_lens,
                                          int num_seqs, int H, int Hkv, int d, int num_blocks,
                                          int max_blocks_per_seq, int block_size, float scale,
                                          void* o, float* lse, attn_stream_t stream);

/*
 * paged_prefill -- chunked prefill over a paged KV cache: each sequence's Nq
 * newest tokens (the chunk being prefilled) attend the sequence's cached keys,
 * read through the block table, with the same tiled single-pass kernel as
 * attn_fwd.
 *
 * Defined by: tutorial "第 3 章 进阶原理:性能模型与数值稳定性", section 3.0.6
 * (FlashAttention-2 and PagedAttention used together: the fused kernel reads
 * the paged cache) and the definition of attn_fwd.
 *
 *   q            [num_seqs, H, Nq, d]                  bf16: the chunk's queries
 *   k_cache      [num_blocks, Hkv, block_size, d]      bf16 pool (as paged_decode)
 *   v_cache      [num_blocks, Hkv, block_size, d]      bf16
 *   block_table  [num_seqs, max_blocks_per_seq]        int32 (as paged_decode)
 *   seq_lens     [num_seqs]                            int32: cached tokens of each
 *                sequence, the chunk's own keys included (its last Nq tokens).
 *   o            [num_seqs, H, Nq, d]                  bf16 output
 *   lse          [num_seqs, H, Nq]                     fp32 output or NULL
 *   causal 1: query row i is token seq_lens[s] - Nq + i and attends key j iff
 *          j <= i + seq_lens[s] - Nq (rows with no key: o = 0, lse = -inf);
 *          0: every cached key.
 *
 * Cache slots past a sequence's length may hold any bits (even NaN).  A
 * block_table entry outside [0, num_blocks) is read as zeros and a seq_lens
 * entry outside [0, 16 * max_blocks_per_seq] is clamped; both are recorded as
 * device errors (attn_device_status).
 *
 * Requirements: block_size == 16; H % Hkv == 0; d in {64, 128};
 * num_blocks * Hkv * 16 < 2^31 - 16; pointers 16-byte aligned (block_table,
 * seq_lens and lse: 4-byte aligned).  No workspace; nothing is allocated.
 */
ATTN_API attn_status paged_prefill(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_table, const int32_t* seq_lens,
                                   int num_seqs, int H, int Hkv, int Nq, int d, int num_blocks,
                                   int max_blocks_per_seq, int block_size, float scale, int causal,
                                   void* o, float* lse, attn_stream_t stream);

/*
 * kv_append_workspace_size -- bytes of device workspace kv_append needs
 * (int32 scratch: 2 per pool block + 5 per sequence + 1).  0 for invalid
 * sizes.  Pure host function.
 */
ATTN_API size_t kv_append_workspace_size(int num_seqs, int num_blocks);

/*
 * kv_append -- append T new tokens' K/V to every sequence of a paged cache,
 * copying a shared block before writing into it (copy-on-write).
 *
 * Defined by: tutorial "第 3 章 进阶原理:性能模型与数值稳定性", section 3.0.6
 * (PagedAttention: block table, sharing between sequences, copy-on-write)
 * and 3.0.7 (block size 16; parallel sampling shares prefix blocks).  The
 * pages name copy-on-write without detail; the reading implemented: sequence
 * s's tokens seq_lens[s] .. seq_lens[s]+T-1 are written; a write into a block
 * with ref_counts > 1 first copies that block into a fresh one (the table
 * then points at the copy, the old block loses one reference), except that
 * when every holder of the block is writing into it this step, the
 * highest-numbered holder writes in place -- exactly what handling the
 * sequences one at a time in index order gives.  Tokens that start a block
 * take a fresh block.  Fresh blocks are popped off the free stack in sequence
 * order: the a-th block taken this call is free_ids[*free_top - 1 - a].
 *
 *   k_new, v_new  [num_seqs, T, Hkv, d]               bf16 (read)
 *   k_cache       [num_blocks, Hkv, 16, d]            bf16 (written)
 *   v_cache       [num_blocks, Hkv, 16, d]            bf16 (written)
 *   block_table   [num_seqs, max_blocks_per_seq]      int32 (updated)
 *   seq_lens      [num_seqs]                          int32 (each += T)
 *   ref_counts    [num_blocks]                        int32 (updated): number of
 *                 (sequence, logical block) table entries holding each block
 *   free_ids      [>= *free_top]                      int32 free block ids (read)
 *   free_top      [1]                                 int32 stack height (updated)
 *   workspace     >= kv_append_workspace_size(num_seqs, num_blocks) bytes,
 *                 16-byte aligned; clobbered.
 * All pointers are device pointers; nothing is read back to the host.  If a
 * length is negative or would pass 16 * max_blocks_per_seq, a table entry to
 * be written through is not a block id, or the stack holds too few blocks,
 * nothing is modified and attn_device_status() reports the error.
 *
 * Requirements: block_size == 16; d in {64, 128}; num_seqs, Hkv <= 65535;
 * k_new, v_new, caches and workspace 16-byte aligned.  Blocks in the stack
 * must have ref_counts 0.
 */
ATTN_API attn_status kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                               int32_t* block_table, int32_t* seq_lens, int32_t* ref_counts,
                               const int32_t* free_ids, int32_t* free_top, int num_seqs, int T,
                               int Hkv, int d, int num_blocks, int max_blocks_per_seq,
                               int block_size, void* workspace, size_t workspace_bytes,
                               attn_stream_t stream);

/*
 * attn_selftest_wait_timeout -- diagnostic for the library's failure
 * detection (the source pages have no counterpart).  Every wait inside the
 * kernels is bounded: if the data it waits for never arrives, it gives up,
 * records an error code read by attn_device_status() and lets the kernel
 * return, so a broken pipeline never hangs the GPU.  This call launches one
 * warp that waits on a barrier nothing will ever signal, with a limit of
 * limit_us microseconds (1 .. 1e6), synchronises `stream` and checks that the
 * expiry was detected and reported.  Returns ATTN_OK if it was, ATTN_EDEVICE
 * if not, ATTN_EINVAL for a bad limit, ATTN_ECUDA if a CUDA call failed.
 * It does not touch the error words attn_device_status() reads.
 */
ATTN_API attn_status attn_selftest_wait_timeout(unsigned limit_us, attn_stream_t stream);

/* Message for the last non-OK status returned on the calling thread. */
ATTN_API const char* attn_last_error(void);

/*
 * attn_device_status -- synchronises `stream`, then reads and clears the
 * device error words the kernels set (a bounded wait that timed out, an
 * out-of-range block id).  Returns ATTN_OK, ATTN_EDEVICE (message holds the
 * codes) or ATTN_ECUDA.  The words are shared by every stream and launch on
 * the device and keep the first code recorded since the last read; the
 * launch that recorded it has undefined outputs, other launches do not.
 */
ATTN_API attn_status attn_device_status(attn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_B300_H_ */
