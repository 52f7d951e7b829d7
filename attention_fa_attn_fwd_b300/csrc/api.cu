// C ABI of libattn_b300.so (declared in include/attn_b300.h): argument
// validation, device check, TMA descriptor encoding, kernel dispatch.
// Nothing is launched on invalid input.

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "attn_b300.h"
#include "attn_internal.h"

namespace {

thread_local char g_msg[512] = "";

attn_status fail(attn_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Returns ATTN_OK if the current device is sm_103 (B300).
attn_status check_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(ATTN_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  static std::mutex mu;
  static int known[64];
  static bool init = false;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!init) {
      for (int& x : known) x = -1;
      init = true;
    }
    if (dev >= 0 && dev < 64 && known[dev] >= 0) {
      return known[dev] ? ATTN_OK
                        : fail(ATTN_EUNSUPPORTED, "device %d is not sm_103 (B300)", dev);
    }
  }
  int major = 0, minor = 0;
  e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e != cudaSuccess) return fail(ATTN_ECUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
  const bool okdev = (major == 10 && minor == 3);
  {
    std::lock_guard<std::mutex> lk(mu);
    if (dev >= 0 && dev < 64) known[dev] = okdev ? 1 : 0;
  }
  if (!okdev) return fail(ATTN_EUNSUPPORTED, "device %d is sm_%d%d, need sm_103", dev, major, minor);
  return ATTN_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn(const char** err) {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  if (!fn && err) *err = "cuTensorMapEncodeTiled is unavailable";
  return fn;
}

}  // namespace

namespace attn {

bool encode_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                      const uint64_t* strides_bytes, const uint32_t* box, bool swizzle128,
                      const char** err) {
  auto fn = get_encode_fn(err);
  if (!fn) return false;
  cuuint64_t gd[5];
  cuuint64_t gs[4];
  cuuint32_t bx[5];
  cuuint32_t es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) gs[i] = strides_bytes[i];
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cuuint32_t(rank), const_cast<void*>(base),
                  gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    if (err) *err = "cuTensorMapEncodeTiled failed";
    return false;
  }
  return true;
}

unsigned next_launch_id() {
  static std::atomic<unsigned> seq{0};
  unsigned id = seq.fetch_add(1, std::memory_order_relaxed) + 1;
  if (id == 0) id = seq.fetch_add(1, std::memory_order_relaxed) + 1;  // skip 0 on wrap
  return id;
}

void set_last_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
}

}  // namespace attn

extern "C" {

const char* attn_last_error(void) { return g_msg; }

attn_status attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int H, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                        unsigned flags, attn_stream_t stream) {
  if (!q || !k || !v || !o) return fail(ATTN_EINVAL, "attn_fwd: null q/k/v/o pointer");
  if (B < 1 || H < 1 || Hkv < 1 || Nq < 1 || Nk < 1)
    return fail(ATTN_EINVAL, "attn_fwd: sizes must be >= 1 (B=%d H=%d Hkv=%d Nq=%d Nk=%d)", B, H,
                Hkv, Nq, Nk);
  if (H % Hkv != 0) return fail(ATTN_EINVAL, "attn_fwd: H=%d is not a multiple of Hkv=%d", H, Hkv);
  if (!(scale > 0.f) || !(scale < 3.0e38f))
    return fail(ATTN_EINVAL, "attn_fwd: scale must be positive and finite");
  if (causal != 0 && causal != 1) return fail(ATTN_EINVAL, "attn_fwd: causal must be 0 or 1");
  if (flags & ~unsigned(ATTN_FWD_EXP2_FMA | ATTN_FWD_DIAG_WAIT_EXPIRES))
    return fail(ATTN_EINVAL, "attn_fwd: unknown flags 0x%x", flags);
  if (d != 64 && d != 128) return fail(ATTN_EUNSUPPORTED, "attn_fwd: head dim %d (need 64 or 128)", d);
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      (lse && !aligned(lse, 4)))
    return fail(ATTN_EINVAL, "attn_fwd: pointers must be 16-byte aligned");
  const long long ctas = (long long)B * H * ((Nq + 127) / 128);
  if (ctas >= (1LL << 31)) return fail(ATTN_EINVAL, "attn_fwd: problem too large");
  attn_status st = check_device();
  if (st != ATTN_OK) return st;
  const char* err = nullptr;
  // The diagnostic wait's limit: 1 ms.
  const unsigned diag_ns = (flags & ATTN_FWD_DIAG_WAIT_EXPIRES) ? 1000000u : 0u;
  cudaError_t e = attn::prefill_launch(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, scale, causal,
                                       (flags & ATTN_FWD_EXP2_FMA) != 0, diag_ns,
                                       reinterpret_cast<cudaStream_t>(stream), &err);
  if (err) return fail(ATTN_ECUDA, "attn_fwd: %s", err);
  if (e != cudaSuccess) return fail(ATTN_ECUDA, "attn_fwd launch: %s", cudaGetErrorString(e));
  return ATTN_OK;
}

attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                     attn_stream_t stream) {
  return attn_fwd_ex(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, scale, causal, 0u, stream);
}

size_t attn_fwd_host_workspace_size(int B, int H, int Hkv, int Nq, int Nk, int d) {
  if (B < 1 || H < 1 || Hkv < 1 || Nq < 1 || Nk < 1 || H % Hkv != 0 || (d != 64 && d != 128))
    return 0;
  return attn::fwd_host_workspace_bytes(B, H, Hkv, Nq, Nk, d);
}

attn_status attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                          int H, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                          void* workspace, size_t workspace_bytes, int chunks,
                          attn_stream_t stream) {
  if (!q || !k || !v || !o || !workspace)
    return fail(ATTN_EINVAL, "attn_fwd_host: null q/k/v/o/workspace pointer");
  if (B < 1 || H < 1 || Hkv < 1 || Nq < 1 || Nk < 1)
    return fail(ATTN_EINVAL, "attn_fwd_host: sizes must be >= 1 (B=%d H=%d Hkv=%d Nq=%d Nk=%d)",
                B, H, Hkv, Nq, Nk);
  if (H % Hkv != 0)
    return fail(ATTN_EINVAL, "attn_fwd_host: H=%d is not a multiple of Hkv=%d", H, Hkv);
  if (!(scale > 0.f) || !(scale < 3.0e38f))
    return fail(ATTN_EINVAL, "attn_fwd_host: scale must be positive and finite");
  if (causal != 0 && causal != 1) return fail(ATTN_EINVAL, "attn_fwd_host: causal must be 0 or 1");
  if (d != 64 && d != 128)
    return fail(ATTN_EUNSUPPORTED, "attn_fwd_host: head dim %d (need 64 or 128)", d);
  if (chunks < 0 || chunks > attn::fwd_host_max_chunks())
    return fail(ATTN_EINVAL, "attn_fwd_host: chunks=%d (0 = automatic, else 1..%d)", chunks,
                attn::fwd_host_max_chunks());
  if (!aligned(workspace, 256))
    return fail(ATTN_EINVAL, "attn_fwd_host: workspace must be 256-byte aligned");
  const long long ctas = (long long)B * H * ((Nq + 127) / 128);
  if (ctas >= (1LL << 31)) return fail(ATTN_EINVAL, "attn_fwd_host: problem too large");
  const size_t need = attn::fwd_host_workspace_bytes(B, H, Hkv, Nq, Nk, d);
  if (workspace_bytes < need)
    return fail(ATTN_EINVAL, "attn_fwd_host: workspace of %zu bytes, need %zu", workspace_bytes,
                need);
  attn_status st = check_device();
  if (st != ATTN_OK) return st;
  const char* err = nullptr;
  cudaError_t e = attn::fwd_host_launch(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, scale, causal,
                                        workspace, chunks, reinterpret_cast<cudaStream_t>(stream),
                                        &err);
  if (err) return fail(ATTN_ECUDA, "attn_fwd_host: %s", err);
  if (e != cudaSuccess) return fail(ATTN_ECUDA, "attn_fwd_host: %s", cudaGetErrorString(e));
  return ATTN_OK;
}

attn_status paged_prefill(const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_table, const int32_t* seq_lens, int num_seqs, int H,
                          int Hkv, int Nq, int d, int num_blocks, int max_blocks_per_seq,
                          int block_size, float scale, int causal, void* o, float* lse,
                          attn_stream_t stream) {
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !o)
    return fail(ATTN_EINVAL, "paged_prefill: null pointer argument");
  if (num_seqs < 1 || H < 1 || Hkv < 1 || Nq < 1 || num_blocks < 1 || max_blocks_per_seq < 1)
    return fail(ATTN_EINVAL, "paged_prefill: sizes must be >= 1");
  if (H % Hkv != 0) return fail(ATTN_EINVAL, "paged_prefill: H=%d not a multiple of Hkv=%d", H, Hkv);
  if (block_size != 16) return fail(ATTN_EINVAL, "paged_prefill: block_size must be 16");
  if (!(scale > 0.f) || !(scale < 3.0e38f))
    return fail(ATTN_EINVAL, "paged_prefill: scale must be positive and finite");
  if (causal != 0 && causal != 1) return fail(ATTN_EINVAL, "paged_prefill: causal must be 0 or 1");
  if (d != 64 && d != 128) return fail(ATTN_EUNSUPPORTED, "paged_prefill: head dim %d", d);
  if ((long long)num_blocks * Hkv * 16 >= (1LL << 31) - 16)
    return fail(ATTN_EINVAL, "paged_prefill: KV pool too large for 32-bit row coordinates");
  if ((long long)max_blocks_per_seq * 16 >= (1LL << 31))
    return fail(ATTN_EINVAL, "paged_prefill: max_blocks_per_seq too large");
  if ((long long)num_seqs * H * ((Nq + 255) / 256) >= (1LL << 31))
    return fail(ATTN_EINVAL, "paged_prefill: problem too large");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(o, 16) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4) || (lse && !aligned(lse, 4)))
    return fail(ATTN_EINVAL, "paged_prefill: misaligned pointer");
  attn_status st = check_device();
  if (st != ATTN_OK) return st;
  const char* err = nullptr;
  cudaError_t e = attn::paged_prefill_launch(q, k_cache, v_cache, block_table, seq_lens, num_seqs,
                                             H, Hkv, Nq, d, num_blocks, max_blocks_per_seq, scale,
                                             causal, o, lse, reinterpret_cast<cudaStream_t>(stream),
                                             &err);
  if (err) return fail(ATTN_ECUDA, "paged_prefill: %s", err);
  if (e != cudaSuccess) return fail(ATTN_ECUDA, "paged_prefill launch: %s", cudaGetErrorString(e));
  return ATTN_OK;
}

size_t attn_bwd_workspace_size(int B, int H, int Nq, int d) {
  if (B < 1 || H < 1 || Nq < 1 || (d != 64 && d != 128)) return 0;
  return attn::backward_workspace_bytes(B, H, Nq, d, false);
}

attn_status attn_bwd_ex(const void* q, const void* k, const void* v, const void* o,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                        int H, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                        void* workspace, size_t workspace_bytes, unsigned flags,
                        attn_stream_t stream) {
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace)
    return fail(ATTN_EINVAL, "attn_bwd: null pointer argument");
  if (B < 1 || H < 1 || Hkv < 1 || Nq < 1 || Nk < 1)
    return fail(ATTN_EINVAL, "attn_bwd: sizes must be >= 1 (B=%d H=%d Hkv=%d Nq=%d Nk=%d)", B, H,
                Hkv, Nq, Nk);
  if (H % Hkv != 0) return fail(ATTN_EINVAL, "attn_bwd: H=%d is not a multiple of Hkv=%d", H, Hkv);
  if (!(scale > 0.f) || !(scale < 3.0e38f))
    return fail(ATTN_EINVAL, "attn_bwd: scale must be positive and finite");
  if (causal != 0 && causal != 1) return fail(ATTN_EINVAL, "attn_bwd: causal must be 0 or 1");
  if (flags & ~unsigned(ATTN_BWD_DETERMINISTIC | ATTN_BWD_DIAG_WAIT_EXPIRES))
    return fail(ATTN_EINVAL, "attn_bwd: unknown flags 0x%x", flags);
  if (d != 64 && d != 128) return fail(ATTN_EUNSUPPORTED, "attn_bwd: head dim %d (need 64 or 128)", d);
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(lse, 4) || !aligned(workspace, 16))
    return fail(ATTN_EINVAL, "attn_bwd: misaligned pointer");
  if ((long long)B * H * ((Nq + 127) / 128) >= (1LL << 31) ||
      (long long)B * Hkv * ((Nk + 127) / 128) >= (1LL << 31))
    return fail(ATTN_EINVAL, "attn_bwd: problem too large");
  const bool det = (flags & ATTN_BWD_DETERMINISTIC) != 0;
  const size_t need = attn::backward_workspace_bytes(B, H, Nq, d, det);
  if (workspace_bytes < need)
    return fail(ATTN_EINVAL, "attn_bwd: workspace %zu bytes < required %zu", workspace_bytes, need);
  attn_status st = check_device();
  if (st != ATTN_OK) return st;
  const char* err = nullptr;
  // The diagnostic wait's limit: 1 ms.
  const unsigned diag_ns = (flags & ATTN_BWD_DIAG_WAIT_EXPIRES) ? 1000000u : 0u;
  cudaError_t e = attn::backward_launch(q, k, v, o, dout, lse, dq, dk, dv, B, H, Hkv, Nq, Nk, d,
                                        scale, causal, det, diag_ns, workspace,
                                        reinterpret_cast<cudaStream_t>(stream), &err);
  if (err) return fail(ATTN_ECUDA, "attn_bwd: %s", err);
  if (e != cudaSuccess) return fail(ATTN_ECUDA, "attn_bwd launch: %s", cudaGetErrorString(e));
  return ATTN_OK;
}

attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, int B, int H, int Hkv, int Nq,
                     int Nk, int d, float scale, int causal, void* workspace,
                     size_t workspace_bytes, attn_stream_t stream) {
  return attn_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, B, H, Hkv, Nq, Nk, d, scale, causal,
                     workspace, workspace_bytes, 0u, stream);
}

size_t kv_append_workspace_size(int num_seqs, int num_blocks) {
  if (num_seqs < 1 || num_blocks < 1) return 0;
  return attn::kv_append_workspace_bytes(num_seqs, num_blocks);
}

attn_status kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                      int32_t* block_table, int32_t* seq_lens, int32_t* ref_counts,
                      const int32_t* free_ids, int32_t* free_top, int num_seqs, int T, int Hkv,
                      int d, int num_blocks, int max_blocks_per_seq, int block_size,
                      void* workspace, size_t workspace_bytes, attn_stream_t stream) {
  if (!k_new || !v_new || !k_cache || !v_cache || !block_table || !seq_lens || !ref_counts ||
      !free_ids || !free_top || !workspace)
    return fail(ATTN_EINVAL, "kv_append: null pointer argument");
  if (num_seqs < 1 || T < 1 || Hkv < 1 || num_blocks < 1 || max_blocks_per_seq < 1)
    return fail(ATTN_EINVAL, "kv_append: sizes must be >= 1");
  if (block_size != 16) return fail(ATTN_EINVAL, "kv_append: block_size must be 16");
  if (d != 64 && d != 128) return fail(ATTN_EUNSUPPORTED, "kv_append: head dim %d", d);
  if (num_seqs > 65535 || Hkv > 65535)
    return fail(ATTN_EINVAL, "kv_append: num_seqs and Hkv must be <= 65535");
  if ((long long)max_blocks_per_seq * 16 >= (1LL << 31) ||
      (long long)num_blocks * 2 + (long long)num_seqs * 5 >= (1LL << 31))
    return fail(ATTN_EINVAL, "kv_append: sizes too large");
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
      !aligned(ref_counts, 4) || !aligned(free_ids, 4) || !aligned(free_top, 4) ||
      !aligned(workspace, 16))
    return fail(ATTN_EINVAL, "kv_append: misaligned pointer");
  const size_t need = attn::kv_append_workspace_bytes(num_seqs, num_blocks);
  if (workspace_bytes < need)
    return fail(ATTN_EINVAL, "kv_append: workspace %zu bytes < required %zu", workspace_bytes, need);
  attn_status st = check_device();
  if (st != ATTN_OK) return st;
  cudaError_t e = attn::kv_append_launch(k_new, v_new, k_cache, v_cache, block_table, seq_lens,
                                         ref_counts, free_ids, free_top, num_seqs, T, Hkv, d,
                                         num_blocks, max_blocks_per_seq, workspace,
                                         reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(ATTN_ECUDA, "kv_append launch: %s", cudaGetErrorString(e));
  return ATTN_OK;
}

size_t paged_decode_workspace_size(int num_seqs, int H, int Hkv, int d, int max_blocks_per_seq) {
  if (num_seqs < 1 || H < 1 || Hkv < 1 || H % Hkv || max_blocks_per_seq < 1 || (d != 64 && d != 128))
    return 0;
  return attn::decode_plan(num_seqs, H, Hkv, d, max_blocks_per_seq).workspace_bytes;
}

attn_status paged_decode(const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_table, const int32_t* seq_lens, int num_seqs, int H,
                         int Hkv, int d, int num_blocks, int max_blocks_per_seq, int block_size,
                         float scale, void* o, float* lse, void* workspace,
                         size_t workspace_bytes, attn_stream_t stream) {
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !o || !workspace)
    return fail(ATTN_EINVAL, "paged_decode: null pointer argument");
  if (num_seqs < 1 || H < 1 || Hkv < 1 || num_blocks < 1 || max_blocks_per_seq < 1)
    return fail(ATTN_EINVAL, "paged_decode: sizes must be >= 1");
  if (H % Hkv != 0) return fail(ATTN_EINVAL, "paged_decode: H=%d not a multiple of Hkv=%d", H, Hkv);
  if (block_size != 16) return fail(ATTN_EINVAL, "paged_decode: block_size must be 16");
  if (!(scale > 0.f) || !(scale < 3.0e38f))
    return fail(ATTN_EINVAL, "paged_decode: scale must be positive and finite");
  if (d != 64 && d != 128) return fail(ATTN_EUNSUPPORTED, "paged_decode: head dim %d", d);
  if (H / Hkv > 16) return fail(ATTN_EUNSUPPORTED, "paged_decode: H/Hkv=%d > 16", H / Hkv);
  if ((long long)num_blocks * Hkv * 16 >= (1LL << 31))
    return fail(ATTN_EINVAL, "paged_decode: KV pool too large for 32-bit row coordinates");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(o, 16) ||
      !aligned(workspace, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
      (lse && !aligned(lse, 4)))
    return fail(ATTN_EINVAL, "paged_decode: misaligned pointer");
  const attn::DecodePlan plan = attn::decode_plan(num_seqs, H, Hkv, d, max_blocks_per_seq);
  if (workspace_bytes < plan.workspace_bytes)
    return fail(ATTN_EINVAL, "paged_decode: workspace %zu bytes < required %zu", workspace_bytes,
                plan.workspace_bytes);
  attn_status st = check_device();
  if (st != ATTN_OK) return st;
  const char* err = nullptr;
  cudaError_t e = attn::decode_launch(q, k_cache, v_cache, block_table, seq_lens, num_seqs, H, Hkv,
                                      d, num_blocks, max_blocks_per_seq, scale, o, lse, workspace,
                                      plan, reinterpret_cast<cudaStream_t>(stream), &err);
  if (err) return fail(ATTN_ECUDA, "paged_decode: %s", err);
  if (e != cudaSuccess) return fail(ATTN_ECUDA, "paged_decode launch: %s", cudaGetErrorString(e));
  return ATTN_OK;
}

attn_status attn_device_status(attn_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(ATTN_ECUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
  const int a = attn::prefill_take_device_error();
  const int b = attn::decode_take_device_error();
  const int c = attn::backward_take_device_error();
  const int f = attn::append_take_device_error();
  if (a < 0 || b < 0 || c < 0 || f < 0)
    return fail(ATTN_ECUDA, "reading the device error word failed");
  if (a || b || c || f)
    return fail(ATTN_EDEVICE, "device error: prefill 0x%x, decode 0x%x, backward 0x%x, append 0x%x",
                a, b, c, f);
  return ATTN_OK;
}

}  // extern "C"
