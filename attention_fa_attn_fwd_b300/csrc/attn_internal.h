// Internal declarations shared by the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace attn {

// Encodes a tiled TMA descriptor; returns false on failure (message in err).
bool encode_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                      const uint64_t* strides_bytes, const uint32_t* box, bool swizzle128,
                      const char** err);

// ---- prefill (prefill_sm103.cu)
cudaError_t prefill_launch(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                           int H, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                           bool poly_exp, unsigned diag_wait_ns, cudaStream_t stream,
                           const char** err);
cudaError_t paged_prefill_launch(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* block_table, const int32_t* kv_lens, int B, int H,
                                 int Hkv, int Nq, int d, int num_blocks, int max_blocks,
                                 float scale, int causal, void* o, float* lse,
                                 cudaStream_t stream, const char** err);
int prefill_take_device_error();  // reads and clears (synchronous)

// ---- forward from host buffers, copies overlapped (host_pipeline.cu)
size_t fwd_host_workspace_bytes(int B, int H, int Hkv, int Nq, int Nk, int d);
int fwd_host_max_chunks();
cudaError_t fwd_host_launch(const void* q_h, const void* k_h, const void* v_h, void* o_h,
                            float* lse_h, int B, int H, int Hkv, int Nq, int Nk, int d,
                            float scale, int causal, void* workspace, int chunks,
                            cudaStream_t stream, const char** err);

// ---- paged decode (decode_sm103.cu)
struct DecodePlan {
  int blocks_per_split;
  int max_splits;
  size_t workspace_bytes;
};
DecodePlan decode_plan(int num_seqs, int H, int Hkv, int d, int max_blocks_per_seq);
cudaError_t decode_launch(const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_table, const int32_t* seq_lens, int num_seqs, int H,
                          int Hkv, int d, int num_blocks, int max_blocks_per_seq, float scale,
                          void* o, float* lse, void* workspace, const DecodePlan& plan,
                          cudaStream_t stream, const char** err);
int decode_take_device_error();

// ---- backward (backward_sm103.cu)
size_t backward_workspace_bytes(int B, int H, int Nq, int d, bool deterministic);
cudaError_t backward_launch(const void* q, const void* k, const void* v, const void* o,
                            const void* dout, const float* lse, void* dq, void* dk, void* dv,
                            int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                            bool deterministic, unsigned diag_wait_ns, void* workspace,
                            cudaStream_t stream, const char** err);
int backward_take_device_error();

// ---- paged-cache append (kv_append.cu)
size_t kv_append_workspace_bytes(int num_seqs, int num_blocks);
cudaError_t kv_append_launch(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             int32_t* block_table, int32_t* seq_lens, int32_t* ref_counts,
                             const int32_t* free_ids, int32_t* free_top, int num_seqs, int T,
                             int Hkv, int d, int num_blocks, int max_blocks, void* workspace,
                             cudaStream_t stream);
int append_take_device_error();

// Sets the calling thread's attn_last_error() message (printf-style).
void set_last_error(const char* fmt, ...);

// A fresh id for one kernel launch (process-wide counter, never 0): a kernel
// whose bounded wait expires records it, and only CTAs of that same launch
// skip their work because of it.
unsigned next_launch_id();

}  // namespace attn
