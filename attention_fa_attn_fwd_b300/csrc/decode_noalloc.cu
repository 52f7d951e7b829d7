// paged_decode_noalloc: paged decode for callers that cannot allocate device
// memory.
//
// Some callers of this library are not allowed to allocate: for example a
// plugin whose host framework hands it only its input and output buffers (no
// workspace hook), or a serving process that reserves all device memory for
// its KV-cache pool at start-up and forbids cudaMalloc afterwards (a late
// cudaMalloc there can fail, or stall the device while it synchronises).
// paged_decode needs a workspace for its per-split partial results; this
// entry point takes that workspace from a fixed array compiled into the
// library instead, and allocates nothing itself.
//
// The scratch array below is kScratchBytes (32 MiB) on every GPU that loads
// this library, held until the process exits.  All calls share it:
//   * calls whose kernels may overlap on the GPU (different streams, or
//     different host threads on one device) race on it and give wrong
//     results -- serialise them on one stream;
//   * it keeps the previous call's contents; nothing in it needs to start at
//     zero, because the merge kernel reads only partials that the split
//     kernel of the same call has just written -- when the call succeeds.
//     After a call in which a bounded wait expired (attn_device_status then
//     reports ATTN_EDEVICE), o and lse are undefined and may hold values
//     computed from an earlier call's partials.
// The host needs the array's device address, not the name: in host code the
// name is a host-side stand-in.  The first call on each device therefore
// looks the address up (cudaGetSymbolAddress, with that device current) and
// caches it; make that first call before any stream capture.  The cached
// address belongs to the device's current context: resetting the device
// (cudaDeviceReset) after the first call is not supported, because later
// calls would keep using the old address.

#include <cstdio>
#include <mutex>

#include "attn_b300.h"
#include "attn_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device (looked up once
// per device).  Returns nullptr and sets *e on failure.
void* scratch_on_current_device(cudaError_t* e) {
  int dev = 0;
  *e = cudaGetDevice(&dev);
  if (*e != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *e = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    *e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (*e != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" {

attn_status paged_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* block_table, const int32_t* seq_lens,
                                 int num_seqs, int H, int Hkv, int d, int num_blocks,
                                 int max_blocks_per_seq, int block_size, float scale, void* o,
                                 float* lse, attn_stream_t stream) {
  const size_t need = paged_decode_workspace_size(num_seqs, H, Hkv, d, max_blocks_per_seq);
  if (need > kScratchBytes) {
    attn::set_last_error(
        "paged_decode_noalloc: these sizes need %zu bytes of scratch but the library's static "
        "scratch holds %zu; use paged_decode with a caller workspace",
        need, kScratchBytes);
    return ATTN_EINVAL;
  }
  if (need == 0) {
    // Invalid sizes: let paged_decode report exactly which argument is wrong.
    // The stand-in workspace pointer below is never dereferenced: paged_decode
    // rejects these sizes before it launches anything; it is non-null only so
    // that the null-workspace check does not hide the real error.
    return paged_decode(q, k_cache, v_cache, block_table, seq_lens, num_seqs, H, Hkv, d,
                        num_blocks, max_blocks_per_seq, block_size, scale, o, lse,
                        reinterpret_cast<void*>(uintptr_t(256)), 0, stream);
  }
  cudaError_t e = cudaSuccess;
  void* scratch = scratch_on_current_device(&e);
  if (scratch == nullptr) {
    attn::set_last_error("paged_decode_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    return ATTN_ECUDA;
  }
  return paged_decode(q, k_cache, v_cache, block_table, seq_lens, num_seqs, H, Hkv, d, num_blocks,
                      max_blocks_per_seq, block_size, scale, o, lse, scratch, kScratchBytes,
                      stream);
}

}  // extern "C"
