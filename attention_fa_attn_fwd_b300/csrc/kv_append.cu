// Appending tokens to a paged KV cache, with copy-on-write of shared blocks.
//
// PagedAttention keeps each sequence's K/V in 16-token blocks behind a block
// table, lets sequences with a common prefix share physical blocks, and
// copies a shared block before writing into it (tutorial "第 3 章
// 进阶原理:性能模型与数值稳定性", section 3.0.6: block table, sharing,
// copy-on-write; 3.0.7: block size 16, parallel sampling shares prefixes).
//
// The whole step runs on the GPU, so a decode loop needs no host round trip:
//   kv_append_plan_kernel   one CTA does the bookkeeping: for every sequence,
//                           is its write target shared (copy first), which
//                           fresh blocks does it need, then pops those blocks
//                           off the free stack in sequence order (an
//                           exclusive scan), rewrites the block table, the
//                           reference counts, the lengths and the stack top.
//                           Among the sequences that write into one shared
//                           block, all but the highest-numbered copy it when
//                           they are its only holders; otherwise all copy --
//                           the outcome of handling the sequences one by one
//                           in index order, so the result is deterministic.
//   kv_append_write_kernel  per (sequence, KV head): the block copy (valid
//                           rows only) and the new tokens' K/V rows, 16-byte
//                           vector loads and stores.
// If the stack runs dry, a length is out of range or a table entry is not a
// block id, the plan kernel records a device error and changes nothing.

#include <climits>
#include <cstdio>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {

__device__ int g_append_error;

namespace {

constexpr int kBlock = 16;
constexpr int kPlanThreads = 1024;

struct AppendWs {  // views into the caller's int32 workspace
  int* cnt;         // [num_blocks] writers into each touched shared block
  int* last;        // [num_blocks] highest writer index of each touched block
  int* need;        // [S] blocks this sequence takes off the stack
  int* base;        // [S] exclusive scan of need
  int* pos;         // [S] length before the append
  int* src;         // [S] block copied (or -1)
  int* dst;         // [S] its private copy
  int* skip;        // [1] set when the plan found an error
};

__device__ __forceinline__ AppendWs carve(int* w, int S, int num_blocks) {
  AppendWs a;
  a.cnt = w;
  a.last = a.cnt + num_blocks;
  a.need = a.last + num_blocks;
  a.base = a.need + S;
  a.pos = a.base + S;
  a.src = a.pos + S;
  a.dst = a.src + S;
  a.skip = a.dst + S;
  return a;
}

__global__ void __launch_bounds__(kPlanThreads)
    kv_append_plan_kernel(int32_t* __restrict__ bt, int32_t* __restrict__ seq_lens,
                          int32_t* __restrict__ ref, const int32_t* __restrict__ free_ids,
                          int32_t* __restrict__ free_top, int* __restrict__ wsp, int S, int T,
                          int num_blocks, int max_blocks) {
  __shared__ int s_err;
  __shared__ int s_warp[kPlanThreads / 32];
  __shared__ int s_carry;
  const AppendWs w = carve(wsp, S, num_blocks);
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_err = 0;
    s_carry = 0;
  }
  __syncthreads();

  // 1. validate; reset the counters of every block a sequence writes into
  for (int s = tid; s < S; s += kPlanThreads) {
    const int p = seq_lens[s];
    w.pos[s] = p;
    if (p < 0 || (long long)p + T > (long long)max_blocks * kBlock) {
      atomicCAS(&s_err, 0, kErrAppendTable);
      continue;
    }
    if (p % kBlock != 0) {
      const int P = bt[(size_t)s * max_blocks + p / kBlock];
      if (P < 0 || P >= num_blocks) {
        atomicCAS(&s_err, 0, kErrAppendBlock);
        continue;
      }
      w.cnt[P] = 0;
      w.last[P] = -1;
    }
  }
  __syncthreads();
  if (s_err == 0) {
    // 2. writers per shared block and the last of them
    for (int s = tid; s < S; s += kPlanThreads) {
      const int p = w.pos[s];
      if (p % kBlock != 0) {
        const int P = bt[(size_t)s * max_blocks + p / kBlock];
        atomicAdd(&w.cnt[P], 1);
        atomicMax(&w.last[P], s);
      }
    }
  }
  __syncthreads();
  // 3. blocks each sequence needs: a private copy, plus the blocks its new
  //    tokens open
  for (int s = tid; s < S && s_err == 0; s += kPlanThreads) {
    const int p = w.pos[s];
    int copy = 0;
    if (p % kBlock != 0) {
      const int P = bt[(size_t)s * max_blocks + p / kBlock];
      const int r = ref[P];
      copy = (r > 1 && !(r == w.cnt[P] && s == w.last[P])) ? 1 : 0;
      w.src[s] = copy ? P : -1;
    } else {
      w.src[s] = -1;
    }
    const int opened = (p + T + kBlock - 1) / kBlock - (p + kBlock - 1) / kBlock;
    w.need[s] = copy + opened;
  }
  __syncthreads();
  // 4. exclusive scan of need in sequence order (chunks of kPlanThreads)
  for (int c0 = 0; c0 < S && s_err == 0; c0 += kPlanThreads) {
    const int s = c0 + tid;
    const int v = s < S ? w.need[s] : 0;
    int x = v;
    const int lane = tid & 31, wid = tid >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[wid] = x;
    __syncthreads();
    if (wid == 0) {
      int t = s_warp[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= o) t += y;
      }
      s_warp[lane] = t;
    }
    __syncthreads();
    const int incl = x + (wid > 0 ? s_warp[wid - 1] : 0) + s_carry;
    if (s < S) w.base[s] = incl - v;
    __syncthreads();
    if (tid == kPlanThreads - 1) s_carry = incl;
    __syncthreads();
  }
  const int top = *free_top;
  if (tid == 0 && s_err == 0 && (s_carry > top || top > num_blocks)) s_err = kErrAppendNoFree;
  __syncthreads();
  if (s_err != 0) {
    if (tid == 0) {
      atomicCAS(&g_append_error, 0, s_err);
      *w.skip = 1;
    }
    return;
  }
  // 5. take the blocks off the stack (top first, in scan order), rewrite the
  //    table, the reference counts and the lengths
  for (int s = tid; s < S; s += kPlanThreads) {
    const int p = w.pos[s];
    int a = w.base[s];
    int32_t* row = bt + (size_t)s * max_blocks;
    if (w.src[s] >= 0) {
      const int P = w.src[s];
      const int dst = free_ids[top - 1 - a++];
      w.dst[s] = dst;
      row[p / kBlock] = dst;
      ref[dst] = 1;
      atomicSub(&ref[P], 1);
    }
    for (int lb = (p + kBlock - 1) / kBlock; lb <= (p + T - 1) / kBlock; ++lb) {
      const int id = free_ids[top - 1 - a++];
      row[lb] = id;
      ref[id] = 1;
    }
    seq_lens[s] = p + T;
  }
  if (tid == 0) {
    *free_top = top - s_carry;
    *w.skip = 0;
  }
}

// One CTA per (sequence, KV head); D/8 threads per 16-byte-vector row.
template <int D>
__global__ void __launch_bounds__(128)
    kv_append_write_kernel(const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
                           uint16_t* __restrict__ k_cache, uint16_t* __restrict__ v_cache,
                           const int32_t* __restrict__ bt, const int* __restrict__ wsp, int S,
                           int T, int Hkv, int num_blocks, int max_blocks) {
  const AppendWs w = carve(const_cast<int*>(wsp), S, num_blocks);
  if (*w.skip) return;
  constexpr int VPR = D / 8;              // uint4 per row
  constexpr int RPI = 128 / VPR;          // rows per pass of the CTA
  const int s = blockIdx.x, g = blockIdx.y;
  const int tid = threadIdx.x;
  const int p = w.pos[s];
  auto row_ptr = [&](uint16_t* base, int blk, int r) {
    return reinterpret_cast<uint4*>(base + ((size_t(blk) * Hkv + g) * kBlock + r) * D);
  };
  // copy-on-write: the valid rows of the shared block
  if (w.src[s] >= 0) {
    const int src = w.src[s], dst = w.dst[s], n = p % kBlock;
    for (int i = tid; i < n * VPR; i += 128) {
      const int r = i / VPR, c = i % VPR;
      row_ptr(k_cache, dst, r)[c] = row_ptr(k_cache, src, r)[c];
      row_ptr(v_cache, dst, r)[c] = row_ptr(v_cache, src, r)[c];
    }
  }
  // the new tokens
  const int32_t* row = bt + (size_t)s * max_blocks;
  for (int t0 = 0; t0 < T; t0 += RPI) {
    const int t = t0 + tid / VPR, c = tid % VPR;
    if (t < T) {
      const int q = p + t;
      const int blk = row[q / kBlock];
      const size_t in = ((size_t(s) * T + t) * Hkv + g) * D;
      row_ptr(k_cache, blk, q % kBlock)[c] = reinterpret_cast<const uint4*>(k_new + in)[c];
      row_ptr(v_cache, blk, q % kBlock)[c] = reinterpret_cast<const uint4*>(v_new + in)[c];
    }
  }
}

}  // namespace

size_t kv_append_workspace_bytes(int num_seqs, int num_blocks) {
  const size_t n = 2 * size_t(num_blocks) + 5 * size_t(num_seqs) + 1;
  return (n * sizeof(int) + 255) / 256 * 256;
}

cudaError_t kv_append_launch(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             int32_t* block_table, int32_t* seq_lens, int32_t* ref_counts,
                             const int32_t* free_ids, int32_t* free_top, int num_seqs, int T,
                             int Hkv, int d, int num_blocks, int max_blocks, void* workspace,
                             cudaStream_t stream) {
  int* wsp = static_cast<int*>(workspace);
  kv_append_plan_kernel<<<1, kPlanThreads, 0, stream>>>(block_table, seq_lens, ref_counts, free_ids,
                                                        free_top, wsp, num_seqs, T, num_blocks,
                                                        max_blocks);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 grid(num_seqs, Hkv);
  if (d == 128)
    kv_append_write_kernel<128><<<grid, 128, 0, stream>>>(
        static_cast<const uint16_t*>(k_new), static_cast<const uint16_t*>(v_new),
        static_cast<uint16_t*>(k_cache), static_cast<uint16_t*>(v_cache), block_table, wsp,
        num_seqs, T, Hkv, num_blocks, max_blocks);
  else
    kv_append_write_kernel<64><<<grid, 128, 0, stream>>>(
        static_cast<const uint16_t*>(k_new), static_cast<const uint16_t*>(v_new),
        static_cast<uint16_t*>(k_cache), static_cast<uint16_t*>(v_cache), block_table, wsp,
        num_seqs, T, Hkv, num_blocks, max_blocks);
  return cudaGetLastError();
}

int append_take_device_error() {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_append_error, sizeof(int)) != cudaSuccess) return -1;
  if (v != 0) cudaMemcpyToSymbol(g_append_error, &zero, sizeof(int));
  return v;
}

}  // namespace attn
