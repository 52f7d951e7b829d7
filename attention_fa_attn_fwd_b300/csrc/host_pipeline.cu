// Attention forward with host-resident inputs and outputs, the transfers
// overlapped with the kernels.
//
// The (batch, KV head) units of a GQA problem are independent and contiguous
// in every tensor ([B, H, N, d] with H = Hkv * G: unit u = b * Hkv + g owns
// query heads g*G .. g*G+G-1 of batch b, i.e. G*N consecutive rows of Q, O
// and LSE, and N consecutive rows of K and V).  So a contiguous range of
// units is itself a problem of the same kind (B = 1, H = n*G, Hkv = n) on
// offset pointers.  The call splits the units into `chunks` ranges and runs,
// for each range c:
//   copy stream "in":   Q, K, V of range c, host -> device workspace
//   caller's stream:    the forward kernel on range c (after its inputs)
//   copy stream "out":  O, LSE of range c, device -> host (after its kernel)
// so the inputs of range c+1 travel while range c computes and range c-1's
// outputs travel back (PCIe is full duplex; each direction has its own copy
// engine).  Events tie the three streams to the caller's: the copies start
// after the work already queued on `stream`, and `stream` continues only
// after the last output copy, so the call is stream-ordered like every other
// entry point.
//
// The two copy streams and the events are created once per calling thread
// and device and kept for later calls (no device memory is allocated here).

#include <cstdio>

#include "attn_internal.h"

namespace attn {

namespace {

constexpr int kMaxPipeChunks = 16;
constexpr int kMaxDevices = 64;

struct Pipe {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t loaded[kMaxPipeChunks] = {};
  cudaEvent_t computed[kMaxPipeChunks] = {};
};

thread_local Pipe g_pipes[kMaxDevices];

cudaError_t get_pipe(Pipe** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  Pipe& p = g_pipes[dev];
  if (!p.ready) {
    e = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.done, cudaEventDisableTiming);
    for (int c = 0; c < kMaxPipeChunks && e == cudaSuccess; ++c) {
      e = cudaEventCreateWithFlags(&p.loaded[c], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.computed[c], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return e;
    p.ready = true;
  }
  *out = &p;
  return cudaSuccess;
}

size_t round256(size_t n) { return (n + 255) / 256 * 256; }

struct Layout {
  size_t q, kv, o, lse;           // bytes of each device buffer
  size_t off_k, off_v, off_o, off_lse, total;
};

Layout layout(int B, int H, int Hkv, int Nq, int Nk, int d) {
  Layout L;
  L.q = size_t(B) * H * Nq * d * 2;
  L.kv = size_t(B) * Hkv * Nk * d * 2;
  L.o = L.q;
  L.lse = size_t(B) * H * Nq * 4;
  L.off_k = round256(L.q);
  L.off_v = L.off_k + round256(L.kv);
  L.off_o = L.off_v + round256(L.kv);
  L.off_lse = L.off_o + round256(L.o);
  L.total = L.off_lse + round256(L.lse);
  return L;
}

}  // namespace

size_t fwd_host_workspace_bytes(int B, int H, int Hkv, int Nq, int Nk, int d) {
  return layout(B, H, Hkv, Nq, Nk, d).total;
}

int fwd_host_max_chunks() { return kMaxPipeChunks; }

cudaError_t fwd_host_launch(const void* q_h, const void* k_h, const void* v_h, void* o_h,
                            float* lse_h, int B, int H, int Hkv, int Nq, int Nk, int d,
                            float scale, int causal, void* workspace, int chunks,
                            cudaStream_t stream, const char** err) {
  Pipe* p = nullptr;
  cudaError_t e = get_pipe(&p);
  if (e != cudaSuccess) return e;
  const Layout L = layout(B, H, Hkv, Nq, Nk, d);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* dq = ws;
  uint8_t* dk = ws + L.off_k;
  uint8_t* dv = ws + L.off_v;
  uint8_t* dout = ws + L.off_o;
  float* dlse = reinterpret_cast<float*>(ws + L.off_lse);

  const int G = H / Hkv;
  const int units = B * Hkv;
  if (chunks <= 0) chunks = 8;
  chunks = chunks < units ? chunks : units;
  if (chunks > kMaxPipeChunks) chunks = kMaxPipeChunks;
  const size_t q_unit = size_t(G) * Nq * d * 2;   // bytes of Q (and O) per unit
  const size_t kv_unit = size_t(Nk) * d * 2;      // bytes of K (and V) per unit
  const size_t lse_unit = size_t(G) * Nq;         // floats of LSE per unit
  const uint8_t* qh = static_cast<const uint8_t*>(q_h);
  const uint8_t* kh = static_cast<const uint8_t*>(k_h);
  const uint8_t* vh = static_cast<const uint8_t*>(v_h);
  uint8_t* oh = static_cast<uint8_t*>(o_h);

  auto range = [&](int c, int* u0, int* n) {
    *u0 = int((long long)units * c / chunks);
    *n = int((long long)units * (c + 1) / chunks) - *u0;
  };
  // On a failure part-way, `stream` still waits for whatever the copy
  // streams already hold, so the workspace is not reused under them.
  auto fail_joined = [&](cudaError_t why) {
    if (cudaEventRecord(p->done, p->in) == cudaSuccess) cudaStreamWaitEvent(stream, p->done, 0);
    if (cudaEventRecord(p->done, p->out) == cudaSuccess) cudaStreamWaitEvent(stream, p->done, 0);
    return why;
  };

  // Inputs, in order, on the "in" stream (after the work already on `stream`).
  if ((e = cudaEventRecord(p->start, stream)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(p->in, p->start, 0)) != cudaSuccess) return e;
  for (int c = 0; c < chunks; ++c) {
    int u0, n;
    range(c, &u0, &n);
    if ((e = cudaMemcpyAsync(dq + u0 * q_unit, qh + u0 * q_unit, n * q_unit,
                             cudaMemcpyHostToDevice, p->in)) != cudaSuccess ||
        (e = cudaMemcpyAsync(dk + u0 * kv_unit, kh + u0 * kv_unit, n * kv_unit,
                             cudaMemcpyHostToDevice, p->in)) != cudaSuccess ||
        (e = cudaMemcpyAsync(dv + u0 * kv_unit, vh + u0 * kv_unit, n * kv_unit,
                             cudaMemcpyHostToDevice, p->in)) != cudaSuccess ||
        (e = cudaEventRecord(p->loaded[c], p->in)) != cudaSuccess)
      return fail_joined(e);
  }
  // Kernels on `stream`, each after its inputs; outputs on the "out" stream.
  for (int c = 0; c < chunks; ++c) {
    int u0, n;
    range(c, &u0, &n);
    if ((e = cudaStreamWaitEvent(stream, p->loaded[c], 0)) != cudaSuccess) return fail_joined(e);
    e = prefill_launch(dq + u0 * q_unit, dk + u0 * kv_unit, dv + u0 * kv_unit, dout + u0 * q_unit,
                       lse_h ? dlse + u0 * lse_unit : nullptr, 1, n * G, n, Nq, Nk, d, scale,
                       causal, false, 0u, stream, err);
    if (e != cudaSuccess || (err && *err))
      return fail_joined(e != cudaSuccess ? e : cudaErrorInvalidValue);
    if ((e = cudaEventRecord(p->computed[c], stream)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(p->out, p->computed[c], 0)) != cudaSuccess ||
        (e = cudaMemcpyAsync(oh + u0 * q_unit, dout + u0 * q_unit, n * q_unit,
                             cudaMemcpyDeviceToHost, p->out)) != cudaSuccess)
      return fail_joined(e);
    if (lse_h && (e = cudaMemcpyAsync(lse_h + u0 * lse_unit, dlse + u0 * lse_unit,
                                      n * lse_unit * sizeof(float), cudaMemcpyDeviceToHost,
                                      p->out)) != cudaSuccess)
      return fail_joined(e);
  }
  if ((e = cudaEventRecord(p->done, p->out)) != cudaSuccess) return fail_joined(e);
  return cudaStreamWaitEvent(stream, p->done, 0);
}

}  // namespace attn
