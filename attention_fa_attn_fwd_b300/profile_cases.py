"""Run one hot-path workload a fixed number of times (for Nsight Compute).

    python -m attention_fa_attn_fwd_b300.profile_cases --case prefill --iters 3
    python -m attention_fa_attn_fwd_b300.profile_cases --case decode --iters 3
    python -m attention_fa_attn_fwd_b300.profile_cases --case step --iters 3
    python -m attention_fa_attn_fwd_b300.profile_cases --case paged_prefill --iters 3

``prefill``: attn_fwd on the long-context causal GQA workload (B1 H32 Hkv8
N16384 d128; 335 MB on the device, larger than L2).  ``decode``: paged_decode
on the 64-sequence workload (2.3 GB pool).  ``step``: both, as one bench step.
``paged_prefill``: chunked prefill of 8 x 2048 tokens over a paged cache.
``backward``: attn_bwd on the prefill workload (after one untimed attn_fwd).
``sweep``: attn_fwd over the sequence-length sweep at B*N = 16384 tokens
(N 512..16384, d 64/128, causal and not); prints TFLOP/s per configuration.
``configs``: attn_fwd on each named prefill workload (tiny, B2 H16 N2048,
long-context GQA), with and without the FMA exp2, and the d64 sweep points
with the FMA exp2; prints TFLOP/s.
``decode_sweep``: paged_decode of 64 sequences (32 at 16384) of one fixed
context length (512..16384 tokens, H32 Hkv8 d128); prints KV GB/s per length.
An L2 flush (``measure.L2Flush``: torch kernels, not this library's)
precedes every kernel, as in bench.py.  Prints the CUDA-event time of each launch.
"""

from __future__ import annotations

import argparse

import torch

from . import binding, workloads
from .measure import L2Flush


def _time(fn, flush, iters: int) -> float:
    """Mean CUDA-event time (ms) of fn over iters runs after 2 warm-ups, each
    run preceded by an L2 flush outside the events."""
    for _ in range(2):
        flush()
        fn()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(iters)]
    for a, b in evs:
        flush()
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / iters


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", choices=["prefill", "decode", "step", "paged_prefill", "backward", "sweep",
                             "decode_sweep", "configs"], default="step")
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--prefill", default="gqa_b1h32kv8_n16384_d128_causal")
    ap.add_argument("--decode-seqs", type=int, default=64,
                    help="sequences of the decode workload (fewer: smaller pool for long captures)")
    args = ap.parse_args(argv)
    binding.load_library()
    dev = torch.device("cuda", 0)
    flush = L2Flush(dev)
    runs = []
    if args.case in ("prefill", "step"):
        cfg = dict(workloads.PREFILL_WORKLOADS.get(args.prefill) or workloads.sweep_workloads()[args.prefill])
        q, k, v = (t.to(dev) for t in workloads.prefill_inputs(**cfg))
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
        runs.append(("attn_fwd", lambda: binding.attn_fwd(q, k, v, causal=cfg["causal"], o=o, lse=lse)))
    if args.case in ("decode", "step"):
        dcfg = dict(workloads.PAGED_WORKLOADS["paged_decode_s64_h32kv8_d128"])
        dcfg["num_seqs"] = args.decode_seqs
        pb = workloads.paged_decode_inputs(**dcfg)
        dq, kc, vc = pb.q.to(dev), pb.k_cache.to(dev), pb.v_cache.to(dev)
        bt, sl = pb.block_table.to(dev), pb.seq_lens.to(dev)
        do = torch.empty_like(dq)
        dl = torch.empty(dq.shape[:2], dtype=torch.float32, device=dev)
        n = binding.paged_decode_workspace_size(dq.shape[0], dq.shape[1], kc.shape[1], dq.shape[2],
                                                bt.shape[1])
        ws = torch.empty(n, dtype=torch.uint8, device=dev)
        runs.append(("paged_decode", lambda: binding.paged_decode(dq, kc, vc, bt, sl, o=do, lse=dl,
                                                                  workspace=ws)))
    if args.case == "paged_prefill":
        pcfg = workloads.PAGED_PREFILL_WORKLOADS["paged_prefill_s8_h32kv8_q2048_d128"]
        pp = workloads.paged_prefill_inputs(**pcfg)
        pq, pkc, pvc = pp.q.to(dev), pp.k_cache.to(dev), pp.v_cache.to(dev)
        pbt, psl = pp.block_table.to(dev), pp.seq_lens.to(dev)
        po = torch.empty_like(pq)
        pl = torch.empty(pq.shape[:3], dtype=torch.float32, device=dev)
        runs.append(("paged_prefill", lambda: binding.paged_prefill(pq, pkc, pvc, pbt, psl,
                                                                    o=po, lse=pl)))
    if args.case == "backward":
        cfg = dict(workloads.PREFILL_WORKLOADS.get(args.prefill) or workloads.sweep_workloads()[args.prefill])
        q, k, v = (t.to(dev) for t in workloads.prefill_inputs(**cfg))
        do = workloads.grad_output(q.shape).to(dev)
        o, lse = binding.attn_fwd(q, k, v, causal=cfg["causal"])
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        bws = torch.empty(binding.attn_bwd_workspace_size(*q.shape[:3]), dtype=torch.uint8,
                          device=dev)
        runs.append(("attn_bwd", lambda: binding.attn_bwd(q, k, v, o, do, lse, causal=cfg["causal"],
                                                          dq=dq, dk=dk, dv=dv, workspace=bws)))
    if args.case == "configs":
        todo = [(n, c, False) for n, c in workloads.PREFILL_WORKLOADS.items()]
        todo += [(n, c, True) for n, c in workloads.PREFILL_WORKLOADS.items()]
        todo += [(n, c, True) for n, c in workloads.sweep_workloads().items() if c["d"] == 64]
        for name, cfg, fma in todo:
            q, k, v = (t.to(dev) for t in workloads.prefill_inputs(**cfg))
            o = torch.empty_like(q)
            lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
            ms = _time(lambda: binding.attn_fwd(q, k, v, causal=cfg["causal"], o=o, lse=lse,
                                                exp2_fma=fma), flush, args.iters)
            fl = 4.0 * cfg["B"] * cfg["H"] * cfg["Nq"] * cfg["Nk"] * cfg["d"]
            fl = fl / 2 if cfg["causal"] else fl
            tag = " exp2_fma" if fma else ""
            print(f"{name}{tag}: {ms:.4f} ms  {fl / ms / 1e9:.1f} TFLOP/s", flush=True)
            del q, k, v, o, lse
        return
    if args.case == "sweep":
        for name, cfg in workloads.sweep_workloads().items():
            q, k, v = (t.to(dev) for t in workloads.prefill_inputs(**cfg))
            o = torch.empty_like(q)
            lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
            ms = _time(lambda: binding.attn_fwd(q, k, v, causal=cfg["causal"], o=o, lse=lse),
                       flush, args.iters)
            fl = 4.0 * cfg["B"] * cfg["H"] * cfg["Nq"] * cfg["Nk"] * cfg["d"]
            fl = fl / 2 if cfg["causal"] else fl
            print(f"{name}: {ms:.4f} ms  {fl / ms / 1e9:.1f} TFLOP/s", flush=True)
            del q, k, v, o, lse
        return
    if args.case == "decode_sweep":
        for L in (512, 1024, 2048, 4096, 8192, 16384):
            S = min(64, 64 * 8192 // L)
            pb = workloads.paged_decode_inputs(num_seqs=S, H=32, Hkv=8, d=128, min_len=L,
                                               max_len=L, group=1, shared_tokens=0, seed=0)
            dq, kc, vc = pb.q.to(dev), pb.k_cache.to(dev), pb.v_cache.to(dev)
            bt, sl = pb.block_table.to(dev), pb.seq_lens.to(dev)
            do = torch.empty_like(dq)
            dl = torch.empty(dq.shape[:2], dtype=torch.float32, device=dev)
            n = binding.paged_decode_workspace_size(S, 32, 8, 128, bt.shape[1])
            ws = torch.empty(n, dtype=torch.uint8, device=dev)
            ms = _time(lambda: binding.paged_decode(dq, kc, vc, bt, sl, o=do, lse=dl, workspace=ws),
                       flush, args.iters)
            nbytes = pb.unique_valid_tokens() * 8 * 128 * 2 * 2
            print(f"decode_s{S}_len{L}: {ms * 1e3:.1f} us  {nbytes / ms / 1e6:.1f} GB/s", flush=True)
            del dq, kc, vc, bt, sl, do, dl, ws
        return
    for it in range(args.iters):
        for name, fn in runs:
            flush()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            print(f"{name} iter {it}: {a.elapsed_time(b):.3f} ms", flush=True)
    assert binding.device_status() == 0


if __name__ == "__main__":
    main()
