"""Benchmark of the attention hot path on B300: prints ONE JSON line.

A step is one pass of the whole hot path over one batch of synthetic input:
  * prefill: attn_fwd on the long-context causal GQA workload
    (B=1, H=32, Hkv=8, Nq=Nk=16384, d=128, Q,K ~ N(0,1)*1.5, V ~ N(0,1));
  * decode:  paged_decode on 64 sequences x 1 query token, H=32, Hkv=8,
    d=128, lengths U{1024..8192}, block 16, groups of 4 sharing a 512-token
    prefix, permuted NaN-poisoned pool.
``value`` is the prefill throughput in TFLOP/s (FLOPs = 4*B*H*Nq*Nk*d, halved
for causal); the decode throughput (KV GB/s over the unique bytes read) is
reported beside it.  Kernel times are CUDA events on the launching stream,
with an L2 flush (outside the events) before every kernel: a 256 MiB write,
then a 256 MiB read so the lines left in L2 are clean (``measure.L2Flush``).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same step on its own GPU
(independent replicas: weak scaling); times are the max over ranks.
``--impl reference`` times the fp64 CPU oracle on a bounded sample of the same
workload (the reference arm of this benchmark).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from attention_fa_attn_fwd_b300 import workloads  # noqa: E402
from attention_fa_attn_fwd_b300.measure import L2Flush  # noqa: E402

PREFILL = "gqa_b1h32kv8_n16384_d128_causal"
DECODE = "paged_decode_s64_h32kv8_d128"
PAGED_PREFILL = "paged_prefill_s8_h32kv8_q2048_d128"
METRIC = "prefill attn TFLOP/s & % BF16 tensor peak; paged decode KV GB/s & % HBM"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p["bf16_tflops_sustained"]), "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
                "source": "fallback"}


def prefill_flops(cfg) -> float:
    f = 4.0 * cfg["B"] * cfg["H"] * cfg["Nq"] * cfg["Nk"] * cfg["d"]
    return f / 2 if cfg["causal"] else f


def paged_prefill_flops(seq_lens, H: int, Nq: int, d: int, causal: bool = True) -> float:
    """4*H*d FLOPs per (query, unmasked key) pair; query i of a chunk of Nq in a
    cache of n tokens sees min(n, i + n - Nq + 1) keys under the causal mask."""
    pairs = 0
    for n in (int(x) for x in seq_lens):
        if not causal:
            pairs += Nq * n
            continue
        for i in range(Nq):
            pairs += max(0, min(n, i + n - Nq + 1))
    return 4.0 * H * d * pairs


def source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "attention_fa_attn_fwd_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str, files):
    """DRAM bytes per launch from the committed ncu summary, if the kernel
    source is unchanged since it was captured; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
            t = json.load(fh)[kernel]
        if t.get("source_sha256") == source_hash(files):
            return float(t["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 20 ms."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = [r for (t, r) in self.samples if t0 <= t <= t1 + 0.05]
        if not rows:
            rows = [r for (_, r) in self.samples[-3:]]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        smax = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if len(r) > 6 + i and r[6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


def spread(ms):
    """Mean, median, p10 and p90 (ms) of a list of event times."""
    xs = sorted(ms)
    n = len(xs)

    def q(f):
        i = f * (n - 1)
        lo = int(math.floor(i))
        hi = min(n - 1, lo + 1)
        return xs[lo] + (xs[hi] - xs[lo]) * (i - lo)

    return {"ms_mean": statistics.mean(xs), "ms_median": q(0.5), "ms_p10": q(0.1),
            "ms_p90": q(0.9), "iters": n}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return ws, rank, local


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- CPU oracle

def oracle_prefill_sample(q, k, v, cfg, budget_s: float, seed: int = 0):
    """Time the fp64 oracle on seeded query rows of the prefill workload until
    ~budget_s of CPU work; returns (TFLOP/s, description, flops, seconds)."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(seed)
    f = lambda t: oracle.bf16_bits_to_f64(t.contiguous().view(torch.int16).numpy())
    scale = 1.0 / math.sqrt(cfg["d"])
    G = cfg["H"] // cfg["Hkv"]
    flops = 0.0
    rows_done = 0
    t_total = 0.0
    t_start = time.perf_counter()
    while time.perf_counter() - t_start < budget_s:
        h = int(rng.integers(cfg["H"]))
        rows = np.sort(rng.choice(cfg["Nq"], size=16, replace=False))
        qh = f(q[:, h:h + 1])
        kh = f(k[:, h // G:h // G + 1])
        vh = f(v[:, h // G:h // G + 1])
        t0 = time.perf_counter()
        oracle.attention_ref(qh, kh, vh, scale, cfg["causal"], rows=rows)
        t_total += time.perf_counter() - t0
        for i in rows:
            keys = (min(cfg["Nk"], i + 1 + cfg["Nk"] - cfg["Nq"]) if cfg["causal"] else cfg["Nk"])
            flops += 4.0 * cfg["d"] * keys
        rows_done += len(rows)
    desc = f"{rows_done} seeded query rows (16 per sampled head) of {PREFILL}"
    return flops / t_total / 1e12, desc, flops, t_total


def oracle_decode_sample(pb, budget_s: float):
    import numpy as np
    import oracle
    f = lambda t: oracle.bf16_bits_to_f64(t.contiguous().view(torch.int16).numpy())
    scale = 1.0 / math.sqrt(pb.q.shape[-1])
    nbytes = 0
    t_total = 0.0
    n = 0
    t_start = time.perf_counter()
    per_tok = pb.k_cache.shape[1] * pb.k_cache.shape[3] * 2 * 2
    while time.perf_counter() - t_start < budget_s and n < pb.num_seqs:
        k, v = pb.logical_kv(n)
        kk, vv, qq = f(k), f(v), f(pb.q[n:n + 1])
        t0 = time.perf_counter()
        oracle.paged_decode_ref(qq, [kk], [vv], scale)
        t_total += time.perf_counter() - t0
        nbytes += int(pb.seq_lens[n]) * per_tok
        n += 1
    return nbytes / t_total / 1e9, f"{n} of {pb.num_seqs} sequences of {DECODE}", t_total


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        n = max((i.get("num_threads", 1) for i in info if i.get("user_api") == "blas"), default=1)
        return int(n)
    except Exception:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- single cases
# ``--case NAME`` runs one hot-path workload a fixed number of times instead of
# the benchmark line (the commands of the Nsight Compute summaries under
# profiles/ use these), or a timing sweep:
#   prefill        attn_fwd on --prefill (default: the long-context GQA workload)
#   decode         paged_decode on the 64-sequence workload (--decode-seqs fewer)
#   step           prefill then decode, as one bench step
#   paged_prefill  chunked prefill of 8 x 2048 tokens over a paged cache
#   backward       attn_bwd on --prefill (after one untimed attn_fwd);
#                  --deterministic selects ATTN_BWD_DETERMINISTIC
#   sweep          attn_fwd over the length sweep at B*N = 16384 tokens
#   configs        attn_fwd on each named prefill workload, with and without
#                  the FMA exp2, and the d64 sweep points with it
#   decode_sweep   paged_decode of 64 sequences (32 at 16384 tokens) of one
#                  fixed context length, 512 .. 16384
# An L2 flush precedes every kernel; each launch's CUDA-event time is printed
# (sweeps: median of --iters runs and TFLOP/s or GB/s).

def _time(fn, flush, iters: int) -> float:
    """Median CUDA-event time (ms) of fn over iters runs after 2 warm-ups, each
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
    return statistics.median(a.elapsed_time(b) for a, b in evs)


def run_case(args):
    from attention_fa_attn_fwd_b300 import binding
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
        bws = torch.empty(binding.attn_bwd_workspace_size(*q.shape[:3], q.shape[3]),
                          dtype=torch.uint8, device=dev)
        runs.append(("attn_bwd", lambda: binding.attn_bwd(q, k, v, o, do, lse, causal=cfg["causal"],
                                                          dq=dq, dk=dk, dv=dv, workspace=bws,
                                                          deterministic=args.deterministic)))
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



# ---------------------------------------------------------------- arms

def run_reference(args, ws, rank):
    """Reference arm: the fp64 CPU oracle, bounded sample per step."""
    if rank != 0:
        return
    cfg = workloads.PREFILL_WORKLOADS[PREFILL]
    q, k, v = workloads.prefill_inputs(**cfg, seed=0)
    pb = workloads.paged_decode_inputs(**workloads.PAGED_WORKLOADS[DECODE], seed=0)
    per_step = max(0.5, min(6.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_prefill_sample(q, k, v, cfg, per_step * 0.2)
    vals, dec, secs = [], [], []
    for i in range(args.steps):
        tf, desc, _, t = oracle_prefill_sample(q, k, v, cfg, per_step * 0.8, seed=i + 1)
        gbs, ddesc, td = oracle_decode_sample(pb, per_step * 0.2)
        vals.append(tf)
        dec.append(gbs)
        secs.append(t + td)
    value = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.mean(secs), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{PREFILL} + {DECODE}", "prefill": cfg,
                   "decode": workloads.PAGED_WORKLOADS[DECODE]},
        "timing": {"l2": "n/a (CPU)", "parallelism": "rank 0 only", "aggregate": "mean",
                   "step_s": spread([1e3 * x for x in secs])},
        "decode": {"value": statistics.mean(dec), "unit": "GB/s"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": blas_threads(),
                         "kind": "oracle", "sample": f"per step: {desc}; decode {ddesc}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def run_ours(args, ws, rank, local):
    from attention_fa_attn_fwd_b300 import binding
    binding.load_library()  # fails loudly if the CUDA library is missing
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    cfg = workloads.PREFILL_WORKLOADS[PREFILL]
    dcfg = workloads.PAGED_WORKLOADS[DECODE]
    q_h, k_h, v_h = workloads.prefill_inputs(**cfg, seed=rank)
    pb = workloads.paged_decode_inputs(**dcfg, seed=rank)
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(cfg["B"], cfg["H"], cfg["Nq"], dtype=torch.float32, device=dev)
    dq, kc, vc = pb.q.to(dev), pb.k_cache.to(dev), pb.v_cache.to(dev)
    bt, sl = pb.block_table.to(dev), pb.seq_lens.to(dev)
    do = torch.empty_like(dq)
    dlse = torch.empty(dq.shape[0], dq.shape[1], dtype=torch.float32, device=dev)
    wsb = binding.paged_decode_workspace_size(dq.shape[0], dq.shape[1], kc.shape[1], dq.shape[2],
                                              bt.shape[1])
    wsp = torch.empty(wsb, dtype=torch.uint8, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    def prefill():
        binding.attn_fwd(q, k, v, causal=True, o=o, lse=lse, stream=stream)

    def decode():
        binding.paged_decode(dq, kc, vc, bt, sl, o=do, lse=dlse, workspace=wsp, stream=stream)

    for _ in range(args.warmup):
        flush()
        prefill()
        flush()
        decode()
    torch.cuda.synchronize()
    assert binding.device_status(stream) == 0

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.6)
    barrier(ws)
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(K):
        flush()
        evs[i][0].record(stream)
        prefill()
        evs[i][1].record(stream)
        flush()
        evs[i][2].record(stream)
        decode()
        evs[i][3].record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    t1 = time.time()
    time.sleep(0.25)
    sampler.stop()
    launches = 3 * K
    p_ms = [evs[i][0].elapsed_time(evs[i][1]) for i in range(K)]
    d_ms = [evs[i][2].elapsed_time(evs[i][3]) for i in range(K)]
    p_mean = max_over_ranks(statistics.mean(p_ms), ws)
    d_mean = max_over_ranks(statistics.mean(d_ms), ws)
    p_spread, d_spread = spread(p_ms), spread(d_ms)
    assert binding.device_status(stream) == 0

    # Whole-job throughput: every rank ran the same step (independent replicas),
    # timed by the slowest rank.
    flops = prefill_flops(cfg) * ws
    tflops = flops / (p_mean * 1e-3) / 1e12
    per_tok = kc.shape[1] * kc.shape[3] * 2 * 2
    uniq_bytes = pb.unique_valid_tokens() * per_tok
    logical_bytes = pb.logical_tokens() * per_tok
    small_bytes = (dq.numel() * 2 * 2 + bt.numel() * 4 + sl.numel() * 4 + dlse.numel() * 4)
    dec_gbs = ws * (uniq_bytes + small_bytes) / (d_mean * 1e-3) / 1e9

    # ---- the opt-in FMA-pipe exp2 variant of the prefill kernel (beside the step)
    def prefill_fma():
        binding.attn_fwd(q, k, v, causal=True, o=o, lse=lse, stream=stream, exp2_fma=True)

    for _ in range(3):
        flush()
        prefill_fma()
    Kx = max(3, min(K, 50))
    x_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(Kx)]
    for i in range(Kx):
        flush()
        x_evs[i][0].record(stream)
        prefill_fma()
        x_evs[i][1].record(stream)
    torch.cuda.synchronize()
    assert binding.device_status(stream) == 0
    px_ms = max_over_ranks(statistics.mean(e[0].elapsed_time(e[1]) for e in x_evs), ws)
    px_tflops = flops / (px_ms * 1e-3) / 1e12

    # ---- chunked prefill over the paged cache (reported beside the step)
    ppc = workloads.PAGED_PREFILL_WORKLOADS[PAGED_PREFILL]
    pp = workloads.paged_prefill_inputs(**ppc, seed=rank)
    pq, pkc, pvc = pp.q.to(dev), pp.k_cache.to(dev), pp.v_cache.to(dev)
    pbt, psl = pp.block_table.to(dev), pp.seq_lens.to(dev)
    po = torch.empty_like(pq)
    plse = torch.empty(pq.shape[:3], dtype=torch.float32, device=dev)

    def paged_prefill():
        binding.paged_prefill(pq, pkc, pvc, pbt, psl, causal=True, o=po, lse=plse, stream=stream)

    for _ in range(3):
        flush()
        paged_prefill()
    Kp = max(3, min(K, 100))
    p_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(Kp)]
    for i in range(Kp):
        flush()
        p_evs[i][0].record(stream)
        paged_prefill()
        p_evs[i][1].record(stream)
    torch.cuda.synchronize()
    assert binding.device_status(stream) == 0
    pp_ms = max_over_ranks(statistics.mean(e[0].elapsed_time(e[1]) for e in p_evs), ws)
    pp_flops = paged_prefill_flops(pp.seq_lens, ppc["H"], ppc["Nq"], ppc["d"]) * ws
    pp_tflops = pp_flops / (pp_ms * 1e-3) / 1e12
    del pq, pkc, pvc, pbt, psl, po, plse

    # ---- KV append for a run of decode steps (reported beside the step).
    # One append is two tiny launches, far shorter than the host-side call, so
    # a run of APPEND_STEPS appends is captured once as a CUDA graph and the
    # replay is timed; the table gets spare columns so no sequence overflows.
    APPEND_STEPS = 16
    nblk = [(int(n) + 15) // 16 for n in pb.seq_lens]
    refs_h = torch.zeros(pb.num_blocks, dtype=torch.int32)
    for s_ in range(pb.num_seqs):
        for b_ in pb.block_table[s_, :nblk[s_]].tolist():
            refs_h[b_] += 1
    free_h = torch.nonzero(refs_h == 0).flatten().to(torch.int32)
    bt_wide = torch.zeros(pb.num_seqs, pb.max_blocks_per_seq + 2, dtype=torch.int32)
    bt_wide[:, :pb.max_blocks_per_seq] = pb.block_table
    a_bt, a_sl, a_rf = bt_wide.to(dev), sl.clone(), refs_h.to(dev)
    a_free = free_h.to(dev)
    a_top = torch.tensor([free_h.numel()], dtype=torch.int32, device=dev)
    saved = (a_bt.clone(), a_sl.clone(), a_rf.clone(), a_top.clone())
    g_ = torch.Generator().manual_seed(rank)
    a_kn = torch.randn(APPEND_STEPS, pb.num_seqs, 1, kc.shape[1], kc.shape[3],
                       generator=g_).to(torch.bfloat16).to(dev)
    a_vn = torch.randn(a_kn.shape, generator=g_).to(torch.bfloat16).to(dev)
    a_ws = torch.empty(binding.kv_append_workspace_size(pb.num_seqs, pb.num_blocks),
                       dtype=torch.uint8, device=dev)
    a_kc, a_vc = kc.clone(), vc.clone()

    def restore():
        for dst_, src_ in zip((a_bt, a_sl, a_rf, a_top), saved):
            dst_.copy_(src_)

    def append_run():
        for i_ in range(APPEND_STEPS):
            binding.kv_append(a_kn[i_], a_vn[i_], a_kc, a_vc, a_bt, a_sl, a_rf, a_free, a_top,
                              workspace=a_ws)

    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        restore()
        append_run()  # warm-up outside capture (first-call device queries)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        append_run()
    Ka = max(3, min(K, 50))
    a_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(Ka)]
    for i in range(Ka):
        restore()
        flush()
        a_evs[i][0].record(stream)
        graph.replay()
        a_evs[i][1].record(stream)
    torch.cuda.synchronize()
    assert binding.device_status(stream) == 0
    assert int(a_sl[0]) == int(saved[1][0]) + APPEND_STEPS
    ap_ms = max_over_ranks(statistics.mean(e[0].elapsed_time(e[1]) for e in a_evs), ws)
    ap_ms /= APPEND_STEPS
    del a_kc, a_vc, graph

    # ---- backward pass of the prefill workload (reported beside the step)
    do_ = workloads.grad_output(q_h.shape, seed=rank).to(dev)
    dq_, dk_, dv_ = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    bws = torch.empty(binding.attn_bwd_workspace_size(cfg["B"], cfg["H"], cfg["Nq"], cfg["d"]),
                      dtype=torch.uint8, device=dev)
    prefill()

    def time_backward(det: bool):
        def backward():
            binding.attn_bwd(q, k, v, o, do_, lse, causal=True, dq=dq_, dk=dk_, dv=dv_,
                             workspace=bws, stream=stream, deterministic=det)

        for _ in range(3):
            flush()
            backward()
        Kb = max(3, min(K, 50))
        b_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(Kb)]
        for i in range(Kb):
            flush()
            b_evs[i][0].record(stream)
            backward()
            b_evs[i][1].record(stream)
        torch.cuda.synchronize()
        assert binding.device_status(stream) == 0
        ms = [e[0].elapsed_time(e[1]) for e in b_evs]
        return max_over_ranks(statistics.mean(ms), ws), spread(ms)

    bw_ms, bw_spread = time_backward(False)
    bwd_ms, bwd_spread = time_backward(True)
    bw_flops = 2.5 * prefill_flops(cfg) * ws  # 5 matrix products vs the forward's 2
    bw_tflops = bw_flops / (bw_ms * 1e-3) / 1e12
    bwd_tflops = bw_flops / (bwd_ms * 1e-3) / 1e12
    del do_, dq_, dk_, dv_, bws

    # ---- end to end through the public API with pinned host buffers
    qp, kp, vp = q_h.pin_memory(), k_h.pin_memory(), v_h.pin_memory()
    op = torch.empty(q_h.shape, dtype=torch.bfloat16).pin_memory()
    lp = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    dqp, btp, slp = pb.q.pin_memory(), pb.block_table.pin_memory(), pb.seq_lens.pin_memory()
    dop = torch.empty(pb.q.shape, dtype=torch.bfloat16).pin_memory()
    dlp = torch.empty(dlse.shape, dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (qp, kp, vp, dqp, btp, slp))
    d2h = sum(t.numel() * t.element_size() for t in (op, lp, dop, dlp))
    Ke = max(3, min(K, 10))
    e_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(Ke)]
    # The prefill leg is one attn_fwd_host call on the pinned host buffers:
    # Q, K, V in and O, LSE out, the transfers overlapped with the kernels
    # inside the call (ranges of KV-head groups, copy streams joined to this one).
    host_ws = torch.empty(binding.attn_fwd_host_workspace_size(
        cfg["B"], cfg["H"], cfg["Hkv"], cfg["Nq"], cfg["Nk"], cfg["d"]), dtype=torch.uint8,
        device=dev)

    def e2e_step(ev):
        flush()
        if ev:
            ev[0].record(stream)
        binding.attn_fwd_host(qp, kp, vp, causal=cfg["causal"], o=op, lse=lp,
                              workspace=host_ws, stream=stream)
        if ev:
            ev[1].record(stream)
        dq.copy_(dqp, non_blocking=True)
        bt.copy_(btp, non_blocking=True)
        sl.copy_(slp, non_blocking=True)
        decode()
        dop.copy_(do, non_blocking=True)
        dlp.copy_(dlse, non_blocking=True)
        if ev:
            ev[2].record(stream)

    e2e_step(None)  # untimed warm-up
    for i in range(Ke):
        e2e_step(e_evs[i])
    torch.cuda.synchronize()
    ep = max_over_ranks(statistics.mean(e_evs[i][0].elapsed_time(e_evs[i][1]) for i in range(Ke)), ws)
    ed = max_over_ranks(statistics.mean(e_evs[i][1].elapsed_time(e_evs[i][2]) for i in range(Ke)), ws)
    e2e_tflops = flops / (ep * 1e-3) / 1e12  # flops already counts every rank

    if rank != 0:
        return
    clocks = sampler.summary(t0, t1)
    traffic = committed_traffic("prefill_fwd_kernel", ["prefill_sm103.cu", "ptx.cuh"])
    cpu_tf, cpu_desc, _, _ = oracle_prefill_sample(q_h, k_h, v_h, cfg, args.cpu_budget)
    cpu_dec, cpu_ddesc, _ = oracle_decode_sample(pb, max(1.0, args.cpu_budget / 4))
    peak_tf = peaks["bf16_tflops"]
    k_tflops = tflops / ws  # one replica's kernel against one GPU's peak
    k_gbs = dec_gbs / ws
    line = {
        "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": p_mean + d_mean, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{PREFILL} + {DECODE}", "prefill": cfg, "decode": dcfg},
        "timing": {"l2": "L2 flush before every timed kernel, outside the events: write 256 MiB, "
                         "then read 256 MiB (clean lines)",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "aggregate": "mean of the K event times (rank 0's spread beside it)"},
        "prefill": {"ms": p_mean, "tflops": tflops, "frac_burst": k_tflops / peak_tf,
                    "frac_sustained": k_tflops / peaks["bf16_tflops_sustained"], **p_spread,
                    "tflops_median": flops / ws / (p_spread["ms_median"] * 1e-3) / 1e12},
        "decode": {"ms": d_mean, "value": dec_gbs, "unit": "GB/s", **d_spread,
                   "unique_kv_bytes": uniq_bytes, "logical_kv_bytes": logical_bytes,
                   "logical_gbs": ws * (logical_bytes + small_bytes) / (d_mean * 1e-3) / 1e9,
                   "frac_hbm_measured": k_gbs / peaks["hbm_gbs"], "frac_hbm_8tbs": k_gbs / 8000.0},
        "roofline": {"bound": "tensor", "achieved": k_tflops, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": k_tflops / peak_tf, "traffic": traffic,
                     "kernel": "prefill_fwd_kernel<128>", "peak_kind": f"bf16 burst ({peaks['source']})"},
        "roofline_decode": {"bound": "hbm", "achieved": k_gbs, "peak": peaks["hbm_gbs"],
                            "unit": "GB/s", "frac": k_gbs / peaks["hbm_gbs"],
                            "traffic": committed_traffic("decode_split_kernel", ["decode_sm103.cu", "ptx.cuh"]),
                            "kernel": "decode_split_kernel<128> + decode_merge_kernel<128>"},
        "prefill_exp2_fma": {"ms": px_ms, "tflops": px_tflops, "frac_burst": px_tflops / ws / peak_tf,
                             "note": "attn_fwd_ex(ATTN_FWD_EXP2_FMA): half the exponentials "
                                     "on the FMA pipe"},
        "paged_prefill": {"workload": PAGED_PREFILL, "config": ppc, "ms": pp_ms,
                          "tflops": pp_tflops, "frac_burst": pp_tflops / ws / peak_tf,
                          "flops": pp_flops / ws, "kernel": "prefill_fwd_kernel<128, paged>",
                          "kv_lens": [int(x) for x in pp.seq_lens]},
        "kv_append": {"workload": f"{DECODE}, one token per sequence per step",
                      "us_per_step": 1e3 * ap_ms,
                      "kernels": "kv_append_plan_kernel + kv_append_write_kernel<128>",
                      "note": f"CUDA graph of {APPEND_STEPS} decode-step appends, time / steps; "
                              "latency-bound: 2 launches, 262 KB of new K/V rows per step"},
        "backward": {"workload": PREFILL, "ms": bw_ms, "tflops": bw_tflops,
                     "frac_burst": bw_tflops / ws / peak_tf, **bw_spread,
                     "flops": bw_flops / ws, "flops_note": "algorithmic: 2.5 x forward (5 products)",
                     "kernels": "bwd_delta_kernel + bwd_fused_kernel + bwd_dq_convert_kernel"},
        "backward_deterministic": {"workload": PREFILL, "ms": bwd_ms, "tflops": bwd_tflops,
                                   "frac_burst": bwd_tflops / ws / peak_tf, **bwd_spread,
                                   "kernels": "bwd_delta_kernel + bwd_dq_kernel<128> + "
                                              "bwd_dkdv_kernel<128> (ATTN_BWD_DETERMINISTIC)"},
        "e2e": {"value": e2e_tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "prefill_ms": ep, "decode_ms": ed,
                "path": "prefill: attn_fwd_host on pinned host buffers (copies overlapped with "
                        "the kernels inside the call); decode: host copies around paged_decode",
                "decode_gbs": ws * (uniq_bytes + small_bytes) / (ed * 1e-3) / 1e9},
        "gpu_launches": launches,
        "clocks": clocks,
        "cpu_baseline": {"value": cpu_tf, "unit": "TFLOP/s", "cores": blas_threads(),
                         "kind": "oracle", "sample": cpu_desc,
                         "decode_gbs": cpu_dec, "decode_sample": cpu_ddesc},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of CPU oracle work for the cpu_baseline")
    ap.add_argument("--case", choices=["prefill", "decode", "step", "paged_prefill", "backward",
                                       "sweep", "decode_sweep", "configs"], default=None,
                    help="run one workload (for Nsight Compute) or a sweep instead of the bench line")
    ap.add_argument("--iters", type=int, default=3, help="--case: runs per workload")
    ap.add_argument("--prefill", default=PREFILL, help="--case prefill/backward: workload name")
    ap.add_argument("--decode-seqs", type=int, default=64,
                    help="--case decode/step: sequences of the decode workload")
    ap.add_argument("--deterministic", action="store_true",
                    help="--case backward: ATTN_BWD_DETERMINISTIC")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.case:
        run_case(args)
        return
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_ours(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
