"""Benchmark of the chunked gated delta rule forward + backward on GB300.

One step = one training pass of the whole hot path over one batch: the
forward (gate cumsum, WY matrix, state recurrence and output, saving g_cumsum
and A) followed by the backward (state recompute, reverse state-gradient
chain, per-chunk gradients), on synthetic seeded inputs of the dense prefill
workload B=2, T=4096, H_q=H_v=32, K=V=128, bf16, q/k L2-normalised in the
kernels.

Prints one JSON line.  --impl reference times the fp64 CPU oracle instead
(a bounded sample of the same workload on the host cores).
"""

from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from gated_delta_rule_38_gb300.inputs import WORKLOADS, make_inputs  # noqa: E402

METRIC = "GDN fwd+bwd tokens/s & TFLOP/s (H=32,K=V=128,bf16) vs roofline, 1xGB300"
# DRAM bytes (read + write) per launch on the dense workload from one ncu capture of each kernel as it
# stands (profiles/*_dense_B2_T4096_H32.md); an entry must be removed when its kernel changes.
NCU_TRAFFIC = {"wy_fwd": 172.6e6, "chain_fwd": 496.5e6, "chain_rev": 437.7e6, "chunk_p": 151.4e6,
               "bwd_chunk": 884.1e6}
C = 64
L2_BYTES = 129 * 2 ** 20


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def work(w, backward=True):
    """Algorithmic FLOPs and bytes of one step (forward saving A and g_cumsum, plus backward).

    FLOPs per token and value head (multiply-add = 2, C = 64, K = V = 128):
    forward Hq/Hv * 4CK + 2C(K+2V) + 6KV; backward twice the forward plus 4C^2.
    Bytes: every tensor the pass must read or write once.
    """
    K = V = 128
    tok = w.tokens
    e = 2
    fwd_f = tok * (w.Hq * 4 * C * K + w.Hv * (2 * C * (K + 2 * V) + 6 * K * V))
    bwd_f = 2 * fwd_f + tok * w.Hv * 4 * C * C
    N = w.num_seqs
    st = N * w.Hv * K * V * 4
    qk = 2 * tok * w.Hq * K * e
    vv = tok * w.Hv * V * e
    gb = 2 * tok * w.Hv * e
    fwd_b = qk + vv + gb + vv + tok * w.Hv * (C * e + 4)  # in; o; A and g_cumsum out
    if w.has_h0:
        fwd_b += st
    if w.final_state:
        fwd_b += st
    bwd_b = qk + vv + tok * w.Hv * (4 + e + C * e) + vv + qk + vv + gb  # q,k,v,g_cs,beta,A,do in; grads out
    if w.has_h0:
        bwd_b += 2 * st
    if w.final_state:
        bwd_b += st
    return (fwd_f, fwd_b, bwd_f, bwd_b) if backward else (fwd_f, fwd_b, 0, 0)


def rank_seed(rank: int) -> int:
    """Each rank draws its own batch (weak scaling over independent streams; no data-path collective)."""
    return 42 + rank


def max_over_ranks(x: float, dist, device) -> float:
    """The job's time is the slowest rank's (max-reduce; the identity without a process group)."""
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, seconds: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank * world / seconds


class Clocks:
    """nvidia-smi sampler running during the timed region."""

    def __init__(self, index=0):
        self.index = index
        self.rows = []
        self.proc = None

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + q,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 8:
                self.rows.append(parts)

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm = sorted(float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit())
        mx = max(float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit())
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(self.rows)}


def run_ours(args):
    import gated_delta_rule_38_gb300 as gdr
    from gated_delta_rule_38_gb300 import _lib

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    w = WORKLOADS[args.workload]
    l2 = not w.host_l2
    x = make_inputs(w, seed=rank_seed(rank))  # every rank: its own batch (weak scaling, no collective)
    dev = torch.device("cuda", local)
    d = {k: (v.to(dev) if v is not None else None) for k, v in x.items()}
    cu = None if w.cu_seqlens is None else torch.tensor(w.cu_seqlens, dtype=torch.int32, device=dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    # the forward hands its decayed causal blocks and q/k norms to the backward (one buffer, reused by the steps)
    saved = gdr.saved_buffer(d["q"], d["v"], d["g"], cu_seqlens=cu, use_qk_l2norm_in_kernel=l2)

    def step(dd):
        gcs, A, o, _, fin = gdr.chunk_gated_delta_rule_fwd(
            dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], initial_state=dd["h0"],
            output_final_state=w.final_state, cu_seqlens=cu, use_qk_l2norm_in_kernel=l2, saved=saved)
        grads = gdr.chunk_gated_delta_rule_bwd(
            dd["q"], dd["k"], dd["v"], gcs, dd["beta"], A, dd["do"], dht=dd["dht"], initial_state=dd["h0"],
            cu_seqlens=cu, use_qk_l2norm_in_kernel=l2, saved=saved)
        return o, grads

    for _ in range(args.warmup):
        step(d)
    torch.cuda.synchronize()

    # ---- device-resident timing: per step events, L2 flushed between steps (outside the events).  The
    # library's per-kernel event profiler stays off here (its event pairs would sit between the step's
    # kernels); a second pass of the same steps with it on gives the per-kernel times and the launch count.
    stream = torch.cuda.current_stream(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        for i in range(args.steps):
            flush.zero_()
            evs[i][0].record(stream)
            step(d)
            evs[i][1].record(stream)
        torch.cuda.synchronize()
    ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in evs) / args.steps, dist, dev)
    _lib.profile_enable(True)
    for i in range(args.steps):
        flush.zero_()
        step(d)
    torch.cuda.synchronize()
    _lib.profile_enable(False)
    prof = _lib.profile_read()

    # ---- end to end: pinned host inputs -> device, step, every output -> pinned host buffers.  Steps are
    # pipelined over two device input sets: the copy stream brings step i+1's inputs in while step i
    # computes, and the read-back stream takes step i's outputs out while step i+1 computes.
    keys = ["q", "k", "v", "g", "beta", "do"] + [k for k in ("h0", "dht") if x[k] is not None]
    hx = {k: x[k].pin_memory() for k in keys}
    h2d = sum(hx[k].numel() * hx[k].element_size() for k in keys)
    bufs = [{k: torch.empty_like(d[k]) for k in keys} for _ in range(2)]
    o, grads = step(d)
    shapes = [t for t in (o,) + tuple(grads) if t is not None]
    hout = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in shapes] for _ in range(2)]
    d2h = sum(t.numel() * t.element_size() for t in shapes)
    copy_s, read_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    buf_free = [None, None]
    for it in range(args.warmup + args.steps):
        if it == args.warmup:
            torch.cuda.synchronize()
            if dist:
                dist.barrier()
            t0 = time.perf_counter()
        j = it % 2
        with torch.cuda.stream(copy_s):
            if buf_free[j] is not None:
                copy_s.wait_event(buf_free[j])
            for k in keys:
                bufs[j][k].copy_(hx[k], non_blocking=True)
            in_ready[j].record(copy_s)
        stream.wait_event(in_ready[j])
        dd = dict(d)
        dd.update(bufs[j])
        o, grads = step(dd)
        buf_free[j] = torch.cuda.Event()
        buf_free[j].record(stream)
        outs = [t for t in (o,) + tuple(grads) if t is not None]
        with torch.cuda.stream(read_s):
            read_s.wait_event(buf_free[j])
            for t, h in zip(outs, hout[j]):
                h.copy_(t, non_blocking=True)
                t.record_stream(read_s)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / args.steps, dist, dev)

    fwd_f, fwd_b, bwd_f, bwd_b = work(w)
    hbm, tf_burst, tf_sus, src = peaks()
    tokens = w.tokens * world
    value = job_throughput(w.tokens, world, ms * 1e-3)
    # dominant kernel by measured time share
    tot = sum(v[1] for v in prof.values()) or 1.0
    name, (cnt, kms) = max(prof.items(), key=lambda kv: kv[1][1])
    per_launch_ms = kms / cnt
    kernel_bytes = {
        # algorithmic bytes one launch of each kernel must move: the per-chunk gradient kernel reads every
        # input of the backward and writes every gradient; the forward recurrence reads the forward's inputs
        # and writes o
        "bwd_chunk": bwd_b, "chain_fwd": fwd_b, "chain_bwd": bwd_b * 0.5, "chain_fwd_recompute": fwd_b,
        "chain_pair": bwd_b * 0.5, "chain_rev": bwd_b * 0.5, "wy_fwd": fwd_b * 0.4, "chunk_p": fwd_b * 0.4,
    }
    kb = kernel_bytes.get(name, fwd_b + bwd_b)
    achieved = kb / (per_launch_ms * 1e-3) / 1e9
    traffic = NCU_TRAFFIC.get(name) if args.workload == "dense" else None
    roofline = {"kernel": name, "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "traffic": traffic, "peak_source": src,
                "share": round(kms / tot, 3), "algorithmic_bytes": int(kb)}
    rl_us = max((fwd_b + bwd_b) / (hbm * 1e9), (fwd_f + bwd_f) / (tf_sus * 1e12)) * 1e6
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == torch.bfloat16 else "fp16", "data": "synthetic",
        "config": {"workload": "dense prefill B=%d T=%d Hq=%d Hv=%d K=V=128 l2norm-in-kernel" % (
            w.B, w.T, w.Hq, w.Hv) if args.workload == "dense" else args.workload,
            "B": w.B, "T": w.T, "Hq": w.Hq, "Hv": w.Hv, "chunk": C,
            "l2": "flushed between steps (256 MiB write outside the timed events)", "parallelism": "replicas"},
        "tflops": round((fwd_f + bwd_f) / (ms * 1e-3) / 1e12, 2),
        "step_roofline_us": round(rl_us, 2), "step_roofline_frac": round(rl_us / (ms * 1e3), 4),
        "kernels_ms_per_step": {k: round(v[1] / args.steps, 4) for k, v in prof.items()},
        "roofline": roofline,
        "e2e": {"value": round(tokens / e2e_s, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": int(sum(v[0] for v in prof.values())),
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def cpu_baseline(w, budget_s):
    """The fp64 oracle on a bounded sample of the workload (whole sequences, a subset of heads)."""
    import oracle
    nthreads = oracle.max_threads()
    x = make_inputs(w)
    pb = oracle.Problem(B=w.B, T=w.T, Hq=w.Hq, Hv=w.Hv, l2norm=not w.host_l2, cu_seqlens=w.cu_seqlens)
    heads = [0]
    t0 = time.perf_counter()
    oracle.fwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"], heads=heads, nthreads=nthreads)
    oracle.bwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], h0=x["h0"], dht=x["dht"], heads=heads,
               nthreads=nthreads)
    dt = time.perf_counter() - t0
    nh = 1
    # grow the sample (more heads) while it stays inside the budget
    while dt * 2.2 < budget_s and nh * 2 <= w.Hv:
        nh *= 2
        heads = list(range(nh))
        t0 = time.perf_counter()
        oracle.fwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"], heads=heads, nthreads=nthreads)
        oracle.bwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], h0=x["h0"], dht=x["dht"],
                   heads=heads, nthreads=nthreads)
        dt = time.perf_counter() - t0
    token_heads = w.tokens * nh
    return {"value": round(token_heads / w.Hv / dt, 1), "unit": "tokens/s", "cores": nthreads, "kind": "oracle",
            "sample": "fwd+bwd of all %d tokens on %d of %d value heads (%.1f s); tokens/s scaled to all heads"
                      % (w.tokens, nh, w.Hv, dt)}


def run_reference(args):
    """The oracle as the reference arm: fp64 CPU, bounded sample, on rank 0 only."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    samples = []
    for i in range(args.warmup + args.steps):
        cb = cpu_baseline(w, args.cpu_seconds / max(1, args.steps))
        if i >= args.warmup:
            samples.append(cb)
    v = sum(s["value"] for s in samples) / len(samples)
    tokens = w.tokens
    line = {"metric": METRIC, "impl": "reference", "value": round(v, 1), "unit": "tokens/s",
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tokens / v * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "dense prefill B=%d T=%d Hq=%d Hv=%d K=V=128 l2norm-in-kernel" % (
                w.B, w.T, w.Hq, w.Hv) if args.workload == "dense" else args.workload},
            "cpu_baseline": {"value": round(v, 1), "unit": "tokens/s", "kind": "oracle",
                             "cores": samples[-1]["cores"], "sample": samples[-1]["sample"]},
            "e2e": {"value": round(v, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_decode(args):
    """Recurrent decode: one token for each of 256 rows x 32 heads from resident fp32 states (the state cache
    of autoregressive inference), updated in place.  HBM-bound on the states (64 KB per row and head, read and
    written every step); the 537 MB of states exceed L2, so no flush is needed between steps."""
    import gated_delta_rule_38_gb300 as gdr
    from gated_delta_rule_38_gb300.inputs import custom

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    w = custom(name="decode", B=256, T=1, Hq=32, Hv=32, host_l2=False)
    x = make_inputs(w)
    d = {k: (v.to(dev) if v is not None else None) for k, v in x.items()}
    state = d["h0"].clone()

    def step(dd):
        return gdr.recurrent_gated_delta_rule(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], initial_state=state,
                                              use_qk_l2norm_in_kernel=True, inplace=True)[0]

    for _ in range(args.warmup):
        step(d)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with Clocks(0) as clk:
        for i in range(args.steps):
            evs[i][0].record(stream)
            step(d)
            evs[i][1].record(stream)
        torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    # end to end: the step's token inputs from pinned host memory and its output back (the states stay resident)
    names = ["q", "k", "v", "g", "beta"]
    hin = {k: x[k].pin_memory() for k in names}
    hout = torch.empty(d["v"].shape, dtype=d["v"].dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in hin.values())
    d2h = hout.numel() * hout.element_size()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        dd = {k: hin[k].to(dev, non_blocking=True) for k in names}
        hout.copy_(step(dd), non_blocking=True)
    torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - t0) / args.steps
    tokens = w.B * w.T
    sbytes = w.B * w.Hv * 128 * 128 * 4
    tok_bytes = tokens * (2 * w.Hq * 128 * 2 + 2 * w.Hv * 128 * 2 + 2 * w.Hv * 2)
    algo = 2 * sbytes + tok_bytes
    hbm, _, _, src = peaks()
    achieved = algo / (ms * 1e-3) / 1e9
    line = {
        "metric": "GDN recurrent decode tokens/s (B=256 rows, T=1, H=32, K=V=128, fp32 state), 1xGB300",
        "value": round(tokens / (ms * 1e-3), 1), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "decode B=256 T=1 Hq=Hv=32 K=V=128 l2norm-in-kernel, fp32 states resident and "
                               "updated in place", "l2": "states (537 MB) larger than L2: no flush"},
        "roofline": {"kernel": "decode", "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "traffic": None, "peak_source": src,
                     "algorithmic_bytes": int(algo)},
        "e2e": {"value": round(tokens / e2e_s, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        import oracle
        pb = oracle.Problem(B=w.B, T=w.T, Hq=w.Hq, Hv=w.Hv, l2norm=True)
        heads = [0, 1]
        t0 = time.perf_counter()
        oracle.fwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"], heads=heads,
                   nthreads=oracle.max_threads())
        dt = time.perf_counter() - t0
        all_heads_s = dt * w.Hv / len(heads)  # the sample's time scaled to every head
        line["cpu_baseline"] = {"value": round(tokens / all_heads_s, 1), "unit": "tokens/s",
                                "cores": oracle.max_threads(), "kind": "oracle",
                                "sample": "all %d rows on %d of %d value heads (%.2f s); tokens/s scaled to all heads"
                                          % (w.B, len(heads), w.Hv, dt)}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="dense", choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode", action="store_true", help="time the recurrent decode instead of the training step")
    args = ap.parse_args()
    if args.decode and args.impl == "ours":
        run_decode(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
