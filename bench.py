"""Benchmark of the chunked gated delta rule forward + backward on GB300.

One step = one training pass of the whole hot path over one batch: the
forward (gate cumsum, WY matrix, state recurrence and output, saving g_cumsum
and A, and handing its states to the backward) followed by the backward
(reverse state-gradient chain, per-chunk gradients), on synthetic seeded
inputs of the dense prefill workload B=2, T=4096, H_q=H_v=32, K=V=128, bf16,
q/k L2-normalised in the kernels.

Prints one JSON line: the headline (tokens/s of exactly --steps timed steps),
each direction's time, throughput and roofline fraction (inference forward,
training forward, backward), the same per direction for the varlen, GVA,
long, activated-gate and head-dimension-64 workloads, per-kernel times, the end-to-end figure through host memory,
the clocks under load and the fp64 oracle on the host cores.
--impl reference times the oracle alone (a bounded sample of the workload).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
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
C = 64
L2_BYTES = 129 * 2 ** 20
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic_dense_B2_T4096_H32.json")
WORKLOAD_TEXT = {
    "dense": "dense prefill B=2 T=4096 Hq=32 Hv=32 K=V=128 l2norm-in-kernel",
    "varlen": "varlen packed T=5311 lengths [512,1024,768,3000,7] H=32 K=V=128, initial and final states",
    "gva": "GVA B=4 T=8192 Hq=16 Hv=32 K=V=128 fp16, initial and final states",
    "long": "long single sequence B=1 T=65536 H=16 K=V=128, slow decay, intra-GPU sequence split",
    "tiny": "tiny B=1 T=256 H=2 K=V=128",
    "dense_act": "dense prefill B=2 T=4096 H=32 K=V=128 l2norm-in-kernel, raw gate and beta logits activated in "
                 "the kernels (logsigmoid gate, sigmoid beta, negative eigenvalues allowed)",
    "dense_hd64": "dense prefill B=2 T=4096 H=32 K=V=64 l2norm-in-kernel (run zero-padded to 128 in the chunked "
                  "kernels; bytes and FLOPs counted at 64)",
}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def work(w):
    """Algorithmic FLOPs and bytes of each direction of one pass over workload ``w``.

    FLOPs per token and value head (multiply-add = 2, C = 64, the workload's K and V): forward Hq/Hv * 4CK + 2C(K+2V) +
    6KV; backward twice the forward plus 4C^2.  Bytes: every tensor the direction must read or write once --
    forward-only (inference): q, k, v, g, beta in, o out (and the initial / final states when used); the
    training forward adds A (input dtype) and g_cumsum (fp32) out; the backward reads q, k, v, g_cumsum, beta,
    A, do (and h0, dht) and writes dq, dk, dv, dg, dbeta (and dh0).
    """
    K, V = w.K, w.V
    tok = w.tokens
    e = 2
    fwd_f = tok * (w.Hq * 4 * C * K + w.Hv * (2 * C * (K + 2 * V) + 6 * K * V))
    bwd_f = 2 * fwd_f + tok * w.Hv * 4 * C * C
    N = w.num_seqs
    st = N * w.Hv * K * V * 4
    qk = 2 * tok * w.Hq * K * e
    vv = tok * w.Hv * V * e
    gb = 2 * tok * w.Hv * e
    fwd_only_b = qk + vv + gb + vv + (st if w.has_h0 else 0) + (st if w.final_state else 0)
    train_fwd_b = fwd_only_b + tok * w.Hv * (C * e + 4)
    bwd_b = qk + vv + tok * w.Hv * (4 + e + C * e) + vv + qk + vv + gb
    if w.has_h0:
        bwd_b += 2 * st
    if w.final_state:
        bwd_b += st
    return {"fwd_flops": fwd_f, "fwd_only_bytes": fwd_only_b, "train_fwd_bytes": train_fwd_b, "bwd_flops": bwd_f,
            "bwd_bytes": bwd_b, "parts": {"qk": qk, "v": vv, "gates": gb, "A_gcs": tok * w.Hv * (C * e + 4),
                                          "gcs_beta_A": tok * w.Hv * (4 + e + C * e), "state": st}}


def kernel_bytes(name, w, wk):
    """Algorithmic bytes of one launch of a kernel: the tensors of the direction's list that the kernel
    itself must read or write (intermediates it exchanges with another kernel are not counted)."""
    p = wk["parts"]
    st_in = p["state"] if w.has_h0 else 0
    st_out = p["state"] if w.final_state else 0
    table = {
        # q, k, g, beta in; A and g_cumsum out
        "wy_fwd": p["qk"] + p["gates"] + p["A_gcs"],
        # q, k, v, beta, g_cumsum, A in; o out (initial / final states)
        "chain_fwd": p["qk"] + 2 * p["v"] + p["gcs_beta_A"] + st_in + st_out,
        # q, k, do, g_cumsum, beta, A in (dht in, dh0 out)
        "chain_rev": p["qk"] + p["v"] + p["gcs_beta_A"] + st_out + (p["state"] if w.has_h0 else 0),
        # every input of the backward in, every gradient out
        "bwd_chunk": wk["bwd_bytes"],
    }
    return table.get(name)


def recorded_traffic(name):
    """DRAM bytes (read + write) of one launch of a kernel on the dense workload, from the committed ncu
    record, or None when the record is missing or the kernel's sources changed since it was taken."""
    import hashlib
    try:
        rec = json.load(open(TRAFFIC_FILE))["kernels"][name]
    except Exception:
        return None
    h = hashlib.sha256()
    for f in rec["sources"]:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return float(rec["dram_bytes"]) if h.hexdigest()[:16] == rec["sources_sha16"] else None


def direction_report(ms, flops, nbytes, tokens, hbm, tflops, median_ms=None):
    """Throughput and roofline fraction of one direction from its mean time (roofline = the slower of bytes at
    HBM bandwidth and FLOPs at dense bf16 tensor peak); the median time beside it when given."""
    rl_us = max(nbytes / (hbm * 1e9), flops / (tflops * 1e12)) * 1e6
    extra = {} if median_ms is None else {"us_median": round(median_ms * 1e3, 2)}
    return {"us": round(ms * 1e3, 2), **extra, "tokens_per_s": round(tokens / (ms * 1e-3), 1),
            "tflops": round(flops / (ms * 1e-3) / 1e12, 2), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
            "roofline_us": round(rl_us, 2), "roofline_frac": round(rl_us / (ms * 1e3), 4),
            "algorithmic_bytes": int(nbytes), "algorithmic_flops": int(flops)}


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

    def __init__(self, index=0, interval_ms=50):
        self.index = index
        self.interval_ms = interval_ms
        self.rows = []
        self.proc = None

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + q,
                                          "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
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


def _inputs_on(w, seed, dev):
    x = make_inputs(w, seed=seed)
    d = {k: (v.to(dev) if v is not None else None) for k, v in x.items()}
    cu = None if w.cu_seqlens is None else torch.tensor(w.cu_seqlens, dtype=torch.int32, device=dev)
    return x, d, cu


def act_options(w):
    """The library's activation options for a workload whose gate and beta are raw logits."""
    if not w.activations:
        return {}
    return dict(use_gate_in_kernel=True, use_beta_sigmoid_in_kernel=True, allow_neg_eigval=True)


def saved_for(gdr, w, d, cu):
    """The forward-to-backward buffer of workload ``w`` (reused by every step)."""
    return gdr.saved_buffer(d["q"], d["v"], d["g"], cu_seqlens=cu, use_qk_l2norm_in_kernel=not w.host_l2,
                            **act_options(w))


def _make_step(gdr, w, cu, saved):
    l2 = not w.host_l2
    act = act_options(w)

    def fwd(dd, save=True):
        if not save:
            return gdr.chunk_gated_delta_rule_fwd(
                dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], initial_state=dd["h0"],
                output_final_state=w.final_state, cu_seqlens=cu, use_qk_l2norm_in_kernel=l2,
                save_for_backward=False, **act)
        return gdr.chunk_gated_delta_rule_fwd(
            dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], initial_state=dd["h0"],
            output_final_state=w.final_state, cu_seqlens=cu, use_qk_l2norm_in_kernel=l2, saved=saved, **act)

    def bwd(dd, f):
        gcs, A = f[0], f[1]
        return gdr.chunk_gated_delta_rule_bwd(
            dd["q"], dd["k"], dd["v"], gcs, dd["beta"], A, dd["do"], dht=dd["dht"], initial_state=dd["h0"],
            cu_seqlens=cu, use_qk_l2norm_in_kernel=l2, saved=saved, **act)

    def step(dd):
        f = fwd(dd)
        return f[2], bwd(dd, f)

    return fwd, bwd, step


def _direction_times(fwd, bwd, d, steps, flush, stream):
    """Mean device ms of the training forward, the backward, and an inference forward (no saving), each step
    timed with CUDA events on the launching stream and the L2 flushed before it; and their medians (a dict)."""
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        ev[i][0].record(stream)
        f = fwd(d)
        ev[i][1].record(stream)
        bwd(d, f)
        ev[i][2].record(stream)
    inf = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        inf[i][0].record(stream)
        fwd(d, save=False)
        inf[i][1].record(stream)
    torch.cuda.synchronize()
    f_ms = [e[0].elapsed_time(e[1]) for e in ev]
    b_ms = [e[1].elapsed_time(e[2]) for e in ev]
    i_ms = [a.elapsed_time(b) for a, b in inf]
    fb_ms = [x + y for x, y in zip(f_ms, b_ms)]
    med = {"train_fwd": statistics.median(f_ms), "bwd": statistics.median(b_ms), "fwd_only": statistics.median(i_ms),
           "fwd_bwd": statistics.median(fb_ms)}
    return sum(f_ms) / steps, sum(b_ms) / steps, sum(i_ms) / steps, med


def _directions(w, tf, tb, ti, hbm, tflops, med=None):
    wk = work(w)
    med = med or {}
    return {
        "fwd_only": direction_report(ti, wk["fwd_flops"], wk["fwd_only_bytes"], w.tokens, hbm, tflops,
                                     med.get("fwd_only")),
        "train_fwd": direction_report(tf, wk["fwd_flops"], wk["train_fwd_bytes"], w.tokens, hbm, tflops,
                                      med.get("train_fwd")),
        "bwd": direction_report(tb, wk["bwd_flops"], wk["bwd_bytes"], w.tokens, hbm, tflops, med.get("bwd")),
        "fwd_bwd": direction_report(tf + tb, wk["fwd_flops"] + wk["bwd_flops"],
                                    wk["train_fwd_bytes"] + wk["bwd_bytes"], w.tokens, hbm, tflops, med.get("fwd_bwd")),
    }


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
    dev = torch.device("cuda", local)
    x, d, cu = _inputs_on(w, rank_seed(rank), dev)  # every rank: its own batch (weak scaling, no collective)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    # the forward hands P, the q/k norms, its states and Delta to the backward (one buffer, reused by the steps)
    saved = saved_for(gdr, w, d, cu)
    fwd, bwd, step = _make_step(gdr, w, cu, saved)
    hbm, tf_burst, tf_sus, src = peaks()

    for _ in range(args.warmup):
        step(d)
    torch.cuda.synchronize()

    # ---- the headline: exactly K training steps, device time per step from CUDA events on the launching
    # stream, the L2 flushed between steps (outside the events).  The clock sampler runs from a loaded
    # stretch of steps just before the timed ones until they end, so it sees the GPU under this load.
    stream = torch.cuda.current_stream(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with Clocks(local) as clk:
        t_load = time.perf_counter()
        n_load = 0
        while time.perf_counter() - t_load < args.load_seconds:
            for _ in range(20):
                flush.zero_()
                step(d)
            n_load += 20
            torch.cuda.synchronize()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.zero_()
            evs[i][0].record(stream)
            step(d)
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
    ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in evs) / args.steps, dist, dev)

    # ---- per direction (events between the forward and the backward), and the inference forward
    tf, tb, ti, med = _direction_times(fwd, bwd, d, args.steps, flush, stream)
    tf, tb, ti = (max_over_ranks(t, dist, dev) for t in (tf, tb, ti))

    # ---- per kernel: the library's own event pairs around each launch, in a pass of its own
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

    wk = work(w)
    tokens = w.tokens * world
    value = job_throughput(w.tokens, world, ms * 1e-3)
    directions = _directions(w, tf, tb, ti, hbm, tf_sus, med if world == 1 else None)
    # dominant kernel by measured time share; its algorithmic bytes are the direction's tensors it must move
    tot = sum(v[1] for v in prof.values()) or 1.0
    name, (cnt, kms) = max(prof.items(), key=lambda kv: kv[1][1])
    per_launch_ms = kms / cnt
    kb = kernel_bytes(name, w, wk)
    roofline = {"kernel": name, "bound": "hbm", "achieved": None, "peak": hbm, "unit": "GB/s", "frac": None,
                "traffic": recorded_traffic(name) if args.workload == "dense" else None,
                "peak_source": src, "share": round(kms / tot, 3), "algorithmic_bytes": kb,
                "launch_ms": round(per_launch_ms, 4)}
    if kb:
        achieved = kb / (per_launch_ms * 1e-3) / 1e9
        roofline["achieved"] = round(achieved, 1)
        roofline["frac"] = round(achieved / hbm, 4)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == torch.bfloat16 else "fp16", "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT.get(args.workload, args.workload),
                   "B": w.B, "T": w.T, "Hq": w.Hq, "Hv": w.Hv, "K": w.K, "V": w.V, "chunk": C,
                   "l2": "flushed between steps (256 MiB write outside the timed events)", "parallelism": "replicas"},
        "tflops": round((wk["fwd_flops"] + wk["bwd_flops"]) / (ms * 1e-3) / 1e12, 2),
        "directions": directions,
        "kernels_ms_per_step": {k: round(v[1] / args.steps, 4) for k, v in prof.items()},
        "roofline": roofline,
        "e2e": {"value": round(tokens / e2e_s, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": int(sum(v[0] for v in prof.values())),
        "clocks": dict(clk.summary(), load_steps_before_timed=n_load),
    }
    # the other workloads, each direction on its own (one GPU only: the per-workload report is a 1-GPU one)
    if world == 1 and not args.headline_only:
        del saved, bufs, hout
        configs = {}
        for other in ("varlen", "gva", "long", "dense_act", "dense_hd64"):
            if other == args.workload:
                continue
            wo = WORKLOADS[other]
            xo, do_, cuo = _inputs_on(wo, 42, dev)
            svo = saved_for(gdr, wo, do_, cuo)
            fo, bo, so = _make_step(gdr, wo, cuo, svo)
            for _ in range(max(3, args.warmup)):
                so(do_)
            torch.cuda.synchronize()
            n = max(3, min(args.steps, 50))
            a, b, c, mo = _direction_times(fo, bo, do_, n, flush, stream)
            _lib.profile_enable(True)
            so(do_)
            torch.cuda.synchronize()
            _lib.profile_enable(False)
            kp = _lib.profile_read()
            configs[other] = {"workload": WORKLOAD_TEXT[other], "steps": n,
                              "directions": _directions(wo, a, b, c, hbm, tf_sus, mo),
                              "kernels_ms": {k: round(v[1], 4) for k, v in kp.items()}}
            del xo, do_, cuo, svo, fo, bo, so
            torch.cuda.empty_cache()
        line["configs"] = configs
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def _oracle_sample(w, x, nh, nthreads):
    """fwd + bwd of the oracle over every token of ``w`` on its first ``nh`` value heads; returns seconds."""
    import oracle
    pb = oracle.Problem(B=w.B, T=w.T, Hq=w.Hq, Hv=w.Hv, K=w.K, V=w.V, l2norm=not w.host_l2,
                        state_v_first=w.state_v_first, cu_seqlens=w.cu_seqlens, gate_in_kernel=w.activations,
                        beta_sigmoid=w.activations, neg_eigval=w.activations)
    heads = list(range(nh))
    t0 = time.perf_counter()
    oracle.fwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"], heads=heads, nthreads=nthreads)
    oracle.bwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], h0=x["h0"], dht=x["dht"], heads=heads,
               nthreads=nthreads)
    return time.perf_counter() - t0


def _first_heads(w, nthreads):
    """Fewest value heads whose (sequence, head) pairs keep every oracle thread busy (it parallelises over
    those pairs)."""
    return min(w.Hv, max(1, -(-nthreads // max(1, w.num_seqs))))


def cpu_baseline(w, budget_s):
    """The fp64 oracle on a bounded sample of the workload (every token, a subset of the value heads large
    enough to occupy every thread), grown while it stays inside the budget."""
    import oracle
    nthreads = oracle.max_threads()
    x = make_inputs(w)
    nh = _first_heads(w, nthreads)
    dt = _oracle_sample(w, x, nh, nthreads)
    while dt * 2.2 < budget_s and nh * 2 <= w.Hv:
        nh *= 2
        dt = _oracle_sample(w, x, nh, nthreads)
    return {"value": round(w.tokens * nh / w.Hv / dt, 1), "unit": "tokens/s", "cores": nthreads,
            "host_cpus": os.cpu_count(), "kind": "oracle",
            "sample": "fwd+bwd of all %d tokens on %d of %d value heads (%.2f s, %d threads); tokens/s scaled to "
                      "all heads" % (w.tokens, nh, w.Hv, dt, nthreads)}


def run_reference(args):
    """The oracle as the reference arm: fp64 CPU on the host cores, rank 0 only.  Each step is a timed sample
    of the workload: fwd + bwd of every token on as many value heads as keep every oracle thread busy."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    w = WORKLOADS[args.workload]
    nthreads = oracle.max_threads()
    x = make_inputs(w)
    nh = _first_heads(w, nthreads)
    times = []
    for i in range(args.warmup + args.steps):
        dt = _oracle_sample(w, x, nh, nthreads)
        if i >= args.warmup:
            times.append(dt)
    t = sum(times) / len(times)
    v = w.tokens * nh / w.Hv / t
    sample = ("each step: fwd+bwd of all %d tokens on %d of %d value heads (%d threads, %d host CPUs); "
              "tokens/s scaled to all heads" % (w.tokens, nh, w.Hv, nthreads, os.cpu_count()))
    line = {"metric": METRIC, "impl": "reference", "value": round(v, 1), "unit": "tokens/s",
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD_TEXT.get(args.workload, args.workload),
                       "step": "a timed sample: %d of %d value heads" % (nh, w.Hv)},
            "cpu_baseline": {"value": round(v, 1), "unit": "tokens/s", "kind": "oracle", "cores": nthreads,
                             "host_cpus": os.cpu_count(), "sample": sample},
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
    ap.add_argument("--load-seconds", type=float, default=1.0,
                    help="loaded stretch of steps before the timed ones, inside the clock sampler's window")
    ap.add_argument("--headline-only", action="store_true", help="skip the per-workload direction report")
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
