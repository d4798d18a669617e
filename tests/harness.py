"""Shared helpers for the parity tests: run the CUDA path and the oracle on
the same seeded inputs and compare them by relative L2 error (fp64)."""

from __future__ import annotations

import numpy as np
import torch

import oracle
from gated_delta_rule_38_gb300.inputs import Workload, make_inputs

# Acceptance bound: relative L2 error <= 8e-3 for every output and gradient
# (PR #998 test plan: fwd+bwd ratio <= 0.008).
TOL = 8e-3


def rel_l2(got, want) -> float:
    a = np.asarray(got, dtype=np.float64)
    b = np.asarray(want, dtype=np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    assert np.isfinite(a).all(), "non-finite values in the CUDA result"
    den = np.linalg.norm(b.ravel())
    return float(np.linalg.norm((a - b).ravel()) / max(den, 1e-300))


def np64(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def act_options(w: Workload) -> dict:
    """The library's activation options for a workload whose gate and beta are raw logits."""
    if not w.activations:
        return {}
    return dict(use_gate_in_kernel=True, use_beta_sigmoid_in_kernel=True, allow_neg_eigval=True)


def oracle_problem(w: Workload, kernel_l2: bool) -> oracle.Problem:
    return oracle.Problem(B=w.B, T=w.T, Hq=w.Hq, Hv=w.Hv, K=w.K, V=w.V, l2norm=kernel_l2,
                          state_v_first=w.state_v_first, cu_seqlens=w.cu_seqlens, gate_in_kernel=w.activations,
                          beta_sigmoid=w.activations, neg_eigval=w.activations)


def to_dev(x, dev="cuda"):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


_CU = {}


def cu_tensor(w: Workload, dev="cuda"):
    """The workload's cu_seqlens on the device, made once per (lengths, device) and shared (read-only): a call
    captured in a CUDA graph must not copy it from host memory."""
    if w.cu_seqlens is None:
        return None
    key = (tuple(w.cu_seqlens), str(dev))
    if key not in _CU:
        _CU[key] = torch.tensor(w.cu_seqlens, dtype=torch.int32, device=dev)
    return _CU[key]


def gpu_fwd(w: Workload, d, kernel_l2: bool, output_h=False, num_segments=0, gate_f32=False, saved=None):
    import gated_delta_rule_38_gb300 as gdr
    g, beta = d["g"], d["beta"]
    if gate_f32:
        g, beta = g.float(), beta.float()
    return gdr.chunk_gated_delta_rule_fwd(
        d["q"], d["k"], d["v"], g, beta, initial_state=d["h0"], output_final_state=w.final_state,
        cu_seqlens=cu_tensor(w), use_qk_l2norm_in_kernel=kernel_l2, state_v_first=w.state_v_first,
        num_segments=num_segments, output_h=output_h, saved=saved, **act_options(w))


def gpu_bwd(w: Workload, d, gcs, A, kernel_l2: bool, num_segments=0, gate_f32=False, saved=None):
    import gated_delta_rule_38_gb300 as gdr
    beta = d["beta"].float() if gate_f32 else d["beta"]
    return gdr.chunk_gated_delta_rule_bwd(
        d["q"], d["k"], d["v"], gcs, beta, A, d["do"], dht=d["dht"], initial_state=d["h0"],
        cu_seqlens=cu_tensor(w), use_qk_l2norm_in_kernel=kernel_l2, state_v_first=w.state_v_first,
        num_segments=num_segments, saved=saved, **act_options(w))


def gpu_saved(w: Workload, d, kernel_l2: bool, num_segments=0, gate_f32=False):
    """The forward-to-backward buffer for this workload."""
    import gated_delta_rule_38_gb300 as gdr
    g = d["g"].float() if gate_f32 else d["g"]
    return gdr.saved_buffer(d["q"], d["v"], g, cu_seqlens=cu_tensor(w), use_qk_l2norm_in_kernel=kernel_l2,
                            state_v_first=w.state_v_first, num_segments=num_segments, **act_options(w))


def train_step(w: Workload, d, nseg=0, poison=False, sync=True):
    """One forward + backward of ``w`` through the saved buffer (as the training step runs it), synchronised;
    returns copies of every output and gradient.  ``poison`` fills the fresh saved buffer with a byte pattern
    first (nothing may depend on what it held).  ``sync=False``: no synchronisation, the tensors themselves
    (still being written on the current stream)."""
    import torch
    kernel_l2 = not w.host_l2
    saved = gpu_saved(w, d, kernel_l2, num_segments=nseg)
    if poison and saved is not None:
        saved.fill_(0xA5)
    gcs, A, o, _, fin = gpu_fwd(w, d, kernel_l2, num_segments=nseg, saved=saved)
    dq, dk, dv, db, dg, dh0 = gpu_bwd(w, d, gcs, A, kernel_l2, num_segments=nseg, saved=saved)
    out = {"g_cumsum": gcs, "A": A, "o": o, "final_state": fin, "dq": dq, "dk": dk, "dv": dv, "dbeta": db,
           "dg": dg, "dh0": dh0}
    if not sync:
        return {k: v for k, v in out.items() if v is not None}
    torch.cuda.current_stream().synchronize()
    return {k: v.clone() for k, v in out.items() if v is not None}


def assert_bit_identical(first, second, what):
    import torch
    assert first.keys() == second.keys()
    for k in first:
        a, b = first[k], second[k]
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), (what, k, (a.float() - b.float()).abs().max().item())
