"""Intra-GPU sequence split: a sequence cut into segments whose affine state maps are
composed on the GPU gives the oracle's results (forward and backward), for explicit
segment counts, packed batches with empty and short sequences, and the state outputs."""

import pytest
import torch

import oracle
from gated_delta_rule_38_gb300.inputs import custom, make_inputs
from harness import TOL, gpu_bwd, gpu_fwd, gpu_saved, np64, oracle_problem, rel_l2, to_dev

pytestmark = pytest.mark.gpu


def run_split(w, kernel_l2, nseg, saved=False):
    """Forward and backward with nseg segments per sequence; without the saved buffer the forward also
    returns the per-chunk states (checked) and the backward recomputes them, with it the backward runs the
    reverse segment passes on the forward's states."""
    x = make_inputs(w)
    d = to_dev(x)
    sv = gpu_saved(w, d, kernel_l2, num_segments=nseg) if saved else None
    gcs, A, o, h, fin = gpu_fwd(w, d, kernel_l2, num_segments=nseg, output_h=not saved, saved=sv)
    grads = gpu_bwd(w, d, gcs, A, kernel_l2, num_segments=nseg, saved=sv)
    torch.cuda.synchronize()
    pb = oracle_problem(w, kernel_l2)
    ref = oracle.fwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"], want_h=not saved)
    gref = oracle.bwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], h0=x["h0"], dht=x["dht"])
    errs = {"o": rel_l2(np64(o), ref["o"])}
    if not saved:
        errs["h"] = rel_l2(np64(h[:ref["h"].shape[0]]), ref["h"])
    if w.final_state:
        errs["final_state"] = rel_l2(np64(fin), ref["final_state"])
    for key, val in zip(("dq", "dk", "dv", "dbeta", "dg", "dh0"), grads):
        if val is None:
            continue
        errs[key] = rel_l2(np64(val), gref[key])
    for key, e in errs.items():
        assert e <= TOL, (key, e, errs)
    return o, grads


@pytest.mark.parametrize("nseg", [2, 3, 7])
def test_dense_segments(nseg):
    w = custom(B=1, T=64 * 20 + 17, Hq=1, Hv=2, host_l2=False, mu_g=2.0)
    run_split(w, True, nseg)


def test_varlen_segments():
    w = custom(seq_lens=(700, 0, 130, 5, 64), Hq=2, Hv=2, mu_g=1.0)
    run_split(w, False, 4)


@pytest.mark.parametrize("nseg", [2, 3, 7])
def test_dense_segments_saved(nseg):
    w = custom(B=1, T=64 * 20 + 17, Hq=1, Hv=2, host_l2=False, mu_g=2.0)
    run_split(w, True, nseg, saved=True)


def test_varlen_segments_saved():
    """Segments of a packed batch with empty, one-chunk and ragged sequences (segments past a short
    sequence's end are empty), through the saved buffer."""
    w = custom(seq_lens=(700, 0, 130, 5, 64), Hq=2, Hv=2, mu_g=1.0)
    run_split(w, False, 4, saved=True)


def test_segments_saved_gva_fp16_state_v_first():
    w = custom(B=2, T=64 * 7 + 30, Hq=1, Hv=2, dtype=torch.float16, host_l2=False, state_v_first=True)
    run_split(w, True, 3, saved=True)


def test_split_matches_unsplit():
    w = custom(B=1, T=64 * 12, Hq=2, Hv=2, mu_g=2.0)
    x = to_dev(make_inputs(w))
    o1 = gpu_fwd(w, x, False, num_segments=1)[2]
    o4 = gpu_fwd(w, x, False, num_segments=4)[2]
    torch.cuda.synchronize()
    # the split forward starts its segments from states composed of the segment-affine passes (other kernels,
    # other rounding points than the unsplit running state), each within TOL of the oracle; they agree to
    # within that same bound
    assert rel_l2(np64(o4), np64(o1)) < TOL


def test_split_state_v_first_bit_exact():
    w = custom(B=1, T=64 * 9 + 3, Hq=1, Hv=1, dtype=torch.float16)
    x = to_dev(make_inputs(w))
    a = gpu_fwd(w, x, False, num_segments=3, output_h=True)
    wt = custom(B=1, T=64 * 9 + 3, Hq=1, Hv=1, dtype=torch.float16, state_v_first=True)
    xt = dict(x)
    xt["h0"] = x["h0"].transpose(-1, -2).contiguous()
    b = gpu_fwd(wt, xt, False, num_segments=3, output_h=True)
    torch.cuda.synchronize()
    assert torch.equal(a[2], b[2])
    assert torch.equal(a[4], b[4].transpose(-1, -2))
