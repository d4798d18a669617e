"""Intra-GPU sequence split: a sequence cut into segments whose affine state maps are
composed on the GPU gives the oracle's results (forward and backward), for explicit
segment counts, packed batches with empty and short sequences, and the state outputs."""

import pytest
import torch

import oracle
from gated_delta_rule_38_gb300.inputs import custom, make_inputs
from harness import TOL, gpu_bwd, gpu_fwd, np64, oracle_problem, rel_l2, to_dev

pytestmark = pytest.mark.gpu


def run_split(w, kernel_l2, nseg):
    x = make_inputs(w)
    d = to_dev(x)
    gcs, A, o, h, fin = gpu_fwd(w, d, kernel_l2, num_segments=nseg, output_h=True)
    grads = gpu_bwd(w, d, gcs, A, kernel_l2, num_segments=nseg)
    torch.cuda.synchronize()
    pb = oracle_problem(w, kernel_l2)
    ref = oracle.fwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"], want_h=True)
    gref = oracle.bwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], h0=x["h0"], dht=x["dht"])
    errs = {"o": rel_l2(np64(o), ref["o"]), "h": rel_l2(np64(h)[:ref["h"].shape[0]], ref["h"])}
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


def test_split_matches_unsplit():
    w = custom(B=1, T=64 * 12, Hq=2, Hv=2, mu_g=2.0)
    x = to_dev(make_inputs(w))
    o1 = gpu_fwd(w, x, False, num_segments=1)[2]
    o4 = gpu_fwd(w, x, False, num_segments=4)[2]
    torch.cuda.synchronize()
    # the unsplit forward and the split forward are different kernels (different rounding points), each
    # within TOL of the oracle; they agree to within that same bound
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
