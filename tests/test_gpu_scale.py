"""A caller-chosen output scale (not K^-1/2) reaches every term that carries it: the output and, in the
backward, dq, dk (through the causal block's gradient), dv, dbeta, dg and dh0, against the fp64 oracle at the
same scale (whose scale handling is pinned on its own by the closed-form T = 1 tests)."""

import dataclasses

import pytest
import torch

import oracle
from gated_delta_rule_38_gb300.inputs import custom, make_inputs
from harness import TOL, cu_tensor, np64, oracle_problem, rel_l2, to_dev

pytestmark = pytest.mark.gpu

SCALE = 0.3


@pytest.mark.parametrize("name,w,saved", [
    ("dense, states", custom(name="sc_dense", B=2, T=200, Hq=2, Hv=4, host_l2=False, has_h0=True, final_state=True),
     True),
    ("dense, states, no saved buffer", custom(name="sc_dense", B=2, T=200, Hq=2, Hv=4, host_l2=False, has_h0=True,
                                              final_state=True), False),
    ("packed", custom(name="sc_varlen", Hq=2, Hv=2, seq_lens=(100, 1, 140), host_l2=False, has_h0=True,
                      final_state=True), True),
], ids=lambda x: x if isinstance(x, str) else "")
def test_custom_scale(name, w, saved):
    import gated_delta_rule_38_gb300 as gdr
    x = make_inputs(w, seed=31)
    d = to_dev(x)
    cu = cu_tensor(w)
    sv = (gdr.saved_buffer(d["q"], d["v"], d["g"], scale=SCALE, cu_seqlens=cu, use_qk_l2norm_in_kernel=True)
          if saved else None)
    gcs, A, o, _, fin = gdr.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=SCALE,
                                                       initial_state=d["h0"], output_final_state=True,
                                                       cu_seqlens=cu, use_qk_l2norm_in_kernel=True, saved=sv)
    dq, dk, dv, db, dg, dh0 = gdr.chunk_gated_delta_rule_bwd(d["q"], d["k"], d["v"], gcs, d["beta"], A, d["do"],
                                                             dht=d["dht"], scale=SCALE, initial_state=d["h0"],
                                                             cu_seqlens=cu, use_qk_l2norm_in_kernel=True, saved=sv)
    torch.cuda.synchronize()
    pb = dataclasses.replace(oracle_problem(w, True), scale=SCALE)
    ref = oracle.fwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"])
    gref = oracle.bwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], h0=x["h0"], dht=x["dht"])
    got = {"o": o, "final_state": fin, "dq": dq, "dk": dk, "dv": dv, "dbeta": db, "dg": dg, "dh0": dh0}
    want = {**ref, **gref}
    errs = {k: rel_l2(np64(v), want[k]) for k, v in got.items()}
    assert all(e <= TOL for e in errs.values()), errs
    # and the scale matters: the default scale's output differs from the oracle's at this one
    pb0 = oracle_problem(w, True)
    o0 = oracle.fwd(pb0, x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"])["o"]
    assert rel_l2(o0, ref["o"]) > 10 * TOL


def test_custom_scale_decode():
    import gated_delta_rule_38_gb300 as gdr
    w = custom(name="sc_dec", B=3, T=2, Hq=2, Hv=4, host_l2=False, has_h0=True, final_state=True)
    x = make_inputs(w, seed=32)
    d = to_dev(x)
    o, fin = gdr.recurrent_gated_delta_rule(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=SCALE,
                                            initial_state=d["h0"], use_qk_l2norm_in_kernel=True)
    torch.cuda.synchronize()
    pb = dataclasses.replace(oracle_problem(w, True), scale=SCALE)
    ref = oracle.fwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"])
    assert rel_l2(np64(o), ref["o"]) <= TOL and rel_l2(np64(fin), ref["final_state"]) <= TOL
