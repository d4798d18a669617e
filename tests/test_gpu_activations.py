"""The gate / beta activation options on the GPU (use_gate_in_kernel, use_beta_sigmoid_in_kernel and
allow_neg_eigval, the options the FlashQLA backend's verifier names in PR #998) against the fp64 oracle:
forward and backward (gradients w.r.t. the raw gate and beta), the split path, the recurrent decode and the
autograd op."""

import pytest
import torch

import oracle
from gated_delta_rule_38_gb300.inputs import custom, make_inputs
from harness import TOL, cu_tensor, np64, rel_l2, to_dev

pytestmark = pytest.mark.gpu

ALL = dict(use_gate_in_kernel=True, use_beta_sigmoid_in_kernel=True, allow_neg_eigval=True)


def raw_inputs(w, seed):
    """The workload's inputs with the gate and beta replaced by raw logits (std 2, both signs)."""
    x = make_inputs(w, seed=seed)
    gen = torch.Generator().manual_seed(seed + 1000)
    x["g"] = (2.0 * torch.randn(x["g"].shape, generator=gen)).to(w.dtype)
    x["beta"] = (2.0 * torch.randn(x["beta"].shape, generator=gen)).to(w.dtype)
    return x


def oracle_pb(w, l2, act):
    return oracle.Problem(B=w.B, T=w.T, Hq=w.Hq, Hv=w.Hv, l2norm=l2, state_v_first=w.state_v_first,
                          cu_seqlens=w.cu_seqlens, gate_in_kernel=act.get("use_gate_in_kernel", False),
                          beta_sigmoid=act.get("use_beta_sigmoid_in_kernel", False),
                          neg_eigval=act.get("allow_neg_eigval", False))


def run(w, x, l2, act, saved=True, num_segments=0, gate_f32=False):
    import gated_delta_rule_38_gb300 as gdr
    d = to_dev(x)
    g, beta = d["g"], d["beta"]
    if gate_f32:
        g, beta = g.float(), beta.float()
    cu = cu_tensor(w)
    sv = gdr.saved_buffer(d["q"], d["v"], g, cu_seqlens=cu, use_qk_l2norm_in_kernel=l2,
                          state_v_first=w.state_v_first, num_segments=num_segments, **act) if saved else None
    gcs, A, o, _, fin = gdr.chunk_gated_delta_rule_fwd(
        d["q"], d["k"], d["v"], g, beta, initial_state=d["h0"], output_final_state=w.final_state, cu_seqlens=cu,
        use_qk_l2norm_in_kernel=l2, state_v_first=w.state_v_first, num_segments=num_segments, saved=sv, **act)
    grads = gdr.chunk_gated_delta_rule_bwd(
        d["q"], d["k"], d["v"], gcs, beta, A, d["do"], dht=d["dht"], initial_state=d["h0"], cu_seqlens=cu,
        use_qk_l2norm_in_kernel=l2, state_v_first=w.state_v_first, num_segments=num_segments, saved=sv, **act)
    torch.cuda.synchronize()
    return o, fin, grads, gcs, A


def check(w, l2, act, seed, **kw):
    x = raw_inputs(w, seed)
    o, fin, (dq, dk, dv, db, dg, dh0), gcs, A = run(w, x, l2, act, **kw)
    pb = oracle_pb(w, l2, act)
    ref = oracle.fwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"])
    gref = oracle.bwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], h0=x["h0"], dht=x["dht"])
    got = {"o": o, "final_state": fin, "dq": dq, "dk": dk, "dv": dv, "dbeta": db, "dg": dg, "dh0": dh0}
    want = {**ref, **gref}
    errs = {key: rel_l2(np64(val), want[key]) for key, val in got.items() if val is not None}
    # the processed gate is the chunk-local cumsum of the activated gate
    errs["g_cumsum"] = rel_l2(np64(gcs), oracle.g_cumsum(pb, x["g"]))
    errs["A"] = rel_l2(np64(A), oracle.wy_matrix(pb, x["k"], x["g"], x["beta"]))
    for key, e in errs.items():
        assert e <= TOL, (key, e, errs)
    return errs


@pytest.mark.parametrize("T", [64, 200])
def test_all_options_dense(T):
    check(custom(B=2, T=T, Hq=2, Hv=2, host_l2=False), True, ALL, seed=31)


def test_all_options_varlen():
    check(custom(seq_lens=(7, 0, 130, 64, 1, 65), Hq=2, Hv=2), False, ALL, seed=32)


def test_all_options_gva_fp16_state_v_first():
    check(custom(B=2, T=150, Hq=1, Hv=4, dtype=torch.float16, host_l2=False, state_v_first=True), True, ALL,
          seed=33)


def test_all_options_fp32_gates():
    check(custom(B=1, T=190, Hq=2, Hv=2), False, ALL, seed=34, gate_f32=True)


@pytest.mark.parametrize("act", [dict(use_beta_sigmoid_in_kernel=True), dict(allow_neg_eigval=True),
                                 dict(use_beta_sigmoid_in_kernel=True, allow_neg_eigval=True)],
                         ids=["sigmoid", "neg_eigval", "sigmoid_neg_eigval"])
def test_beta_options_without_saved_buffer(act):
    """Without the in-kernel gate the backward needs no saved buffer."""
    w = custom(B=2, T=150, Hq=2, Hv=2, host_l2=False)
    x = raw_inputs(w, 36)
    x["g"] = torch.nn.functional.logsigmoid(x["g"].float()).to(w.dtype)   # a plain log-decay gate
    if not act.get("use_beta_sigmoid_in_kernel"):
        # beta as given (doubled): drawn in (0, 1), so the used beta spans (0, 2)
        x["beta"] = torch.sigmoid(x["beta"].float()).to(w.dtype)
    o, fin, (dq, dk, dv, db, dg, dh0), _, _ = run(w, x, True, act, saved=False)
    pb = oracle_pb(w, True, act)
    ref = oracle.fwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"])
    gref = oracle.bwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], h0=x["h0"], dht=x["dht"])
    got = {"o": o, "final_state": fin, "dq": dq, "dk": dk, "dv": dv, "dbeta": db, "dg": dg, "dh0": dh0}
    want = {**ref, **gref}
    for key, val in got.items():
        assert rel_l2(np64(val), want[key]) <= TOL, key


def test_all_options_split_path():
    """The intra-GPU sequence split with the saved buffer (the forward keeps its states for the backward)."""
    check(custom(B=1, T=700, Hq=1, Hv=2, host_l2=False), True, ALL, seed=37, num_segments=3)


def test_gate_backward_without_saved_buffer_is_refused():
    import gated_delta_rule_38_gb300 as gdr
    w = custom(B=1, T=64, Hq=1, Hv=1, host_l2=False)
    d = to_dev(raw_inputs(w, 38))
    gcs, A, _, _, _ = gdr.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                                     use_qk_l2norm_in_kernel=True, **ALL)
    with pytest.raises(gdr.GdrError) as e:
        gdr.chunk_gated_delta_rule_bwd(d["q"], d["k"], d["v"], gcs, d["beta"], A, d["do"],
                                       use_qk_l2norm_in_kernel=True, **ALL)
    assert e.value.status == 4


def test_decode_with_all_options():
    import gated_delta_rule_38_gb300 as gdr
    w = custom(name="decode", B=3, T=4, Hq=2, Hv=4, host_l2=False)
    x = raw_inputs(w, 39)
    d = to_dev(x)
    o, fin = gdr.recurrent_gated_delta_rule(d["q"], d["k"], d["v"], d["g"], d["beta"], initial_state=d["h0"],
                                            use_qk_l2norm_in_kernel=True, **ALL)
    torch.cuda.synchronize()
    ref = oracle.fwd(oracle_pb(w, True, ALL), x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"])
    assert rel_l2(np64(o), ref["o"]) <= TOL
    assert rel_l2(np64(fin), ref["final_state"]) <= TOL


def test_autograd_with_all_options():
    import gated_delta_rule_38_gb300 as gdr
    w = custom(B=1, T=130, Hq=1, Hv=2, host_l2=False)
    x = raw_inputs(w, 40)
    d = {k: (v.cuda().requires_grad_(True) if v is not None and k in ("q", "k", "v", "g", "beta", "h0") else
             (v.cuda() if v is not None else None)) for k, v in x.items()}
    o, fin = gdr.chunk_gated_delta_rule(d["q"], d["k"], d["v"], d["g"], d["beta"], initial_state=d["h0"],
                                        output_final_state=True, use_qk_l2norm_in_kernel=True, **ALL)
    (o.float() * d["do"].float()).sum().add_((fin * d["dht"]).sum()).backward()
    pb = oracle_pb(w, True, ALL)
    ref = oracle.bwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], h0=x["h0"], dht=x["dht"])
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta"), ("h0", "dh0")):
        assert rel_l2(np64(d[name].grad), ref[key]) <= TOL, name
