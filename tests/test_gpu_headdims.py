"""Head dimensions below 128 on the GPU (the head-size list of the FlashQLA skill page; the chunked kernels
are built for K = V = 128 and run smaller sizes on zero-padded copies, the decode masks them) against the
fp64 oracle, which is dimension-generic."""

import pytest
import torch

import oracle
from gated_delta_rule_38_gb300.inputs import custom, make_inputs
from harness import TOL, gpu_bwd, gpu_fwd, gpu_saved, np64, oracle_problem, rel_l2, to_dev

pytestmark = pytest.mark.gpu


def check(w, kernel_l2, saved, **act):
    x = make_inputs(w, seed=50)
    d = to_dev(x)
    sv = gpu_saved(w, d, kernel_l2) if saved else None
    gcs, A, o, _, fin = gpu_fwd(w, d, kernel_l2, saved=sv)
    dq, dk, dv, db, dg, dh0 = gpu_bwd(w, d, gcs, A, kernel_l2, saved=sv)
    torch.cuda.synchronize()
    pb = oracle_problem(w, kernel_l2)
    ref = oracle.fwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"])
    gref = oracle.bwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], h0=x["h0"], dht=x["dht"])
    got = {"o": o, "final_state": fin, "dq": dq, "dk": dk, "dv": dv, "dbeta": db, "dg": dg, "dh0": dh0}
    want = {**ref, **gref}
    errs = {key: rel_l2(np64(val), want[key]) for key, val in got.items() if val is not None}
    errs["A"] = rel_l2(np64(A), oracle.wy_matrix(pb, x["k"], x["g"], x["beta"]))
    for key, e in errs.items():
        assert e <= TOL, (key, e, errs)
    assert o.shape[-1] == w.V and dq.shape[-1] == w.K


@pytest.mark.parametrize("K,V", [(64, 64), (64, 128), (128, 32), (32, 96), (8, 8)])
def test_dense_head_dims(K, V):
    check(custom(B=2, T=200, Hq=2, Hv=2, K=K, V=V, host_l2=False), True, saved=True)


def test_head_dim_64_without_saved_buffer():
    check(custom(B=1, T=150, Hq=2, Hv=2, K=64, V=64, host_l2=False), True, saved=False)


def test_head_dim_64_varlen():
    check(custom(seq_lens=(7, 0, 130, 64, 1, 65), Hq=2, Hv=2, K=64, V=64), False, saved=True)


def test_head_dims_gva_fp16_state_v_first():
    check(custom(B=2, T=150, Hq=1, Hv=4, K=64, V=96, dtype=torch.float16, host_l2=False, state_v_first=True),
          True, saved=True)


def test_head_dim_64_split_path():
    w = custom(B=1, T=500, Hq=1, Hv=2, K=64, V=64, host_l2=False)
    x = make_inputs(w, seed=51)
    d = to_dev(x)
    gcs, A, o, _, fin = gpu_fwd(w, d, True, num_segments=3)
    dq, dk, dv, db, dg, dh0 = gpu_bwd(w, d, gcs, A, True, num_segments=3)
    torch.cuda.synchronize()
    pb = oracle_problem(w, True)
    ref = oracle.fwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"])
    gref = oracle.bwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], h0=x["h0"], dht=x["dht"])
    for key, val in (("o", o), ("final_state", fin), ("dq", dq), ("dk", dk), ("dv", dv), ("dg", dg),
                     ("dbeta", db), ("dh0", dh0)):
        assert rel_l2(np64(val), (ref if key in ref else gref)[key]) <= TOL, key


@pytest.mark.parametrize("K,V", [(64, 64), (32, 96)])
def test_head_dims_split_path_saved(K, V):
    """Head dims below 128 on the intra-GPU split with the saved buffer (segments on the warp-specialised
    chains, clipped stores of o, dq, dk, dv)."""
    w = custom(B=1, T=64 * 9 + 21, Hq=1, Hv=2, K=K, V=V, host_l2=False)
    x = make_inputs(w, seed=54)
    d = to_dev(x)
    sv = gpu_saved(w, d, True, num_segments=3)
    gcs, A, o, _, fin = gpu_fwd(w, d, True, num_segments=3, saved=sv)
    dq, dk, dv, db, dg, dh0 = gpu_bwd(w, d, gcs, A, True, num_segments=3, saved=sv)
    torch.cuda.synchronize()
    pb = oracle_problem(w, True)
    ref = oracle.fwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"])
    gref = oracle.bwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], h0=x["h0"], dht=x["dht"])
    for key, val in (("o", o), ("final_state", fin), ("dq", dq), ("dk", dk), ("dv", dv), ("dg", dg),
                     ("dbeta", db), ("dh0", dh0)):
        assert rel_l2(np64(val), (ref if key in ref else gref)[key]) <= TOL, key


def test_per_chunk_states_not_offered_when_padded():
    import gated_delta_rule_38_gb300 as gdr
    w = custom(B=1, T=64, Hq=1, Hv=1, K=64, V=64)
    d = to_dev(make_inputs(w, seed=52))
    with pytest.raises(gdr.GdrError) as e:
        gdr.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], output_h=True)
    assert e.value.status == 4


@pytest.mark.parametrize("K,V,vf", [(64, 64, False), (32, 96, True), (128, 48, False)])
def test_decode_head_dims(K, V, vf):
    import gated_delta_rule_38_gb300 as gdr
    w = custom(name="decode", B=3, T=4, Hq=2, Hv=4, K=K, V=V, host_l2=False, state_v_first=vf)
    x = make_inputs(w, seed=53)
    d = to_dev(x)
    o, fin = gdr.recurrent_gated_delta_rule(d["q"], d["k"], d["v"], d["g"], d["beta"], initial_state=d["h0"],
                                            use_qk_l2norm_in_kernel=True, state_v_first=vf)
    torch.cuda.synchronize()
    ref = oracle.fwd(oracle_problem(w, True), x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"])
    assert rel_l2(np64(o), ref["o"]) <= TOL
    assert rel_l2(np64(fin), ref["final_state"]) <= TOL
