"""Edge cases of the recurrence on the GPU, against the fp64 oracle.

* strong decay: chunk sums of the log-gate far below -50 (a factored exp(-G) would overflow fp16) and
  reset tokens with g = -30 (exp(g) ~ 1e-13: the state is all but wiped);
* the invariant of the "Core API" recurrence that beta = 0 with g = 0 leaves the state unchanged
  (o_t = scale h0^T q_t and final_state = h0);
* state_v_first changes only the layout of the state tensors, also on the path the training step runs
  (the forward's saved buffer handed to the backward): every result bit-identical.
"""

import pytest
import torch

import oracle
from gated_delta_rule_38_gb300.inputs import custom, make_inputs
from harness import TOL, gpu_bwd, gpu_fwd, gpu_saved, np64, oracle_problem, rel_l2, to_dev

pytestmark = pytest.mark.gpu

GRADS = ("dq", "dk", "dv", "dbeta", "dg", "dh0")


def parity(w, x, kernel_l2, saved):
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
    for key, e in errs.items():
        assert e <= TOL, (key, e, errs)
    return got, errs


RESET_TOKENS = (5, 70, 130, 199)


@pytest.mark.parametrize("mu_g", [0.0, -3.0])
@pytest.mark.parametrize("saved", [False, True])
def test_strong_decay_fp16_with_resets(mu_g, saved):
    # mu_g = 0: chunk sums of g near -52; mu_g = -3: near -200.  Four tokens per head carry g = -30.
    w = custom(B=2, T=260, Hq=2, Hv=4, dtype=torch.float16, host_l2=False, mu_g=mu_g)
    x = make_inputs(w, seed=7)
    g = x["g"].clone()
    g[:, list(RESET_TOKENS), :] = -30.0
    x["g"] = g.to(w.dtype)
    parity(w, x, kernel_l2=True, saved=saved)


def test_strong_decay_varlen_bf16():
    w = custom(seq_lens=(200, 1, 64, 130), Hq=2, Hv=2, mu_g=-3.0)
    x = make_inputs(w, seed=8)
    g = x["g"].clone()
    g[:, [0, 100, 201, 300], :] = -30.0
    x["g"] = g.to(w.dtype)
    parity(w, x, kernel_l2=False, saved=True)


@pytest.mark.parametrize("saved", [False, True])
def test_zero_beta_zero_gate_keeps_the_state(saved):
    """beta = 0 and g = 0: every step is the identity on the state."""
    w = custom(B=2, T=200, Hq=2, Hv=2, host_l2=False)
    x = make_inputs(w, seed=9)
    x["g"] = torch.zeros_like(x["g"])
    x["beta"] = torch.zeros_like(x["beta"])
    got, _ = parity(w, x, kernel_l2=True, saved=saved)
    h0 = x["h0"].cuda()
    torch.testing.assert_close(got["final_state"], h0, rtol=1e-6, atol=1e-7)
    # o_t = scale h0^T q^_t: the oracle's output equals that closed form
    pb = oracle_problem(w, True)
    q = np64(x["q"])
    qn = q / (((q ** 2).sum(-1, keepdims=True) + oracle.L2_EPS) ** 0.5)
    o_closed = (128 ** -0.5) * torch.einsum("btik,bikv->btiv", torch.from_numpy(qn),
                                              torch.from_numpy(np64(x["h0"]))).numpy()
    assert rel_l2(np64(got["o"]), o_closed) <= TOL
    ref = oracle.fwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"])
    assert rel_l2(ref["o"], o_closed) < 1e-12


def test_state_v_first_bit_exact_with_saved_buffer():
    """The training step's path (the forward keeps its states and Delta, the backward runs the reverse chain
    alone): the [V,K] state layout gives bit-identical results."""
    w = custom(B=2, T=200, Hq=1, Hv=2, dtype=torch.float16, host_l2=False)
    d = to_dev(make_inputs(w, seed=10))
    sv = gpu_saved(w, d, True)
    gcs, A, o, _, fin = gpu_fwd(w, d, True, saved=sv)
    ga = gpu_bwd(w, d, gcs, A, True, saved=sv)
    wt = custom(B=2, T=200, Hq=1, Hv=2, dtype=torch.float16, host_l2=False, state_v_first=True)
    dt = dict(d)
    dt["h0"] = d["h0"].transpose(-1, -2).contiguous()
    dt["dht"] = d["dht"].transpose(-1, -2).contiguous()
    svt = gpu_saved(wt, dt, True)
    gcs_t, A_t, o_t, _, fin_t = gpu_fwd(wt, dt, True, saved=svt)
    gb = gpu_bwd(wt, dt, gcs_t, A_t, True, saved=svt)
    torch.cuda.synchronize()
    assert torch.equal(o, o_t) and torch.equal(A, A_t) and torch.equal(gcs, gcs_t)
    assert torch.equal(fin, fin_t.transpose(-1, -2))
    for a, b in zip(ga[:5], gb[:5]):
        assert torch.equal(a, b)
    assert torch.equal(ga[5], gb[5].transpose(-1, -2))


@pytest.mark.parametrize("packed", [False, True])
@pytest.mark.parametrize("saved", [False, True])
def test_no_tokens_at_all(packed, saved):
    """A call with no tokens (a dense batch with T = 0, or a packed batch whose every sequence is empty) runs
    no recurrence step: the final states are the initial ones and dh0 is dht, bit for bit."""
    import gated_delta_rule_38_gb300 as gdr
    H, D, N = 2, 128, 3
    B = 1 if packed else N
    gen = torch.Generator(device="cuda").manual_seed(11)
    q = torch.zeros(B, 0, H, D, dtype=torch.bfloat16, device="cuda")
    g = torch.zeros(B, 0, H, dtype=torch.bfloat16, device="cuda")
    h0 = torch.randn(N, H, D, D, device="cuda", generator=gen)
    dht = torch.randn(N, H, D, D, device="cuda", generator=gen)
    cu = torch.zeros(N + 1, dtype=torch.int32, device="cuda") if packed else None
    sv = gdr.saved_buffer(q, q, g, cu_seqlens=cu) if saved else None
    gcs, A, o, _, fin = gdr.chunk_gated_delta_rule_fwd(q, q, q, g, g, initial_state=h0, output_final_state=True,
                                                       cu_seqlens=cu, saved=sv)
    assert o.numel() == 0 and torch.equal(fin, h0)
    dq, dk, dv, db, dg, dh0 = gdr.chunk_gated_delta_rule_bwd(q, q, q, gcs, g, A, q, dht=dht, initial_state=h0,
                                                             cu_seqlens=cu, saved=sv)
    torch.cuda.synchronize()
    assert gdr.get_error() == 0
    assert dq.numel() == 0 and dg.numel() == 0 and torch.equal(dh0, dht)


@pytest.mark.parametrize("packed", [False, True])
@pytest.mark.parametrize("saved", [False, True])
def test_infinite_gate_is_a_hard_reset(packed, saved):
    """A log-gate of -inf at some tokens (e^g = 0: the state is wiped there, a hard reset) against the oracle,
    which applies the token recurrence literally; the chunk form, which subtracts cumulative gates, takes such
    gates at its floor, whose factor is already zero at fp32 resolution."""
    if packed:
        w = custom(name="neginf_v", Hq=2, Hv=2, seq_lens=(150, 70, 1), host_l2=False, has_h0=True,
                   final_state=True)
    else:
        w = custom(name="neginf", B=2, T=200, Hq=2, Hv=2, host_l2=False, has_h0=True, final_state=True)
    x = make_inputs(w, seed=13)
    g = x["g"].clone()
    g[0, 0] = float("-inf")  # the first token of one sequence only: a reference dh0 of all zeros has no scale
    for t in (37, 64, 65, 130, 151):  # inside chunks, a chunk's first token, inside a later sequence
        if t < g.shape[1]:
            g[:, t] = float("-inf")
    x["g"] = g
    got, errs = parity(w, x, kernel_l2=True, saved=saved)
    assert all(torch.isfinite(v).all() for v in got.values() if v is not None)
