"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test fixes the oracle to something the pages or the mathematics decide:
finite differences (the backward against the forward), the single-token
closed form written in the state-first orientation of the stated recurrence
S_t = e^{g_t} S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T, invariants
(beta = 0 with g = 0 keeps the state; g = -inf resets it), the delta rule's
textbook behaviour on orthonormal keys, structural equalities (continuation,
varlen = separate calls, grouped heads = repeated heads), the chunked
identities that the GPU path uses, and the chunk-table example printed on
the FlashQLA documentation page.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import Problem

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(rng, *shape):
    return rng.standard_normal(shape)


def small_inputs(rng, pb: Problem, g_scale=1.0, with_h0=True):
    Tt = pb.total_tokens
    lead = (pb.B, pb.T) if pb.cu_seqlens is None else (1, Tt)
    q = rnd(rng, *lead, pb.Hq, pb.K)
    k = rnd(rng, *lead, pb.Hq, pb.K)
    if not pb.l2norm:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rnd(rng, *lead, pb.Hv, pb.V)
    g = -np.log1p(np.exp(-rnd(rng, *lead, pb.Hv))) * g_scale
    beta = 1.0 / (1.0 + np.exp(-rnd(rng, *lead, pb.Hv)))
    sshape = (pb.num_seqs, pb.Hv, pb.V, pb.K) if pb.state_v_first else (pb.num_seqs, pb.Hv, pb.K, pb.V)
    h0 = 0.3 * rnd(rng, *sshape) if with_h0 else None
    return dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0)


# ---------------------------------------------------------------- chunk tables

def test_prepare_lens_golden():
    gold = json.load(open(os.path.join(GOLDEN, "prepare_lens.json")))
    assert oracle.prepare_lens(gold["cu_seqlens"]) == gold["lens"]


def test_chunk_tables_golden():
    gold = json.load(open(os.path.join(GOLDEN, "chunk_tables.json")))
    for case in gold["cases"]:
        offs, tot = oracle.prepare_chunk_offsets(case["cu_seqlens"], case["chunk_size"])
        assert offs == case["chunk_offsets"]
        assert tot == case["total_chunks"]
        idx = oracle.prepare_chunk_indices(case["cu_seqlens"], case["chunk_size"])
        assert len(idx) == tot
        if "chunk_indices" in case:
            assert idx == case["chunk_indices"]


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("vf", [False, True])
def test_single_token_closed_form(vf):
    """T = 1: S_1 = e^g S_0 (I - b k k^T) + b v k^T and o = scale S_1 q (S = state^T)."""
    rng = np.random.default_rng(1)
    K, V = 6, 5
    pb = Problem(B=1, T=1, Hq=1, Hv=1, K=K, V=V, scale=0.37, state_v_first=vf)
    q = rnd(rng, K); k = rnd(rng, K); k /= np.linalg.norm(k); v = rnd(rng, V)
    g, b = -0.4, 0.7
    S0 = rnd(rng, V, K)                       # value-by-key state
    S1 = math.exp(g) * S0 @ (np.eye(K) - b * np.outer(k, k)) + b * np.outer(v, k)
    o_ref = pb.scale * S1 @ q
    h0 = S0 if vf else S0.T.copy()
    out = oracle.fwd(pb, q.reshape(1, 1, 1, K), k.reshape(1, 1, 1, K), v.reshape(1, 1, 1, V),
                     np.full((1, 1, 1), g), np.full((1, 1, 1), b), h0=h0.reshape((1, 1) + h0.shape))
    np.testing.assert_allclose(out["o"].reshape(V), o_ref, rtol=1e-13, atol=1e-13)
    fin = out["final_state"].reshape(h0.shape)
    np.testing.assert_allclose(fin, S1 if vf else S1.T, rtol=1e-13, atol=1e-13)


def test_single_token_closed_form_gradients():
    """T = 1 gradients, derived by hand from S_1 = e^g S_0 (I - b k k^T) + b v k^T, o = c S_1 q."""
    rng = np.random.default_rng(2)
    K, V = 5, 4
    c = 0.5
    pb = Problem(B=1, T=1, Hq=1, Hv=1, K=K, V=V, scale=c, state_v_first=True)
    q = rnd(rng, K); k = rnd(rng, K); v = rnd(rng, V)
    g, b = -0.3, 0.6
    a = math.exp(g)
    S0 = rnd(rng, V, K)
    dO = rnd(rng, V)
    dS1 = rnd(rng, V, K)                      # gradient arriving at the final state
    S1 = a * S0 @ (np.eye(K) - b * np.outer(k, k)) + b * np.outer(v, k)
    G = dS1 + c * np.outer(dO, q)             # total gradient w.r.t. S_1
    dq = c * S1.T @ dO
    dS0 = a * G @ (np.eye(K) - b * np.outer(k, k))
    dv = b * G @ k
    dbeta = float(np.sum(G * (np.outer(v, k) - a * S0 @ np.outer(k, k))))
    dg = float(np.sum(G * (a * S0 @ (np.eye(K) - b * np.outer(k, k)))))
    # d/dk of -a b S0 k k^T + b v k^T:  -a b (S0^T G k + G^T S0 k) + b G^T v
    dk = -a * b * (S0.T @ G @ k + G.T @ S0 @ k) + b * G.T @ v
    res = oracle.bwd(pb, q.reshape(1, 1, 1, K), k.reshape(1, 1, 1, K), v.reshape(1, 1, 1, V),
                     np.full((1, 1, 1), g), np.full((1, 1, 1), b), dO.reshape(1, 1, 1, V),
                     h0=S0.reshape(1, 1, V, K), dht=dS1.reshape(1, 1, V, K))
    np.testing.assert_allclose(res["dq"].reshape(K), dq, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(res["dk"].reshape(K), dk, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(res["dv"].reshape(V), dv, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(res["dbeta"].item(), dbeta, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(res["dg"].item(), dg, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(res["dh0"].reshape(V, K), dS0, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- invariants

def test_zero_beta_zero_gate_keeps_state():
    rng = np.random.default_rng(3)
    pb = Problem(B=1, T=7, Hq=1, Hv=1, K=8, V=6, scale=0.9)
    x = small_inputs(rng, pb)
    x["beta"][:] = 0.0
    x["g"][:] = 0.0
    out = oracle.fwd(pb, **x)
    assert np.array_equal(out["final_state"], x["h0"])
    h0 = x["h0"][0, 0]
    o_ref = pb.scale * np.einsum("kv,tk->tv", h0, x["q"][0, :, 0])
    np.testing.assert_allclose(out["o"][0, :, 0], o_ref, rtol=1e-14, atol=1e-14)


def test_minus_infinity_gate_resets_state():
    rng = np.random.default_rng(4)
    pb = Problem(B=1, T=9, Hq=1, Hv=1, K=8, V=6, l2norm=True)
    x = small_inputs(rng, pb)
    x["g"][0, 4, 0] = -np.inf
    a = oracle.fwd(pb, **x)
    x2 = dict(x)
    x2["h0"] = 100.0 * x["h0"]                      # any start state
    b = oracle.fwd(pb, **x2)
    # outputs from the reset token on do not depend on the start state
    np.testing.assert_allclose(a["o"][0, 4:], b["o"][0, 4:], rtol=1e-13, atol=1e-13)
    assert not np.allclose(a["o"][0, :4], b["o"][0, :4])
    # a reset at the last token leaves beta k v^T
    x3 = dict(x)
    x3["g"] = x["g"].copy()
    x3["g"][0, -1, 0] = -np.inf
    c = oracle.fwd(pb, **x3)
    kk = x["k"][0, -1, 0]
    kk = kk / np.sqrt(kk @ kk + oracle.L2_EPS)
    ref = x["beta"][0, -1, 0] * np.outer(kk, x["v"][0, -1, 0])
    np.testing.assert_allclose(c["final_state"][0, 0], ref, rtol=1e-13, atol=1e-15)


def test_orthonormal_keys_overwrite_rows():
    """g = 0, beta = 1, k_t = e_t: the delta rule replaces row t of the [K,V] state by v_t."""
    rng = np.random.default_rng(5)
    K, V, T = 8, 5, 6
    pb = Problem(B=1, T=T, Hq=1, Hv=1, K=K, V=V, scale=1.0)
    q = rnd(rng, 1, T, 1, K)
    k = np.zeros((1, T, 1, K))
    for t in range(T):
        k[0, t, 0, t] = 1.0
    v = rnd(rng, 1, T, 1, V)
    h0 = rnd(rng, 1, 1, K, V)
    out = oracle.fwd(pb, q, k, v, np.zeros((1, T, 1)), np.ones((1, T, 1)), h0=h0)
    for t in range(T):
        h = h0[0, 0].copy()
        h[: t + 1] = v[0, : t + 1, 0]
        np.testing.assert_allclose(out["o"][0, t, 0], h.T @ q[0, t, 0], rtol=1e-14, atol=1e-14)
    h = h0[0, 0].copy()
    h[:T] = v[0, :, 0]
    np.testing.assert_allclose(out["final_state"][0, 0], h, rtol=0, atol=1e-14)


def test_state_v_first_is_exact_transpose():
    rng = np.random.default_rng(6)
    pb = Problem(B=2, T=11, Hq=1, Hv=2, K=6, V=5, l2norm=True, chunk=4)
    x = small_inputs(rng, pb)
    dO = rnd(rng, 2, 11, 2, 5)
    dht = rnd(rng, 2, 2, 6, 5)
    a = oracle.fwd(pb, **x, want_h=True)
    ga = oracle.bwd(pb, **x, do=dO, dht=dht)
    pbt = Problem(B=2, T=11, Hq=1, Hv=2, K=6, V=5, l2norm=True, chunk=4, state_v_first=True)
    xt = dict(x)
    xt["h0"] = np.ascontiguousarray(np.swapaxes(x["h0"], -1, -2))
    b = oracle.fwd(pbt, **xt, want_h=True)
    gb = oracle.bwd(pbt, **xt, do=dO, dht=np.ascontiguousarray(np.swapaxes(dht, -1, -2)))
    assert np.array_equal(a["o"], b["o"])
    assert np.array_equal(a["final_state"], np.swapaxes(b["final_state"], -1, -2))
    assert np.array_equal(a["h"], np.swapaxes(b["h"], -1, -2))
    for key in ("dq", "dk", "dv", "dg", "dbeta"):
        assert np.array_equal(ga[key], gb[key]), key
    assert np.array_equal(ga["dh0"], np.swapaxes(gb["dh0"], -1, -2))


# ---------------------------------------------------------------- finite differences

FD_CASES = [
    dict(B=2, T=9, Hq=1, Hv=1, l2norm=False, cu=None, vf=False),
    dict(B=1, T=8, Hq=1, Hv=1, l2norm=True, cu=[0, 3, 3, 8], vf=False),
    dict(B=1, T=7, Hq=1, Hv=2, l2norm=True, cu=None, vf=True),
]


@pytest.mark.parametrize("case", FD_CASES, ids=["dense", "varlen", "gva_vfirst"])
def test_gradients_match_finite_differences(case):
    rng = np.random.default_rng(7)
    K = V = 4
    pb = Problem(B=case["B"], T=case["T"], Hq=case["Hq"], Hv=case["Hv"], K=K, V=V, scale=0.8,
                 l2norm=case["l2norm"], state_v_first=case["vf"], cu_seqlens=case["cu"], chunk=3)
    x = small_inputs(rng, pb)
    out = oracle.fwd(pb, **x)
    Ro = rnd(rng, *out["o"].shape)
    Rh = rnd(rng, *out["final_state"].shape)

    def loss(xx):
        r = oracle.fwd(pb, **xx)
        return float(np.sum(r["o"] * Ro) + np.sum(r["final_state"] * Rh))

    grads = oracle.bwd(pb, **x, do=Ro, dht=Rh)
    names = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta", "h0": "dh0"}
    eps = 1e-6
    for name, gname in names.items():
        base = x[name]
        num = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = {kk: (vv.copy() if kk == name else vv) for kk, vv in x.items()}
            xm = {kk: (vv.copy() if kk == name else vv) for kk, vv in x.items()}
            xp[name][idx] += eps
            xm[name][idx] -= eps
            num[idx] = (loss(xp) - loss(xm)) / (2 * eps)
        ana = grads[gname]
        err = np.max(np.abs(ana - num)) / max(1e-3, np.max(np.abs(num)))
        assert err < 1e-6, (name, err)


# ---------------------------------------------------------------- structural equalities

def test_continuation_through_final_state():
    rng = np.random.default_rng(8)
    pb = Problem(B=1, T=150, Hq=1, Hv=2, K=16, V=8, l2norm=True)
    x = small_inputs(rng, pb)
    full = oracle.fwd(pb, **x)
    T1 = 70
    pa = Problem(B=1, T=T1, Hq=1, Hv=2, K=16, V=8, l2norm=True)
    pbb = Problem(B=1, T=150 - T1, Hq=1, Hv=2, K=16, V=8, l2norm=True)
    xa = {kk: (vv[:, :T1] if kk != "h0" else vv) for kk, vv in x.items()}
    ra = oracle.fwd(pa, **xa)
    xb = {kk: (vv[:, T1:] if kk != "h0" else ra["final_state"]) for kk, vv in x.items()}
    rb = oracle.fwd(pbb, **xb)
    np.testing.assert_allclose(np.concatenate([ra["o"], rb["o"]], axis=1), full["o"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(rb["final_state"], full["final_state"], rtol=1e-12, atol=1e-12)


def test_varlen_equals_separate_calls():
    rng = np.random.default_rng(9)
    lens = [5, 0, 70, 1]
    cu = [0, 5, 5, 75, 76]
    pb = Problem(B=1, T=76, Hq=2, Hv=2, K=8, V=8, cu_seqlens=cu, chunk=16, l2norm=True)
    x = small_inputs(rng, pb)
    do = rnd(rng, 1, 76, 2, 8)
    dht = rnd(rng, 4, 2, 8, 8)
    r = oracle.fwd(pb, **x, want_h=True)
    gr = oracle.bwd(pb, **x, do=do, dht=dht)
    for n, L in enumerate(lens):
        s = slice(cu[n], cu[n + 1])
        p1 = Problem(B=1, T=L, Hq=2, Hv=2, K=8, V=8, chunk=16, l2norm=True)
        xn = {kk: (vv[:, s] if kk != "h0" else vv[n:n + 1]) for kk, vv in x.items()}
        rn = oracle.fwd(p1, **xn)
        gn = oracle.bwd(p1, **xn, do=do[:, s], dht=dht[n:n + 1])
        np.testing.assert_allclose(r["o"][:, s], rn["o"], rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(r["final_state"][n], rn["final_state"][0], rtol=1e-13, atol=1e-13)
        for key in ("dq", "dk", "dv", "dg", "dbeta"):
            np.testing.assert_allclose(gr[key][:, s], gn[key], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(gr["dh0"][n], gn["dh0"][0], rtol=1e-12, atol=1e-12)
    # empty sequence: final state = initial state, dh0 = dht
    assert np.array_equal(r["final_state"][1], x["h0"][1])
    assert np.array_equal(gr["dh0"][1], dht[1])


def test_grouped_heads_equal_repeated_heads():
    rng = np.random.default_rng(10)
    pb = Problem(B=2, T=20, Hq=2, Hv=4, K=8, V=4, l2norm=True, chunk=8)
    x = small_inputs(rng, pb)
    do = rnd(rng, 2, 20, 4, 4)
    r = oracle.fwd(pb, **x)
    gr = oracle.bwd(pb, **x, do=do)
    pr = Problem(B=2, T=20, Hq=4, Hv=4, K=8, V=4, l2norm=True, chunk=8)
    xr = dict(x)
    xr["q"] = np.repeat(x["q"], 2, axis=2)
    xr["k"] = np.repeat(x["k"], 2, axis=2)
    rr = oracle.fwd(pr, **xr)
    grr = oracle.bwd(pr, **xr, do=do)
    np.testing.assert_allclose(r["o"], rr["o"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(gr["dv"], grr["dv"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(gr["dq"], grr["dq"].reshape(2, 20, 2, 2, 8).sum(3), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(gr["dk"], grr["dk"].reshape(2, 20, 2, 2, 8).sum(3), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- chunked identities

def test_chunked_identities_pin_g_cumsum_A_and_h():
    """The per-chunk quantities reproduce the token recurrence exactly (fp64):

    Delta = A (diag(beta) V - diag(beta e^G) K h_c) equals the per-token delta,
    O = scale (diag(e^G) Q h_c + (Q K^T o Gamma o M) Delta) equals o, and
    e^{G_last} h_c + (diag(e^{G_last - G}) K)^T Delta equals the next chunk's state.
    """
    rng = np.random.default_rng(11)
    C = 16
    cu = [0, 37, 37 + 16, 37 + 16 + 5]
    pb = Problem(B=1, T=58, Hq=1, Hv=2, K=8, V=6, l2norm=True, cu_seqlens=cu, chunk=C, scale=0.7)
    x = small_inputs(rng, pb)
    r = oracle.fwd(pb, **x, want_h=True, want_delta=True)
    G = oracle.g_cumsum(pb, x["g"])[0]
    A = oracle.wy_matrix(pb, x["k"], x["g"], x["beta"])[0]
    kk = x["k"][0] / np.sqrt((x["k"][0] ** 2).sum(-1, keepdims=True) + oracle.L2_EPS)
    qq = x["q"][0] / np.sqrt((x["q"][0] ** 2).sum(-1, keepdims=True) + oracle.L2_EPS)
    offs, _ = oracle.prepare_chunk_offsets(cu, C)
    for n in range(3):
        s0, L = cu[n], cu[n + 1] - cu[n]
        for c, c0 in enumerate(range(0, L, C)):
            m = min(C, L - c0)
            sl = slice(s0 + c0, s0 + c0 + m)
            for j in range(2):
                hc = r["h"][offs[n] + c, j]
                Gc = G[sl, j]
                Kc, Qc = kk[sl, 0], qq[sl, 0]
                Ac = A[sl, j, :m]
                b = x["beta"][0, sl, j]
                rhs = b[:, None] * x["v"][0, sl, j] - (b * np.exp(Gc))[:, None] * (Kc @ hc)
                D = Ac @ rhs
                np.testing.assert_allclose(D, r["delta"][0, sl, j], rtol=1e-11, atol=1e-12)
                Gam = np.tril(np.exp(Gc[:, None] - Gc[None, :]))
                O = pb.scale * (np.exp(Gc)[:, None] * (Qc @ hc) + ((Qc @ Kc.T) * Gam) @ D)
                np.testing.assert_allclose(O, r["o"][0, sl, j], rtol=1e-11, atol=1e-12)
                hn = np.exp(Gc[-1]) * hc + (np.exp(Gc[-1] - Gc)[:, None] * Kc).T @ D
                nxt = r["h"][offs[n] + c + 1, j] if c0 + C < L else r["final_state"][n, j]
                np.testing.assert_allclose(hn, nxt, rtol=1e-11, atol=1e-12)


def test_h_rows_are_prefix_final_states():
    rng = np.random.default_rng(12)
    pb = Problem(B=1, T=50, Hq=1, Hv=1, K=8, V=8, chunk=16)
    x = small_inputs(rng, pb)
    r = oracle.fwd(pb, **x, want_h=True)
    for c in range(4):
        T1 = 16 * c
        if T1 == 0:
            np.testing.assert_array_equal(r["h"][0], x["h0"][0])
            continue
        pp = Problem(B=1, T=T1, Hq=1, Hv=1, K=8, V=8, chunk=16)
        rp = oracle.fwd(pp, **{kk: (vv[:, :T1] if kk != "h0" else vv) for kk, vv in x.items()})
        np.testing.assert_allclose(r["h"][c], rp["final_state"][0], rtol=1e-13, atol=1e-14)


def test_gate_gradient_identity():
    """With h_t = e^{G_t} h~_t the gate enters only through e^{G_t} q_t, e^{-G_t} v_t and the final
    state, so dg_s = sum_{t>=s} (<q_t, dq_t> - <v_t, dv_t>) + <dh_T, h_T> per sequence and head."""
    rng = np.random.default_rng(13)
    cu = [0, 29, 29, 90]
    pb = Problem(B=1, T=90, Hq=2, Hv=2, K=8, V=6, scale=0.7, chunk=16, cu_seqlens=cu)
    x = small_inputs(rng, pb)
    dO = rnd(rng, 1, 90, 2, 6)
    dht = rnd(rng, 3, 2, 8, 6)
    f = oracle.fwd(pb, **x)
    r = oracle.bwd(pb, **x, do=dO, dht=dht)
    D = (x["q"] * r["dq"]).sum(-1) - (x["v"] * r["dv"]).sum(-1)
    for n in range(3):
        s = slice(cu[n], cu[n + 1])
        ident = np.flip(np.cumsum(np.flip(D[0, s], 0), 0), 0) + (dht[n] * f["final_state"][n]).sum((-1, -2))
        np.testing.assert_allclose(ident, r["dg"][0, s], rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- activation options

ACT = dict(gate_in_kernel=True, beta_sigmoid=True, neg_eigval=True)


def test_activations_equal_library_routines():
    """With the options set, the oracle equals the plain recurrence on inputs activated by scipy's own
    logistic routines (an implementation other than the oracle's)."""
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(21)
    base = dict(B=2, T=11, Hq=1, Hv=2, K=4, V=4, scale=0.7, chunk=4)
    x = small_inputs(rng, Problem(**base))
    graw = 3.0 * rnd(rng, *x["g"].shape)          # raw gate logits, both signs, some large
    braw = 3.0 * rnd(rng, *x["beta"].shape)
    for opts in (dict(gate_in_kernel=True), dict(beta_sigmoid=True), dict(neg_eigval=True), ACT):
        pa = Problem(**base, **opts)
        ga = special.log_expit(graw) if opts.get("gate_in_kernel") else graw
        ba = special.expit(braw) if opts.get("beta_sigmoid") else braw
        if opts.get("neg_eigval"):
            ba = 2.0 * ba
        got = oracle.fwd(pa, x["q"], x["k"], x["v"], graw, braw, h0=x["h0"])
        want = oracle.fwd(Problem(**base), x["q"], x["k"], x["v"], ga, ba, h0=x["h0"])
        for key in ("o", "final_state"):
            assert np.allclose(got[key], want[key], rtol=1e-13, atol=1e-13), (opts, key)


def test_negative_eigenvalue_reflects_the_key_direction():
    """beta = 2 (raw beta = 1 doubled), g = 0, v = 0: the step is the Householder reflection I - 2 k k^T of
    the state, so a state k u^T becomes -k u^T (eigenvalue -1 along k) and directions orthogonal to k stay."""
    K = V = 4
    pb = Problem(B=1, T=1, Hq=1, Hv=1, K=K, V=V, scale=1.0, neg_eigval=True)
    k = np.zeros((1, 1, 1, K)); k[..., 1] = 1.0
    u = np.array([0.5, -1.0, 2.0, 0.25])
    w = np.array([0.0, 0.0, 3.0, 0.0])            # orthogonal to k
    h0 = (np.outer(k[0, 0, 0], u) + np.outer(np.array([1.0, 0, 0, 0]), w))[None, None]
    out = oracle.fwd(pb, np.zeros((1, 1, 1, K)), k, np.zeros((1, 1, 1, V)), np.zeros((1, 1, 1)),
                     np.ones((1, 1, 1)), h0=h0)
    want = -np.outer(k[0, 0, 0], u) + np.outer(np.array([1.0, 0, 0, 0]), w)
    assert np.allclose(out["final_state"][0, 0], want, atol=1e-15)


@pytest.mark.parametrize("opts", [dict(gate_in_kernel=True), dict(beta_sigmoid=True), ACT],
                         ids=["gate", "beta_sigmoid", "all"])
def test_activation_gradients_match_finite_differences(opts):
    """Gradients w.r.t. the raw gate and beta (chain rule through the activations) against central
    differences of the whole forward."""
    rng = np.random.default_rng(22)
    pb = Problem(B=1, T=7, Hq=1, Hv=2, K=4, V=4, scale=0.8, l2norm=True, cu_seqlens=[0, 3, 7], chunk=3, **opts)
    x = small_inputs(rng, pb)
    x["g"] = 2.0 * rnd(rng, *x["g"].shape)
    x["beta"] = 2.0 * rnd(rng, *x["beta"].shape)
    out = oracle.fwd(pb, **x)
    Ro = rnd(rng, *out["o"].shape)
    Rh = rnd(rng, *out["final_state"].shape)

    def loss(xx):
        r = oracle.fwd(pb, **xx)
        return float(np.sum(r["o"] * Ro) + np.sum(r["final_state"] * Rh))

    grads = oracle.bwd(pb, **x, do=Ro, dht=Rh)
    eps = 1e-6
    for name, gname in (("g", "dg"), ("beta", "dbeta"), ("k", "dk")):
        base = x[name]
        num = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = {kk: (vv.copy() if kk == name else vv) for kk, vv in x.items()}
            xm = {kk: (vv.copy() if kk == name else vv) for kk, vv in x.items()}
            xp[name][idx] += eps
            xm[name][idx] -= eps
            num[idx] = (loss(xp) - loss(xm)) / (2 * eps)
        err = np.max(np.abs(grads[gname] - num)) / max(1e-3, np.max(np.abs(num)))
        assert err < 1e-6, (name, err)
