"""Recurrent decode parity: gdr_decode (through the C ABI) against the fp64 oracle's token-level forward on
the same seeded inputs.  The oracle applies the recurrence token by token, which is exactly what the
decode computes, so its output and final state are the expected values."""

import pytest
import torch

import oracle
from gated_delta_rule_38_gb300.inputs import custom, make_inputs
from harness import TOL, gpu_fwd, np64, oracle_problem, rel_l2, to_dev

pytestmark = pytest.mark.gpu


def check_decode(w, kernel_l2, gate_f32=False, inplace=False):
    import gated_delta_rule_38_gb300 as gdr
    x = make_inputs(w)
    d = to_dev(x)
    g, beta = d["g"], d["beta"]
    if gate_f32:
        g, beta = g.float(), beta.float()
    h0 = d["h0"].clone() if (inplace and d["h0"] is not None) else d["h0"]
    o, fin = gdr.recurrent_gated_delta_rule(d["q"], d["k"], d["v"], g, beta, initial_state=h0,
                                            use_qk_l2norm_in_kernel=kernel_l2, state_v_first=w.state_v_first,
                                            inplace=inplace)
    torch.cuda.synchronize()
    if inplace:
        assert fin.data_ptr() == h0.data_ptr()
    ref = oracle.fwd(oracle_problem(w, kernel_l2), x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"])
    eo, ef = rel_l2(np64(o), ref["o"]), rel_l2(np64(fin), ref["final_state"])
    assert eo <= TOL and ef <= TOL, (eo, ef)
    return o, fin


def test_one_token_kernel_l2norm_gva():
    check_decode(custom(B=3, T=1, Hq=2, Hv=4, host_l2=False), kernel_l2=True)


def test_few_tokens_fp16_state_v_first():
    check_decode(custom(B=2, T=5, Hq=1, Hv=2, dtype=torch.float16, state_v_first=True), kernel_l2=False)


def test_zero_state_fp32_gates():
    check_decode(custom(B=2, T=3, Hq=2, Hv=2, has_h0=False, host_l2=False), kernel_l2=True, gate_f32=True)


def test_in_place_state():
    check_decode(custom(B=2, T=2, Hq=2, Hv=2, host_l2=False), kernel_l2=True, inplace=True)


def test_decode_continues_the_chunked_forward():
    """The chunked forward over the first tokens, then decode of the next ones from its final state, gives the
    oracle's result over all tokens (the state cache hand-off of autoregressive inference)."""
    import gated_delta_rule_38_gb300 as gdr
    T0, T1 = 70, 3
    w = custom(B=2, T=T0 + T1, Hq=1, Hv=2, host_l2=False)
    x = make_inputs(w)
    d = to_dev(x)
    part = lambda t, a, b: t[:, a:b].contiguous()
    _, _, o0, _, fin0 = gdr.chunk_gated_delta_rule_fwd(part(d["q"], 0, T0), part(d["k"], 0, T0),
                                                       part(d["v"], 0, T0), part(d["g"], 0, T0),
                                                       part(d["beta"], 0, T0), initial_state=d["h0"],
                                                       use_qk_l2norm_in_kernel=True)
    o1, fin = gdr.recurrent_gated_delta_rule(part(d["q"], T0, T0 + T1), part(d["k"], T0, T0 + T1),
                                             part(d["v"], T0, T0 + T1), part(d["g"], T0, T0 + T1),
                                             part(d["beta"], T0, T0 + T1), initial_state=fin0,
                                             use_qk_l2norm_in_kernel=True)
    torch.cuda.synchronize()
    ref = oracle.fwd(oracle_problem(w, True), x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"])
    assert rel_l2(np64(torch.cat([o0, o1], dim=1)), ref["o"]) <= TOL
    assert rel_l2(np64(fin), ref["final_state"]) <= TOL


def test_zero_tokens_copies_the_state():
    import gated_delta_rule_38_gb300 as gdr
    w = custom(B=2, T=4, Hq=1, Hv=2, host_l2=False)
    d = to_dev(make_inputs(w))
    e = lambda t: t[:, :0].contiguous()
    _, fin = gdr.recurrent_gated_delta_rule(e(d["q"]), e(d["k"]), e(d["v"]), e(d["g"]), e(d["beta"]),
                                            initial_state=d["h0"])
    torch.cuda.synchronize()
    assert torch.equal(fin, d["h0"])


@pytest.mark.parametrize("hq,hv", [(3, 6), (5, 5)])
def test_head_counts_not_powers_of_two(hq, hv):
    """The decode's block -> (row, value head) -> q/k head mapping at head counts that are not powers of two."""
    check_decode(custom(B=3, T=2, Hq=hq, Hv=hv, host_l2=False), kernel_l2=True)
