"""Seeded combinations of the recurrent decode's options against the oracle's token recurrence: batch and
token counts, GVA grouping, head dims, dtype, norm placement, state layout, initial state or none, the
activation options, fp32 gates and the in-place state update.  The decode keeps the states in fp32, so the
plain bound holds."""

import random

import pytest
import torch

import oracle
from gated_delta_rule_38_gb300.inputs import custom, make_inputs
from harness import TOL, act_options, np64, oracle_problem, rel_l2, to_dev

pytestmark = pytest.mark.gpu

HEADS = [(1, 1), (1, 2), (2, 2), (2, 4), (4, 8)]
DIMS = [(128, 128), (128, 128), (64, 64), (32, 96), (128, 48), (8, 16)]


def draw(seed):
    r = random.Random(seed)
    hq, hv = r.choice(HEADS)
    k, v = r.choice(DIMS)
    spec = dict(B=r.choice([1, 3, 17]), T=r.choice([1, 1, 2, 5]), Hq=hq, Hv=hv, K=k, V=v,
                dtype=r.choice([torch.bfloat16, torch.float16]), host_l2=r.random() < 0.5,
                state_v_first=r.random() < 0.3, has_h0=r.random() < 0.8, final_state=True,
                activations=r.random() < 0.3, mu_g=r.choice([0.0, 1.0, 2.0]))
    inplace = spec["has_h0"] and r.random() < 0.5
    gate_f32 = r.random() < 0.3
    return spec, inplace, gate_f32


@pytest.mark.parametrize("seed", range(60))
def test_decode_combinations(seed):
    import gated_delta_rule_38_gb300 as gdr
    spec, inplace, gate_f32 = draw(5000 + seed)
    w = custom(name="dec_combo", **spec)
    kernel_l2 = not w.host_l2
    x = make_inputs(w, seed=6000 + seed)
    d = to_dev(x)
    g, beta = d["g"], d["beta"]
    if gate_f32:
        g, beta = g.float(), beta.float()
    h0 = d["h0"].clone() if inplace else d["h0"]
    o, fin = gdr.recurrent_gated_delta_rule(d["q"], d["k"], d["v"], g, beta, initial_state=h0,
                                            use_qk_l2norm_in_kernel=kernel_l2, state_v_first=w.state_v_first,
                                            inplace=inplace, **act_options(w))
    torch.cuda.synchronize()
    if inplace:
        assert fin.data_ptr() == h0.data_ptr()
    ref = oracle.fwd(oracle_problem(w, kernel_l2), x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"])
    eo, ef = rel_l2(np64(o), ref["o"]), rel_l2(np64(fin), ref["final_state"])
    assert eo <= TOL and ef <= TOL, (eo, ef, spec, inplace, gate_f32)
