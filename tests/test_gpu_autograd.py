"""Two layers in one autograd graph, the second reading the first's output as its queries: both forwards run
first (each keeps its own saved buffer), then both backwards in reverse order on the autograd engine's
thread.  Every gradient equals, bit for bit, the same sequence of calls made by hand through the low-level
forward and backward (the kernels are deterministic)."""

import pytest
import torch

import gated_delta_rule_38_gb300 as gdr

pytestmark = pytest.mark.gpu

B, T, H, D = 2, 150, 2, 128


def test_two_chained_layers():
    gen = torch.Generator(device="cuda").manual_seed(51)
    r = lambda *s: torch.randn(*s, device="cuda", generator=gen)
    x = r(B, T, H, D).bfloat16()
    k1, v1, k2, v2 = (r(B, T, H, D).bfloat16() for _ in range(4))
    g1, g2 = (torch.nn.functional.logsigmoid(r(B, T, H) + 2).bfloat16() for _ in range(2))
    b1, b2 = (torch.sigmoid(r(B, T, H)).bfloat16() for _ in range(2))
    h0 = r(B, H, D, D)
    wgt = r(B, T, H, D).bfloat16()
    opts = dict(use_qk_l2norm_in_kernel=True)

    # by hand: forward 1, forward 2, backward 2, backward 1 (dO of layer 1 = dq of layer 2)
    s1 = gdr.saved_buffer(x, v1, g1, **opts)
    gc1, A1, o1, _, _ = gdr.chunk_gated_delta_rule_fwd(x, k1, v1, g1, b1, initial_state=h0, saved=s1, **opts)
    s2 = gdr.saved_buffer(o1, v2, g2, **opts)
    gc2, A2, o2, _, _ = gdr.chunk_gated_delta_rule_fwd(o1, k2, v2, g2, b2, saved=s2, **opts)
    dq2, dk2, dv2, db2, dg2, _ = gdr.chunk_gated_delta_rule_bwd(o1, k2, v2, gc2, b2, A2, wgt, saved=s2, **opts)
    dq1, dk1, dv1, db1, dg1, dh01 = gdr.chunk_gated_delta_rule_bwd(x, k1, v1, gc1, b1, A1, dq2, initial_state=h0,
                                                                   saved=s1, **opts)
    torch.cuda.synchronize()

    # the same through the differentiable op
    leaves = [t.clone().requires_grad_(True) for t in (x, k1, v1, g1, b1, k2, v2, g2, b2, h0)]
    X, K1, V1, G1, B1, K2, V2, G2, B2, H0 = leaves
    y1, _ = gdr.chunk_gated_delta_rule(X, K1, V1, G1, B1, initial_state=H0, **opts)
    y2, _ = gdr.chunk_gated_delta_rule(y1, K2, V2, G2, B2, **opts)
    y2.backward(wgt)
    torch.cuda.synchronize()
    assert torch.equal(y2.detach(), o2)
    want = [dq1, dk1, dv1, dg1, db1, dk2, dv2, dg2, db2, dh01]
    for name, leaf, w in zip(("x", "k1", "v1", "g1", "beta1", "k2", "v2", "g2", "beta2", "h0"), leaves, want):
        assert torch.equal(leaf.grad, w), name


def test_initial_state_in_bf16():
    """A bf16 initial state that requires grad: the library runs the states in fp32, and the gradient comes
    back in the leaf's dtype (the fp32 state's gradient, rounded)."""
    gen = torch.Generator(device="cuda").manual_seed(52)
    r = lambda *s: torch.randn(*s, device="cuda", generator=gen)
    q, k, v = (r(B, T, H, D).bfloat16() for _ in range(3))
    g = torch.nn.functional.logsigmoid(r(B, T, H) + 2).bfloat16()
    beta = torch.sigmoid(r(B, T, H)).bfloat16()
    h0 = r(B, H, D, D).bfloat16()
    wgt = r(B, T, H, D).bfloat16()
    hb = h0.clone().requires_grad_(True)
    hf = h0.float().requires_grad_(True)
    ob, fb = gdr.chunk_gated_delta_rule(q, k, v, g, beta, initial_state=hb, output_final_state=True,
                                        use_qk_l2norm_in_kernel=True)
    of, ff = gdr.chunk_gated_delta_rule(q, k, v, g, beta, initial_state=hf, output_final_state=True,
                                        use_qk_l2norm_in_kernel=True)
    assert torch.equal(ob, of) and torch.equal(fb, ff)
    (ob.float() * wgt.float()).sum().backward()
    (of.float() * wgt.float()).sum().backward()
    assert hb.grad.dtype == torch.bfloat16
    assert torch.equal(hb.grad, hf.grad.bfloat16())
