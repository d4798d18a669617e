"""The Python binding refuses, before any launch, every tensor the library would read or write as something
it is not (wrong shape, dtype, device or layout, a saved buffer made for a smaller problem); the
differentiable op accepts views (q, k, v sliced from one fused projection) and gives what contiguous
copies give."""

import pytest
import torch

import gated_delta_rule_38_gb300 as gdr

pytestmark = pytest.mark.gpu

B, T, H, D = 2, 100, 2, 128


def _inputs(seed=0):
    gen = torch.Generator(device="cuda").manual_seed(seed)
    r = lambda *s: torch.randn(*s, device="cuda", generator=gen)
    q, k, v = (r(B, T, H, D).bfloat16() for _ in range(3))
    g = torch.nn.functional.logsigmoid(r(B, T, H) + 2).bfloat16()
    beta = torch.sigmoid(r(B, T, H)).bfloat16()
    return q, k, v, g, beta


def test_forward_refusals():
    q, k, v, g, beta = _inputs()
    cases = [
        (dict(q=q.transpose(1, 2).contiguous().transpose(1, 2)), "contiguous"),
        (dict(k=k[:, :T - 1]), "shape"),
        (dict(k=k.half()), "dtype"),
        (dict(g=g[..., :1]), "shape"),
        (dict(beta=beta.float()), "dtype"),
        (dict(initial_state=torch.zeros(B, H, D, D - 8, device="cuda")), "shape"),
        (dict(cu_seqlens=torch.tensor([0, 2 * T], dtype=torch.int32)), "CUDA tensor"),
    ]
    for over, msg in cases:
        kw = dict(q=q, k=k, v=v, g=g, beta=beta)
        kw.update(over)
        with pytest.raises(ValueError, match=msg):
            gdr.chunk_gated_delta_rule_fwd(**kw)
    small = gdr.saved_buffer(q[:, :64], v[:, :64], g[:, :64])
    with pytest.raises(ValueError, match="saved"):
        gdr.chunk_gated_delta_rule_fwd(q, k, v, g, beta, saved=small)


def test_backward_refusals():
    q, k, v, g, beta = _inputs()
    gcs, A, o, _, _ = gdr.chunk_gated_delta_rule_fwd(q, k, v, g, beta)
    do = torch.randn_like(o)
    cases = [
        (dict(g=gcs.bfloat16()), "dtype"),
        (dict(A=A.half()), "dtype"),
        (dict(A=A[..., :32].contiguous()), "shape"),
        (dict(do=do[:, :T - 1]), "shape"),
        (dict(dht=torch.zeros(B, H, D, D + 8, device="cuda")), "shape"),
        (dict(beta=beta.float(), gate_dtype=torch.bfloat16), "dtype"),
    ]
    for over, msg in cases:
        kw = dict(q=q, k=k, v=v, g=gcs, beta=beta, A=A, do=do)
        kw.update(over)
        with pytest.raises(ValueError, match=msg):
            gdr.chunk_gated_delta_rule_bwd(**kw)
    torch.cuda.synchronize()
    assert gdr.get_error() == 0


def test_differentiable_op_takes_views_of_a_fused_projection():
    q, k, v, g, beta = _inputs(1)
    fused = torch.cat([q, k, v], dim=-1).requires_grad_(True)  # [B, T, H, 3D]
    fv = [fused[..., i * D:(i + 1) * D] for i in range(3)]  # strided views
    assert not fv[0].is_contiguous()
    copies = [t.detach().clone().contiguous().requires_grad_(True) for t in fv]
    o1, _ = gdr.chunk_gated_delta_rule(*fv, g, beta, use_qk_l2norm_in_kernel=True)
    o2, _ = gdr.chunk_gated_delta_rule(*copies, g, beta, use_qk_l2norm_in_kernel=True)
    assert torch.equal(o1, o2)
    do = torch.randn_like(o1)
    o1.backward(do)
    o2.backward(do)
    want = torch.cat([c.grad for c in copies], dim=-1)
    assert torch.equal(fused.grad, want)
