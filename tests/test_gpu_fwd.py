"""Forward parity: the CUDA path (through the C ABI) against the fp64 oracle."""

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_38_gb300.inputs import WORKLOADS, custom, make_inputs
from harness import TOL, gpu_fwd, np64, oracle_problem, rel_l2, to_dev

pytestmark = pytest.mark.gpu


def check_fwd(w, kernel_l2, heads=None, check_chunks=True, gate_f32=False):
    x = make_inputs(w)
    d = to_dev(x)
    gcs, A, o, h, fin = gpu_fwd(w, d, kernel_l2, output_h=check_chunks, gate_f32=gate_f32)
    torch.cuda.synchronize()
    pb = oracle_problem(w, kernel_l2)
    ref = oracle.fwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"], heads=heads,
                     want_h=check_chunks)
    sel = slice(None) if heads is None else list(heads)
    errs = {"o": rel_l2(np64(o)[:, :, sel], ref["o"][:, :, sel])}
    if w.final_state:
        errs["final_state"] = rel_l2(np64(fin)[:, sel], ref["final_state"][:, sel])
    if check_chunks:
        nrows = ref["h"].shape[0]
        errs["h"] = rel_l2(np64(h[:nrows])[:, sel], ref["h"][:, sel])  # (rows past the chunk count are unused)
        gref = oracle.g_cumsum(pb, x["g"])
        assert rel_l2(np64(gcs)[..., sel], gref[..., sel]) < 1e-5
        Aref = oracle.wy_matrix(pb, x["k"], x["g"], x["beta"])
        errs["A"] = rel_l2(np64(A)[:, :, sel], Aref[:, :, sel])
    for key, e in errs.items():
        assert e <= TOL, (key, e, errs)
    return errs


def test_tiny():
    check_fwd(WORKLOADS["tiny"], kernel_l2=False)


def test_tiny_kernel_l2norm():
    w = custom(B=1, T=256, Hq=2, Hv=2, host_l2=False)
    check_fwd(w, kernel_l2=True)


@pytest.mark.parametrize("T", [1, 63, 64, 65, 129, 200])
def test_ragged_lengths(T):
    w = custom(B=2, T=T, Hq=1, Hv=2, host_l2=False)
    check_fwd(w, kernel_l2=True)


def test_varlen_with_empty_and_short_sequences():
    w = custom(seq_lens=(7, 0, 130, 64, 1, 65), Hq=2, Hv=2)
    check_fwd(w, kernel_l2=False)


def test_gva_fp16():
    w = custom(B=2, T=150, Hq=1, Hv=4, dtype=torch.float16, host_l2=False)
    check_fwd(w, kernel_l2=True)


def test_fp32_gates():
    w = custom(B=1, T=190, Hq=2, Hv=2)
    check_fwd(w, kernel_l2=False, gate_f32=True)


def test_no_initial_state_no_final_state():
    w = custom(B=1, T=100, Hq=1, Hv=1, has_h0=False, final_state=False)
    check_fwd(w, kernel_l2=False)


def test_state_v_first_bit_exact():
    """state_v_first changes only the state layout: every result is bit-identical."""
    w = custom(B=2, T=200, Hq=1, Hv=2, dtype=torch.float16)
    x = to_dev(make_inputs(w))
    a = gpu_fwd(w, x, False, output_h=True)
    wt = custom(B=2, T=200, Hq=1, Hv=2, dtype=torch.float16, state_v_first=True)
    xt = dict(x)
    xt["h0"] = x["h0"].transpose(-1, -2).contiguous()
    b = gpu_fwd(wt, xt, False, output_h=True)
    torch.cuda.synchronize()
    assert torch.equal(a[2], b[2])                                  # o
    assert torch.equal(a[4], b[4].transpose(-1, -2))                # final state
    assert torch.equal(a[3], b[3].transpose(-1, -2))                # h
    assert torch.equal(a[1], b[1]) and torch.equal(a[0], b[0])      # A, g_cumsum


def test_rejects_unaligned_and_missing():
    import gated_delta_rule_38_gb300 as gdr
    w = custom(B=1, T=64, Hq=1, Hv=1)
    x = to_dev(make_inputs(w))
    with pytest.raises(gdr.GdrError) as e:
        gdr.chunk_gated_delta_rule_fwd(x["q"].float(), x["k"].float(), x["v"].float(), x["g"], x["beta"])
    assert e.value.status == 3
    buf = torch.empty(x["q"].numel() + 8, dtype=x["q"].dtype, device="cuda")
    qmis = buf[1:1 + x["q"].numel()].view_as(x["q"])
    qmis.copy_(x["q"])
    with pytest.raises(gdr.GdrError) as e:
        gdr.chunk_gated_delta_rule_fwd(qmis, x["k"], x["v"], x["g"], x["beta"])
    assert e.value.status == 6


# ---------------------------------------------------------------- full-size workloads (every head)

# (per-chunk states are not offered for the long split path nor for head dimensions below 128)
@pytest.mark.parametrize("name", ["dense", "varlen", "gva", "long", "dense_act", "dense_hd64"])
def test_full_size_all_heads(name):
    w = WORKLOADS[name]
    check_fwd(w, kernel_l2=not w.host_l2, check_chunks=name not in ("long", "dense_hd64"))


# q/k head counts that are not powers of two (the kernels' item -> chunk slot, q/k head arithmetic divides by Hq
# and by the chunks per sequence)
@pytest.mark.parametrize("hq,hv", [(3, 3), (3, 6), (5, 10)])
def test_head_counts_not_powers_of_two(hq, hv):
    check_fwd(custom(B=3, T=201, Hq=hq, Hv=hv, host_l2=False), kernel_l2=True)
    check_fwd(custom(seq_lens=(65, 0, 7, 130), Hq=hq, Hv=hv), kernel_l2=False)
