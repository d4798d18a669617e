"""Backward parity: the CUDA path (through the C ABI) against the fp64 oracle's
reverse-mode gradients, on the same seeded inputs."""

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_38_gb300.inputs import WORKLOADS, custom, make_inputs
from harness import TOL, gpu_bwd, gpu_fwd, gpu_saved, np64, oracle_problem, rel_l2, to_dev

pytestmark = pytest.mark.gpu

GRADS = ("dq", "dk", "dv", "dbeta", "dg", "dh0")


def check_bwd(w, kernel_l2, heads=None, gate_f32=False, num_segments=0, saved=False):
    x = make_inputs(w)
    d = to_dev(x)
    sv = gpu_saved(w, d, kernel_l2, num_segments=num_segments, gate_f32=gate_f32) if saved else None
    gcs, A, o, _, fin = gpu_fwd(w, d, kernel_l2, num_segments=num_segments, gate_f32=gate_f32, saved=sv)
    dq, dk, dv, db, dg, dh0 = gpu_bwd(w, d, gcs, A, kernel_l2, num_segments=num_segments, gate_f32=gate_f32,
                                      saved=sv)
    torch.cuda.synchronize()
    pb = oracle_problem(w, kernel_l2)
    ref = oracle.bwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], h0=x["h0"], dht=x["dht"],
                     heads=heads)
    got = {"dq": dq, "dk": dk, "dv": dv, "dbeta": db, "dg": dg, "dh0": dh0}
    if heads is None:
        vsel = qsel = slice(None)
    else:
        grp = w.Hv // w.Hq
        vsel = list(heads)
        qsel = sorted({h // grp for h in heads})
    errs = {}
    for key in GRADS:
        if got[key] is None:
            assert x["h0"] is None and key == "dh0"
            continue
        a = np64(got[key])
        b = ref[key]
        if key in ("dq", "dk"):
            a, b = a[:, :, qsel], b[:, :, qsel]
        elif key == "dh0":
            a, b = a[:, vsel], b[:, vsel]
        else:
            a, b = a[:, :, vsel], b[:, :, vsel]
        errs[key] = rel_l2(a, b)
    for key, e in errs.items():
        assert e <= TOL, (key, e, errs)
    return errs


def test_tiny():
    check_bwd(WORKLOADS["tiny"], kernel_l2=False)


def test_tiny_kernel_l2norm():
    check_bwd(custom(B=1, T=256, Hq=2, Hv=2, host_l2=False), kernel_l2=True)


# the forward's decayed causal blocks and q/k norms handed to the backward (no recompute there)
@pytest.mark.parametrize("kernel_l2", [False, True])
def test_saved_blocks(kernel_l2):
    check_bwd(custom(B=2, T=200, Hq=2, Hv=2, host_l2=not kernel_l2), kernel_l2=kernel_l2, saved=True)


def test_saved_blocks_varlen():
    check_bwd(custom(seq_lens=(7, 0, 130, 64, 1, 65), Hq=2, Hv=2, host_l2=False), kernel_l2=True, saved=True)


def test_saved_state_v_first():
    check_bwd(custom(B=2, T=150, Hq=1, Hv=2, state_v_first=True), kernel_l2=False, saved=True)


def test_saved_no_initial_state():
    check_bwd(custom(B=1, T=100, Hq=1, Hv=1, has_h0=False, final_state=False), kernel_l2=False, saved=True)


def test_saved_blocks_gva_fp16():
    check_bwd(custom(B=2, T=150, Hq=1, Hv=4, dtype=torch.float16, host_l2=False), kernel_l2=True, saved=True)


@pytest.mark.parametrize("T", [1, 63, 64, 65, 129, 200])
def test_ragged_lengths(T):
    check_bwd(custom(B=2, T=T, Hq=1, Hv=2, host_l2=False), kernel_l2=True)


def test_varlen_with_empty_and_short_sequences():
    check_bwd(custom(seq_lens=(7, 0, 130, 64, 1, 65), Hq=2, Hv=2), kernel_l2=False)


@pytest.mark.parametrize("saved", [False, True])
def test_varlen_many_sequences_with_equal_lengths(saved):
    """The chains start a packed batch's longest sequences first (a rank by length, ties by index): many
    sequences, repeated lengths, empty ones and more chains than SMs; forward and backward."""
    lens = (64, 130, 64, 1, 300, 130, 0, 64, 7, 300, 65, 1, 0, 129, 300, 2)
    w = custom(seq_lens=lens, Hq=4, Hv=8, host_l2=False)
    check_bwd(w, kernel_l2=True, saved=saved)
    check_fwd_states(w)


@pytest.mark.parametrize("saved", [False, True])
def test_varlen_more_sequences_than_the_order_table(saved):
    """More than 2,048 sequences: the chunk-table kernel ranks at most 2,048 by length and otherwise starts
    the chains in index order.  2,500 sequences of 0 to 40 tokens (empty ones included), states given;
    forward and backward against the oracle."""
    rng = np.random.default_rng(7)
    lens = tuple(int(n) for n in rng.integers(0, 41, size=2500))
    w = custom(name="many_seqs", seq_lens=lens, Hq=1, Hv=2, host_l2=False, has_h0=True, final_state=True)
    check_bwd(w, kernel_l2=True, saved=saved)
    check_fwd_states(w)


def test_reverse_chain_whole_width():
    """Equal-length batches whose 64-column reverse-chain slices would need an extra wave of SMs run it in
    whole-width CTAs: 2 sequences x 80 heads (320 slices, 160 whole-width CTAs), through the saved buffer."""
    check_bwd(custom(B=2, T=130, Hq=40, Hv=80, host_l2=False), kernel_l2=True, saved=True)


def check_fwd_states(w):
    """The forward's output and final states of a packed batch against the oracle."""
    x = make_inputs(w)
    d = to_dev(x)
    _, _, o, _, fin = gpu_fwd(w, d, True)
    torch.cuda.synchronize()
    ref = oracle.fwd(oracle_problem(w, True), x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"])
    assert rel_l2(np64(o), ref["o"]) <= TOL
    assert rel_l2(np64(fin), ref["final_state"]) <= TOL


def test_gva_fp16():
    check_bwd(custom(B=2, T=150, Hq=1, Hv=4, dtype=torch.float16, host_l2=False), kernel_l2=True)


def test_fp32_gates():
    check_bwd(custom(B=1, T=190, Hq=2, Hv=2), kernel_l2=False, gate_f32=True)


def test_no_initial_state():
    check_bwd(custom(B=1, T=100, Hq=1, Hv=1, has_h0=False, final_state=False), kernel_l2=False)


def test_state_v_first_bit_exact():
    w = custom(B=2, T=150, Hq=1, Hv=2, dtype=torch.float16)
    d = to_dev(make_inputs(w))
    gcs, A, _, _, _ = gpu_fwd(w, d, False)
    ga = gpu_bwd(w, d, gcs, A, False)
    wt = custom(B=2, T=150, Hq=1, Hv=2, dtype=torch.float16, state_v_first=True)
    dt = dict(d)
    dt["h0"] = d["h0"].transpose(-1, -2).contiguous()
    dt["dht"] = d["dht"].transpose(-1, -2).contiguous()
    gb = gpu_bwd(wt, dt, gcs, A, False)
    torch.cuda.synchronize()
    for a, b in zip(ga[:5], gb[:5]):
        assert torch.equal(a, b)
    assert torch.equal(ga[5], gb[5].transpose(-1, -2))


def test_autograd_function():
    import gated_delta_rule_38_gb300 as gdr
    w = custom(B=1, T=130, Hq=1, Hv=2, host_l2=False)
    x = make_inputs(w)
    d = {k: (v.cuda().requires_grad_(True) if v is not None and k in ("q", "k", "v", "g", "beta", "h0") else
             (v.cuda() if v is not None else None)) for k, v in x.items()}
    o, fin = gdr.chunk_gated_delta_rule(d["q"], d["k"], d["v"], d["g"], d["beta"], initial_state=d["h0"],
                                        output_final_state=True, use_qk_l2norm_in_kernel=True)
    (o.float() * d["do"].float()).sum().add_((fin * d["dht"]).sum()).backward()
    pb = oracle_problem(w, True)
    ref = oracle.bwd(pb, x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], h0=x["h0"], dht=x["dht"])
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta"), ("h0", "dh0")):
        assert rel_l2(np64(d[name].grad), ref[key]) <= TOL, name


# full sizes: the dense case as the training step runs it (the forward's saved buffer, the reverse chain alone)
# and without the buffer (forward recompute beside the reverse chain); the long sequence runs the split path;
# the dense variants with in-kernel activations and with head dimension 64 run as the benchmark times them
@pytest.mark.parametrize("name,saved", [("dense", True), ("dense", False), ("varlen", True), ("gva", True),
                                        ("long", False), ("long", True), ("dense_act", True), ("dense_hd64", True)])
def test_full_size_all_heads(name, saved):
    w = WORKLOADS[name]
    check_bwd(w, kernel_l2=not w.host_l2, saved=saved)


def test_back_to_back_steps_bit_identical():
    """Forward + backward steps issued back to back on one stream, with no host synchronisation between
    them (each kernel may begin launching while its predecessor finishes), give bit-identical results:
    every kernel waits for its predecessor's results before touching global memory."""
    import gated_delta_rule_38_gb300 as gdr
    w = custom(B=2, T=300, Hq=2, Hv=2, host_l2=False)
    d = to_dev(make_inputs(w))
    runs = []
    for _ in range(3):
        sv = gdr.saved_buffer(d["q"], d["v"], d["g"], use_qk_l2norm_in_kernel=True)
        gcs, A, o, _, fin = gdr.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                                           initial_state=d["h0"], use_qk_l2norm_in_kernel=True,
                                                           saved=sv)
        grads = gdr.chunk_gated_delta_rule_bwd(d["q"], d["k"], d["v"], gcs, d["beta"], A, d["do"], dht=d["dht"],
                                               initial_state=d["h0"], use_qk_l2norm_in_kernel=True, saved=sv)
        runs.append([o, fin] + [t for t in grads if t is not None])
    torch.cuda.synchronize()
    for other in runs[1:]:
        for a, b in zip(runs[0], other):
            assert torch.equal(a, b)


# q/k head counts that are not powers of two, with and without the saved buffer (the kernels' item -> chunk
# slot, q/k head arithmetic divides by Hq and by the chunks per sequence)
@pytest.mark.parametrize("saved", [False, True])
@pytest.mark.parametrize("hq,hv", [(3, 3), (3, 6), (5, 10)])
def test_head_counts_not_powers_of_two(hq, hv, saved):
    check_bwd(custom(B=3, T=201, Hq=hq, Hv=hv, host_l2=False), kernel_l2=True, saved=saved)
    check_bwd(custom(seq_lens=(65, 0, 7, 130), Hq=hq, Hv=hv), kernel_l2=False, saved=saved)
