"""Varlen chunk tables on the GPU (gdr_prepare_chunks, through the C ABI) against the oracle, bit for bit.

The tables are the FlashQLA documentation page's utilities (prepare_lens, prepare_chunk_offsets,
prepare_chunk_indices): integers, so every entry must match exactly.  The malformed-input paths latch an
error code in the device error word and write nothing but a zero total.
"""

import ctypes
import json
import os

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_38_gb300 import _lib

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = json.load(open(os.path.join(HERE, "golden", "chunk_tables.json")))["cases"]


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


SENTINEL = -7


def call(cu, chunk, total_tokens, max_chunks):
    """Run gdr_prepare_chunks; returns (status, idx, off, total) with the table pre-filled by a sentinel."""
    lib = _lib.load()
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    N = len(cu) - 1
    idx = torch.full((max(max_chunks, 1), 2), SENTINEL, dtype=torch.int32, device="cuda")
    off = torch.full((N + 1,), SENTINEL, dtype=torch.int32, device="cuda")
    tot = torch.full((1,), SENTINEL, dtype=torch.int32, device="cuda")
    st = lib.gdr_prepare_chunks(_p(cu_d), N, total_tokens, chunk, _p(idx), max_chunks, _p(off), _p(tot), _stream())
    torch.cuda.synchronize()
    return st, idx.cpu().numpy(), off.cpu().numpy(), int(tot.item())


def bound(cu, chunk):
    return (cu[-1] + (len(cu) - 1) * (chunk - 1)) // chunk


def check_exact(cu, chunk, with_total):
    mc = bound(cu, chunk)
    st, idx, off, tot = call(cu, chunk, cu[-1] if with_total else -1, mc)
    assert st == 0
    assert lib_error() == 0
    want_off, want_tot = oracle.prepare_chunk_offsets(cu, chunk)
    want_idx = np.array(oracle.prepare_chunk_indices(cu, chunk), dtype=np.int64).reshape(-1, 2)
    assert tot == want_tot
    assert off.tolist() == list(want_off)
    assert np.array_equal(idx[:tot], want_idx)
    assert (idx[tot:] == SENTINEL).all()   # rows past the total are left untouched
    return idx, off, tot


def lib_error():
    return int(_lib.load().gdr_get_error(_stream()))


@pytest.mark.parametrize("with_total", [True, False])
@pytest.mark.parametrize("case", range(len(GOLDEN)))
def test_golden_tables(case, with_total):
    c = GOLDEN[case]
    idx, off, tot = check_exact(c["cu_seqlens"], c["chunk_size"], with_total)
    assert tot == c["total_chunks"]
    assert off.tolist() == c["chunk_offsets"]
    if "chunk_indices" in c:
        assert idx[:tot].tolist() == c["chunk_indices"]


@pytest.mark.parametrize("chunk", [1, 2, 7, 64, 128])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_tables_with_empty_and_single_token_sequences(chunk, seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 3000))
    lens = rng.integers(0, 300, size=n)
    lens[rng.random(n) < 0.2] = 0       # empty sequences
    lens[rng.random(n) < 0.2] = 1       # single tokens
    cu = [0] + np.cumsum(lens).tolist()
    for with_total in (True, False):
        check_exact(cu, chunk, with_total)


def test_prepare_chunks_binding_sizes_the_table_without_total():
    """The Python binding without total_tokens sizes the table from cu_seqlens[-1] (no truncation)."""
    import gated_delta_rule_38_gb300 as gdr
    cu = [0, 512, 1536, 2304, 5304, 5311]
    idx, off, tot = gdr.prepare_chunks(torch.tensor(cu, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    want = oracle.prepare_chunk_indices(cu, 64)
    assert int(tot.item()) == 84 and idx.shape[0] >= 84
    assert idx[:84].cpu().tolist() == want
    assert off.cpu().tolist() == [0, 8, 24, 36, 83, 84]


@pytest.mark.parametrize("cu,total_tokens", [
    ([0, 5, 3, 9], 9),          # decreasing
    ([0, 5, 9], 10),            # last entry != T
    ([2, 5, 9], 9),             # not starting at 0
    ([0, 5, 3, 9], -1),         # decreasing, without the total check
])
def test_malformed_cu_seqlens_latch_error(cu, total_tokens):
    assert lib_error() == 0
    st, idx, off, tot = call(cu, 4, total_tokens, 64)
    assert st == 0                       # the host cannot see the device array: the kernel reports it
    assert lib_error() == 8              # GDR_ERR_CUSEQLENS
    assert lib_error() == 0              # reading clears the word
    assert tot == 0
    assert (idx == SENTINEL).all() and (off == SENTINEL).all()   # nothing else written


def test_table_too_small_latches_shape_error():
    """With total_tokens = -1 the host cannot bound the table; the kernel counts first and refuses."""
    cu = [0, 100, 300]
    st, idx, off, tot = call(cu, 64, -1, 3)        # needs 2 + 4 = 6 rows
    assert st == 0
    assert lib_error() == 2              # GDR_ERR_SHAPE
    assert tot == 0 and (idx == SENTINEL).all() and (off == SENTINEL).all()
    # the host-side bound check with the total given
    lib = _lib.load()
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    buf = torch.zeros(16, dtype=torch.int32, device="cuda")
    assert lib.gdr_prepare_chunks(_p(cu_d), 2, 300, 64, _p(buf), 3, _p(buf), _p(buf), _stream()) == 2


@pytest.mark.parametrize("cu", [[0, 70, 40, 200], [0, 70, 150, 180]], ids=["decreasing", "last_entry_short"])
@pytest.mark.parametrize("saved", [False, True])
def test_malformed_cu_seqlens_in_forward_and_backward(cu, saved):
    """The forward and backward with a malformed cu_seqlens latch GDR_ERR_CUSEQLENS: their kernels treat
    every sequence as empty (the final states equal the initial ones, dh0 equals dht, nothing is read or
    written past the tables), and the next call with a valid cu_seqlens matches the oracle."""
    import gated_delta_rule_38_gb300 as gdr
    from gated_delta_rule_38_gb300.inputs import custom, make_inputs
    from harness import TOL, np64, oracle_problem, rel_l2, to_dev
    w = custom(seq_lens=(70, 60, 70), Hq=2, Hv=2, host_l2=False)
    x = make_inputs(w)
    d = to_dev(x)
    bad = torch.tensor(cu, dtype=torch.int32, device="cuda")
    assert gdr.get_error() == 0
    sv = gdr.saved_buffer(d["q"], d["v"], d["g"], cu_seqlens=bad, use_qk_l2norm_in_kernel=True) if saved else None
    gcs, A, o, _, fin = gdr.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                                       initial_state=d["h0"], cu_seqlens=bad,
                                                       use_qk_l2norm_in_kernel=True, saved=sv)
    assert gdr.get_error() == 8                    # GDR_ERR_CUSEQLENS
    assert torch.equal(fin, d["h0"])               # every sequence empty: the states pass through
    grads = gdr.chunk_gated_delta_rule_bwd(d["q"], d["k"], d["v"], gcs, d["beta"], A, d["do"], dht=d["dht"],
                                           initial_state=d["h0"], cu_seqlens=bad, use_qk_l2norm_in_kernel=True,
                                           saved=sv)
    assert gdr.get_error() == 8
    assert torch.equal(grads[5], d["dht"])
    # the context is intact: a valid call next
    good = torch.tensor(w.cu_seqlens, dtype=torch.int32, device="cuda")
    _, _, o, _, fin = gdr.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], initial_state=d["h0"],
                                                     cu_seqlens=good, use_qk_l2norm_in_kernel=True)
    torch.cuda.synchronize()
    assert gdr.get_error() == 0
    ref = oracle.fwd(oracle_problem(w, True), x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"])
    assert rel_l2(np64(o), ref["o"]) <= TOL and rel_l2(np64(fin), ref["final_state"]) <= TOL
