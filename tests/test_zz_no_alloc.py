"""The allocation-free forward (gdr_fwd_noalloc) against the workspace forward (gdr_fwd).

gdr_fwd_noalloc serves callers that may not allocate device memory: it runs the
forward on a scratch array built into the library instead of a caller workspace.
These tests call both entry points through the C ABI on the same inputs and
require the same outputs, on two calls in a row (the second call must not be
disturbed by what the first left in the shared scratch).  This file is collected
last so that a run stopping at the first failure has run every other test.
"""

import ctypes

import pytest
import torch

import gated_delta_rule_38_gb300 as gdr
from gated_delta_rule_38_gb300 import _lib
from gated_delta_rule_38_gb300.inputs import custom, make_inputs
from harness import TOL, np64, rel_l2


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _inputs(seed, w):
    x = make_inputs(w, seed=seed)
    return {k: (v.cuda() if v is not None else None) for k, v in x.items()}


def _run_both(lib, w, x, cu, l2):
    pb = gdr.problem(x["q"], x["v"], x["g"], None, cu, l2)
    o_ref = torch.empty_like(x["v"])
    fin_ref = torch.empty(x["h0"].shape, dtype=torch.float32, device="cuda")
    nbytes = gdr.workspace_bytes(pb, False)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device="cuda")
    st = lib.gdr_fwd(ctypes.byref(pb), _p(x["q"]), _p(x["k"]), _p(x["v"]), _p(x["g"]), _p(x["beta"]), _p(x["h0"]),
                     _p(o_ref), _p(fin_ref), None, None, None, _p(ws), nbytes, _stream())
    assert st == 0, _lib.status_string(st)
    o = torch.full_like(x["v"], float("nan"))
    fin = torch.full_like(fin_ref, float("nan"))
    st = lib.gdr_fwd_noalloc(ctypes.byref(pb), _p(x["q"]), _p(x["k"]), _p(x["v"]), _p(x["g"]), _p(x["beta"]),
                             _p(x["h0"]), _p(o), _p(fin), _stream())
    assert st == 0, _lib.status_string(st)
    torch.cuda.synchronize()
    assert rel_l2(np64(o), np64(o_ref)) <= TOL
    assert rel_l2(np64(fin), np64(fin_ref)) <= TOL


@pytest.mark.gpu
def test_no_alloc_forward_matches_workspace_forward_twice():
    lib = _lib.load()
    w = custom(B=2, T=300, Hq=2, Hv=4, host_l2=False)
    _run_both(lib, w, _inputs(1, w), None, True)
    # a second call, on different (packed, variable-length) inputs, after the first left its scratch behind
    w2 = custom(seq_lens=(130, 7, 0, 260), Hq=2, Hv=2)
    cu = torch.tensor(w2.cu_seqlens, dtype=torch.int32, device="cuda")
    _run_both(lib, w2, _inputs(2, w2), cu, False)


def _big_problem():
    """A forward whose workspace (about 70 MB: 262,144 token-heads x 268 bytes) exceeds the 64 MiB scratch."""
    p = _lib.Problem()
    p.B, p.T, p.Hq, p.Hv, p.K, p.V = 1, 16384, 16, 16, 128, 128
    p.dtype = p.gate_dtype = _lib.GDR_BF16
    p.scale = 128 ** -0.5
    p.cu_seqlens = None
    p.num_seqs = 0
    p.flags = 0
    p.num_segments = 1
    return p


def test_no_alloc_rejects_problems_beyond_its_scratch_without_gpu():
    """A forward whose workspace exceeds the built-in scratch is refused on the host (made-up addresses,
    so only on a machine without a GPU)."""
    if torch.cuda.is_available():
        pytest.skip("the GPU variant below uses real buffers")
    from gated_delta_rule_38_gb300 import build as gbuild
    gbuild.build()
    lib = _lib.load()
    p = _big_problem()
    P = ctypes.c_void_p(0x100000)
    assert lib.gdr_fwd_noalloc(ctypes.byref(p), P, P, P, P, P, None, P, None, None) == 7


@pytest.mark.gpu
def test_no_alloc_rejects_problems_beyond_its_scratch():
    """The same refusal with real buffers of the problem's sizes."""
    lib = _lib.load()
    p = _big_problem()
    x = torch.zeros(1, 16384, 16, 128, dtype=torch.bfloat16, device="cuda")
    gb = torch.zeros(1, 16384, 16, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(x)
    assert lib.gdr_fwd_noalloc(ctypes.byref(p), _p(x), _p(x), _p(x), _p(gb), _p(gb), None, _p(o), None,
                               _stream()) == 7


@pytest.mark.gpu
def test_no_alloc_allocates_nothing_and_runs_the_split_layout():
    """After a first (set-up) call, further calls leave the device's free memory unchanged; a problem that
    runs the intra-GPU sequence split (two segments: its own workspace layout) still fits the scratch."""
    lib = _lib.load()
    w = custom(B=1, T=1000, Hq=2, Hv=2)
    x = _inputs(3, w)
    pb = gdr.problem(x["q"], x["v"], x["g"], None, None, False, num_segments=2)
    nbytes = gdr.workspace_bytes(pb, False)
    assert 0 < nbytes <= 64 << 20
    o_ref = torch.empty_like(x["v"])
    fin_ref = torch.empty(x["h0"].shape, dtype=torch.float32, device="cuda")
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    st = lib.gdr_fwd(ctypes.byref(pb), _p(x["q"]), _p(x["k"]), _p(x["v"]), _p(x["g"]), _p(x["beta"]),
                     _p(x["h0"]), _p(o_ref), _p(fin_ref), None, None, None, _p(ws), nbytes, _stream())
    assert st == 0
    o = torch.empty_like(x["v"])
    fin = torch.empty_like(fin_ref)

    def call():
        s = lib.gdr_fwd_noalloc(ctypes.byref(pb), _p(x["q"]), _p(x["k"]), _p(x["v"]), _p(x["g"]), _p(x["beta"]),
                                _p(x["h0"]), _p(o), _p(fin), _stream())
        assert s == 0, _lib.status_string(s)
        torch.cuda.synchronize()

    call()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        call()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert rel_l2(np64(o), np64(o_ref)) <= TOL
    assert rel_l2(np64(fin), np64(fin_ref)) <= TOL
