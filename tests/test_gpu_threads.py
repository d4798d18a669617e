"""Calls from a host thread that has made no CUDA call of its own (a framework's worker thread, such as the
autograd engine's): the library makes the device's primary context current before it builds its TMA
tensor maps (a driver call that needs one), so the C-ABI calls succeed there and give, bit for bit, what
the same calls give on the main thread.  Every buffer is allocated on the main thread, so the worker
thread's first CUDA call is the library's."""

import ctypes
import threading

import pytest
import torch

import gated_delta_rule_38_gb300 as gdr
from gated_delta_rule_38_gb300 import _lib

pytestmark = pytest.mark.gpu

B, T, H, D = 2, 100, 2, 128


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_first_call_of_a_fresh_thread():
    lib = _lib.load()
    gen = torch.Generator(device="cuda").manual_seed(3)
    r = lambda *s: torch.randn(*s, device="cuda", generator=gen)
    q, k, v, do = (r(B, T, H, D).bfloat16() for _ in range(4))
    g = torch.nn.functional.logsigmoid(r(B, T, H) + 2).bfloat16()
    beta = torch.sigmoid(r(B, T, H)).bfloat16()
    p = gdr.problem(q, v, g, use_qk_l2norm_in_kernel=True)
    saved = gdr.saved_buffer(q, v, g, use_qk_l2norm_in_kernel=True)
    o, A = torch.empty_like(v), torch.empty(B, T, H, 64, dtype=q.dtype, device="cuda")
    gcs = torch.empty(B, T, H, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dg, db = torch.empty_like(beta), torch.empty_like(beta)
    nf, nb = gdr.workspace_bytes(p, False, saved), gdr.workspace_bytes(p, True, saved)
    wf = torch.empty(max(nf, 1), dtype=torch.uint8, device="cuda")
    wb = torch.empty(max(nb, 1), dtype=torch.uint8, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def step():
        st_f = lib.gdr_fwd_ex(ctypes.byref(p), _p(q), _p(k), _p(v), _p(g), _p(beta), None, _p(o), None, _p(gcs),
                              _p(A), None, _p(wf), nf, _p(saved), stream)
        st_b = lib.gdr_bwd_ex(ctypes.byref(p), _p(q), _p(k), _p(v), _p(gcs), _p(beta), _p(A), _p(do), None, None,
                              _p(dq), _p(dk), _p(dv), _p(dg), _p(db), None, _p(wb), nb, _p(saved), stream)
        return st_f, st_b

    assert step() == (0, 0)
    torch.cuda.synchronize()
    want = [t.clone() for t in (o, A, gcs, dq, dk, dv, dg, db)]
    for t in (o, A, gcs, dq, dk, dv, dg, db):
        t.fill_(float("nan"))
    torch.cuda.synchronize()
    result = {}

    def worker():
        result["status"] = step()
        if result["status"] != (0, 0):
            result["why"] = _lib.last_cuda_error()

    th = threading.Thread(target=worker)
    th.start()
    th.join()
    assert result["status"] == (0, 0), result
    torch.cuda.synchronize()
    assert gdr.get_error() == 0
    for a, b in zip(want, (o, A, gcs, dq, dk, dv, dg, db)):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
