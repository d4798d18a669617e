"""The C ABI without a GPU: the library loads, exports every declared symbol,
and rejects bad arguments on the host before touching a device.

The rejection cases mirror the FlashQLA backend verifier's branches (PR #998
"[GDN] Add FlashQLA backend dispatch": K != 128, V != 128, gate or beta
activation in the kernel, negative eigenvalues, inter-card CP, fp32 inputs).
"""

import ctypes
import os
import re

import pytest

from gated_delta_rule_38_gb300 import _lib
from gated_delta_rule_38_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return _lib.load()


@pytest.fixture
def fake_ptrs():
    """Tests that pass made-up device addresses to check host-side rejections run only without a GPU:
    there no call can reach a kernel, whatever order the host checks take (the GPU tests make real calls)."""
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("made-up device addresses are only passed on machines without a GPU")
    except ImportError:
        pass


def prob(**kw):
    p = _lib.Problem()
    p.B, p.T, p.Hq, p.Hv, p.K, p.V = 2, 256, 4, 4, 128, 128
    p.dtype = _lib.GDR_BF16
    p.gate_dtype = _lib.GDR_BF16
    p.scale = 128 ** -0.5
    p.cu_seqlens = None
    p.num_seqs = 0
    p.flags = 0
    p.num_segments = 0
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def test_exports_match_header(lib):
    hdr = open(os.path.join(ROOT, "include", "gdr.h")).read()
    declared = set(re.findall(r"^\s*(?:[\w\s\*]+?)\b(gdr_\w+)\s*\(", hdr, flags=re.M))
    assert declared == set(_lib.EXPORTS)
    for name in _lib.EXPORTS:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(12):
        s = lib.gdr_status_string(code)
        assert s and len(s) > 1
    assert lib.gdr_version() >= 100


def fwd_call(lib, p, ptr=0x100000, ws=0x200000, ws_bytes=1 << 40, **over):
    args = dict(q=ptr, k=ptr, v=ptr, g=ptr, beta=ptr, h0=None, o=ptr, fin=None, gcs=None, A=None, h=None)
    args.update(over)
    return lib.gdr_fwd(ctypes.byref(p), args["q"], args["k"], args["v"], args["g"], args["beta"], args["h0"],
                       args["o"], args["fin"], args["gcs"], args["A"], args["h"], ws, ws_bytes, None)


@pytest.mark.parametrize("field,value,status", [
    ("K", 60, 2), ("K", 256, 2), ("V", 4, 2), ("V", 0, 2), ("Hv", 6, 2), ("T", -1, 2), ("B", 0, 2),
    ("dtype", _lib.GDR_FP32, 3), ("gate_dtype", _lib.GDR_FP16, 3),
    ("flags", _lib.GDR_INTER_CARD_CP, 4), ("flags", 1 << 20, 4),
])
def test_verifier_rejections(lib, fake_ptrs, field, value, status):
    p = prob(**{field: value})
    assert fwd_call(lib, p) == status
    n = ctypes.c_size_t()
    assert lib.gdr_fwd_workspace_size(ctypes.byref(p), ctypes.byref(n)) == status


def test_packed_batch_needs_single_row(lib, fake_ptrs):
    p = prob(cu_seqlens=0x100000, num_seqs=3)
    assert fwd_call(lib, p) == 2
    p = prob(B=1, cu_seqlens=0x100000, num_seqs=0)
    assert fwd_call(lib, p) == 2


def test_null_align_workspace(lib, fake_ptrs):
    p = prob()
    assert fwd_call(lib, p, q=None) == 1
    assert fwd_call(lib, p, o=None) == 1
    assert fwd_call(lib, p, k=0x100008) == 6
    assert fwd_call(lib, p, ws=None) == 7
    assert fwd_call(lib, p, ws_bytes=16) == 7
    assert fwd_call(lib, p, ws=0x200010) == 6


def test_valid_call_without_gpu_never_succeeds(lib):
    """On a machine without a usable sm_103a device a valid call fails loudly."""
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("a GPU is present")
    except ImportError:
        pass
    assert fwd_call(lib, prob()) in (5, 10)


def test_workspace_sizes_and_max_chunks(lib):
    p = prob(B=2, T=4096, Hq=32, Hv=32)
    assert lib.gdr_max_chunks(ctypes.byref(p)) == 128
    n = ctypes.c_size_t()
    assert lib.gdr_fwd_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 0
    tok = 2 * 4096 * 32
    assert n.value >= tok * 4 + tok * 64 * 2
    assert lib.gdr_bwd_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 0
    assert n.value >= 2 * 128 * 32 * 128 * 128 * 2
    pv = prob(B=1, T=5311, Hq=32, Hv=32, cu_seqlens=0x100000, num_seqs=5)
    assert lib.gdr_max_chunks(ctypes.byref(pv)) == (5311 + 5 * 63) // 64


def test_prepare_chunks_host_checks(lib, fake_ptrs):
    P = 0x100000
    # table too small for the bound (T + N*(C-1)) / C
    assert lib.gdr_prepare_chunks(P, 2, 8, 2, P, 4, P, P, None) == 2
    assert lib.gdr_prepare_chunks(None, 2, 8, 2, P, 5, P, P, None) == 1
    assert lib.gdr_prepare_chunks(P, 0, 8, 2, P, 5, P, P, None) == 2


def test_saved_buffer_size_and_exclusive_states(lib, fake_ptrs):
    """The saved buffer holds P, the q/k norms, the per-chunk states and Delta; it excludes an h output."""
    p = prob(B=2, T=4096, Hq=32, Hv=32)
    n = ctypes.c_size_t()
    assert lib.gdr_saved_bytes(ctypes.byref(p), ctypes.byref(n)) == 0
    tok, rows = 2 * 4096 * 32, 128 * 32
    assert n.value == tok * 64 * 2 + 2 * tok * 4 + rows * 128 * 128 * 2 + rows * 64 * 128 * 2
    P = 0x100000
    st = lib.gdr_fwd_ex(ctypes.byref(p), P, P, P, P, P, None, P, None, None, None, P, 0x200000, 1 << 40, P, None)
    assert st == 4
    # the intra-GPU split keeps the same parts (its forward stores the states for its backward too) and the
    # segments' transfer matrices (1 sequence x 16 heads x 4 segments x 128 x 128 fp32)
    ps = prob(B=1, T=65536, Hq=16, Hv=16, num_segments=4)
    assert lib.gdr_saved_bytes(ctypes.byref(ps), ctypes.byref(n)) == 0
    tok, rows = 65536 * 16, 1024 * 16
    assert n.value == tok * 64 * 2 + 2 * tok * 4 + rows * 128 * 128 * 2 + rows * 64 * 128 * 2 + 16 * 4 * 128 * 128 * 4
    st = lib.gdr_fwd_ex(ctypes.byref(ps), P, P, P, P, P, None, P, None, None, None, P, 0x200000, 1 << 40, P, None)
    assert st == 4


def test_binding_rejects_states_with_saved():
    import torch
    import gated_delta_rule_38_gb300 as gdr
    x = torch.zeros(1, 64, 1, 128, dtype=torch.bfloat16)
    g = torch.zeros(1, 64, 1)
    with pytest.raises(ValueError):
        gdr.chunk_gated_delta_rule_fwd(x, x, x, g, g, output_h=True, saved=torch.zeros(16, dtype=torch.uint8))


def test_saved_workspace_sizes(lib):
    """With a saved buffer the workspaces leave out what the buffer holds (P and norms; states and Delta)."""
    p = prob(B=2, T=4096, Hq=32, Hv=32, flags=_lib.GDR_L2NORM_QK)
    n, m = ctypes.c_size_t(), ctypes.c_size_t()
    tok, rows = 2 * 4096 * 32, 128 * 32
    for backward in (0, 1):
        full = lib.gdr_bwd_workspace_size if backward else lib.gdr_fwd_workspace_size
        assert full(ctypes.byref(p), ctypes.byref(n)) == 0
        assert lib.gdr_saved_workspace_size(ctypes.byref(p), backward, ctypes.byref(m)) == 0
        kept = tok * 64 * 2 + 2 * tok * 4 + (rows * 128 * 128 * 2 + rows * 64 * 128 * 2 if backward else 0)
        assert n.value - m.value == kept
    # the intra-GPU split (no in-kernel L2 norm): the forward leaves out P; the backward, whose recompute
    # without the buffer needs no P, leaves out the states and Delta
    ps = prob(B=1, T=65536, Hq=16, Hv=16, num_segments=4)
    tok, rows = 65536 * 16, 1024 * 16
    for backward in (0, 1):
        full = lib.gdr_bwd_workspace_size if backward else lib.gdr_fwd_workspace_size
        assert full(ctypes.byref(ps), ctypes.byref(n)) == 0
        assert lib.gdr_saved_workspace_size(ctypes.byref(ps), backward, ctypes.byref(m)) == 0
        kept = rows * 128 * 128 * 2 + rows * 64 * 128 * 2 if backward else tok * 64 * 2
        assert n.value - m.value == kept
    assert lib.gdr_saved_workspace_size(ctypes.byref(prob(K=60)), 1, ctypes.byref(m)) == 2


def test_decode_host_checks(lib, fake_ptrs):
    """gdr_decode validates its arguments on the host before touching a device."""
    P = 0x100000

    def dec(p, q=P, out=P, o=P):
        return lib.gdr_decode(ctypes.byref(p), q, P, P, P, P, None, out, o, None)

    assert dec(prob(T=1, cu_seqlens=P, B=1, num_seqs=2)) == 4   # packed rows: not a decode layout
    assert dec(prob(T=1, K=72, V=256)) == 2
    assert dec(prob(T=1), out=None) == 1
    assert dec(prob(T=1), o=None) == 1
    assert dec(prob(T=1), q=0x100008) == 6
    assert dec(prob(T=1, dtype=_lib.GDR_FP32)) == 3
    # a valid call (T = 0 needs only the state) reaches the device check; only without a GPU, since the
    # pointers here are not device memory
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except ImportError:
        has_gpu = False
    if not has_gpu:
        assert dec(prob(T=0), q=None, o=None) in (5, 10)


def test_activation_options_are_accepted_and_the_gate_backward_needs_saved(lib, fake_ptrs):
    """The gate / beta activation options pass the host checks; the in-kernel gate's backward without the
    forward's saved buffer is refused (the activation's derivative lives there)."""
    n = ctypes.c_size_t()
    act = _lib.GDR_GATE_IN_KERNEL | _lib.GDR_BETA_SIGMOID_IN_KERNEL | _lib.GDR_ALLOW_NEG_EIGVAL
    p = prob(flags=act)
    assert lib.gdr_fwd_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 0
    assert lib.gdr_saved_bytes(ctypes.byref(p), ctypes.byref(n)) == 0 and n.value > 0
    # the gate activation's derivative (tokens x Hv fp32) comes first, then the parts of the plain buffer
    ps = prob(B=1, T=65536, Hq=16, Hv=16, num_segments=4, flags=_lib.GDR_GATE_IN_KERNEL)
    m = ctypes.c_size_t()
    assert lib.gdr_saved_bytes(ctypes.byref(prob(B=1, T=65536, Hq=16, Hv=16, num_segments=4)), ctypes.byref(m)) == 0
    assert lib.gdr_saved_bytes(ctypes.byref(ps), ctypes.byref(n)) == 0 and n.value == m.value + 65536 * 16 * 4
    P = 0x100000
    st = lib.gdr_bwd(ctypes.byref(p), P, P, P, P, P, P, P, None, None, P, P, P, P, P, None, 0x200000, 1 << 40, None)
    assert st == 4


def test_smaller_head_dims_run_padded(lib):
    """K or V below 128 are accepted; their workspaces hold zero-padded copies on top of the 128-wide ones."""
    n, m = ctypes.c_size_t(), ctypes.c_size_t()
    p128 = prob(B=2, T=256, Hq=4, Hv=4)
    p64 = prob(B=2, T=256, Hq=4, Hv=4, K=64, V=64)
    for backward, fn in ((0, lib.gdr_fwd_workspace_size), (1, lib.gdr_bwd_workspace_size)):
        assert fn(ctypes.byref(p128), ctypes.byref(n)) == 0
        assert fn(ctypes.byref(p64), ctypes.byref(m)) == 0
        assert m.value > n.value
    assert lib.gdr_saved_bytes(ctypes.byref(p64), ctypes.byref(m)) == 0
    assert lib.gdr_saved_bytes(ctypes.byref(p128), ctypes.byref(n)) == 0 and m.value == n.value
