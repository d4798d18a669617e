"""GB300-native chunked Gated Delta Rule.

Python surface of the C library declared in ``include/gdr.h``.  Every step of
the computation runs in the library's CUDA kernels; this module only
allocates outputs with PyTorch, marshals pointers and passes the current CUDA
stream.  There is no CPU fallback: without the built library every call
raises.

API (shapes follow the FlashQLA skill page, "Core API" / "Low-Level API"):

* ``chunk_gated_delta_rule_fwd(q, k, v, g, beta, ...) -> (g_cumsum, A, o, h, final_state)``
* ``chunk_gated_delta_rule_bwd(q, k, v, g_cumsum, beta, A, do, ...) -> (dq, dk, dv, dbeta, dg, dh0)``
* ``chunk_gated_delta_rule(q, k, v, g, beta, ...) -> (o, final_state)`` (autograd)
* ``prepare_chunks(cu_seqlens, chunk_size=64) -> (chunk_indices, chunk_offsets, total_chunks)``
"""

from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _lib

__all__ = ["chunk_gated_delta_rule", "chunk_gated_delta_rule_fwd", "chunk_gated_delta_rule_bwd", "saved_buffer",
           "recurrent_gated_delta_rule", "prepare_chunks", "GdrError", "problem", "workspace_bytes"]

GdrError = _lib.GdrError

_DT = {torch.bfloat16: _lib.GDR_BF16, torch.float16: _lib.GDR_FP16, torch.float32: _lib.GDR_FP32}


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(t, name, shape=None, dtype=None, like=None, optional=False, contiguous=True):
    """The library reads and writes every tensor through a raw device pointer as a contiguous row-major array
    of the problem's shape: anything else is refused here, before a kernel could read past its end."""
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if like is not None and t.device != like.device:
        raise ValueError(f"{name} is on {t.device}, the other tensors on {like.device}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check_tokens(q, k, v, g=None, beta=None):
    """q, k [B,T,Hq,K] and v [B,T,Hv,V] of one dtype; g, beta [B,T,Hv] of one dtype."""
    _check(q, "q")
    if q.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k and v must be [B, T, H, D]")
    B, T = q.shape[0], q.shape[1]
    _check(k, "k", q.shape, q.dtype, q)
    _check(v, "v", (B, T) + tuple(v.shape[2:]), q.dtype, q)
    if g is not None or beta is not None:
        _check(g, "g", (B, T, v.shape[2]), None, q)
        _check(beta, "beta", (B, T, v.shape[2]), g.dtype, q)


def _check_state(t, name, p, v_first, like):
    # (states are copied to contiguous fp32 by the callers below when they are not already)
    if t is not None:
        _check(t, name, _state_shape(p, v_first), None, like, contiguous=False)


def _check_cu(cu, q):
    if cu is not None:
        _check(cu, "cu_seqlens", (cu.numel(),), torch.int32, q)
        if q.shape[0] != 1:
            raise ValueError("a packed batch (cu_seqlens) has B = 1")


def _check_saved(saved, p, q):
    if saved is None:
        return
    _check(saved, "saved", None, torch.uint8, q)
    n = ctypes.c_size_t(0)
    _lib.check(_lib.load().gdr_saved_bytes(ctypes.byref(p), ctypes.byref(n)), "gdr_saved_bytes")
    if saved.numel() < n.value:
        raise ValueError(f"saved holds {saved.numel()} bytes, this problem needs {n.value} (saved_buffer)")


def problem(q, v, g, scale=None, cu_seqlens=None, use_qk_l2norm_in_kernel=False, state_v_first=False,
            num_segments=0, extra_flags=0, use_gate_in_kernel=False, use_beta_sigmoid_in_kernel=False,
            allow_neg_eigval=False) -> _lib.Problem:
    """The gdr_problem struct describing a call with these tensors."""
    B, T, Hq, K = q.shape
    Hv, V = v.shape[2], v.shape[3]
    flags = extra_flags
    if use_qk_l2norm_in_kernel:
        flags |= _lib.GDR_L2NORM_QK
    if state_v_first:
        flags |= _lib.GDR_STATE_V_FIRST
    if use_gate_in_kernel:
        flags |= _lib.GDR_GATE_IN_KERNEL
    if use_beta_sigmoid_in_kernel:
        flags |= _lib.GDR_BETA_SIGMOID_IN_KERNEL
    if allow_neg_eigval:
        flags |= _lib.GDR_ALLOW_NEG_EIGVAL
    p = _lib.Problem()
    p.B, p.T, p.Hq, p.Hv, p.K, p.V = B, T, Hq, Hv, K, V
    p.dtype = _DT.get(q.dtype, 99)
    p.gate_dtype = _DT.get(g.dtype, 99)
    p.scale = float(K ** -0.5 if scale is None else scale)
    if cu_seqlens is not None:
        p.cu_seqlens = cu_seqlens.data_ptr()
        p.num_seqs = cu_seqlens.numel() - 1
    else:
        p.cu_seqlens = None
        p.num_seqs = 0
    p.flags = flags
    p.num_segments = int(num_segments)
    return p


def workspace_bytes(p: _lib.Problem, backward: bool, saved=None) -> int:
    """Workspace bytes of the forward or backward (smaller with a saved buffer, which holds some parts)."""
    lib = _lib.load()
    n = ctypes.c_size_t(0)
    if saved is not None:
        _lib.check(lib.gdr_saved_workspace_size(ctypes.byref(p), int(backward), ctypes.byref(n)),
                   "gdr_saved_workspace_size")
        return int(n.value)
    fn = lib.gdr_bwd_workspace_size if backward else lib.gdr_fwd_workspace_size
    _lib.check(fn(ctypes.byref(p), ctypes.byref(n)), fn.__name__)
    return int(n.value)


def _state_shape(p, v_first):
    N = p.num_seqs if p.cu_seqlens else p.B
    return (N, p.Hv, p.V, p.K) if v_first else (N, p.Hv, p.K, p.V)


def _cu(cu_seqlens):
    if cu_seqlens is None:
        return None
    if cu_seqlens.dtype != torch.int32:
        cu_seqlens = cu_seqlens.to(torch.int32)
    return cu_seqlens.contiguous()


def saved_buffer(q, v, g, scale=None, cu_seqlens=None, use_qk_l2norm_in_kernel=False, state_v_first=False,
                 num_segments=0, **act):
    """A device buffer for what the forward keeps for the backward (``saved=`` of the forward and backward
    below): the decayed causal blocks, the q/k norms, the state before every chunk and Delta of every chunk,
    and with ``use_gate_in_kernel`` the gate activation's derivative.  ``act``: the activation options."""
    lib = _lib.load()
    p = problem(q, v, g, scale, _cu(cu_seqlens), use_qk_l2norm_in_kernel, state_v_first, num_segments, **act)
    n = ctypes.c_size_t(0)
    _lib.check(lib.gdr_saved_bytes(ctypes.byref(p), ctypes.byref(n)), "gdr_saved_bytes")
    return torch.empty(int(n.value), dtype=torch.uint8, device=q.device) if n.value else None


def chunk_gated_delta_rule_fwd(q, k, v, g, beta, scale=None, initial_state=None, output_final_state=True,
                               cu_seqlens=None, use_qk_l2norm_in_kernel=False, state_v_first=False,
                               num_segments=0, output_h=False, save_for_backward=True, out=None, saved=None,
                               use_gate_in_kernel=False, use_beta_sigmoid_in_kernel=False, allow_neg_eigval=False):
    """Forward.  Returns (g_cumsum, A, o, h, final_state); h is None unless output_h.

    g_cumsum and A are None when save_for_backward is False.  For packed
    batches h has gdr_max_chunks rows; rows past the true chunk count are unused.
    ``saved`` (from saved_buffer) receives the decayed causal blocks, q/k norms, states and Delta for the
    backward; it excludes ``output_h`` (the states then live in ``saved``).  With ``use_gate_in_kernel`` g
    holds raw gate logits (the recurrence uses logsigmoid(g)); with ``use_beta_sigmoid_in_kernel`` beta holds
    raw logits (sigmoid(beta)); ``allow_neg_eigval`` doubles beta.
    """
    if output_h and saved is not None:
        raise ValueError("output_h and saved are exclusive: with saved, the states are kept in the saved buffer")
    _check_tokens(q, k, v, g, beta)
    lib = _lib.load()
    cu = _cu(cu_seqlens)
    _check_cu(cu, q)
    p = problem(q, v, g, scale, cu, use_qk_l2norm_in_kernel, state_v_first, num_segments,
                use_gate_in_kernel=use_gate_in_kernel, use_beta_sigmoid_in_kernel=use_beta_sigmoid_in_kernel,
                allow_neg_eigval=allow_neg_eigval)
    _check_state(initial_state, "initial_state", p, state_v_first, q)
    _check(out, "out", v.shape, v.dtype, q, optional=True)
    _check_saved(saved, p, q)
    dev = q.device
    B, T, Hv, V = v.shape
    o = out if out is not None else torch.empty_like(v)
    fin = torch.empty(_state_shape(p, state_v_first), dtype=torch.float32, device=dev) if output_final_state else None
    gcs = A = None
    if save_for_backward:
        gcs = torch.empty((B, T, Hv), dtype=torch.float32, device=dev)
        A = torch.empty((B, T, Hv, _lib.GDR_CHUNK), dtype=q.dtype, device=dev)
    h = None
    if output_h:
        rows = int(lib.gdr_max_chunks(ctypes.byref(p)))
        h = torch.empty((rows, Hv) + _state_shape(p, state_v_first)[2:], dtype=q.dtype, device=dev)
    nbytes = workspace_bytes(p, False, saved)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    h0 = None if initial_state is None else initial_state.to(torch.float32).contiguous()
    st = lib.gdr_fwd_ex(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(o),
                        _ptr(fin), _ptr(gcs), _ptr(A), _ptr(h), _ptr(ws), nbytes, _ptr(saved), _stream(dev))
    _lib.check(st, "gdr_fwd_ex")
    return gcs, A, o, h, fin


def recurrent_gated_delta_rule(q, k, v, g, beta, scale=None, initial_state=None, use_qk_l2norm_in_kernel=False,
                               state_v_first=False, inplace=False, out=None, use_gate_in_kernel=False,
                               use_beta_sigmoid_in_kernel=False, allow_neg_eigval=False):
    """Recurrent decode: the T tokens of every row applied one by one to its cached fp32 state.

    Returns (o, final_state).  ``initial_state`` [B,Hv,K,V] fp32 ([B,Hv,V,K] with state_v_first) or None
    (zero states); with ``inplace`` the final state is written into ``initial_state`` itself (contiguous
    fp32).  Same recurrence as chunk_gated_delta_rule over the same tokens; meant for T = 1 or a few.
    """
    _check_tokens(q, k, v, g, beta)
    lib = _lib.load()
    p = problem(q, v, g, scale, None, use_qk_l2norm_in_kernel, state_v_first, 0,
                use_gate_in_kernel=use_gate_in_kernel, use_beta_sigmoid_in_kernel=use_beta_sigmoid_in_kernel,
                allow_neg_eigval=allow_neg_eigval)
    _check_state(initial_state, "initial_state", p, state_v_first, q)
    _check(out, "out", v.shape, v.dtype, q, optional=True)
    dev = q.device
    B, T, Hv, V = v.shape
    o = out if out is not None else torch.empty_like(v)
    if inplace:
        if initial_state is None or initial_state.dtype != torch.float32 or not initial_state.is_contiguous():
            raise ValueError("inplace needs a contiguous fp32 initial_state")
        h0 = fin = initial_state
    else:
        h0 = None if initial_state is None else initial_state.to(torch.float32).contiguous()
        fin = torch.empty(_state_shape(p, state_v_first), dtype=torch.float32, device=dev)
    st = lib.gdr_decode(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(fin),
                        _ptr(o), _stream(dev))
    _lib.check(st, "gdr_decode")
    return o, fin


def chunk_gated_delta_rule_bwd(q, k, v, g, beta, A, do, dht=None, scale=None, initial_state=None,
                               cu_seqlens=None, use_qk_l2norm_in_kernel=False, state_v_first=False,
                               num_segments=0, gate_dtype=None, saved=None, use_gate_in_kernel=False,
                               use_beta_sigmoid_in_kernel=False, allow_neg_eigval=False):
    """Backward.  ``g`` is the forward's g_cumsum (fp32).  Returns (dq, dk, dv, dbeta, dg, dh0).

    dg and dbeta take beta's dtype (or ``gate_dtype``); dh0 is None without an initial state.
    ``saved`` is the buffer the forward filled for the same problem and inputs (the backward then skips
    recomputing the decayed causal blocks, the states and Delta); None recomputes them.  With the activation
    options, beta is the raw beta and dg, dbeta are gradients w.r.t. the raw inputs; ``use_gate_in_kernel``
    needs ``saved``.
    """
    _check_tokens(q, k, v)
    B, T, Hv, V = v.shape
    gd = gate_dtype or beta.dtype
    _check(g, "g_cumsum", (B, T, Hv), torch.float32, q)
    _check(beta, "beta", (B, T, Hv), gd, q)
    _check(A, "A", (B, T, Hv, _lib.GDR_CHUNK), q.dtype, q)
    _check(do, "do", v.shape, v.dtype, q)
    lib = _lib.load()
    cu = _cu(cu_seqlens)
    _check_cu(cu, q)
    p = problem(q, v, torch.empty(0, dtype=gd), scale, cu, use_qk_l2norm_in_kernel, state_v_first, num_segments,
                use_gate_in_kernel=use_gate_in_kernel, use_beta_sigmoid_in_kernel=use_beta_sigmoid_in_kernel,
                allow_neg_eigval=allow_neg_eigval)
    _check_state(initial_state, "initial_state", p, state_v_first, q)
    _check_state(dht, "dht", p, state_v_first, q)
    _check_saved(saved, p, q)
    dev = q.device
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    dg = torch.empty(beta.shape, dtype=gd, device=dev)
    db = torch.empty(beta.shape, dtype=gd, device=dev)
    h0 = None if initial_state is None else initial_state.to(torch.float32).contiguous()
    dh0 = torch.empty(_state_shape(p, state_v_first), dtype=torch.float32, device=dev) if h0 is not None else None
    dht_ = None if dht is None else dht.to(torch.float32).contiguous()
    nbytes = workspace_bytes(p, True, saved)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    st = lib.gdr_bwd_ex(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(A), _ptr(do),
                        _ptr(dht_), _ptr(h0), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(db), _ptr(dh0), _ptr(ws),
                        nbytes, _ptr(saved), _stream(dev))
    _lib.check(st, "gdr_bwd_ex")
    return dq, dk, dv, db, dg, dh0


def prepare_chunks(cu_seqlens: torch.Tensor, chunk_size: int = _lib.GDR_CHUNK, total_tokens: int = -1):
    """Chunk tables of a packed batch, computed on the GPU.

    Returns (chunk_indices [max_chunks,2] int32, chunk_offsets [N+1] int32, total_chunks int32 [1]);
    rows of chunk_indices past total_chunks are zero.  Without ``total_tokens`` the table is sized from
    ``cu_seqlens[-1]``, read back to the host once (a synchronisation); passing it avoids that read.
    """
    lib = _lib.load()
    cu = _cu(cu_seqlens)
    _check(cu, "cu_seqlens", (cu.numel(),), torch.int32)
    N = cu.numel() - 1
    T = int(total_tokens)
    if T < 0:
        T = int(cu[-1].item())
    bound = (max(T, 0) + N * (chunk_size - 1)) // chunk_size
    max_chunks = max(bound, 1)
    idx = torch.zeros((max_chunks, 2), dtype=torch.int32, device=cu.device)
    off = torch.empty((N + 1,), dtype=torch.int32, device=cu.device)
    tot = torch.empty((1,), dtype=torch.int32, device=cu.device)
    st = lib.gdr_prepare_chunks(_ptr(cu), N, T, chunk_size, _ptr(idx), max_chunks, _ptr(off), _ptr(tot),
                                _stream(cu.device))
    _lib.check(st, "gdr_prepare_chunks")
    return idx, off, tot


def get_error(device=None) -> int:
    """Synchronise the current stream and return (and clear) the device error word."""
    return int(_lib.load().gdr_get_error(_stream(device)))


class _GDR(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, g, beta, scale, initial_state, output_final_state, cu_seqlens,
                use_qk_l2norm_in_kernel, state_v_first, num_segments, act):
        saved = saved_buffer(q, v, g, scale=scale, cu_seqlens=cu_seqlens,
                             use_qk_l2norm_in_kernel=use_qk_l2norm_in_kernel, state_v_first=state_v_first,
                             num_segments=num_segments, **act)
        gcs, A, o, _, fin = chunk_gated_delta_rule_fwd(
            q, k, v, g, beta, scale=scale, initial_state=initial_state, output_final_state=output_final_state,
            cu_seqlens=cu_seqlens, use_qk_l2norm_in_kernel=use_qk_l2norm_in_kernel, state_v_first=state_v_first,
            num_segments=num_segments, saved=saved, **act)
        ctx.save_for_backward(q, k, v, gcs, beta, A, initial_state, cu_seqlens, saved)
        ctx.opts = (scale, use_qk_l2norm_in_kernel, state_v_first, num_segments, g.dtype, act)
        return o, fin

    @staticmethod
    def backward(ctx, do, dht):
        q, k, v, gcs, beta, A, h0, cu, saved = ctx.saved_tensors
        scale, l2, vf, nseg, gdt, act = ctx.opts
        dq, dk, dv, db, dg, dh0 = chunk_gated_delta_rule_bwd(
            q, k, v, gcs, beta, A, do.contiguous(), dht=dht, scale=scale, initial_state=h0, cu_seqlens=cu,
            use_qk_l2norm_in_kernel=l2, state_v_first=vf, num_segments=nseg, gate_dtype=gdt, saved=saved, **act)
        return dq, dk, dv, dg, db, None, dh0, None, None, None, None, None, None


def chunk_gated_delta_rule(q, k, v, g, beta, scale=None, initial_state=None, output_final_state=False,
                           cu_seqlens=None, use_qk_l2norm_in_kernel=False, state_v_first=False, num_segments=0,
                           use_gate_in_kernel=False, use_beta_sigmoid_in_kernel=False, allow_neg_eigval=False):
    """Differentiable op: returns (o, final_state or None).  The activation options: see
    chunk_gated_delta_rule_fwd (gradients are w.r.t. the raw g and beta)."""
    act = dict(use_gate_in_kernel=use_gate_in_kernel, use_beta_sigmoid_in_kernel=use_beta_sigmoid_in_kernel,
               allow_neg_eigval=allow_neg_eigval)
    # the library reads contiguous arrays: views (q, k, v sliced from one fused projection) are copied first
    q, k, v, g, beta = (t.contiguous() for t in (q, k, v, g, beta))
    return _GDR.apply(q, k, v, g, beta, scale, initial_state, output_final_state, cu_seqlens,
                      use_qk_l2norm_in_kernel, state_v_first, num_segments, act)
