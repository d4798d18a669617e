"""Oracle for the chunked Gated Delta Rule -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The product (the CUDA library
under ``gated_delta_rule_38_gb300``) never imports it, and the two share no
code: the only module both sides use is the seeded input generator
``gated_delta_rule_38_gb300.inputs``, which holds none of the method's
arithmetic.

Contents
--------
* ``fwd`` / ``bwd``: the token-by-token fp64 recurrence and its reverse-mode
  gradient, implemented in C (``gdr_oracle.c``) and called through ctypes.
  They follow the recurrence of the "Gated Delta Rule" op (FlashQLA skill
  page, "Core API" section for the tensor roles and shapes).
* ``g_cumsum``, ``wy_matrix``: the per-chunk quantities that the low-level
  forward returns ("processed gate tensor" and "intra-chunk attention
  matrix", FlashQLA skill page, "Low-Level API" section), written from their
  definitions with numpy fp64.
* ``prepare_lens``, ``prepare_chunk_offsets``, ``prepare_chunk_indices``:
  the varlen chunk tables (FlashQLA documentation page, utilities section),
  as plain Python loops.

Readings where the pages are silent (each is listed in the design notes):
the log-gate ``g`` is used as ``exp(g)`` with no activation unless one of the
activation options is set (``gate_in_kernel``: g = logsigmoid(raw), the log of
the sigmoid decay in (0, 1) that the skill page's module example applies;
``beta_sigmoid``: beta = sigmoid(raw); ``neg_eigval``: beta doubled, so that the
eigenvalue 1 - beta of the transition along k spans (-1, 1)); the L2 norm is
``x / sqrt(sum x^2 + 1e-6)``; the chunk size is 64; ``g_cumsum`` is the
chunk-local inclusive cumulative sum reset at every chunk and sequence start;
``A`` is stored per token as row ``t mod 64`` of its chunk's inverse;
``chunk_indices`` rows are ``(sequence, chunk-within-sequence)``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdr_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libgdr_oracle.so")

CHUNK = 64
L2_EPS = 1e-6

_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc + OpenMP (no CUDA involved)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _SO + ".tmp%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32 = ctypes.c_int
        lib.gdr_oracle_fwd.restype = i32
        lib.gdr_oracle_fwd.argtypes = [i32, P, P, i32, i32, i32, i32, ctypes.c_double, i32, i32, i32,
                                       P, P, P, P, P, P, P, P, P, P, P, P, i32]
        lib.gdr_oracle_bwd.restype = i32
        lib.gdr_oracle_bwd.argtypes = [i32, P, P, i32, i32, i32, i32, ctypes.c_double, i32, i32, i32,
                                       P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, i32]
        lib.gdr_oracle_max_threads.restype = i32
        _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().gdr_oracle_max_threads())


@dataclass
class Problem:
    """Shapes and options of one call (dense when ``cu_seqlens`` is None)."""
    B: int
    T: int
    Hq: int
    Hv: int
    K: int = 128
    V: int = 128
    scale: Optional[float] = None
    l2norm: bool = False
    state_v_first: bool = False
    cu_seqlens: Optional[List[int]] = None
    chunk: int = CHUNK
    # activations applied to the raw per-token scalars before the recurrence (the options the FlashQLA
    # backend's verifier names: use_gate_in_kernel, use_beta_sigmoid_in_kernel, allow_neg_eigval)
    gate_in_kernel: bool = False   # g <- logsigmoid(g): the log of a sigmoid decay in (0, 1)
    beta_sigmoid: bool = False     # beta <- sigmoid(beta)
    neg_eigval: bool = False       # beta <- 2 beta: the transition's eigenvalue along k spans (-1, 1)

    def __post_init__(self):
        if self.scale is None:
            self.scale = self.K ** -0.5

    @property
    def num_seqs(self) -> int:
        return len(self.cu_seqlens) - 1 if self.cu_seqlens is not None else self.B

    def seq_bounds(self):
        """(start, length) of every sequence in the packed token axis."""
        if self.cu_seqlens is not None:
            cu = self.cu_seqlens
            return [(int(cu[n]), int(cu[n + 1]) - int(cu[n])) for n in range(len(cu) - 1)]
        return [(b * self.T, self.T) for b in range(self.B)]

    @property
    def total_tokens(self) -> int:
        return self.B * self.T


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(a) -> Optional[np.ndarray]:
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor on the CPU
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _sigmoid(x: np.ndarray) -> np.ndarray:
    """1 / (1 + e^{-x}), evaluated without overflow for either sign of x."""
    e = np.exp(-np.abs(x))
    return np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def _logsigmoid(x: np.ndarray) -> np.ndarray:
    """log(1 / (1 + e^{-x})) = min(x, 0) - log(1 + e^{-|x|})."""
    return np.minimum(x, 0.0) - np.log1p(np.exp(-np.abs(x)))


def activate(pb: Problem, g, beta):
    """The gate and beta the recurrence uses, from the raw inputs (fp64); unchanged without the options."""
    g, beta = _f64(g), _f64(beta)
    if pb.gate_in_kernel:
        g = _logsigmoid(g)
    if pb.beta_sigmoid:
        beta = _sigmoid(beta)
    if pb.neg_eigval:
        beta = 2.0 * beta
    return g, beta


def activate_grads(pb: Problem, g_raw, beta_raw, dg, dbeta):
    """Chain rule through ``activate``: gradients w.r.t. the raw g and beta from those w.r.t. the used ones.
    d logsigmoid(x)/dx = sigmoid(-x); d sigmoid(x)/dx = sigmoid(x) sigmoid(-x)."""
    if pb.gate_in_kernel:
        dg = dg * _sigmoid(-_f64(g_raw)).reshape(dg.shape)
    if pb.neg_eigval:
        dbeta = 2.0 * dbeta
    if pb.beta_sigmoid:
        b = _f64(beta_raw).reshape(dbeta.shape)
        dbeta = dbeta * _sigmoid(b) * _sigmoid(-b)
    return dg, dbeta


def _chunk_base(pb: Problem) -> np.ndarray:
    base, acc = [], 0
    for _, ln in pb.seq_bounds():
        base.append(acc)
        acc += (ln + pb.chunk - 1) // pb.chunk
    return np.asarray(base + [acc], dtype=np.int64)


def fwd(pb: Problem, q, k, v, g, beta, h0=None, heads=None, want_h=False, want_delta=False,
        nthreads: int = 0):
    """Token-level forward.  Returns dict(o, final_state[, h][, delta]).

    Inputs are in the API layouts ([B,T,H,D] dense or [1,T,H,D] packed);
    values are upcast to fp64 exactly.  ``heads``: optional list of v-heads to
    evaluate (outputs of the other heads are NaN).
    """
    lib = _load()
    g, beta = activate(pb, g, beta)
    q, k, v, g, beta, h0 = (_f64(x) for x in (q, k, v, g, beta, h0))
    Ttot = pb.total_tokens
    N = pb.num_seqs
    bounds = pb.seq_bounds()
    st = np.asarray([s for s, _ in bounds], dtype=np.int64)
    ln = np.asarray([n for _, n in bounds], dtype=np.int64)
    sel = None
    if heads is not None:
        sel = np.zeros(pb.Hv, dtype=np.uint8)
        sel[list(heads)] = 1
    o = np.full((Ttot, pb.Hv, pb.V), np.nan)
    shape_state = (N, pb.Hv, pb.V, pb.K) if pb.state_v_first else (N, pb.Hv, pb.K, pb.V)
    ht = np.full(shape_state, np.nan)
    base = _chunk_base(pb)
    hc = None
    if want_h:
        hc = np.full((int(base[-1]),) + shape_state[1:], np.nan)
    dl = np.full((Ttot, pb.Hv, pb.V), np.nan) if want_delta else None
    rc = lib.gdr_oracle_fwd(N, _ptr(st), _ptr(ln), pb.Hq, pb.Hv, pb.K, pb.V, float(pb.scale),
                            int(pb.l2norm), int(pb.state_v_first), pb.chunk,
                            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(sel),
                            _ptr(o), _ptr(ht), _ptr(hc), _ptr(base), _ptr(dl), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle fwd failed with code %d" % rc)
    lead = (pb.B, pb.T) if pb.cu_seqlens is None else (1, Ttot)
    out = {"o": o.reshape(lead + (pb.Hv, pb.V)), "final_state": ht}
    if want_h:
        out["h"] = hc
    if want_delta:
        out["delta"] = dl.reshape(lead + (pb.Hv, pb.V))
    return out


def bwd(pb: Problem, q, k, v, g, beta, do, h0=None, dht=None, heads=None, nthreads: int = 0):
    """Reverse-mode gradient of ``fwd``.  Returns dict(dq, dk, dv, dg, dbeta, dh0).

    ``dh0`` is the gradient of the initial state (all-zero start when h0 is None).
    With ``heads``, only those v-heads contribute (dq/dk of a q/k head are
    exact when every v-head of its group is selected).
    """
    lib = _load()
    g_raw, beta_raw = g, beta
    g, beta = activate(pb, g, beta)
    q, k, v, g, beta, h0, do, dht = (_f64(x) for x in (q, k, v, g, beta, h0, do, dht))
    Ttot = pb.total_tokens
    N = pb.num_seqs
    bounds = pb.seq_bounds()
    st = np.asarray([s for s, _ in bounds], dtype=np.int64)
    ln = np.asarray([n for _, n in bounds], dtype=np.int64)
    sel = None
    if heads is not None:
        sel = np.zeros(pb.Hv, dtype=np.uint8)
        sel[list(heads)] = 1
    dq = np.full((Ttot, pb.Hq, pb.K), np.nan)
    dk = np.full((Ttot, pb.Hq, pb.K), np.nan)
    dv = np.full((Ttot, pb.Hv, pb.V), np.nan)
    dg = np.full((Ttot, pb.Hv), np.nan)
    db = np.full((Ttot, pb.Hv), np.nan)
    shape_state = (N, pb.Hv, pb.V, pb.K) if pb.state_v_first else (N, pb.Hv, pb.K, pb.V)
    dh0 = np.full(shape_state, np.nan)
    rc = lib.gdr_oracle_bwd(N, _ptr(st), _ptr(ln), pb.Hq, pb.Hv, pb.K, pb.V, float(pb.scale),
                            int(pb.l2norm), int(pb.state_v_first), pb.chunk,
                            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(do),
                            _ptr(dht), _ptr(sel), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(db),
                            _ptr(dh0), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle bwd failed with code %d" % rc)
    dg, db = activate_grads(pb, g_raw, beta_raw, dg, db)
    lead = (pb.B, pb.T) if pb.cu_seqlens is None else (1, Ttot)
    return {"dq": dq.reshape(lead + (pb.Hq, pb.K)), "dk": dk.reshape(lead + (pb.Hq, pb.K)),
            "dv": dv.reshape(lead + (pb.Hv, pb.V)), "dg": dg.reshape(lead + (pb.Hv,)),
            "dbeta": db.reshape(lead + (pb.Hv,)), "dh0": dh0}


# ---------------------------------------------------------------------------
# Chunk-level quantities, from their definitions (numpy fp64).
# ---------------------------------------------------------------------------

def _l2n(x: np.ndarray) -> np.ndarray:
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + L2_EPS)


def g_cumsum(pb: Problem, g) -> np.ndarray:
    """Processed gate: inclusive cumsum of g inside each chunk of each sequence.

    Returns [B,T,Hv] (or [1,Ttot,Hv]) fp64.  Restarts at every chunk start and
    at every sequence start (reading of the "processed gate tensor").
    """
    g = activate(pb, g, np.zeros(1))[0].reshape(pb.total_tokens, pb.Hv)
    out = np.zeros_like(g)
    for s0, L in pb.seq_bounds():
        for c0 in range(0, L, pb.chunk):
            c1 = min(L, c0 + pb.chunk)
            out[s0 + c0:s0 + c1] = np.cumsum(g[s0 + c0:s0 + c1], axis=0)
    lead = (pb.B, pb.T) if pb.cu_seqlens is None else (1, pb.total_tokens)
    return out.reshape(lead + (pb.Hv,))


def wy_matrix(pb: Problem, k, g, beta) -> np.ndarray:
    """Intra-chunk matrix A = (I + L)^-1 per chunk and v-head, stored per token.

    L[r,s] = beta_r exp(G_r - G_s) (k_r . k_s) for s < r (strictly lower),
    with G the chunk-local cumsum of g and k L2-normalised when the option is
    on.  Row r of the chunk's inverse is stored at token (chunk start + r),
    columns 0..63; entries past the sequence end stay zero.
    Returns [B,T,Hv,chunk] (or [1,Ttot,Hv,chunk]) fp64.
    """
    kk = _f64(k).reshape(pb.total_tokens, pb.Hq, pb.K)
    if pb.l2norm:
        kk = _l2n(kk)
    bb = activate(pb, np.zeros(1), beta)[1].reshape(pb.total_tokens, pb.Hv)
    G = g_cumsum(pb, g).reshape(pb.total_tokens, pb.Hv)
    grp = pb.Hv // pb.Hq
    out = np.zeros((pb.total_tokens, pb.Hv, pb.chunk))
    for s0, L in pb.seq_bounds():
        for c0 in range(0, L, pb.chunk):
            n = min(L, c0 + pb.chunk) - c0
            sl = slice(s0 + c0, s0 + c0 + n)
            for j in range(pb.Hv):
                kc = kk[sl, j // grp]
                Gc = G[sl, j]
                gram = kc @ kc.T
                decay = np.exp(Gc[:, None] - Gc[None, :])
                Lm = np.tril(bb[sl, j][:, None] * gram * decay, -1)
                out[sl, j, :n] = np.linalg.inv(np.eye(n) + Lm)
    lead = (pb.B, pb.T) if pb.cu_seqlens is None else (1, pb.total_tokens)
    return out.reshape(lead + (pb.Hv, pb.chunk))


# ---------------------------------------------------------------------------
# Varlen chunk tables (FlashQLA documentation page, utilities section).
# ---------------------------------------------------------------------------

def prepare_lens(cu_seqlens) -> List[int]:
    """Per-sequence lengths: consecutive differences of cu_seqlens."""
    cu = [int(x) for x in cu_seqlens]
    return [cu[n + 1] - cu[n] for n in range(len(cu) - 1)]


def prepare_chunk_offsets(cu_seqlens, chunk_size: int):
    """(offsets, total): offsets has the shape of cu_seqlens; offsets[n] is the
    number of chunks before sequence n, offsets[N] = total."""
    offs = [0]
    for ln in prepare_lens(cu_seqlens):
        offs.append(offs[-1] + (ln + chunk_size - 1) // chunk_size)
    return offs, offs[-1]


def prepare_chunk_indices(cu_seqlens, chunk_size: int) -> List[List[int]]:
    """One row per chunk: [sequence index, chunk index within the sequence]."""
    rows = []
    for n, ln in enumerate(prepare_lens(cu_seqlens)):
        for c in range((ln + chunk_size - 1) // chunk_size):
            rows.append([n, c])
    return rows
