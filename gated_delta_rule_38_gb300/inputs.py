"""Seeded synthetic inputs for the gated delta rule.

This module only draws random tensors with the distributions of the
workloads; it holds none of the method's arithmetic.  It is the one module
that both the CUDA path's tests/benchmark and the CPU oracle read from.

Recipe (all draws on a CPU ``torch.Generator`` seeded with 42, in the fixed
order q, k, v, g, beta, h0, do, dht, in fp32, then cast once to the input
dtype; the oracle reads the cast values):

* q, k ~ N(0, 1); for the workloads marked ``host_l2`` they are divided by
  their per-token, per-head Euclidean norm before the cast (the kernel's own
  L2-norm option is then off), otherwise the kernel normalises them.
* v ~ N(0, 1).
* g = logsigmoid(N(mu_g, 1)) (a log-space decay <= 0); beta = sigmoid(N(0, 1)).
  For the workloads marked ``activations`` the same draws are handed over
  raw (g = N(mu_g, 1), beta = N(0, 1): the logits before the activations),
  and they run with the in-kernel gate and beta activations.
* h0 = 0.1 N(0, 1) in fp32 when the workload has an initial state.
* do ~ N(0, 1); dht = 0.1 N(0, 1) in fp32 when the final state is an output.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    Hq: int
    Hv: int
    K: int = 128
    V: int = 128
    dtype: torch.dtype = torch.bfloat16
    host_l2: bool = True          # q,k normalised on the host (kernel option off)
    has_h0: bool = True
    final_state: bool = True
    state_v_first: bool = False
    mu_g: float = 0.0
    seq_lens: Optional[tuple] = None   # varlen: packed lengths (B must be 1)
    activations: bool = False     # g, beta drawn as raw logits; run with the in-kernel activations

    @property
    def cu_seqlens(self) -> Optional[List[int]]:
        if self.seq_lens is None:
            return None
        cu = [0]
        for n in self.seq_lens:
            cu.append(cu[-1] + int(n))
        return cu

    @property
    def num_seqs(self) -> int:
        return len(self.seq_lens) if self.seq_lens is not None else self.B

    @property
    def tokens(self) -> int:
        return self.B * self.T


# The workloads: a tiny correctness case, dense prefill, a packed
# variable-length batch, grouped value attention and one long sequence; and
# two variants of dense prefill, one with raw gate / beta logits activated in
# the kernels and one with head dimension 64.
WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", B=1, T=256, Hq=2, Hv=2),
    "dense": Workload("dense", B=2, T=4096, Hq=32, Hv=32, host_l2=False, has_h0=False,
                      final_state=False),
    "varlen": Workload("varlen", B=1, T=5311, Hq=32, Hv=32, seq_lens=(512, 1024, 768, 3000, 7)),
    "gva": Workload("gva", B=4, T=8192, Hq=16, Hv=32, dtype=torch.float16),
    "long": Workload("long", B=1, T=65536, Hq=16, Hv=16, mu_g=2.0),
    "dense_act": Workload("dense_act", B=2, T=4096, Hq=32, Hv=32, host_l2=False, has_h0=False,
                          final_state=False, activations=True),
    "dense_hd64": Workload("dense_hd64", B=2, T=4096, Hq=32, Hv=32, K=64, V=64, host_l2=False, has_h0=False,
                           final_state=False),
}


def custom(name="custom", **kw) -> Workload:
    """A workload with explicit sizes (used by edge-case tests)."""
    if "seq_lens" in kw and kw["seq_lens"] is not None:
        kw["seq_lens"] = tuple(int(x) for x in kw["seq_lens"])
        kw.setdefault("B", 1)
        kw["T"] = sum(kw["seq_lens"])
    return Workload(name, **kw)


def make_inputs(w: Workload, seed: int = 42) -> Dict[str, torch.Tensor]:
    """Draw the inputs of ``w`` on the CPU.  Returns a dict of CPU tensors.

    Keys: q, k, v, g, beta (input dtype), h0, dht (fp32 or None), do.
    Layouts: q,k [B,T,Hq,K]; v,do [B,T,Hv,V]; g,beta [B,T,Hv];
    h0,dht [N,Hv,K,V] ([N,Hv,V,K] when state_v_first).
    """
    gen = torch.Generator().manual_seed(seed)
    B, T = w.B, w.T
    dt = w.dtype

    def randn(*shape):
        return torch.randn(*shape, generator=gen, dtype=torch.float32)

    q = randn(B, T, w.Hq, w.K)
    k = randn(B, T, w.Hq, w.K)
    if w.host_l2:
        q = q / q.norm(dim=-1, keepdim=True)
        k = k / k.norm(dim=-1, keepdim=True)
    v = randn(B, T, w.Hv, w.V)
    g = randn(B, T, w.Hv) + w.mu_g
    beta = randn(B, T, w.Hv)
    if not w.activations:
        g = torch.nn.functional.logsigmoid(g)
        beta = torch.sigmoid(beta)
    N = w.num_seqs
    sshape = (N, w.Hv, w.V, w.K) if w.state_v_first else (N, w.Hv, w.K, w.V)
    h0 = 0.1 * randn(*sshape) if w.has_h0 else None
    do = randn(B, T, w.Hv, w.V)
    dht = 0.1 * randn(*sshape) if w.final_state else None
    return {
        "q": q.to(dt), "k": k.to(dt), "v": v.to(dt), "g": g.to(dt), "beta": beta.to(dt),
        "h0": h0, "do": do.to(dt), "dht": dht,
    }
