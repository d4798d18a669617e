"""The library's per-kernel event profiler (gdr_profile_enable / gdr_profile_read, which the benchmark's
per-kernel table reads) and the forward's caller-provided output buffer."""

import pytest
import torch

import gated_delta_rule_38_gb300 as gdr
from gated_delta_rule_38_gb300 import _lib
from gated_delta_rule_38_gb300.inputs import custom, make_inputs
from harness import to_dev, train_step

pytestmark = pytest.mark.gpu


def test_profiler_counts_each_launch_of_a_step():
    w = custom(name="prof", B=2, T=300, Hq=2, Hv=2, host_l2=False)
    d = to_dev(make_inputs(w, seed=41))
    train_step(w, d)  # warm
    _lib.profile_enable(True)
    for _ in range(3):
        train_step(w, d)
    _lib.profile_enable(False)
    prof = _lib.profile_read()
    for name in ("wy_fwd", "chain_fwd", "chain_rev", "bwd_chunk"):
        launches, ms = prof[name]
        assert launches == 3 and ms > 0, (name, prof[name])
    # nothing is recorded while it is off; enabling again clears the totals
    train_step(w, d)
    assert _lib.profile_read() == prof
    _lib.profile_enable(True)
    _lib.profile_enable(False)
    assert all(n == 0 for n, _ in _lib.profile_read().values())


def test_forward_into_a_callers_output_buffer():
    w = custom(name="outbuf", B=2, T=130, Hq=2, Hv=2, host_l2=False)
    d = to_dev(make_inputs(w, seed=42))
    _, _, o, _, _ = gdr.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                                   use_qk_l2norm_in_kernel=True)
    out = torch.full_like(d["v"], float("nan"))
    _, _, o2, _, _ = gdr.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                                    use_qk_l2norm_in_kernel=True, out=out)
    torch.cuda.synchronize()
    assert o2.data_ptr() == out.data_ptr() and torch.equal(out, o)
