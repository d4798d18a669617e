"""Run-to-run determinism: every reduction of the forward and backward kernels runs in a fixed order, so two
training steps on the same inputs give bit-identical outputs, states and gradients.  Before the second step
freed device memory is filled with NaN and its fresh saved buffer with a byte pattern, so a value that a run
leaves unwritten, or reads from a stale buffer, shows as a difference too."""

import pytest
import torch

from gated_delta_rule_38_gb300.inputs import WORKLOADS, custom, make_inputs
from harness import assert_bit_identical, to_dev, train_step

pytestmark = pytest.mark.gpu

CASES = [
    ("dense full size", WORKLOADS["dense"], 0),
    ("ragged, states", custom(name="det_ragged", B=2, T=333, Hq=4, Hv=4, has_h0=True, final_state=True), 0),
    ("packed batch", custom(name="det_varlen", Hq=4, Hv=4, seq_lens=(200, 0, 1, 64, 511), has_h0=True,
                            final_state=True), 0),
    ("GVA fp16, [V,K] states", custom(name="det_gva", B=1, T=700, Hq=2, Hv=8, dtype=torch.float16,
                                      state_v_first=True, has_h0=True, final_state=True), 0),
    ("split, 3 segments", custom(name="det_split", B=1, T=2000, Hq=2, Hv=2, has_h0=True, final_state=True), 3),
    ("activations, head dims 64", custom(name="det_act", B=2, T=300, Hq=4, Hv=4, K=64, V=64, activations=True,
                                         has_h0=True, final_state=True), 0),
]


@pytest.mark.parametrize("name,w,nseg", CASES, ids=[c[0] for c in CASES])
def test_two_steps_are_bit_identical(name, w, nseg):
    d = to_dev(make_inputs(w, seed=77))
    first = train_step(w, d, nseg)
    # scribble over freed memory so that the second step's fresh buffers do not start as copies of the first's
    junk = torch.full((64 << 20,), float("nan"), device="cuda")
    del junk
    second = train_step(w, d, nseg, poison=True)
    assert_bit_identical(first, second, name)
