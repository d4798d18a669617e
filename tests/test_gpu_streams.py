"""Every launch of a call goes to the caller's stream.  The step runs on a side stream behind a long sleep
kernel, so a launch that went to another stream would run before its inputs exist; the results must equal,
bit for bit, those of the same step on the default stream (the kernels are deterministic)."""

import pytest
import torch

from gated_delta_rule_38_gb300.inputs import custom, make_inputs
from harness import assert_bit_identical, to_dev, train_step

pytestmark = pytest.mark.gpu

CASES = [
    ("packed batch", custom(name="st_varlen", Hq=4, Hv=4, seq_lens=(300, 1, 0, 129), has_h0=True,
                            final_state=True), 0),
    ("split, 3 segments, GVA", custom(name="st_split", B=1, T=3000, Hq=2, Hv=4, has_h0=True, final_state=True), 3),
    ("activations", custom(name="st_act", B=2, T=257, Hq=4, Hv=4, activations=True, final_state=True), 0),
]


@pytest.mark.parametrize("name,w,nseg", CASES, ids=[c[0] for c in CASES])
def test_side_stream_behind_a_sleep(name, w, nseg):
    d = to_dev(make_inputs(w, seed=5))
    torch.cuda.synchronize()
    want = train_step(w, d, nseg)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        torch.cuda._sleep(50_000_000)  # tens of milliseconds of one spinning thread on the side stream
        got = train_step(w, d, nseg)
    torch.cuda.synchronize()
    assert_bit_identical(want, got, name)
