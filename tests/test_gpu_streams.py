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


def test_two_problems_on_two_streams_at_once():
    """Two independent steps (a dense batch and a packed one) issued on two streams without synchronising
    between them give, bit for bit, what each gives alone: the calls share no device state that they write."""
    w1 = custom(name="st_two_a", B=2, T=700, Hq=4, Hv=4, has_h0=True, final_state=True)
    w2 = custom(name="st_two_b", Hq=2, Hv=4, seq_lens=(500, 3, 129), has_h0=True, final_state=True)
    d1, d2 = to_dev(make_inputs(w1, seed=21)), to_dev(make_inputs(w2, seed=22))
    torch.cuda.synchronize()
    want1, want2 = train_step(w1, d1), train_step(w2, d2)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        # both steps in flight at once: nothing waits between the two streams' launches
        with torch.cuda.stream(s1):
            got1 = train_step(w1, d1, sync=False)
        with torch.cuda.stream(s2):
            got2 = train_step(w2, d2, sync=False)
        torch.cuda.synchronize()
    assert_bit_identical(want1, got1, "dense")
    assert_bit_identical(want2, got2, "packed")
