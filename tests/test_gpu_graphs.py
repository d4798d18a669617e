"""A training step (forward + backward through the saved buffer) captured in a CUDA graph and replayed gives,
bit for bit, what the same calls give eagerly: no call reads device memory on the host, synchronises or
allocates outside the caller's stream, and the overlapped (programmatic) launches survive capture."""

import pytest
import torch

from gated_delta_rule_38_gb300.inputs import WORKLOADS, custom, make_inputs
from harness import assert_bit_identical, gpu_bwd, gpu_fwd, gpu_saved, to_dev, train_step

pytestmark = pytest.mark.gpu

CASES = [
    ("dense full size", WORKLOADS["dense"], 0),
    ("packed batch", custom(name="gr_varlen", Hq=4, Hv=4, seq_lens=(300, 1, 0, 129), has_h0=True,
                            final_state=True), 0),
    ("split, 3 segments", custom(name="gr_split", B=1, T=3000, Hq=2, Hv=2, has_h0=True, final_state=True), 3),
    ("activations", custom(name="gr_act", B=2, T=257, Hq=4, Hv=4, activations=True, final_state=True), 0),
]


@pytest.mark.parametrize("name,w,nseg", CASES, ids=[c[0] for c in CASES])
def test_captured_step_replays_bit_identically(name, w, nseg):
    d = to_dev(make_inputs(w, seed=9))
    torch.cuda.synchronize()
    want = train_step(w, d, nseg)
    kernel_l2 = not w.host_l2
    saved = gpu_saved(w, d, kernel_l2, num_segments=nseg)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # one eager warm-up call on the capture stream (library state, tensor maps)
        gpu_bwd(w, d, *gpu_fwd(w, d, kernel_l2, num_segments=nseg, saved=saved)[:2], kernel_l2,
                num_segments=nseg, saved=saved)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gcs, A, o, _, fin = gpu_fwd(w, d, kernel_l2, num_segments=nseg, saved=saved)
        dq, dk, dv, db, dg, dh0 = gpu_bwd(w, d, gcs, A, kernel_l2, num_segments=nseg, saved=saved)
    outs = {"g_cumsum": gcs, "A": A, "o": o, "final_state": fin, "dq": dq, "dk": dk, "dv": dv, "dbeta": db,
            "dg": dg, "dh0": dh0}
    for t in outs.values():
        if t is not None:
            t.fill_(float("nan")) if t.is_floating_point() else t.zero_()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    got = {k: v.clone() for k, v in outs.items() if v is not None}
    assert_bit_identical(want, got, name)
