"""Bounded device-side waits: a wait that runs out of polls gives up, the kernel reports GDR_ERR_TIMEOUT
through the device error word and returns cleanly (its loads and MMA drained, its tensor memory freed),
and the next normal call is correct.

The poll budget of the backward's decayed-block kernel is cut to zero polls through
gdr_debug_set_wait_polls, so its first wait gives up before the tile loads it waits for can land.  The
producers are untouched and nothing faults, traps or spins without a bound.
"""

import ctypes

import pytest
import torch

import oracle
from gated_delta_rule_38_gb300 import _lib
from gated_delta_rule_38_gb300.inputs import custom, make_inputs
from harness import TOL, gpu_bwd, gpu_fwd, np64, oracle_problem, rel_l2, to_dev

pytestmark = pytest.mark.gpu


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def test_expired_wait_reports_timeout_and_the_next_call_is_correct():
    lib = _lib.load()
    w = custom(B=2, T=300, Hq=2, Hv=2, host_l2=False)
    x = make_inputs(w, seed=11)
    d = to_dev(x)
    gcs, A, _, _, _ = gpu_fwd(w, d, True)
    assert int(lib.gdr_get_error(_stream())) == 0
    assert lib.gdr_debug_set_wait_polls(0) == 0
    try:
        gpu_bwd(w, d, gcs, A, True)          # no saved buffer: the decayed-block kernel runs first
        assert int(lib.gdr_get_error(_stream())) == 9   # GDR_ERR_TIMEOUT, and the call returned
    finally:
        assert lib.gdr_debug_set_wait_polls(-1) == 0
    assert int(lib.gdr_get_error(_stream())) == 0
    # every kernel of the next call allocates tensor memory on every SM: it runs only if the timed-out
    # blocks freed theirs
    dq, dk, dv, db, dg, dh0 = gpu_bwd(w, d, gcs, A, True)
    torch.cuda.synchronize()
    assert int(lib.gdr_get_error(_stream())) == 0
    ref = oracle.bwd(oracle_problem(w, True), x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], h0=x["h0"],
                     dht=x["dht"])
    for key, val in (("dq", dq), ("dk", dk), ("dv", dv), ("dbeta", db), ("dg", dg), ("dh0", dh0)):
        assert rel_l2(np64(val), ref[key]) <= TOL, key
