"""Failure detection without a GPU fault: a kernel whose bounded wait runs
out reports W4A16_ERR_DEVICE_TIMEOUT through the device error word, returns,
and leaves the device usable.

The test loads the debug build of the library (a separate .so outside the
package; the product never loads it): its waits give up after 5 ms instead
of 2 s, and a test hook makes the producer of the fragment-path linear's
first CTA leave out one ring stage (no copies, no arrival), so the
consumers' wait on that stage runs out. Every access stays inside its buffer
and every wait is bounded.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_linear_close, bf16_bits, bf16_to_dev, canon_to_dev, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def D():
    from speculative_decode_verify_w4a16_gb300 import _lib, build

    oracle.build()
    L = ctypes.CDLL(build.build_debug())
    for name, (res, args) in _lib.SIGNATURES.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    L.w4a16_test_set_skip_stage.argtypes = [ctypes.c_int]
    L.w4a16_test_set_skip_stage.restype = ctypes.c_int
    return L


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_wait_runs_out_then_the_device_recovers(D):
    M, N, K = 4, 8192, 8192  # 4096 units: every CTA fills more than five ring stages
    x_h = synth.activations(M, K, seed=700)
    qw_h, sc_h = oracle.quantize(synth.weights(N, K, seed=701))
    ref = oracle.linear(x_h, qw_h, sc_h)
    qw, sc = canon_to_dev(qw_h, sc_h)
    qp = torch.empty(N * K // 2, dtype=torch.uint8, device=dev())
    sp = torch.empty(N * K // 64, dtype=torch.uint8, device=dev())
    assert D.w4a16_prepack(_p(qw), _p(sc), N, K, _p(qp), _p(sp), None) == 0
    x = bf16_to_dev(x_h)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev())
    nb = D.w4a16_linear_workspace_bytes(M, N, K)
    ws = torch.zeros(nb, dtype=torch.uint8, device=dev())

    def call():
        return D.w4a16_linear(_p(x), M, K, _p(qp), _p(sp), N, _p(out), _p(ws), nb, None)

    assert call() == 0 and D.w4a16_check_device_status(None) == 0
    assert_linear_close(bf16_bits(out), ref, "before the timeout")

    assert D.w4a16_test_set_skip_stage(4) == 0  # CTA 0 leaves out its fifth ring stage
    try:
        assert call() == 0  # the launch itself succeeds; the failure is found on the device
        assert D.w4a16_check_device_status(None) == 4  # W4A16_ERR_DEVICE_TIMEOUT
        assert D.w4a16_check_device_status(None) == 0  # the read cleared it
    finally:
        assert D.w4a16_test_set_skip_stage(-1) == 0

    # the context is still usable: after re-zeroing the workspace (its
    # counters may have been left mid-count) the same call is correct again
    ws.zero_()
    out.fill_(float("nan"))
    assert call() == 0 and D.w4a16_check_device_status(None) == 0
    assert_linear_close(bf16_bits(out), ref, "after the timeout")
    torch.cuda.synchronize()
