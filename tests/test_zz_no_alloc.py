"""The allocation-free linear (w4a16_linear_noalloc) against the regular
w4a16_linear, through the C ABI.

The allocation-free entry point serves callers that cannot allocate device
memory at the call site (a plugin slot that only passes inputs and outputs, a
runtime that owns every allocation); it keeps its scratch in a static device
array instead of a caller workspace. This file is collected last so that a
run stopping at its first failure has already run every other test.
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
def L():
    from speculative_decode_verify_w4a16_gb300 import _lib, build
    build.build()
    oracle.build()
    return _lib.lib()


@pytest.mark.parametrize("M,N,K", [(4, 2048, 2048), (64, 1152, 3072)])
def test_noalloc_matches_workspace_linear_twice(L, M, N, K):
    import speculative_decode_verify_w4a16_gb300 as sv

    x_h = synth.activations(M, K, seed=900 + M)
    qw, sc = oracle.quantize(synth.weights(N, K, seed=901 + M))
    w = sv.prepack(*canon_to_dev(qw, sc))
    x = bf16_to_dev(x_h)
    ref_out = torch.empty((M, N), dtype=torch.bfloat16, device=dev())
    ws = torch.zeros(L.w4a16_linear_workspace_bytes(M, N, K), dtype=torch.uint8, device=dev())
    stream = torch.cuda.current_stream().cuda_stream
    assert L.w4a16_linear(ctypes.c_void_p(x.data_ptr()), M, K, ctypes.c_void_p(w.qweight.data_ptr()),
                          ctypes.c_void_p(w.scales.data_ptr()), N, ctypes.c_void_p(ref_out.data_ptr()),
                          ctypes.c_void_p(ws.data_ptr()), ws.numel(), ctypes.c_void_p(stream)) == 0
    ref = bf16_bits(ref_out)
    outs = []
    for i in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev())
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        alloc0 = torch.cuda.memory_allocated()
        assert L.w4a16_linear_noalloc(ctypes.c_void_p(x.data_ptr()), M, K, ctypes.c_void_p(w.qweight.data_ptr()),
                                      ctypes.c_void_p(w.scales.data_ptr()), N, ctypes.c_void_p(out.data_ptr()),
                                      ctypes.c_void_p(stream)) == 0
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        # the call allocates nothing: no tensor, and (after the first call,
        # which may load the library's kernels) no device memory, whose
        # allocations come in pages of 2 MB or more
        assert torch.cuda.memory_allocated() == alloc0
        if i > 0:
            assert free0 - free1 < (2 << 20), (free0, free1)
        outs.append(bf16_bits(out))
    assert L.w4a16_check_device_status(ctypes.c_void_p(stream)) == 0
    for o in outs:
        assert_linear_close(o, ref, "noalloc vs workspace linear")
    assert_linear_close(outs[0], oracle.linear(x_h, qw, sc), "noalloc vs oracle")
    assert L.w4a16_linear_noalloc_scratch_bytes() == 24 << 20


def test_noalloc_rejects_bad_arguments(L):
    p = ctypes.c_void_p(0x10000)
    assert L.w4a16_linear_noalloc(None, 4, 2048, p, p, 2048, p, None) == 1
    assert L.w4a16_linear_noalloc(p, 81, 2048, p, p, 2048, p, None) == 2
