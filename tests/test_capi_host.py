"""Host-side checks of the C-ABI library (no GPU needed): it loads, exports
every symbol the header declares, and rejects bad arguments before touching
the device; the stream-K work split covers every unit exactly once."""
import ctypes
import os
import re

import pytest

import __graft_entry__  # noqa: F401  (puts the repo root on sys.path)
from speculative_decode_verify_w4a16_gb300 import _lib
from speculative_decode_verify_w4a16_gb300 import build as sv_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    sv_build.build()
    return _lib.lib()


def _header_functions():
    text = open(os.path.join(ROOT, "include", "w4a16sv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_0-9]+)\s*\(", text)) - {"if", "sizeof"})


def test_header_symbols_exported(L):
    names = _header_functions()
    assert "w4a16_linear" in names and "spec_accept" in names
    for n in names:
        assert hasattr(L, n), n
        assert n in _lib.SIGNATURES, f"binding lacks {n}"


def test_no_torch_types_in_header():
    text = open(os.path.join(ROOT, "include", "w4a16sv.h")).read()
    for bad in ("torch", "at::", "Tensor", "c10"):
        assert bad not in text


def test_status_strings(L):
    for code, name in [(0, "W4A16_OK"), (1, "W4A16_ERR_INVALID_ARG"), (2, "W4A16_ERR_UNSUPPORTED"),
                       (4, "W4A16_ERR_DEVICE_TIMEOUT"), (6, "W4A16_ERR_WORKSPACE")]:
        assert _lib.status_string(code) == name
    assert _lib.status_string(99) == "W4A16_ERR_UNKNOWN"
    assert L.w4a16_abi_version() == 1


def test_size_functions(L):
    assert L.w4a16_packed_weight_bytes(8192, 8192) == 8192 * 8192 // 2
    assert L.w4a16_packed_scale_bytes(8192, 8192) == 8192 * 8192 // 64
    assert L.w4a16_packed_weight_bytes(100, 8192) == 0  # N not a multiple of 128
    assert L.w4a16_packed_weight_bytes(128, 100) == 0
    assert L.spec_accept_workspace_bytes(16, 4, 128256) > 0
    assert L.spec_accept_workspace_bytes(0, 4, 128256) == 0
    assert L.spec_accept_workspace_bytes(16, 2000, 128256) == 0
    assert L.spec_accept_workspace_bytes(16, 4, 1) == 0


def test_linear_rejects_bad_arguments_before_any_launch(L):
    p = ctypes.c_void_p(0x10000)  # never dereferenced: every call below fails validation
    ws = ctypes.c_void_p(0x20000)
    args = lambda x, M, K, N, ws_, nbytes: L.w4a16_linear(x, M, K, p, p, N, p, ws_, nbytes, None)
    assert args(None, 4, 2048, 2048, ws, 1 << 20) == _lib.ERR_INVALID_ARG
    assert args(p, 0, 2048, 2048, ws, 1 << 20) == _lib.ERR_INVALID_ARG
    assert args(p, 4, 2000, 2048, ws, 1 << 20) == _lib.ERR_INVALID_ARG
    assert args(p, 4, 2048, 2000, ws, 1 << 20) == _lib.ERR_INVALID_ARG
    assert args(p, 81, 2048, 2048, ws, 1 << 20) == _lib.ERR_UNSUPPORTED
    assert args(p, 4, 512, 2048, ws, 1 << 20) == _lib.ERR_UNSUPPORTED
    assert args(ctypes.c_void_p(0x10008), 4, 2048, 2048, ws, 1 << 20) == _lib.ERR_INVALID_ARG  # misaligned x
    assert args(p, 4, 2048, 2048, None, 1 << 20) == _lib.ERR_WORKSPACE
    assert args(p, 4, 2048, 2048, ctypes.c_void_p(0x20010), 1 << 20) == _lib.ERR_WORKSPACE


def test_accept_rejects_bad_arguments_before_any_launch(L):
    p = ctypes.c_void_p(0x10000)
    ws = ctypes.c_void_p(0x20000)
    f = L.spec_accept
    assert f(None, None, p, None, None, 1, 4, 100, p, p, ws, 1 << 20, None) == _lib.ERR_INVALID_ARG
    assert f(p, p, p, p, p, 1, 4, 131076, p, p, ws, 1 << 30, None) == _lib.ERR_UNSUPPORTED  # stochastic tree, V
    assert f(p, p, p, p, None, 1, 4, 100, p, p, ws, 1 << 20, None) == _lib.ERR_INVALID_ARG  # stochastic tree, no u
    assert f(p, p, p, None, None, 1, 4, 100, p, p, ws, 1 << 20, None) == _lib.ERR_INVALID_ARG  # no uniforms
    assert f(p, None, p, None, None, 0, 4, 100, p, p, ws, 1 << 20, None) == _lib.ERR_INVALID_ARG
    assert f(p, None, p, None, None, 1, 0, 100, p, p, ws, 1 << 20, None) == _lib.ERR_INVALID_ARG
    assert f(p, None, p, None, None, 1, 4, 1, p, p, ws, 1 << 20, None) == _lib.ERR_INVALID_ARG
    assert f(ctypes.c_void_p(0x10004), None, p, None, None, 1, 4, 100, p, p, ws, 1 << 20,
             None) == _lib.ERR_INVALID_ARG  # V % 4 == 0 wants 16-byte rows
    assert f(p, None, p, None, None, 1, 4, 100, p, p, None, 1 << 20, None) == _lib.ERR_WORKSPACE
    assert f(p, None, p, None, None, 1, 4, 100, p, p, ws, 16, None) == _lib.ERR_WORKSPACE


def test_fused_lm_head_and_prestat_accept_reject_bad_arguments(L):
    p = ctypes.c_void_p(0x10000)
    ws = ctypes.c_void_p(0x20000)
    lg = lambda x, M, K, N, logits, stats, ws_: L.w4a16_linear_logits(x, M, K, p, p, N, logits, stats, ws_, 1 << 20,
                                                                      None)
    assert lg(None, 4, 2048, 2048, p, p, ws) == _lib.ERR_INVALID_ARG
    assert lg(p, 4, 2048, 2048, p, None, ws) == _lib.ERR_INVALID_ARG
    assert lg(p, 81, 2048, 2048, p, p, ws) == _lib.ERR_UNSUPPORTED
    assert lg(p, 4, 2048, 2000, p, p, ws) == _lib.ERR_INVALID_ARG
    assert lg(p, 4, 2048, 2048, p, ctypes.c_void_p(0x10004), ws) == _lib.ERR_INVALID_ARG  # stats 8-byte aligned
    assert lg(p, 4, 2048, 2048, p, p, None) == _lib.ERR_WORKSPACE
    assert L.w4a16_linear_logits_workspace_bytes(0, 2048, 2048) == 0
    f = L.spec_accept_prestat
    assert f(p, None, p, p, p, 1, 4, 128, p, p, ws, 1 << 20, None) == _lib.ERR_INVALID_ARG  # no target statistics
    assert f(p, p, None, p, p, 1, 4, 128, p, p, ws, 1 << 20, None) == _lib.ERR_INVALID_ARG  # stochastic only
    assert f(p, p, p, p, p, 1, 4, 100, p, p, ws, 1 << 20, None) == _lib.ERR_INVALID_ARG  # V % 32 != 0
    assert f(p, p, p, p, p, 1, 4, 128, p, p, ws, 16, None) == _lib.ERR_WORKSPACE


def test_attention_compaction_and_node_accept_reject_bad_arguments(L):
    p = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10008)  # 8-byte, not 16-byte aligned
    ws = ctypes.c_void_p(0x20000)
    f32 = ctypes.c_float

    def att(q=p, lens=p, B=2, n=5, H=64, Hkv=8, D=128, Lcap=4096, max_len=4000, scale=f32(0.088)):
        return L.tree_attention(q, p, p, lens, None, B, n, H, Hkv, D, Lcap, max_len, scale, p, ws, 1 << 30, None)

    assert att(q=None) == _lib.ERR_INVALID_ARG
    assert att(lens=None) == _lib.ERR_INVALID_ARG
    assert att(D=64) == _lib.ERR_UNSUPPORTED
    assert att(n=65) == _lib.ERR_UNSUPPORTED
    assert att(H=60, Hkv=8) == _lib.ERR_INVALID_ARG  # H not a multiple of Hkv
    assert att(max_len=4092) == _lib.ERR_INVALID_ARG  # max_len + n > Lcap
    assert att(q=odd) == _lib.ERR_INVALID_ARG
    assert att(scale=f32(0.0)) == _lib.ERR_INVALID_ARG
    assert att(scale=f32(float("nan"))) == _lib.ERR_INVALID_ARG
    assert L.tree_attention_workspace_bytes(2, 5, 64, 8, 64, 4096, 4000) == 0
    assert L.tree_attention_workspace_bytes(2, 5, 64, 8, 128, 4096, 4095) == 0

    def comp(kc=p, node=p, n=5, Hkv=8, D=128, Lcap=4096, layers=80):
        return L.kv_compact(kc, p, p, None, node, 2, n, Hkv, D, Lcap, layers, p, None)

    assert comp(kc=None) == _lib.ERR_INVALID_ARG
    assert comp(node=None) == _lib.ERR_INVALID_ARG
    assert comp(D=12) == _lib.ERR_INVALID_ARG
    assert comp(n=65) == _lib.ERR_UNSUPPORTED
    assert comp(Hkv=1024) == _lib.ERR_UNSUPPORTED  # one node's keys and values exceed a pass
    assert comp(kc=odd) == _lib.ERR_INVALID_ARG
    assert comp(Lcap=4) == _lib.ERR_INVALID_ARG
    a = L.spec_accept_node
    assert a(p, None, p, None, None, 2, 4, 128, p, p, None, ws, 1 << 20, None) == _lib.ERR_INVALID_ARG
    assert a(p, None, p, None, None, 2, 4, 128, p, p, ctypes.c_void_p(0x10002), ws, 1 << 20, None) == \
        _lib.ERR_INVALID_ARG


def test_format_calls_reject_bad_arguments(L):
    p = ctypes.c_void_p(0x10000)
    assert L.w4a16_quantize(None, 128, 128, p, p, None) == _lib.ERR_INVALID_ARG
    assert L.w4a16_quantize(p, 100, 128, p, p, None) == _lib.ERR_INVALID_ARG
    assert L.w4a16_prepack(p, p, 128, 128, ctypes.c_void_p(0x10004), p, None) == _lib.ERR_INVALID_ARG


@pytest.mark.parametrize("U,C,min_units,max_rounds", [
    (1, 1, 2, 8), (7, 3, 2, 8), (256, 256, 2, 8), (1024, 456, 2, 8), (4096, 608, 2, 8), (64128, 456, 2, 8),
    (28672, 608, 2, 8), (28672, 608, 2, 3), (14336, 152, 4, 8), (33, 32, 2, 8), (5120, 608, 2, 1)])
def test_item_schedule_covers_each_unit_once(L, U, C, min_units, max_rounds):
    rb = (ctypes.c_int64 * 9)()
    R = L.w4a16_item_rounds(U, C, min_units, max_rounds, rb)
    assert 1 <= R <= max_rounds
    rb = list(rb)[:R + 1]
    assert rb[0] == 0 and rb[-1] == U
    # every round holds at least C units (no empty item); rounds shrink
    lens = [rb[r + 1] - rb[r] for r in range(R)]
    assert all(n >= C for n in lens)
    assert all(lens[r + 1] <= lens[r] for r in range(R - 2))
    # all but the last round are at least 2*C*min_units long (split only when that leaves >= C*min_units)
    assert all(n >= C * min_units for n in lens[:-1])
    begins = [L.w4a16_item_begin(U, C, min_units, max_rounds, i) for i in range(R * C + 1)]
    assert begins[0] == 0 and begins[-1] == U
    assert all(begins[i + 1] > begins[i] for i in range(R * C))  # no empty item
    for r in range(R):  # inside a round, item sizes differ by at most one
        sizes = [begins[r * C + j + 1] - begins[r * C + j] for j in range(C)]
        assert max(sizes) - min(sizes) <= 1
    step = max(1, U // 3000)
    for u in list(range(0, U, step)) + [U - 1]:
        i = L.w4a16_item_owner(U, C, min_units, max_rounds, u)
        assert begins[i] <= u < begins[i + 1]
    assert L.w4a16_item_owner(U, C, min_units, max_rounds, U) == -1
    assert L.w4a16_item_begin(U, C, min_units, max_rounds, R * C + 1) == -1
    assert L.w4a16_item_rounds(C - 1, C, min_units, max_rounds, (ctypes.c_int64 * 9)()) == 0
