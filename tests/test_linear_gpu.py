"""GPU parity of the W4A16 verify linear against the CPU oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decode_verify_w4a16_gb300 as sv
import synth
from helpers import assert_linear_close, bf16_bits, bf16_to_dev, canon_to_dev, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decode_verify_w4a16_gb300 import build
    build.build()
    oracle.build()


def _case(M, N, K, seed):
    x = synth.activations(M, K, seed=seed)
    qw, sc = oracle.quantize(synth.weights(N, K, seed=seed + 1))
    return x, qw, sc


def _gpu_linear(x, qw, sc):
    w = sv.prepack(*canon_to_dev(qw, sc))
    out = sv.linear(bf16_to_dev(x), w)
    torch.cuda.synchronize()
    assert sv.check_device_status() == 0
    return bf16_bits(out)


def test_gpu_quantizer_bit_exact():
    N, K = 384, 2048
    w = synth.weights(N, K, seed=100)
    w[5, 256:384] = 0.0
    w[7, 0] = 1e-9  # tiny group max: subnormal fp16 scale
    qw_r, sc_r = oracle.quantize(w)
    qw, sc = sv.quantize(torch.from_numpy(w).to(dev()))
    torch.cuda.synchronize()
    assert np.array_equal(qw.cpu().numpy().view(np.uint32), qw_r)
    assert np.array_equal(sc.cpu().numpy().view(np.uint16), sc_r)


def test_config_single_linear_m4():
    # x bf16 [4, 2048] ~ N(0,1); W 2048 x 2048 ~ N(0, 0.02), int4 g128; seed 0
    x, qw, sc = _case(4, 2048, 2048, seed=0)
    assert_linear_close(_gpu_linear(x, qw, sc), oracle.linear(x, qw, sc), "config 2048x2048 M=4")


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 7, 8, 9, 15, 16, 17, 24, 32, 33, 48, 63, 64, 65, 72, 80])
def test_all_token_counts(M):
    # several tiles along N and K, K range split across CTAs
    x, qw, sc = _case(M, 640, 3072, seed=10 + M)
    assert_linear_close(_gpu_linear(x, qw, sc), oracle.linear(x, qw, sc), f"M={M}")


@pytest.mark.parametrize("M,N,K", [(1, 128, 1024), (4, 128, 8192), (8, 1024, 1024), (2, 4096, 1152),
                                   (16, 256, 2048), (64, 128, 1024), (3, 1152, 5120)])
def test_shapes(M, N, K):
    x, qw, sc = _case(M, N, K, seed=M * 7 + N + K)
    assert_linear_close(_gpu_linear(x, qw, sc), oracle.linear(x, qw, sc), f"{M}x{N}x{K}")


@pytest.mark.parametrize("M", [4, 40, 64])
def test_output_not_16_byte_aligned(M):
    # an output that starts 4 bytes past a 16-byte boundary takes the
    # per-element store path (tiles are otherwise written by TMA stores);
    # the rows around it are untouched
    x, qw, sc = _case(M, 640, 3072, seed=200 + M)
    w = sv.prepack(*canon_to_dev(qw, sc))
    buf = torch.full((M * 640 + 16,), 7.0, dtype=torch.bfloat16, device=dev())
    out = buf[2:2 + M * 640].view(M, 640)
    assert out.data_ptr() % 16 == 4
    sv.linear(bf16_to_dev(x), w, out=out)
    torch.cuda.synchronize()
    assert sv.check_device_status() == 0
    assert_linear_close(bf16_bits(out), oracle.linear(x, qw, sc), f"unaligned out M={M}")
    assert torch.all(buf[:2] == 7.0) and torch.all(buf[2 + M * 640:] == 7.0)


@pytest.mark.parametrize("M", [1, 6, 8, 13, 40])
def test_one_hot_codes_select_columns_exactly(M):
    # W[n, cols[n]] = 1 (scale 1) selects column cols[n] of x. Both paths
    # multiply exact codes, so the selection is bit-exact for any tokens: this
    # pins the index mapping of the packed layout, the token tiles and the
    # output tiles (integer tokens times a power of two per row, and N(0, 1)).
    N, K = 384, 1024
    g = synth.rng(40 + M)
    cols = g.integers(0, K, size=N)
    codes = np.zeros((N, K), dtype=np.int8)
    codes[np.arange(N), cols] = 1
    sc = np.full((N, K // 128), np.float16(1.0)).view(np.uint16)
    qw = oracle.pack_codes(codes)
    xi = g.integers(-64, 65, size=(M, K)).astype(np.float32) * (2.0 ** g.integers(-20, 20, size=(M, 1)))
    x = synth.bf16_bits_from_f32(xi.astype(np.float32))
    assert np.array_equal(_gpu_linear(x, qw, sc), x[:, cols])
    xn = synth.activations(M, K, seed=41)
    assert np.array_equal(_gpu_linear(xn, qw, sc), xn[:, cols])


@pytest.mark.parametrize("M", [1, 5, 8, 15])
def test_token_rows_of_very_different_magnitude(M):
    # token rows from 2^-30 to 2^30 (and a zero row) in one call must each
    # meet the tolerance
    N, K = 256, 2048
    j = np.round(np.linspace(-30, 30, M)).astype(np.int32)[:, None]
    x = synth.bf16_bits_to_f32(synth.activations(M, K, seed=46)) * (2.0 ** j).astype(np.float32)  # exact
    zero_row = M // 2 if M > 2 else -1
    if zero_row >= 0:
        x[zero_row] = 0.0
    xb = synth.bf16_bits_from_f32(x.astype(np.float32))
    _, qw, sc = _case(M, N, K, seed=47)
    got, ref = _gpu_linear(xb, qw, sc), oracle.linear(xb, qw, sc)
    if zero_row >= 0:
        assert np.all(got[zero_row] == 0) and np.all(ref[zero_row] == 0)
    # undo each row's power of two (exact on bf16 values in the normal range) and apply the usual bar
    unscale = lambda b: synth.bf16_bits_from_f32(synth.bf16_bits_to_f32(b) * (2.0 ** -j).astype(np.float32))
    for m in range(M):
        if m != zero_row:
            assert_linear_close(unscale(got)[m:m + 1], unscale(ref)[m:m + 1], f"row {m} (x scaled by 2^{j[m, 0]})")


@pytest.mark.parametrize("M", [2, 8])
def test_groups_of_very_different_magnitude(M):
    # within one token row, each 128-wide group scaled by its own power of two
    # (2^-8 .. 2^0): the per-group partial sums must combine correctly
    N, K = 512, 4096
    g = synth.rng(48 + M)
    j = g.integers(-8, 1, size=(M, K // 128))
    x = synth.bf16_bits_to_f32(synth.activations(M, K, seed=49 + M)).reshape(M, K // 128, 128)
    x = (x * (2.0 ** j)[:, :, None]).reshape(M, K).astype(np.float32)
    xb = synth.bf16_bits_from_f32(x)
    _, qw, sc = _case(M, N, K, seed=50 + M)
    assert_linear_close(_gpu_linear(xb, qw, sc), oracle.linear(xb, qw, sc), f"M={M} groups 2^-8..2^0")


def test_zero_input_gives_zero():
    M, N, K = 2, 256, 1024
    x = np.zeros((M, K), dtype=np.uint16)
    _, qw, sc = _case(M, N, K, seed=43)
    assert np.all(_gpu_linear(x, qw, sc) == 0)


def test_repeated_calls_reuse_workspace():
    # the split-tile counters must reset themselves between calls
    x, qw, sc = _case(5, 1024, 4096, seed=44)
    ref = oracle.linear(x, qw, sc)
    w = sv.prepack(*canon_to_dev(qw, sc))
    xt = bf16_to_dev(x)
    first = None
    for _ in range(4):
        out = bf16_bits(sv.linear(xt, w))
        if first is None:
            first = out
        assert np.array_equal(out, first)  # deterministic
    assert_linear_close(first, ref, "repeat")
    assert sv.check_device_status() == 0


def test_workspace_errors():
    x, qw, sc = _case(4, 256, 1024, seed=45)
    w = sv.prepack(*canon_to_dev(qw, sc))
    xt = bf16_to_dev(x)
    small = torch.zeros(16, dtype=torch.uint8, device=dev())
    with pytest.raises(sv.W4A16Error) as e:
        sv.linear(xt, w, ws=small)
    assert e.value.status == 6


# --------------------------------------------------- Llama-3-70B full shapes
SHAPES = [("qkv", 8192, 10240), ("o", 8192, 8192), ("gate_up", 8192, 57344), ("down", 28672, 8192),
          ("lm_head", 8192, 128256)]


@pytest.fixture(scope="module")
def full_weights():
    cache = {}

    def get(name, K, N):
        if name not in cache:
            cache.clear()
            w = synth.weights(N, K, seed=1000 + len(name))
            qw, sc = oracle.quantize(w)
            del w
            cache[name] = (qw, sc, sv.prepack(*canon_to_dev(qw, sc)))
        return cache[name]

    return get


@pytest.mark.parametrize("name,K,N", SHAPES)
def test_llama70b_shapes_sampled(full_weights, name, K, N):
    """Full Llama-3-70B shapes in the launch configuration the benchmark times,
    checked on sampled output columns (first/last tiles plus random ones)."""
    qw, sc, w = full_weights(name, K, N)
    g = synth.rng(2000 + N)
    cols = np.unique(np.concatenate([np.arange(0, 128), np.arange(N - 128, N), g.integers(0, N, 256)]))
    for M in (1, 4, 8, 9, 16, 40, 64, 80):  # the fragment path and five token-tile widths of the tcgen05 path
        x = synth.activations(M, K, seed=3000 + M)
        out = bf16_bits(sv.linear(bf16_to_dev(x), w))
        ref = oracle.linear_cols(x, qw, sc, cols)
        assert_linear_close(out[:, cols], ref, f"{name} M={M}")
    assert sv.check_device_status() == 0
