"""Python binding of libw4a16sv: argument marshalling from torch tensors to the
C ABI (include/w4a16sv.h). PyTorch supplies device memory and the current
CUDA stream; every step of the computation runs in the library's kernels.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from ._lib import W4A16Error, check, lib

GROUP = 128


def _stream(stream: Optional[torch.cuda.Stream] = None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        # the library launches on, and keeps its state for, the current device
        raise ValueError(f"{name} is on {t.device}, the current device is cuda:{torch.cuda.current_device()}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


# --------------------------------------------------------------- workspace
_ws_cache: dict = {}


def workspace(nbytes: int, device: Optional[torch.device] = None, key: str = "default") -> torch.Tensor:
    """A zero-filled scratch buffer of at least nbytes on `device`, cached per
    (device, key). The kernels leave it zeroed after every call."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    k = (dev.index if dev.index is not None else torch.cuda.current_device(), key)
    buf = _ws_cache.get(k)
    if buf is None or buf.numel() < nbytes:
        buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=dev)
        _ws_cache[k] = buf
    return buf


# ------------------------------------------------------------------ format

def packed_weight_bytes(N: int, K: int) -> int:
    return int(lib().w4a16_packed_weight_bytes(N, K))


def packed_scale_bytes(N: int, K: int) -> int:
    return int(lib().w4a16_packed_scale_bytes(N, K))


def quantize(w: torch.Tensor, stream=None):
    """w fp32 [N, K] (CUDA) -> canonical (qweight int32 [N, K/8] holding the
    uint32 words, scales fp16 [N, K/128])."""
    _need(w, "w", torch.float32)
    N, K = w.shape
    qw = torch.empty((N, K // 8), dtype=torch.int32, device=w.device)
    sc = torch.empty((N, K // GROUP), dtype=torch.float16, device=w.device)
    check(lib().w4a16_quantize(_ptr(w), N, K, _ptr(qw), _ptr(sc), _stream(stream)), "w4a16_quantize")
    return qw, sc


@dataclass
class PackedWeight:
    """A prepacked W4A16 weight (N x K) ready for linear()."""
    N: int
    K: int
    qweight: torch.Tensor  # uint8 [N*K/2], streaming layout
    scales: torch.Tensor   # uint8 [N*K/64], streaming layout

    @property
    def nbytes(self) -> int:
        return self.qweight.numel() + self.scales.numel()


def prepack(qweight: torch.Tensor, scales: torch.Tensor, stream=None) -> PackedWeight:
    """Canonical (qweight int32/uint32 [N, K/8], scales fp16 [N, K/128]) -> PackedWeight."""
    if qweight.dtype not in (torch.int32, torch.uint32):
        raise ValueError("qweight must hold 32-bit words")
    _need(qweight, "qweight", qweight.dtype)
    _need(scales, "scales", torch.float16)
    N, K8 = qweight.shape
    K = K8 * 8
    if tuple(scales.shape) != (N, K // GROUP):
        raise ValueError("scales shape mismatch")
    qp = torch.empty(packed_weight_bytes(N, K), dtype=torch.uint8, device=qweight.device)
    sp = torch.empty(packed_scale_bytes(N, K), dtype=torch.uint8, device=qweight.device)
    if qp.numel() == 0:
        raise W4A16Error(1, "w4a16_prepack: N and K must be positive multiples of 128")
    check(lib().w4a16_prepack(_ptr(qweight), _ptr(scales), N, K, _ptr(qp), _ptr(sp), _stream(stream)),
          "w4a16_prepack")
    return PackedWeight(N, K, qp, sp)


# ------------------------------------------------------------------ linear

def linear_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib().w4a16_linear_workspace_bytes(M, N, K))


def linear(x: torch.Tensor, w: PackedWeight, out: Optional[torch.Tensor] = None,
           ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out[M, N] = bf16(x[M, K] . W^T) with W the dequantised int4 weight."""
    _need(x, "x", torch.bfloat16)
    M, K = x.shape
    if K != w.K:
        raise ValueError(f"x has K={K}, weight has K={w.K}")
    if out is None:
        out = torch.empty((M, w.N), dtype=torch.bfloat16, device=x.device)
    _need(out, "out", torch.bfloat16, (M, w.N))
    if ws is None:
        ws = workspace(linear_workspace_bytes(M, w.N, K), x.device, "linear")
    check(lib().w4a16_linear(_ptr(x), M, K, _ptr(w.qweight), _ptr(w.scales), w.N, _ptr(out), _ptr(ws),
                             ws.numel(), _stream(stream)), "w4a16_linear")
    return out


def linear_noalloc(x: torch.Tensor, w: PackedWeight, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """linear() without a workspace: the library uses its static device scratch
    (see w4a16_linear_noalloc in the header for the rules on sharing it)."""
    _need(x, "x", torch.bfloat16)
    M, K = x.shape
    if K != w.K:
        raise ValueError(f"x has K={K}, weight has K={w.K}")
    if out is None:
        out = torch.empty((M, w.N), dtype=torch.bfloat16, device=x.device)
    _need(out, "out", torch.bfloat16, (M, w.N))
    check(lib().w4a16_linear_noalloc(_ptr(x), M, K, _ptr(w.qweight), _ptr(w.scales), w.N, _ptr(out),
                                     _stream(stream)), "w4a16_linear_noalloc")
    return out


def linear_logits_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib().w4a16_linear_logits_workspace_bytes(M, N, K))


def linear_logits(x: torch.Tensor, w: PackedWeight, logits: Optional[torch.Tensor] = None,
                  stats: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None, stream=None):
    """The lm_head of the verify pass with fused softmax statistics:
    returns (logits fp32 [M, N], stats fp32 [M, N/32, 2] = (max, sum exp(l - max))
    per 32-logit slice)."""
    _need(x, "x", torch.bfloat16)
    M, K = x.shape
    if K != w.K:
        raise ValueError(f"x has K={K}, weight has K={w.K}")
    if logits is None:
        logits = torch.empty((M, w.N), dtype=torch.float32, device=x.device)
    if stats is None:
        stats = torch.empty((M, w.N // 32, 2), dtype=torch.float32, device=x.device)
    _need(logits, "logits", torch.float32, (M, w.N))
    _need(stats, "stats", torch.float32, (M, w.N // 32, 2))
    if ws is None:
        ws = workspace(linear_logits_workspace_bytes(M, w.N, K), x.device, "linear")
    check(lib().w4a16_linear_logits(_ptr(x), M, K, _ptr(w.qweight), _ptr(w.scales), w.N, _ptr(logits), _ptr(stats),
                                    _ptr(ws), ws.numel(), _stream(stream)), "w4a16_linear_logits")
    return logits, stats


# ------------------------------------------------------------------ accept

def accept_workspace_bytes(B: int, n: int, V: int) -> int:
    return int(lib().spec_accept_workspace_bytes(B, n, V))


def spec_accept(p_logits: torch.Tensor, draft_ids: torch.Tensor, q_logits: Optional[torch.Tensor] = None,
                tree_parents: Optional[torch.Tensor] = None, uniforms: Optional[torch.Tensor] = None,
                accepted_len: Optional[torch.Tensor] = None, next_token: Optional[torch.Tensor] = None,
                ws: Optional[torch.Tensor] = None, stream=None):
    """Speculative accept step; see the header for the three modes.
    Returns (accepted_len int32 [B], next_token int32 [B])."""
    _need(p_logits, "p_logits", torch.float32)
    _need(draft_ids, "draft_ids", torch.int32)
    B, rows, V = p_logits.shape
    if tree_parents is not None:
        n = rows
        _need(tree_parents, "tree_parents", torch.int32, (B, n))
        _need(draft_ids, "draft_ids", torch.int32, (B, n))
    else:
        n = rows - 1
        _need(draft_ids, "draft_ids", torch.int32, (B, n))
    if q_logits is not None:
        _need(q_logits, "q_logits", torch.float32, (B, n, V))
    if uniforms is not None:  # stochastic tree: [B, n] (u_0 draws); sequence: [B, n + 1]
        _need(uniforms, "uniforms", torch.float32, (B, n) if tree_parents is not None else (B, n + 1))
    if accepted_len is None:
        accepted_len = torch.empty(B, dtype=torch.int32, device=p_logits.device)
    if next_token is None:
        next_token = torch.empty(B, dtype=torch.int32, device=p_logits.device)
    if ws is None:
        ws = workspace(accept_workspace_bytes(B, n, V), p_logits.device, "accept")
    check(lib().spec_accept(_ptr(p_logits), _ptr(q_logits), _ptr(draft_ids), _ptr(tree_parents), _ptr(uniforms),
                            B, n, V, _ptr(accepted_len), _ptr(next_token), _ptr(ws), ws.numel(),
                            _stream(stream)), "spec_accept")
    return accepted_len, next_token


def spec_accept_prestat(p_logits: torch.Tensor, p_stats: torch.Tensor, draft_ids: torch.Tensor,
                        q_logits: torch.Tensor, uniforms: torch.Tensor, accepted_len: Optional[torch.Tensor] = None,
                        next_token: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None, stream=None):
    """Stochastic sequence accept with the target rows' statistics supplied
    (p_stats [B, n+1, V/32, 2] from linear_logits). Returns (accepted_len, next_token)."""
    _need(p_logits, "p_logits", torch.float32)
    B, n1, V = p_logits.shape
    n = n1 - 1
    _need(p_stats, "p_stats", torch.float32, (B, n1, V // 32, 2))
    _need(draft_ids, "draft_ids", torch.int32, (B, n))
    _need(q_logits, "q_logits", torch.float32, (B, n, V))
    _need(uniforms, "uniforms", torch.float32, (B, n + 1))
    if accepted_len is None:
        accepted_len = torch.empty(B, dtype=torch.int32, device=p_logits.device)
    if next_token is None:
        next_token = torch.empty(B, dtype=torch.int32, device=p_logits.device)
    if ws is None:
        ws = workspace(accept_workspace_bytes(B, n, V), p_logits.device, "accept")
    check(lib().spec_accept_prestat(_ptr(p_logits), _ptr(p_stats), _ptr(q_logits), _ptr(draft_ids), _ptr(uniforms),
                                    B, n, V, _ptr(accepted_len), _ptr(next_token), _ptr(ws), ws.numel(),
                                    _stream(stream)), "spec_accept_prestat")
    return accepted_len, next_token


def spec_accept_node(p_logits: torch.Tensor, draft_ids: torch.Tensor, q_logits: Optional[torch.Tensor] = None,
                     tree_parents: Optional[torch.Tensor] = None, uniforms: Optional[torch.Tensor] = None,
                     ws: Optional[torch.Tensor] = None, stream=None):
    """spec_accept that also returns the accepted node:
    (accepted_len, next_token, accepted_node), int32 [B] each."""
    _need(p_logits, "p_logits", torch.float32)
    B, rows, V = p_logits.shape
    n = rows if tree_parents is not None else rows - 1
    _need(draft_ids, "draft_ids", torch.int32, (B, n))
    if tree_parents is not None:
        _need(tree_parents, "tree_parents", torch.int32, (B, n))
    if q_logits is not None:
        _need(q_logits, "q_logits", torch.float32, (B, n, V))
    if uniforms is not None:
        _need(uniforms, "uniforms", torch.float32, (B, n) if tree_parents is not None else (B, n + 1))
    acc, nxt, node = (torch.empty(B, dtype=torch.int32, device=p_logits.device) for _ in range(3))
    if ws is None:
        ws = workspace(accept_workspace_bytes(B, n, V), p_logits.device, "accept")
    check(lib().spec_accept_node(_ptr(p_logits), _ptr(q_logits), _ptr(draft_ids), _ptr(tree_parents),
                                 _ptr(uniforms), B, n, V, _ptr(acc), _ptr(nxt), _ptr(node), _ptr(ws), ws.numel(),
                                 _stream(stream)), "spec_accept_node")
    return acc, nxt, node


# ------------------------------------------------------ verify attention

def tree_attention_workspace_bytes(B: int, n: int, H: int, Hkv: int, D: int, Lcap: int, max_len: int) -> int:
    return int(lib().tree_attention_workspace_bytes(B, n, H, Hkv, D, Lcap, max_len))


def tree_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, lens: torch.Tensor,
                   tree_parents: Optional[torch.Tensor] = None, max_len: Optional[int] = None,
                   scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                   ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Tree-masked verify attention. q bf16 [B, n, H, D]; caches bf16
    [B, Hkv, Lcap, D] (prefix at 0..lens-1, the tree nodes at lens..lens+n-1);
    lens int32 [B]; tree_parents int32 [B, n] or None (chain); max_len: an
    upper bound of lens (default Lcap - n). Returns bf16 [B, n, H, D]."""
    _need(q, "q", torch.bfloat16)
    B, n, H, D = q.shape
    _need(k_cache, "k_cache", torch.bfloat16)
    Hkv, Lcap = k_cache.shape[1], k_cache.shape[2]
    _need(k_cache, "k_cache", torch.bfloat16, (B, Hkv, Lcap, D))
    _need(v_cache, "v_cache", torch.bfloat16, (B, Hkv, Lcap, D))
    _need(lens, "lens", torch.int32, (B,))
    if tree_parents is not None:
        _need(tree_parents, "tree_parents", torch.int32, (B, n))
    max_len = Lcap - n if max_len is None else int(max_len)
    scale = D ** -0.5 if scale is None else float(scale)
    if out is None:
        out = torch.empty((B, n, H, D), dtype=torch.bfloat16, device=q.device)
    _need(out, "out", torch.bfloat16, (B, n, H, D))
    nbytes = tree_attention_workspace_bytes(B, n, H, Hkv, D, Lcap, max_len)
    if ws is None and nbytes > 0:
        ws = workspace(nbytes, q.device, "attention")
    check(lib().tree_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(lens), _ptr(tree_parents), B, n, H, Hkv,
                               D, Lcap, max_len, scale, _ptr(out), _ptr(ws), 0 if ws is None else ws.numel(),
                               _stream(stream)), "tree_attention")
    return out


def kv_compact(k_cache: torch.Tensor, v_cache: torch.Tensor, lens: torch.Tensor, accepted_node: torch.Tensor,
               tree_parents: Optional[torch.Tensor] = None, n: Optional[int] = None,
               new_lens: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Moves the accepted root path's keys/values to lens..lens+depth in
    place. Caches bf16 [layers, B, Hkv, Lcap, D] (or [B, Hkv, Lcap, D]);
    tree_parents [B, n] or None (chain, then n is required). Returns new_lens."""
    _need(k_cache, "k_cache", torch.bfloat16)
    kc, vc = (k_cache, v_cache) if k_cache.dim() == 5 else (k_cache.unsqueeze(0), v_cache.unsqueeze(0))
    layers, B, Hkv, Lcap, D = kc.shape
    _need(vc, "v_cache", torch.bfloat16, (layers, B, Hkv, Lcap, D))
    _need(lens, "lens", torch.int32, (B,))
    _need(accepted_node, "accepted_node", torch.int32, (B,))
    if tree_parents is not None:
        n = tree_parents.shape[1]
        _need(tree_parents, "tree_parents", torch.int32, (B, n))
    elif n is None:
        raise ValueError("n is required for a sequence draft")
    if new_lens is None:
        new_lens = torch.empty(B, dtype=torch.int32, device=lens.device)
    check(lib().kv_compact(_ptr(kc), _ptr(vc), _ptr(lens), _ptr(tree_parents), _ptr(accepted_node), B, int(n), Hkv,
                           D, Lcap, layers, _ptr(new_lens), _stream(stream)), "kv_compact")
    return new_lens


def check_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    return int(lib().w4a16_check_device_status(_stream(stream)))
