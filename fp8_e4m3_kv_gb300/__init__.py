"""fp8_e4m3_kv_gb300 -- Python binding of libfp8kv, an FP8 e4m3 paged KV
cache with attention over it, in hand-written CUDA for GB300 (sm_103a).

This module only marshals arguments: torch tensors become device pointers,
sizes and the current CUDA stream, and a non-zero status becomes an
exception.  Every step of the computation runs in the library's kernels; if
``libfp8kv.so`` is missing the import fails (build it with
``python fp8_e4m3_kv_gb300/build.py`` or ``__graft_entry__.build()``).

The entry points and their C signatures are declared in ``include/fp8kv.h``.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfp8kv.so")

OK, ERR_ARG, ERR_SCALE, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_LAUNCH, ERR_DEVICE = range(7)
DEVERR_WAIT_TIMEOUT, DEVERR_BAD_BLOCK, DEVERR_BAD_SLOT = 0x1, 0x2, 0x4

if not os.path.exists(LIB_PATH):
    raise ImportError(
        "libfp8kv.so is not built (%s); run `python fp8_e4m3_kv_gb300/build.py`" % LIB_PATH)

_lib = ctypes.CDLL(LIB_PATH)

P = ctypes.c_void_p
i32, i64, f32, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t


class CacheStruct(ctypes.Structure):
    _fields_ = [("k", P), ("v", P), ("num_blocks", i64), ("block_size", i32),
                ("num_kv_heads", i32), ("head_dim", i32)]


def _sig(name, restype, argtypes):
    f = getattr(_lib, name)
    f.restype = restype
    f.argtypes = argtypes
    return f


_kv_store = _sig("kv_store_e4m3", ctypes.c_int,
                 [ctypes.POINTER(CacheStruct), P, P, i64, i64, P, i64, f32, f32, P])
_decode_ex = _sig("paged_attn_fp8_decode_ex", ctypes.c_int,
                  [ctypes.POINTER(CacheStruct), P, i32, P, i32, P, i32, f32, f32, f32, f32, P,
                   i64, i32, i32, P, P, sz, i32, P])
_decode = _sig("paged_attn_fp8_decode", ctypes.c_int,
               [ctypes.POINTER(CacheStruct), P, i32, P, i32, P, i32, f32, f32, f32, f32, P,
                i64, i32, i32, P, P, sz, P])
_decode_noalloc = _sig("paged_attn_fp8_decode_noalloc", ctypes.c_int,
                       [ctypes.POINTER(CacheStruct), P, i32, P, i32, P, i32, f32, f32, f32, f32,
                        P, i64, i32, i32, P, P])
_decode_store = _sig("paged_attn_fp8_decode_store", ctypes.c_int,
                     [ctypes.POINTER(CacheStruct), P, i32, P, P, P, i32, P, i32, f32, f32, f32,
                      f32, P, i64, i32, i32, P, P, P, P, sz, P])
_store_pt = _sig("kv_store_e4m3_per_token", ctypes.c_int,
                 [ctypes.POINTER(CacheStruct), P, P, i64, i64, P, i64, P, P, P])
_decode_pt = _sig("paged_attn_fp8_decode_per_token", ctypes.c_int,
                  [ctypes.POINTER(CacheStruct), P, i32, P, i32, P, i32, f32, f32, P, P, P, i64,
                   i32, i32, P, P, sz, P])
_prefill_pt = _sig("attn_fp8_varlen_prefill_per_token", ctypes.c_int,
                   [ctypes.POINTER(CacheStruct), P, i32, P, P, P, i32, i32, i32, f32, f32, P, P, P,
                    i64, i32, i32, P, P])
_ws_size = _sig("fp8kv_decode_workspace_size", sz, [i32, i32, i32, i32, i32, i32, i32, i32])
_prefill = _sig("attn_fp8_varlen_prefill", ctypes.c_int,
                [ctypes.POINTER(CacheStruct), P, i32, P, P, P, i32, i32, i32, f32, f32, f32,
                 f32, P, i64, i32, i32, P, P, sz, P])
_amax = _sig("kv_amax_calibrate", ctypes.c_int, [P, P, i64, i64, P, i64, i32, i32, P, P, P])
_band_counts = _sig("kv_band_counts", ctypes.c_int, [P, i64, P, i64, i32, f32, P, P])
_scale_from_amax = _sig("fp8kv_scale_from_amax", ctypes.c_int, [f32, i32, ctypes.POINTER(f32)])
_cache_bytes = _sig("fp8kv_cache_bytes", sz, [i64, i32, i32, i32])
_prefill_max_ctas = _sig("fp8kv_set_prefill_max_ctas", ctypes.c_int, [i32])
_drop_first_copy = _sig("fp8kv_test_drop_first_copy", ctypes.c_int, [i32])
_device_error = _sig("fp8kv_device_error", ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), i32])
_status_string = _sig("fp8kv_status_string", ctypes.c_char_p, [ctypes.c_int])

EXPORTED = ("kv_store_e4m3", "paged_attn_fp8_decode", "paged_attn_fp8_decode_ex",
            "paged_attn_fp8_decode_noalloc", "paged_attn_fp8_decode_store",
            "kv_store_e4m3_per_token", "paged_attn_fp8_decode_per_token",
            "fp8kv_decode_workspace_size", "attn_fp8_varlen_prefill",
            "attn_fp8_varlen_prefill_per_token",
            "fp8kv_set_prefill_max_ctas", "kv_amax_calibrate",
            "kv_band_counts",
            "fp8kv_scale_from_amax", "fp8kv_cache_bytes", "fp8kv_device_error",
            "fp8kv_test_drop_first_copy",
            "fp8kv_status_string")


class Fp8KVError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (call, status_string(status), status))


def status_string(status: int) -> str:
    return _status_string(int(status)).decode()


def _check(status: int, call: str):
    if status != OK:
        raise Fp8KVError(status, call)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> int:
    """The CUDA stream handle: the given torch stream, else the current one."""
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(torch.cuda.current_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _need(t: torch.Tensor, dtype, name: str, device=None):
    if t.dtype is not dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if device is not None:
        # a CUDA device compares by index (no device object per check)
        ok = (t.is_cuda and t.get_device() == device.index) if device.type == "cuda" \
            else t.device == device
        if not ok:
            raise ValueError("%s must be on %s" % (name, device))


class KVCache:
    """The paged e4m3 cache: K and V uint8 tensors
    [num_blocks][num_kv_heads][block_size][head_dim], each byte an e4m3 code."""

    def __init__(self, k: torch.Tensor, v: torch.Tensor):
        if k.shape != v.shape or k.dim() != 4:
            raise ValueError("k and v must be [num_blocks][num_kv_heads][block_size][head_dim]")
        _need(k, torch.uint8, "cache k")
        _need(v, torch.uint8, "cache v")
        if not (k.is_contiguous() and v.is_contiguous()):
            raise ValueError("cache arrays must be contiguous")
        self.k, self.v = k, v
        self._device = k.device
        self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim = k.shape
        self._c = CacheStruct(k.data_ptr(), v.data_ptr(), self.num_blocks, self.block_size,
                              self.num_kv_heads, self.head_dim)

    @classmethod
    def empty(cls, num_blocks, block_size, num_kv_heads, head_dim, device="cuda",
              fill: int = 0) -> "KVCache":
        shape = (num_blocks, num_kv_heads, block_size, head_dim)
        k = torch.full(shape, fill, dtype=torch.uint8, device=device)
        v = torch.full(shape, fill, dtype=torch.uint8, device=device)
        return cls(k, v)

    @property
    def device(self):
        return self._device

    def c(self):
        return ctypes.byref(self._c)


def cache_bytes(num_blocks, block_size, num_kv_heads, head_dim) -> int:
    return int(_cache_bytes(num_blocks, block_size, num_kv_heads, head_dim))


def _rows(x: torch.Tensor, name: str, row: int):
    """[T][H][D] (or [T][H*D]) bf16 with contiguous rows -> token stride."""
    _need(x, torch.bfloat16, name)
    if x.dim() == 3:
        if x.stride(2) != 1 or x.stride(1) != x.shape[2] or x.shape[1] * x.shape[2] != row:
            raise ValueError("%s rows must be contiguous [T][H][D]" % name)
    elif x.dim() == 2:
        if x.stride(1) != 1 or x.shape[1] != row:
            raise ValueError("%s rows must be contiguous [T][H*D]" % name)
    else:
        raise ValueError("%s must be [T][H][D]" % name)
    return x.stride(0)


def kv_store_e4m3(cache: KVCache, k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                  k_scale: float, v_scale: float, stream=None) -> None:
    """Quantize bf16 k, v [T][Hkv][D] (x / scale, clamp +-448, e4m3 RNE) and
    store them at slot_mapping (int64 [T]; negative = skip)."""
    row = cache.num_kv_heads * cache.head_dim
    ks, vs = _rows(k, "k", row), _rows(v, "v", row)
    _need(slot_mapping, torch.int64, "slot_mapping", cache.device)
    T = k.shape[0]
    if v.shape[0] != T or slot_mapping.numel() != T or not slot_mapping.is_contiguous():
        raise ValueError("k, v and slot_mapping must have the same token count")
    _check(_kv_store(cache.c(), _ptr(k), _ptr(v), ks, vs, _ptr(slot_mapping), T, k_scale,
                     v_scale, _stream(stream)), "kv_store_e4m3")


def kv_amax_calibrate(k: Optional[torch.Tensor], v: Optional[torch.Tensor],
                      amax_k: Optional[torch.Tensor], amax_v: Optional[torch.Tensor],
                      slot_mapping: Optional[torch.Tensor] = None, stream=None) -> None:
    """amax_k = max(amax_k, max|k|) over tokens with slot >= 0 (same for v);
    amax_* are device float32 scalars updated in place."""
    ref = k if k is not None else v
    H, D = (ref.shape[1], ref.shape[2]) if ref.dim() == 3 else (1, ref.shape[1])
    ks = _rows(k, "k", H * D) if k is not None else 0
    vs = _rows(v, "v", H * D) if v is not None else 0
    for a in (amax_k, amax_v):
        if a is not None:
            _need(a, torch.float32, "amax")
    if slot_mapping is not None:
        _need(slot_mapping, torch.int64, "slot_mapping")
    _check(_amax(_ptr(k), _ptr(v), ks, vs, _ptr(slot_mapping), ref.shape[0], H, D, _ptr(amax_k),
                 _ptr(amax_v), _stream(stream)), "kv_amax_calibrate")


BAND_COUNTS_BYTES = 40   # fp8kv_band_counts: four uint64 counters and a double


def kv_band_counts(x: torch.Tensor, scale: float, slot_mapping: Optional[torch.Tensor] = None,
                   counts: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Adds the clip / flush-to-zero counters and the round-trip error sum of
    quantizing the stored rows of x ([T][H][D] or [T][H*D] bf16) at `scale`
    into `counts` (a zeroed device uint8 tensor of BAND_COUNTS_BYTES when
    None) and returns it; read it with band_counts_dict."""
    row = int(x.shape[1] * (x.shape[2] if x.dim() == 3 else 1))
    stride = _rows(x, "x", row)
    if counts is None:
        counts = torch.zeros(BAND_COUNTS_BYTES, dtype=torch.uint8, device=x.device)
    _need(counts, torch.uint8, "counts", x.device)
    if counts.numel() < BAND_COUNTS_BYTES or not counts.is_contiguous():
        raise ValueError("counts must be a contiguous uint8 tensor of %d bytes" % BAND_COUNTS_BYTES)
    if slot_mapping is not None:
        _need(slot_mapping, torch.int64, "slot_mapping", x.device)
    _check(_band_counts(_ptr(x), stride, _ptr(slot_mapping), x.shape[0], row, float(scale),
                        _ptr(counts), _stream(stream)), "kv_band_counts")
    return counts


def band_counts_dict(counts: torch.Tensor) -> dict:
    """The fields of a fp8kv_band_counts tensor (copies it to the host)."""
    import struct
    c, nz, clip, flush, err = struct.unpack("<4Qd", bytes(counts[:BAND_COUNTS_BYTES].cpu().numpy()))
    return {"count": c, "nonzero": nz, "clipped": clip, "flushed": flush, "rt_err_sum": err}


def scale_from_amax(amax: float, rule: int = 0) -> float:
    s = f32()
    _check(_scale_from_amax(float(amax), int(rule), ctypes.byref(s)), "fp8kv_scale_from_amax")
    return float(s.value)


def decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                          block_size, window=0, split_tokens=0) -> int:
    return int(_ws_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                        block_size, window, split_tokens))


def _table_and_lens(block_table: torch.Tensor, seq_lens: torch.Tensor, B: int, device):
    """block_table int32 [B][max_blocks] and seq_lens int32 [B], contiguous, on
    the cache's device: the kernels read them through raw device pointers."""
    _need(block_table, torch.int32, "block_table", device)
    _need(seq_lens, torch.int32, "seq_lens", device)
    if block_table.dim() != 2 or block_table.shape[0] != B or not block_table.is_contiguous():
        raise ValueError("block_table must be contiguous [B][max_blocks]")
    if seq_lens.numel() != B or not seq_lens.is_contiguous():
        raise ValueError("seq_lens must be contiguous [B]")


def _bias_args(rel_bias, Hq):
    if rel_bias is None:
        return None, 0, 0
    _need(rel_bias, torch.bfloat16, "rel_bias")
    if rel_bias.dim() != 3 or rel_bias.shape[1] != Hq or rel_bias.stride(2) != 1 or \
            rel_bias.stride(1) != rel_bias.shape[2]:
        raise ValueError("rel_bias must be [T][Hq][E] with contiguous [Hq][E] rows")
    return rel_bias, rel_bias.stride(0), rel_bias.shape[2]


def paged_attn_fp8_decode(cache: KVCache, q: torch.Tensor, block_table: torch.Tensor,
                          seq_lens: torch.Tensor, q_scale: float, k_scale: float,
                          v_scale: float, softmax_scale: Optional[float] = None,
                          rel_bias: Optional[torch.Tensor] = None, window: int = 0,
                          out: Optional[torch.Tensor] = None,
                          workspace: Optional[torch.Tensor] = None, split_tokens: int = 0,
                          stream=None) -> torch.Tensor:
    """Decode attention of q [B][Hq][D] (one token per sequence, at position
    seq_len-1) over the cache; returns out [B][Hq][D] bf16."""
    _need(q, torch.bfloat16, "q", cache.device)
    if q.dim() != 3 or not q.is_contiguous() or q.shape[2] != cache.head_dim:
        raise ValueError("q must be contiguous [B][Hq][D]")
    B, Hq, D = q.shape
    _table_and_lens(block_table, seq_lens, B, cache.device)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    rel, bstride, E = _bias_args(rel_bias, Hq)
    if out is None:
        out = torch.empty_like(q)
    mb = block_table.shape[1]
    if workspace is None:
        n = decode_workspace_size(B, Hq, cache.num_kv_heads, D, mb, cache.block_size, window,
                                  split_tokens)
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=cache.device)
    _check(_decode_ex(cache.c(), _ptr(q), Hq, _ptr(block_table), mb, _ptr(seq_lens), B,
                      q_scale, k_scale, v_scale, softmax_scale, _ptr(rel), bstride, E, window,
                      _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                      split_tokens, _stream(stream)), "paged_attn_fp8_decode")
    return out


class DecodeStep:
    """A decode call bound to fixed buffers, validated once.

    ``run()`` launches paged_attn_fp8_decode (or, with k_new and v_new,
    paged_attn_fp8_decode_store) over the buffers' current contents with no
    per-call argument checks: only the stream is looked up.  It is meant for
    decode loops that update q, k_new / v_new, seq_lens and the block table in
    place, as a serving loop or a captured CUDA graph does.  The buffers must
    keep their shapes and stay alive (the object holds references to them);
    the results are those of the one-shot calls, bit for bit."""

    def __init__(self, cache: KVCache, q: torch.Tensor, block_table: torch.Tensor,
                 seq_lens: torch.Tensor, q_scale: float, k_scale: float, v_scale: float,
                 softmax_scale: Optional[float] = None, rel_bias: Optional[torch.Tensor] = None,
                 window: int = 0, out: Optional[torch.Tensor] = None,
                 workspace: Optional[torch.Tensor] = None, k_new: Optional[torch.Tensor] = None,
                 v_new: Optional[torch.Tensor] = None, amax_k: Optional[torch.Tensor] = None,
                 amax_v: Optional[torch.Tensor] = None):
        _need(q, torch.bfloat16, "q", cache.device)
        if q.dim() != 3 or not q.is_contiguous() or q.shape[2] != cache.head_dim:
            raise ValueError("q must be contiguous [B][Hq][D]")
        B, Hq, D = q.shape
        fused = k_new is not None or v_new is not None
        if fused:
            for name, t in (("k_new", k_new), ("v_new", v_new)):
                if t is None:
                    raise ValueError("k_new and v_new go together")
                _need(t, torch.bfloat16, name, cache.device)
                if tuple(t.shape) != (B, cache.num_kv_heads, D) or not t.is_contiguous():
                    raise ValueError("%s must be contiguous [B][Hkv][D]" % name)
            for a in (amax_k, amax_v):
                if a is not None:
                    _need(a, torch.float32, "amax", cache.device)
        elif amax_k is not None or amax_v is not None:
            raise ValueError("amax_k / amax_v need k_new and v_new")
        _table_and_lens(block_table, seq_lens, B, cache.device)
        if softmax_scale is None:
            softmax_scale = 1.0 / math.sqrt(D)
        rel, bstride, E = _bias_args(rel_bias, Hq)
        if out is None:
            out = torch.empty_like(q)
        _need(out, torch.bfloat16, "out", cache.device)
        if tuple(out.shape) != tuple(q.shape) or not out.is_contiguous():
            raise ValueError("out must be contiguous [B][Hq][D]")
        mb = block_table.shape[1]
        n = decode_workspace_size(B, Hq, cache.num_kv_heads, D, mb, cache.block_size, window, 0)
        if workspace is None:
            workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=cache.device)
        _need(workspace, torch.uint8, "workspace", cache.device)
        if workspace.numel() < n or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous uint8 tensor of >= %d bytes" % n)
        self.out = out
        self._keep = (cache, q, block_table, seq_lens, rel, out, workspace, k_new, v_new, amax_k,
                      amax_v)
        ws_bytes = workspace.numel()
        if fused:
            self._fn, self._name = _decode_store, "paged_attn_fp8_decode_store"
            self._args = (cache.c(), _ptr(q), Hq, _ptr(k_new), _ptr(v_new), _ptr(block_table), mb,
                          _ptr(seq_lens), B, q_scale, k_scale, v_scale, softmax_scale, _ptr(rel),
                          bstride, E, window, _ptr(amax_k), _ptr(amax_v), _ptr(out),
                          _ptr(workspace), ws_bytes)
        else:
            self._fn, self._name = _decode_ex, "paged_attn_fp8_decode"
            self._args = (cache.c(), _ptr(q), Hq, _ptr(block_table), mb, _ptr(seq_lens), B,
                          q_scale, k_scale, v_scale, softmax_scale, _ptr(rel), bstride, E, window,
                          _ptr(out), _ptr(workspace), ws_bytes, 0)

    def run(self, stream=None) -> torch.Tensor:
        _check(self._fn(*self._args, _stream(stream)), self._name)
        return self.out

    def cuda_graph(self, pre=None, post=None) -> "torch.cuda.CUDAGraph":
        """Capture one step into a CUDA graph: ``pre()`` (for example the copy
        of the step's inputs from pinned host memory into the bound buffers),
        ``run()``, then ``post()`` (for example the copy of out to the host).
        ``graph.replay()`` then runs the whole step as one launch on the
        current stream, reading the buffers' contents at replay time.  The
        step runs once before the capture (on the current stream, which is
        then synchronized), so the launch set-up is done outside it."""
        self.run()
        torch.cuda.current_stream().synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            if pre is not None:
                pre()
            self.run()
            if post is not None:
                post()
        return graph


def kv_store_e4m3_per_token(cache: KVCache, k: torch.Tensor, v: torch.Tensor,
                            slot_mapping: torch.Tensor, k_scales: torch.Tensor,
                            v_scales: torch.Tensor, stream=None) -> None:
    """Quantize k, v [T][Hkv][D] bf16 with one scale per token and head
    (max|x|/448) into the cache; the scales go to k_scales / v_scales, float32
    [num_blocks][Hkv][block_size] on the cache's device."""
    row = cache.num_kv_heads * cache.head_dim
    ks, vs = _rows(k, "k", row), _rows(v, "v", row)
    _need(slot_mapping, torch.int64, "slot_mapping", cache.device)
    shape = (cache.num_blocks, cache.num_kv_heads, cache.block_size)
    for name, t in (("k_scales", k_scales), ("v_scales", v_scales)):
        _need(t, torch.float32, name, cache.device)
        if tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError("%s must be contiguous float32 %s" % (name, shape))
    _check(_store_pt(cache.c(), _ptr(k), _ptr(v), ks, vs, _ptr(slot_mapping), k.shape[0],
                     _ptr(k_scales), _ptr(v_scales), _stream(stream)), "kv_store_e4m3_per_token")


def paged_attn_fp8_decode_per_token(cache: KVCache, q: torch.Tensor, block_table: torch.Tensor,
                                    seq_lens: torch.Tensor, q_scale: float,
                                    k_scales: torch.Tensor, v_scales: torch.Tensor,
                                    softmax_scale: Optional[float] = None,
                                    rel_bias: Optional[torch.Tensor] = None, window: int = 0,
                                    out: Optional[torch.Tensor] = None,
                                    workspace: Optional[torch.Tensor] = None,
                                    stream=None) -> torch.Tensor:
    """Decode over a cache written by kv_store_e4m3_per_token (its scale
    arrays k_scales, v_scales); returns out [B][Hq][D] bf16."""
    _need(q, torch.bfloat16, "q", cache.device)
    if q.dim() != 3 or not q.is_contiguous() or q.shape[2] != cache.head_dim:
        raise ValueError("q must be contiguous [B][Hq][D]")
    B, Hq, D = q.shape
    shape = (cache.num_blocks, cache.num_kv_heads, cache.block_size)
    for name, t in (("k_scales", k_scales), ("v_scales", v_scales)):
        _need(t, torch.float32, name, cache.device)
        if tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError("%s must be contiguous float32 %s" % (name, shape))
    _table_and_lens(block_table, seq_lens, B, cache.device)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    rel, bstride, E = _bias_args(rel_bias, Hq)
    if out is None:
        out = torch.empty_like(q)
    mb = block_table.shape[1]
    if workspace is None:
        n = decode_workspace_size(B, Hq, cache.num_kv_heads, D, mb, cache.block_size, window, 0)
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=cache.device)
    _check(_decode_pt(cache.c(), _ptr(q), Hq, _ptr(block_table), mb, _ptr(seq_lens), B, q_scale,
                      softmax_scale, _ptr(k_scales), _ptr(v_scales), _ptr(rel), bstride, E, window,
                      _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                      _stream(stream)), "paged_attn_fp8_decode_per_token")
    return out


def paged_attn_fp8_decode_store(cache: KVCache, q: torch.Tensor, k_new: torch.Tensor,
                                v_new: torch.Tensor, block_table: torch.Tensor,
                                seq_lens: torch.Tensor, q_scale: float, k_scale: float,
                                v_scale: float, softmax_scale: Optional[float] = None,
                                rel_bias: Optional[torch.Tensor] = None, window: int = 0,
                                amax_k: Optional[torch.Tensor] = None,
                                amax_v: Optional[torch.Tensor] = None,
                                out: Optional[torch.Tensor] = None,
                                workspace: Optional[torch.Tensor] = None,
                                stream=None) -> torch.Tensor:
    """One decode step: store k_new / v_new [B][Hkv][D] (each sequence's new
    token, at position seq_len-1) into the cache, raise amax_k / amax_v
    (device float32 scalars, optional), and attend; returns out [B][Hq][D]."""
    _need(q, torch.bfloat16, "q", cache.device)
    if q.dim() != 3 or not q.is_contiguous() or q.shape[2] != cache.head_dim:
        raise ValueError("q must be contiguous [B][Hq][D]")
    B, Hq, D = q.shape
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        _need(t, torch.bfloat16, name, cache.device)
        if tuple(t.shape) != (B, cache.num_kv_heads, D) or not t.is_contiguous():
            raise ValueError("%s must be contiguous [B][Hkv][D]" % name)
    for a in (amax_k, amax_v):
        if a is not None:
            _need(a, torch.float32, "amax", cache.device)
    _table_and_lens(block_table, seq_lens, B, cache.device)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    rel, bstride, E = _bias_args(rel_bias, Hq)
    if out is None:
        out = torch.empty_like(q)
    mb = block_table.shape[1]
    if workspace is None:
        n = decode_workspace_size(B, Hq, cache.num_kv_heads, D, mb, cache.block_size, window, 0)
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=cache.device)
    _check(_decode_store(cache.c(), _ptr(q), Hq, _ptr(k_new), _ptr(v_new), _ptr(block_table), mb,
                         _ptr(seq_lens), B, q_scale, k_scale, v_scale, softmax_scale, _ptr(rel),
                         bstride, E, window, _ptr(amax_k), _ptr(amax_v), _ptr(out),
                         _ptr(workspace), workspace.numel() * workspace.element_size(),
                         _stream(stream)), "paged_attn_fp8_decode_store")
    return out


def paged_attn_fp8_decode_noalloc(cache: KVCache, q: torch.Tensor, block_table: torch.Tensor,
                                  seq_lens: torch.Tensor, q_scale: float, k_scale: float,
                                  v_scale: float, softmax_scale: Optional[float] = None,
                                  rel_bias: Optional[torch.Tensor] = None, window: int = 0,
                                  out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """paged_attn_fp8_decode for callers that cannot supply a workspace: the
    split partials go to the library's fixed 16 MiB device buffer (see
    include/fp8kv.h).  Calls that may overlap on the GPU race on that buffer.
    The arguments are checked like paged_attn_fp8_decode's before the call."""
    _need(q, torch.bfloat16, "q", cache.device)
    if q.dim() != 3 or not q.is_contiguous() or q.shape[2] != cache.head_dim:
        raise ValueError("q must be contiguous [B][Hq][D]")
    B, Hq, D = q.shape
    _table_and_lens(block_table, seq_lens, B, cache.device)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    rel, bstride, E = _bias_args(rel_bias, Hq)
    if out is None:
        out = torch.empty_like(q)
    _check(_decode_noalloc(cache.c(), _ptr(q), Hq, _ptr(block_table), block_table.shape[1],
                           _ptr(seq_lens), B, q_scale, k_scale, v_scale, softmax_scale,
                           _ptr(rel), bstride, E, window, _ptr(out), _stream(stream)),
           "paged_attn_fp8_decode_noalloc")
    return out


def attn_fp8_varlen_prefill(cache: KVCache, q: torch.Tensor, cu_seqlens_q: torch.Tensor,
                            seq_lens_k: torch.Tensor, block_table: torch.Tensor,
                            max_seqlen_q: int, q_scale: float, k_scale: float, v_scale: float,
                            softmax_scale: Optional[float] = None,
                            rel_bias: Optional[torch.Tensor] = None, window: int = 0,
                            out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Causal (optionally windowed) prefill of q [Tq][Hq][D] over the cache;
    sequence b's queries are the last cu_seqlens_q[b+1]-cu_seqlens_q[b] of its
    seq_lens_k[b] keys.  Returns out [Tq][Hq][D] bf16."""
    _need(q, torch.bfloat16, "q", cache.device)
    if q.dim() != 3 or not q.is_contiguous() or q.shape[2] != cache.head_dim:
        raise ValueError("q must be contiguous [Tq][Hq][D]")
    Tq, Hq, D = q.shape
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q", cache.device)
    _need(seq_lens_k, torch.int32, "seq_lens_k", cache.device)
    _need(block_table, torch.int32, "block_table", cache.device)
    B = seq_lens_k.numel()
    if cu_seqlens_q.numel() != B + 1 or block_table.shape[0] != B or \
            not block_table.is_contiguous():
        raise ValueError("cu_seqlens_q [B+1], seq_lens_k [B], block_table [B][max_blocks]")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    rel, bstride, E = _bias_args(rel_bias, Hq)
    if out is None:
        out = torch.empty_like(q)
    _check(_prefill(cache.c(), _ptr(q), Hq, _ptr(cu_seqlens_q), _ptr(seq_lens_k),
                    _ptr(block_table), block_table.shape[1], B, int(max_seqlen_q), q_scale,
                    k_scale, v_scale, softmax_scale, _ptr(rel), bstride, E, window, _ptr(out),
                    None, 0, _stream(stream)), "attn_fp8_varlen_prefill")
    return out


def attn_fp8_varlen_prefill_per_token(cache: KVCache, q: torch.Tensor, cu_seqlens_q: torch.Tensor,
                                      seq_lens_k: torch.Tensor, block_table: torch.Tensor,
                                      max_seqlen_q: int, q_scale: float, k_scales: torch.Tensor,
                                      v_scales: torch.Tensor, softmax_scale: Optional[float] = None,
                                      rel_bias: Optional[torch.Tensor] = None, window: int = 0,
                                      out: Optional[torch.Tensor] = None,
                                      stream=None) -> torch.Tensor:
    """attn_fp8_varlen_prefill over a cache written by kv_store_e4m3_per_token
    (its scale arrays k_scales, v_scales); returns out [Tq][Hq][D] bf16."""
    _need(q, torch.bfloat16, "q", cache.device)
    if q.dim() != 3 or not q.is_contiguous() or q.shape[2] != cache.head_dim:
        raise ValueError("q must be contiguous [Tq][Hq][D]")
    Tq, Hq, D = q.shape
    shape = (cache.num_blocks, cache.num_kv_heads, cache.block_size)
    for name, t in (("k_scales", k_scales), ("v_scales", v_scales)):
        _need(t, torch.float32, name, cache.device)
        if tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError("%s must be contiguous float32 %s" % (name, shape))
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q", cache.device)
    _need(seq_lens_k, torch.int32, "seq_lens_k", cache.device)
    _need(block_table, torch.int32, "block_table", cache.device)
    B = seq_lens_k.numel()
    if cu_seqlens_q.numel() != B + 1 or block_table.shape[0] != B or \
            not block_table.is_contiguous():
        raise ValueError("cu_seqlens_q [B+1], seq_lens_k [B], block_table [B][max_blocks]")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    rel, bstride, E = _bias_args(rel_bias, Hq)
    if out is None:
        out = torch.empty_like(q)
    _check(_prefill_pt(cache.c(), _ptr(q), Hq, _ptr(cu_seqlens_q), _ptr(seq_lens_k),
                       _ptr(block_table), block_table.shape[1], B, int(max_seqlen_q), q_scale,
                       softmax_scale, _ptr(k_scales), _ptr(v_scales), _ptr(rel), bstride, E, window,
                       _ptr(out), _stream(stream)), "attn_fp8_varlen_prefill_per_token")
    return out


def set_prefill_max_ctas(max_ctas: int) -> None:
    """Caps the CTAs of the persistent head_dim-128 prefill (0: one per SM)."""
    _check(_prefill_max_ctas(int(max_ctas)), "fp8kv_set_prefill_max_ctas")


def test_drop_first_copy(on: bool = True) -> None:
    """Test hook: the next decode launch skips each CTA's first key-tile copy,
    so its bounded wait runs out (see include/fp8kv.h)."""
    _check(_drop_first_copy(1 if on else 0), "fp8kv_test_drop_first_copy")


def device_error(clear: bool = True) -> int:
    """The current device's error word (synchronizes); 0 when clean."""
    w = ctypes.c_uint32()
    _check(_device_error(ctypes.byref(w), 1 if clear else 0), "fp8kv_device_error")
    return int(w.value)


__all__ = ["KVCache", "Fp8KVError", "DecodeStep", "kv_store_e4m3", "kv_amax_calibrate", "kv_band_counts",
           "band_counts_dict", "BAND_COUNTS_BYTES", "scale_from_amax",
           "paged_attn_fp8_decode", "paged_attn_fp8_decode_noalloc", "paged_attn_fp8_decode_store",
           "kv_store_e4m3_per_token", "paged_attn_fp8_decode_per_token",
           "attn_fp8_varlen_prefill", "attn_fp8_varlen_prefill_per_token", "set_prefill_max_ctas",
           "decode_workspace_size",
           "cache_bytes", "device_error", "status_string", "LIB_PATH", "EXPORTED"]
