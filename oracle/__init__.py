"""CPU oracle for the fp8 e4m3 KV cache path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  The product library never does,
and this package never imports the product (``fp8_e4m3_kv_gb300``): the two
share nothing but the seeded input generators in ``workloads``.

The arithmetic lives in ``fp8kv_oracle.c`` (plain C, float64 attention); this
module only compiles it and marshals numpy arrays.  Every function cites, in
the C source, the page section it follows:

* e4m3 decode / encode (nearest-even, saturating to +-448): OCP E4M3 and
  vLLM PR 54705, "Purpose" (quant-on-store clamp).  Pinned by the OCP code
  table, the pages' printed values (448; |V| = 1,272 clips at scale 1 but not
  at 3) and an exhaustive cross-check against torch's float8_e4m3fn cast.
* store quantization and paged scatter: PR 54705 "Purpose".  Pinned through
  the codec pins and a layout round trip.
* amax and scale rules: Qwen3.8-27B-FP8-KVcal card ("What it fixes",
  "Rebuild / reproduce") and PR 54705's calibration paragraph.  Pinned by the
  printed 1,272 -> 3.69 and amax -> 448 mapping.
* attention (form 4: descale fold; form 5: dequantize-then-attend): PR 54705
  "Purpose", descale handling.  Pinned by closed forms (one key, constant
  keys, bias selecting one distance, window/causal counts), by scipy softmax
  on tiny cases, and by form 4 == form 5.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8kv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

E4M3_MAX = 448.0


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` with gcc (OpenMP on)."""
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    ):
        tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c99",
             "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    i64, i32, f32, f64 = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_double
    lib.or_e4m3_decode.restype = f64
    lib.or_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.or_e4m3_encode.restype = ctypes.c_uint8
    lib.or_e4m3_encode.argtypes = [f32]
    lib.or_quantize.restype = ctypes.c_uint8
    lib.or_quantize.argtypes = [ctypes.c_uint16, f32]
    lib.or_quantize_array.restype = None
    lib.or_quantize_array.argtypes = [P, i64, f32, P]
    lib.or_decode_array.restype = None
    lib.or_decode_array.argtypes = [P, i64, P]
    lib.or_kv_store.restype = ctypes.c_int
    lib.or_kv_store.argtypes = [P, P, i64, i32, i32, i32, P, P, i64, i64, P, i64, f32, f32]
    lib.or_amax.restype = f32
    lib.or_amax.argtypes = [P, i64, P, i64, i32, i32, f32]
    lib.or_scale_from_amax.restype = ctypes.c_int
    lib.or_row_scale.argtypes = [P, i32]
    lib.or_row_scale.restype = f32
    lib.or_quantize_per_token.argtypes = [P, i64, i32, P, P]
    lib.or_quantize_per_token.restype = None
    lib.or_attend_row_pt.argtypes = [i32, P, P, P, i64, P, P, i64, i64, f64, f64, P, i32, i32, P]
    lib.or_attend_row_pt.restype = None
    lib.or_band_counts.argtypes = [P, i64, P, i64, i32, f32, P, P]
    lib.or_band_counts.restype = None
    lib.or_scale_from_amax.argtypes = [f32, ctypes.c_int, ctypes.POINTER(f32)]
    lib.or_attend_row.restype = None
    lib.or_attend_row.argtypes = [i32, P, P, P, i64, i64, i64, f64, f64, f64, f64,
                                  P, i32, i32, ctypes.c_int, P]
    lib.or_attend_rows.restype = None
    lib.or_attend_rows.argtypes = [i64, i32, P, P, P, P, P, i64, P, P, f64, f64, f64,
                                   f64, P, P, i32, i32, ctypes.c_int, P]
    lib.or_num_threads.restype = ctypes.c_int
    lib.or_num_threads.argtypes = []
    _lib = lib
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(x) -> np.ndarray:
    """bf16 data as its raw uint16 bit patterns (numpy has no bf16 dtype)."""
    x = np.asarray(x)
    if x.dtype != np.uint16:
        raise TypeError("bf16 arrays are passed as uint16 bit patterns")
    return np.ascontiguousarray(x)


# ---------------------------------------------------------------- codec
def e4m3_decode(b: int) -> float:
    return _load().or_e4m3_decode(int(b))


def e4m3_encode(x: float) -> int:
    return int(_load().or_e4m3_encode(float(x)))


def decode_array(codes: np.ndarray) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _load().or_decode_array(_ptr(c), c.size, _ptr(out))
    return out


def quantize(x_bf16: np.ndarray, scale: float) -> np.ndarray:
    """bf16 (uint16 bits) -> e4m3 bytes: fp32 x/scale, clamp +-448, RNE."""
    x = _u16(x_bf16)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().or_quantize_array(_ptr(x), x.size, float(scale), _ptr(out))
    return out


def encode_f32(x: np.ndarray) -> np.ndarray:
    """fp32 values -> e4m3 bytes (no division), one at a time."""
    lib = _load()
    x = np.asarray(x, dtype=np.float32).ravel()
    return np.array([lib.or_e4m3_encode(float(v)) for v in x], dtype=np.uint8)


# ---------------------------------------------------------------- store / amax
def kv_store(cache_k, cache_v, k_bf16, v_bf16, slot_mapping, k_scale, v_scale,
             block_size):
    """Quantize and scatter k/v ([T][Hkv][D] uint16 bits) into the caches
    ([num_blocks][Hkv][block_size][D] uint8), in place."""
    k = _u16(k_bf16)
    v = _u16(v_bf16)
    T, H, D = k.shape
    nb = cache_k.shape[0]
    assert cache_k.shape == (nb, H, block_size, D)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    assert cache_k.flags.c_contiguous and cache_v.flags.c_contiguous
    rc = _load().or_kv_store(_ptr(cache_k), _ptr(cache_v), nb, block_size, H, D,
                             _ptr(k), _ptr(v), H * D, H * D, _ptr(sm), T,
                             float(k_scale), float(v_scale))
    if rc != 0:
        raise ValueError("slot out of range")


def amax(x_bf16, slot_mapping=None, amax_in: float = 0.0) -> float:
    x = _u16(x_bf16)
    T = x.shape[0]
    row = int(np.prod(x.shape[1:]))
    sm = None if slot_mapping is None else np.ascontiguousarray(slot_mapping, dtype=np.int64)
    return float(_load().or_amax(_ptr(x), row, _ptr(sm), T, 1, row, float(amax_in)))


def band_counts(x_bf16, scale: float, slot_mapping=None) -> dict:
    """Clip / flush-to-zero counters and round-trip error sum of quantizing
    the stored values (rows of x, skipping tokens with slot < 0) at scale."""
    x = _u16(x_bf16)
    T = x.shape[0]
    row = int(np.prod(x.shape[1:]))
    sm = None if slot_mapping is None else np.ascontiguousarray(slot_mapping, dtype=np.int64)
    counts = np.zeros(4, dtype=np.int64)
    err = np.zeros(1, dtype=np.float64)
    _load().or_band_counts(_ptr(x), row, _ptr(sm), T, row, float(scale), _ptr(counts), _ptr(err))
    return {"count": int(counts[0]), "nonzero": int(counts[1]), "clipped": int(counts[2]),
            "flushed": int(counts[3]), "rt_err_sum": float(err[0])}


def quantize_per_token(x_bf16, row_len: int):
    """Rows of row_len bf16 values -> (codes uint8 [rows][row_len], scales
    float32 [rows]), one scale per row (a token's head)."""
    x = _u16(x_bf16).reshape(-1, row_len)
    codes = np.zeros(x.shape, dtype=np.uint8)
    scales = np.zeros(x.shape[0], dtype=np.float32)
    _load().or_quantize_per_token(_ptr(x), x.shape[0], row_len, _ptr(codes), _ptr(scales))
    return codes, scales


def attend_row_pt(q8, k8, v8, sk, sv, pos_q, sigma, s_q, bias=None, window=0):
    """One query row over keys with per-token scales (k8, v8 [len][D] codes,
    sk, sv [len] float32)."""
    q8 = np.ascontiguousarray(q8, dtype=np.uint8)
    k8 = np.ascontiguousarray(k8, dtype=np.uint8)
    v8 = np.ascontiguousarray(v8, dtype=np.uint8)
    sk = np.ascontiguousarray(sk, dtype=np.float32)
    sv = np.ascontiguousarray(sv, dtype=np.float32)
    D = q8.shape[0]
    out = np.zeros(D, dtype=np.float64)
    b = None if bias is None else _u16(bias)
    E = 0 if b is None else b.shape[0]
    _load().or_attend_row_pt(D, _ptr(q8), _ptr(k8), _ptr(v8), D, _ptr(sk), _ptr(sv), k8.shape[0],
                             int(pos_q), float(sigma), float(s_q), _ptr(b), E, int(window),
                             _ptr(out))
    return out


def scale_from_amax(a: float, rule: int = 0) -> float:
    s = ctypes.c_float()
    rc = _load().or_scale_from_amax(float(a), int(rule), ctypes.byref(s))
    if rc != 0:
        raise ValueError("scale would not be finite and positive")
    return float(s.value)


# ---------------------------------------------------------------- attention
def attend_row(q8, k8, v8, pos_q, sigma, s_q, s_k, s_v, bias=None, window=0,
               form=4):
    """One query row.  q8: [D] e4m3 bytes; k8, v8: [len_k][D] e4m3 bytes in
    token order; bias: None or [E] uint16 bf16 bits indexed by distance."""
    q8 = np.ascontiguousarray(q8, dtype=np.uint8)
    k8 = np.ascontiguousarray(k8, dtype=np.uint8)
    v8 = np.ascontiguousarray(v8, dtype=np.uint8)
    D = q8.shape[-1]
    L = k8.shape[0]
    b = None if bias is None else _u16(bias)
    E = 0 if b is None else b.shape[-1]
    out = np.zeros(D, dtype=np.float64)
    _load().or_attend_row(D, _ptr(q8), _ptr(k8), _ptr(v8), D, L, int(pos_q),
                          float(sigma), float(s_q), float(s_k), float(s_v), _ptr(b),
                          E, int(window), int(form), _ptr(out))
    return out


def attend_rows(head_dim, q8, q_off, k8, v8, kv_off, ld, len_k, pos_q, sigma, s_q,
                s_k, s_v, bias=None, bias_off=None, rel_extent=0, window=0, form=4):
    """Many rows (see or_attend_rows).  Offsets are element offsets into the
    flat q8 / k8 / v8 / bias arrays; returns [n_rows][D] float64."""
    q8 = np.ascontiguousarray(q8, dtype=np.uint8)
    k8 = np.ascontiguousarray(k8, dtype=np.uint8)
    v8 = np.ascontiguousarray(v8, dtype=np.uint8)
    q_off = np.ascontiguousarray(q_off, dtype=np.int64)
    kv_off = np.ascontiguousarray(kv_off, dtype=np.int64)
    len_k = np.ascontiguousarray(len_k, dtype=np.int64)
    pos_q = np.ascontiguousarray(pos_q, dtype=np.int64)
    n = q_off.shape[0]
    D = int(head_dim)
    b = None if bias is None else _u16(bias)
    bo = None if bias is None else np.ascontiguousarray(bias_off, dtype=np.int64)
    out = np.zeros((n, D), dtype=np.float64)
    _load().or_attend_rows(n, D, _ptr(q8), _ptr(q_off), _ptr(k8), _ptr(v8),
                           _ptr(kv_off), int(ld), _ptr(len_k), _ptr(pos_q),
                           float(sigma), float(s_q), float(s_k), float(s_v), _ptr(b),
                           _ptr(bo), int(rel_extent), int(window), int(form), _ptr(out))
    return out


def num_threads() -> int:
    return int(_load().or_num_threads())
