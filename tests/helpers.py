"""Shared helpers of the GPU parity tests: run the library on seeded inputs
and compute the oracle's rows for the same inputs."""
import math

import numpy as np
import torch

import oracle
import workloads

ATOL = 2e-2
RTOL = 2e-2


def bits(t):
    return workloads.bf16_bits(t)


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    if bad.any():
        i = np.unravel_index(np.argmax(err - (ATOL + RTOL * np.abs(ref))), err.shape)
        raise AssertionError("%s: %d of %d outside 2e-2 abs + 2e-2 rel; worst at %s: got %r "
                             "ref %r" % (what, int(bad.sum()), bad.size, i, got[i], ref[i]))
    return float(err.max()) if err.size else 0.0


class OracleKV:
    """Oracle-side quantized keys/values of a PagedKV, per (sequence, KV head),
    computed from the bf16 inputs on demand (never from the GPU cache)."""

    def __init__(self, kv, k_scale, v_scale):
        self.kv, self.sk, self.sv = kv, k_scale, v_scale
        self.starts = kv.tok_start.cpu().tolist()
        self.lens = kv.seq_lens.cpu().tolist()
        self._memo = {}

    def seq(self, b, kvh):
        key = (b, kvh)
        if key not in self._memo:
            s, L = self.starts[b], self.lens[b]
            k = self.kv.k[s:s + L, kvh].contiguous()
            v = self.kv.v[s:s + L, kvh].contiguous()
            self._memo = {key: (oracle.quantize(bits(k), self.sk), oracle.quantize(bits(v), self.sv))}
        return self._memo[key]


def oracle_decode_rows(inp, rows, q_scale, k_scale, v_scale, softmax_scale=None, window=0,
                       rel=None):
    """Oracle output rows [len(rows)][D] for decode rows (b, h): the query of
    sequence b, head h at position len-1."""
    kv = inp["kv"]
    q = inp["q"]
    B, Hq, D = q.shape
    Hkv = kv.k.shape[1]
    G = Hq // Hkv
    sigma = softmax_scale if softmax_scale is not None else 1 / math.sqrt(D)
    okv = OracleKV(kv, k_scale, v_scale)
    out = []
    for b, h in sorted(rows, key=lambda r: (r[0], r[1] // G)):
        k8, v8 = okv.seq(b, h // G)
        q8 = oracle.quantize(bits(q[b, h].contiguous()), q_scale)
        bias = None if rel is None else bits(rel[b, h].contiguous())
        L = okv.lens[b]
        out.append(((b, h), oracle.attend_row(q8, k8, v8, L - 1, sigma, q_scale, k_scale, v_scale,
                                              bias=bias, window=window)))
    d = dict(out)
    return np.stack([d[(b, h)] for b, h in rows]) if rows else np.zeros((0, D))


def oracle_store(kv, k_scale, v_scale, fill=0xA5):
    """Oracle's paged cache for the whole PagedKV (small cases only)."""
    shape = (kv.num_blocks, kv.k.shape[1], kv.block_size, kv.k.shape[2])
    ck = np.full(shape, fill, dtype=np.uint8)
    cv = np.full(shape, fill, dtype=np.uint8)
    oracle.kv_store(ck, cv, bits(kv.k.cpu()), bits(kv.v.cpu()), kv.slot_mapping.cpu().numpy(),
                    k_scale, v_scale, kv.block_size)
    return ck, cv


def to_device(kv, dev):
    return workloads.PagedKV(k=kv.k.to(dev), v=kv.v.to(dev), seq_lens=kv.seq_lens.to(dev),
                             tok_start=kv.tok_start.to(dev), block_table=kv.block_table.to(dev),
                             slot_mapping=kv.slot_mapping.to(dev), num_blocks=kv.num_blocks,
                             block_size=kv.block_size)


def oracle_prefill_rows(inp, rows, q_scale, k_scale, v_scale, softmax_scale=None, window=0,
                        rel=None):
    """Oracle output rows for prefill rows (t, h): query token t (global index
    into q) of head h; its sequence's queries are the last q_len of k_len keys."""
    kv = inp["kv"]
    q = inp["q"]
    Tq, Hq, D = q.shape
    Hkv = kv.k.shape[1]
    G = Hq // Hkv
    sigma = softmax_scale if softmax_scale is not None else 1 / math.sqrt(D)
    cu = inp["cu_seqlens_q"].cpu().tolist()
    okv = OracleKV(kv, k_scale, v_scale)
    q_lens, k_lens = inp["q_lens"], inp["k_lens"]
    res = {}
    seq_of = np.searchsorted(np.asarray(cu), np.asarray([t for t, _ in rows]), side="right") - 1
    order = sorted(range(len(rows)), key=lambda i: (seq_of[i], rows[i][1] // G))
    for i in order:
        t, h = rows[i]
        b = int(seq_of[i])
        k8, v8 = okv.seq(b, h // G)
        pos = k_lens[b] - q_lens[b] + (t - cu[b])
        q8 = oracle.quantize(bits(q[t, h].contiguous()), q_scale)
        bias = None if rel is None else bits(rel[t, h].contiguous())
        res[i] = oracle.attend_row(q8, k8, v8, pos, sigma, q_scale, k_scale, v_scale, bias=bias,
                                   window=window)
    return np.stack([res[i] for i in range(len(rows))]) if rows else np.zeros((0, D))
