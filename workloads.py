"""Seeded synthetic inputs for the fp8 e4m3 KV cache path.

This module only draws random tensors and lays out the paged-cache
book-keeping (sequence lengths, block tables, slot mappings).  It holds none
of the method's arithmetic: no quantization, no attention.  Both the CUDA
library's tests / bench and the CPU oracle take their inputs from here.

The value distributions stand in for the pages' model activations (vLLM PR
54705, evidence document Tier 2 table: |K| max 55.8-73.5, |V| max up to
1,272, V clipping at unity scale ~1.3e-4 in the worst pool; Qwen3.8-27B-
FP8-KVcal card, "Honesty notes": post-norm K amax 11.6-23.1, V amax
14.9-114.6).  No dataset is read.

Tensors are torch tensors on the requested device; random draws use a
torch.Generator seeded per workload, so a workload is reproducible on one
machine and torch version.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import torch

# |V| = 17.47 * t(3): 448 / 17.47 = 25.64 is the 1 - 6.5e-5 quantile of a
# Student t with 3 degrees of freedom, so |V| > 448 (clipping at unity scale)
# occurs with probability ~1.3e-4, the worst-pool rate of the Tier 2 table.
V_T3_SCALE = 17.47
V_CLAMP = 1272.0          # the largest |V| the Tier 2 table reports


@dataclasses.dataclass
class PagedKV:
    """K/V tokens of a batch of sequences plus their paged-cache placement.

    k, v:          bf16 [T][Hkv][D], the tokens of all sequences, sequence
                   after sequence, each in position order.
    seq_lens:      int32 [B] keys per sequence.
    tok_start:     int64 [B+1] offset of each sequence's first token in k, v.
    block_table:   int32 [B][max_blocks], physical block of each logical block
                   (-1 past the sequence end).
    slot_mapping:  int64 [T], block*block_size + offset for each token.
    num_blocks:    physical blocks in the pool (a random permutation is used,
                   plus spare blocks no sequence owns).
    """
    k: torch.Tensor
    v: torch.Tensor
    seq_lens: torch.Tensor
    tok_start: torch.Tensor
    block_table: torch.Tensor
    slot_mapping: torch.Tensor
    num_blocks: int
    block_size: int

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, g, device, dtype=torch.float32):
    return torch.randn(shape, generator=g, device=device, dtype=dtype)


def _student_t3(shape, g, device):
    """Student t with 3 degrees of freedom: z0 / sqrt((z1^2+z2^2+z3^2)/3)."""
    z0 = _normal(shape, g, device)
    chi2 = torch.zeros(shape, device=device)
    for _ in range(3):
        z = _normal(shape, g, device)
        chi2.add_(z * z)
    return z0 / torch.sqrt(chi2 / 3.0)


def draw_values(shape, dist: str, g, device, amax: Optional[float] = None) -> torch.Tensor:
    """bf16 values of one of the recipes:
    normal   N(0, 1)
    v_t3     17.47 * t(3) clamped to +-1272 (heavy-tailed V of a global layer)
    t3_amax  t(3) rescaled so max|x| = amax
    n_amax   N(0, 1) rescaled so max|x| = amax
    zeros    all zero
    """
    if dist == "normal":
        x = _normal(shape, g, device)
    elif dist == "v_t3":
        x = (V_T3_SCALE * _student_t3(shape, g, device)).clamp_(-V_CLAMP, V_CLAMP)
    elif dist in ("t3_amax", "n_amax"):
        x = _student_t3(shape, g, device) if dist == "t3_amax" else _normal(shape, g, device)
        x = x * (float(amax) / float(x.abs().max()))
    elif dist == "zeros":
        x = torch.zeros(shape, device=device)
    else:
        raise ValueError(dist)
    return x.to(torch.bfloat16)


def make_paged_kv(seq_lens: List[int], Hkv: int, D: int, block_size: int, *,
                  g, device, k_dist="normal", v_dist="normal", k_amax=None,
                  v_amax=None, spare_blocks: int = 3, plant_v: bool = False,
                  max_blocks: Optional[int] = None) -> PagedKV:
    B = len(seq_lens)
    T = int(sum(seq_lens))
    k = draw_values((T, Hkv, D), k_dist, g, device, k_amax)
    v = draw_values((T, Hkv, D), v_dist, g, device, v_amax)
    if plant_v and T > 0:
        # one element at the clamp value, at a drawn position and sign
        idx = int(torch.randint(0, T * Hkv * D, (1,), generator=g, device=device).item())
        sign = 1.0 if int(torch.randint(0, 2, (1,), generator=g, device=device).item()) else -1.0
        v.view(-1)[idx] = sign * V_CLAMP
    nblk = [(L + block_size - 1) // block_size for L in seq_lens]
    mb = max(nblk + [1]) if max_blocks is None else max_blocks
    num_blocks = sum(nblk) + spare_blocks
    perm = torch.randperm(num_blocks, generator=g, device=device).to(torch.int32)
    bt = torch.full((B, mb), -1, dtype=torch.int32, device=device)
    tok_start = [0]
    slots = []
    used = 0
    for b, L in enumerate(seq_lens):
        n = nblk[b]
        bt[b, :n] = perm[used:used + n]
        used += n
        if L > 0:
            pos = torch.arange(L, device=device, dtype=torch.int64)
            slots.append(bt[b, pos // block_size].to(torch.int64) * block_size + pos % block_size)
        tok_start.append(tok_start[-1] + L)
    slot_mapping = torch.cat(slots) if slots else torch.zeros(0, dtype=torch.int64, device=device)
    return PagedKV(k=k, v=v,
                   seq_lens=torch.tensor(seq_lens, dtype=torch.int32, device=device),
                   tok_start=torch.tensor(tok_start, dtype=torch.int64, device=device),
                   block_table=bt, slot_mapping=slot_mapping,
                   num_blocks=num_blocks, block_size=block_size)


# ---------------------------------------------------------------------------
# Workloads.  Each returns a dict of tensors; names say what they are.
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class DecodeSpec:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    block_size: int
    ctx_lo: int
    ctx_hi: int
    k_dist: str = "normal"
    v_dist: str = "normal"
    k_amax_range: Optional[tuple] = None
    v_amax_range: Optional[tuple] = None
    rel_extent: int = 0
    bias_std: float = 0.5
    window: int = 0
    plant_v: bool = False
    scales: tuple = (1.0, 1.0, 1.0)      # (q, k, v); None entries = calibrate


@dataclasses.dataclass
class PrefillSpec:
    name: str
    q_lens: Optional[List[int]]
    q_lo: int
    q_hi: int
    n_seqs: int
    Hq: int
    Hkv: int
    D: int
    block_size: int
    rel_extent: int = 0
    bias_std: float = 0.5
    windows: tuple = (0,)        # window of each group of sequences
    prefix: int = 0              # cached keys before each chunk (seq_len_k = q_len + prefix)
    scales: tuple = (1.0, 1.0, 1.0)


TINY_DECODE = DecodeSpec("decode_tiny_b1_h4x1_d128_ctx256", B=1, Hq=4, Hkv=1, D=128,
                         block_size=16, ctx_lo=256, ctx_hi=256)
DECODE_32K = DecodeSpec("decode_b64_h32x4_d128_ctx1k-32k_bias1024", B=64, Hq=32, Hkv=4,
                        D=128, block_size=16, ctx_lo=1024, ctx_hi=32768, v_dist="v_t3",
                        rel_extent=1024, plant_v=True)
PREFILL_16K = PrefillSpec("prefill_8seq_q512-4096_h32x4_d128_causal_sw512", q_lens=None,
                          q_lo=512, q_hi=4096, n_seqs=8, Hq=32, Hkv=4, D=128,
                          block_size=16, rel_extent=128, windows=(0, 512))
# one 4,096-query chunk over a 61,440-key cached prefix (65,536 keys in all):
# the pages' "chunked prefill 64K" kernel case
PREFILL_CHUNK_64K = PrefillSpec("prefill_chunk_q4096_k65536_h32x4_d128", q_lens=[4096], q_lo=4096,
                                q_hi=4096, n_seqs=1, Hq=32, Hkv=4, D=128, block_size=16,
                                rel_extent=128, windows=(0,), prefix=61440)
DECODE_128K_CAL = DecodeSpec("decode_b8_h24x4_d256_ctx128k_calibrated", B=8, Hq=24, Hkv=4,
                             D=256, block_size=16, ctx_lo=131072, ctx_hi=131072,
                             k_dist="n_amax", v_dist="t3_amax",
                             k_amax_range=(11.6, 23.1), v_amax_range=(14.9, 114.6),
                             scales=(None, None, None))
DECODE_1M = DecodeSpec("decode_b1_h32x4_d128_ctx1m", B=1, Hq=32, Hkv=4, D=128,
                       block_size=16, ctx_lo=1048576, ctx_hi=1048576)

WORKLOADS = {w.name: w for w in (TINY_DECODE, DECODE_32K, PREFILL_16K, PREFILL_CHUNK_64K,
                                 DECODE_128K_CAL, DECODE_1M)}


def make_decode(spec: DecodeSpec, *, device="cpu", seed: int = 0, lens=None,
                B: Optional[int] = None, max_blocks: Optional[int] = None):
    """Inputs of one decode step: the cache contents (every sequence's keys,
    including the step's own token, which is the last one) and the queries.
    lens / B override the drawn lengths for smaller parity cases."""
    g = _gen(device, seed)
    nb = spec.B if B is None else B
    if lens is None:
        if spec.ctx_lo == spec.ctx_hi:
            lens = [spec.ctx_lo] * nb
        else:
            lens = torch.randint(spec.ctx_lo, spec.ctx_hi + 1, (nb,), generator=g,
                                 device=device).tolist()
    k_amax = v_amax = None
    if spec.k_amax_range:
        lo, hi = spec.k_amax_range
        k_amax = lo + (hi - lo) * float(torch.rand((1,), generator=g, device=device).item())
    if spec.v_amax_range:
        lo, hi = spec.v_amax_range
        v_amax = lo + (hi - lo) * float(torch.rand((1,), generator=g, device=device).item())
    kv = make_paged_kv(list(lens), spec.Hkv, spec.D, spec.block_size, g=g, device=device,
                       k_dist=spec.k_dist, v_dist=spec.v_dist, k_amax=k_amax, v_amax=v_amax,
                       plant_v=spec.plant_v, max_blocks=max_blocks)
    q = draw_values((nb, spec.Hq, spec.D), "normal", g, device)
    rel = None
    if spec.rel_extent:
        rel = (spec.bias_std * _normal((nb, spec.Hq, spec.rel_extent), g, device)).to(torch.bfloat16)
    return dict(kv=kv, q=q, rel=rel, lens=list(lens), k_amax=k_amax, v_amax=v_amax)


def make_prefill(spec: PrefillSpec, *, device="cpu", seed: int = 0, q_lens=None,
                 k_lens=None):
    """Inputs of one varlen prefill chunk: K/V of every sequence (k_lens tokens,
    the chunk's queries being the last q_len of them), queries [Tq][Hq][D],
    cu_seqlens_q, and a per-query-token bias [Tq][Hq][E]."""
    g = _gen(device, seed)
    if q_lens is None:
        q_lens = spec.q_lens or torch.randint(spec.q_lo, spec.q_hi + 1, (spec.n_seqs,),
                                              generator=g, device=device).tolist()
    q_lens = [int(x) for x in q_lens]
    if k_lens is None:
        k_lens = [L + spec.prefix for L in q_lens]
    kv = make_paged_kv(list(k_lens), spec.Hkv, spec.D, spec.block_size, g=g, device=device)
    Tq = sum(q_lens)
    q = draw_values((Tq, spec.Hq, spec.D), "normal", g, device)
    cu = [0]
    for L in q_lens:
        cu.append(cu[-1] + L)
    rel = None
    if spec.rel_extent:
        rel = (spec.bias_std * _normal((Tq, spec.Hq, spec.rel_extent), g, device)).to(torch.bfloat16)
    return dict(kv=kv, q=q, rel=rel, q_lens=q_lens, k_lens=list(k_lens),
                cu_seqlens_q=torch.tensor(cu, dtype=torch.int32, device=device))


def bf16_bits(t: torch.Tensor):
    """Raw uint16 bit patterns of a bf16 tensor, as a host numpy array."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


__all__ = ["PagedKV", "DecodeSpec", "PrefillSpec", "TINY_DECODE", "DECODE_32K", "PREFILL_16K",
           "PREFILL_CHUNK_64K",
           "DECODE_128K_CAL", "DECODE_1M", "WORKLOADS", "make_decode", "make_prefill",
           "make_paged_kv", "draw_values", "bf16_bits", "ceil_div"]
