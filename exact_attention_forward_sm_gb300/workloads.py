"""Seeded synthetic inputs for the attention forward pass.

This module only draws inputs; it holds none of the attention arithmetic.  The
CUDA path's tests, the benchmark and the CPU oracle's tests all take their
inputs from here, so every side sees the same 16-bit values.

Recipe (all draws on the CPU, ``torch.Generator().manual_seed(seed)``):

* packed variable-length workloads first draw their sequence lengths, then
  Q, K, V;
* Q, K, V are drawn in fp32 as N(0, sigma^2) and cast (round to nearest) to the
  16-bit dtype; the oracle reads those same rounded values;
* the rising-bias workload reserves channel D-1 of Q and K to carry a per-key
  bias b(j) in log2 units: q[..., D-1] = 1 and k[j, ..., D-1] =
  b(j) * ln2 / scale, so scale * <q_i, k_j> gains exactly b(j) * ln2 (natural
  units), i.e. b(j) log2 units.  b is constant within a 128-key block and grows
  by 0.5 * (blk mod 25) log2 units at block blk >= 1, so successive block maxima
  rise by 0 .. 12 log2 units and both skipped and performed lazy rescales occur
  when the keys are walked in ascending order.

Score variants (local window, soft cap, ALiBi) are carried on the case as plain
parameters; ALiBi slopes follow the geometric sequence 2^(-8 (h + 1) / H) of
the ALiBi paper (for H a power of two), one per query head.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}
DTYPE_CODE = {"fp16": 0, "bf16": 1}


@dataclass(frozen=True)
class Workload:
    """One attention forward problem, described by its sizes and draw recipe."""
    name: str
    B: int
    Hq: int
    Hkv: int
    S: int                 # Sq = Sk for dense problems; unused for packed ones
    D: int
    dtype: str
    causal: bool
    sigma: float = 1.0
    rising_bias: bool = False
    varlen_count: int = 0  # >0: packed problem with this many sequences
    varlen_min: int = 0
    varlen_max: int = 0
    seed: int = 0
    window: tuple = (-1, -1)   # local window (left, right), -1 = unbounded
    softcap: float = 0.0
    alibi: bool = False        # geometric ALiBi slopes, one per query head
    Sk: int = 0                # dense keys per sequence when != S (0: Sk = S)
    splits: int = -1           # split-KV chunks: -1 unsplit path, 0 chosen, >= 1 forced


# The five workloads the method is validated and measured on.  Seeds are
# 1000 + index.  ``attention fwd`` throughput is quoted on the second one.
WORKLOADS = [
    Workload("b1_h2_s128_d64_fp16_noncausal", 1, 2, 2, 128, 64, "fp16", False,
             seed=1000),
    Workload("b4_h16_s2048_d128_bf16_causal", 4, 16, 16, 2048, 128, "bf16", True,
             seed=1001),
    Workload("b2_hq32_hkv8_s4096_d128_bf16_causal_risingbias", 2, 32, 8, 4096, 128,
             "bf16", True, rising_bias=True, seed=1002),
    Workload("varlen16_l64to8192_h16_d64_fp16_causal", 16, 16, 16, 0, 64, "fp16",
             True, varlen_count=16, varlen_min=64, varlen_max=8192, seed=1003),
    Workload("b1_h8_s32768_d128_bf16_noncausal_sigma2", 1, 8, 8, 32768, 128, "bf16",
             False, sigma=math.sqrt(2.0), seed=1004),
]
# Score-variant workloads (local window, soft cap, ALiBi): the shapes of the
# causal benchmark problem and a long sliding-window problem.  They are not
# part of the five validation workloads; seeds are 1100 + index.
VARIANT_WORKLOADS = [
    Workload("b4_h16_s2048_d128_bf16_causal_softcap30", 4, 16, 16, 2048, 128, "bf16", True,
             seed=1100, softcap=30.0),
    Workload("b4_h16_s2048_d128_bf16_causal_alibi", 4, 16, 16, 2048, 128, "bf16", True,
             seed=1101, alibi=True),
    Workload("b2_h16_s16384_d128_bf16_causal_window1024", 2, 16, 16, 16384, 128, "bf16",
             True, seed=1102, window=(1024, 0)),
    Workload("b4_h16_s2048_d128_bf16_window32_32", 4, 16, 16, 2048, 128, "bf16", False,
             seed=1103, window=(32, 32)),
]
# Split-KV workloads: too few query tiles to fill the GPU, many K/V tiles each
# (a prefill chunk at the end of a long context; one query row per sequence and
# head, as in decoding).  Seeds 1200 + index; the split count is chosen by the
# library.
SPLIT_WORKLOADS = [
    Workload("b1_h32_sq512_sk16384_d128_bf16_causal_chunk", 1, 32, 32, 512, 128, "bf16",
             True, seed=1200, Sk=16384, splits=0),
    Workload("b8_h8_sq1_sk8192_d128_bf16_decode", 8, 8, 8, 1, 128, "bf16", True,
             seed=1201, Sk=8192, splits=0),
]
# Head dim 256 (the fork's v1.7 notes validate D = 256 in section 4.3).  Seeds
# 1400 + index.
D256_WORKLOADS = [
    Workload("b2_h16_s4096_d256_bf16_causal", 2, 16, 16, 4096, 256, "bf16", True, seed=1400),
    Workload("b1_h8_s16384_d256_bf16_noncausal", 1, 8, 8, 16384, 256, "bf16", False,
             seed=1401),
]
BY_NAME = {w.name: w for w in WORKLOADS + VARIANT_WORKLOADS + SPLIT_WORKLOADS + D256_WORKLOADS}


@dataclass
class Case:
    """Drawn inputs plus the C-ABI size arguments that describe them."""
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    B: int
    Hq: int
    Hkv: int
    Sq: int              # dense: rows per sequence; packed: total_q
    Sk: int              # dense: keys per sequence; packed: total_k
    D: int
    scale: float
    causal: bool
    dtype: str
    cu_seqlens_q: Optional[torch.Tensor] = None   # int32 [B + 1] (CPU)
    cu_seqlens_k: Optional[torch.Tensor] = None
    meta: dict = field(default_factory=dict)
    window_left: int = -1                         # -1: unbounded
    window_right: int = -1
    softcap: float = 0.0                          # 0: off
    alibi_slopes: Optional[torch.Tensor] = None   # fp32 [Hq] (CPU) or None

    @property
    def has_variants(self) -> bool:
        return (self.window_left >= 0 or self.window_right >= 0 or self.softcap > 0
                or self.alibi_slopes is not None)

    @property
    def varlen(self) -> bool:
        return self.cu_seqlens_q is not None

    def seq_lengths(self):
        """(Lq, Lk) per sequence."""
        if not self.varlen:
            return [(self.Sq, self.Sk)] * self.B
        cq = self.cu_seqlens_q.tolist()
        ck = self.cu_seqlens_k.tolist()
        return [(cq[b + 1] - cq[b], ck[b + 1] - ck[b]) for b in range(self.B)]

    def lse_rows(self) -> int:
        """Number of query rows (= LSE entries)."""
        return self.Hq * (self.Sq if self.varlen else self.B * self.Sq)


def rising_bias_log2(n_keys: int, block: int = 128, period: int = 25,
                     step: float = 0.5) -> torch.Tensor:
    """Per-key bias b(j) in log2 units (constant within each key block)."""
    nblk = (n_keys + block - 1) // block
    rise = torch.tensor([0.0] + [step * (i % period) for i in range(1, nblk)],
                        dtype=torch.float64)
    per_block = torch.cumsum(rise, 0)
    return per_block.repeat_interleave(block)[:n_keys]


def alibi_slopes_geometric(H: int) -> torch.Tensor:
    """ALiBi slopes 2^(-8 (h + 1) / H), h = 0 .. H-1 (fp32)."""
    return torch.tensor([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)], dtype=torch.float32)


def _draw(shape, sigma, dtype, g):
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if sigma != 1.0:
        x = x * sigma
    return x.to(DTYPES[dtype])


def make_case(B, Hq, Hkv, Sq, Sk, D, dtype="bf16", causal=False, seed=0,
              sigma=1.0, rising_bias=False, seqlens_q=None, seqlens_k=None,
              scale=None, zero_q=False, window=(-1, -1), softcap=0.0,
              alibi_slopes=None) -> Case:
    """Draw one problem.

    Dense when ``seqlens_q`` is None (q [B, Sq, Hq, D], k/v [B, Sk, Hkv, D]);
    packed otherwise (q [sum Lq, Hq, D], k/v [sum Lk, Hkv, D], B = number of
    sequences, Sq / Sk = the packed totals).
    """
    g = torch.Generator().manual_seed(int(seed))
    scale = (1.0 / math.sqrt(D)) if scale is None else float(scale)
    cu_q = cu_k = None
    if seqlens_q is not None:
        seqlens_k = seqlens_q if seqlens_k is None else seqlens_k
        lq = [int(x) for x in seqlens_q]
        lk = [int(x) for x in seqlens_k]
        B = len(lq)
        cu_q = torch.tensor([0] + lq, dtype=torch.int64).cumsum(0).to(torch.int32)
        cu_k = torch.tensor([0] + lk, dtype=torch.int64).cumsum(0).to(torch.int32)
        Sq, Sk = int(cu_q[-1]), int(cu_k[-1])
        q_shape, kv_shape = (Sq, Hq, D), (Sk, Hkv, D)
    else:
        q_shape, kv_shape = (B, Sq, Hq, D), (B, Sk, Hkv, D)
    q = _draw(q_shape, sigma, dtype, g)
    k = _draw(kv_shape, sigma, dtype, g)
    v = _draw(kv_shape, sigma, dtype, g)
    if zero_q:
        q.zero_()
    if rising_bias:
        # channel D-1 carries b(j) log2 units: scale * q . k gains b(j) * ln2
        q[..., D - 1] = 1.0
        if cu_k is None:
            bias = rising_bias_log2(Sk) * math.log(2.0) / scale
            k[..., D - 1] = bias.view(1, Sk, 1).to(k.dtype)
        else:
            for b in range(B):
                s0, s1 = int(cu_k[b]), int(cu_k[b + 1])
                bias = rising_bias_log2(s1 - s0) * math.log(2.0) / scale
                k[s0:s1, :, D - 1] = bias.view(-1, 1).to(k.dtype)
    if alibi_slopes is not None:
        alibi_slopes = torch.as_tensor(alibi_slopes, dtype=torch.float32).reshape(Hq)
    return Case(q, k, v, B, Hq, Hkv, Sq, Sk, D, scale, bool(causal), dtype, cu_q, cu_k,
                window_left=int(window[0]), window_right=int(window[1]),
                softcap=float(softcap), alibi_slopes=alibi_slopes)


def _variants(w: Workload) -> dict:
    return {"window": tuple(w.window), "softcap": w.softcap,
            "alibi_slopes": alibi_slopes_geometric(w.Hq) if w.alibi else None}


def make_workload(w: Workload) -> Case:
    """Draw the inputs of one named workload."""
    if w.varlen_count:
        g = torch.Generator().manual_seed(int(w.seed))
        lens = torch.randint(w.varlen_min, w.varlen_max + 1, (w.varlen_count,),
                             generator=g).tolist()
        case = make_case(w.varlen_count, w.Hq, w.Hkv, 0, 0, w.D, w.dtype, w.causal,
                         seed=w.seed + 7919, sigma=w.sigma,
                         rising_bias=w.rising_bias, seqlens_q=lens, **_variants(w))
    else:
        case = make_case(w.B, w.Hq, w.Hkv, w.S, w.Sk or w.S, w.D, w.dtype, w.causal,
                         seed=w.seed, sigma=w.sigma, rising_bias=w.rising_bias,
                         **_variants(w))
    case.meta["workload"] = w.name
    return case


def visible_pairs(case: Case) -> int:
    """Number of (query, key) pairs the mask leaves visible, summed over the
    sequences of one head (bottom-right aligned causal mask and local window)."""
    total = 0
    for lq, lk in case.seq_lengths():
        if not case.causal and case.window_left < 0 and case.window_right < 0:
            total += lq * lk
            continue
        diag = torch.arange(lq, dtype=torch.int64) + (lk - lq)
        hi = torch.full_like(diag, lk - 1)
        if case.causal:
            hi = torch.minimum(hi, diag)
        if case.window_right >= 0:
            hi = torch.minimum(hi, diag + case.window_right)
        lo = torch.zeros_like(diag)
        if case.window_left >= 0:
            lo = torch.maximum(lo, diag - case.window_left)
        total += int((hi - lo + 1).clamp(min=0).sum())
    return total


def attention_flops(case: Case) -> int:
    """FLOPs of the two contractions (QK^T and PV): 4 * D * Hq * visible pairs."""
    pairs = visible_pairs(case)
    return 4 * case.D * case.Hq * pairs


def algorithmic_bytes(case: Case) -> int:
    """Q, K, V read once plus O written (16-bit) and LSE written (fp32)."""
    el = 2
    return (case.q.numel() + case.k.numel() + case.v.numel() + case.q.numel()) * el \
        + case.lse_rows() * 4


# ----------------------------------------------------------------- KV caches

@dataclass(frozen=True)
class CacheWorkload:
    """Decoding over a KV cache: Sq new tokens per sequence against a cache of
    cache_seqlens[b] keys, drawn uniformly in [min_len, capacity] (all equal to
    capacity when min_len is 0); paged with page_rows rows per page (pages in a
    random order) or contiguous (page_rows 0)."""
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    D: int
    dtype: str
    causal: bool
    capacity: int
    page_rows: int = 0
    min_len: int = 0
    seed: int = 0
    splits: int = 0        # split-KV chunks: 0 = chosen by the library


@dataclass
class KVCase:
    """Drawn decoding problem: q [B, Sq, Hq, D]; cache [pages, page_rows, Hkv, D]
    (contiguous: pages = B, page_rows = capacity); int32 seqlens / block table (CPU)."""
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    cache_seqlens: torch.Tensor
    block_table: Optional[torch.Tensor]
    B: int
    Hq: int
    Hkv: int
    Sq: int
    D: int
    scale: float
    causal: bool
    dtype: str
    page_rows: int
    num_pages: int
    max_blocks: int
    meta: dict = field(default_factory=dict)

    def lse_rows(self) -> int:
        return self.B * self.Hq * self.Sq


CACHE_WORKLOADS = [
    CacheWorkload("decode_b64_hq32_hkv8_sq1_d128_bf16_paged256_len2k4k", 64, 32, 8, 1, 128,
                  "bf16", True, capacity=4096, page_rows=256, min_len=2048, seed=1300),
    CacheWorkload("decode_b8_hq64_hkv8_sq1_d128_bf16_len16k", 8, 64, 8, 1, 128, "bf16", True,
                  capacity=16384, seed=1301),
    CacheWorkload("decode_b32_hq32_hkv8_sq4_d128_bf16_paged256_len4k", 32, 32, 8, 4, 128,
                  "bf16", True, capacity=4096, page_rows=256, seed=1302),
]
CACHE_BY_NAME = {w.name: w for w in CACHE_WORKLOADS}


def make_cache_workload(w: CacheWorkload, seed=None) -> KVCase:
    """Draw the lengths, then q, then the cache pages, then the page order."""
    g = torch.Generator().manual_seed(int(w.seed if seed is None else seed))
    if w.min_len:
        lens = torch.randint(w.min_len, w.capacity + 1, (w.B,), generator=g)
    else:
        lens = torch.full((w.B,), w.capacity, dtype=torch.int64)
    q = _draw((w.B, w.Sq, w.Hq, w.D), 1.0, w.dtype, g)
    if w.page_rows:
        max_blocks = (w.capacity + w.page_rows - 1) // w.page_rows
        pages = w.B * max_blocks
        shape = (pages, w.page_rows, w.Hkv, w.D)
    else:
        max_blocks, pages = 1, w.B
        shape = (w.B, w.capacity, w.Hkv, w.D)
    kc = _draw(shape, 1.0, w.dtype, g)
    vc = _draw(shape, 1.0, w.dtype, g)
    table = None
    if w.page_rows:
        table = torch.randperm(pages, generator=g).reshape(w.B, max_blocks).to(torch.int32)
    case = KVCase(q, kc, vc, lens.to(torch.int32), table, w.B, w.Hq, w.Hkv, w.Sq, w.D,
                  1.0 / math.sqrt(w.D), w.causal, w.dtype, w.page_rows or w.capacity, pages,
                  max_blocks)
    case.meta["workload"] = w.name
    return case


def kv_visible_per_row(c: KVCase):
    """Visible keys of every row in [B, Hq, Sq] order (bottom-right causal)."""
    out = []
    for lk in c.cache_seqlens.tolist():
        i = torch.arange(c.Sq, dtype=torch.int64)
        n = (i + lk - c.Sq + 1).clamp(min=0, max=lk) if c.causal else torch.full_like(i, lk)
        out.append(n.repeat(c.Hq))
    return torch.cat(out)


def kv_flops(c: KVCase) -> int:
    """4 * D * (visible (query row, key) pairs over all query heads)."""
    return 4 * c.D * int(kv_visible_per_row(c).sum())


def kv_algorithmic_bytes(c: KVCase) -> int:
    """q and o (16-bit), LSE (fp32), and every cache row some query token of its
    sequence sees, K and V, once per K/V head."""
    rows = sum(c.cache_seqlens.tolist())  # the newest token sees every key, causal or not
    return 2 * 2 * c.q.numel() + 4 * c.lse_rows() + 2 * 2 * rows * c.Hkv * c.D
