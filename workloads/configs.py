"""Synthetic workloads of the flash-attention forward pages, and their seeded inputs.

Each workload is named by what it is, with its sizes.  Inputs are i.i.d. N(0, 1)
rounded to bf16 (see ``workloads.rng``), drawn from one counter-based stream per
tensor, so the oracle side can regenerate any row or head by itself:

* prefill Q element (b, h, i, x)  -> counter ((b*hq + h)*sq + i)*d + x  of stream "q"
* prefill K/V element (b, g, j, x) -> counter ((b*hkv + g)*skv + j)*d + x of stream "k"/"v"
* the long-context workload multiplies each Q element by 8 when the uniform draw of
  stream "q_outlier" at the same counter is below 0.01 (exact in bf16).
* decode: cache_len[b] = lo + floor(u_b * (hi - lo + 1)) (stream "cache_len"); cached
  K/V at logical position j < cache_len - s_active come from stream "k_cache"/"v_cache"
  at counter ((b*hkv + g)*hi + j)*d + x; the s_active appended tokens come from
  "k_new"/"v_new" at ((b*hkv + g)*s_active + t)*d + x; query element (b, h, t, x)
  from "q" at ((b*hq + h)*s_active + t)*d + x.  Logical page p of sequence b holds
  tokens [page*p, page*p + page); physical pages are the stable argsort of stream
  "page_perm" over all pages in use; slots past cache_len in a last page are NaN.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

from . import rng


@dataclass(frozen=True)
class PrefillWorkload:
    name: str
    b: int
    hq: int
    hkv: int
    sq: int
    skv: int
    d: int
    causal: bool
    window: int = 0
    o_dtype: str = "bf16"  # "bf16" or "f32"
    outlier_frac: float = 0.0
    seed: int = 0xA77E0000

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def q_pos(self, i):
        """Position of query row i: queries sit at the tail of the keys (bottom-right)."""
        return i + (self.skv - self.sq)

    def allowed_pairs_per_head(self) -> int:
        """Exact number of (query, key) pairs the mask allows, for one head."""
        i = np.arange(self.sq, dtype=np.int64)
        qp = self.q_pos(i)
        hi = np.minimum(self.skv - 1, qp) if self.causal else np.full_like(qp, self.skv - 1)
        lo = np.maximum(0, qp - self.window + 1) if self.window > 0 else np.zeros_like(qp)
        return int(np.clip(hi - lo + 1, 0, None).sum())

    def flops(self) -> float:
        """Causal/window-adjusted FLOPs: 4*d per allowed pair (two matmuls, multiply+add)."""
        return 4.0 * self.d * self.allowed_pairs_per_head() * self.b * self.hq

    def io_bytes(self) -> int:
        """Algorithmic HBM bytes: Q, K, V read once, O and LSE written once."""
        ob = 2 if self.o_dtype == "bf16" else 4
        q = self.b * self.hq * self.sq * self.d * 2
        kv = 2 * self.b * self.hkv * self.skv * self.d * 2
        o = self.b * self.hq * self.sq * self.d * ob
        lse = self.b * self.hq * self.sq * 4
        return q + kv + o + lse

    def with_(self, **kw) -> "PrefillWorkload":
        f = dict(self.__dict__)
        f.update(kw)
        return PrefillWorkload(**f)


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    b: int
    hq: int
    hkv: int
    d: int
    s_active: int
    page_size: int = 32
    len_lo: int = 1024
    len_hi: int = 32768
    paged: bool = True
    o_dtype: str = "bf16"
    seed: int = 0xA77E0004
    fixed_lens: tuple = field(default=())

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def max_pages_per_seq(self) -> int:
        return -(-self.len_hi // self.page_size)

    def with_(self, **kw) -> "DecodeWorkload":
        f = dict(self.__dict__)
        f.update(kw)
        return DecodeWorkload(**f)


# The five workloads of the pages' problem statement, at full size.
TINY_PREFILL = PrefillWorkload("tiny_prefill_b1_h1_s128_d64", 1, 1, 1, 128, 128, 64,
                               causal=False, o_dtype="f32", seed=0xA77E0000)
CAUSAL_PREFILL_2K = PrefillWorkload("causal_prefill_b1_h32_s2048_d128", 1, 32, 32, 2048, 2048,
                                    128, causal=True, seed=0xA77E0001)
GQA_PREFILL_32K = PrefillWorkload("gqa_causal_prefill_b1_h32kv8_s32768_d128_outliers", 1, 32, 8,
                                  32768, 32768, 128, causal=True, outlier_frac=0.01,
                                  seed=0xA77E0002)
SWA_PREFILL_8K = PrefillWorkload("swa_prefill_b2_h32kv16_s8192_d256_w1024", 2, 32, 16, 8192,
                                 8192, 256, causal=True, window=1024, seed=0xA77E0003)
PAGED_DECODE = DecodeWorkload("paged_decode_b64_h32kv8_d128_sa1", 64, 32, 8, 128, 1,
                              seed=0xA77E0004)
PAGED_DECODE_SPEC4 = DecodeWorkload("paged_decode_b64_h32kv8_d128_sa4", 64, 32, 8, 128, 4,
                                    seed=0xA77E0005)

ALL_PREFILL = (TINY_PREFILL, CAUSAL_PREFILL_2K, GQA_PREFILL_32K, SWA_PREFILL_8K)
ALL_DECODE = (PAGED_DECODE, PAGED_DECODE_SPEC4)

# Reduced variants of the same kernels, sized for profiler captures (a few hundred MB).
GQA_PREFILL_8K = GQA_PREFILL_32K.with_(name="gqa_causal_prefill_b1_h32kv8_s8192_d128_outliers",
                                       sq=8192, skv=8192)
SWA_PREFILL_8K_B1 = SWA_PREFILL_8K.with_(name="swa_prefill_b1_h32kv16_s8192_d256_w1024", b=1)
PAGED_DECODE_B16 = PAGED_DECODE.with_(name="paged_decode_b16_h32kv8_d128_sa1", b=16)
PAGED_DECODE_SPEC4_B16 = PAGED_DECODE_SPEC4.with_(name="paged_decode_b16_h32kv8_d128_sa4", b=16)

# head_dim 256 decode (the pages' head_dim bound), 32 sequences of the same length mix.
PAGED_DECODE_D256 = DecodeWorkload("paged_decode_b32_h32kv8_d256_sa1", 32, 32, 8, 256, 1,
                                   seed=0xA77E0006)

PAGED_DECODE_D256_B8 = PAGED_DECODE_D256.with_(name="paged_decode_b8_h32kv8_d256_sa1", b=8)

REGISTRY = {w.name: w for w in ALL_PREFILL + ALL_DECODE + (
    GQA_PREFILL_8K, SWA_PREFILL_8K_B1, PAGED_DECODE_B16, PAGED_DECODE_SPEC4_B16,
    PAGED_DECODE_D256, PAGED_DECODE_D256_B8)}


# =========================================================================== prefill
def _prefill_q_counter(w: PrefillWorkload, b: int, h: int, i0: int) -> int:
    return ((b * w.hq + h) * w.sq + i0) * w.d


def _prefill_kv_counter(w: PrefillWorkload, b: int, g: int, j0: int) -> int:
    return ((b * w.hkv + g) * w.skv + j0) * w.d


def _apply_outliers_np(w: PrefillWorkload, bits: np.ndarray, start: int) -> np.ndarray:
    if w.outlier_frac <= 0:
        return bits
    u = rng.uniform_np(rng.stream_seed(w.seed, "q_outlier"), start, bits.size)
    x = rng.bf16_bits_to_f32_np(bits.reshape(-1)).copy()
    x[u < w.outlier_frac] *= 8.0
    return rng.f32_to_bf16_bits_np(x).reshape(bits.shape)


def prefill_q_rows_np(w: PrefillWorkload, b: int, h: int, i0: int, n: int) -> np.ndarray:
    """Q rows [i0, i0+n) of head (b, h) as bf16 bits, shape [n, d]."""
    start = _prefill_q_counter(w, b, h, i0)
    bits = rng.normal_bf16_np(rng.stream_seed(w.seed, "q"), start, n * w.d)
    return _apply_outliers_np(w, bits, start).reshape(n, w.d)


def prefill_kv_head_np(w: PrefillWorkload, which: str, b: int, g: int) -> np.ndarray:
    """Whole K (which='k') or V ('v') of kv head (b, g) as bf16 bits, shape [skv, d]."""
    start = _prefill_kv_counter(w, b, g, 0)
    return rng.normal_bf16_np(rng.stream_seed(w.seed, which), start, w.skv * w.d).reshape(w.skv, w.d)


def prefill_inputs_np(w: PrefillWorkload):
    """Full Q, K, V as bf16 bits ([b,hq,sq,d], [b,hkv,skv,d] x2). For small workloads."""
    q = np.stack([np.stack([prefill_q_rows_np(w, b, h, 0, w.sq) for h in range(w.hq)])
                  for b in range(w.b)])
    k = np.stack([np.stack([prefill_kv_head_np(w, "k", b, g) for g in range(w.hkv)])
                  for b in range(w.b)])
    v = np.stack([np.stack([prefill_kv_head_np(w, "v", b, g) for g in range(w.hkv)])
                  for b in range(w.b)])
    return q, k, v


def prefill_inputs_torch(w: PrefillWorkload, device):
    """Full Q, K, V as bf16 torch tensors on ``device`` (same values as the numpy side)."""
    import torch

    nq = w.b * w.hq * w.sq * w.d
    q = rng.normal_bf16_torch(rng.stream_seed(w.seed, "q"), 0, nq, device)
    if w.outlier_frac > 0:
        u = rng.uniform_torch(rng.stream_seed(w.seed, "q_outlier"), 0, nq, device)
        qf = q.float()
        qf = torch.where(u < w.outlier_frac, qf * 8.0, qf)
        q = qf.to(torch.bfloat16)  # exact: a power-of-two multiple of a bf16 value
        del u, qf
    nkv = w.b * w.hkv * w.skv * w.d
    k = rng.normal_bf16_torch(rng.stream_seed(w.seed, "k"), 0, nkv, device)
    v = rng.normal_bf16_torch(rng.stream_seed(w.seed, "v"), 0, nkv, device)
    return (q.view(w.b, w.hq, w.sq, w.d), k.view(w.b, w.hkv, w.skv, w.d),
            v.view(w.b, w.hkv, w.skv, w.d))


# =========================================================================== decode
def decode_cache_lens(w: DecodeWorkload) -> np.ndarray:
    if w.fixed_lens:
        lens = np.asarray(w.fixed_lens, dtype=np.int64)
        assert lens.shape == (w.b,)
    else:
        u = rng.uniform_np(rng.stream_seed(w.seed, "cache_len"), 0, w.b)
        lens = w.len_lo + np.floor(u * (w.len_hi - w.len_lo + 1)).astype(np.int64)
    assert lens.min() >= w.s_active and lens.max() <= w.len_hi
    return lens.astype(np.int32)


def decode_block_table(w: DecodeWorkload, lens: np.ndarray, permute: bool = True):
    """uint32 [b, max_pages_per_seq] page table (unused entries 0xFFFFFFFF) and page count."""
    npages = -(-lens.astype(np.int64) // w.page_size)
    total = int(npages.sum())
    if permute:
        keys = rng.u64_np(rng.stream_seed(w.seed, "page_perm"), 0, total)
        phys = np.argsort(keys, kind="stable").astype(np.uint32)
    else:
        phys = np.arange(total, dtype=np.uint32)
    table = np.full((w.b, w.max_pages_per_seq), 0xFFFFFFFF, dtype=np.uint32)
    off = 0
    for b in range(w.b):
        table[b, : npages[b]] = phys[off: off + npages[b]]
        off += npages[b]
    return table, total


def decode_q_np(w: DecodeWorkload, b: int, h: int) -> np.ndarray:
    start = ((b * w.hq + h) * w.s_active) * w.d
    return rng.normal_bf16_np(rng.stream_seed(w.seed, "q"), start, w.s_active * w.d).reshape(
        w.s_active, w.d)


def decode_kv_logical_np(w: DecodeWorkload, which: str, b: int, g: int, length: int) -> np.ndarray:
    """Logical K ('k') or V ('v') rows [0, length) of (b, kv head g), bf16 bits [length, d]."""
    prior = length - w.s_active
    out = np.empty((length, w.d), dtype=np.uint16)
    if prior > 0:
        start = ((b * w.hkv + g) * w.len_hi) * w.d
        out[:prior] = rng.normal_bf16_np(rng.stream_seed(w.seed, which + "_cache"), start,
                                         prior * w.d).reshape(prior, w.d)
    start = ((b * w.hkv + g) * w.s_active) * w.d
    out[prior:] = rng.normal_bf16_np(rng.stream_seed(w.seed, which + "_new"), start,
                                     w.s_active * w.d).reshape(w.s_active, w.d)
    return out


def _decode_kv_logical_torch(w: DecodeWorkload, which: str, b: int, length: int, device):
    """Logical [hkv, length, d] bf16 for sequence b (cached part, then the appended tokens)."""
    import torch

    prior = length - w.s_active
    parts = []
    for g in range(w.hkv):
        rows = []
        if prior > 0:
            start = ((b * w.hkv + g) * w.len_hi) * w.d
            rows.append(rng.normal_bf16_torch(rng.stream_seed(w.seed, which + "_cache"), start,
                                              prior * w.d, device).view(prior, w.d))
        start = ((b * w.hkv + g) * w.s_active) * w.d
        rows.append(rng.normal_bf16_torch(rng.stream_seed(w.seed, which + "_new"), start,
                                          w.s_active * w.d, device).view(w.s_active, w.d))
        parts.append(torch.cat(rows, 0))
    return torch.stack(parts, 0)


def decode_inputs_torch(w: DecodeWorkload, device, permute: bool = True):
    """Device tensors for one decode call.

    Returns dict(q [b,hq,s_active,d] bf16, k_cache, v_cache, block_table (int32 view of
    the uint32 table, or None for a flat cache), cache_len int32 [b], lens (numpy),
    table (numpy uint32 or None), num_pages, max_cache_len).
    Paged cache: [num_pages, hkv, page, d]; flat cache: [b, hkv, len_hi, d].
    """
    import torch

    lens = decode_cache_lens(w)
    nq = w.b * w.hq * w.s_active * w.d
    q = rng.normal_bf16_torch(rng.stream_seed(w.seed, "q"), 0, nq, device).view(
        w.b, w.hq, w.s_active, w.d)
    nan = torch.tensor(rng.BF16_NAN_BITS, dtype=torch.int16).view(torch.bfloat16).item()
    out = dict(q=q, lens=lens, cache_len=torch.from_numpy(lens).to(device))
    if w.paged:
        table, total = decode_block_table(w, lens, permute)
        caches = {}
        for which in ("k", "v"):
            cache = torch.empty((total, w.hkv, w.page_size, w.d), dtype=torch.bfloat16,
                                device=device)
            for b in range(w.b):
                n = int(lens[b])
                npg = -(-n // w.page_size)
                logical = torch.full((w.hkv, npg * w.page_size, w.d), nan, dtype=torch.bfloat16,
                                     device=device)
                logical[:, :n] = _decode_kv_logical_torch(w, which, b, n, device)
                pages = logical.view(w.hkv, npg, w.page_size, w.d).permute(1, 0, 2, 3)
                idx = torch.from_numpy(table[b, :npg].astype(np.int64)).to(device)
                cache[idx] = pages
            caches[which] = cache
        out.update(k_cache=caches["k"], v_cache=caches["v"], table=table, num_pages=total,
                   block_table=torch.from_numpy(table.view(np.int32)).to(device),
                   max_cache_len=w.max_pages_per_seq * w.page_size)
    else:
        caches = {}
        for which in ("k", "v"):
            cache = torch.full((w.b, w.hkv, w.len_hi, w.d), nan, dtype=torch.bfloat16,
                               device=device)
            for b in range(w.b):
                n = int(lens[b])
                cache[b, :, :n] = _decode_kv_logical_torch(w, which, b, n, device)
            caches[which] = cache
        out.update(k_cache=caches["k"], v_cache=caches["v"], table=None, num_pages=0,
                   block_table=None, max_cache_len=w.len_hi)
    return out


# Packed prefill: nseq sequences along the sequence axis of one batch, seeded query
# lengths in [q_lo, q_hi] and cached-prefix lengths in [0, prefix_hi] (more keys than
# queries), each sequence causal inside itself.
@dataclass(frozen=True)
class PackedPrefillWorkload:
    name: str
    hq: int
    hkv: int
    d: int
    nseq: int
    q_lo: int
    q_hi: int
    prefix_hi: int
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def offsets(self):
        """(cu_q, cu_k) int32 [nseq + 1]."""
        u = rng.u64_np(self.seed, 0, 2 * self.nseq)
        nq = self.q_lo + (u[: self.nseq] % np.uint64(self.q_hi - self.q_lo + 1)).astype(np.int64)
        pre = (u[self.nseq:] % np.uint64(self.prefix_hi + 1)).astype(np.int64)
        cu_q = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
        cu_k = np.concatenate([[0], np.cumsum(nq + pre)]).astype(np.int32)
        return cu_q, cu_k

    def flops(self) -> float:
        """4 d per allowed (query, key) pair: query i of a sequence with nq queries after
        a prefix of p keys sees p + i + 1 keys."""
        cu_q, cu_k = self.offsets()
        nq = np.diff(cu_q).astype(np.float64)
        pre = np.diff(cu_k).astype(np.float64) - nq
        pairs = (nq * pre + nq * (nq + 1) / 2).sum()
        return 4.0 * self.d * self.hq * pairs

    def io_bytes(self) -> int:
        cu_q, cu_k = self.offsets()
        sq, skv = int(cu_q[-1]), int(cu_k[-1])
        return 2 * self.hq * sq * self.d * 2 + 2 * self.hkv * skv * self.d * 2 + self.hq * sq * 4

    def as_prefill(self) -> "PrefillWorkload":
        """The b = 1 problem the sequences are packed into (for its input tensors)."""
        cu_q, cu_k = self.offsets()
        return PrefillWorkload(self.name, 1, self.hq, self.hkv, int(cu_q[-1]), int(cu_k[-1]),
                               self.d, True, 0, seed=self.seed)


PACKED_PREFILL = PackedPrefillWorkload("packed_prefill_h32kv8_d128_16seqs", 32, 8, 128, 16, 256,
                                       4096, 1024, seed=0x9ACC)
REGISTRY[PACKED_PREFILL.name] = PACKED_PREFILL


# Attention-sink logits, one per query head (scaled-score units): a fixed cycle of a
# neutral, moderate, dominant (e^9 and e^60 outweigh every key of an N(0,1) row),
# negligible and absent (-inf) sink, so every regime of the sink is present in a run.
SINK_CYCLE = (0.0, 2.5, -1.75, 9.0, -40.0, float("-inf"), 0.75, 60.0)


def sink_logits(hq: int) -> np.ndarray:
    """fp32 [hq] sink logits of the query heads."""
    return np.array([SINK_CYCLE[h % len(SINK_CYCLE)] for h in range(hq)], dtype=np.float32)


def decode_inputs_e4m3_torch(w: DecodeWorkload, device, permute: bool = True):
    """decode_inputs_torch with the caches rounded to e4m3 (torch.float8_e4m3fn, round to
    nearest even): the FP8-e4m3 cache of the same synthetic values.  The NaN padding
    slots stay NaN codes; N(0,1) samples never come near e4m3's largest value, 448."""
    import torch

    t = decode_inputs_torch(w, device, permute)
    for which in ("k_cache", "v_cache"):
        t[which] = t[which].to(torch.float8_e4m3fn)
    return t


def decode_io_bytes(w: DecodeWorkload, lens: np.ndarray, kv_bytes: int = 2, window: int = 0) -> int:
    """Algorithmic HBM bytes of one decode call: each needed K/V byte once (kv_bytes per
    element: 2 for bf16, 1 for e4m3; with a window only the window + s_active - 1 newest
    positions are needed), the page table entries in use, cache_len, Q and O (bf16) and LSE."""
    lens = lens.astype(np.int64)
    need = np.minimum(lens, window + w.s_active - 1) if window > 0 else lens
    kv = int(need.sum()) * w.hkv * w.d * kv_bytes * 2
    first = lens - need  # the oldest needed position
    pages = int((-(-lens // w.page_size) - first // w.page_size).sum()) * 4 if w.paged else 0
    qo = 2 * w.b * w.hq * w.s_active * w.d * 2
    lse = w.b * w.hq * w.s_active * 4
    return kv + pages + w.b * 4 + qo + lse
