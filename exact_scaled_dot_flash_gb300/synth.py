"""Seeded synthetic inputs for exact scaled-dot-product attention.

This module is the one piece shared by the GPU path's tests/bench and by the
float64 oracle: it draws Q, K, V (and, for the key-padding workload, the
per-batch valid lengths and the additive fp32 bias) and rounds them to the
storage dtype. It holds none of the attention arithmetic.

Recipe (identical on both sides, stated once here):
  * bit generator: numpy's Philox-4x64 counter-based generator, keyed by the
    pair (seed, stream) through ``np.random.SeedSequence``; each tensor has its
    own stream (0 = Q, 1 = K, 2 = V, 3 = kv_lens, 4 = bias), so every tensor
    is independent of the shapes of the others;
  * values: standard normal draws in float32 times sigma, then rounded
    round-to-nearest-even to the storage dtype (fp32 stays as drawn; fp16 via
    numpy's IEEE conversion; bf16 by rounding the fp32 bit pattern);
  * key-padding lengths: integers uniform on [lo, hi] inclusive;
  * bias: fp32 standard normal, never rounded.

Storage format returned to callers: ``np.float32`` for F32, ``np.float16``
for F16, and ``np.uint16`` bit patterns for BF16 (numpy has no bfloat16).

The workload table ``WORKLOADS`` describes the benchmark shapes of the
attention pages: a small F32 causal case, a char-transformer-sized BF16 block
(B=8, H=8, S=128, D in {32, 64}), a long-context causal MHA (B=4, H=32,
S=4096, D=128, plus a wide-score variant with Q,K ~ N(0, 3^2)), a GQA case
(Hq=32, Hkv=8, S=8192) and an F16 key-padding + bias case. One more shape
exercises split-KV: the newest 256 query rows of a 32768-key GQA context
(B=1, Hq=32, Hkv=8, D=128, bottom-right causal), where one CTA per 256-row
block would leave most of the GPU idle.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

F32, F16, BF16 = "f32", "f16", "bf16"
DTYPES = (F32, F16, BF16)

# Mask kinds are bit flags, the same values the C ABI uses.
MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING = 0, 1, 2

STREAM_Q, STREAM_K, STREAM_V, STREAM_LENS, STREAM_BIAS = 0, 1, 2, 3, 4


def _gen(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([int(seed), int(stream)])))


def normal_f32(seed: int, stream: int, shape, sigma: float = 1.0) -> np.ndarray:
    """float32 N(0, sigma^2) draws for (seed, stream), C-contiguous."""
    x = _gen(seed, stream).standard_normal(size=tuple(shape), dtype=np.float32)
    if sigma != 1.0:
        x *= np.float32(sigma)
    return x


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bfloat16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def to_storage(x_f32: np.ndarray, dtype: str) -> np.ndarray:
    """Round a float32 array to the storage dtype (see module docstring)."""
    if dtype == F32:
        return np.ascontiguousarray(x_f32, dtype=np.float32)
    if dtype == F16:
        return np.ascontiguousarray(x_f32.astype(np.float16))
    if dtype == BF16:
        return f32_to_bf16_bits(x_f32)
    raise ValueError(f"unknown dtype {dtype!r}")


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention problem: shapes, dtype, mask, bias layout and input recipe."""
    name: str
    dtype: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Sk: int
    D: int
    mask: int = MASK_NONE
    bias: bool = False
    bias_b: int = 1
    bias_h: int = 1
    seed: int = 0
    sigma_qk: float = 1.0
    sigma_v: float = 1.0
    kv_len_range: tuple | None = None   # (lo, hi) inclusive, key-padding only
    scale: float | None = None          # default 1/sqrt(D)

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.D)

    @property
    def causal(self) -> bool:
        return bool(self.mask & MASK_CAUSAL)

    def flops(self) -> float:
        """Nominal attention FLOPs 4*B*Hq*Sq*Sk*D, halved for a causal mask."""
        f = 4.0 * self.B * self.Hq * self.Sq * self.Sk * self.D
        return f / 2.0 if self.causal else f

    def io_bytes(self) -> int:
        """Bytes read and written once: Q, K, V, O (+ bias, + kv_lens)."""
        es = {F32: 4, F16: 2, BF16: 2}[self.dtype]
        n = (2 * self.B * self.Hq * self.Sq + 2 * self.B * self.Hkv * self.Sk) * self.D * es
        if self.bias:
            n += self.bias_b * self.bias_h * self.Sq * self.Sk * 4
        if self.mask & MASK_KEY_PADDING:
            n += 4 * self.B
        return n

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "f32_causal_small": Workload("f32_causal_small", F32, 2, 2, 2, 64, 64, 16,
                                 mask=MASK_CAUSAL, seed=0),
    "bf16_block_d32": Workload("bf16_block_d32", BF16, 8, 8, 8, 128, 128, 32,
                               mask=MASK_CAUSAL, seed=1),
    "bf16_block_d64": Workload("bf16_block_d64", BF16, 8, 8, 8, 128, 128, 64,
                               mask=MASK_CAUSAL, seed=1),
    "bf16_causal_4k": Workload("bf16_causal_4k", BF16, 4, 32, 32, 4096, 4096, 128,
                               mask=MASK_CAUSAL, seed=2),
    "bf16_causal_4k_wide": Workload("bf16_causal_4k_wide", BF16, 4, 32, 32, 4096, 4096, 128,
                                    mask=MASK_CAUSAL, seed=3, sigma_qk=3.0),
    "bf16_gqa_8k": Workload("bf16_gqa_8k", BF16, 2, 32, 8, 8192, 8192, 128,
                            mask=MASK_CAUSAL, seed=4),
    "f16_padding_bias": Workload("f16_padding_bias", F16, 16, 16, 16, 1024, 1024, 64,
                                 mask=MASK_KEY_PADDING, bias=True, bias_b=1, bias_h=16,
                                 seed=5, kv_len_range=(256, 1024)),
    "bf16_gqa_chunk_32k": Workload("bf16_gqa_chunk_32k", BF16, 1, 32, 8, 256, 32768, 128,
                                   mask=MASK_CAUSAL, seed=6),
}


def make_inputs(w: Workload) -> dict:
    """Draw the inputs of workload ``w``.

    Returns a dict with ``q`` [B,Hq,Sq,D], ``k``/``v`` [B,Hkv,Sk,D] in storage
    format, ``kv_lens`` int32 [B] or None, ``bias`` float32
    [bias_b,bias_h,Sq,Sk] or None, plus ``scale`` (float) and ``mask`` (int).
    """
    q = to_storage(normal_f32(w.seed, STREAM_Q, (w.B, w.Hq, w.Sq, w.D), w.sigma_qk), w.dtype)
    k = to_storage(normal_f32(w.seed, STREAM_K, (w.B, w.Hkv, w.Sk, w.D), w.sigma_qk), w.dtype)
    v = to_storage(normal_f32(w.seed, STREAM_V, (w.B, w.Hkv, w.Sk, w.D), w.sigma_v), w.dtype)
    kv_lens = None
    if w.mask & MASK_KEY_PADDING:
        lo, hi = w.kv_len_range if w.kv_len_range is not None else (0, w.Sk)
        kv_lens = _gen(w.seed, STREAM_LENS).integers(lo, hi, size=w.B, endpoint=True).astype(np.int32)
    bias = None
    if w.bias:
        bias = normal_f32(w.seed, STREAM_BIAS, (w.bias_b, w.bias_h, w.Sq, w.Sk))
    return {"q": q, "k": k, "v": v, "kv_lens": kv_lens, "bias": bias,
            "scale": w.softmax_scale, "mask": w.mask}


# --------------------------------------------------------------- paged caches
STREAM_PAGED_Q, STREAM_PAGED_K, STREAM_PAGED_V, STREAM_PAGED_META = 8, 9, 10, 11
STREAM_MLA_QP, STREAM_MLA_KP = 12, 13


@dataclasses.dataclass(frozen=True)
class PagedWorkload:
    """Packed queries over a paged key/value cache (serving-shaped inputs)."""
    name: str
    dtype: str
    num_seqs: int
    Hq: int
    Hkv: int
    D: int
    page_size: int
    ctx_range: tuple          # (lo, hi) inclusive key lengths per sequence
    q_range: tuple            # (lo, hi) inclusive new queries per sequence (capped by its length)
    seed: int = 0
    causal: bool = True
    explicit_positions: bool = False  # random increasing positions instead of the newest tokens
    spare_pages: int = 3              # unused physical pages mixed into the cache
    scale: float | None = None

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.D)

    def replace(self, **kw) -> "PagedWorkload":
        return dataclasses.replace(self, **kw)


def make_paged_inputs(w: PagedWorkload) -> dict:
    """Draw a paged problem: per-sequence key lengths and query counts, a cache
    whose physical pages are a random permutation (so page tables scatter), and
    packed queries. Unused page-table entries are -1. Returns q [queries, Hq, D],
    k_cache/v_cache [pages, page_size, Hkv, D] in storage format, block_table
    int32 [num_seqs, max_pages], seq_lens, q_offsets [num_seqs + 1], positions
    (int32 [queries] or None) and scale.
    """
    meta = _paged_meta(w)
    total_q, pages, P = int(meta["q_offsets"][-1]), meta.pop("pages"), w.page_size
    q = to_storage(normal_f32(w.seed, STREAM_PAGED_Q, (total_q, w.Hq, w.D)), w.dtype)
    k = to_storage(normal_f32(w.seed, STREAM_PAGED_K, (pages, P, w.Hkv, w.D)), w.dtype)
    v = to_storage(normal_f32(w.seed, STREAM_PAGED_V, (pages, P, w.Hkv, w.D)), w.dtype)
    return {"q": q, "k_cache": k, "v_cache": v, **meta, "scale": w.softmax_scale}


def _paged_meta(w) -> dict:
    """Sequence lengths, query counts, scattered page tables, query offsets and
    (optional) explicit positions of a paged workload ``w``."""
    g = _gen(w.seed, STREAM_PAGED_META)
    lens = g.integers(w.ctx_range[0], w.ctx_range[1], size=w.num_seqs, endpoint=True).astype(np.int32)
    nq = np.array([g.integers(min(w.q_range[0], L), min(w.q_range[1], L), endpoint=True) if L > 0 else 0
                   for L in lens], dtype=np.int32)
    P = w.page_size
    need = (lens + P - 1) // P
    max_pages = max(1, int(need.max()) if w.num_seqs else 1)
    pages = int(need.sum()) + w.spare_pages
    perm = g.permutation(pages).astype(np.int32)
    table = np.full((w.num_seqs, max_pages), -1, dtype=np.int32)
    at = 0
    for s in range(w.num_seqs):
        table[s, :need[s]] = perm[at:at + need[s]]
        at += need[s]
    q_off = np.zeros(w.num_seqs + 1, dtype=np.int32)
    q_off[1:] = np.cumsum(nq)
    positions = None
    if w.explicit_positions:
        positions = np.concatenate([np.sort(g.choice(int(L), size=int(n), replace=False)) if n else
                                    np.zeros(0, dtype=np.int64) for L, n in zip(lens, nq)]).astype(np.int32)
    return {"block_table": table, "seq_lens": lens, "q_offsets": q_off, "positions": positions, "pages": pages}


@dataclasses.dataclass(frozen=True)
class MlaWorkload:
    """MLA with absorbed projections over a paged latent cache."""
    name: str
    dtype: str
    num_seqs: int
    H: int
    R: int                    # latent rank (query, latent and output width)
    Pd: int                   # positional (rope) width
    page_size: int
    ctx_range: tuple
    q_range: tuple
    seed: int = 0
    causal: bool = True
    explicit_positions: bool = False
    spare_pages: int = 3
    scale: float | None = None  # the original model's QK scale; default 1/sqrt(R + Pd)

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.R + self.Pd)

    def replace(self, **kw) -> "MlaWorkload":
        return dataclasses.replace(self, **kw)


def make_mla_inputs(w: MlaWorkload) -> dict:
    """q [queries, H, R], qp [queries, H, Pd], latent [pages, page_size, 1, R],
    kpos [pages, page_size, 1, Pd] in storage format, plus the paged metadata."""
    meta = _paged_meta(w)
    total_q, pages, P = int(meta["q_offsets"][-1]), meta.pop("pages"), w.page_size
    q = to_storage(normal_f32(w.seed, STREAM_PAGED_Q, (total_q, w.H, w.R)), w.dtype)
    qp = to_storage(normal_f32(w.seed, STREAM_MLA_QP, (total_q, w.H, w.Pd)), w.dtype)
    lat = to_storage(normal_f32(w.seed, STREAM_PAGED_K, (pages, P, 1, w.R)), w.dtype)
    kp = to_storage(normal_f32(w.seed, STREAM_MLA_KP, (pages, P, 1, w.Pd)), w.dtype)
    return {"q": q, "qp": qp, "latent": lat, "kpos": kp, **meta, "scale": w.softmax_scale}


PAGED_WORKLOADS = {
    # serving decode step: one new token per sequence over 1k-8k keys
    "bf16_paged_decode": PagedWorkload("bf16_paged_decode", BF16, 64, 32, 8, 128, 64, (1024, 8192), (1, 1),
                                       seed=20),
    # chunked prefill: 128-512 new tokens per sequence over 0.5k-4k keys
    "bf16_paged_prefill": PagedWorkload("bf16_paged_prefill", BF16, 16, 32, 8, 128, 64, (512, 4096),
                                        (128, 512), seed=21),
}


MLA_WORKLOADS = {
    # MLA decode step: 128 heads over a 512-rank latent (+64 positional) cache, 1k-8k tokens
    "bf16_mla_decode": MlaWorkload("bf16_mla_decode", BF16, 64, 128, 512, 64, 64, (1024, 8192), (1, 1), seed=30),
}
