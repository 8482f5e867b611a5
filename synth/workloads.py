"""Workload shapes and seeded input draws for absorbed-MLA decode.

Shapes follow the pages: the V2-Lite attention layer (16 heads, kv_lora_rank
512, RoPE key 64, nope head 128, value head 128) and the DeepSeek-V3 layer
(128 heads, same latent sizes).  Values are drawn with numpy's PCG64
generator, keyed by (seed, stream, index) so that one sequence of a large
batch can be re-drawn on its own.

Value recipe (identical for every workload unless noted):
  * c_KV: N(0,1) per element, then scaled to unit RMS per token (the
    RMSNorm that precedes caching, without a learned gain).  The quantized
    workload instead keeps raw N(0,1) values and multiplies a fixed, seeded
    1% of the 512 channels by 8 (per-channel outliers).
  * k_pe, q_pe: N(0,1), then rotated with interleaved-pair RoPE (theta
    10000) at the token's position; the query sits at position seqlen-1.
  * q_nope: N(0,1).
  * wkv_b (W_UKV): N(0, 1/sqrt(512)) per element, shape [H*(128+128), 512].
Every tensor is rounded to bfloat16 (round-to-nearest-even) before use; the
arrays returned here are the bf16 bit patterns (uint16).
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

D_C = 512      # kv_lora_rank: width of the cached latent c_KV
D_R = 64       # qk_rope_head_dim: width of the shared RoPE key k_pe
D_NOPE = 128   # qk_nope_head_dim
D_V = 128      # v_head_dim
PAGE = 64      # tokens per cache page

# stream ids inside one workload seed
_S_WEIGHTS, _S_QUERY, _S_SEQLEN, _S_PAGES, _S_OUTLIER, _S_SEQ = 0, 1, 2, 3, 4, 100
_S_PROJ_W, _S_PROJ_X = 5, 200


@dataclass(frozen=True)
class Workload:
    name: str
    H: int
    B: int
    seqlen: int            # uniform length; ignored when ragged
    seed: int
    ragged: bool = False   # lognormal lengths (median 4096, sigma 1, clip 256..32768)
    paged: bool = True     # seeded random page permutation; False = contiguous pages
    dist: str = "rmsnorm"  # "rmsnorm" or "outlier"
    fmts: tuple = ("bf16",)
    prefill: int = 0       # tokens appended before the decode token (tiny case)
    q_len: int = 1         # query tokens per row (the row's last q_len cached tokens, causal)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(D_NOPE + D_R)


WORKLOADS = {
    # V2-Lite single layer: 25-token prefill, then 1 decode token (26 cached)
    "v2lite_tiny": Workload("v2lite_tiny", H=16, B=1, seqlen=26, seed=0, paged=False, prefill=25),
    # V2-Lite shape decode batch over a contiguous cache
    "v2lite_batch": Workload("v2lite_batch", H=16, B=32, seqlen=4096, seed=1, paged=False),
    # DeepSeek-V3 shape decode over a paged cache with a random page table
    "v3_paged": Workload("v3_paged", H=128, B=64, seqlen=8192, seed=2),
    # V3 shape, ragged lognormal lengths
    "v3_ragged": Workload("v3_ragged", H=128, B=128, seqlen=0, seed=3, ragged=True),
    # V3 shape over a quantized cache (INT8, then INT4), latents with outlier channels
    "v3_quant": Workload("v3_quant", H=128, B=64, seqlen=32768, seed=4, dist="outlier",
                         fmts=("int8", "int4")),
    # several query tokens per row (speculative / multi-token-prediction decode):
    # the V2-Lite batch's cache with 8 causal queries per row, and the V3 paged
    # cache with 2
    "v2lite_mtp": Workload("v2lite_mtp", H=16, B=32, seqlen=4096, seed=1, paged=False, q_len=8),
    "v3_mtp": Workload("v3_mtp", H=128, B=64, seqlen=8192, seed=2, q_len=2),
}


def get_workload(name: str) -> Workload:
    return WORKLOADS[name]


# ----------------------------------------------------------------------------
# bfloat16 bit handling (input preparation only)
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(x) -> np.ndarray:
    """Round float32 values to bfloat16, nearest-even; returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def rope_interleaved(x: np.ndarray, pos) -> np.ndarray:
    """Rotate pairs (2i, 2i+1) of the last axis by pos * 10000^(-2i/d), in fp64."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    i = np.arange(d // 2, dtype=np.float64)
    theta = 10000.0 ** (-2.0 * i / d)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * theta
    c, s = np.cos(ang), np.sin(ang)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


# ----------------------------------------------------------------------------
# draws
# ----------------------------------------------------------------------------

def _rng(seed: int, *stream: int) -> np.random.Generator:
    return np.random.default_rng([seed, *stream])


def gen_seqlens(w: Workload) -> np.ndarray:
    if not w.ragged:
        return np.full(w.B, w.seqlen, dtype=np.int32)
    z = _rng(w.seed, _S_SEQLEN).standard_normal(w.B)
    n = np.rint(np.exp(math.log(4096.0) + 1.0 * z))
    return np.clip(n, 256, 32768).astype(np.int32)


def gen_weights(H: int, seed: int) -> np.ndarray:
    """wkv_b: [H*(D_NOPE+D_V), D_C] bf16 bits, N(0, 1/sqrt(512))."""
    w = _rng(seed, _S_WEIGHTS).standard_normal((H * (D_NOPE + D_V), D_C), dtype=np.float32)
    return f32_to_bf16_bits(w * np.float32(1.0 / math.sqrt(D_C)))


def gen_queries(H: int, seqlens, seed: int):
    """q_nope [B,H,128] and RoPE-rotated q_pe [B,H,64] (position seqlen-1), bf16 bits."""
    seqlens = np.asarray(seqlens)
    B = len(seqlens)
    r = _rng(seed, _S_QUERY)
    q_nope = r.standard_normal((B, H, D_NOPE), dtype=np.float32)
    q_pe = r.standard_normal((B, H, D_R), dtype=np.float32)
    pos = np.maximum(seqlens.astype(np.int64) - 1, 0)[:, None] * np.ones((1, H))
    q_pe = rope_interleaved(q_pe, pos).astype(np.float32)
    return f32_to_bf16_bits(q_nope), f32_to_bf16_bits(q_pe)


def gen_queries_multi(H: int, T: int, seqlens, seed: int):
    """T query tokens per row: q_nope [B,T,H,128] and q_pe [B,T,H,64] rotated at
    their positions n_b - T + t (the row's last T tokens), bf16 bits."""
    seqlens = np.asarray(seqlens)
    B = len(seqlens)
    r = _rng(seed, _S_QUERY, T)
    q_nope = r.standard_normal((B, T, H, D_NOPE), dtype=np.float32)
    q_pe = r.standard_normal((B, T, H, D_R), dtype=np.float32)
    pos = (seqlens.astype(np.int64)[:, None] - T + np.arange(T)[None, :]).clip(min=0)
    q_pe = rope_interleaved(q_pe, pos[:, :, None] * np.ones((1, 1, H))).astype(np.float32)
    return f32_to_bf16_bits(q_nope), f32_to_bf16_bits(q_pe)


def _outlier_channels(seed: int) -> np.ndarray:
    return np.sort(_rng(seed, _S_OUTLIER).choice(D_C, size=max(1, D_C // 100), replace=False))


def gen_sequence(seed: int, b: int, n: int, dist: str = "rmsnorm", start: int = 0):
    """Tokens [start, start+n) of sequence b: c_kv [n,512], k_pe [n,64] (bf16 bits).

    Token t is drawn from a stream keyed by (seed, b) so a sequence can be
    drawn in pieces (prefill then decode) with the same result.
    """
    r = _rng(seed, _S_SEQ, b)
    total = start + n
    x = r.standard_normal((total, D_C + D_R), dtype=np.float32)[start:]
    c = x[:, :D_C]
    if dist == "rmsnorm":
        ms = np.mean(c.astype(np.float64) ** 2, axis=1, keepdims=True)
        c = (c / np.sqrt(ms + 1e-6)).astype(np.float32)
    elif dist == "outlier":
        c = c.copy()
        c[:, _outlier_channels(seed)] *= np.float32(8.0)
    else:
        raise ValueError(dist)
    pos = np.arange(start, total, dtype=np.float64)
    k_pe = rope_interleaved(x[:, D_C:], pos).astype(np.float32)
    return f32_to_bf16_bits(c), f32_to_bf16_bits(k_pe)


def make_page_table(seqlens, seed: int, paged: bool, spare_pages: int = 0):
    """Logical→physical page map [B, max_pages] int32 (unused entries -1).

    paged=True assigns a seeded random permutation of the physical pages;
    paged=False gives each sequence a contiguous run (identity order).
    Returns (page_table, num_pages).
    """
    seqlens = np.asarray(seqlens, dtype=np.int64)
    npg = (seqlens + PAGE - 1) // PAGE
    max_pages = int(max(1, npg.max(initial=1)))
    num_pages = int(npg.sum()) + spare_pages
    phys = np.arange(num_pages, dtype=np.int32)
    if paged:
        phys = _rng(seed, _S_PAGES).permutation(num_pages).astype(np.int32)
    table = np.full((len(seqlens), max_pages), -1, dtype=np.int32)
    k = 0
    for b, m in enumerate(npg):
        table[b, :m] = phys[k:k + m]
        k += m
    return table, max(num_pages, 1)


# ----------------------------------------------------------------------------
# inputs of the cache producer (down-projection, RMSNorm, RoPE before append)
# ----------------------------------------------------------------------------
# hidden width of the attention input: 2048 for the V2-Lite layer (its outputs
# are [1, 1, 2048]), 7168 for DeepSeek-V3 ("dim" of its config)
HIDDEN = {"v2lite": 2048, "v3": 7168}


def gen_project_weights(hidden: int, seed: int):
    """wkv_a [576, hidden] ~ N(0, 1/sqrt(hidden)) and kv_norm weight [512] ~
    1 + 0.1 N(0,1), both as bf16 bits (the latent rows first, then the 64
    RoPE-key rows)."""
    r = _rng(seed, _S_PROJ_W)
    w = r.standard_normal((D_C + D_R, hidden), dtype=np.float32) * np.float32(1.0 / math.sqrt(hidden))
    g = np.float32(1.0) + np.float32(0.1) * r.standard_normal(D_C, dtype=np.float32)
    return f32_to_bf16_bits(w), f32_to_bf16_bits(g)


def gen_out_weights(H: int, hidden: int, seed: int) -> np.ndarray:
    """Wo [hidden, H*128] ~ N(0, 1/sqrt(H*128)) as bf16 bits (the layer's output
    projection after the heads)."""
    w = _rng(seed, _S_PROJ_W, 1).standard_normal((hidden, H * D_V), dtype=np.float32)
    return f32_to_bf16_bits(w * np.float32(1.0 / math.sqrt(H * D_V)))


def gen_hidden(hidden: int, seed: int, b: int, n: int) -> np.ndarray:
    """Attention inputs of n tokens of row b, [n, hidden] bf16 bits, N(0,1) (the
    layer input after its own RMSNorm has unit scale per element)."""
    x = _rng(seed, _S_PROJ_X, b).standard_normal((n, hidden), dtype=np.float32)
    return f32_to_bf16_bits(x)
