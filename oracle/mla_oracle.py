"""fp64 CPU oracle for absorbed Multi-head Latent Attention decode.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by
the CPU-baseline leg of the bench, never by the product package.  Nothing in
here is blocked, fused or reordered beyond what the definitions state; numpy
matrix products serve as single steps.

Sources (pages are cited by title and section):
  [audit]    "DeepSeek MLA 吸收式缓存：真实权重执行与 FlashMLA 架构边界"
             (DEEPSEEK_MLA_ABSORB_AUDIT.md)
  [report]   "DeepSeek-V2-Lite MLA 吸收式 KV 缓存优化 — 完整实验报告"
             (mla_absorbed_cache_report.md)
  [tutorial] "手搓 MLA:从 MHA 到 weight absorption,看懂 DeepSeek 的 KV 压缩"
  [budget]   "kv_budget.py" (算子实战 IV：MoE 与 MLA · 代码)

Pins (tests/test_oracle.py): the worked example's byte counts ([audit] §4.1,
§4.2), naive == absorbed to 1e-10 in fp64 ([audit] §2.2/§2.3, [tutorial] §四),
pure-Python brute-force attention on tiny inputs, closed forms (one token,
zero query, one dominant token), and hand-worked quantizer vectors.  The
producer of the cache payload (down-projection, RMSNorm, RoPE) is pinned by
hand-worked values, closed forms (unit RMS, scale invariance, rotation by
position 0 and by one radian), the relative-position property of RoPE and a
pure-Python brute force on odd tiny dimensions.  Causal attention of several
query tokens is pinned by a brute force, the first-prefill-token closed form
and the prefill-then-decode split of the V2-Lite case; the output projection
and the other quantizers of [report] §3.2 by hand-worked vectors, brute force
and error bounds.
The quantizer's rounding rules are readings of [report] §3.2, which gives no
formula; the pages' own error figures use an unstated metric, so the
quantization *error* is parity unpinned (the codes themselves are pinned to
the stated rules by hand-worked vectors).
"""

from __future__ import annotations

import math

import numpy as np

D_C = 512
D_R = 64
D_NOPE = 128
D_V = 128
PAGE = 64

__all__ = [
    "D_C", "D_R", "D_NOPE", "D_V", "PAGE",
    "split_wkv_b", "naive_decode", "absorbed_decode", "softmax",
    "latent_cache_bytes", "expanded_cache_bytes", "decode_arithmetic_intensity",
    "bf16_round", "bf16_from_bits", "bf16_to_bits",
    "quantize_int8", "quantize_int4_asym", "dequantize_int8", "dequantize_int4",
    "pack_nibbles", "page_bytes", "PAGE_LAYOUT",
    "quantize_token", "dequantized_tokens", "expected_page_pool",
    "rms_norm", "rope", "project_latent",
    "naive_attend_causal", "absorbed_attend_causal",
    "output_projection", "quantize_int8_per_token", "quantize_int8_per_tensor", "quantize_int4_sym",
    "dequantize_int4_sym",
]


# ----------------------------------------------------------------------------
# weights
# ----------------------------------------------------------------------------

def split_wkv_b(wkv_b, H: int, d_nope: int = D_NOPE, d_v: int = D_V):
    """Split the up-projection wkv_b [H*(d_nope+d_v), d_c] into W_UK, W_UV.

    [tutorial] §三 ("k_nope, v = split(kv_up)") splits the up-projected
    vector per head into the no-RoPE key part and the value part; read as a
    per-head interleave, rows [h*(dn+dv), h*(dn+dv)+dn) are W_UK[h] and the
    next dv rows are W_UV[h].  Returns fp64 arrays W_UK [H, dn, dc] and
    W_UV [H, dv, dc], index order h, d, c as in the absorbed einsums of
    [tutorial] §四.
    """
    W = np.asarray(wkv_b, dtype=np.float64)
    W = W.reshape(H, d_nope + d_v, W.shape[-1])
    return W[:, :d_nope, :].copy(), W[:, d_nope:, :].copy()


# ----------------------------------------------------------------------------
# attention, both paths
# ----------------------------------------------------------------------------

def softmax(s: np.ndarray) -> np.ndarray:
    """Softmax over the last axis: subtract the max, exponentiate, normalise."""
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def naive_decode(q_nope, q_pe, c_kv, k_pe, W_UK, W_UV, scale: float):
    """Expand-then-attend decode for one query token over n cached tokens.

    [audit] §2.1: every head expands each cached latent into its own key
    k_t = W_UK c_t and value v_t = W_UV c_t; [audit] §2.4 / [tutorial] §三:
    the key is concatenated with the shared RoPE key, k = [k_nope; k_pe], and
    the query is [q_nope; q_pe].  Standard attention follows.

    q_nope [H, dn], q_pe [H, dr], c_kv [n, dc], k_pe [n, dr] -> out [H, dv].
    """
    q_nope = np.asarray(q_nope, np.float64)
    q_pe = np.asarray(q_pe, np.float64)
    C = np.asarray(c_kv, np.float64)
    Kpe = np.asarray(k_pe, np.float64)
    H = q_nope.shape[0]
    n = C.shape[0]
    out = np.zeros((H, W_UV.shape[1]), dtype=np.float64)
    if n == 0:
        return out
    for h in range(H):
        k_nope = C @ W_UK[h].T                       # [n, dn]: k_t = W_UK[h] c_t
        v = C @ W_UV[h].T                            # [n, dv]: v_t = W_UV[h] c_t
        K = np.concatenate([k_nope, Kpe], axis=1)    # [n, dn+dr]
        q = np.concatenate([q_nope[h], q_pe[h]])     # [dn+dr]
        p = softmax(scale * (K @ q))
        out[h] = p @ v
    return out


def absorbed_decode(q_nope, q_pe, c_kv, k_pe, W_UK, W_UV, scale: float):
    """Absorbed decode for one query token over n cached tokens.

    [audit] §2.2: q^T (W_UK c_t) = (W_UK^T q)^T c_t, so the query is moved
    into latent space, q_lat = W_UK^T q_nope, and dotted with the cached
    latent directly; the RoPE part q_pe . k_pe_t is added unchanged
    ([audit] §2.4).  [audit] §2.3: sum_t p_t W_UV c_t = W_UV (sum_t p_t c_t),
    so the probabilities weight the latents and W_UV is applied once.
    [tutorial] §四 writes the same steps as einsums.

    Returns out [H, dv], o_lat [H, dc] and lse [H] (natural-log sum of the
    exponentiated scaled scores; -inf when n == 0).
    """
    q_nope = np.asarray(q_nope, np.float64)
    q_pe = np.asarray(q_pe, np.float64)
    C = np.asarray(c_kv, np.float64)
    Kpe = np.asarray(k_pe, np.float64)
    H = q_nope.shape[0]
    n = C.shape[0]
    if n == 0:
        return (np.zeros((H, W_UV.shape[1])), np.zeros((H, C.shape[1])),
                np.full(H, -np.inf))
    q_lat = np.einsum("hd,hdc->hc", q_nope, W_UK)    # W_UK[h]^T q_nope[h]
    s = scale * (q_lat @ C.T + q_pe @ Kpe.T)         # [H, n]
    m = np.max(s, axis=1, keepdims=True)
    e = np.exp(s - m)
    l = np.sum(e, axis=1, keepdims=True)
    o_lat = (e / l) @ C                              # sum_t p_t c_t
    out = np.einsum("hc,hdc->hd", o_lat, W_UV)       # W_UV[h] o_lat[h]
    lse = m[:, 0] + np.log(l[:, 0])
    return out, o_lat, lse


# ----------------------------------------------------------------------------
# several query tokens per row (prefill chunk, incremental decode), causal
# ----------------------------------------------------------------------------

def _causal_visible(n: int, q_pos):
    """[T, n] boolean: cached token s is visible to query t iff s <= q_pos[t]."""
    return np.arange(n)[None, :] <= np.asarray(q_pos)[:, None]


def naive_attend_causal(q_nope, q_pe, c_kv, k_pe, W_UK, W_UV, scale: float, q_pos=None):
    """Expand-then-attend for T query tokens over n cached tokens, causal.

    [audit] §3.4 runs the same layer as a 25-token prefill and a 1-token
    incremental decode on the causal path; [audit] §2.1 expands every cached
    latent into per-head keys W_UK c_t (with the shared RoPE key appended,
    §2.4) and values W_UV c_t.  Query t sits at position q_pos[t] (default: the
    last T positions, n-T .. n-1) and sees cached tokens 0 .. q_pos[t].

    q_nope [T, H, dn], q_pe [T, H, dr], c_kv [n, dc], k_pe [n, dr] -> out [T, H, dv].
    """
    q_nope = np.asarray(q_nope, np.float64)
    q_pe = np.asarray(q_pe, np.float64)
    C = np.asarray(c_kv, np.float64)
    Kpe = np.asarray(k_pe, np.float64)
    T, H = q_nope.shape[:2]
    n = C.shape[0]
    q_pos = np.arange(n - T, n) if q_pos is None else np.asarray(q_pos)
    vis = _causal_visible(n, q_pos)
    out = np.zeros((T, H, W_UV.shape[1]))
    for h in range(H):
        K = np.concatenate([C @ W_UK[h].T, Kpe], axis=1)     # [n, dn+dr]
        V = C @ W_UV[h].T                                    # [n, dv]
        Q = np.concatenate([q_nope[:, h], q_pe[:, h]], axis=1)  # [T, dn+dr]
        s = np.where(vis, scale * (Q @ K.T), -np.inf)        # [T, n]
        out[:, h] = softmax(s) @ V
    return out


def absorbed_attend_causal(q_nope, q_pe, c_kv, k_pe, W_UK, W_UV, scale: float, q_pos=None):
    """Absorbed attention for T query tokens over n cached tokens, causal.

    The einsums of [tutorial] §四 with the query-token axis t and the cached
    axis s: q_lat = einsum("thd,hdc->thc"), scores = einsum("thc,sc->hts") +
    einsum("thd,sd->hts") (the RoPE key shared by all heads), a causal mask
    (query t sees s <= q_pos[t], [audit] §3.4), softmax over s, o_lat =
    einsum("hts,sc->thc"), out = einsum("thc,hdc->thd").  Returns out
    [T, H, dv] and o_lat [T, H, dc].
    """
    q_nope = np.asarray(q_nope, np.float64)
    q_pe = np.asarray(q_pe, np.float64)
    C = np.asarray(c_kv, np.float64)
    Kpe = np.asarray(k_pe, np.float64)
    T = q_nope.shape[0]
    n = C.shape[0]
    q_pos = np.arange(n - T, n) if q_pos is None else np.asarray(q_pos)
    q_lat = np.einsum("thd,hdc->thc", q_nope, W_UK)
    s = scale * (np.einsum("thc,sc->hts", q_lat, C) + np.einsum("thd,sd->hts", q_pe, Kpe))
    s = np.where(_causal_visible(n, q_pos)[None, :, :], s, -np.inf)
    p = softmax(s)                                           # over s, per (h, t)
    o_lat = np.einsum("hts,sc->thc", p, C)
    return np.einsum("thc,hdc->thd", o_lat, W_UV), o_lat


# ----------------------------------------------------------------------------
# the step before the cache: down-projection, RMSNorm, RoPE
# ----------------------------------------------------------------------------

def rms_norm(v, weight, eps: float):
    """RMSNorm over the last axis: v / sqrt(mean(v^2) + eps) * weight.

    [tutorial] §三 normalises the down-projected latent before it is cached,
    c_kv = rmsnorm(x @ W_DKV.T, W_KVN); [audit] §3.3 maps the learned gain
    W_KVN to the checkpoint's kv_norm weight.  The page states no epsilon:
    it is an argument here.
    """
    v = np.asarray(v, dtype=np.float64)
    ms = np.mean(v * v, axis=-1, keepdims=True)
    return v / np.sqrt(ms + eps) * np.asarray(weight, dtype=np.float64)


def rope(x, pos, theta: float = 10000.0):
    """Rotary position embedding of the last axis at integer positions `pos`.

    [tutorial] §三 rotates the shared key before caching, k_pe = rope(x @
    W_KR.T).  The pages give no pairing convention; read here as consecutive
    pairs (2i, 2i+1) rotated by the angle pos * theta^(-2i/d):
    (a, b) -> (a cos - b sin, a sin + b cos), all in fp64.
    x [..., d] (d even), pos broadcastable to x.shape[:-1].
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    freq = theta ** (-2.0 * np.arange(d // 2, dtype=np.float64) / d)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * freq
    cos, sin = np.cos(ang), np.sin(ang)
    a, b = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = a * cos - b * sin
    out[..., 1::2] = a * sin + b * cos
    return out


def project_latent(x, wkv_a, kv_norm_w, pos, eps: float, theta: float = 10000.0):
    """The cache payload of n tokens from their attention inputs.

    [tutorial] §三: c_kv = rmsnorm(x @ W_DKV.T, W_KVN) and k_pe =
    rope(x @ W_KR.T).  [audit] §3.3 names the joint projection wkv_a
    (kv_a_proj_with_mqa): its first d_c rows are W_DKV, the remaining d_r rows
    W_KR (the shared RoPE key appended to the latent projection).
    x [n, hidden], wkv_a [d_c + d_r, hidden], kv_norm_w [d_c], pos [n].
    Returns c_kv [n, d_c] and k_pe [n, d_r] in fp64.
    """
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(wkv_a, dtype=np.float64)
    d_c = np.shape(kv_norm_w)[-1]
    y = x @ w.T                                   # [n, d_c + d_r]
    return rms_norm(y[:, :d_c], kv_norm_w, eps), rope(y[:, d_c:], pos, theta)


# ----------------------------------------------------------------------------
# after the up-projection: the layer's output projection
# ----------------------------------------------------------------------------

def output_projection(out_heads, wo):
    """The layer output: the heads' outputs side by side, times Wo^T.

    [tutorial] §三 and §四 end both paths with "@ Wo.T" after reshaping the
    per-head outputs to [T, H*dv] (its MHA listing does the reshape
    explicitly); [audit] §3.3 maps o_proj to wo.  out_heads [T, H, dv],
    wo [hidden, H*dv] -> [T, hidden].
    """
    o = np.asarray(out_heads, dtype=np.float64)
    T = o.shape[0]
    return o.reshape(T, -1) @ np.asarray(wo, dtype=np.float64).T


# ----------------------------------------------------------------------------
# the other cache quantizers [report] §3.2 compares (same rounding rules)
# ----------------------------------------------------------------------------

def quantize_int8_per_token(x):
    """INT8 with one scale per token over all its channels ([report] §3.2
    "per-token INT8"): the symmetric INT8 rule of quantize_int8 with a group
    that spans the whole row."""
    x = np.asarray(x, dtype=np.float32)
    return quantize_int8(x, x.shape[-1])


def quantize_int8_per_tensor(x):
    """INT8 with one scale for the whole tensor ([report] §3.2 "per-tensor
    INT8"): s = bf16(amax / 127) over every element, code = clamp(rint(x / s),
    -127, 127).  Returns int8 codes (shape of x) and the scalar scale."""
    x = np.asarray(x, dtype=np.float32)
    codes, s = quantize_int8(x.reshape(1, -1), x.size)
    return codes.reshape(x.shape), s.reshape(())


def quantize_int4_sym(x, group: int):
    """Symmetric INT4 over contiguous groups ([report] §3.2 "对称 INT4 (32块)" for
    c_KV and "k_pe 对称 INT4 (8块)").  Reading, by analogy with the INT8 rule
    (the page gives no formula): s = bf16(amax / 7) in fp32, code = clamp(
    rint(x / s), -7, 7) half to even, all-zero codes when s is 0; x^ = code * s.
    Returns int8 codes in -7..7 (shape of x) and float32 scales [..., k]."""
    x = np.asarray(x, dtype=np.float32)
    g = x.reshape(*x.shape[:-1], x.shape[-1] // group, group)
    amax = np.max(np.abs(g), axis=-1)
    s = bf16_round(amax / np.float32(7.0))
    safe = np.where(s == 0, np.float32(1.0), s).astype(np.float32)
    q = np.clip(np.rint(g / safe[..., None]), -7, 7)
    q = np.where((s == 0)[..., None], 0, q)
    return q.astype(np.int8).reshape(x.shape), s


def dequantize_int4_sym(codes, scales, group: int) -> np.ndarray:
    return dequantize_int8(codes, scales, group)


# ----------------------------------------------------------------------------
# byte accounting
# ----------------------------------------------------------------------------

def latent_cache_bytes(ntok: int, d_c: int = D_C, d_r: int = D_R, elem_bytes: int = 2) -> int:
    """Absorbed cache: one c_KV and one k_pe per token ([audit] §2.4, §4.1)."""
    return ntok * (d_c + d_r) * elem_bytes


def expanded_cache_bytes(ntok: int, H: int, d_qk: int = D_NOPE + D_R, d_v: int = D_V,
                         elem_bytes: int = 2) -> int:
    """Naive cache: per-head expanded key (nope+rope) and value ([audit] §2.1, §4.1)."""
    return ntok * H * (d_qk + d_v) * elem_bytes


def decode_arithmetic_intensity(H: int, d_c: int = D_C, d_r: int = D_R, elem_bytes: int = 2) -> float:
    """FLOP per cached byte of one absorbed decode query ([budget] part B):
    each token costs 2*H*(d_c+d_r) for the scores and 2*H*d_c for the
    latent sum over (d_c+d_r)*elem_bytes bytes."""
    return 2.0 * H * (2 * d_c + d_r) / (elem_bytes * (d_c + d_r))


# ----------------------------------------------------------------------------
# bfloat16 and the cache quantizers (fp32 decisions, bit-exact)
# ----------------------------------------------------------------------------

def bf16_round(x) -> np.ndarray:
    """float32 -> nearest-even bfloat16, returned as float32 values."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16))
    return (r.astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_to_bits(x) -> np.ndarray:
    """bfloat16-representable float32 values -> uint16 bit patterns."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_from_bits(bits) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def quantize_int8(x, group: int):
    """Symmetric INT8 over contiguous groups of `group` channels of one token.

    [report] §3.2 lists per-channel INT8 in 32-element blocks for c_KV and
    INT8 in 8-element blocks for k_pe.  Reading (no formula on the page):
    scale s = bf16(amax / 127) computed in fp32, code = clamp(rint(x / s),
    -127, 127) with round-half-even; a group whose s is 0 stores all-zero
    codes.  x: float32 [..., k*group].  Returns int8 codes (same shape) and
    float32 scales [..., k] holding bf16 values.
    """
    x = np.asarray(x, dtype=np.float32)
    g = x.reshape(*x.shape[:-1], x.shape[-1] // group, group)
    amax = np.max(np.abs(g), axis=-1)
    s = bf16_round(amax / np.float32(127.0))
    safe = np.where(s == 0, np.float32(1.0), s).astype(np.float32)
    q = np.rint(g / safe[..., None])
    q = np.clip(q, -127, 127)
    q = np.where((s == 0)[..., None], 0, q)
    return q.astype(np.int8).reshape(x.shape), s


def quantize_int4_asym(x, group: int = 32):
    """Asymmetric INT4 over contiguous groups of one token's channels.

    [report] §3.2 names asymmetric INT4 in 32-element blocks (scale + zero).
    Reading: mn, mx = group min and max; s = bf16((mx - mn) / 15) in fp32;
    zero = bf16(mn); code = clamp(rint((x - zero) / s), 0, 15), all-zero codes
    when s is 0.  Dequantised value = code * s + zero.  Returns uint8 codes
    0..15 (unpacked, same shape as x), float32 scales and zeros [..., k].
    """
    x = np.asarray(x, dtype=np.float32)
    g = x.reshape(*x.shape[:-1], x.shape[-1] // group, group)
    mn = np.min(g, axis=-1)
    mx = np.max(g, axis=-1)
    s = bf16_round((mx - mn) / np.float32(15.0))
    z = bf16_round(mn)
    safe = np.where(s == 0, np.float32(1.0), s).astype(np.float32)
    q = np.rint((g - z[..., None]) / safe[..., None])
    q = np.clip(q, 0, 15)
    q = np.where((s == 0)[..., None], 0, q)
    return q.astype(np.uint8).reshape(x.shape), s, z


def dequantize_int8(codes, scales, group: int) -> np.ndarray:
    c = np.asarray(codes, dtype=np.float64)
    c = c.reshape(*c.shape[:-1], c.shape[-1] // group, group)
    return (c * np.asarray(scales, np.float64)[..., None]).reshape(np.shape(codes))


def dequantize_int4(codes, scales, zeros, group: int = 32) -> np.ndarray:
    c = np.asarray(codes, dtype=np.float64)
    c = c.reshape(*c.shape[:-1], c.shape[-1] // group, group)
    v = c * np.asarray(scales, np.float64)[..., None] + np.asarray(zeros, np.float64)[..., None]
    return v.reshape(np.shape(codes))


def pack_nibbles(codes) -> np.ndarray:
    """Two 4-bit codes per byte: element 2i in the low nibble, 2i+1 in the high."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


# ----------------------------------------------------------------------------
# page format (the cache contract of the library, restated independently)
# ----------------------------------------------------------------------------
# Each physical page holds PAGE token slots.  Sections (byte offset, dtype,
# per-token shape) in page order:
PAGE_LAYOUT = {
    "bf16": [("tok", "bf16", (D_C + D_R,))],            # c_kv then k_pe per slot
    "int8": [("c_code", "i8", (D_C,)), ("pe_code", "i8", (D_R,)),
             ("c_scale", "bf16", (D_C // 32,)), ("pe_scale", "bf16", (D_R // 8,))],
    "int4": [("c_code", "u4x2", (D_C // 2,)), ("pe_code", "i8", (D_R,)),
             ("c_scale", "bf16", (D_C // 32,)), ("c_zero", "bf16", (D_C // 32,)),
             ("pe_scale", "bf16", (D_R // 8,))],
}
# the per-token INT8, symmetric INT4 and 4-bit k_pe quantizers of [report] §3.2
# write the INT8 and INT4 page layouts (the library's reading: one page form per
# code width; the 4-bit k_pe codes -7..7 sit in the INT8 k_pe code section)
PAGE_LAYOUT["int8_token"] = PAGE_LAYOUT["int8"]
PAGE_LAYOUT["int4_sym"] = PAGE_LAYOUT["int4"]
PAGE_LAYOUT["int4_pe4"] = PAGE_LAYOUT["int4"]
_ELEM = {"bf16": 2, "i8": 1, "u4x2": 1}


def _sections(fmt: str, page: int = PAGE):
    off = 0
    out = {}
    for name, dt, shp in PAGE_LAYOUT[fmt]:
        nbytes = page * int(np.prod(shp)) * _ELEM[dt]
        out[name] = (off, dt, shp, nbytes)
        off += nbytes
    return out, off


def page_bytes(fmt: str, page: int = PAGE) -> int:
    return _sections(fmt, page)[1]


def quantize_token(fmt: str, c_kv, k_pe):
    """Per-token payload of one format, as {section: array} for `n` tokens.

    c_kv [n, dc], k_pe [n, dr] are bf16-representable float32 values.
    """
    c = np.asarray(c_kv, np.float32)
    p = np.asarray(k_pe, np.float32)
    if fmt == "bf16":
        return {"tok": bf16_to_bits(np.concatenate([c, p], axis=1))}
    # k_pe: INT8 in 8-dim groups, or symmetric INT4 in 8-dim groups ("k_pe 对称 INT4 (8块)")
    pc, ps = quantize_int4_sym(p, 8) if fmt == "int4_pe4" else quantize_int8(p, 8)
    if fmt == "int8":
        cc, cs = quantize_int8(c, 32)
        return {"c_code": cc, "pe_code": pc, "c_scale": bf16_to_bits(cs),
                "pe_scale": bf16_to_bits(ps)}
    if fmt in ("int4", "int4_pe4"):
        cc, cs, cz = quantize_int4_asym(c, 32)
        return {"c_code": pack_nibbles(cc), "pe_code": pc, "c_scale": bf16_to_bits(cs),
                "c_zero": bf16_to_bits(cz), "pe_scale": bf16_to_bits(ps)}
    if fmt == "int8_token":
        # one scale per token, repeated in the token's 16 group-scale slots
        cc, cs = quantize_int8_per_token(c)
        return {"c_code": cc, "pe_code": pc, "c_scale": bf16_to_bits(np.repeat(cs, D_C // 32, axis=-1)),
                "pe_scale": bf16_to_bits(ps)}
    if fmt == "int4_sym":
        # codes q in -7..7 stored as q + 8, zero -8 s: code * s + zero = q * s
        q, cs = quantize_int4_sym(c, 32)
        return {"c_code": pack_nibbles((q.astype(np.int16) + 8).astype(np.uint8)), "pe_code": pc,
                "c_scale": bf16_to_bits(cs), "c_zero": bf16_to_bits(np.float32(-8.0) * cs),
                "pe_scale": bf16_to_bits(ps)}
    raise ValueError(fmt)


def dequantized_tokens(fmt: str, c_kv, k_pe):
    """The real values a decode over a `fmt` cache attends to (fp64)."""
    c = np.asarray(c_kv, np.float32)
    p = np.asarray(k_pe, np.float32)
    if fmt == "bf16":
        return c.astype(np.float64), p.astype(np.float64)
    if fmt == "int4_pe4":
        pc, ps = quantize_int4_sym(p, 8)
        pe = dequantize_int4_sym(pc, ps, 8)
    else:
        pc, ps = quantize_int8(p, 8)
        pe = dequantize_int8(pc, ps, 8)
    if fmt == "int8":
        cc, cs = quantize_int8(c, 32)
        return dequantize_int8(cc, cs, 32), pe
    if fmt == "int8_token":
        cc, cs = quantize_int8_per_token(c)
        return dequantize_int8(cc, cs, D_C), pe
    if fmt == "int4_sym":
        q, cs = quantize_int4_sym(c, 32)
        return dequantize_int4_sym(q, cs, 32), pe
    cc, cs, cz = quantize_int4_asym(c, 32)
    return dequantize_int4(cc, cs, cz, 32), pe


def expected_page_pool(fmt: str, num_pages: int, writes, page: int = PAGE) -> np.ndarray:
    """Byte image of a page pool after appending tokens, starting from zeros.

    writes: iterable of (page_table_row, pos, c_kv [T, dc], k_pe [T, dr]);
    token t of the row lands in physical page row[(pos+t) // page], slot
    (pos+t) % page.  Returns uint8 [num_pages, page_bytes(fmt)].
    """
    secs, pb = _sections(fmt, page)
    pool = np.zeros((num_pages, pb), dtype=np.uint8)
    for row, pos, c, p in writes:
        payload = quantize_token(fmt, c, p)
        for t in range(np.shape(c)[0]):
            lp = (pos + t) // page
            slot = (pos + t) % page
            phys = int(row[lp])
            for name, arr in payload.items():
                off, dt, shp, nbytes = secs[name]
                per_tok = nbytes // page
                raw = np.ascontiguousarray(arr[t]).view(np.uint8).reshape(-1)
                assert raw.size == per_tok
                pool[phys, off + slot * per_tok: off + (slot + 1) * per_tok] = raw
    return pool
