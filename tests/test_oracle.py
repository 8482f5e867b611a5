"""Pins for the CPU oracle: values the pages print, closed forms, brute force.

None of these compare the oracle with itself: each expected value is either
printed on a page (tests/golden/*.json, with the citation inside), follows
from a closed form of a special case, or comes from a separate pure-Python
brute-force loop.
"""

import json
import math
import os
import random

import numpy as np
import pytest

import oracle as O
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------
# byte accounting: the worked example of the audit page
# ----------------------------------------------------------------------------

def test_cache_bytes_worked_example():
    g = _gold("audit_cache_bytes.json")
    H, n, slots = g["H"], g["active_tokens"], g["allocated_slots"]
    a = g["active_bytes"]
    assert O.latent_cache_bytes(n) == a["absorb_total"]
    assert O.latent_cache_bytes(n, d_r=0) == a["absorb_latent"]
    assert O.latent_cache_bytes(n, d_c=0) == a["absorb_rope"]
    assert O.expanded_cache_bytes(n, H) == a["naive_total"]
    assert O.expanded_cache_bytes(n, H, d_v=0) == a["naive_key"]
    assert O.expanded_cache_bytes(n, H, d_qk=0) == a["naive_value"]
    al = g["allocated_bytes"]
    assert O.latent_cache_bytes(slots) == al["absorb_total"]
    assert O.expanded_cache_bytes(slots, H) == al["naive_total"]
    assert O.expanded_cache_bytes(slots, H, d_v=0) == al["naive_key"]
    ratio = O.expanded_cache_bytes(n, H) / O.latent_cache_bytes(n)
    assert abs(ratio - g["ratio_naive_over_absorb"]) < 1e-6
    assert ratio == pytest.approx(80.0 / 9.0)
    assert 100.0 * (1 - 1 / ratio) == pytest.approx(g["reduction_percent"])
    e = g["elements_per_token"]
    assert O.expanded_cache_bytes(1, H, elem_bytes=1) == e["naive_total"]
    assert O.latent_cache_bytes(1, elem_bytes=1) == e["absorbed_total"]


def test_cache_bytes_against_real_buffers():
    """Count the bytes of actual arrays shaped like both caches (audit §4.1)."""
    g = _gold("audit_cache_bytes.json")
    n, H = g["active_tokens"], g["H"]
    k = np.zeros((1, n, H, O.D_NOPE + O.D_R), dtype=np.uint16)
    v = np.zeros((1, n, H, O.D_V), dtype=np.uint16)
    lat = np.zeros((1, n, O.D_C), dtype=np.uint16)
    pe = np.zeros((1, n, O.D_R), dtype=np.uint16)
    assert k.nbytes == g["active_bytes"]["naive_key"]
    assert v.nbytes == g["active_bytes"]["naive_value"]
    assert lat.nbytes == g["active_bytes"]["absorb_latent"]
    assert pe.nbytes == g["active_bytes"]["absorb_rope"]


def test_v3_bytes_table():
    g = _gold("tutorial_v3_bytes.json")
    assert O.latent_cache_bytes(1, elem_bytes=1) == g["per_token_layer"]["MLA"]["elements"]
    assert O.latent_cache_bytes(1) == g["per_token_layer"]["MLA"]["bf16_bytes"]
    mha = g["per_token_layer"]["MHA"]["elements"]
    assert round(mha / O.latent_cache_bytes(1, elem_bytes=1)) == g["mha_over_mla_approx"]
    kb = O.latent_cache_bytes(1) * g["layers"] / 1000   # 70,272 B: "about 70 KB"
    assert round(kb) == g["mla_61_layer_kb_approx"]


def test_report_quantized_sizes():
    """Codes-only per-token sizes over 27 layers (report §3.1, §4.1)."""
    g = _gold("report_quant_sizes.json")
    L = g["layers"]
    mha = O.expanded_cache_bytes(1, 16) * L
    assert mha == g["mha_equiv_bytes"]
    absorbed = O.latent_cache_bytes(1) * L
    int8 = O.latent_cache_bytes(1, elem_bytes=1) * L
    int4 = O.latent_cache_bytes(1, elem_bytes=1) * L // 2
    assert round(absorbed / 1024, 1) == g["absorbed_kb"]
    assert round(int8 / 1024, 1) == g["int8_kb"]
    assert round(int4 / 1024, 1) == g["int4_kb"]
    assert round(mha / absorbed, 1) == g["ratio_absorbed"]
    assert round(mha / int8, 1) == g["ratio_int8"]
    assert round(mha / int4, 1) == g["ratio_int4"]


def test_page_formats():
    """Per-token page payload: 1152 B bf16, 624 B INT8, 400 B INT4 (codes+scales+zeros)."""
    assert O.page_bytes("bf16") == 64 * 1152
    assert O.page_bytes("int8") == 64 * (512 + 64 + 2 * 16 + 2 * 8)
    assert O.page_bytes("int4") == 64 * (256 + 64 + 2 * 16 + 2 * 16 + 2 * 8)


def test_arithmetic_intensity_closed_form():
    # kv_budget.py part B: 2*Hq*(2dc+dr)/(b*(dc+dr)); V3 shape -> 241.8 FLOP/B
    assert O.decode_arithmetic_intensity(128) == pytest.approx(2 * 128 * 1088 / 1152)
    # heads needed to reach a 1000/3 FLOP/B machine balance (H100 spec on the page)
    need = (1000.0 / 3.0) * 2 * 576 / (2 * 1088)
    assert round(need) == 176


# ----------------------------------------------------------------------------
# weight split
# ----------------------------------------------------------------------------

def test_split_wkv_b_rows():
    H = 3
    w = np.arange(H * 256, dtype=np.float64)[:, None] * np.ones((1, 5))
    uk, uv = O.split_wkv_b(w, H)
    for h in range(H):
        assert np.all(uk[h][:, 0] == h * 256 + np.arange(128))
        assert np.all(uv[h][:, 0] == h * 256 + 128 + np.arange(128))


# ----------------------------------------------------------------------------
# attention: brute force, associativity, closed forms
# ----------------------------------------------------------------------------

def _bruteforce(q_nope, q_pe, C, Kpe, Wuk, Wuv, scale):
    """Pure-Python loops: expand K/V per head, softmax by max-subtract-exp-divide."""
    H, dn = len(q_nope), len(q_nope[0])
    n, dc = len(C), len(C[0])
    dv = len(Wuv[0])
    out = []
    for h in range(H):
        s = []
        vs = []
        for t in range(n):
            k = [math.fsum(Wuk[h][d][c] * C[t][c] for c in range(dc)) for d in range(dn)]
            k += list(Kpe[t])
            q = list(q_nope[h]) + list(q_pe[h])
            s.append(scale * math.fsum(a * b for a, b in zip(q, k)))
            vs.append([math.fsum(Wuv[h][d][c] * C[t][c] for c in range(dc)) for d in range(dv)])
        m = max(s)
        e = [math.exp(x - m) for x in s]
        z = math.fsum(e)
        out.append([math.fsum(e[t] / z * vs[t][d] for t in range(n)) for d in range(dv)])
    return out


def _rand(rng, *shape):
    return rng.standard_normal(shape)


@pytest.mark.parametrize("n", [1, 2, 5])
def test_bruteforce_tiny_odd_dims(n):
    """Odd, unequal dims so a transposed or swapped operand fails."""
    rng = np.random.default_rng(11 + n)
    H, dn, dr, dc, dv = 2, 3, 2, 7, 5
    q_nope, q_pe = _rand(rng, H, dn), _rand(rng, H, dr)
    C, Kpe = _rand(rng, n, dc), _rand(rng, n, dr)
    Wuk, Wuv = _rand(rng, H, dn, dc), _rand(rng, H, dv, dc)
    scale = 0.37
    ref = np.array(_bruteforce(q_nope.tolist(), q_pe.tolist(), C.tolist(), Kpe.tolist(),
                               Wuk.tolist(), Wuv.tolist(), scale))
    naive = O.naive_decode(q_nope, q_pe, C, Kpe, Wuk, Wuv, scale)
    absorbed, _, _ = O.absorbed_decode(q_nope, q_pe, C, Kpe, Wuk, Wuv, scale)
    assert np.max(np.abs(naive - ref)) < 1e-12
    assert np.max(np.abs(absorbed - ref)) < 1e-12


def test_lse_bruteforce():
    rng = np.random.default_rng(5)
    H, n = 2, 6
    q_nope, q_pe = _rand(rng, H, 3), _rand(rng, H, 2)
    C, Kpe = _rand(rng, n, 4), _rand(rng, n, 2)
    Wuk, Wuv = _rand(rng, H, 3, 4), _rand(rng, H, 2, 4)
    _, _, lse = O.absorbed_decode(q_nope, q_pe, C, Kpe, Wuk, Wuv, 0.5)
    for h in range(H):
        s = []
        for t in range(n):
            k = [sum(Wuk[h][d][c] * C[t][c] for c in range(4)) for d in range(3)] + list(Kpe[t])
            q = list(q_nope[h]) + list(q_pe[h])
            s.append(0.5 * sum(a * b for a, b in zip(q, k)))
        assert lse[h] == pytest.approx(math.log(math.fsum(math.exp(x) for x in s)), abs=1e-12)


def _tiny_inputs():
    w = synth.get_workload("v2lite_tiny")
    wkv = synth.bf16_bits_to_f32(synth.gen_weights(w.H, w.seed))
    qn, qp = synth.gen_queries(w.H, [w.seqlen], w.seed)
    c, p = synth.gen_sequence(w.seed, 0, w.seqlen)
    Wuk, Wuv = O.split_wkv_b(wkv, w.H)
    return (synth.bf16_bits_to_f32(qn)[0], synth.bf16_bits_to_f32(qp)[0],
            synth.bf16_bits_to_f32(c), synth.bf16_bits_to_f32(p), Wuk, Wuv, w.scale)


def test_naive_equals_absorbed_v2lite_tiny():
    """Associativity (audit §2.2, §2.3; tutorial §四): equal to 1e-10 in fp64."""
    qn, qp, C, P, Wuk, Wuv, sc = _tiny_inputs()
    a, _, _ = O.absorbed_decode(qn, qp, C, P, Wuk, Wuv, sc)
    b = O.naive_decode(qn, qp, C, P, Wuk, Wuv, sc)
    assert a.shape == (16, 128)
    assert np.max(np.abs(a - b)) <= 1e-10


def test_naive_equals_absorbed_v3_shape():
    w = synth.get_workload("v3_paged")
    wkv = synth.bf16_bits_to_f32(synth.gen_weights(w.H, w.seed))
    Wuk, Wuv = O.split_wkv_b(wkv, w.H)
    n = 96
    qn, qp = synth.gen_queries(w.H, [n], w.seed)
    c, p = synth.gen_sequence(w.seed, 0, n)
    args = (synth.bf16_bits_to_f32(qn)[0], synth.bf16_bits_to_f32(qp)[0],
            synth.bf16_bits_to_f32(c), synth.bf16_bits_to_f32(p), Wuk, Wuv, w.scale)
    a, _, _ = O.absorbed_decode(*args)
    b = O.naive_decode(*args)
    assert np.max(np.abs(a - b)) <= 1e-10


def test_single_token_closed_form():
    """n = 1: the softmax weight is 1, so o_lat = c_0 and out = W_UV c_0."""
    qn, qp, C, P, Wuk, Wuv, sc = _tiny_inputs()
    out, o_lat, lse = O.absorbed_decode(qn, qp, C[:1], P[:1], Wuk, Wuv, sc)
    assert np.array_equal(o_lat, np.broadcast_to(C[0].astype(np.float64), o_lat.shape))
    for h in range(16):
        assert np.allclose(out[h], Wuv[h] @ C[0], atol=1e-13)


def test_zero_query_is_mean():
    """q = 0: all scores equal, so o_lat is the plain mean of the latents."""
    qn, qp, C, P, Wuk, Wuv, sc = _tiny_inputs()
    out, o_lat, lse = O.absorbed_decode(qn * 0, qp * 0, C, P, Wuk, Wuv, sc)
    assert np.allclose(o_lat, C.astype(np.float64).mean(axis=0)[None, :], atol=1e-14)
    assert np.allclose(lse, math.log(C.shape[0]), atol=1e-14)


def test_dominant_rope_token():
    """A RoPE key aligned with every head's q_pe and scaled up selects that token."""
    qn, qp, C, P, Wuk, Wuv, sc = _tiny_inputs()
    H = qp.shape[0]
    qp = np.ones_like(qp)           # identical q_pe for all heads
    P = P.copy()
    j = 7
    P[j] = 1.0e3                    # q_pe . k_pe_j = 64e3, far above every other score
    out, o_lat, _ = O.absorbed_decode(qn, qp, C, P, Wuk, Wuv, sc)
    assert np.allclose(o_lat, np.broadcast_to(C[j], (H, C.shape[1])), atol=1e-12)
    for h in range(H):
        assert np.allclose(out[h], Wuv[h] @ C[j], atol=1e-12)


def test_empty_sequence():
    qn, qp, C, P, Wuk, Wuv, sc = _tiny_inputs()
    out, o_lat, lse = O.absorbed_decode(qn, qp, C[:0], P[:0], Wuk, Wuv, sc)
    assert np.all(out == 0) and np.all(o_lat == 0) and np.all(np.isneginf(lse))


def test_scale_is_inverse_sqrt_192():
    assert synth.get_workload("v3_paged").scale == pytest.approx(1 / math.sqrt(128 + 64))


# ----------------------------------------------------------------------------
# bf16 rounding and quantizers: hand-worked vectors
# ----------------------------------------------------------------------------

def test_bf16_round_hand_values():
    x = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -7, -2.5, 1 + 2 ** -8 + 2 ** -20,
                  3.4e38], dtype=np.float32)   # above the largest finite bf16 (3.3895e38)
    want = np.array([1.0, 1.0, 1 + 2 ** -6, 1 + 2 ** -7, -2.5, 1 + 2 ** -7, np.inf],
                    dtype=np.float32)
    got = O.bf16_round(x)
    assert np.array_equal(got, want)


def test_bf16_bit_patterns_by_hand():
    # sign | 8-bit exponent (bias 127) | 7-bit fraction, the top half of a float32
    bits = np.array([0x3F80, 0xC040, 0x0000, 0x8000, 0x7F80, 0x3F81, 0x0001], dtype=np.uint16)
    vals = np.array([1.0, -3.0, 0.0, -0.0, np.inf, 1 + 2 ** -7, 2.0 ** -133], dtype=np.float32)
    got = O.bf16_from_bits(bits)
    assert np.array_equal(got, vals)
    assert np.array_equal(np.signbit(got), np.signbit(vals))
    assert np.array_equal(O.bf16_to_bits(vals), bits)


def test_int8_hand_vector():
    # amax 127 -> s = 1 exactly; codes = round-half-even of x
    x = np.zeros(32, dtype=np.float32)
    x[:8] = [127, -127, 63.5, 62.5, -0.5, 1.5, 2.5, -3.5]
    codes, s = O.quantize_int8(x, 32)
    assert s.tolist() == [1.0]
    assert codes[:8].tolist() == [127, -127, 64, 62, 0, 2, 2, -4]
    assert np.all(codes[8:] == 0)


def test_int8_scale_rounding():
    # amax 1 -> 1/127 = 0.0078740157..., bf16 -> 0.00787353515625 (mantissa 1.0078125 * 2^-7)
    x = np.zeros(8, dtype=np.float32)
    x[0], x[1] = 1.0, -0.5
    codes, s = O.quantize_int8(x, 8)
    assert s.tolist() == [0.00787353515625]
    assert codes[0] == 127                 # 1/s = 127.007 -> 127
    assert codes[1] == -64                 # -0.5/s = -63.5039 -> -64
    # an all-zero group keeps scale 0 and zero codes
    c0, s0 = O.quantize_int8(np.zeros(8, np.float32), 8)
    assert s0.tolist() == [0.0] and np.all(c0 == 0)


def test_int4_hand_vector():
    # mn = -1, mx = 2: s = bf16(3/15 = 0.2) = 0.2001953125, zero = -1
    x = np.full(32, -1.0, dtype=np.float32)
    x[1], x[2], x[3] = 2.0, 0.0, -0.9
    codes, s, z = O.quantize_int4_asym(x, 32)
    assert s.tolist() == [0.2001953125] and z.tolist() == [-1.0]
    # (2+1)/s = 14.985 -> 15; (0+1)/s = 4.995 -> 5; (0.1)/s = 0.4995 -> 0
    assert codes[:4].tolist() == [0, 15, 5, 0]
    # constant group: s = 0, zero = value, dequantises exactly
    c, s2, z2 = O.quantize_int4_asym(np.full(32, 0.75, np.float32), 32)
    assert s2.tolist() == [0.0] and z2.tolist() == [0.75] and np.all(c == 0)
    assert np.all(O.dequantize_int4(c, s2, z2, 32) == 0.75)


def test_nibble_packing():
    assert O.pack_nibbles(np.array([1, 2, 15, 0], np.uint8)).tolist() == [0x21, 0x0F]


@pytest.mark.parametrize("fmt,group", [("int8", 32), ("int8", 8), ("int4", 32)])
def test_quantizer_error_bound(fmt, group):
    """|x - dequant(x)| <= s/2 (plus the bf16 rounding slack of s itself)."""
    rng = np.random.default_rng(3)
    x = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(
        rng.standard_normal((200, 512)).astype(np.float32) * 3))
    if fmt == "int8":
        c, s = O.quantize_int8(x, group)
        xr = O.dequantize_int8(c, s, group)
    else:
        c, s, z = O.quantize_int4_asym(x, group)
        xr = O.dequantize_int4(c, s, z, group)
    err = np.abs(x.astype(np.float64) - xr).reshape(200, -1, group).max(axis=-1)
    assert np.all(err <= s.astype(np.float64) * 0.5 * (1 + 2 ** -6) + 1e-30)


def test_expected_page_pool_placement():
    """Token t of row b lands in page_table[b][(pos+t)//64], slot (pos+t)%64."""
    rng = np.random.default_rng(0)
    row = np.array([3, 0, 2], np.int32)
    c = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(rng.standard_normal((70, 512)).astype(np.float32)))
    p = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(rng.standard_normal((70, 64)).astype(np.float32)))
    pool = O.expected_page_pool("bf16", 4, [(row, 60, c, p)])
    tok = pool.view(np.uint16).reshape(4, 64, 576)
    assert np.array_equal(tok[3, 60], O.bf16_to_bits(np.concatenate([c[0], p[0]])))
    assert np.array_equal(tok[0, 0], O.bf16_to_bits(np.concatenate([c[4], p[4]])))
    assert np.array_equal(tok[0, 63], O.bf16_to_bits(np.concatenate([c[67], p[67]])))
    assert np.array_equal(tok[2, 1], O.bf16_to_bits(np.concatenate([c[69], p[69]])))
    assert np.all(tok[1] == 0) and np.all(tok[3, :60] == 0)


def test_quant_pool_sections():
    rng = np.random.default_rng(1)
    c = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(rng.standard_normal((2, 512)).astype(np.float32)))
    p = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(rng.standard_normal((2, 64)).astype(np.float32)))
    pool = O.expected_page_pool("int4", 1, [(np.array([0]), 5, c, p)])[0]
    codes, s, z = O.quantize_int4_asym(c, 32)
    assert np.array_equal(pool[5 * 256:6 * 256], O.pack_nibbles(codes[0]))
    off_scale = 64 * 256 + 64 * 64
    got_s = pool[off_scale + 6 * 32: off_scale + 6 * 32 + 32].view(np.uint16)
    assert np.array_equal(got_s, O.bf16_to_bits(s[1]))
    off_zero = off_scale + 64 * 32
    got_z = pool[off_zero + 5 * 32: off_zero + 6 * 32].view(np.uint16)
    assert np.array_equal(got_z, O.bf16_to_bits(z[0]))


def test_int8_pool_sections():
    """INT8 page image, indexed by hand: c codes int8 [64][512] from byte 0,
    k_pe codes int8 [64][64] from 64*512 = 32768, c scales bf16 [64][16] from
    32768 + 64*64 = 36864, k_pe scales bf16 [64][8] from 36864 + 64*16*2 =
    38912; the page ends at 38912 + 64*8*2 = 39936.  Two tokens at slots 5, 6."""
    rng = np.random.default_rng(2)
    c = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(rng.standard_normal((2, 512)).astype(np.float32)))
    p = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(rng.standard_normal((2, 64)).astype(np.float32)))
    pool = O.expected_page_pool("int8", 1, [(np.array([0]), 5, c, p)])[0]
    assert pool.size == 39936
    cc, cs = O.quantize_int8(c, 32)
    pc, ps = O.quantize_int8(p, 8)
    for k, slot in enumerate((5, 6)):
        assert np.array_equal(pool[slot * 512:(slot + 1) * 512].view(np.int8), cc[k])
        assert np.array_equal(pool[32768 + slot * 64:32768 + (slot + 1) * 64].view(np.int8), pc[k])
        assert np.array_equal(pool[36864 + slot * 32:36864 + (slot + 1) * 32].view(np.uint16), O.bf16_to_bits(cs[k]))
        assert np.array_equal(pool[38912 + slot * 16:38912 + (slot + 1) * 16].view(np.uint16), O.bf16_to_bits(ps[k]))
    # every other byte of the page is untouched
    mask = np.zeros(pool.size, bool)
    for slot in (5, 6):
        for off, per in ((0, 512), (32768, 64), (36864, 32), (38912, 16)):
            mask[off + slot * per:off + (slot + 1) * per] = True
    assert not pool[~mask].any()


def test_random_roundtrip_rope_norm():
    """Generator sanity (not oracle): RoPE keeps pair norms, c_KV rows have unit RMS."""
    c, p = synth.gen_sequence(0, 0, 30)
    cf = synth.bf16_bits_to_f32(c).astype(np.float64)
    assert np.allclose(np.sqrt(np.mean(cf ** 2, axis=1)), 1.0, atol=5e-3)
    x = np.random.default_rng(0).standard_normal((3, 64))
    y = synth.rope_interleaved(x, np.array([0.0, 5.0, 77.0]))
    assert np.allclose(x[0], y[0])
    assert np.allclose(np.hypot(x[:, 0::2], x[:, 1::2]), np.hypot(y[:, 0::2], y[:, 1::2]))
    random.seed(0)


# ----------------------------------------------------------------------------
# the cache payload producer: c_kv = rmsnorm(x W_DKV^T, W_KVN), k_pe = rope(x W_KR^T)
# ("手搓 MLA" §三; weight names "DeepSeek MLA 吸收式缓存" §3.3)
# ----------------------------------------------------------------------------

def test_rms_norm_hand_values():
    """[1, 2, 3, 4]: mean square 30/4 = 7.5, so each entry is divided by sqrt(7.5)
    = 2.7386127875258306; then the gain multiplies elementwise."""
    out = O.rms_norm(np.array([1.0, 2.0, 3.0, 4.0]), np.array([1.0, 1.0, 2.0, -1.0]), 0.0)
    want = [0.3651483716701107, 0.7302967433402214, 2.1908902300206643, -1.4605934866804429]
    assert np.allclose(out, want, rtol=0, atol=1e-15)
    # a constant vector normalises to the gain itself; eps enters under the root
    g = np.linspace(0.5, 1.5, 512)
    assert np.allclose(O.rms_norm(np.full(512, -3.0), g, 0.0), -g, atol=1e-15)
    assert O.rms_norm(np.full(4, 2.0), np.ones(4), 12.0)[0] == pytest.approx(2.0 / 4.0, abs=1e-15)


def test_rms_norm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(3)
    v = rng.standard_normal((5, 512)) * 7.0
    out = O.rms_norm(v, np.ones(512), 0.0)
    assert np.allclose(np.sqrt(np.mean(out ** 2, axis=1)), 1.0, atol=1e-14)
    assert np.allclose(O.rms_norm(v * 1e-3, np.ones(512), 0.0), out, atol=1e-12)
    # the normalisation is per row: a row scaled alone does not move the others
    v2 = v.copy()
    v2[2] *= 50.0
    assert np.allclose(O.rms_norm(v2, np.ones(512), 0.0), out, atol=1e-12)


def test_rope_position_zero_and_one_radian():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 64))
    assert np.array_equal(O.rope(x, np.zeros(3)), x)
    # pair 0 turns by exactly pos radians (theta^0 = 1): (1, 0) at pos 1 -> (cos 1, sin 1)
    e0 = np.zeros(64)
    e0[0] = 1.0
    r = O.rope(e0, 1)
    assert r[0] == pytest.approx(0.5403023058681398, abs=1e-15)
    assert r[1] == pytest.approx(0.8414709848078965, abs=1e-15)
    assert np.all(r[2:] == 0.0)
    # pair 1 (dims 2, 3) turns by 10000^(-2/64) = 0.7498942093324559 radians per position:
    # (0, 1) at pos 2 -> (-sin 1.4997884186649117, cos 1.4997884186649117)
    e3 = np.zeros(64)
    e3[3] = 1.0
    r = O.rope(e3, 2)
    assert r[2] == pytest.approx(-math.sin(1.4997884186649117), abs=1e-14)
    assert r[3] == pytest.approx(math.cos(1.4997884186649117), abs=1e-14)
    assert np.all(np.delete(r, [2, 3]) == 0.0)
    # the last pair (dims 62, 63) turns by 10000^(-62/64) = 1.333521432163324e-4 per position
    e62 = np.zeros(64)
    e62[62] = 1.0
    r = O.rope(e62, 1000)
    assert r[62] == pytest.approx(math.cos(0.1333521432163324), abs=1e-14)
    assert r[63] == pytest.approx(math.sin(0.1333521432163324), abs=1e-14)


def test_rope_relative_position_and_norm():
    """The defining property: <rope(q, m), rope(k, n)> depends on m - n only; each
    pair keeps its length; rotations by a and then b compose to a + b."""
    rng = np.random.default_rng(6)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    d1 = np.dot(O.rope(q, 37), O.rope(k, 5))
    d2 = np.dot(O.rope(q, 1032), O.rope(k, 1000))
    assert d1 == pytest.approx(d2, abs=1e-9)
    assert d1 != pytest.approx(np.dot(O.rope(q, 38), O.rope(k, 5)), abs=1e-3)
    x = rng.standard_normal(64)
    r = O.rope(x, 12345)
    assert np.allclose(np.hypot(r[0::2], r[1::2]), np.hypot(x[0::2], x[1::2]), atol=1e-12)
    assert np.allclose(O.rope(O.rope(x, 300), 45), O.rope(x, 345), atol=1e-10)


def _project_bruteforce(x, w, g, pos, eps, theta, dc):
    """Explicit loops, math.fsum: the projection, RMSNorm and RoPE as written."""
    out_c, out_p = [], []
    for t, row in enumerate(x):
        y = [math.fsum(row[k] * w[j][k] for k in range(len(row))) for j in range(len(w))]
        lat, rot = y[:dc], y[dc:]
        inv = 1.0 / math.sqrt(math.fsum(v * v for v in lat) / dc + eps)
        out_c.append([lat[j] * inv * g[j] for j in range(dc)])
        d = len(rot)
        pr = []
        for i in range(d // 2):
            ang = pos[t] * theta ** (-2.0 * i / d)
            a, b = rot[2 * i], rot[2 * i + 1]
            pr += [a * math.cos(ang) - b * math.sin(ang), a * math.sin(ang) + b * math.cos(ang)]
        out_p.append(pr)
    return np.array(out_c), np.array(out_p)


@pytest.mark.parametrize("n", [1, 3])
def test_project_latent_bruteforce_odd_dims(n):
    """Odd, unequal dims (hidden 5, latent 3, RoPE key 4): a transposed weight, the
    latent/key row split taken the other way round or the norm over the wrong
    axis fails."""
    rng = np.random.default_rng(20 + n)
    hidden, dc, dr = 5, 3, 4
    x = rng.standard_normal((n, hidden))
    w = rng.standard_normal((dc + dr, hidden))
    g = rng.standard_normal(dc)
    pos = np.arange(7, 7 + n)
    c, p = O.project_latent(x, w, g, pos, eps=0.25, theta=100.0)
    bc, bp = _project_bruteforce(x.tolist(), w.tolist(), g.tolist(), pos.tolist(), 0.25, 100.0, dc)
    assert c.shape == (n, dc) and p.shape == (n, dr)
    assert np.max(np.abs(c - bc)) < 1e-12
    assert np.max(np.abs(p - bp)) < 1e-12


# ----------------------------------------------------------------------------
# several query tokens per row, causal ("DeepSeek MLA 吸收式缓存" §3.4 prefill +
# incremental decode; the t axis of the "手搓 MLA" §四 einsums)
# ----------------------------------------------------------------------------

def _bruteforce_causal(q_nope, q_pe, C, Kpe, Wuk, Wuv, scale, q_pos):
    """Explicit loops: for each query token and head, expand the visible keys and
    values, exponentiate, normalise with math.fsum, sum."""
    T, H = len(q_nope), len(q_nope[0])
    dn, dc, dv = len(Wuk[0]), len(C[0]), len(Wuv[0])
    out = []
    for t in range(T):
        rows = []
        for h in range(H):
            s = []
            for j in range(q_pos[t] + 1):
                k = [math.fsum(Wuk[h][d][c] * C[j][c] for c in range(dc)) for d in range(dn)] + list(Kpe[j])
                q = list(q_nope[t][h]) + list(q_pe[t][h])
                s.append(scale * math.fsum(a * b for a, b in zip(q, k)))
            m = max(s)
            e = [math.exp(x - m) for x in s]
            z = math.fsum(e)
            v = [[math.fsum(Wuv[h][d][c] * C[j][c] for c in range(dc)) for d in range(dv)] for j in range(len(s))]
            rows.append([math.fsum(e[j] / z * v[j][d] for j in range(len(s))) for d in range(dv)])
        out.append(rows)
    return np.array(out)


@pytest.mark.parametrize("q_pos", [[2, 3, 4], [0, 1, 2], [4, 1, 3]])
def test_causal_bruteforce_tiny_odd_dims(q_pos):
    """T = 3 queries over n = 5 tokens, odd unequal dims; the last positions, a
    full prefill of the first three tokens, and an unordered set of positions."""
    rng = np.random.default_rng(40)
    T, H, dn, dr, dc, dv, n = 3, 2, 3, 2, 7, 5, 5
    qn, qp = rng.standard_normal((T, H, dn)), rng.standard_normal((T, H, dr))
    C, Kpe = rng.standard_normal((n, dc)), rng.standard_normal((n, dr))
    Wuk, Wuv = rng.standard_normal((H, dn, dc)), rng.standard_normal((H, dv, dc))
    ref = _bruteforce_causal(qn.tolist(), qp.tolist(), C.tolist(), Kpe.tolist(), Wuk.tolist(), Wuv.tolist(), 0.41,
                             q_pos)
    naive = O.naive_attend_causal(qn, qp, C, Kpe, Wuk, Wuv, 0.41, q_pos)
    absorbed, _ = O.absorbed_attend_causal(qn, qp, C, Kpe, Wuk, Wuv, 0.41, q_pos)
    assert np.max(np.abs(naive - ref)) < 1e-12
    assert np.max(np.abs(absorbed - ref)) < 1e-12


def test_causal_first_prefill_token_sees_only_itself():
    """Full prefill (T = n): query 0 sees token 0 alone, so its latent sum is c_0
    and its output W_UV c_0 for every head, whatever the scores."""
    rng = np.random.default_rng(41)
    T = n = 6
    H, dc = 3, 8
    qn, qp = rng.standard_normal((T, H, 4)) * 30, rng.standard_normal((T, H, 2)) * 30
    C, Kpe = rng.standard_normal((n, dc)), rng.standard_normal((n, 2))
    Wuk, Wuv = rng.standard_normal((H, 4, dc)), rng.standard_normal((H, 5, dc))
    out, o_lat = O.absorbed_attend_causal(qn, qp, C, Kpe, Wuk, Wuv, 0.3, np.arange(n))
    assert np.allclose(o_lat[0], np.broadcast_to(C[0], (H, dc)), atol=1e-14)
    assert np.allclose(out[0], Wuv @ C[0], atol=1e-12)


def test_causal_v2lite_prefill_and_decode_agree():
    """The 26-token V2-Lite case run as [audit] §3.4 runs it: a 25-token causal
    prefill, then the 26th token as an incremental decode.  Naive and absorbed
    agree to 1e-10 (associativity); the prefill's last query sees the same 25
    tokens as a decode over the first 25, and the decode token as a decode
    over all 26."""
    qn1, qp1, C, P, Wuk, Wuv, sc = _tiny_inputs()
    rng = np.random.default_rng(42)
    T, H = 25, qn1.shape[0]
    qn = np.concatenate([rng.standard_normal((T, H, 128)), qn1[None]], axis=0)
    qp = np.concatenate([rng.standard_normal((T, H, 64)), qp1[None]], axis=0)
    a, _ = O.absorbed_attend_causal(qn, qp, C, P, Wuk, Wuv, sc)   # positions 0..25
    nv = O.naive_attend_causal(qn, qp, C, P, Wuk, Wuv, sc)
    assert np.max(np.abs(a - nv)) < 1e-10
    last_prefill, _, _ = O.absorbed_decode(qn[24], qp[24], C[:25], P[:25], Wuk, Wuv, sc)
    assert np.max(np.abs(a[24] - last_prefill)) < 1e-12
    decode, _, _ = O.absorbed_decode(qn[25], qp[25], C, P, Wuk, Wuv, sc)
    assert np.max(np.abs(a[25] - decode)) < 1e-12


# ----------------------------------------------------------------------------
# the layer output projection and the other quantizers of [report] §3.2
# ----------------------------------------------------------------------------

def test_output_projection_picks_head_and_dim():
    """A one-hot Wo row reads one (head, dim) of the side-by-side head outputs:
    the reshape is head-major ([T, H*dv], head h at columns h*dv .. h*dv+dv-1)."""
    rng = np.random.default_rng(50)
    T, H, dv = 2, 3, 4
    out = rng.standard_normal((T, H, dv))
    wo = np.zeros((2, H * dv))
    wo[0, 1 * dv + 2] = 1.0      # head 1, dim 2
    wo[1, 2 * dv + 0] = -2.0     # head 2, dim 0
    y = O.output_projection(out, wo)
    assert np.array_equal(y[:, 0], out[:, 1, 2])
    assert np.array_equal(y[:, 1], -2.0 * out[:, 2, 0])


def test_output_projection_bruteforce():
    rng = np.random.default_rng(51)
    T, H, dv, hidden = 2, 3, 5, 7
    out = rng.standard_normal((T, H, dv))
    wo = rng.standard_normal((hidden, H * dv))
    y = O.output_projection(out, wo)
    for t in range(T):
        for j in range(hidden):
            want = math.fsum(wo[j][h * dv + d] * out[t][h][d] for h in range(H) for d in range(dv))
            assert y[t, j] == pytest.approx(want, abs=1e-12)


def test_int4_sym_hand_vector():
    """amax 7 gives s = 1 exactly; -3.5, 0.5, 1.5 and 2.5 are ties, rounded to even."""
    x = np.array([[7.0, -3.5, 0.5, 1.5, -7.0, 2.5, 0.0, 3.0]], dtype=np.float32)
    codes, s = O.quantize_int4_sym(x, 8)
    assert s.tolist() == [[1.0]]
    assert codes.tolist() == [[7, -4, 0, 2, -7, 2, 0, 3]]
    # amax 1: s = bf16(1/7) = 146/128 * 2^-3 = 0.142578125, and 1/s = 7.01 rounds to 7
    codes, s = O.quantize_int4_sym(np.array([1.0, -0.5] + [0.0] * 6, dtype=np.float32), 8)
    assert s.tolist() == [0.142578125]
    assert codes.tolist() == [7, -4, 0, 0, 0, 0, 0, 0]   # -0.5/s = -3.51 -> -4
    codes, s = O.quantize_int4_sym(np.zeros(8, dtype=np.float32), 8)
    assert s.tolist() == [0.0] and not codes.any()


def test_int8_per_token_and_per_tensor_hand_vectors():
    # per token: amax 254 gives s = 2; 63.5 / 2 = 31.75 -> 32, -63.5 / 2 -> -32, 0.5 / 2 -> 0
    codes, s = O.quantize_int8_per_token(np.array([[63.5, -63.5, 0.5, 254.0], [1.0, 0.0, 0.0, 0.0]],
                                                  dtype=np.float32))
    assert s.tolist() == [[2.0], [0.00787353515625]]  # bf16(1/127) = 129/128 * 2^-7
    assert codes.tolist() == [[32, -32, 0, 127], [127, 0, 0, 0]]
    # per tensor: amax 4 gives s = bf16(4/127) = 129/128 * 2^-5 = 0.031494140625
    codes, s = O.quantize_int8_per_tensor(np.array([[1.0, -2.0], [0.5, 4.0]], dtype=np.float32))
    assert float(s) == 0.031494140625
    assert codes.tolist() == [[32, -64], [16, 127]]   # 31.75, -63.50, 15.88, 127.01


@pytest.mark.parametrize("kind", ["int4_sym_32", "int4_sym_8", "int8_token", "int8_tensor"])
def test_quantizer_variants_error_bound(kind):
    """|x - x^| <= s/2 for every element (no clamping occurs at these scales)."""
    rng = np.random.default_rng(52)
    x = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(rng.standard_normal((16, 512)).astype(np.float32) * 3))
    if kind.startswith("int4_sym"):
        g = int(kind.rsplit("_", 1)[1])
        codes, s = O.quantize_int4_sym(x, g)
        xh = O.dequantize_int4_sym(codes, s, g)
        bound = np.repeat(np.asarray(s, np.float64), g, axis=-1) / 2
        assert np.abs(codes).max() <= 7
    elif kind == "int8_token":
        codes, s = O.quantize_int8_per_token(x)
        xh = O.dequantize_int8(codes, s, 512)
        bound = np.repeat(np.asarray(s, np.float64), 512, axis=-1) / 2
    else:
        codes, s = O.quantize_int8_per_tensor(x)
        xh = codes.astype(np.float64) * float(s)
        bound = float(s) / 2
    assert np.all(np.abs(x - xh) <= bound * (1 + 1e-12))


def _variant_errors(c):
    """Relative RMS error ||x - x^|| / ||x|| of each c_KV quantizer on latents c [n, 512]."""
    def rel(xh):
        return float(np.linalg.norm(c - xh) / np.linalg.norm(c))
    codes, s = O.quantize_int8(c, 32)
    e = {"int8_channel32": rel(O.dequantize_int8(codes, s, 32))}
    codes, s = O.quantize_int8_per_token(c)
    e["int8_token"] = rel(O.dequantize_int8(codes, s, 512))
    codes, s = O.quantize_int8_per_tensor(c)
    e["int8_tensor"] = rel(codes.astype(np.float64) * float(s))
    codes, s, z = O.quantize_int4_asym(c, 32)
    e["int4_asym32"] = rel(O.dequantize_int4(codes, s, z, 32))
    codes, s = O.quantize_int4_sym(c, 32)
    e["int4_sym32"] = rel(O.dequantize_int4_sym(codes, s, 32))
    return e


def test_quantizer_variants_order_on_outlier_latents():
    """On the quantized workload's latents (N(0,1) with 1 % of the channels x8) the
    variants order as [report] §3.2 finds on real weights: 32-channel INT8 beats
    per-token INT8, which beats per-tensor INT8 (an outlier channel widens every
    scale it shares); asymmetric INT4 beats symmetric INT4 (16 levels over
    [min, max] instead of 15 over [-amax, amax]).  The page's error metric is not
    stated, so its figures are not reproduced (parity unpinned); this checks the
    ordering only."""
    c, _ = synth.gen_sequence(4, 0, 256, "outlier")
    e = _variant_errors(synth.bf16_bits_to_f32(c).astype(np.float32))
    assert e["int8_channel32"] < e["int8_token"] < e["int8_tensor"]
    assert e["int4_asym32"] < e["int4_sym32"]
    assert e["int8_channel32"] < e["int4_asym32"]


# ----------------------------------------------------------------------------
# the seeded input generators both sides take their inputs from (not oracle pins)
# ----------------------------------------------------------------------------

def test_generator_draws_in_pieces_equal_whole():
    """A sequence drawn as a 25-token prefill then one decode token equals the
    26-token draw, bit for bit; the same seed gives the same bits again."""
    c, p = synth.gen_sequence(0, 3, 26)
    c1, p1 = synth.gen_sequence(0, 3, 25)
    c2, p2 = synth.gen_sequence(0, 3, 1, start=25)
    assert np.array_equal(c, np.concatenate([c1, c2])) and np.array_equal(p, np.concatenate([p1, p2]))
    c3, _ = synth.gen_sequence(0, 3, 26)
    assert np.array_equal(c, c3)
    x = synth.gen_hidden(2048, 1, 2, 5)
    assert np.array_equal(x, synth.gen_hidden(2048, 1, 2, 5)) and x.shape == (5, 2048)


def test_generator_page_tables_and_lengths():
    """Each physical page belongs to exactly one (row, logical page); rows get the
    pages their lengths need; ragged lengths stay in the stated clip range."""
    w = synth.get_workload("v3_ragged")
    lens = synth.gen_seqlens(w)
    assert lens.min() >= 256 and lens.max() <= 32768 and len(lens) == w.B
    table, num_pages = synth.make_page_table(lens, w.seed, True, spare_pages=2)
    need = (lens.astype(np.int64) + 63) // 64
    used = np.concatenate([table[b, :need[b]] for b in range(len(lens))])
    assert len(used) == need.sum() and len(np.unique(used)) == len(used)
    assert used.min() >= 0 and used.max() < num_pages and num_pages == need.sum() + 2
    assert all(np.all(table[b, need[b]:] == -1) for b in range(len(lens)))
    ident, _ = synth.make_page_table([70, 10], 0, False)
    assert ident.tolist() == [[0, 1], [2, -1]]


def test_variant_pool_sections():
    """The per-token INT8, symmetric INT4 and 4-bit RoPE-key quantizers in their page images,
    indexed by hand: per-token INT8 keeps the INT8 layout with the token's one
    scale s = bf16(amax / 127) in all 16 group-scale slots; symmetric INT4 keeps
    the INT4 layout with nibbles q + 8 and zero = -8 s, so that code * s + zero
    equals q * s (the symmetric dequantization)."""
    rng = np.random.default_rng(3)
    c = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(rng.standard_normal((1, 512)).astype(np.float32) * 2))
    p = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(rng.standard_normal((1, 64)).astype(np.float32)))
    # per-token INT8, slot 9
    pool = O.expected_page_pool("int8_token", 1, [(np.array([0]), 9, c, p)])[0]
    s_tok = float(np.asarray(O.bf16_round(np.max(np.abs(c)) / np.float32(127.0))).reshape(-1)[0])
    scales = pool[36864 + 9 * 32:36864 + 10 * 32].view(np.uint16)
    assert np.all(scales == O.bf16_to_bits(np.float32(s_tok)))
    codes = pool[9 * 512:10 * 512].view(np.int8).astype(np.float64)
    assert np.all(np.abs(codes) <= 127) and np.max(np.abs(codes)) == 127
    assert np.allclose(codes * float(s_tok), O.dequantized_tokens("int8_token", c, p)[0][0], rtol=0, atol=0)
    # symmetric INT4, slot 3
    pool = O.expected_page_pool("int4_sym", 1, [(np.array([0]), 3, c, p)])[0]
    q, s = O.quantize_int4_sym(c, 32)
    nib = pool[3 * 256:4 * 256]
    lo, hi = (nib & 0xF).astype(np.int16), (nib >> 4).astype(np.int16)
    assert np.array_equal(lo - 8, q[0, 0::2]) and np.array_equal(hi - 8, q[0, 1::2])
    sc = synth.bf16_bits_to_f32(pool[20480 + 3 * 32:20480 + 4 * 32].view(np.uint16))
    zr = synth.bf16_bits_to_f32(pool[22528 + 3 * 32:22528 + 4 * 32].view(np.uint16))
    assert np.array_equal(sc, s[0]) and np.array_equal(zr, -8 * s[0])
    codes = np.empty(512)
    codes[0::2], codes[1::2] = lo, hi
    g = np.repeat(np.arange(16), 32)
    assert np.array_equal(codes * sc[g].astype(np.float64) + zr[g], q[0] * s[0][g].astype(np.float64))
    assert np.array_equal(O.dequantized_tokens("int4_sym", c, p)[0][0], q[0] * s[0][g].astype(np.float64))
    # 4-bit RoPE key (symmetric INT4 in 8-dim groups) in the INT4 layout, slot 5: the
    # latent sections are those of the plain INT4 image, the k_pe codes are -7..7 in
    # the INT8 k_pe section with s = bf16(amax / 7) in the k_pe scale slots
    pool4 = O.expected_page_pool("int4", 1, [(np.array([0]), 5, c, p)])[0]
    pool = O.expected_page_pool("int4_pe4", 1, [(np.array([0]), 5, c, p)])[0]
    assert np.array_equal(pool[:16384], pool4[:16384])                    # c codes
    assert np.array_equal(pool[20480:24576], pool4[20480:24576])          # c scales and zeros
    kq = pool[16384 + 5 * 64:16384 + 6 * 64].view(np.int8)
    ks = synth.bf16_bits_to_f32(pool[24576 + 5 * 16:24576 + 6 * 16].view(np.uint16))
    amax = np.max(np.abs(p[0].reshape(8, 8)), axis=1)
    assert np.array_equal(ks, O.bf16_round(amax / np.float32(7.0)))
    assert np.all(np.abs(kq) <= 7) and np.max(np.abs(kq)) == 7
    assert np.all(np.abs(kq.astype(np.float64) * np.repeat(ks, 8) - p[0]) <= np.repeat(ks, 8) / 2 + 1e-12)
    assert np.array_equal(O.dequantized_tokens("int4_pe4", c, p)[1][0], kq * np.repeat(ks, 8).astype(np.float64))
    assert np.array_equal(O.dequantized_tokens("int4_pe4", c, p)[0], O.dequantized_tokens("int4", c, p)[0])
