"""GPU parity of the fused cache producer (mla_cache_project_append) against the
fp64 oracle ("手搓 MLA" §三: c_kv = rmsnorm(x W_DKV^T, W_KVN), k_pe =
rope(x W_KR^T); weight names "DeepSeek MLA 吸收式缓存" §3.3).

Tolerance of the produced payload: the kernel rounds each value once to bf16
(at most 2^-9 relative) after fp32 accumulation (relative error of order 1e-6
at these depths), so |got - ref| <= 2^-8 |ref| + 1e-4 elementwise and a
relative RMS error <= 2^-8 per token.  Page placement and the quantized codes
and scales are bit-exact: they are checked against the oracle's page image
built from the bf16 payload the same call returned (latent_out), so both sides
take the quantization decisions on the same bf16 values.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")]

import oracle as O  # noqa: E402
import synth  # noqa: E402
from synth.device import bits_to_device  # noqa: E402
from tests.parity import assert_close  # noqa: E402

RTOL = 2.0 ** -8
ATOL = 1e-4
EPS = 1e-6
THETA = 10000.0


def _np_bf16(t):
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def _status():
    import mla_absorbed_latent_gb300 as mla
    return mla.mla_get_device_status()


class Produced:
    """x, wkv_a and kv_norm of B rows x T new tokens at positions pos0[b] + t,
    a zeroed page pool covering every row's positions, and one producer call."""

    def __init__(self, hidden, B, T, pos0, seed, fmt="bf16", paged=True):
        import mla_absorbed_latent_gb300 as mla
        self.mla, self.hidden, self.B, self.T, self.fmt = mla, hidden, B, T, fmt
        self.pos0 = np.asarray(pos0, dtype=np.int32)
        w, g = synth.gen_project_weights(hidden, seed)
        self.w_bits, self.g_bits = w, g
        self.x_bits = np.stack([synth.gen_hidden(hidden, seed, b, T) for b in range(B)])  # [B, T, hidden]
        self.page_table, self.num_pages = synth.make_page_table(self.pos0 + T, seed, paged)
        self.pool = torch.zeros(self.num_pages * mla.mla_cache_page_bytes(fmt), dtype=torch.uint8, device="cuda")
        self.cache = mla.cache_struct(fmt, self.num_pages, self.pool)
        self.x = bits_to_device(self.x_bits)
        self.w = bits_to_device(w)
        self.g = bits_to_device(g)
        self.pt = torch.from_numpy(self.page_table).cuda()
        self.pos = torch.from_numpy(self.pos0).cuda()
        self.latent = torch.full((B, T, 576), float("nan"), dtype=torch.bfloat16, device="cuda")

    def run(self, k_splits=0, pos=None):
        m = self.mla
        nbytes = m.mla_cache_project_workspace_bytes(self.B, self.T, self.hidden, k_splits)
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")
        m.mla_cache_project_append(self.cache, self.x, self.hidden, self.w, self.g, EPS, THETA, self.pt,
                                   self.page_table.shape[1], self.pos if pos is None else pos, self.B, self.T,
                                   self.latent, k_splits, ws, nbytes)
        torch.cuda.synchronize()
        return nbytes

    def latent_f32(self):
        return synth.bf16_bits_to_f32(_np_bf16(self.latent))  # [B, T, 576]

    def oracle(self, b, tokens=None):
        """fp64 (c_kv, k_pe) of row b at the listed token indices (all by default)."""
        t = np.arange(self.T) if tokens is None else np.asarray(tokens)
        x = synth.bf16_bits_to_f32(self.x_bits[b][t])
        return O.project_latent(x, synth.bf16_bits_to_f32(self.w_bits), synth.bf16_bits_to_f32(self.g_bits),
                                self.pos0[b] + t, EPS, THETA)

    def expected_pool(self):
        lat = self.latent_f32()
        writes = [(self.page_table[b], int(self.pos0[b]), lat[b, :, :512], lat[b, :, 512:]) for b in range(self.B)]
        return O.expected_page_pool(self.fmt, self.num_pages, writes)

    def pool_bytes(self):
        return self.pool.cpu().numpy().reshape(self.num_pages, -1)


def _check_payload(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref)
    bad = err > RTOL * np.abs(ref) + ATOL
    assert not bad.any(), f"{bad.sum()} values out of tolerance, max err {err.max():.3e}"
    rel = np.linalg.norm(got - ref, axis=-1) / np.linalg.norm(ref, axis=-1)
    assert rel.max() <= RTOL, f"worst token rel-RMS {rel.max():.3e}"


def _check_rows(p, rows=None, tokens=None):
    lat = p.latent_f32()
    for b in (range(p.B) if rows is None else rows):
        c, k = p.oracle(b, tokens)
        t = slice(None) if tokens is None else np.asarray(tokens)
        _check_payload(lat[b, t, :512], c)
        _check_payload(lat[b, t, 512:], k)


@pytest.mark.parametrize("k_splits", [1, 0, 5])
def test_project_bf16_v2lite_rows_mid_page(k_splits):
    """V2-Lite width (hidden 2048), three rows whose 45 new tokens start mid-page
    and cross pages (two 128-token tiles, a ragged tail); one pair per tile, the
    automatic split and a forced split of the hidden dimension."""
    p = Produced(2048, B=3, T=45, pos0=[0, 10, 70], seed=31)
    p.run(k_splits)
    assert _status() == (0, 0)
    _check_rows(p)
    assert np.array_equal(p.pool_bytes(), p.expected_pool())


@pytest.mark.parametrize("fmt", ["int8", "int4"])
def test_project_quantized_pool_bitexact(fmt):
    """The quantized page image equals the oracle's quantizer applied to the bf16
    payload of the same call; the payload itself is within tolerance."""
    p = Produced(2048, B=2, T=70, pos0=[5, 64], seed=32, fmt=fmt)
    p.run()
    assert _status() == (0, 0)
    _check_rows(p)
    assert np.array_equal(p.pool_bytes(), p.expected_pool())


def test_project_v3_decode_shape():
    """DeepSeek-V3 width (hidden 7168), one new token for each of 64 rows at seeded
    positions up to 8191 (the decode-time append: one tile, K split over pairs,
    the pairs' partials summed in split order: bit-identical on a second call)."""
    pos0 = np.random.default_rng(33).integers(0, 8192, size=64).astype(np.int32)
    p = Produced(7168, B=64, T=1, pos0=pos0, seed=33)
    nbytes = p.run()
    assert nbytes > 0  # few tokens: the hidden dimension is split
    assert _status() == (0, 0)
    _check_rows(p)
    assert np.array_equal(p.pool_bytes(), p.expected_pool())
    first = _np_bf16(p.latent).copy()
    p.run()
    assert np.array_equal(_np_bf16(p.latent), first)


@pytest.mark.parametrize("hidden,fmt,B,T", [(64, "bf16", 1, 1), (2048, "int8", 5, 7), (2048, "int4", 5, 7),
                                             (7168, "bf16", 3, 21), (65536, "bf16", 1, 3)])
def test_project_few_tokens(hidden, fmt, B, T):
    """At most 64 tokens with the automatic split: the warp-level MMA producer
    (the hidden dimension in slices of at most 512, the 576 columns in groups of
    64, token rows past the last one read as zeros).  Payload against the oracle,
    page image bit-exact, and within one bf16 ulp of the forced tcgen05 path."""
    p = Produced(hidden, B=B, T=T, pos0=[3 + 61 * b for b in range(B)], seed=35 + hidden % 7)
    assert p.run() > 0
    assert _status() == (0, 0)
    _check_rows(p)
    assert np.array_equal(p.pool_bytes(), p.expected_pool())
    small = p.latent_f32().astype(np.float64)
    p.run(k_splits=1)
    assert _status() == (0, 0)
    # two bf16 roundings of (nearly) the same fp32 value: at most one ulp apart
    other = p.latent_f32().astype(np.float64)
    assert np.all(np.abs(small - other) <= 2.0 ** -7 * np.abs(other) + 2 * ATOL)


@pytest.mark.parametrize("k_splits", [0, 1, 3])
def test_project_far_positions(k_splits):
    """Positions near 2^20, 2^22 and 2^24 (rotation angles of up to 1.7e7 rad on
    the fastest pair): the angle is reduced to one turn in 64-bit fixed point,
    so the RoPE key stays within tolerance of the fp64 oracle.  The few-token
    kernel with its finishing kernel, the tcgen05 kernel's own epilogue, and the
    tcgen05 kernel split three ways with the finishing kernel."""
    far = np.array([(1 << 20) - 1, (1 << 20) + 12345, 3 * (1 << 22) + 7, (1 << 24) - 1], dtype=np.int32)
    p = Produced(2048, B=4, T=1, pos0=[0, 0, 0, 0], seed=36)
    max_pages = (1 << 24) // 64
    table = np.repeat(p.page_table[:, :1], max_pages, axis=1).astype(np.int32)  # every page: the row's own
    p.page_table, p.pos0 = np.ascontiguousarray(table), far
    p.pt = torch.from_numpy(p.page_table).cuda()
    p.pos = torch.from_numpy(far).cuda()
    p.run(k_splits)
    assert _status() == (0, 0)
    _check_rows(p)
    assert np.array_equal(p.pool_bytes(), p.expected_pool())


def test_project_v3_prefill_many_tiles():
    """V3 width, 4 rows x 2500 tokens (79 tiles, enough for one pair per tile:
    no K split, deterministic): sampled tokens of every row against the oracle,
    including the last tile's ragged tail; the whole pool against the payload."""
    p = Produced(7168, B=4, T=2500, pos0=[0, 1, 64, 4000], seed=34)
    nbytes = p.run()
    assert nbytes == 0
    assert _status() == (0, 0)
    tokens = np.unique(np.concatenate([np.random.default_rng(34).integers(0, 2500, size=40), [0, 127, 128, 2499]]))
    _check_rows(p, tokens=tokens)
    assert np.array_equal(p.pool_bytes(), p.expected_pool())
    first = _np_bf16(p.latent).copy()
    p.run()
    assert np.array_equal(_np_bf16(p.latent), first)  # no K split: bit-identical on a second call


def test_project_bad_position_is_reported_not_written():
    import mla_absorbed_latent_gb300 as mla
    p = Produced(2048, B=2, T=3, pos0=[0, 0], seed=35)
    bad = torch.tensor([0, 64 * p.page_table.shape[1]], dtype=torch.int32, device="cuda")  # row 1 past its pages
    p.run(pos=bad)
    st, info = _status()
    assert st == mla.MLA_ERR_BOUNDS and info == 1
    lat = p.latent_f32()
    assert np.all(np.isfinite(lat))  # the payload is still produced for every token
    pool = p.pool_bytes()
    want = O.expected_page_pool("bf16", p.num_pages, [(p.page_table[0], 0, lat[0, :, :512], lat[0, :, 512:])])
    assert np.array_equal(pool, want)  # row 0 written, nothing of row 1
    assert _status() == (0, 0)


def test_project_then_decode():
    """A cache filled by the producer decodes like the oracle over the same
    payload (V2-Lite heads over two rows)."""
    import mla_absorbed_latent_gb300 as mla
    H, T, seed = 16, 200, 36
    p = Produced(2048, B=2, T=T, pos0=[0, 0], seed=seed)
    p.run()
    assert _status() == (0, 0)
    seqlens = np.array([T, T], dtype=np.int32)
    wkv = synth.gen_weights(H, seed)
    q_nope, q_pe = synth.gen_queries(H, seqlens, seed)
    W_UK = torch.empty((H, 512, 128), dtype=torch.bfloat16, device="cuda")
    W_UV = torch.empty((H, 128, 512), dtype=torch.bfloat16, device="cuda")
    mla.mla_absorb_weights(bits_to_device(wkv), H, W_UK, W_UV)
    ws_bytes = mla.mla_decode_workspace_bytes(2, H)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.empty((2, H, 128), dtype=torch.bfloat16, device="cuda")
    scale = 1.0 / 192 ** 0.5
    mla.mla_decode(bits_to_device(q_nope), bits_to_device(q_pe), W_UK, W_UV, H, p.cache, p.pt,
                   p.page_table.shape[1], torch.from_numpy(seqlens).cuda(), 2, scale, ws, ws_bytes, out)
    torch.cuda.synchronize()
    assert _status() == (0, 0)
    Wuk, Wuv = O.split_wkv_b(synth.bf16_bits_to_f32(wkv), H)
    lat = p.latent_f32()
    got = synth.bf16_bits_to_f32(_np_bf16(out)).astype(np.float64)
    for b in range(2):
        ref, _, _ = O.absorbed_decode(synth.bf16_bits_to_f32(q_nope)[b], synth.bf16_bits_to_f32(q_pe)[b],
                                      lat[b, :, :512], lat[b, :, 512:], Wuk, Wuv, scale)
        assert_close(got[b], ref, what=f"out[{b}]")
