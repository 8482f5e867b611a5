"""GPU parity of the causal multi-query decode (mla_decode_q): T query tokens
per row, query t at position n - T + t seeing tokens 0 .. n - T + t, against
the fp64 oracle's absorbed_attend_causal ("手搓 MLA" §四 with its query-token
axis; "DeepSeek MLA 吸收式缓存" §3.4's causal prefill and incremental decode).
Tolerance as for the single-query decode (abs 2e-2 + rel 1e-2 elementwise,
rel-RMS 1e-2 per head, cosine 0.9999).
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")]

import oracle as O  # noqa: E402
import synth  # noqa: E402
from synth.device import DeviceDecode, bits_to_device, make_problem  # noqa: E402
from tests.parity import assert_close, weights  # noqa: E402


def _f64(t):
    return synth.bf16_bits_to_f32(t.detach().view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)


def _status_ok():
    import mla_absorbed_latent_gb300 as mla
    st, info = mla.mla_get_device_status()
    assert st == mla.MLA_OK, (mla.mla_status_string(st), info)


def _decode_q(dev, T, qn, qp, seqlens=None):
    """mla_decode_q over dev's cache; returns (out [B,T,H,128] f64, o_lat [B,T,H,512] f64)."""
    import mla_absorbed_latent_gb300 as mla
    prob = dev.prob
    B, H = prob.B, prob.H
    lens = dev.seqlens if seqlens is None else torch.tensor(seqlens, dtype=torch.int32, device="cuda")
    ws_bytes = mla.mla_decode_q_workspace_bytes(B, H, T)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.full((B, T, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    ol = torch.full((B, T, H, 512), float("nan"), dtype=torch.float32, device="cuda")
    mla.mla_decode_q(bits_to_device(qn), bits_to_device(qp), dev.W_UK, dev.W_UV, H, T, dev.cache, dev.page_table,
                     prob.max_pages, lens, B, prob.scale, ws, ws_bytes, out, ol)
    torch.cuda.synchronize()
    return _f64(out), ol.cpu().numpy().astype(np.float64)


def _oracle(prob, qn, qp, b, n, T):
    """out [T,H,128], o_lat [T,H,512] of row b over its first n tokens, queries at n-T .. n-1."""
    Wuk, Wuv = weights(prob)
    c, p = prob.sequence(b, 0, n)
    C, P = O.dequantized_tokens(prob.fmt, synth.bf16_bits_to_f32(c), synth.bf16_bits_to_f32(p))
    return O.absorbed_attend_causal(synth.bf16_bits_to_f32(qn[b]), synth.bf16_bits_to_f32(qp[b]), C, P, Wuk, Wuv,
                                    prob.scale)


def _check(prob, qn, qp, out, ol, T, lens=None, check_lat=True):
    lens = prob.seqlens if lens is None else lens
    for b in range(prob.B):
        ref, ref_lat = _oracle(prob, qn, qp, b, int(lens[b]), T)
        assert_close(out[b], ref, what=f"out[{b}]")
        if check_lat:
            if prob.fmt == "bf16":
                assert_close(ol[b], ref_lat, what=f"o_lat[{b}]")
            else:
                # dequantized values rounded to bf16 and bf16 split partials: 2^-8 of the
                # channel's largest magnitude on top (as for the single-query decode)
                c, p = prob.sequence(b, 0, int(lens[b]))
                C, _ = O.dequantized_tokens(prob.fmt, synth.bf16_bits_to_f32(c), synth.bf16_bits_to_f32(p))
                bound = 2e-2 + 1e-2 * np.abs(ref_lat) + 2.0 ** -8 * np.max(np.abs(C), axis=0)
                assert np.all(np.abs(ol[b] - ref_lat) <= bound), f"o_lat[{b}]"


def test_multi_v2lite_prefill_chunk_then_decode():
    """The V2-Lite layer case: a 25-token causal chunk over the first 25 cached
    tokens (query t sees tokens 0..t), then the incremental decode of token 25
    over all 26; both against the oracle, and the decode against mla_decode."""
    H = 16
    prob = make_problem(H, [26], seed=0, paged=False)
    dev = DeviceDecode(prob, prefill=25)
    qn25, qp25 = synth.gen_queries_multi(H, 25, [25], seed=0)
    out, ol = _decode_q(dev, 25, qn25, qp25, seqlens=[25])
    _status_ok()
    _check(prob, qn25, qp25, out, ol, 25, lens=[25])
    # the decode step: the single-query queries of the workload, through both entry points
    qn1 = prob.q_nope[:, None]
    qp1 = prob.q_pe[:, None]
    out1, ol1 = _decode_q(dev, 1, qn1, qp1)
    _status_ok()
    _check(prob, qn1, qp1, out1, ol1, 1)
    ref = _f64(dev.decode())
    torch.cuda.synchronize()
    assert_close(out1[:, 0], ref, what="mla_decode_q T=1 vs mla_decode")


def test_multi_h16_t8_ragged():
    """H=16, 8 query tokens per row (128 virtual heads, one pass over each row's
    cache): lengths at and around page edges, random page table."""
    T = 8
    seqlens = [8, 9, 63, 64, 65, 71, 130, 700, 2000, 4096]
    prob = make_problem(16, seqlens, seed=81)
    dev = DeviceDecode(prob)
    qn, qp = synth.gen_queries_multi(16, T, seqlens, seed=81)
    out, ol = _decode_q(dev, T, qn, qp)
    _status_ok()
    _check(prob, qn, qp, out, ol, T)


@pytest.mark.parametrize("T", [3, 25])
def test_multi_h16_padding_lanes(T):
    """H=16 with T not a multiple of 8: the last virtual row of each row carries
    padding lanes (and T=25 four virtual rows per row, each with its own view)."""
    seqlens = [25, 26, 64, 100, 1000]
    prob = make_problem(16, seqlens, seed=82 + T)
    dev = DeviceDecode(prob)
    qn, qp = synth.gen_queries_multi(16, T, seqlens, seed=82 + T)
    out, ol = _decode_q(dev, T, qn, qp)
    _status_ok()
    _check(prob, qn, qp, out, ol, T)


def test_multi_h128_t2():
    """H=128, 2 query tokens per row: one token per pass (G=1), each its own view."""
    T = 2
    seqlens = [2, 63, 64, 65, 500, 3000]
    prob = make_problem(128, seqlens, seed=83)
    dev = DeviceDecode(prob)
    qn, qp = synth.gen_queries_multi(128, T, seqlens, seed=83)
    out, ol = _decode_q(dev, T, qn, qp)
    _status_ok()
    _check(prob, qn, qp, out, ol, T)


@pytest.mark.parametrize("fmt", ["int8", "int4", "int8_token", "int4_sym", "int4_pe4"])
def test_multi_quantized_pools(fmt):
    """Causal multi-query decode over INT8 / INT4 pools (H=16, T=5; H=128, T=2)."""
    for H, T, seed in ((16, 5, 84), (128, 2, 85)):
        seqlens = [5, 64, 77, 900]
        prob = make_problem(H, seqlens, seed=seed, fmt=fmt, dist="outlier")
        dev = DeviceDecode(prob)
        qn, qp = synth.gen_queries_multi(H, T, seqlens, seed=seed)
        out, ol = _decode_q(dev, T, qn, qp)
        _status_ok()
        _check(prob, qn, qp, out, ol, T)


def test_multi_h16_t1_matches_single_query_decodes():
    """T=1 at H=16 runs on the fifth-generation tensor cores (7 of 8 token lanes
    padding) and must agree with the oracle and with both 16-head single-query
    kernels (warp-level MMA, CUDA cores)."""
    import mla_absorbed_latent_gb300 as mla
    seqlens = [1, 64, 65, 4096, 333]
    prob = make_problem(16, seqlens, seed=86)
    dev = DeviceDecode(prob)
    out, ol = _decode_q(dev, 1, prob.q_nope[:, None], prob.q_pe[:, None])
    _status_ok()
    _check(prob, prob.q_nope[:, None], prob.q_pe[:, None], out, ol, 1)
    try:
        for kind in (mla.MLA_KERNEL_MMA, mla.MLA_KERNEL_CUDA_CORES):
            mla.mla_decode_select_kernel(16, kind)
            ref = _f64(dev.decode())
            torch.cuda.synchronize()
            _status_ok()
            assert_close(out[:, 0], ref, what=f"tcgen05 vs single-query kernel {kind}")
    finally:
        mla.mla_decode_select_kernel(16, mla.MLA_KERNEL_MMA)


def test_multi_range_jump_is_exact():
    """H=16, T=8: one cached token's RoPE key is 200 x head 3's q_pe of query 7,
    far past the fast path's tracked range for the virtual heads that see it;
    the flagged row is recomputed per virtual head over its own causal view
    (queries 0..6 do not see that token when it sits at position n-1)."""
    T = 8
    n = 64 * 40
    prob = make_problem(16, [n, 500], seed=87, paged=False)
    dev = DeviceDecode(prob)
    qn, qp = synth.gen_queries_multi(16, T, [n, 500], seed=87)
    qpe = synth.bf16_bits_to_f32(qp)[0, T - 1, 3]
    for token in (64 * 7 + 3, n - 1):
        bits = synth.f32_to_bf16_bits((200.0 * qpe).astype(np.float32))
        page, slot = divmod(token, 64)
        off = int(dev.page_table[0, page]) * dev.page_bytes + slot * 1152 + 1024
        dev.pool[off:off + 128] = torch.from_numpy(bits.view(np.uint8).copy()).to(dev.pool.device)
    out, ol = _decode_q(dev, T, qn, qp)
    _status_ok()
    # the oracle on the same modified cache
    Wuk, Wuv = weights(prob)
    c, p = prob.sequence(0)
    C, P = synth.bf16_bits_to_f32(c).astype(np.float64), synth.bf16_bits_to_f32(p).astype(np.float64)
    for token in (64 * 7 + 3, n - 1):
        P[token] = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits((200.0 * qpe).astype(np.float32)))
    ref, ref_lat = O.absorbed_attend_causal(synth.bf16_bits_to_f32(qn[0]), synth.bf16_bits_to_f32(qp[0]), C, P, Wuk,
                                            Wuv, prob.scale)
    assert_close(out[0], ref, what="out[0]")
    assert_close(ol[0], ref_lat, what="o_lat[0]")
    ref1, _ = _oracle(prob, qn, qp, 1, 500, T)
    assert_close(out[1], ref1, what="out[1]")


def test_multi_short_row_reports_bounds():
    import mla_absorbed_latent_gb300 as mla
    prob = make_problem(128, [3], seed=88)
    dev = DeviceDecode(prob)
    qn, qp = synth.gen_queries_multi(128, 4, [3], seed=88)
    _decode_q(dev, 4, qn, qp)
    st, info = mla.mla_get_device_status()
    assert st == mla.MLA_ERR_BOUNDS and info == 0
