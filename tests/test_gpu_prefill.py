"""GPU parity of the unabsorbed causal prefill (mla_prefill): keys and values
expanded once per cached token ("手搓 MLA" §三: k_nope, v = split(kv_up)), then
standard causal attention, against the fp64 oracle's expand-then-attend path
(naive_attend_causal) at the decode tolerance (abs 2e-2 + rel 1e-2
elementwise, rel-RMS 1e-2 per head, cosine 0.9999), and against the absorbed
multi-query decode on the same inputs.
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


def _status():
    import mla_absorbed_latent_gb300 as mla
    return mla.mla_get_device_status()


def _prefill(dev, T, qn, qp, seqlens=None):
    import mla_absorbed_latent_gb300 as mla
    prob = dev.prob
    B, H = prob.B, prob.H
    lens = dev.seqlens if seqlens is None else torch.tensor(seqlens, dtype=torch.int32, device="cuda")
    ws_bytes = mla.mla_prefill_workspace_bytes(B, H, prob.max_pages)
    ws = torch.full((ws_bytes,), 0xFF, dtype=torch.uint8, device="cuda")  # NaN bit patterns: every read is written first
    out = torch.full((B, T, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    mla.mla_prefill(bits_to_device(qn), bits_to_device(qp), dev.wkv, H, T, dev.cache, dev.page_table, prob.max_pages,
                    lens, B, prob.scale, ws, ws_bytes, out)
    torch.cuda.synchronize()
    return _f64(out)


def _naive(prob, qn, qp, b, n, T):
    Wuk, Wuv = weights(prob)
    c, p = prob.sequence(b, 0, n)
    return O.naive_attend_causal(synth.bf16_bits_to_f32(qn[b]), synth.bf16_bits_to_f32(qp[b]),
                                 synth.bf16_bits_to_f32(c), synth.bf16_bits_to_f32(p), Wuk, Wuv, prob.scale)


def test_prefill_v2lite_25_tokens():
    """The V2-Lite layer's 25-token prefill: query t at position t sees tokens 0..t."""
    prob = make_problem(16, [25], seed=0, paged=False)
    dev = DeviceDecode(prob)
    qn, qp = synth.gen_queries_multi(16, 25, [25], seed=0)
    out = _prefill(dev, 25, qn, qp)
    st, info = _status()
    assert st == 0, info
    assert_close(out[0], _naive(prob, qn, qp, 0, 25, 25))


@pytest.mark.parametrize("H,T,seqlens", [(16, 64, [300, 64, 129]), (128, 130, [130, 257]),
                                         (16, 300, [700, 300]), (128, 1, [1, 65, 1000])])
def test_prefill_ragged_rows(H, T, seqlens):
    """Several query tiles (T > 128), key tiles crossing the causal diagonal and the
    rows' last pages, paged random table; every row against the oracle."""
    prob = make_problem(H, seqlens, seed=90 + H + T)
    dev = DeviceDecode(prob)
    qn, qp = synth.gen_queries_multi(H, T, seqlens, seed=90 + H + T)
    out = _prefill(dev, T, qn, qp)
    st, info = _status()
    assert st == 0, info
    for b, n in enumerate(seqlens):
        assert_close(out[b], _naive(prob, qn, qp, b, n, T), what=f"row {b}")


def test_prefill_matches_absorbed_decode():
    """The same causal queries through both forms (expanded and absorbed)."""
    import mla_absorbed_latent_gb300 as mla
    H, T, seqlens = 128, 3, [500, 64, 200]
    prob = make_problem(H, seqlens, seed=97)
    dev = DeviceDecode(prob)
    qn, qp = synth.gen_queries_multi(H, T, seqlens, seed=97)
    a = _prefill(dev, T, qn, qp)
    ws_bytes = mla.mla_decode_q_workspace_bytes(prob.B, H, T)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.empty((prob.B, T, H, 128), dtype=torch.bfloat16, device="cuda")
    mla.mla_decode_q(bits_to_device(qn), bits_to_device(qp), dev.W_UK, dev.W_UV, H, T, dev.cache, dev.page_table,
                     prob.max_pages, dev.seqlens, prob.B, prob.scale, ws, ws_bytes, out)
    torch.cuda.synchronize()
    assert_close(a, _f64(out), what="unabsorbed vs absorbed")


def test_prefill_rejects_quantized_pool_and_reports_short_rows():
    import mla_absorbed_latent_gb300 as mla
    prob = make_problem(16, [10], seed=98, fmt="int8")
    dev = DeviceDecode(prob)
    qn, qp = synth.gen_queries_multi(16, 4, [10], seed=98)
    ws = torch.empty(mla.mla_prefill_workspace_bytes(1, 16, prob.max_pages), dtype=torch.uint8, device="cuda")
    out = torch.empty((1, 4, 16, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mla.MLAError) as e:
        mla.mla_prefill(bits_to_device(qn), bits_to_device(qp), dev.wkv, 16, 4, dev.cache, dev.page_table,
                        prob.max_pages, dev.seqlens, 1, prob.scale, ws, ws.numel(), out)
    assert e.value.status == mla.MLA_ERR_UNSUPPORTED
    # a row shorter than its queries
    prob = make_problem(16, [3], seed=99)
    dev = DeviceDecode(prob)
    qn, qp = synth.gen_queries_multi(16, 5, [3], seed=99)
    _prefill(dev, 5, qn, qp)
    st, info = _status()
    assert st == mla.MLA_ERR_BOUNDS and info == 0
