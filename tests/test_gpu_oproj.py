"""GPU parity of the output projection after the value up-projection
(mla_output_projection: y = o Wo^T over the heads side by side, "手搓 MLA"
§三/§四 "@ Wo.T") against the fp64 oracle's output_projection, alone and
chained after a decode, at the decode tolerance."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")]

import oracle as O  # noqa: E402
import synth  # noqa: E402
from synth.device import DeviceDecode, bits_to_device, make_problem  # noqa: E402
from tests.parity import assert_close, oracle_outputs  # noqa: E402


def _f64(t):
    return synth.bf16_bits_to_f32(t.detach().view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)


def _project(o, H, hidden, wo_bits):
    import mla_absorbed_latent_gb300 as mla
    R = o.shape[0]
    y = torch.full((R, hidden), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws_bytes = mla.mla_output_projection_workspace_bytes(R, H, hidden)
    ws = torch.full((max(ws_bytes, 256),), 0xFF, dtype=torch.uint8, device="cuda")
    mla.mla_output_projection(o, bits_to_device(wo_bits), R, H, hidden, y, ws, ws_bytes)
    torch.cuda.synchronize()
    st, info = mla.mla_get_device_status()
    assert st == 0, info
    return _f64(y)


@pytest.mark.parametrize("H,hidden,R", [(16, 2048, 1), (16, 2048, 32), (128, 7168, 64), (128, 7168, 200),
                                        (128, 1024, 65)])
def test_output_projection_random_rows(H, hidden, R):
    """Rows of N(0,1) bf16 head outputs (row tiles with a ragged last one, split and
    unsplit reductions) against the oracle."""
    rng = np.random.default_rng(H + R)
    o_bits = synth.f32_to_bf16_bits(rng.standard_normal((R, H, 128)).astype(np.float32))
    wo = synth.gen_out_weights(H, hidden, seed=R)
    got = _project(bits_to_device(o_bits), H, hidden, wo)
    ref = O.output_projection(synth.bf16_bits_to_f32(o_bits), synth.bf16_bits_to_f32(wo))
    assert_close(got, ref, what="y")


def test_output_projection_after_decode():
    """The chain decode -> output projection on one stream (the projection reads the
    decode's bf16 output), against the oracle's decode followed by its projection
    (of the bf16-rounded decode output, as the library rounds it)."""
    H, hidden = 128, 7168
    seqlens = [1000, 64, 3000, 5]
    prob = make_problem(H, seqlens, seed=120)
    dev = DeviceDecode(prob)
    out = dev.decode()
    wo = synth.gen_out_weights(H, hidden, seed=121)
    got = _project(out, H, hidden, wo)
    ref_heads = oracle_outputs(prob, range(prob.B))
    o_ref = np.stack([ref_heads[b] for b in range(prob.B)])
    assert_close(_f64(out), o_ref, what="decode out")
    ref = O.output_projection(_f64(out), synth.bf16_bits_to_f32(wo))
    assert_close(got, ref, what="y")
