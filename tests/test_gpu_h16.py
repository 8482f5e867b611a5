"""GPU parity of the two 16-head attend kernels (the V2-Lite layer, "DeepSeek MLA
吸收式缓存" §2.2–§2.4 with H = 16): the warp-level MMA kernel (mma.sync
m16n8k16, the default) and the CUDA-core kernel, each selected through
mla_decode_select_kernel and checked against the fp64 oracle at the decode
tolerance (abs 2e-2 + rel 1e-2 elementwise, rel-RMS 1e-2 per head, cosine
0.9999), and against each other.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")]

import oracle as O  # noqa: E402
import synth  # noqa: E402
from synth.device import DeviceDecode, make_problem, problem_from_workload  # noqa: E402
from tests.parity import assert_close, oracle_outputs, oracle_rows, weights  # noqa: E402

KINDS = ["mma", "cuda_cores"]


def _kind(name):
    import mla_absorbed_latent_gb300 as mla
    return {"mma": mla.MLA_KERNEL_MMA, "cuda_cores": mla.MLA_KERNEL_CUDA_CORES}[name]


@pytest.fixture
def select():
    """Selects a 16-head kernel for the test and restores the default after it."""
    import mla_absorbed_latent_gb300 as mla

    def _select(name):
        mla.mla_decode_select_kernel(16, _kind(name))
        assert mla.mla_decode_kernel_kind(16) == _kind(name)
    yield _select
    mla.mla_decode_select_kernel(16, mla.MLA_KERNEL_MMA)


def _f64(t):
    return synth.bf16_bits_to_f32(t.detach().view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)


def _status_ok():
    import mla_absorbed_latent_gb300 as mla
    st, info = mla.mla_get_device_status()
    assert st == mla.MLA_OK, (mla.mla_status_string(st), info)


def test_default_16_head_kernel_is_mma():
    import mla_absorbed_latent_gb300 as mla
    assert mla.mla_decode_kernel_kind(16) == mla.MLA_KERNEL_MMA
    assert mla.mla_decode_kernel_kind(128) == mla.MLA_KERNEL_TCGEN05
    with pytest.raises(mla.MLAError):
        mla.mla_decode_select_kernel(128, mla.MLA_KERNEL_MMA)
    with pytest.raises(mla.MLAError):
        mla.mla_decode_select_kernel(16, mla.MLA_KERNEL_TCGEN05)


@pytest.mark.parametrize("kind", KINDS)
def test_h16_ragged_edges(kind, select):
    """Lengths at and around the half-page and page edges, an empty row, several
    split workers per row; out and o_lat of every row against the oracle."""
    select(kind)
    seqlens = [1, 2, 31, 32, 33, 63, 64, 65, 0, 97, 200, 1000, 4097, 129]
    prob = make_problem(16, seqlens, seed=120)
    dev = DeviceDecode(prob)
    o_lat = torch.full((prob.B, 16, 512), float("nan"), dtype=torch.float32, device="cuda")
    dev.workspace.fill_(0xFF)
    dev.decode_steps(o_lat)
    torch.cuda.synchronize()
    _status_ok()
    rows = [b for b, n in enumerate(seqlens) if n > 0]
    ref = oracle_rows(prob, rows)
    got = _f64(dev.out)
    lat = o_lat.cpu().numpy().astype(np.float64)
    for b in rows:
        assert_close(got[b], ref[b][0], what=f"out[{b}]")
        assert_close(lat[b], ref[b][1], what=f"o_lat[{b}]")
    empty = seqlens.index(0)
    assert torch.count_nonzero(dev.out[empty]) == 0


@pytest.mark.parametrize("kind", KINDS)
def test_h16_v2lite_batch_full(kind, select):
    """The V2-Lite batch workload (B=32, 4,096 tokens each): every row."""
    select(kind)
    prob = problem_from_workload(synth.get_workload("v2lite_batch"))
    dev = DeviceDecode(prob)
    dev.decode()
    torch.cuda.synchronize()
    _status_ok()
    ref = oracle_outputs(prob, range(prob.B))
    got = _f64(dev.out)
    for b in range(prob.B):
        assert_close(got[b], ref[b], what=f"out[{b}]")


def test_h16_kernels_agree(select):
    """The same problem through both kernels: within tolerance of each other."""
    seqlens = [5000, 33, 640, 1, 2222]
    prob = make_problem(16, seqlens, seed=121)
    dev = DeviceDecode(prob)
    outs = {}
    for kind in KINDS:
        select(kind)
        dev.decode()
        torch.cuda.synchronize()
        _status_ok()
        outs[kind] = _f64(dev.out)
    assert_close(outs["mma"], outs["cuda_cores"], what="mma vs cuda cores")


@pytest.mark.parametrize("kind", KINDS)
def test_h16_garbage_past_row_end_is_ignored(kind, select):
    """The page slots past each row's length hold all-ones bytes (NaN in bf16):
    they are neither keys nor values of the row (the MMA kernel multiplies whole
    32-token blocks, so it must mask the scores and zero those value rows)."""
    select(kind)
    seqlens = [1, 33, 63, 100, 129, 2000]
    prob = make_problem(16, seqlens, seed=122)
    dev = DeviceDecode(prob)
    for b, n in enumerate(seqlens):
        last = (n - 1) // 64
        page = int(dev.page_table[b, last])
        lo = page * dev.page_bytes + (n - 64 * last) * 1152
        dev.pool[lo:(page + 1) * dev.page_bytes] = 0xFF
    dev.decode()
    torch.cuda.synchronize()
    _status_ok()
    ref = oracle_rows(prob, range(prob.B))
    got = _f64(dev.out)
    for b in range(prob.B):
        assert_close(got[b], ref[b][0], what=f"out[{b}]")


@pytest.mark.parametrize("kind", KINDS)
def test_h16_extreme_scores_are_exact(kind, select):
    """RoPE keys 200 x a head's q_pe (a score about 1,300 log2 units above the
    rest) in the middle of the row and in its last half page, for two heads: the
    16-head kernels rescale at every new maximum, so the result is the defined
    softmax (against the oracle on the same modified cache)."""
    select(kind)
    n = 64 * 60 + 17
    prob = make_problem(16, [n, 300], seed=123, paged=False)
    dev = DeviceDecode(prob)
    qp = synth.bf16_bits_to_f32(prob.q_pe)
    c, p = prob.sequence(0)
    C, P = synth.bf16_bits_to_f32(c).astype(np.float64), synth.bf16_bits_to_f32(p).astype(np.float64)
    for head, token in ((3, 64 * 21 + 40), (11, n - 1)):
        bits = synth.f32_to_bf16_bits((200.0 * qp[0, head]).astype(np.float32))
        P[token] = synth.bf16_bits_to_f32(bits)
        page, slot = divmod(token, 64)
        off = int(dev.page_table[0, page]) * dev.page_bytes + slot * 1152 + 1024
        dev.pool[off:off + 128] = torch.from_numpy(bits.view(np.uint8).copy()).to(dev.pool.device)
    o_lat = torch.empty((2, 16, 512), dtype=torch.float32, device="cuda")
    dev.decode_steps(o_lat)
    torch.cuda.synchronize()
    _status_ok()
    Wuk, Wuv = weights(prob)
    ref, ref_lat, _ = O.absorbed_decode(synth.bf16_bits_to_f32(prob.q_nope)[0], qp[0], C, P, Wuk, Wuv, prob.scale)
    assert_close(_f64(dev.out)[0], ref)
    assert_close(o_lat[0].cpu().numpy(), ref_lat, what="o_lat")
    assert_close(_f64(dev.out)[1], oracle_rows(prob, [1])[1][0], what="out[1]")


@pytest.mark.parametrize("kind", KINDS)
def test_h16_long_row_many_segments(kind, select):
    """One 40,000-token row (625 pages) beside short rows: every split worker takes
    a piece of the long row, so its merge has more than 32 segments (the merge's
    weights go out in chunks of 32) and the short rows sit inside one worker's
    range.  Out and o_lat of every row against the oracle."""
    select(kind)
    seqlens = [40000, 3, 64, 1000]
    prob = make_problem(16, seqlens, seed=125)
    dev = DeviceDecode(prob)
    o_lat = torch.empty((prob.B, 16, 512), dtype=torch.float32, device="cuda")
    dev.decode_steps(o_lat)
    torch.cuda.synchronize()
    _status_ok()
    ref = oracle_rows(prob, range(prob.B))
    got = _f64(dev.out)
    lat = o_lat.cpu().numpy().astype(np.float64)
    for b in range(prob.B):
        assert_close(got[b], ref[b][0], what=f"out[{b}]")
        assert_close(lat[b], ref[b][1], what=f"o_lat[{b}]")
