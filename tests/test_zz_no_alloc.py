"""mla_decode_noalloc: the decode entry point for callers that cannot allocate
device memory (no workspace argument; the library keeps a fixed scratch array
in device memory).  Called through the C ABI and compared with mla_decode, the
entry point that takes a caller workspace, on two calls in a row, within the
parity tolerance of the other tests.  Kept in a file that pytest collects last.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")]

import synth  # noqa: E402
from synth.device import DeviceDecode, make_problem  # noqa: E402
from tests.parity import assert_close  # noqa: E402


def _f64(t):
    return synth.bf16_bits_to_f32(t.detach().view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)


@pytest.mark.parametrize("H,seqlens", [(16, [26, 4096, 1, 700]), (128, [8192, 65, 0, 3000, 64])])
def test_noalloc_matches_workspace_decode_twice(H, seqlens):
    import mla_absorbed_latent_gb300 as mla
    prob = make_problem(H, seqlens, seed=40 + H)
    dev = DeviceDecode(prob)
    ref = _f64(dev.decode())
    torch.cuda.synchronize()
    for _ in range(2):                     # two calls in a row share the scratch
        out = torch.full_like(dev.out, float("nan"))
        mla.mla_decode_noalloc(dev.q_nope, dev.q_pe, dev.W_UK, dev.W_UV, H, dev.cache, dev.page_table,
                               prob.max_pages, dev.seqlens, prob.B, prob.scale, out)
        torch.cuda.synchronize()
        st, info = mla.mla_get_device_status()
        assert st == mla.MLA_OK, (mla.mla_status_string(st), info)
        assert_close(_f64(out), ref, what="noalloc vs workspace decode")


def _noalloc_twice_vs_workspace(prob, dev):
    import mla_absorbed_latent_gb300 as mla
    ref = _f64(dev.decode())
    torch.cuda.synchronize()
    for _ in range(2):
        out = torch.full_like(dev.out, float("nan"))
        mla.mla_decode_noalloc(dev.q_nope, dev.q_pe, dev.W_UK, dev.W_UV, prob.H, dev.cache, dev.page_table,
                               prob.max_pages, dev.seqlens, prob.B, prob.scale, out)
        torch.cuda.synchronize()
        st, info = mla.mla_get_device_status()
        assert st == mla.MLA_OK, (mla.mla_status_string(st), info)
        assert_close(_f64(out), ref, what="noalloc vs workspace decode")
    return out


def test_noalloc_fewer_workers_than_decode():
    """H=128, B=230: the query latent (34 MB) plus the partials of the default
    worker count do not fit the 64 MiB scratch, but fewer workers do, so the
    plan, attend and combine run with a reduced split count (and a partial
    tensor map and merge sized by it); against the workspace decode twice, and
    a few rows against the oracle."""
    import mla_absorbed_latent_gb300 as mla
    from tests.parity import oracle_outputs
    H, B = 128, 230
    # 34 MB of query latent + 76 default workers' partials (B + 76 slots of 131.6 KB) > 64 MiB;
    # one worker's (B + 1 slots) fits
    assert B * H * 576 * 2 + (B + mla.mla_decode_max_workers(H, "bf16")) * H * 1028 > mla.MLA_NOALLOC_SCRATCH_BYTES
    assert B * H * 576 * 2 + (B + 1) * H * 1028 + (1 << 16) < mla.MLA_NOALLOC_SCRATCH_BYTES
    seqlens = [(1, 64, 65, 130, 200, 7)[b % 6] for b in range(B)]
    prob = make_problem(H, seqlens, seed=44)
    dev = DeviceDecode(prob)
    out = _noalloc_twice_vs_workspace(prob, dev)
    rows = [0, 1, 2, 3, 4, 5, 117, 229]
    ref = oracle_outputs(prob, rows)
    got = _f64(out)
    for b in rows:
        assert_close(got[b], ref[b], what=f"noalloc out[{b}]")


@pytest.mark.parametrize("fmt", ["int8", "int4", "int8_token", "int4_sym", "int4_pe4"])
def test_noalloc_quantized_pools(fmt):
    """H=128 over INT8 / INT4 pools through the no-allocation entry point,
    against the workspace decode on two calls in a row."""
    prob = make_problem(128, [3000, 1, 129, 640], seed=46, fmt=fmt, dist="outlier")
    dev = DeviceDecode(prob)
    _noalloc_twice_vs_workspace(prob, dev)


def test_noalloc_rejects_batch_beyond_scratch():
    import mla_absorbed_latent_gb300 as mla
    prob = make_problem(128, [64], seed=3)
    dev = DeviceDecode(prob)
    B = 1024                                # q-side latent alone exceeds the fixed scratch
    big = torch.empty((B, 128, 128), dtype=torch.bfloat16, device="cuda")
    pt = torch.zeros((B, 1), dtype=torch.int32, device="cuda")
    with pytest.raises(mla.MLAError) as e:
        mla.mla_decode_noalloc(big, big, dev.W_UK, dev.W_UV, 128, dev.cache, pt, 1, pt, B, prob.scale, big)
    assert e.value.status == mla.MLA_ERR_WORKSPACE


def test_noalloc_16_head_kernels():
    """H=16 with each 16-head attend kernel selected (warp-level MMA, CUDA
    cores): the no-allocation call against the workspace decode with the same
    kernel, twice."""
    import mla_absorbed_latent_gb300 as mla
    prob = make_problem(16, [700, 1, 64, 3000], seed=124)
    dev = DeviceDecode(prob)
    try:
        for kind in (mla.MLA_KERNEL_MMA, mla.MLA_KERNEL_CUDA_CORES):
            mla.mla_decode_select_kernel(16, kind)
            _noalloc_twice_vs_workspace(prob, dev)
    finally:
        mla.mla_decode_select_kernel(16, mla.MLA_KERNEL_MMA)
