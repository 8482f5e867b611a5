"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Bit-exact where the result is a copy or an integer decision (weight split,
page placement, quantized codes and scales); abs 2e-2 + rel 1e-2 elementwise
plus rel-RMS 1e-2 and cosine 0.9999 for the bf16 decode outputs.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")]

import oracle as O  # noqa: E402
import synth  # noqa: E402
from synth.device import DeviceDecode, bits_to_device, make_problem, problem_from_workload  # noqa: E402
from tests.parity import assert_close, oracle_outputs, oracle_rows, weights  # noqa: E402


def _np_bf16(t):
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def _out_f64(t):
    return synth.bf16_bits_to_f32(_np_bf16(t)).astype(np.float64)


def _status_ok():
    import mla_absorbed_latent_gb300 as mla
    st, info = mla.mla_get_device_status()
    assert st == mla.MLA_OK, (mla.mla_status_string(st), info)


# ----------------------------------------------------------------------------
# weights and cache placement: bit-exact
@pytest.mark.parametrize("H", [16, 128])
def test_stepwise_absorb_right_after_weight_split(H):
    """The weight split enqueued directly before the step-wise q-absorb (the plan
    enqueued first), W_UK and W_UV filled with NaN bits beforehand: the q-absorb
    step loads W_UK only after it has waited for the kernel before it, so the
    decode reads the fresh split and matches the oracle."""
    import mla_absorbed_latent_gb300 as mla
    seqlens = [300, 2000, 64, 1]
    prob = make_problem(H, seqlens, seed=70 + H)
    dev = DeviceDecode(prob)
    ref = oracle_outputs(prob, range(prob.B))
    for _ in range(3):
        dev.W_UK.view(torch.int16).fill_(-1)
        dev.W_UV.view(torch.int16).fill_(-1)
        mla.mla_decode_plan(H, "bf16", dev.seqlens, prob.B, prob.max_pages, dev.workspace, dev.ws_bytes)
        mla.mla_absorb_weights(dev.wkv, H, dev.W_UK, dev.W_UV)
        mla.mla_decode_absorb_q(dev.q_nope, dev.q_pe, dev.W_UK, H, prob.B, dev.workspace, dev.ws_bytes)
        mla.mla_decode_attend(H, dev.cache, dev.page_table, prob.max_pages, dev.seqlens, prob.B, prob.scale,
                              dev.workspace, dev.ws_bytes)
        mla.mla_decode_combine(dev.W_UV, H, prob.B, dev.workspace, dev.ws_bytes, dev.out)
        torch.cuda.synchronize()
        _status_ok()
        got = _out_f64(dev.out)
        for bb in range(prob.B):
            assert_close(got[bb], ref[bb], what=f"out[{bb}]")


# ----------------------------------------------------------------------------

@pytest.mark.parametrize("H", [16, 128])
def test_absorb_weights_bitexact(H):
    import mla_absorbed_latent_gb300 as mla
    wkv = synth.gen_weights(H, seed=7)
    W_UK = torch.empty((H, 512, 128), dtype=torch.bfloat16, device="cuda")
    W_UV = torch.empty((H, 128, 512), dtype=torch.bfloat16, device="cuda")
    mla.mla_absorb_weights(bits_to_device(wkv), H, W_UK, W_UV)
    uk, uv = O.split_wkv_b(synth.bf16_bits_to_f32(wkv), H)
    got_uk = synth.bf16_bits_to_f32(_np_bf16(W_UK)).astype(np.float64)
    got_uv = synth.bf16_bits_to_f32(_np_bf16(W_UV)).astype(np.float64)
    assert np.array_equal(got_uk, np.transpose(uk, (0, 2, 1)))
    assert np.array_equal(got_uv, uv)


def _pool_bytes(dev):
    return dev.pool.cpu().numpy().reshape(dev.prob.num_pages, -1)


def _expected_pool(prob, writes):
    return O.expected_page_pool(prob.fmt, prob.num_pages, writes)


@pytest.mark.parametrize("fmt", ["bf16", "int8", "int4", "int8_token", "int4_sym", "int4_pe4"])
def test_append_prefill_then_decode_bitexact(fmt):
    """V2-Lite tiny case: 25-token prefill append, then the decode token at position 25."""
    w = synth.get_workload("v2lite_tiny")
    prob = make_problem(w.H, [26], w.seed, paged=False, fmt=fmt)
    dev = DeviceDecode(prob, prefill=25)
    _status_ok()
    c, p = prob.sequence(0)
    want = _expected_pool(prob, [(prob.page_table[0], 0, synth.bf16_bits_to_f32(c), synth.bf16_bits_to_f32(p))])
    assert np.array_equal(_pool_bytes(dev), want)


@pytest.mark.parametrize("fmt", ["bf16", "int8", "int4", "int8_token", "int4_sym", "int4_pe4"])
def test_append_ragged_paged_bitexact(fmt):
    """Several rows, random page table, appends that start mid-page and cross pages."""
    import mla_absorbed_latent_gb300 as mla
    seqlens = [70, 1, 130, 64, 200]
    prob = make_problem(128, seqlens, seed=21, fmt=fmt, dist="outlier", spare_pages=3)
    dev = DeviceDecode(prob, prefill=None)  # appends tokens 0..n-1 per row
    # second append: 37 more tokens per row at pos = seqlen (rows with room)
    extra = 37
    rows = [0, 2, 3]
    rng = np.random.default_rng(5)
    c_new = synth.f32_to_bf16_bits(rng.standard_normal((len(rows), extra, 512)).astype(np.float32) * 3)
    p_new = synth.f32_to_bf16_bits(rng.standard_normal((len(rows), extra, 64)).astype(np.float32))
    # give those rows fresh pages for the spill-over (the spare pages)
    table = prob.page_table.copy()
    spare = list(range(prob.num_pages - 3, prob.num_pages))
    for r in rows:
        n = seqlens[r]
        need = (n + extra + 63) // 64
        for j in range((n + 63) // 64, need):
            table = np.pad(table, ((0, 0), (0, max(0, j + 1 - table.shape[1]))), constant_values=-1)
            table[r, j] = spare.pop(0)
    pt = torch.from_numpy(np.ascontiguousarray(table[rows])).cuda()
    pos = torch.tensor([seqlens[r] for r in rows], dtype=torch.int32, device="cuda")
    mla.mla_cache_append(dev.cache, bits_to_device(c_new), bits_to_device(p_new), pt, table.shape[1], pos,
                         len(rows), extra)
    torch.cuda.synchronize()
    _status_ok()
    writes = []
    for b, n in enumerate(seqlens):
        c, p = prob.sequence(b)
        writes.append((prob.page_table[b], 0, synth.bf16_bits_to_f32(c), synth.bf16_bits_to_f32(p)))
    for i, r in enumerate(rows):
        writes.append((table[r], seqlens[r], synth.bf16_bits_to_f32(c_new[i]), synth.bf16_bits_to_f32(p_new[i])))
    assert np.array_equal(_pool_bytes(dev), _expected_pool(prob, writes))


def test_append_out_of_bounds_is_reported_not_written():
    import mla_absorbed_latent_gb300 as mla
    prob = make_problem(16, [10], seed=3)
    dev = DeviceDecode(prob)
    before = dev.pool.clone()
    c = torch.zeros((1, 1, 512), dtype=torch.bfloat16, device="cuda")
    p = torch.zeros((1, 1, 64), dtype=torch.bfloat16, device="cuda")
    pos = torch.tensor([64 * prob.max_pages], dtype=torch.int32, device="cuda")   # one past capacity
    mla.mla_cache_append(dev.cache, c, p, dev.page_table, prob.max_pages, pos, 1, 1)
    st, info = mla.mla_get_device_status()
    assert st == mla.MLA_ERR_BOUNDS and info == 0
    bad_table = torch.tensor([[prob.num_pages + 5]], dtype=torch.int32, device="cuda")
    pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_cache_append(dev.cache, c, p, bad_table, 1, pos, 1, 1)
    st, info = mla.mla_get_device_status()
    assert st == mla.MLA_ERR_BOUNDS and info == prob.num_pages + 5
    assert torch.equal(before, dev.pool)
    _status_ok()


# ----------------------------------------------------------------------------
# decode parity
# ----------------------------------------------------------------------------

def _check_all_rows(dev, rows=None):
    """Every listed row (default: all non-empty rows) of dev.out against the fp64
    oracle, the oracle rows computed in parallel worker processes."""
    prob = dev.prob
    rows = [b for b in range(prob.B) if prob.seqlens[b] > 0] if rows is None else rows
    ref = oracle_outputs(prob, rows)
    got = _out_f64(dev.out)
    worst = 0.0
    for b in rows:
        _, r = assert_close(got[b], ref[b], what=f"out[{b}]")
        worst = max(worst, r)
    return worst


def _check_rows(dev, rows, o_lat=None):
    prob = dev.prob
    ref = oracle_rows(prob, rows)
    got = _out_f64(dev.out)
    worst = 0.0
    for b in rows:
        _, r = assert_close(got[b], ref[b][0], what=f"out[{b}]")
        worst = max(worst, r)
        if o_lat is not None:
            assert_close(o_lat[b].cpu().numpy(), ref[b][1], what=f"o_lat[{b}]")
    return worst


def test_decode_v2lite_tiny():
    w = synth.get_workload("v2lite_tiny")
    prob = problem_from_workload(w)
    dev = DeviceDecode(prob, prefill=25)
    o_lat = torch.empty((1, 16, 512), dtype=torch.float32, device="cuda")
    dev.decode_steps(o_lat)
    torch.cuda.synchronize()
    _status_ok()
    _check_rows(dev, [0], o_lat)
    # the oracle's naive path gives the same reference
    Wuk, Wuv = weights(prob)
    c, p = prob.sequence(0)
    naive = O.naive_decode(synth.bf16_bits_to_f32(prob.q_nope)[0], synth.bf16_bits_to_f32(prob.q_pe)[0],
                           synth.bf16_bits_to_f32(c), synth.bf16_bits_to_f32(p), Wuk, Wuv, prob.scale)
    assert_close(_out_f64(dev.out)[0], naive)


@pytest.mark.parametrize("H", [16, 128])
def test_decode_ragged_edges(H):
    """Lengths around the page and half-page edges, an empty row, several tiles."""
    seqlens = [1, 31, 32, 33, 63, 64, 65, 0, 200, 1000, 129]
    prob = make_problem(H, seqlens, seed=11 + H)
    dev = DeviceDecode(prob)
    o_lat = torch.empty((len(seqlens), H, 512), dtype=torch.float32, device="cuda")
    dev.decode_steps(o_lat)
    torch.cuda.synchronize()
    _status_ok()
    rows = [b for b, n in enumerate(seqlens) if n > 0]
    _check_rows(dev, rows, o_lat)
    empty = seqlens.index(0)
    assert torch.count_nonzero(dev.out[empty]) == 0
    assert torch.count_nonzero(o_lat[empty]) == 0


def test_decode_steps_equal_decode():
    prob = make_problem(128, [300, 77, 1], seed=5)
    dev = DeviceDecode(prob)
    a = dev.decode().clone()
    b = dev.decode_steps().clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_decode_page_permutation_bitexact():
    """Same tokens behind a different physical page order: identical output bits."""
    seqlens = [500, 130, 64]
    p1 = make_problem(128, seqlens, seed=9, paged=False)
    p2 = make_problem(128, seqlens, seed=9, paged=True)
    assert not np.array_equal(p1.page_table, p2.page_table)
    a = DeviceDecode(p1).decode().clone()
    b = DeviceDecode(p2).decode().clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_decode_v2lite_batch_full():
    """H=16, B=32, every seqlen 4096, contiguous cache: every row against the oracle."""
    prob = problem_from_workload(synth.get_workload("v2lite_batch"))
    dev = DeviceDecode(prob)
    dev.decode()
    torch.cuda.synchronize()
    _status_ok()
    _check_rows(dev, list(range(prob.B)))


def test_decode_v3_paged_full():
    """H=128, B=64, seqlen 8192, random page table: every row against the oracle."""
    prob = problem_from_workload(synth.get_workload("v3_paged"))
    dev = DeviceDecode(prob)
    o_lat = torch.empty((prob.B, 128, 512), dtype=torch.float32, device="cuda")
    dev.decode_steps(o_lat)
    torch.cuda.synchronize()
    _status_ok()
    _check_all_rows(dev)
    _check_rows(dev, [0, 63], o_lat)
    # every row's o_lat is a convex combination of unit-RMS latents: RMS <= 1
    rms = torch.sqrt(torch.mean(o_lat ** 2, dim=-1))
    assert bool(torch.all(rms <= 1.0 + 1e-3))


def test_decode_v3_ragged_full():
    """H=128, B=128, lognormal lengths (segments cross worker boundaries): every row."""
    prob = problem_from_workload(synth.get_workload("v3_ragged"))
    dev = DeviceDecode(prob)
    dev.decode()
    torch.cuda.synchronize()
    _status_ok()
    _check_all_rows(dev)


@pytest.mark.parametrize("fmt", ["int8", "int4", "int8_token", "int4_sym", "int4_pe4"])
def test_decode_quant_ragged_edges(fmt):
    """H=128 over INT8 / INT4 pages (dequantized in the load stage): lengths
    around the page edges, an empty row, outlier channels; against the oracle
    over the dequantized values."""
    seqlens = [1, 31, 33, 63, 64, 65, 0, 200, 1000, 129]
    prob = make_problem(128, seqlens, seed=31, fmt=fmt, dist="outlier")
    dev = DeviceDecode(prob)
    o_lat = torch.empty((len(seqlens), 128, 512), dtype=torch.float32, device="cuda")
    dev.decode_steps(o_lat)
    torch.cuda.synchronize()
    _status_ok()
    rows = [b for b, n in enumerate(seqlens) if n > 0]
    _check_rows(dev, rows)  # the bf16 outputs, at the stated tolerance
    # o_lat: the dequantized values are rounded once to bf16 for the MMA and
    # each split's partial o_lat is stored in bf16 (each half an ulp, 2^-9
    # relative; both propagate into o_lat as at most 2^-9 of the channel's
    # largest magnitude, o_lat being a convex combination of the latents),
    # which the outlier channels (|x| up to ~40) turn into absolute errors above
    # the output tolerance; bound each channel by 2^-8 of its largest magnitude
    # on top of the usual tolerance
    ref = oracle_rows(prob, rows)
    got = o_lat.cpu().numpy().astype(np.float64)
    for b in rows:
        c, p = prob.sequence(b)
        C, _ = O.dequantized_tokens(fmt, synth.bf16_bits_to_f32(c), synth.bf16_bits_to_f32(p))
        bound = 2e-2 + 1e-2 * np.abs(ref[b][1]) + 2.0 ** -8 * np.max(np.abs(C), axis=0)[None, :]
        err = np.abs(got[b] - ref[b][1])
        assert np.all(err <= bound), f"o_lat[{b}]: worst excess {np.max(err - bound):.3e}"
    empty = seqlens.index(0)
    assert torch.count_nonzero(dev.out[empty]) == 0


@pytest.mark.parametrize("fmt", ["int8", "int4"])
def test_decode_v3_quant_full(fmt):
    """H=128, B=64, seqlen 32768, random page table, quantized pool: every row
    against the oracle over the dequantized values."""
    prob = problem_from_workload(synth.get_workload("v3_quant"), fmt=fmt)
    dev = DeviceDecode(prob)
    dev.decode()
    torch.cuda.synchronize()
    _status_ok()
    _check_all_rows(dev)


# ----------------------------------------------------------------------------
# invariants of the result
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("H", [16, 128])
def test_decode_split_count_invariance(H):
    """The same rows decoded with 1, a few and the default number of split
    workers (so with different cut points, partial counts and merges): each
    result within tolerance of the oracle, and all within tolerance of the
    default plan's."""
    import mla_absorbed_latent_gb300 as mla
    seqlens = [4000, 1, 777, 64, 2049, 0, 130, 9000, 65]
    prob = make_problem(H, seqlens, seed=50 + H)
    dev = DeviceDecode(prob)
    wmax = mla.mla_decode_max_workers(H, "bf16")
    ref = oracle_outputs(prob, [b for b, n in enumerate(seqlens) if n > 0])
    outs = {}
    for w in sorted({1, 3, 37 % wmax or 1, wmax}):
        mla.mla_decode_plan_workers(H, "bf16", dev.seqlens, prob.B, prob.max_pages, w, dev.workspace, dev.ws_bytes)
        mla.mla_decode_absorb_q(dev.q_nope, dev.q_pe, dev.W_UK, H, prob.B, dev.workspace, dev.ws_bytes)
        mla.mla_decode_attend(H, dev.cache, dev.page_table, prob.max_pages, dev.seqlens, prob.B, prob.scale,
                              dev.workspace, dev.ws_bytes)
        mla.mla_decode_combine(dev.W_UV, H, prob.B, dev.workspace, dev.ws_bytes, dev.out)
        torch.cuda.synchronize()
        _status_ok()
        outs[w] = _out_f64(dev.out)
        for b in ref:
            assert_close(outs[w][b], ref[b], what=f"W={w} out[{b}]")
        assert not outs[w][seqlens.index(0)].any()
    for w in outs:
        assert_close(outs[w], outs[wmax], what=f"W={w} vs W={wmax}")
    with pytest.raises(mla.MLAError):
        mla.mla_decode_plan_workers(H, "bf16", dev.seqlens, prob.B, prob.max_pages, wmax + 1, dev.workspace,
                                    dev.ws_bytes)


@pytest.mark.parametrize("B", [20, 37, 65])
def test_decode_h128_merge_row_groups(B):
    """H=128 batches that pick each shape of the merge kernel (16 rows per CTA at
    B=20, 64 rows at B=37 with padding rows past the batch, 32 rows at B=65 with a
    partial last group), seeded lengths from 0 to 2,000 tokens with an empty row
    and a one-token row: out and o_lat of every row against the oracle."""
    rng = np.random.default_rng(400 + B)
    seqlens = [int(n) for n in rng.integers(1, 2000, size=B)]
    seqlens[3], seqlens[B // 2] = 0, 1
    prob = make_problem(128, seqlens, seed=400 + B)
    dev = DeviceDecode(prob)
    o_lat = torch.full((prob.B, 128, 512), float("nan"), dtype=torch.float32, device="cuda")
    dev.workspace.fill_(0xFF)
    dev.decode_steps(o_lat)
    torch.cuda.synchronize()
    _status_ok()
    rows = [b for b, n in enumerate(seqlens) if n > 0]
    ref = oracle_rows(prob, rows)
    got = _out_f64(dev.out)
    lat = o_lat.cpu().numpy().astype(np.float64)
    for b in rows:
        assert_close(got[b], ref[b][0], what=f"out[{b}]")
        assert_close(lat[b], ref[b][1], what=f"o_lat[{b}]")
    assert torch.count_nonzero(dev.out[3]) == 0


def test_decode_row_independence():
    """H=128: a row's output does not depend on the other rows.  Changing every
    other row's queries and cache contents (lengths kept, so the split plan is
    the same) leaves row 2's output bit for bit; changing the other rows'
    lengths (a different plan) keeps it within tolerance of the oracle."""
    import mla_absorbed_latent_gb300 as mla
    seqlens = [3000, 500, 5000, 64, 1200, 7]
    prob = make_problem(128, seqlens, seed=61)
    dev = DeviceDecode(prob)
    a = dev.decode().clone()
    torch.cuda.synchronize()
    # other rows: new queries and new cache contents
    g = torch.Generator(device="cuda").manual_seed(5)
    others = [b for b in range(prob.B) if b != 2]
    for b in others:
        dev.q_nope[b] = torch.randn((128, 128), generator=g, device="cuda").to(torch.bfloat16)
        dev.q_pe[b] = torch.randn((128, 64), generator=g, device="cuda").to(torch.bfloat16)
        for j in range((seqlens[b] + 63) // 64):
            pg = int(dev.page_table[b, j])
            vals = torch.randn(64 * 576, generator=g, device="cuda").to(torch.bfloat16)
            dev.pool[pg * dev.page_bytes:(pg + 1) * dev.page_bytes] = vals.view(torch.uint8)
    b_ = dev.decode().clone()
    torch.cuda.synchronize()
    _status_ok()
    assert torch.equal(a[2], b_[2])
    assert not torch.equal(a[0], b_[0])
    # other rows' lengths change (within their allocated pages): a different plan,
    # row 2 still matches the oracle
    lens = torch.tensor([100, 200, 5000, 1, 64, 3], dtype=torch.int32, device="cuda")
    mla.mla_decode(dev.q_nope, dev.q_pe, dev.W_UK, dev.W_UV, 128, dev.cache, dev.page_table, prob.max_pages, lens,
                   prob.B, prob.scale, dev.workspace, dev.ws_bytes, dev.out)
    torch.cuda.synchronize()
    _status_ok()
    _check_rows(dev, [2])


@pytest.mark.parametrize("H", [16, 128])
def test_decode_nan_workspace(H):
    """A workspace filled with all-ones bytes (NaN in bf16 and fp32) before the
    decode: every value the decode reads from it must have been written by the
    same call (an unwritten partial or flag would show up as NaN or a wrong
    row).  Ragged lengths with an empty row, against the oracle."""
    seqlens = [1, 31, 64, 65, 0, 700, 129, 2000]
    prob = make_problem(H, seqlens, seed=70 + H)
    dev = DeviceDecode(prob)
    dev.workspace.fill_(0xFF)
    o_lat = torch.full((prob.B, H, 512), float("nan"), dtype=torch.float32, device="cuda")
    dev.decode_steps(o_lat)
    torch.cuda.synchronize()
    _status_ok()
    rows = [b for b, n in enumerate(seqlens) if n > 0]
    _check_rows(dev, rows, o_lat)
    assert torch.count_nonzero(dev.out[seqlens.index(0)]) == 0
    assert torch.count_nonzero(o_lat[seqlens.index(0)]) == 0


def test_decode_bad_page_id_reports_bounds():
    import mla_absorbed_latent_gb300 as mla
    prob = make_problem(16, [100], seed=4)
    dev = DeviceDecode(prob)
    dev.page_table[0, 1] = prob.num_pages + 100
    dev.decode()
    st, info = mla.mla_get_device_status()
    assert st == mla.MLA_ERR_BOUNDS and info == prob.num_pages + 100


def test_bounded_wait_times_out_and_reports():
    """The failure path of the decode kernel's bounded waits, run out on
    purpose with no fault: in a CTA pair, CTA 0 waits on a barrier that nothing
    completes; after the limit (about 2 s) it records MLA_ERR_TIMEOUT (detail 1,
    CTA 0's) and raises both abort flags, and CTA 1 leaves its later wait
    through its flag without a report of its own.  Afterwards the context still
    decodes correctly (an H=128 case through the tcgen05 kernel)."""
    import time
    import mla_absorbed_latent_gb300 as mla
    _status_ok()
    t0 = time.time()
    mla.mla_wait_selftest()
    st, info = mla.mla_get_device_status()
    assert st == mla.MLA_ERR_TIMEOUT and info == 1, (mla.mla_status_string(st), info)
    assert time.time() - t0 < 60
    prob = make_problem(128, [300, 64, 1], seed=12)
    dev = DeviceDecode(prob)
    o_lat = torch.empty((prob.B, 128, 512), dtype=torch.float32, device="cuda")
    dev.decode_steps(o_lat)
    torch.cuda.synchronize()
    _status_ok()
    _check_rows(dev, list(range(prob.B)), o_lat)


def _boost_rope_keys(dev, prob, boosts):
    """Replace the RoPE keys of (head, token, lam) triples of row 0 by lam x that
    head's q_pe (in the pool, and in the returned fp64 values the oracle reads);
    each such token's score for that head rises by about lam x 6.7 log2 units."""
    qp = synth.bf16_bits_to_f32(prob.q_pe)
    c, p = prob.sequence(0)
    C, P = synth.bf16_bits_to_f32(c), synth.bf16_bits_to_f32(p)
    for head, token, lam in boosts:
        bits = synth.f32_to_bf16_bits((lam * qp[0, head]).astype(np.float32))
        P[token] = synth.bf16_bits_to_f32(bits)
        page, slot = divmod(token, 64)
        off = int(dev.page_table[0, page]) * dev.page_bytes + slot * 1152 + 1024  # the token's k_pe (bf16 pool)
        dev.pool[off:off + 128] = torch.from_numpy(bits.view(np.uint8).copy()).to(dev.pool.device)
    return C, P


def _check_boosted_row(dev, prob, C, P, o_lat=None):
    import mla_absorbed_latent_gb300 as mla
    st, info = mla.mla_get_device_status()
    assert st == mla.MLA_OK, (mla.mla_status_string(st), info)
    qn = synth.bf16_bits_to_f32(prob.q_nope)
    qp = synth.bf16_bits_to_f32(prob.q_pe)
    Wuk, Wuv = weights(prob)
    ref_out, ref_lat, _ = O.absorbed_decode(qn[0], qp[0], C, P, Wuk, Wuv, prob.scale)
    assert_close(_out_f64(dev.out)[0], ref_out)
    if o_lat is not None:
        assert_close(o_lat[0].cpu().numpy(), ref_lat, what="o_lat")


def test_decode_score_beyond_tracked_range_is_exact():
    """H=128: a token of the second page whose RoPE key is 200 x one head's
    q_pe raises that head's score about 1,300 log2 units above the first
    page's maximum, far past the 2^100 the fast path can weight in its running
    reference; the row is recomputed exactly and must match the oracle (all
    heads, out and o_lat).  The row is long enough (304 pages) that the first
    worker's range holds several pages, so page 1 is not the first page of its
    split."""
    prob = make_problem(128, [64 * 304], seed=6, paged=False)
    dev = DeviceDecode(prob)
    C, P = _boost_rope_keys(dev, prob, [(0, 64, 200.0)])
    o_lat = torch.empty((1, 128, 512), dtype=torch.float32, device="cuda")
    dev.decode_steps(o_lat)
    torch.cuda.synchronize()
    _check_boosted_row(dev, prob, C, P, o_lat)


def test_decode_large_half_scores_are_exact():
    """H=128, paged: RoPE keys 12 x a head's q_pe (about 80 log2 units above the
    rest, within the tracked range) make the half scores the CTA pair exchanges
    exceed what fp16 carries to 2^-7; the row is recomputed exactly.  Two
    further rows stay on the fast path and must still match."""
    prob = make_problem(128, [64 * 40, 777, 64 * 9], seed=8)
    dev = DeviceDecode(prob)
    C, P = _boost_rope_keys(dev, prob, [(3, 64 * 5 + 7, 12.0), (100, 64 * 30 + 63, 12.0), (3, 2000, -12.0)])
    dev.decode()
    torch.cuda.synchronize()
    _check_boosted_row(dev, prob, C, P)
    _check_rows(dev, [1, 2])


@pytest.mark.parametrize("fmt", ["int8", "int4", "int8_token", "int4_sym", "int4_pe4"])
def test_decode_quant_range_jump_is_exact(fmt):
    """H=128 over quantized pools: one token's RoPE key (in its INT8 k_pe codes)
    turned into 127 x sign(q_pe) of one head, scale 2, so that head's score jumps
    far past the tracked range; the exact recompute reads the quantized page
    (codes, scales, zeros) and must match the oracle over the dequantized
    values."""
    prob = make_problem(128, [64 * 150, 300], seed=33, fmt=fmt, dist="outlier")
    dev = DeviceDecode(prob)
    import mla_absorbed_latent_gb300 as mla
    qp = synth.bf16_bits_to_f32(prob.q_pe)[0, 5]
    token = 64 * 3 + 9
    page, slot = divmod(token, 64)
    base = int(dev.page_table[0, page]) * dev.page_bytes
    pe_code, pe_scale = (32768, 38912) if fmt.startswith("int8") else (16384, 24576)
    codes = np.where(qp >= 0, 127, -127).astype(np.int8)
    dev.pool[base + pe_code + slot * 64: base + pe_code + slot * 64 + 64] = torch.from_numpy(
        codes.view(np.uint8).copy()).cuda()
    scale_bits = synth.f32_to_bf16_bits(np.full(8, 2.0, np.float32))
    dev.pool[base + pe_scale + slot * 16: base + pe_scale + slot * 16 + 16] = torch.from_numpy(
        scale_bits.view(np.uint8).copy()).cuda()
    dev.decode()
    torch.cuda.synchronize()
    st, info = mla.mla_get_device_status()
    assert st == mla.MLA_OK, (mla.mla_status_string(st), info)
    # the oracle over the dequantized values, with that token's RoPE key replaced
    c, p = prob.sequence(0)
    Cq, Pq = O.dequantized_tokens(fmt, synth.bf16_bits_to_f32(c), synth.bf16_bits_to_f32(p))
    Pq = Pq.copy()
    Pq[token] = codes.astype(np.float64) * 2.0
    qn = synth.bf16_bits_to_f32(prob.q_nope)
    Wuk, Wuv = weights(prob)
    ref = O.absorbed_decode(qn[0], synth.bf16_bits_to_f32(prob.q_pe)[0], Cq, Pq, Wuk, Wuv, prob.scale)[0]
    assert_close(_out_f64(dev.out)[0], ref)
    _check_rows(dev, [1])


def test_decode_reference_moves_keep_the_result_exact():
    """H=128: tokens of later pages whose RoPE keys are 3x one head's q_pe lift
    that head's scores by about 20 log2 units over the first page's maximum, so
    the kernel moves its running reference (rescaling O) while staying inside
    both its tracked range and the fp16 exchange bound (the fast path); the
    output must still match the oracle on the same modified cache."""
    n = 64 * 304
    prob = make_problem(128, [n], seed=7, paged=False)
    dev = DeviceDecode(prob)
    C, P = _boost_rope_keys(dev, prob, [(0, 64 * 3 + 5, 3.0), (1, 64 * 9 + 40, 3.0), (0, 64 * 40 + 1, 5.0)])
    dev.decode()
    torch.cuda.synchronize()
    _check_boosted_row(dev, prob, C, P)


def test_decode_reference_move_on_a_second_to_last_page_is_exact():
    """H=128, one 304-page row over the default split: a boosted token on the
    second-to-last page of a worker's range moves that split's reference at
    the check made during its last page, after the split's slice sums were
    sent.  The split's log-sum-exp must be taken in the moved reference, or
    the merge overweights the split by the size of the move.  Head 0 also
    gets a larger boost on the first page of another worker's range (the true
    maximum of the row), head 2 only the second-to-last-page one."""
    import mla_absorbed_latent_gb300 as mla
    n_pages = 304
    prob = make_problem(128, [64 * n_pages], seed=9, paged=False)
    dev = DeviceDecode(prob)
    W = mla.mla_decode_max_workers(128, "bf16")
    begin = [w * n_pages // W for w in range(W + 1)]  # the default plan's equal split of the pages
    assert begin[2] - begin[1] >= 3 and begin[6] - begin[5] >= 3 and W > 10
    C, P = _boost_rope_keys(dev, prob, [(0, 64 * (begin[2] - 2) + 5, 3.0), (0, 64 * begin[10] + 7, 4.0),
                                        (2, 64 * (begin[6] - 2) + 33, 3.0)])
    dev.decode()
    torch.cuda.synchronize()
    _check_boosted_row(dev, prob, C, P)


def test_decode_seqlen_over_capacity_reports_bounds():
    import mla_absorbed_latent_gb300 as mla
    prob = make_problem(16, [100], seed=4)
    dev = DeviceDecode(prob)
    dev.seqlens[0] = 64 * prob.max_pages + 1
    dev.decode()
    st, info = mla.mla_get_device_status()
    assert st == mla.MLA_ERR_BOUNDS and info == 0


def test_workspace_too_small_is_rejected():
    import mla_absorbed_latent_gb300 as mla
    prob = make_problem(16, [10], seed=4)
    dev = DeviceDecode(prob)
    with pytest.raises(mla.MLAError) as e:
        mla.mla_decode(dev.q_nope, dev.q_pe, dev.W_UK, dev.W_UV, 16, dev.cache, dev.page_table, prob.max_pages,
                       dev.seqlens, 1, prob.scale, dev.workspace, dev.ws_bytes - 1, dev.out)
    assert e.value.status == mla.MLA_ERR_WORKSPACE


def test_decode_h128_garbage_past_row_end_is_ignored():
    """H=128 over bf16 pages: the slots past each row's length in its last page
    hold all-ones bytes (NaN in bf16).  They are neither keys nor values of the
    row: the tensor-core kernel multiplies whole 64-token pages, so it masks
    their scores and zeroes their value rows before the page's P.V."""
    seqlens = [1, 33, 63, 100, 129, 2000]
    prob = make_problem(128, seqlens, seed=123)
    dev = DeviceDecode(prob)
    for b, n in enumerate(seqlens):
        last = (n - 1) // 64
        page = int(dev.page_table[b, last])
        lo = page * dev.page_bytes + (n - 64 * last) * 1152  # the first slot past the row's end
        dev.pool[lo:(page + 1) * dev.page_bytes] = 0xFF
    dev.decode()
    torch.cuda.synchronize()
    _status_ok()
    _check_rows(dev, range(prob.B))
