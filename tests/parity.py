"""Shared helpers of the parity tests: oracle outputs for a Problem and the
tolerance checks (abs 2e-2 + rel 1e-2 elementwise, plus rel-RMS and cosine,
because at long context the outputs are small enough that the elementwise
bound alone would accept an all-zero result)."""

from __future__ import annotations

import numpy as np

import oracle as O
import synth

ATOL, RTOL = 2e-2, 1e-2
REL_RMS = 1e-2
COSINE = 0.9999


def weights(prob):
    return O.split_wkv_b(synth.bf16_bits_to_f32(prob.wkv), prob.H)


def oracle_rows(prob, rows, W=None):
    """{b: (out [H,128], o_lat [H,512], lse [H])} from the fp64 absorbed oracle,
    over the values the cache format stores (dequantized for INT8/INT4)."""
    Wuk, Wuv = W if W is not None else weights(prob)
    qn = synth.bf16_bits_to_f32(prob.q_nope)
    qp = synth.bf16_bits_to_f32(prob.q_pe)
    res = {}
    for b in rows:
        c, p = prob.sequence(b)
        C, P = O.dequantized_tokens(prob.fmt, synth.bf16_bits_to_f32(c), synth.bf16_bits_to_f32(p))
        res[b] = O.absorbed_decode(qn[b], qp[b], C, P, Wuk, Wuv, prob.scale)
    return res


def assert_close(got, ref, what="out"):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements out of tolerance, max err {err.max():.3e}"
    rows_ref = ref.reshape(-1, ref.shape[-1])
    rows_err = (got - ref).reshape(-1, ref.shape[-1])
    nref = np.linalg.norm(rows_ref, axis=1)
    rel = np.linalg.norm(rows_err, axis=1) / np.maximum(nref, 1e-30)
    live = nref > 0
    assert np.all(rel[live] <= REL_RMS), f"{what}: worst row rel-RMS {rel[live].max():.3e}"
    assert np.all(np.abs(rows_err[~live]) <= ATOL)
    if np.linalg.norm(ref) > 0:
        cos = float(np.sum(got * ref) / (np.linalg.norm(got) * np.linalg.norm(ref)))
        assert cos >= COSINE, f"{what}: cosine {cos}"
    return float(err.max()), float(rel[live].max()) if live.any() else 0.0
