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


def _oracle_rows_task(args):
    prob, rows = args
    return {b: r[0] for b, r in oracle_rows(prob, rows).items()}


def oracle_outputs(prob, rows, procs: int | None = None):
    """{b: out [H,128]} of the fp64 oracle for many rows, computed by a pool of
    spawned worker processes (spawn: the parent may already hold a CUDA
    context), each with single-threaded BLAS."""
    import concurrent.futures as cf
    import multiprocessing as mp
    import os
    rows = list(rows)
    procs = procs or max(1, min(len(rows), (os.cpu_count() or 2) - 1, 16))
    if procs == 1 or len(rows) <= 2:
        return _oracle_rows_task((prob, rows))
    chunks = [rows[i::procs] for i in range(procs)]
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"  # inherited by the spawned workers
    try:
        with cf.ProcessPoolExecutor(max_workers=procs, mp_context=mp.get_context("spawn")) as ex:
            res = {}
            for part in ex.map(_oracle_rows_task, [(prob, c) for c in chunks if c]):
                res.update(part)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
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
