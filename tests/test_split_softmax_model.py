"""A model, in fp64 numpy, of the per-head softmax bookkeeping of the 128-head
tensor-core attend kernel, checked against the exact softmax.

The kernel splits each row's pages among workers (one split per worker and
row) and keeps a lazily moved reference maximum per head: a split's first page
takes the exact page maximum; the check of page j runs at the end of page j+1
and moves the reference (rescaling O and l) only when page j's maximum exceeded
it by more than 2^8; at a split's last page the slice sums are sent before the
check of the page before it, so that check's move reaches them as a factor.
Each split emits O / L and its log-sum-exp, and the merge weights the splits by
their log-sum-exps ("DeepSeek MLA 吸收式缓存" §2.3 and the online softmax it
rests on).  The merged result is exact for any plan and any scores; the case
that needs care is a move made by a split's second-to-last page, whose
log-sum-exp must be taken in the moved reference.  No GPU: the model restates
the bookkeeping, the kernel's own parity is checked by the GPU tests.
"""

import numpy as np
import pytest

RESCALE_LOG2 = 8.0


def _splits(rows, ranges, s, V, lse_in_moved_reference=True):
    """Per row, the (O / L, log2-sum-exp) of each split, as the kernel forms them.

    rows: pages per row; ranges: per worker its global page range [x0, x1);
    s[x]: the log2-domain scores of global page x; V[x]: its values."""
    starts = np.concatenate([[0], np.cumsum(rows)])
    out = {b: [] for b in range(len(rows))}
    for x0, x1 in ranges:
        m_ref, l, alpha_prev = -np.inf, 0.0, 1.0
        O = {}  # per row of this worker: its split's accumulator
        pend = None  # (page, last, row, reference after the previous check, message)
        for x in range(x0, x1 + 1):
            if x < x1:
                b = int(np.searchsorted(starts, x, side="right") - 1)
                first = x == x0 or x == starts[b]
                last = x + 1 == x1 or x + 1 == starts[b + 1]
                mraw = s[x].max()
                if first:
                    m_ref, l, O[b] = mraw, 0.0, np.zeros(V[x].shape[1])
                p = np.exp2(s[x] - m_ref)
                l += p.sum()
                msg = l if last else mraw  # a page's message: its maximum, or the sum at a split's end
                O[b] = O[b] + p @ V[x]
            if pend is not None:  # the check of the page before, at the end of this one
                j, j_last, jb, ref_j, msg_j = pend
                if not j_last:
                    alpha = 1.0
                    if msg_j > ref_j + RESCALE_LOG2:
                        m_new = max(msg_j, m_ref)
                        alpha = np.exp2(m_ref - m_new)
                        l *= alpha
                        m_ref = m_new
                    alpha_prev = alpha
                    O[jb] = O[jb] * alpha  # pages <= j + 1, all of row jb
                else:
                    L = alpha_prev * msg_j
                    alpha_prev = 1.0
                    lse = ref_j + np.log2(L if lse_in_moved_reference else msg_j)
                    out[jb].append((O[jb] / L, lse))
            if x == x1:
                break
            pend = (x, last, b, m_ref, msg)
    return out


def _merge(splits):
    lse = np.array([g[1] for g in splits])
    w = np.exp2(lse - lse.max())
    w /= w.sum()
    return sum(wi * g[0] for wi, g in zip(w, splits))


def _exact(s, V):
    s = np.concatenate(s)
    V = np.concatenate(V)
    p = np.exp2(s - s.max())
    return (p / p.sum()) @ V


def _uniform(T, W):
    return [(w * T // W, (w + 1) * T // W) for w in range(W)]


def _single_page_first(T, W):
    # a plan whose first worker holds one page (a split start charged as 3 pages)
    ctot = T + 3
    b = [max(0, (w * ctot) // W - 3) for w in range(W)] + [T]
    return [(b[w], b[w + 1]) for w in range(W)]


def _problem(rows, boosts, seed):
    rng = np.random.default_rng(seed)
    T = int(sum(rows))
    s = [rng.normal(0.0, 1.0, 64) for _ in range(T)]
    V = [rng.normal(0.0, 1.0, (64, 8)) for _ in range(T)]
    for page, slot, add in boosts:
        s[page][slot] += add
    return s, V


def _max_rel_err(rows, ranges, s, V, **kw):
    starts = np.concatenate([[0], np.cumsum(rows)])
    splits = _splits(rows, ranges, s, V, **kw)
    err = 0.0
    for b in range(len(rows)):
        if rows[b] == 0:
            continue
        ref = _exact(s[starts[b]:starts[b + 1]], V[starts[b]:starts[b + 1]])
        err = max(err, np.linalg.norm(_merge(splits[b]) - ref) / np.linalg.norm(ref))
    return err


@pytest.mark.parametrize("plan", ["uniform76", "uniform37", "uniform33", "single_page_first"])
def test_moves_anywhere_in_a_split_keep_the_merge_exact(plan):
    T = 304
    ranges = {"uniform76": _uniform(T, 76), "uniform37": _uniform(T, 37), "uniform33": _uniform(T, 33),
              "single_page_first": _single_page_first(T, 76)}[plan]
    # a move on every page position of some split: first, middle, second-to-last, last
    for seed, boosts in enumerate([[(3, 5, 20.0), (40, 1, 33.0)], [(9, 40, 20.0)], [(6, 3, 20.0), (40, 7, 27.0)],
                                   [(p, 0, 12.0 + (p % 5)) for p in range(2, T, 7)]]):
        s, V = _problem([T], boosts, seed)
        assert _max_rel_err([T], ranges, s, V) < 1e-12, (plan, boosts)


def test_ragged_rows_with_moves_keep_the_merge_exact():
    rng = np.random.default_rng(5)
    rows = [int(v) for v in rng.integers(0, 40, 23)]
    T = sum(rows)
    for W in (1, 3, 19, 76):
        s, V = _problem(rows, [(int(p), int(p) % 64, 15.0) for p in rng.integers(0, T, 30)], W)
        assert _max_rel_err(rows, _uniform(T, W), s, V) < 1e-12, W


def test_lse_before_the_move_overweights_the_split():
    # the planted mistake: the log-sum-exp of the sums sent before the check of
    # the second-to-last page, in the moved reference
    T = 304
    ranges = _uniform(T, 76)  # worker 1 holds pages 4..7: page 6 is its second-to-last
    s, V = _problem([T], [(6, 3, 20.0), (40, 7, 27.0)], 2)
    assert _max_rel_err([T], ranges, s, V) < 1e-12
    assert _max_rel_err([T], ranges, s, V, lse_in_moved_reference=False) > 0.5
    s, V = _problem([T], [(5, 3, 20.0)], 2)  # page 5: a middle page, not the second-to-last
    assert _max_rel_err([T], ranges, s, V, lse_in_moved_reference=False) < 1e-12
