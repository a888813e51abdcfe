"""The seeded synthetic input generators (no GPU needed)."""
import math

import numpy as np
import pytest

from update_merged_table_gb300 import workloads as W


@pytest.mark.parametrize("s,V", [(1.1, 50), (0.8, 30), (1.3, 200), (1.05, 1000)])
def test_zipf_pmf_chi_square(s, V):
    """Frequencies of the rejection-inversion sampler against the exact pmf k^-s / H(V, s)."""
    rng = np.random.default_rng(int(s * 100) + V)
    n = 300_000
    k = W.zipf_ranks(rng, n, s, V)
    assert k.min() >= 1 and k.max() <= V
    p = np.arange(1, V + 1, dtype=np.float64) ** -s
    p /= p.sum()
    obs = np.bincount(k, minlength=V + 1)[1:]
    exp = n * p
    keep = exp >= 5
    chi2 = ((obs[keep] - exp[keep]) ** 2 / exp[keep]).sum() + \
        ((obs[~keep].sum() - exp[~keep].sum()) ** 2 / max(exp[~keep].sum(), 1e-9) if (~keep).any() else 0.0)
    dof = keep.sum() + (1 if (~keep).any() else 0) - 1
    # mean + 5 standard deviations of chi-square(dof)
    assert chi2 < dof + 5 * math.sqrt(2 * dof), (chi2, dof)


def test_zipf_large_vocab_head():
    """Over 2^32 ranks the head probabilities still follow k^-s."""
    rng = np.random.default_rng(1)
    s, V, n = 1.05, 1 << 32, 400_000
    k = W.zipf_ranks(rng, n, s, V)
    H = sum(j ** -s for j in range(1, 10 ** 6)) + ((V + 0.5) ** (1 - s) - (10 ** 6 - 0.5) ** (1 - s)) / (1 - s)
    for r in (1, 2, 5):
        want = n * r ** -s / H
        assert abs((k == r).sum() - want) < 6 * math.sqrt(want)


def test_bijection32_is_injective():
    x = np.arange(1 << 20, dtype=np.int64)
    y = W.bijection32(x)
    assert np.unique(y).size == x.size
    assert y.min() >= 0 and y.max() < (1 << 32)


def test_jagged_batch_shape():
    b = W.jagged_batch(0, users=256)
    lens = np.diff(b.user_offsets)
    assert lens.min() >= 1 and lens.max() <= 3000
    T = int(lens.sum())
    assert b.n == 4 * T and b.feat_offsets.tolist() == [0, T, 2 * T, 3 * T, 4 * T]
    assert b.table_ids.tolist() == [0, 1, 2, 3]
    assert b.ids.min() >= 0 and b.ids.max() < 1_000_000


def test_jagged_lengths_moments():
    lens = W.jagged_lengths(0, users=20000, cap=10 ** 9)
    # log of floor(lognormal(5, 1)) is close to N(5, 1) for values well above 1
    lg = np.log(lens[lens > 20])
    assert abs(np.median(np.log(lens)) - 5.0) < 0.05
    assert 0.8 < lg.std() < 1.1


def test_merged_batch():
    b = W.merged_batch(0, per_table=1024)
    assert b.n == 8 * 1024
    for k in range(8):
        seg = b.ids[b.feat_offsets[k]:b.feat_offsets[k + 1]]
        assert seg.max() < W.merged_vocab(k)
    assert W.merged_vocab(0) == 10_000 and W.merged_vocab(7) == 1_000_000
    assert W.merged_exponent(0) == 0.8 and abs(W.merged_exponent(7) - 1.3) < 1e-12


def test_churn_stream_fresh_ids():
    cs = W.ChurnStream(0, hot=1 << 12, n=1 << 10, erase=1 << 8)
    b0, e0 = cs.step(0)
    b1, e1 = cs.step(1)
    fresh0 = b0.ids[b0.ids >= (1 << 12)]
    fresh1 = b1.ids[b1.ids >= (1 << 12)]
    assert fresh0.size == round(0.1 * (1 << 10)) and np.intersect1d(fresh0, fresh1).size == 0
    assert e1.max() < cs.next_fresh


def test_churn_erases_only_live_ids():
    """The erase set of each step is distinct and drawn from the IDs live after that step's lookup:
    the prefill, plus every ID handed out, minus every ID erased and not handed out again."""
    hot = 1 << 12
    cs = W.ChurnStream(1, hot=hot, n=1 << 10, erase=1 << 9)
    live = set(range(hot))
    for k in range(6):
        b, er = cs.step(k)
        live.update(b.ids.tolist())
        assert er.size == 1 << 9 and np.unique(er).size == er.size
        assert all(int(x) in live for x in er)
        live.difference_update(er.tolist())
        assert set(cs.live_ids().tolist()) == live
    with pytest.raises(ValueError):
        cs.step(9)  # steps are taken in order


def test_batches_are_deterministic():
    a = W.merged_batch(3, per_table=256)
    b = W.merged_batch(3, per_table=256)
    assert np.array_equal(a.ids, b.ids)
    assert np.array_equal(W.grads_normal(1, 10, 4), W.grads_normal(1, 10, 4))
