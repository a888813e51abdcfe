"""Pooled bags of a jagged batch on the GPU (through the C ABI) against the oracle.

A bag is one user's tokens of one feature of the jagged sequence batch; its
pooled embedding is the sum or mean of its rows.  The pooled backward hands
each position its bag's gradient and feeds the per-unique reduction and Adam
without per-position gradient rows.  Pooled rows and gradient sums are
compared within 1e-5 relative + 1e-6 absolute (both sides round an exact sum
once); Adam-updated bf16 rows within one bf16 ulp.
"""
import numpy as np
import pytest
import torch

import oracle
import update_merged_table_gb300 as mt
from update_merged_table_gb300 import workloads as W
from numerics import ATOL, RTOL, assert_rows_close  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from update_merged_table_gb300 import build_lib
    build_lib.build()
    mt.load_library()
    oracle.build()


def dev():
    return torch.device("cuda", torch.cuda.current_device())


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def jagged_bags(b):
    """Bag offsets of a feature-major jagged batch: feature f, user u -> positions f*T + [uo[u], uo[u+1])."""
    T = int(b.user_offsets[-1])
    F = b.feat_offsets.size - 1
    return np.concatenate([f * T + b.user_offsets[:-1] for f in range(F)] + [[F * T]]).astype(np.int64)


def pooled_step(tab, ref, b, bo, mode, seed, row_dtype, check_rows=True):
    res = tab.lookup(to_dev(b.ids), b.feat_offsets, b.table_ids, gather=False)
    ref.lookup(b.ids, b.feat_offsets, b.table_ids, gather=False)
    got = tab.pool_forward(res, to_dev(bo), mode=mode).cpu().numpy()
    want = ref.pool_forward(bo, mode=1 if mode == "mean" else 0)
    np.testing.assert_allclose(got, want, rtol=RTOL, atol=ATOL)
    B = bo.size - 1
    dp = np.random.default_rng(seed).standard_normal((B, tab.dim), dtype=np.float32)
    gsum = tab.backward_adam_pooled(res, to_dev(bo), to_dev(dp), mode=mode, want_gsum=True)
    ref_gsum = ref.backward_adam_pooled(bo, dp, mode=1 if mode == "mean" else 0, want_gsum=True)
    U = res.U
    np.testing.assert_allclose(gsum[:U].cpu().numpy(), ref_gsum, rtol=RTOL, atol=ATOL)
    if check_rows:
        emb, m, v = tab.read_rows(res.unique_rows[:U])
        e2, m2, v2, pr = ref.get_rows(res.unique_keys[:U].cpu().numpy().view(np.uint64))
        assert pr.all()
        assert_rows_close(emb.cpu().numpy(), e2, row_dtype)
        np.testing.assert_allclose(m.cpu().numpy(), m2, rtol=RTOL, atol=ATOL)
        np.testing.assert_allclose(v.cpu().numpy(), v2, rtol=RTOL, atol=1e-9)
    assert tab.error() == 0 and ref.error == 0
    return res


@pytest.mark.parametrize("mode", ["sum", "mean"])
def test_pooled_jagged_bf16(mode):
    """96 users, 4 features, dim 64 bf16 rows: pooled forward and backward over three steps."""
    tab = mt.Table(18, 64, row_dtype="bf16")
    ref = oracle.Table(18, 64, row_dtype=oracle.BF16)
    for s in range(3):
        b = W.jagged_batch(s, users=96)
        pooled_step(tab, ref, b, jagged_bags(b), mode, 70 + s, "bf16")


def test_pooled_fp32_edge_bags():
    """Empty bags, positions before the first and after the last bag, one-position bags, one bag over many
    chunks, and invalid IDs."""
    rng = np.random.default_rng(5)
    ids = rng.integers(0, 500, size=5000).astype(np.int64)
    ids[[7, 4000]] = -3  # invalid: no row, no gradient
    bo = np.array([10, 10, 11, 12, 75, 75, 64 * 40 + 3, 4000, 4001, 4990, 4990], np.int64)
    tab = mt.Table(12, 16)
    ref = oracle.Table(12, 16)
    b = W.single_feature(ids)
    for mode in ("sum", "mean"):
        res = tab.lookup(to_dev(b.ids), gather=False)
        ref.lookup(b.ids, gather=False)
        got = tab.pool_forward(res, to_dev(bo), mode=mode).cpu().numpy()
        want = ref.pool_forward(bo, mode=1 if mode == "mean" else 0)
        np.testing.assert_allclose(got, want, rtol=RTOL, atol=ATOL)
        assert not got[0].any() and not got[4].any() and not got[9].any()  # empty bags
        dp = rng.standard_normal((bo.size - 1, 16), dtype=np.float32)
        gsum = tab.backward_adam_pooled(res, to_dev(bo), to_dev(dp), mode=mode, want_gsum=True)
        ref_gsum = ref.backward_adam_pooled(bo, dp, mode=1 if mode == "mean" else 0, want_gsum=True)
        np.testing.assert_allclose(gsum[:res.U].cpu().numpy(), ref_gsum, rtol=RTOL, atol=ATOL)
        tab.error(clear=True)  # the invalid IDs latched MT_EKEY
        ref.error  # noqa: B018


@pytest.mark.parametrize("dim,row_dtype", [(16, "f32"), (64, "bf16")])
def test_pooled_many_small_and_empty_bags(dim, row_dtype):
    """Bags of 0 to 3 positions (far more than 32 bags meet one chunk, so the kernel walks several windows of
    offsets), runs of empty bags on chunk boundaries, bags that end exactly on a boundary, one long bag over
    several chunks and positions after the last bag, for sum and mean."""
    rng = np.random.default_rng(21)
    n = 3000
    ids = rng.integers(0, 700, size=n).astype(np.int64)
    lens = rng.choice([0, 0, 1, 2, 3], size=700)
    bo = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)  # ends near position 1050
    tail = bo[-1]
    extra = [128 * k for k in range(tail // 128 + 1, tail // 128 + 4) for _ in range(3)]  # empties on boundaries
    bo = np.concatenate([bo, np.maximum(extra, tail), [2000, 2000, 2600]]).astype(np.int64)
    assert (np.diff(bo) >= 0).all() and bo[-1] < n
    tab = mt.Table(13, dim, row_dtype=row_dtype)
    ref = oracle.Table(13, dim, row_dtype=oracle.BF16 if row_dtype == "bf16" else oracle.F32)
    b = W.single_feature(ids)
    res = tab.lookup(to_dev(b.ids), gather=False)
    ref.lookup(b.ids, gather=False)
    for mode in ("sum", "mean"):
        got = tab.pool_forward(res, to_dev(bo), mode=mode).cpu().numpy()
        want = ref.pool_forward(bo, mode=1 if mode == "mean" else 0)
        np.testing.assert_allclose(got, want, rtol=RTOL, atol=ATOL)
        assert not got[np.diff(bo) == 0].any()  # empty bags are zeros
    assert tab.error() == 0 and ref.error == 0


def test_pooled_backward_equals_expanded_backward():
    """The pooled backward (sum) equals the per-position backward fed the bag gradients expanded to their
    positions, bit for bit: the same rows are summed in the same order."""
    b = W.jagged_batch(3, users=128)
    bo = jagged_bags(b)
    B = bo.size - 1
    dp = np.random.default_rng(8).standard_normal((B, 32), dtype=np.float32)
    lens = np.diff(bo)
    expanded = np.repeat(dp, lens, axis=0)
    out = []
    for pooled in (True, False):
        tab = mt.Table(16, 32)
        res = tab.lookup(to_dev(b.ids), b.feat_offsets, b.table_ids, gather=False)
        if pooled:
            gs = tab.backward_adam_pooled(res, to_dev(bo), to_dev(dp), mode="sum", want_gsum=True)
        else:
            gs = tab.backward_adam(res, to_dev(expanded), want_gsum=True)
        emb, m, v = tab.read_rows(res.unique_rows[:res.U])
        out.append((gs[:res.U].cpu().numpy(), emb.cpu().numpy(), v.cpu().numpy()))
    for a, c in zip(out[0], out[1]):
        assert np.array_equal(a, c)


def test_pooled_invalid_offsets_latch_einval():
    """Decreasing offsets: the device latches MT_EINVAL and every access stays in bounds."""
    ids = np.arange(300, dtype=np.int64)
    tab = mt.Table(10, 8)
    res = tab.lookup(to_dev(ids), gather=False)
    bo = np.array([0, 200, 100, 300], np.int64)
    out = tab.pool_forward(res, to_dev(bo))
    torch.cuda.synchronize()
    assert tab.error() == mt.MT_EINVAL
    assert not out[1].any()  # the bad bag reads as zeros
    tab.error(clear=True)
    tab.backward_adam_pooled(res, to_dev(bo), torch.ones((3, 8), device=dev()))
    assert tab.error() == mt.MT_EINVAL


def test_full_size_pooled_jagged():
    """Full GRM jagged batch (2048 users, 4 features, ~2M IDs, M = 2^24, dim 64 bf16): mean pooling forward and
    backward on the cold step and one fresh step, every bag and every touched row compared."""
    tab = mt.Table(24, 64, row_dtype="bf16")
    ref = oracle.Table(24, 64, row_dtype=oracle.BF16)
    for s, mode in ((0, "mean"), (1, "sum")):
        b = W.jagged_batch(s)
        pooled_step(tab, ref, b, jagged_bags(b), mode, 90 + s, "bf16")


@pytest.mark.parametrize("dim,row_dtype", [(4, "f32"), (32, "bf16"), (128, "f32"), (512, "bf16"), (1024, "f32")])
def test_pooled_team_shapes(dim, row_dtype):
    """Row shapes that give every team size (4 to 32 lanes) and several column groups per lane (d = 512 bf16,
    d = 1024 fp32), on jagged bags with sum and mean pooling, against the oracle."""
    tab = mt.Table(14, dim, row_dtype=row_dtype)
    ref = oracle.Table(14, dim, row_dtype=oracle.BF16 if row_dtype == "bf16" else oracle.F32)
    b = W.jagged_batch(11, users=24)
    bo = jagged_bags(b)
    for s, mode in enumerate(("sum", "mean")):
        pooled_step(tab, ref, b, bo, mode, 300 + s, row_dtype)
