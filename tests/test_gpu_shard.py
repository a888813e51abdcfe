"""Sharded two-stage deduplication: G logical ranks with one shard table each, on one GPU (through the C ABI).

Each rank's unique keys, inverse and counts are its own batch's first-occurrence unique (bit-exact against
the oracle); the rows a rank receives equal those of one table holding every key (bit-exact before any
training); the gradient sums over all ranks and the Adam-updated rows match one oracle table fed the
concatenation of the ranks' batches (fp32 within 1e-5 relative + 1e-6 absolute; bf16 within one ulp: each
rank's sum is rounded to fp32 before the owner adds them); every key lives in one shard only.
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


def run_sharded(G, dim, row_dtype, steps, make_batch, log2=14):
    shards = [mt.Table(log2, dim, row_dtype=row_dtype, init_seed=9, hash_seed=r) for r in range(G)]
    grp = mt.ShardGroup(shards)
    ref = oracle.Table(log2 + 4, dim, row_dtype=oracle.BF16 if row_dtype == "bf16" else oracle.F32, init_seed=9)
    gdt = torch.bfloat16 if row_dtype == "bf16" else torch.float32
    for step in range(steps):
        batches = [make_batch(step, r) for r in range(G)]
        res = grp.lookup([to_dev(b.ids) for b in batches], [b.feat_offsets for b in batches], batches[0].table_ids)
        # the oracle: one table, the ranks' batches one after the other
        keys_all, valid_all = [], []
        for b in batches:
            k, v = oracle.encode(b.ids, b.feat_offsets, b.table_ids)
            keys_all.append(k)
            valid_all.append(v)
        for r, b in enumerate(batches):  # per rank: its own first-occurrence unique
            uq, inv, cnt = oracle.unique(keys_all[r], valid_all[r])
            U = res[r].U
            assert U == uq.size
            assert np.array_equal(res[r].unique_keys[:U].cpu().numpy().view(np.uint64), uq)
            assert np.array_equal(res[r].inverse[:b.n].cpu().numpy(), inv)
            assert np.array_equal(res[r].counts[:U].cpu().numpy(), cnt)
            assert (res[r].unique_rows[:U] == -1).all()
        # one batch of every rank's feature segments in rank order, each with its table id
        offs, tids, ids_cat = [0], [], []
        for b in batches:
            for f in range(b.feat_offsets.size - 1):
                seg = b.ids[b.feat_offsets[f]:b.feat_offsets[f + 1]]
                ids_cat.append(seg)
                offs.append(offs[-1] + seg.size)
                tids.append(int(b.table_ids[f]))
        r_all = ref.lookup(np.concatenate(ids_cat), np.array(offs, np.int64), np.array(tids, np.uint8))
        start = 0
        for r, b in enumerate(batches):
            want = r_all["rows"][start:start + b.n]
            if step == 0:  # untrained rows: bit-exact
                assert np.array_equal(res[r].rows.float().cpu().numpy(), want)
            else:  # rows trained from two-stage sums (rank sums rounded once each): the stated tolerance
                assert_rows_close(res[r].rows.float().cpu().numpy(), want, row_dtype)
            start += b.n
        # backward: every rank's gradients; the oracle sees them concatenated in the same order
        gs = [W.grads_normal(100 * step + r, b.n, dim) for r, b in enumerate(batches)]
        gt = [torch.from_numpy(g).to(gdt) for g in gs]
        gsum = grp.backward_adam(res, [g.to(dev()) for g in gt], want_gsum=True)
        if row_dtype == "bf16":
            gcat = torch.cat(gt).view(torch.int16).numpy().view(np.uint16)
            ref_gsum = ref.backward_adam(gcat, grad_dtype=oracle.BF16, want_gsum=True)
        else:
            ref_gsum = ref.backward_adam(np.concatenate(gs), want_gsum=True)
        ukeys_all = r_all["unique"]
        pos = {int(k): i for i, k in enumerate(ukeys_all)}
        # each rank's sum is rounded to fp32 before the owner adds them (exactly) and rounds once more: with
        # S = sum of |g| over the key's positions, |error| <= 2^-24 * (S + |sum|) <= 2^-23 * S
        gabs = np.abs(torch.cat(gt).float().numpy()).astype(np.float64)
        S = np.zeros((ukeys_all.size, dim), np.float64)
        np.add.at(S, r_all["inverse"], gabs)
        for r in range(G):
            U = res[r].U
            uk = res[r].unique_keys[:U].cpu().numpy().view(np.uint64)
            idx = [pos[int(k)] for k in uk]
            want = ref_gsum[idx]
            got = gsum[r][:U].cpu().numpy()
            bound = RTOL * np.abs(want) + ATOL + 2.0 ** -23 * S[idx]
            assert (np.abs(got.astype(np.float64) - want) <= bound).all()
    # the trained rows, read back through another sharded lookup without inserts
    batches = [make_batch(steps - 1, r) for r in range(G)]
    res = grp.lookup([to_dev(b.ids) for b in batches], [b.feat_offsets for b in batches], batches[0].table_ids,
                     insert_missing=False)
    for r, b in enumerate(batches):
        U = res[r].U
        uk = res[r].unique_keys[:U].cpu().numpy().view(np.uint64)
        e2, _, _, pr = ref.get_rows(uk)
        assert pr.all()
        got = res[r].rows.float().cpu().numpy()
        inv = res[r].inverse[:b.n].cpu().numpy()
        us, first = np.unique(inv, return_index=True)  # the first position of every unique index
        keep = us >= 0
        assert np.array_equal(us[keep], np.arange(U))
        assert_rows_close(got[first[keep]], e2, row_dtype)
    # every key lives in exactly one shard, and together they hold the oracle's keys
    key_sets = [set(s.export()[0].cpu().numpy().view(np.uint64).tolist()) for s in shards]
    total = sum(len(k) for k in key_sets)
    union = set().union(*key_sets)
    assert total == len(union) == ref.live
    assert union == set(ref.live_keys().tolist())
    assert all(s.step == steps for s in shards) and all(s.error() == 0 for s in shards)


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
def test_sharded_merged_batches(G):
    """8 merged feature tables per rank, dim 16 fp32, two steps."""
    run_sharded(G, 16, "f32", 2, lambda step, r: W.merged_batch(1000 * step + r, per_table=512))


@pytest.mark.parametrize("G", [2, 4])
def test_sharded_jagged_bf16(G):
    """Jagged user sequences per rank (4 features), dim 64 bf16 rows, bf16 grads, two steps."""
    run_sharded(G, 64, "bf16", 2, lambda step, r: W.jagged_batch(50 * step + r, users=48), log2=16)


def test_sharded_full_size_jagged():
    """Two ranks, each a full-size GRM jagged batch (2048 users, ~2M IDs), M = 2^22 per shard, dim 64 bf16."""
    run_sharded(2, 64, "bf16", 1, lambda step, r: W.jagged_batch(7 + r), log2=22)
