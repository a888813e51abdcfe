"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bit-exact: unique keys, inverse indices, counts, key presence and gathered
rows (fresh rows come from a counter-based generator keyed by the ID, and
slot placement is not compared).  Within tolerance: gradient sums and
Adam-updated rows (fp32 rows 1e-5 relative + 1e-6 absolute; bf16 rows within
one bf16 ulp), as the table's specification fixes.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import update_merged_table_gb300 as mt
from update_merged_table_gb300 import workloads as W

pytestmark = pytest.mark.gpu

from numerics import ATOL, RTOL, assert_rows_close  # noqa: E402


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


def compare_lookup(res, r, gather=True):
    U = res.U
    assert U == r["U"]
    n = res.n
    uk = res.unique_keys[:U].cpu().numpy().view(np.uint64)
    assert np.array_equal(uk, r["unique"])
    assert np.array_equal(res.inverse[:n].cpu().numpy(), r["inverse"])
    assert np.array_equal(res.counts[:U].cpu().numpy(), r["counts"])
    present = res.unique_rows[:U].cpu().numpy() >= 0
    assert np.array_equal(present, r["present"])
    if gather and n:
        got = res.rows.float().cpu().numpy()
        assert np.array_equal(got, r["rows"])


def compare_after_adam(tab, res, ref, r, row_dtype, gsum=None, ref_gsum=None):
    U = r["U"]
    if gsum is not None:
        np.testing.assert_allclose(gsum[:U].cpu().numpy(), ref_gsum, rtol=RTOL, atol=ATOL)
    emb, m, v = tab.read_rows(res.unique_rows[:U])
    e2, m2, v2, pr = ref.get_rows(r["unique"])
    pres = pr
    assert_rows_close(emb.cpu().numpy()[pres], e2[pres], row_dtype)
    np.testing.assert_allclose(m.cpu().numpy()[pres], m2[pres], rtol=RTOL, atol=ATOL)
    np.testing.assert_allclose(v.cpu().numpy()[pres], v2[pres], rtol=RTOL, atol=1e-9)


def grads_for(seed, n, d, dtype):
    g = W.grads_normal(seed, n, d)
    if dtype == "bf16":
        gb = torch.from_numpy(g).to(torch.bfloat16)
        return gb.to(dev()), gb.view(torch.int16).numpy().view(np.uint16), oracle.BF16
    return to_dev(g), g, oracle.F32


def run_steps(tab, ref, batches, row_dtype="f32", grad_dtype="f32", seed0=100, check_rows_every=1):
    for k, b in enumerate(batches):
        res = tab.lookup(to_dev(b.ids), b.feat_offsets, b.table_ids)
        r = ref.lookup(b.ids, b.feat_offsets, b.table_ids)
        compare_lookup(res, r)
        gd, gh, gdt = grads_for(seed0 + k, b.n, tab.dim, grad_dtype)
        gsum = tab.backward_adam(res, gd, want_gsum=True)
        ref_gsum = ref.backward_adam(gh, grad_dtype=gdt, want_gsum=True)
        if k % check_rows_every == 0:
            compare_after_adam(tab, res, ref, r, row_dtype, gsum, ref_gsum)
    assert tab.error() == 0 and ref.error == 0


# ---------------------------------------------------------------------------
# the workloads, at sizes the oracle finishes in seconds
# ---------------------------------------------------------------------------

def test_single_table_workload():
    """M = 2^16, dim 16 fp32, 4096 IDs Zipf(1.1) over 1e5; lookup+insert then backward+Adam."""
    b = W.single_table_batch(0)
    tab = mt.Table(16, 16)
    ref = oracle.Table(16, 16, simulate=True)
    run_steps(tab, ref, [b])
    st = tab.stats()
    sim = ref.sim_stats()
    assert st["live"] == sim["live"] == ref.live
    assert st["total_displacement"] == sim["total_displacement"]  # insert-only: order-independent
    assert st["step"] == 1 and tab.step == 1


@pytest.mark.parametrize("probe_step", [1, 3, 0x9E3779B97F4A7C15])
def test_merged_tables_steps(probe_step):
    """8 feature tables merged by table id into one table, dim 32 fp32, several steps."""
    tab = mt.Table(18, 32, probe_step=probe_step, hash_seed=7, init_seed=11)
    ref = oracle.Table(18, 32, probe_step=probe_step, hash_seed=7, init_seed=11, simulate=True)
    run_steps(tab, ref, [W.merged_batch(s, per_table=2048) for s in range(4)])
    st, sim = tab.stats(), ref.sim_stats()
    assert st["live"] == sim["live"] and st["total_displacement"] == sim["total_displacement"]


def test_jagged_bf16_rows_and_grads():
    """Jagged user sequences, 4 ID features, dim 64 bf16 rows, fp32 Adam state, bf16 grads."""
    batches = [W.jagged_batch(s, users=96, lengths_seed=s) for s in range(3)]
    tab = mt.Table(18, 64, row_dtype="bf16")
    ref = oracle.Table(18, 64, row_dtype=oracle.BF16)
    run_steps(tab, ref, batches, row_dtype="bf16", grad_dtype="bf16")


def test_bf16_rows_fp32_grads_and_fp32_rows_bf16_grads():
    b = W.merged_batch(3, per_table=512)
    tab = mt.Table(16, 32, row_dtype="bf16")
    ref = oracle.Table(16, 32, row_dtype=oracle.BF16)
    run_steps(tab, ref, [b, b], row_dtype="bf16", grad_dtype="f32")
    tab = mt.Table(16, 32)
    ref = oracle.Table(16, 32)
    run_steps(tab, ref, [b, b], row_dtype="f32", grad_dtype="bf16")


def test_bf16_rows_fp32_grads_past_l2():
    """bf16 rows with fp32 gradients whose matrix is too large to stay in L2 (> 16 MB): the heavy uniques'
    rows go through the shared-memory ring, not the register path small fp32 matrices take."""
    batches = [W.jagged_batch(s, users=256, lengths_seed=s) for s in range(2)]
    assert all(b.n * 64 * 4 > (16 << 20) for b in batches)
    tab = mt.Table(19, 64, row_dtype="bf16")
    ref = oracle.Table(19, 64, row_dtype=oracle.BF16)
    run_steps(tab, ref, batches, row_dtype="bf16", grad_dtype="f32")


def test_large_keyspace_prefilled():
    """Zipf(1.05) over a 2^32 key space, dim 128 fp32, table prefilled to load 0.7."""
    log2 = 16
    tab = mt.Table(log2, 128)
    ref = oracle.Table(log2, 128, simulate=True)
    pre = W.large_table_prefill_ids(int(0.7 * (1 << log2)))
    res = tab.lookup(to_dev(pre), gather=False)
    ref.lookup(pre, gather=False)
    assert res.U == pre.size
    batches = [W.large_table_batch(s, n=8192) for s in range(2)]
    run_steps(tab, ref, batches)
    st, sim = tab.stats(), ref.sim_stats()
    assert st["live"] == sim["live"] == ref.live
    assert st["total_displacement"] == sim["total_displacement"]


def test_churn_with_erase_and_stats():
    """Per step: IDs with 10% never seen before, then erase of random earlier IDs (tombstones)."""
    log2 = 14
    cs = W.ChurnStream(0, hot=1 << 12, n=1 << 11, erase=1 << 9)
    tab = mt.Table(log2, 64)
    ref = oracle.Table(log2, 64, simulate=True)
    pre = cs.prefill_ids()
    tab.lookup(to_dev(pre), gather=False)
    ref.lookup(pre, gather=False)
    for k in range(12):
        b, er = cs.step(k)
        res = tab.lookup(to_dev(b.ids))
        r = ref.lookup(b.ids)
        compare_lookup(res, r)
        gd, gh, _ = grads_for(500 + k, b.n, 64, "f32")
        tab.backward_adam(res, gd)
        ref.backward_adam(gh)
        compare_after_adam(tab, res, ref, r, "f32")
        found = tab.erase(to_dev(er.astype(np.int64)))
        want = ref.erase(er.astype(np.uint64))
        assert np.array_equal(found.cpu().numpy().astype(bool), want)
        st = tab.stats()
        assert st["live"] == ref.live
        assert st["rows_free"] == (1 << log2) - ref.live
        keys, rows = tab.export()
        assert np.array_equal(np.sort(keys.cpu().numpy().view(np.uint64)), np.sort(ref.live_keys()))
        assert np.unique(rows.cpu().numpy()).size == rows.numel()
    sim = ref.sim_stats()
    st = tab.stats()
    # placement under churn depends on insertion order: tolerances
    assert abs(st["tombstones"] - sim["tombstones"]) <= 0.05 * max(sim["tombstones"], 1) + 16
    h1 = st["probe_hist"] / max(1, st["live"])
    h2 = sim["hist"] / max(1, sim["live"])
    assert np.abs(h1 - h2).sum() <= 0.05
    assert abs(st["total_displacement"] - sim["total_displacement"]) <= 0.05 * sim["total_displacement"] + 64
    assert tab.error() == 0


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n", [0, 1, 31, 2047, 2048, 2049, 5000])
def test_ragged_sizes(n):
    rng = np.random.default_rng(n)
    ids = rng.integers(0, max(1, n // 2), size=n)
    tab = mt.Table(14, 16)
    ref = oracle.Table(14, 16)
    b = W.single_feature(ids)
    run_steps(tab, ref, [b, b])


def test_all_positions_one_id():
    ids = np.full(10000, 123456789, np.int64)
    tab = mt.Table(10, 8, row_dtype="bf16")
    ref = oracle.Table(10, 8, row_dtype=oracle.BF16)
    run_steps(tab, ref, [W.single_feature(ids)], row_dtype="bf16")


def test_empty_segments_and_table_ids():
    ids = np.arange(300, dtype=np.int64) % 37
    offs = [0, 0, 100, 100, 250, 300]
    tids = [5, 254, 0, 7, 254]
    tab = mt.Table(12, 16)
    ref = oracle.Table(12, 16)
    res = tab.lookup(to_dev(ids), offs, tids)
    r = ref.lookup(ids, offs, tids)
    compare_lookup(res, r)
    assert (r["unique"] >> np.uint64(56)).max() == 254


def test_invalid_ids_latch_ekey():
    ids = np.array([5, -1, 7, 1 << 56, 5, (1 << 56) - 1], np.int64)
    tab = mt.Table(10, 16)
    ref = oracle.Table(10, 16)
    res = tab.lookup(to_dev(ids))
    r = ref.lookup(ids)
    compare_lookup(res, r)
    assert res.inverse[1].item() == -1 and res.inverse[3].item() == -1
    assert tab.error() == mt.MT_EKEY == ref.error
    assert tab.error(clear=True) == mt.MT_EKEY and tab.error() == 0
    g = torch.ones((ids.size, 16), device=dev())
    tab.backward_adam(res, g)  # invalid positions contribute nothing
    ref.backward_adam(np.ones((ids.size, 16), np.float32))
    compare_after_adam(tab, res, ref, r, "f32")


def test_eval_mode_misses_give_zeros():
    tab = mt.Table(12, 16)
    ref = oracle.Table(12, 16)
    a = np.arange(50, dtype=np.int64)
    compare_lookup(tab.lookup(to_dev(a)), ref.lookup(a))
    b = np.arange(25, 100, dtype=np.int64)
    res = tab.lookup(to_dev(b), insert_missing=False)
    r = ref.lookup(b, insert_missing=False)
    compare_lookup(res, r)
    assert tab.stats()["live"] == 50


def test_row_pool_exhaustion_latches_full():
    tab = mt.Table(10, 16, num_rows=100)
    ids = np.arange(500, dtype=np.int64)
    res = tab.lookup(to_dev(ids))
    torch.cuda.synchronize()
    rows = res.unique_rows[:500].cpu().numpy()
    assert (rows >= 0).sum() == 100 and np.unique(rows[rows >= 0]).size == 100
    assert tab.error() == mt.MT_EFULL
    st = tab.stats()
    assert st["live"] == 100 and st["rows_free"] == 0
    got = res.rows.cpu().numpy()
    for i in np.nonzero(rows >= 0)[0][:20]:
        assert np.array_equal(got[i], oracle.init_row(i, 0, oracle.default_init_scale(16), 16))
    assert np.all(got[rows < 0] == 0)


def test_probe_limit_latches_full_without_hang():
    tab = mt.Table(6, 8, max_probes=2)
    ids = np.arange(64, dtype=np.int64)
    res = tab.lookup(to_dev(ids))
    rows = res.unique_rows[:64].cpu().numpy()
    assert tab.error() == mt.MT_EFULL
    placed = rows >= 0
    assert 0 < placed.sum() < 64
    again = tab.lookup(to_dev(ids), insert_missing=False)
    assert np.array_equal(again.unique_rows[:64].cpu().numpy() >= 0, placed)
    assert np.array_equal(again.unique_rows[:64].cpu().numpy()[placed], rows[placed])


def test_erase_duplicates_and_reinsert():
    tab = mt.Table(10, 16, init_seed=3)
    ref = oracle.Table(10, 16, init_seed=3)
    ids = np.arange(40, dtype=np.int64)
    res = tab.lookup(to_dev(ids))
    r = ref.lookup(ids)
    tab.backward_adam(res, torch.ones((40, 16), device=dev()))
    ref.backward_adam(np.ones((40, 16), np.float32))
    er = np.array([3, 3, 99, 5, 3], np.int64)
    found = tab.erase(to_dev(er)).cpu().numpy()
    assert found.tolist() == [1, 1, 0, 1, 1] == ref.erase(er.astype(np.uint64)).astype(int).tolist()
    st = tab.stats()
    assert st["live"] == 38 and st["tombstones"] == 2 and st["rows_free"] == 1024 - 38
    res = tab.lookup(to_dev(np.array([3, 4], np.int64)))
    r = ref.lookup(np.array([3, 4], np.int64))
    compare_lookup(res, r)  # key 3 is back at its initial row; key 4 keeps its trained row
    st = tab.stats()
    assert st["live"] == 39 and st["tombstones"] <= 2


@pytest.mark.parametrize("probe_step", [1, 3])
def test_compact_drops_tombstones_and_keeps_rows(probe_step):
    """mt_compact after heavy erasing: no tombstones, the same live keys on
    the same rows (lookups gather identical rows), and the table keeps
    training in step with the oracle."""
    rng = np.random.default_rng(9)
    tab = mt.Table(14, 8, probe_step=probe_step, init_seed=4)  # room for every key of the test
    ref = oracle.Table(14, 8, probe_step=probe_step, init_seed=4)
    ids = rng.choice(1 << 20, 2500, replace=False).astype(np.int64)
    res = tab.lookup(to_dev(ids))
    ref.lookup(ids)
    g = W.grads_normal(3, ids.size, 8)
    tab.backward_adam(res, to_dev(g))
    ref.backward_adam(g)
    er = ids[::2].copy()
    tab.erase(to_dev(er))
    ref.erase(er.astype(np.uint64))
    more = rng.choice(1 << 20, 800).astype(np.int64)  # inserts after the erases reuse some tombstones
    tab.lookup(to_dev(more))
    ref.lookup(more)
    st0 = tab.stats()
    assert st0["tombstones"] > 0
    before = tab.lookup(to_dev(ids), insert_missing=False)
    U = before.U
    rows_before, urows_before = before.rows.clone(), before.unique_rows[:U].clone()
    tab.compact()
    st1 = tab.stats()
    assert tab.error() == 0
    assert st1["tombstones"] == 0 and st1["live"] == st0["live"] == ref.live
    assert st1["rows_free"] == st0["rows_free"] and st1["step"] == st0["step"]
    after = tab.lookup(to_dev(ids), insert_missing=False)
    assert after.U == U
    assert torch.equal(after.unique_rows[:U], urows_before)
    assert torch.equal(after.rows, rows_before)
    run_steps(tab, ref, [W.single_feature(rng.choice(1 << 20, 3000).astype(np.int64))], seed0=50)
    # the slot array now lives in the first spare; a second compaction goes back into the key store's
    tab.erase(to_dev(ids[1::2].copy()))
    ref.erase(ids[1::2].astype(np.uint64))
    first_home = tab._slots_buf.data_ptr()
    tab.compact()
    assert tab._slots_buf.data_ptr() != first_home and tab.stats()["tombstones"] == 0
    assert tab.stats()["live"] == ref.live
    run_steps(tab, ref, [W.single_feature(rng.choice(1 << 20, 3000).astype(np.int64))], seed0=51)


@pytest.mark.parametrize("row_dtype", ["f32", "bf16"])
def test_checkpoint_restore_continues_bit_identically(row_dtype):
    """Export keys and rows, read emb/m/v and the Adam state, import them into
    a fresh table: it gathers the same rows and trains on bit-identically."""
    tab = mt.Table(14, 16, row_dtype=row_dtype, init_seed=2)
    g_dt = torch.float32 if row_dtype == "f32" else torch.bfloat16
    for s in range(2):
        b = W.merged_batch(s, per_table=256)
        res = tab.lookup(to_dev(b.ids), b.feat_offsets, b.table_ids)
        tab.backward_adam(res, torch.from_numpy(W.grads_normal(40 + s, b.n, 16)).to(g_dt).to(dev()))
    keys, rows = tab.export()
    emb, m, v = tab.read_rows(rows)
    state = tab.adam_state()
    assert state[0] == 2
    tab2 = mt.Table(14, 16, row_dtype=row_dtype, init_seed=2)
    tab2.import_rows(keys.contiguous(), emb.contiguous(), m.contiguous(), v.contiguous())
    tab2.set_adam_state(*state)
    assert tab2.adam_state() == state and tab2.step == 2
    st1, st2 = tab.stats(), tab2.stats()
    assert st2["live"] == st1["live"] and tab2.error() == 0
    for s in (2, 3):  # the same batches and grads on both tables
        b = W.merged_batch(s, per_table=256)
        r1 = tab.lookup(to_dev(b.ids), b.feat_offsets, b.table_ids)
        r2 = tab2.lookup(to_dev(b.ids), b.feat_offsets, b.table_ids)
        assert torch.equal(r1.unique_keys[:r1.U], r2.unique_keys[:r2.U])
        assert torch.equal(r1.inverse[:b.n], r2.inverse[:b.n])
        assert torch.equal(r1.rows.view(torch.uint8), r2.rows.view(torch.uint8))
        gg = torch.from_numpy(W.grads_normal(50 + s, b.n, 16)).to(g_dt).to(dev())
        tab.backward_adam(r1, gg)
        tab2.backward_adam(r2, gg)
        e1, m1, v1 = tab.read_rows(r1.unique_rows[:r1.U])
        e2, m2, v2 = tab2.read_rows(r2.unique_rows[:r2.U])
        assert torch.equal(e1, e2) and torch.equal(m1, m2) and torch.equal(v1, v2)
    assert tab.error() == 0 and tab2.error() == 0


def test_grow_keeps_keys_rows_and_training():
    """Capacity expansion (2^10 to 2^12 slots, 1024 to 4096 rows) mid-training:
    the same keys on the same rows, the Adam state kept, room for new keys,
    and training continues in step with the oracle."""
    rng = np.random.default_rng(13)
    tab = mt.Table(10, 8, probe_step=3, init_seed=5)
    ref = oracle.Table(13, 8, probe_step=3, init_seed=5)  # its capacity never binds in this test
    ids = rng.choice(1 << 20, 600, replace=False).astype(np.int64)
    run_steps(tab, ref, [W.single_feature(ids)], seed0=60)
    before = tab.lookup(to_dev(ids), insert_missing=False)
    U = before.U
    rows_before, urows_before = before.rows.clone(), before.unique_rows[:U].clone()
    st0, state0 = tab.stats(), tab.adam_state()
    ks_old = tab.lib.mt_keystore_bytes(ctypes.byref(tab.cfg))
    rows_before_grow = tab.arena[ks_old:].clone()  # the first row segment lives after the key store
    tab.grow(12)
    assert torch.equal(tab.arena[ks_old:], rows_before_grow)  # no row was moved or rewritten
    st1 = tab.stats()
    assert tab.error() == 0 and tab.adam_state() == state0
    assert st1["capacity"] == 4096 and st1["live"] == st0["live"] == 600 and st1["tombstones"] == 0
    assert st1["rows_free"] == 4096 - 600
    after = tab.lookup(to_dev(ids), insert_missing=False)
    assert after.U == U and torch.equal(after.unique_rows[:U], urows_before) and torch.equal(after.rows, rows_before)
    more = np.concatenate([ids[:300], rng.choice(1 << 20, 2000).astype(np.int64)])
    run_steps(tab, ref, [W.single_feature(more)], seed0=61)  # 2600 keys: more than the old table held
    assert not torch.equal(tab.arena[ks_old:], rows_before_grow)  # the old keys' rows trained in place
    # a second expansion adds a second new row segment; a compaction then moves the slot array
    tab.grow(13, num_rows=6000)
    assert tab.stats()["rows_free"] == 6000 - ref.live and len(tab._row_bufs) == 3
    tab.compact()
    run_steps(tab, ref, [W.single_feature(rng.choice(1 << 20, 1500).astype(np.int64))], seed0=62)
    assert tab.error() == 0 and tab.stats()["live"] == ref.live


def test_step_counter_and_lazy_rows():
    tab = mt.Table(10, 8)
    ref = oracle.Table(10, 8)
    a = W.single_feature(np.array([1, 2], np.int64))
    b = W.single_feature(np.array([1], np.int64))
    run_steps(tab, ref, [a, b, b])
    emb, _, _ = tab.read_rows(tab.lookup(to_dev(np.array([2], np.int64))).unique_rows[:1])
    assert np.allclose(emb.cpu().numpy()[0], ref.get_row(2)[0])
    assert tab.stats()["step"] == 3 == ref.step


def test_integer_grads_sum_exactly():
    """Integer-valued gradients: every partial sum is exact, so the sums match bit for bit."""
    b = W.merged_batch(5, per_table=4096)
    tab = mt.Table(18, 32)
    ref = oracle.Table(18, 32)
    res = tab.lookup(to_dev(b.ids), b.feat_offsets, b.table_ids)
    r = ref.lookup(b.ids, b.feat_offsets, b.table_ids)
    g = W.grads_small_int(9, b.n, 32)
    gsum = tab.backward_adam(res, to_dev(g), want_gsum=True)
    want = ref.backward_adam(g, want_gsum=True)
    assert np.array_equal(gsum[:r["U"]].cpu().numpy(), want)


@pytest.mark.parametrize("n_unique", [2049, 4096])
@pytest.mark.parametrize("row_dtype,dim", [("f32", 32), ("bf16", 64)])
def test_grouping_plan_boundaries(n_unique, row_dtype, dim):
    """The backward's grouping at its boundaries: keys with 31 | 32 | 33 positions (a light unique has at
    most 32), 255 | 256 | 257 and 513 (one heavy warp-chunk holds 256 positions at these dims), filled with
    single-position keys up to a unique count one past, or exactly at, the end of a 2048-unique block of the
    grouping plan.  Positions are shuffled, gradients are integers (so every sum is exact and compared bit
    for bit), then a second step with normal gradients checks Adam."""
    rng = np.random.default_rng(n_unique + dim)
    special = [1, 2, 31, 32, 33, 255, 256, 257, 513, 1000]
    counts = special + [1] * (n_unique - len(special))
    ids = np.repeat(np.arange(n_unique, dtype=np.int64) * 7919 + 11, counts)
    b = W.single_feature(ids[rng.permutation(ids.size)])
    tab = mt.Table(16, dim, row_dtype=row_dtype)
    ref = oracle.Table(16, dim, row_dtype=oracle.BF16 if row_dtype == "bf16" else oracle.F32)
    res = tab.lookup(to_dev(b.ids), b.feat_offsets, b.table_ids)
    r = ref.lookup(b.ids, b.feat_offsets, b.table_ids)
    compare_lookup(res, r)
    assert r["U"] == n_unique
    g = W.grads_small_int(7, b.n, dim)
    gsum = tab.backward_adam(res, to_dev(g), want_gsum=True)
    want = ref.backward_adam(g, want_gsum=True)
    assert np.array_equal(gsum[:n_unique].cpu().numpy(), want)
    compare_after_adam(tab, res, ref, r, row_dtype)
    run_steps(tab, ref, [b], row_dtype=row_dtype, grad_dtype="f32", seed0=41)


# ---------------------------------------------------------------------------
# full size, in the launch configuration the benchmark times
# ---------------------------------------------------------------------------

def test_full_size_jagged_fresh_steps():
    """2048 users, lognormal(5, 1) lengths capped at 3000, 4 features, M = 2^24, dim 64 bf16: the cold step 0
    and five fresh-seed steps (each a new batch of users, so every step inserts keys), all compared in full."""
    tab = mt.Table(24, 64, row_dtype="bf16")
    ref = oracle.Table(24, 64, row_dtype=oracle.BF16)
    batches = [W.jagged_batch(s) for s in range(6)]
    run_steps(tab, ref, batches, row_dtype="bf16", grad_dtype="bf16")
    assert tab.stats()["live"] == ref.live


def test_full_size_merged():
    """8 tables, 65536 IDs, M = 2^22, dim 32 fp32: all 100 steps, lookups compared every step and
    gradient sums and Adam rows every tenth step."""
    tab = mt.Table(22, 32)
    ref = oracle.Table(22, 32)
    for k in range(100):
        b = W.merged_batch(k)
        res = tab.lookup(to_dev(b.ids), b.feat_offsets, b.table_ids)
        r = ref.lookup(b.ids, b.feat_offsets, b.table_ids, gather=(k % 10 == 0))
        compare_lookup(res, r, gather=(k % 10 == 0))
        gd, gh, gdt = grads_for(300 + k, b.n, 32, "f32")
        check = k % 10 == 0 or k == 99
        gsum = tab.backward_adam(res, gd, want_gsum=check)
        ref_gsum = ref.backward_adam(gh, grad_dtype=gdt, want_gsum=check)
        if check:
            compare_after_adam(tab, res, ref, r, "f32", gsum, ref_gsum)
    assert tab.error() == 0 and ref.error == 0 and tab.step == ref.step == 100


def test_ranks_are_a_permutation_per_key():
    """ranks[i] enumerates the positions of each key: per key a permutation of 0..count-1."""
    b = W.jagged_batch(4, users=64)
    tab = mt.Table(16, 16)
    res = tab.lookup(to_dev(b.ids), b.feat_offsets, b.table_ids)
    U = res.U
    inv = res.inverse[:b.n].cpu().numpy().astype(np.int64)
    rk = res.ranks[:b.n].cpu().numpy().astype(np.int64)
    cnt = res.counts[:U].cpu().numpy()
    assert rk.min() >= 0 and np.all(rk < cnt[inv])
    key = inv * (int(cnt.max()) + 1) + rk          # (unique, rank) pairs are all distinct
    assert np.unique(key).size == b.n


def test_backward_without_ranks_matches_with_ranks():
    """Both ways of grouping positions by key give the same sums and rows."""
    b = W.merged_batch(8, per_table=1024)
    g = to_dev(W.grads_small_int(3, b.n, 32))
    out = []
    for ranks in (True, False):
        tab = mt.Table(16, 32)
        res = tab.new_result(b.n, ranks=ranks)
        tab.lookup(to_dev(b.ids), b.feat_offsets, b.table_ids, result=res)
        gs = tab.backward_adam(res, g, want_gsum=True)
        emb, m, v = tab.read_rows(res.unique_rows[:res.U])
        out.append((gs[:res.U].cpu().numpy(), emb.cpu().numpy()))
    assert np.array_equal(out[0][0], out[1][0]) and np.array_equal(out[0][1], out[1][1])


def test_many_tiles_first_occurrence_order():
    """One lookup of 20M IDs (~10k tiles of 2048 positions): unique keys in
    first-occurrence order, inverse and counts, exactly as numpy's unique
    defines them.  The owners' tile offsets come from a look-back that walks
    thousands of earlier tiles."""
    rng = np.random.default_rng(21)
    n = 20_000_000
    ids = W.bijection32(W.zipf_ranks(rng, n, 1.05, 1 << 24))
    b = W.single_feature(ids, table_id=3)
    tab = mt.Table(24, 4)
    res = tab.new_result(n, gather=False, ranks=False)
    tab.lookup(to_dev(b.ids), b.feat_offsets, b.table_ids, gather=False, result=res)
    keys = (np.uint64(3) << np.uint64(56)) | ids.astype(np.uint64)
    uniq, first, inv, cnt = np.unique(keys, return_index=True, return_inverse=True, return_counts=True)
    order = np.argsort(first, kind="stable")     # unique keys by first position
    rank = np.empty_like(order)
    rank[order] = np.arange(order.size)
    U = res.U
    assert U == uniq.size
    assert np.array_equal(res.unique_keys[:U].cpu().numpy().view(np.uint64), uniq[order])
    assert np.array_equal(res.inverse[:n].cpu().numpy(), rank[inv].astype(np.int32))
    assert np.array_equal(res.counts[:U].cpu().numpy(), cnt[order].astype(np.int32))
    assert tab.error() == 0


def test_full_size_large_table():
    """M = 2^26 slots, dim 128 fp32, prefilled with 0.7 M keys (46,976,204); a 2^20-ID batch Zipf(1.05)
    over a 2^32 key space: unique/inverse/counts bit-exact, sampled gathered rows bit-exact (untouched
    rows hold their initial values), sampled Adam rows within tolerance."""
    log2, dim = 26, 128
    tab = mt.Table(log2, dim)
    pre_n = int(0.7 * (1 << log2))
    pre = W.large_table_prefill_ids(pre_n)
    for s0 in range(0, pre_n, 1 << 22):
        tab.lookup(to_dev(pre[s0:s0 + (1 << 22)]), gather=False)
    del pre
    st = tab.stats()
    assert st["live"] == pre_n and tab.error() == 0
    b = W.large_table_batch(0)
    res = tab.lookup(to_dev(b.ids))
    keys, valid = oracle.encode(b.ids, b.feat_offsets, b.table_ids)
    uq, inv, cnt = oracle.unique(keys, valid)
    U = res.U
    assert U == uq.size
    assert np.array_equal(res.unique_keys[:U].cpu().numpy().view(np.uint64), uq)
    assert np.array_equal(res.inverse[:b.n].cpu().numpy(), inv)
    assert np.array_equal(res.counts[:U].cpu().numpy(), cnt)
    assert (res.unique_rows[:U] >= 0).all()
    rng = np.random.default_rng(0)
    sample = rng.choice(b.n, size=2000, replace=False)
    got = res.rows[torch.from_numpy(sample).to(dev())].cpu().numpy()
    scale = oracle.default_init_scale(dim)
    for r, i in enumerate(sample):
        assert np.array_equal(got[r], oracle.init_row(int(keys[i]), 0, scale, dim))
    # backward on the whole batch; the oracle sees the same keys fresh (same initial rows)
    ref = oracle.Table(log2, dim)
    ref.lookup(b.ids, b.feat_offsets, b.table_ids, gather=False)
    g = W.grads_normal(5, b.n, dim)
    gsum = tab.backward_adam(res, to_dev(g), want_gsum=True)
    ref_gsum = ref.backward_adam(g, want_gsum=True)
    np.testing.assert_allclose(gsum[:U].cpu().numpy(), ref_gsum, rtol=RTOL, atol=ATOL)
    us = rng.choice(U, size=min(U, 20000), replace=False)
    emb, m, v = tab.read_rows(res.unique_rows[torch.from_numpy(us).to(dev())])
    e2, m2, v2, pr = ref.get_rows(uq[us])
    assert pr.all()
    np.testing.assert_allclose(emb.cpu().numpy(), e2, rtol=RTOL, atol=ATOL)
    np.testing.assert_allclose(m.cpu().numpy(), m2, rtol=RTOL, atol=ATOL)
    np.testing.assert_allclose(v.cpu().numpy(), v2, rtol=RTOL, atol=1e-9)
    assert tab.error() == 0


def test_full_size_online_churn():
    """M = 2^24, dim 64 fp32, 2^23 prefilled keys; 200 steps of 2^18 IDs with 10% never seen before,
    backward+Adam, and erase of 2^16 earlier IDs; live counts exact every step, rows and stats checked
    every 20 steps against the oracle and its shadow open-addressing table."""
    log2, dim = 24, 64
    cs = W.ChurnStream(0)
    tab = mt.Table(log2, dim)
    ref = oracle.Table(log2, dim, simulate=True)
    pre = cs.prefill_ids()
    for s0 in range(0, pre.size, 1 << 22):
        tab.lookup(to_dev(pre[s0:s0 + (1 << 22)]), gather=False)
    ref.insert_keys(pre.astype(np.uint64))
    for k in range(200):
        b, er = cs.step(k)
        res = tab.lookup(to_dev(b.ids))
        r = ref.lookup(b.ids, gather=(k % 20 == 0))
        gd, gh, _ = grads_for(900 + k, b.n, dim, "f32")
        tab.backward_adam(res, gd)
        ref.backward_adam(gh)
        found = tab.erase(to_dev(er))
        want = ref.erase(er.astype(np.uint64))
        if k % 20 == 0:
            compare_lookup(res, r)
            assert np.array_equal(found.cpu().numpy().astype(bool), want)
            st = tab.stats()
            sim = ref.sim_stats()
            assert st["live"] == ref.live == sim["live"]
            assert abs(st["tombstones"] - sim["tombstones"]) <= 0.05 * sim["tombstones"] + 64
            h1 = st["probe_hist"] / st["live"]
            h2 = sim["hist"] / sim["live"]
            assert np.abs(h1 - h2).sum() <= 0.05
            # Adam rows of a sample of this step's keys
            U = r["U"]
            us = np.random.default_rng(k).choice(U, size=min(U, 5000), replace=False)
            keys_now = r["unique"][us]
            again = tab.lookup(to_dev(keys_now.astype(np.int64)), insert_missing=False)
            rows_now = again.unique_rows[:again.U]
            emb, m, v = tab.read_rows(rows_now)
            e2, m2, v2, pr = ref.get_rows(keys_now)
            assert np.array_equal(rows_now.cpu().numpy() >= 0, pr)
            np.testing.assert_allclose(emb.cpu().numpy()[pr], e2[pr], rtol=RTOL, atol=ATOL)
            np.testing.assert_allclose(m.cpu().numpy()[pr], m2[pr], rtol=RTOL, atol=ATOL)
            np.testing.assert_allclose(v.cpu().numpy()[pr], v2[pr], rtol=RTOL, atol=1e-9)
    assert tab.error() == 0 and ref.error == 0


def test_graph_capture_needs_reserved_workspaces():
    """A lookup captured in a CUDA graph must not grow a workspace (graphs captured earlier keep the old
    buffer's address); after reserve_workspaces the captured lookup replays to the eager result."""
    tab = mt.Table(14, 16)
    small = to_dev(np.arange(100, dtype=np.int64))
    ids = np.random.default_rng(3).integers(0, 3000, size=6000).astype(np.int64)
    big = to_dev(ids)
    tab.lookup(small)  # workspaces sized for 100 IDs
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    res = tab.new_result(ids.size)
    with pytest.raises(RuntimeError, match="reserve_workspaces"):
        with torch.cuda.graph(torch.cuda.CUDAGraph(), stream=s):
            tab.lookup(big, result=res)
    tab.reserve_workspaces(ids.size)
    eager = tab.lookup(big)  # inserts the keys
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tab.lookup(big, result=res)
    g.replay()
    torch.cuda.synchronize()
    U = eager.U
    assert res.U == U
    assert torch.equal(res.unique_keys[:U], eager.unique_keys[:U])
    assert torch.equal(res.inverse, eager.inverse)
    assert torch.equal(res.counts[:U], eager.counts[:U])
    assert torch.equal(res.rows, eager.rows)
    assert tab.error() == 0
