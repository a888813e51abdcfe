"""Automatic table merging on the GPU: features of dims {16, 32, 64} planned into merged tables, a batch's
feature segments routed to them by mt_lookup_grouped, then per-table backward; every merged table matches an
oracle table fed the same routed segments (unique keys, inverse, counts and rows bit-exact; Adam rows within
the stated tolerances)."""
import numpy as np
import pytest
import torch

import oracle
import update_merged_table_gb300 as mt
from update_merged_table_gb300 import workloads as W
from numerics import ATOL, RTOL, assert_rows_close  # noqa: E402

pytestmark = pytest.mark.gpu

FEATURES = [(16, "f32", 4000), (32, "f32", 4000), (64, "bf16", 4000), (16, "f32", 4000), (64, "bf16", 4000),
            (32, "f32", 4000)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from update_merged_table_gb300 import build_lib
    build_lib.build()
    mt.load_library()
    oracle.build()


def batch(seed, per=1500):
    rng = np.random.default_rng(seed)
    sizes = [per, per // 2, per, 0, per + 7, per // 3]  # one feature absent from this batch
    parts = [W.zipf_ranks(rng, s, 1.1, 3000) - 1 for s in sizes]
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    return np.concatenate(parts).astype(np.int64), offs


def routed(ids, offs, placement, g):
    """The segments of group g's features, in feature order, with offsets and table ids (the routing, by hand)."""
    seg, o, t = [], [0], []
    for f, (gg, tid) in enumerate(placement):
        if gg != g:
            continue
        seg.append(ids[offs[f]:offs[f + 1]])
        o.append(o[-1] + offs[f + 1] - offs[f])
        t.append(tid)
    return np.concatenate(seg), np.array(o, np.int64), np.array(t, np.uint8)


def test_merged_tables_route_and_train():
    mtabs = mt.MergedTables(FEATURES, max_load=0.5, init_seed=3)
    assert [(g["dim"], g["row_dtype"], g["num_features"]) for g in mtabs.groups] == [
        (16, "f32", 2), (32, "f32", 2), (64, "bf16", 2)]
    refs = [oracle.Table(g["log2_slots"], g["dim"], row_dtype=oracle.BF16 if g["row_dtype"] == "bf16" else oracle.F32,
                         init_seed=3) for g in mtabs.groups]
    dev = mtabs.device
    for step in range(3):
        ids, offs = batch(step)
        res = mtabs.lookup(torch.from_numpy(ids).to(dev), offs)
        grads = []
        for g, (r, ref) in enumerate(zip(res, refs)):
            gids, goffs, gtids = routed(ids, offs, mtabs.placement, g)
            want = ref.lookup(gids, goffs, gtids)
            U = r.U
            assert U == want["U"]
            assert np.array_equal(r.unique_keys[:U].cpu().numpy().view(np.uint64), want["unique"])
            assert np.array_equal(r.inverse[:r.n].cpu().numpy(), want["inverse"])
            assert np.array_equal(r.counts[:U].cpu().numpy(), want["counts"])
            assert np.array_equal(r.rows.float().cpu().numpy(), want["rows"])
            assert (r.unique_keys[:U].cpu().numpy().view(np.uint64) >> np.uint64(56)).max() < 2  # two features each
            grads.append(W.grads_normal(10 * step + g, r.n, mtabs.groups[g]["dim"]))
        dgrads = [torch.from_numpy(gr).to(dev) for gr in grads]
        if step < 2:  # all tables' steps side by side (mt_backward_adam_grouped)
            gsums = mtabs.backward_adam(res, dgrads, want_gsum=True)
        else:  # one table at a time
            gsums = [t.backward_adam(r, gr, want_gsum=True) for t, r, gr in zip(mtabs.tables, res, dgrads)]
        for g, (r, ref) in enumerate(zip(res, refs)):
            ref_gsum = ref.backward_adam(grads[g], want_gsum=True)
            np.testing.assert_allclose(gsums[g][:r.U].cpu().numpy(), ref_gsum, rtol=RTOL, atol=ATOL)
            emb, m, v = mtabs.tables[g].read_rows(r.unique_rows[:r.U])
            e2, m2, v2, pr = ref.get_rows(r.unique_keys[:r.U].cpu().numpy().view(np.uint64))
            assert pr.all()
            assert_rows_close(emb.cpu().numpy(), e2, mtabs.groups[g]["row_dtype"])
            np.testing.assert_allclose(m.cpu().numpy(), m2, rtol=RTOL, atol=ATOL)
    assert all(t.error() == 0 for t in mtabs.tables)


def test_group_without_ids_in_the_batch():
    mtabs = mt.MergedTables([(16, "f32", 100), (32, "f32", 100)], max_load=0.5)
    ids = np.arange(50, dtype=np.int64)
    res = mtabs.lookup(torch.from_numpy(ids).to(mtabs.device), [0, 50, 50])
    assert res[0].U == 50 and res[1].n == 0 and res[1].U == 0
    grads = [torch.ones((50, 16), device=mtabs.device), torch.empty((0, 32), device=mtabs.device)]
    gs = mtabs.backward_adam(res, grads, want_gsum=True)
    assert torch.equal(gs[0][:50].cpu(), torch.ones(50, 16))
    assert [t.step for t in mtabs.tables] == [1, 1] and all(t.error() == 0 for t in mtabs.tables)


def test_more_groups_than_side_streams():
    """Six merged tables (six row shapes): more groups than the library's four side streams, so groups share
    streams; every table still matches its oracle table, lookup and a grouped backward step."""
    feats = [(8, "f32", 3000), (16, "f32", 3000), (24, "f32", 3000), (32, "f32", 3000), (48, "f32", 3000),
             (64, "bf16", 3000)]
    mtabs = mt.MergedTables(feats, max_load=0.5, init_seed=5)
    assert len(mtabs.groups) == 6
    refs = [oracle.Table(g["log2_slots"], g["dim"], row_dtype=oracle.BF16 if g["row_dtype"] == "bf16" else oracle.F32,
                         init_seed=5) for g in mtabs.groups]
    rng = np.random.default_rng(11)
    sizes = [900, 1300, 700, 1100, 500, 1600]
    ids = np.concatenate([W.zipf_ranks(rng, s, 1.1, 2500) - 1 for s in sizes]).astype(np.int64)
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    dev = mtabs.device
    for step in range(2):
        res = mtabs.lookup(torch.from_numpy(ids).to(dev), offs)
        grads, wants = [], []
        for g, (r, ref) in enumerate(zip(res, refs)):
            gids, goffs, gtids = routed(ids, offs, mtabs.placement, g)
            want = ref.lookup(gids, goffs, gtids)
            assert r.U == want["U"]
            assert np.array_equal(r.inverse[:r.n].cpu().numpy(), want["inverse"])
            assert np.array_equal(r.rows.float().cpu().numpy(), want["rows"])
            grads.append(W.grads_normal(50 * step + g, r.n, mtabs.groups[g]["dim"]))
        gsums = mtabs.backward_adam(res, [torch.from_numpy(x).to(dev) for x in grads], want_gsum=True)
        for g, (r, ref) in enumerate(zip(res, refs)):
            np.testing.assert_allclose(gsums[g][:r.U].cpu().numpy(), ref.backward_adam(grads[g], want_gsum=True),
                                       rtol=RTOL, atol=ATOL)
    assert all(t.error() == 0 for t in mtabs.tables) and [t.step for t in mtabs.tables] == [2] * 6


def test_grouped_calls_replay_as_cuda_graphs():
    """The grouped lookup and backward captured as CUDA graphs (their side streams become parallel branches)
    and replayed give the same tables as the same calls made eagerly on a twin."""
    eager = mt.MergedTables(FEATURES, max_load=0.5, init_seed=9)
    graphed = mt.MergedTables(FEATURES, max_load=0.5, init_seed=9)
    dev = eager.device
    batches = [batch(20 + j) for j in range(3)]
    ids = [torch.from_numpy(i).to(dev) for i, _ in batches]
    grads = [[torch.from_numpy(W.grads_normal(70 + 5 * j + g, sz, eager.groups[g]["dim"])).to(dev)
              for g, sz in enumerate(eager.group_sizes(o))] for j, (_, o) in enumerate(batches)]
    # step 0 eager on both (it also sizes every workspace); steps 1 and 2: eager against graph replays
    for m in (eager, graphed):
        m.backward_adam(m.lookup(ids[0], batches[0][1]), grads[0])
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream())
    graphs = []
    for j in (1, 2):
        gf, gb = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(gf, stream=stream):
            res = graphed.lookup(ids[j], batches[j][1])
        with torch.cuda.graph(gb, stream=stream):
            graphed.backward_adam(res, grads[j])
        graphs.append((gf, gb, res))
    for j, (gf, gb, res) in zip((1, 2), graphs):
        want = eager.lookup(ids[j], batches[j][1])
        eager.backward_adam(want, grads[j])
        gf.replay()
        gb.replay()
        torch.cuda.synchronize()
        for r, w in zip(res, want):
            assert r.U == w.U
            assert torch.equal(r.unique_keys[:r.U], w.unique_keys[:w.U])
            assert torch.equal(r.inverse[:r.n], w.inverse[:w.n])
            assert torch.equal(r.rows, w.rows)
    for te, tg in zip(eager.tables, graphed.tables):
        k_e, _ = te.export()
        k_g, _ = tg.export()
        assert np.array_equal(np.sort(k_e.cpu().numpy()), np.sort(k_g.cpu().numpy()))
        assert te.step == tg.step == 3 and te.error() == 0 and tg.error() == 0


def test_grouped_calls_from_two_host_threads():
    """Two host threads run grouped lookups and backward steps at the same time, each on its own merged tables
    and its own stream (each thread has its own side streams); every result and every table equals the same
    steps run one thread after the other on twin tables."""
    import threading

    def run(mtabs, steps, seed0, out):
        s = torch.cuda.Stream(device=mtabs.device)
        with torch.cuda.stream(s):
            for j in range(steps):
                ids, offs = batch(seed0 + j)
                res = mtabs.lookup(torch.from_numpy(ids).to(mtabs.device), offs)
                grads = [torch.from_numpy(W.grads_normal(seed0 + 7 * j + g, sz, mtabs.groups[g]["dim"])).to(mtabs.device)
                         for g, sz in enumerate(mtabs.group_sizes(offs))]
                mtabs.backward_adam(res, grads)
                out.append([(r.U, r.unique_keys[:r.U].clone(), r.inverse[:r.n].clone(), r.rows.clone()) for r in res])
        s.synchronize()

    seeds = (40, 60)
    twins = [mt.MergedTables(FEATURES, max_load=0.5, init_seed=s) for s in seeds]
    want = [[], []]
    for k in range(2):
        run(twins[k], 3, seeds[k], want[k])
    tabs = [mt.MergedTables(FEATURES, max_load=0.5, init_seed=s) for s in seeds]
    got = [[], []]
    errs = []

    def worker(k):
        try:
            run(tabs[k], 3, seeds[k], got[k])
        except Exception as e:  # surfaced below
            errs.append(e)

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errs, errs
    torch.cuda.synchronize()
    for k in range(2):
        assert len(got[k]) == len(want[k]) == 3
        for gs, ws in zip(got[k], want[k]):
            for (gu, gk, gi, gr), (wu, wk, wi, wr) in zip(gs, ws):
                assert gu == wu and torch.equal(gk, wk) and torch.equal(gi, wi) and torch.equal(gr, wr)
        for tg, tw in zip(tabs[k].tables, twins[k].tables):
            kg, rg = tg.export()
            kw, rw = tw.export()
            og, ow = torch.argsort(kg), torch.argsort(kw)
            assert torch.equal(kg[og], kw[ow])
            assert torch.equal(tg.read_rows(rg[og])[0], tw.read_rows(rw[ow])[0])
            assert tg.step == tw.step == 3 and tg.error() == 0 and tw.error() == 0
