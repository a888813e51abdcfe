"""mt_lookup_static: the lookup for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace (an operator interface that
passes only inputs and outputs, or a process whose device memory budget is
fixed); mt_lookup_static takes its scratch from a static device array
instead.  Through the C ABI, two calls in a row must give exactly what
mt_lookup gives on an identically configured table, and a batch above the
fixed maximum must be refused.  (This file is collected last on purpose.)
"""
import ctypes

import numpy as np
import pytest
import torch

import update_merged_table_gb300 as mt
from update_merged_table_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from update_merged_table_gb300 import build_lib
    build_lib.build()
    mt.load_library()


def _lookup_static(tab, ids, b, res, insert_missing=True):
    fo = np.ascontiguousarray(b.feat_offsets, np.int64)
    ti = np.ascontiguousarray(b.table_ids, np.uint8)
    st = res.as_struct()
    return mt.load_library().mt_lookup_static(
        tab.h, ids.data_ptr(), b.n, fo.ctypes.data_as(ctypes.c_void_p), ti.ctypes.data_as(ctypes.c_void_p),
        fo.size - 1, int(insert_missing), res.rows.data_ptr(), ctypes.byref(st),
        torch.cuda.current_stream().cuda_stream)


def test_static_lookup_matches_lookup_on_two_calls():
    dev = torch.device("cuda", torch.cuda.current_device())
    ref = mt.Table(16, 32, row_dtype="bf16", device=dev)
    tab = mt.Table(16, 32, row_dtype="bf16", device=dev)
    # two batches in a row: the second repeats the first's hot IDs and brings new ones
    for seed in (1, 2):
        b = W.merged_batch(seed, per_table=4096)
        ids = torch.from_numpy(b.ids).to(dev)
        want = ref.lookup(ids, b.feat_offsets, b.table_ids)
        got = tab.new_result(b.n)
        assert _lookup_static(tab, ids, b, got) == mt.MT_OK
        torch.cuda.synchronize()
        U = want.U
        assert got.U == U
        assert torch.equal(got.unique_keys[:U], want.unique_keys[:U])
        assert torch.equal(got.inverse[:b.n], want.inverse[:b.n])
        assert torch.equal(got.counts[:U], want.counts[:U])
        assert torch.equal(got.unique_rows[:U] >= 0, want.unique_rows[:U] >= 0)
        assert torch.equal(got.rows.view(torch.int16), want.rows.view(torch.int16))
        # same backward on both tables: the same rows within the tests' tolerance
        g = torch.from_numpy(W.grads_normal(seed + 7, b.n, 32)).to(dev)
        ref.backward_adam(want, g)
        tab.backward_adam(got, g)
        e1, m1, v1 = ref.read_rows(want.unique_rows[:U])
        e2, m2, v2 = tab.read_rows(got.unique_rows[:U])
        b1 = e1.to(torch.bfloat16).view(torch.int16).int()
        b2 = e2.to(torch.bfloat16).view(torch.int16).int()
        assert (b1 - b2).abs().max().item() <= 1
        torch.testing.assert_close(m2, m1, rtol=1e-5, atol=1e-6)
        torch.testing.assert_close(v2, v1, rtol=1e-5, atol=1e-9)
    assert tab.error() == 0 and ref.error() == 0


def test_static_lookup_takes_the_largest_batch():
    """Exactly MT_LOOKUP_STATIC_MAX_IDS IDs fit the static workspace; same result as mt_lookup."""
    dev = torch.device("cuda", torch.cuda.current_device())
    n = mt.LOOKUP_STATIC_MAX_IDS
    ids = W.bijection32(W.zipf_ranks(np.random.default_rng(5), n, 1.1, 1 << 20))
    b = W.single_feature(ids)
    ref = mt.Table(18, 8, device=dev)
    tab = mt.Table(18, 8, device=dev)
    d_ids = torch.from_numpy(b.ids).to(dev)
    want = ref.lookup(d_ids, b.feat_offsets, b.table_ids)
    got = tab.new_result(n)
    assert _lookup_static(tab, d_ids, b, got) == mt.MT_OK
    torch.cuda.synchronize()
    U = want.U
    assert got.U == U
    assert torch.equal(got.unique_keys[:U], want.unique_keys[:U])
    assert torch.equal(got.inverse[:n], want.inverse[:n])
    assert torch.equal(got.rows, want.rows)
    assert tab.error() == 0


def test_static_lookup_refuses_oversized_batch():
    dev = torch.device("cuda", torch.cuda.current_device())
    tab = mt.Table(10, 8, device=dev)
    n = mt.LOOKUP_STATIC_MAX_IDS + 1
    b = W.single_feature(np.zeros(n, np.int64))
    res = tab.new_result(n)
    assert _lookup_static(tab, torch.zeros(n, dtype=torch.int64, device=dev), b, res) == mt.MT_ETOOBIG
    assert tab.stats()["live"] == 0  # nothing was enqueued
