"""The C-ABI library on a machine without a GPU: it builds, loads, exports every
symbol include/mt.h declares, and rejects bad arguments on the host (no
compute call is made)."""
import ctypes
import os
import re

import pytest

import update_merged_table_gb300 as mt
from update_merged_table_gb300 import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return mt.load_library()


def _declared():
    src = open(os.path.join(ROOT, "include", "mt.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mt_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("mt_table_create", "mt_lookup", "mt_backward_adam", "mt_erase", "mt_stats"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    assert set(_declared()) == set(mt.ABI_FUNCTIONS)


def test_abi_version_and_strerror(lib):
    assert lib.mt_abi_version() == mt.ABI_VERSION
    for code in (mt.MT_OK, mt.MT_EINVAL, mt.MT_ENOSPACE, mt.MT_EFULL, mt.MT_EKEY, mt.MT_ECUDA, mt.MT_ETOOBIG):
        assert lib.mt_strerror(code) and lib.mt_strerror(code) != b"unknown status"
    assert lib.mt_strerror(-99) == b"unknown status"


def _cfg(**kw):
    base = dict(log2_slots=10, dim=16, row_dtype=mt.MT_F32, max_probes=0, probe_step=1, hash_seed=0, init_seed=0,
                init_scale=0.0, flags=0, num_rows=0)
    base.update(kw)
    return mt._Config(*[base[f] for f, _ in mt._Config._fields_])


def test_table_bytes_layout(lib):
    c = _cfg(log2_slots=10, dim=16)
    nb = lib.mt_table_bytes(ctypes.byref(c))
    # header 1 KiB + 1024 slots x 16 B + 1024 x int32 free list + 1024 rows x (16 + 16 + 16) x 4 B
    assert nb == 1024 + 1024 * 16 + 1024 * 4 + 1024 * 16 * 4 * 3
    c = _cfg(log2_slots=10, dim=64, row_dtype=mt.MT_BF16, num_rows=100)
    # 100 rows x (128 B bf16 emb + 256 B m + 256 B v); free list 400 B padded to 512
    assert lib.mt_table_bytes(ctypes.byref(c)) == 1024 + 1024 * 16 + 512 + 100 * 640


@pytest.mark.parametrize("kw", [
    dict(probe_step=2),                 # Theorem 1: an even step does not cover the table
    dict(probe_step=1024),              # == 0 mod M
    dict(log2_slots=0), dict(log2_slots=32),
    dict(dim=0), dict(dim=6), dict(dim=2048),
    dict(row_dtype=mt.MT_BF16, dim=12),  # bf16 rows need dim % 8 == 0
    dict(row_dtype=7),
    dict(num_rows=-1), dict(num_rows=2048),
    dict(flags=1),
    dict(init_scale=float("nan")),
])
def test_invalid_configs_rejected_on_host(lib, kw):
    c = _cfg(**kw)
    assert lib.mt_table_bytes(ctypes.byref(c)) == 0
    h = ctypes.c_void_p()
    assert lib.mt_table_create(ctypes.byref(c), None, 0, None, ctypes.byref(h)) == mt.MT_EINVAL
    assert not h.value


def test_odd_steps_accepted(lib):
    for S in (1, 3, 1023, 0x9E3779B97F4A7C15):
        assert lib.mt_table_bytes(ctypes.byref(_cfg(probe_step=S))) > 0


def test_keystore_and_rows_bytes(lib):
    c = _cfg(log2_slots=10, dim=16)
    ks = lib.mt_keystore_bytes(ctypes.byref(c))
    assert ks == 1024 + 1024 * 16 + 1024 * 4  # header, slots, free list
    assert lib.mt_rows_bytes(ctypes.byref(c), 1000) == 1000 * 16 * 4 * 3
    assert lib.mt_rows_bytes(ctypes.byref(c), 3) == 768  # 3 x 192 B, padded to 256
    assert lib.mt_table_bytes(ctypes.byref(c)) == ks + lib.mt_rows_bytes(ctypes.byref(c), 1024)
    assert lib.mt_rows_bytes(ctypes.byref(c), -1) == 0


def test_create_split_checks_buffers(lib):
    c = _cfg(log2_slots=10, dim=16)
    h = ctypes.c_void_p()
    ks = lib.mt_keystore_bytes(ctypes.byref(c))
    rb = lib.mt_rows_bytes(ctypes.byref(c), 1024)
    assert lib.mt_table_create_split(ctypes.byref(c), None, ks, 1 << 20, rb, None, ctypes.byref(h)) == mt.MT_ENOSPACE
    assert lib.mt_table_create_split(ctypes.byref(c), 1 << 20, ks - 1, 1 << 30, rb, None,
                                     ctypes.byref(h)) == mt.MT_ENOSPACE
    # the key store and the rows must not overlap (checked before any device call)
    assert lib.mt_table_create_split(ctypes.byref(c), 1 << 20, ks, (1 << 20) + 256, rb, None,
                                     ctypes.byref(h)) == mt.MT_EINVAL
    assert not h.value


def test_create_needs_space(lib):
    c = _cfg()
    h = ctypes.c_void_p()
    assert lib.mt_table_create(ctypes.byref(c), None, 1 << 20, None, ctypes.byref(h)) == mt.MT_ENOSPACE
    # misaligned arena
    assert lib.mt_table_create(ctypes.byref(c), 16, 1 << 30, None, ctypes.byref(h)) == mt.MT_ENOSPACE


def test_null_handles_rejected(lib):
    r = mt._Result(0, 0, 0, 0, 0)
    assert lib.mt_lookup(None, None, 0, None, None, 1, 1, None, ctypes.byref(r), None, 0, None) == mt.MT_EINVAL
    assert lib.mt_backward_adam(None, ctypes.byref(r), 0, None, 0, None, None, None, 0, None) == mt.MT_EINVAL
    assert lib.mt_erase(None, None, 0, None, None, 0, None) == mt.MT_EINVAL
    assert lib.mt_stats(None, None, None) == mt.MT_EINVAL
    assert lib.mt_table_destroy(None) == mt.MT_EINVAL
    assert lib.mt_step(None) == -1
    assert lib.mt_lookup_workspace_bytes(None, 10) == 0
    assert lib.mt_erase_workspace_bytes(1000) >= 4000
    assert lib.mt_compact(None, None, 0, None, None) == mt.MT_EINVAL
    assert lib.mt_table_grow(None, None, None, 0, None, 0, None) == mt.MT_EINVAL
    assert lib.mt_compact_workspace_bytes(None) == 0
    assert lib.mt_import(None, None, 0, None, None, None, None, 0, None) == mt.MT_EINVAL
    assert lib.mt_import_workspace_bytes(1000) >= 4000 and lib.mt_import_workspace_bytes(-1) == 0
    st, b1, b2 = ctypes.c_int64(), ctypes.c_double(), ctypes.c_double()
    assert lib.mt_get_adam_state(None, ctypes.byref(st), ctypes.byref(b1), ctypes.byref(b2), None) == mt.MT_EINVAL
    assert lib.mt_set_adam_state(None, 0, 1.0, 1.0, None) == mt.MT_EINVAL


def test_set_adam_state_rejects_inconsistent_state(lib):
    """Arguments are checked before the handle is used: a zeroed stand-in handle (never a real table
    here) shows which combinations pass validation (they then fail at the CUDA call: no GPU)."""
    fake = ctypes.create_string_buffer(4096)
    h = ctypes.cast(fake, ctypes.c_void_p)
    for step, b1, b2 in [(0, 0.9, 1.0), (0, 1.0, 0.999), (3, 1.0, 0.5), (3, 0.5, 1.0), (-1, 1.0, 1.0),
                         (2, float("nan"), 0.5), (2, 0.5, 1.5), (2, -0.1, 0.5)]:
        assert lib.mt_set_adam_state(h, step, b1, b2, None) == mt.MT_EINVAL, (step, b1, b2)
    for step, b1, b2 in [(0, 1.0, 1.0), (3, 0.729, 0.997002999), (5, 0.0, 0.0)]:
        rc = lib.mt_set_adam_state(h, step, b1, b2, None)
        assert rc != mt.MT_EINVAL, (step, b1, b2)


def test_product_path_has_no_oracle_or_fallback():
    """The package never imports the oracle and has no CPU path."""
    pkg = os.path.join(ROOT, "update_merged_table_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "liboracle" not in text, f


def test_grouped_lookup_workspace_covers_any_split(lib):
    """The grouped lookup gives each group its own lookup workspace; the size it asks for covers the routed
    IDs plus the groups' workspaces for any split of the batch into F feature segments and groups."""
    import numpy as np
    rng = np.random.default_rng(0)
    table = ctypes.c_void_p(16)  # the workspace-size query only checks the handle is not NULL

    def align(x):
        return (x + 255) // 256 * 256

    for n in (1, 100, 2047, 4096, 65536, 1 << 20, 3_000_000):
        for _ in range(25):
            F = int(rng.integers(1, mt.MAX_FEATURES + 1))
            cuts = np.sort(rng.integers(0, n + 1, F - 1))
            sizes = np.diff(np.concatenate([[0], cuts, [n]]))
            need = align(n * 8) + sum(align(lib.mt_lookup_workspace_bytes(table, int(s))) for s in sizes if s > 0)
            assert lib.mt_lookup_grouped_workspace_bytes(n, F) >= need, (n, sizes)
    for F in (2, 17, mt.MAX_FEATURES):  # every group one ID past a tile: the most rounding per group
        sizes = [2049] * F
        n = sum(sizes)
        need = align(n * 8) + sum(align(lib.mt_lookup_workspace_bytes(table, s)) for s in sizes)
        assert lib.mt_lookup_grouped_workspace_bytes(n, F) >= need, F
    assert lib.mt_lookup_grouped_workspace_bytes(10, 0) == 0
    assert lib.mt_lookup_grouped_workspace_bytes(10, mt.MAX_FEATURES + 1) == 0


def test_grouped_backward_rejects_bad_arguments_on_host(lib):
    res = (ctypes.c_byte * 64)()
    gn = (ctypes.c_int64 * 1)(0)
    assert lib.mt_backward_grouped_workspace_bytes(None, 1, gn) == 0
    assert lib.mt_backward_adam_grouped(None, 1, res, gn, None, mt.MT_F32, None, None, None, 0, None) == mt.MT_EINVAL
    tabs = (ctypes.c_void_p * 1)(None)
    assert lib.mt_backward_adam_grouped(tabs, 1, res, gn, None, mt.MT_F32, None, None, None, 0, None) == mt.MT_EINVAL
    assert lib.mt_backward_adam_grouped(tabs, 0, res, gn, None, mt.MT_F32, None, None, None, 0, None) == mt.MT_EINVAL


def test_grouped_lookup_rejects_a_table_in_two_groups(lib):
    """The groups' lookups run side by side, so one table may not serve two groups (checked on the host,
    before any handle is used)."""
    t = ctypes.c_void_p(16)
    tabs = (ctypes.c_void_p * 2)(t, t)
    pl = (ctypes.c_int32 * 2)(0, 0)  # one feature: group 0, table id 0
    fo = (ctypes.c_int64 * 2)(0, 0)
    res = (ctypes.c_byte * 256)()
    gn = (ctypes.c_int64 * 2)()
    ws = ctypes.c_void_p(4096)
    assert lib.mt_lookup_grouped(tabs, 2, pl, None, 0, fo, 1, 1, None, res, gn, ws, 1 << 20, None) == mt.MT_EINVAL


def test_pooled_and_sharded_calls_reject_bad_handles_on_host(lib):
    """The pooled-bag and sharded entry points refuse missing handles, sizes and modes before any device
    call (no GPU here)."""
    r = mt._Result(0, 0, 0, 0, 0)
    assert lib.mt_pool_workspace_bytes(None, 10) == 0
    assert lib.mt_pool_forward(None, ctypes.byref(r), 0, None, 1, mt.POOL_SUM, None, None, 0, None) == mt.MT_EINVAL
    assert lib.mt_backward_pooled_workspace_bytes(None, 10, 10) == 0
    assert lib.mt_backward_adam_pooled(None, ctypes.byref(r), 0, None, 1, mt.POOL_SUM, None, None, None, None, 0,
                                       None) == mt.MT_EINVAL
    out = ctypes.c_void_p(1)
    assert lib.mt_shard_group_create(None, 2, ctypes.byref(out)) == mt.MT_EINVAL and out.value is None
    shards = (ctypes.c_void_p * 2)(None, None)
    assert lib.mt_shard_group_create(shards, 0, ctypes.byref(out)) == mt.MT_EINVAL
    max_shards = int(re.search(r"#define MT_MAX_SHARDS (\d+)", open(os.path.join(ROOT, "include", "mt.h")).read()).group(1))
    assert lib.mt_shard_group_create(shards, max_shards + 1, ctypes.byref(out)) == mt.MT_EINVAL
    assert lib.mt_shard_group_create(shards, 2, None) == mt.MT_EINVAL
    assert lib.mt_shard_group_destroy(None) == mt.MT_EINVAL
    n = (ctypes.c_int64 * 2)(10, 10)
    assert lib.mt_shard_workspace_bytes(None, n) == 0
    assert lib.mt_shard_lookup(None, None, n, None, None, 1, 1, None, None, None, 0, None) == mt.MT_EINVAL
    assert lib.mt_shard_backward_adam(None, None, None, mt.MT_F32, None, None, None, 0, None) == mt.MT_EINVAL
