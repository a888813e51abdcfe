"""CPU oracle for the merged dynamic embedding table -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline (reference)
leg of ``bench.py`` may import this package.  The library path never does: it
has no CPU fallback and fails loudly when its CUDA library is missing.

The oracle is a plain single-threaded C++ library (``oracle.cpp``) loaded with
ctypes.  It shares no code with the CUDA path; ``oracle.cpp`` says which
passage of the pages each function follows.

Pins (tests/test_oracle_pins.py) tie each part to something other than itself:
Theorem 1 of MTGenRec by brute force, unique/inverse against a sort-based
unique and hand-worked goldens, Philox4x64-10 against numpy's independent
``numpy.random.Philox``, bf16 rounding against torch, the gradient sum against
``torch.index_add_`` in float64, Adam against its closed form at t = 1 and
against ``torch.optim.Adam``, and the table against a Python dict under random
insert/erase scripts.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")

F32, BF16 = 0, 1
EMPTY = (1 << 64) - 1
TOMB = (1 << 64) - 2

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (no FMA contraction: each float op rounds once)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                               "-shared", _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P, I64, U64, U32, I32, F = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32,
                                    ctypes.c_int, ctypes.c_float)
        sig = {
            "orc_philox4x64_10": (None, [P, P, P]),
            "orc_init_row": (None, [U64, U64, F, U32, I32, P]),
            "orc_bf16_bits": (ctypes.c_uint16, [F]),
            "orc_home_slot": (U64, [U64, U64, U32]),
            "orc_encode": (None, [P, I64, P, P, I32, P, P]),
            "orc_unique": (I64, [P, P, I64, P, P, P]),
            "orc_unique_sort": (I64, [P, P, I64, P, P]),
            "orc_table_new": (P, [U32, U32, I32, U64, U64, U64, F, U64, I64, I32]),
            "orc_table_free": (None, [P]),
            "orc_lookup": (I64, [P, P, I64, P, P, I32, I32, P, P, P, P, P]),
            "orc_backward_adam": (I32, [P, P, I32, F, F, F, F, P]),
            "orc_erase": (None, [P, P, I64, P]),
            "orc_insert_keys": (I64, [P, P, I64]),
            "orc_get_row": (I32, [P, U64, P, P, P]),
            "orc_get_rows": (None, [P, P, I64, P, P, P, P]),
            "orc_live_count": (I64, [P]),
            "orc_live_keys": (I64, [P, P, I64]),
            "orc_step": (I64, [P]),
            "orc_error": (I32, [P]),
            "orc_sim_stats": (I32, [P, P, P, P, P]),
            "orc_sim_occupancy": (I32, [P, P]),
            "orc_sim_new": (P, [U32, U64, U64, U64]),
            "orc_sim_free": (None, [P]),
            "orc_sim_insert": (I32, [P, U64]),
            "orc_sim_erase": (I32, [P, U64]),
            "orc_sim_find": (I64, [P, U64]),
            "orc_sim_placed": (I64, [P, U64]),
            "orc_sim_sequence": (None, [P, U64, U64, P]),
            "orc_sim_raw_occupancy": (I64, [P, P]),
            "orc_pool_forward": (I32, [P, P, I64, I32, P]),
            "orc_backward_adam_pooled": (I32, [P, P, I64, I32, P, F, F, F, F, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- plain functions ---------------------------------------------------------

def philox4x64_10(ctr, key) -> np.ndarray:
    """Philox4x64-10 block function: 4 counter words, 2 key words -> 4 words."""
    c = _c(ctr, np.uint64)
    k = _c(key, np.uint64)
    out = np.zeros(4, np.uint64)
    lib().orc_philox4x64_10(_p(c), _p(k), _p(out))
    return out


def init_row(key: int, seed: int, scale: float, dim: int, dtype: int = F32) -> np.ndarray:
    """Initial embedding of `key` as float32 (values already rounded to the storage dtype)."""
    out = np.zeros(dim, np.float32)
    lib().orc_init_row(int(key), int(seed), float(scale), dim, dtype, _p(out))
    return out


def bf16_bits(x: float) -> int:
    return int(lib().orc_bf16_bits(float(x)))


def home_slot(key: int, seed: int, n: int) -> int:
    return int(lib().orc_home_slot(int(key), int(seed), n))


def default_init_scale(dim: int) -> float:
    """fp32(1/sqrt(dim)), computed in double."""
    return float(np.float32(1.0 / np.sqrt(float(dim))))


def encode(ids, feat_offsets, table_ids):
    ids = _c(ids, np.int64)
    fo = _c(feat_offsets, np.int64)
    ti = _c(table_ids, np.uint8)
    keys = np.zeros(ids.size, np.uint64)
    valid = np.zeros(ids.size, np.uint8)
    lib().orc_encode(_p(ids), ids.size, _p(fo), _p(ti), ti.size, _p(keys), _p(valid))
    return keys, valid.astype(bool)


def unique(keys, valid=None, method: str = "map"):
    """(uniq, inverse, counts) in first-occurrence order.  counts is None for method="sort"."""
    keys = _c(keys, np.uint64)
    valid = np.ones(keys.size, np.uint8) if valid is None else _c(valid, np.uint8)
    uniq = np.zeros(keys.size, np.uint64)
    inv = np.zeros(keys.size, np.int32)
    if method == "map":
        cnt = np.zeros(keys.size, np.int32)
        U = lib().orc_unique(_p(keys), _p(valid), keys.size, _p(uniq), _p(inv), _p(cnt))
        return uniq[:U].copy(), inv, cnt[:U].copy()
    U = lib().orc_unique_sort(_p(keys), _p(valid), keys.size, _p(uniq), _p(inv))
    return uniq[:U].copy(), inv, None


class Table:
    """The oracle's dynamic table: an unordered_map from merged key to row."""

    def __init__(self, log2_slots: int, dim: int, row_dtype: int = F32, probe_step: int = 1, hash_seed: int = 0,
                 init_seed: int = 0, init_scale: float | None = None, max_probes: int = 0, num_rows: int = 0,
                 simulate: bool = False):
        if init_scale is None:
            init_scale = default_init_scale(dim)
        self.dim, self.dtype, self.log2_slots = dim, row_dtype, log2_slots
        self.init_seed, self.init_scale = init_seed, init_scale
        self._U = 0
        self.h = lib().orc_table_new(log2_slots, dim, row_dtype, probe_step, hash_seed, init_seed, init_scale,
                                     max_probes, num_rows, 1 if simulate else 0)
        if not self.h:
            raise ValueError("oracle rejected the table configuration")

    def __del__(self):
        h = getattr(self, "h", None)
        if h:
            lib().orc_table_free(h)
            self.h = None

    def lookup(self, ids, feat_offsets=None, table_ids=None, insert_missing=True, gather=True):
        ids = _c(ids, np.int64)
        n = ids.size
        fo = _c([0, n] if feat_offsets is None else feat_offsets, np.int64)
        ti = _c([0] if table_ids is None else table_ids, np.uint8)
        out = np.zeros((n, self.dim), np.float32) if gather else None
        uniq = np.zeros(n, np.uint64)
        inv = np.zeros(n, np.int32)
        cnt = np.zeros(n, np.int32)
        present = np.zeros(n, np.uint8)
        U = lib().orc_lookup(self.h, _p(ids), n, _p(fo), _p(ti), ti.size, 1 if insert_missing else 0, _p(out),
                             _p(uniq), _p(inv), _p(cnt), _p(present))
        self._U = int(U)
        return dict(rows=out, unique=uniq[:U].copy(), inverse=inv, counts=cnt[:U].copy(),
                    present=present[:U].astype(bool), U=int(U))

    def backward_adam(self, grads, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, grad_dtype=F32, want_gsum=False):
        """grads: float32 [n, dim], or uint16 bf16 bit patterns [n, dim] with grad_dtype=BF16."""
        g = np.ascontiguousarray(grads)
        if grad_dtype == BF16:
            if g.dtype != np.uint16:
                raise TypeError("bf16 grads are passed as uint16 bit patterns")
        else:
            g = g.astype(np.float32, copy=False)
        gsum = np.zeros((self._U, self.dim), np.float32) if want_gsum else None
        rc = lib().orc_backward_adam(self.h, _p(g), grad_dtype, lr, beta1, beta2, eps, _p(gsum))
        if rc != 0:
            raise RuntimeError(f"oracle backward failed: {rc}")
        return gsum

    def pool_forward(self, bag_offsets, mode: int = 0):
        """Pooled rows [B, dim] fp32 of the last lookup: per bag of positions [bo[b], bo[b+1]) the sum
        (mode 0) or mean (mode 1) of the rows, in double, rounded once."""
        bo = _c(bag_offsets, np.int64)
        B = bo.size - 1
        out = np.zeros((max(B, 0), self.dim), np.float32)
        if lib().orc_pool_forward(self.h, _p(bo), B, mode, _p(out)) != 0:
            raise ValueError("bag offsets must be non-decreasing within [0, n]")
        return out

    def backward_adam_pooled(self, bag_offsets, dpooled, mode: int = 0, lr=1e-3, beta1=0.9, beta2=0.999,
                             eps=1e-8, want_gsum=False):
        """Backward of pool_forward followed by the table's backward + Adam; dpooled: fp32 [B, dim]."""
        bo = _c(bag_offsets, np.int64)
        dp = _c(dpooled, np.float32)
        gsum = np.zeros((self._U, self.dim), np.float32) if want_gsum else None
        rc = lib().orc_backward_adam_pooled(self.h, _p(bo), bo.size - 1, mode, _p(dp), lr, beta1, beta2, eps,
                                            _p(gsum))
        if rc != 0:
            raise ValueError("bag offsets must be non-decreasing within [0, n]")
        return gsum

    def insert_keys(self, keys) -> int:
        k = _c(keys, np.uint64)
        return int(lib().orc_insert_keys(self.h, _p(k), k.size))

    def get_row(self, key: int):
        e = np.zeros(self.dim, np.float32)
        m = np.zeros(self.dim, np.float32)
        v = np.zeros(self.dim, np.float32)
        ok = lib().orc_get_row(self.h, int(key), _p(e), _p(m), _p(v))
        return (e, m, v) if ok else None

    def get_rows(self, keys):
        """(emb, m, v, present) for an array of merged keys; absent keys give zero rows."""
        k = _c(keys, np.uint64)
        e = np.zeros((k.size, self.dim), np.float32)
        m = np.zeros_like(e)
        v = np.zeros_like(e)
        pr = np.zeros(k.size, np.uint8)
        lib().orc_get_rows(self.h, _p(k), k.size, _p(e), _p(m), _p(v), _p(pr))
        return e, m, v, pr.astype(bool)

    def erase(self, keys):
        k = _c(keys, np.uint64)
        found = np.zeros(k.size, np.uint8)
        lib().orc_erase(self.h, _p(k), k.size, _p(found))
        return found.astype(bool)

    @property
    def live(self) -> int:
        return int(lib().orc_live_count(self.h))

    def live_keys(self) -> np.ndarray:
        n = self.live
        out = np.zeros(n, np.uint64)
        lib().orc_live_keys(self.h, _p(out), n)
        return out

    @property
    def step(self) -> int:
        return int(lib().orc_step(self.h))

    @property
    def error(self) -> int:
        return int(lib().orc_error(self.h))

    def sim_stats(self):
        live = np.zeros(1, np.int64)
        tombs = np.zeros(1, np.int64)
        hist = np.zeros(64, np.int64)
        disp = np.zeros(1, np.int64)
        rc = lib().orc_sim_stats(self.h, _p(live), _p(tombs), _p(hist), _p(disp))
        if rc != 0:
            raise RuntimeError("table was created without the simulator")
        return dict(live=int(live[0]), tombstones=int(tombs[0]), hist=hist, total_displacement=int(disp[0]))

    def sim_occupancy(self) -> np.ndarray:
        out = np.zeros(1 << self.log2_slots, np.uint8)
        if lib().orc_sim_occupancy(self.h, _p(out)) != 0:
            raise RuntimeError("table was created without the simulator")
        return out


class Simulator:
    """Serial open-addressing table with probe sequence h_t = (h0 + t*S) mod 2^n."""

    def __init__(self, log2_slots: int, probe_step: int, hash_seed: int = 0, max_probes: int = 0):
        self.M = 1 << log2_slots
        self.h = lib().orc_sim_new(log2_slots, probe_step, hash_seed, max_probes)

    def __del__(self):
        h = getattr(self, "h", None)
        if h:
            lib().orc_sim_free(h)
            self.h = None

    def insert(self, key: int) -> int:
        return int(lib().orc_sim_insert(self.h, int(key)))

    def erase(self, key: int) -> bool:
        return bool(lib().orc_sim_erase(self.h, int(key)))

    def find(self, key: int) -> int:
        return int(lib().orc_sim_find(self.h, int(key)))

    def placed(self, key: int) -> int:
        return int(lib().orc_sim_placed(self.h, int(key)))

    def sequence(self, h0: int, count: int) -> np.ndarray:
        out = np.zeros(count, np.uint64)
        lib().orc_sim_sequence(self.h, h0, count, _p(out))
        return out

    def occupancy(self):
        """(per-slot code 0 empty / 1 live / 2 tombstone, total displacement)."""
        out = np.zeros(self.M, np.uint8)
        D = int(lib().orc_sim_raw_occupancy(self.h, _p(out)))
        return out, D
