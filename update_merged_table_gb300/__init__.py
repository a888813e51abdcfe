"""Merged dynamic embedding table on GB300: thin Python binding of ``libmt.so``.

The binding only marshals arguments: it allocates device memory with torch,
passes raw pointers and the current CUDA stream to the C ABI declared in
``include/mt.h``, and wraps the outputs as torch tensors.  Every step of the
lookup and backward path runs in the library's CUDA kernels.  There is no CPU
fallback: without the built library every call raises.

The path follows "MTGenRec: An Efficient Distributed Training System for
Generative Recommendation Models in Meituan" (TL;DR and abstract: dynamic
hash embedding tables whose keys are inserted and deleted while training
runs, feature tables merged into one table, ID deduplication in two stages; Theorem 1: probing h_t = (h0 + t*S) mod
2^n with odd S) and "MTGR" section 5 (Embedding Management, Embedding Lookup).
"""
from __future__ import annotations

import ctypes
import dataclasses
import os

import numpy as np

__all__ = ["Table", "ShardGroup", "MergedTables", "plan_merge", "LookupResult", "load_library", "MTError", "MT_F32", "MT_BF16", "POOL_SUM", "POOL_MEAN",
           "KEY_EMPTY", "KEY_TOMBSTONE",
           "ABI_FUNCTIONS", "profile_enable", "profile_report", "kernel_launches"]

MT_OK, MT_EINVAL, MT_ENOSPACE, MT_EFULL, MT_EKEY, MT_ECUDA, MT_ETOOBIG = 0, -1, -2, -3, -4, -5, -6
ABI_VERSION = 2
LOOKUP_STATIC_MAX_IDS = 65536
MT_F32, MT_BF16 = 0, 1
POOL_SUM, POOL_MEAN = 0, 1
KEY_EMPTY = (1 << 64) - 1
KEY_TOMBSTONE = (1 << 64) - 2
HIST_BINS = 64
MAX_FEATURES = 256

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmt.so")


class MTError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: status {code} ({_strerror(code)})")
        self.code = code


class _Config(ctypes.Structure):
    _fields_ = [("log2_slots", ctypes.c_uint32), ("dim", ctypes.c_uint32), ("row_dtype", ctypes.c_uint32),
                ("max_probes", ctypes.c_uint32), ("probe_step", ctypes.c_uint64), ("hash_seed", ctypes.c_uint64),
                ("init_seed", ctypes.c_uint64), ("init_scale", ctypes.c_float), ("flags", ctypes.c_uint32),
                ("num_rows", ctypes.c_int64)]


class _Result(ctypes.Structure):
    _fields_ = [("unique_keys", ctypes.c_void_p), ("inverse", ctypes.c_void_p), ("counts", ctypes.c_void_p),
                ("unique_rows", ctypes.c_void_p), ("num_unique", ctypes.c_void_p), ("ranks", ctypes.c_void_p)]


class _Adam(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float), ("eps", ctypes.c_float)]


class _Stats(ctypes.Structure):
    _fields_ = [("live", ctypes.c_int64), ("tombstones", ctypes.c_int64), ("capacity", ctypes.c_int64),
                ("num_rows", ctypes.c_int64), ("rows_free", ctypes.c_int64), ("step", ctypes.c_int64),
                ("total_displacement", ctypes.c_int64), ("load_factor", ctypes.c_double),
                ("probe_hist", ctypes.c_int64 * HIST_BINS), ("device_error", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


_P, _I64, _SZ, _I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int
# name -> (restype, argtypes); every entry point of include/mt.h
ABI_FUNCTIONS = {
    "mt_abi_version": (_I32, []),
    "mt_strerror": (ctypes.c_char_p, [_I32]),
    "mt_table_bytes": (_SZ, [_P]),
    "mt_table_create": (_I32, [_P, _P, _SZ, _P, _P]),
    "mt_table_destroy": (_I32, [_P]),
    "mt_table_config": (_I32, [_P, _P]),
    "mt_table_grow": (_I32, [_P, _P, _P, _SZ, _P, _SZ, _P]),
    "mt_keystore_bytes": (_SZ, [_P]),
    "mt_rows_bytes": (_SZ, [_P, _I64]),
    "mt_table_create_split": (_I32, [_P, _P, _SZ, _P, _SZ, _P, _P]),
    "mt_lookup_workspace_bytes": (_SZ, [_P, _I64]),
    "mt_lookup": (_I32, [_P, _P, _I64, _P, _P, _I32, _I32, _P, _P, _P, _SZ, _P]),
    "mt_lookup_static": (_I32, [_P, _P, _I64, _P, _P, _I32, _I32, _P, _P, _P]),
    "mt_backward_workspace_bytes": (_SZ, [_P, _I64]),
    "mt_pool_workspace_bytes": (_SZ, [_P, _I64]),
    "mt_pool_forward": (_I32, [_P, _P, _I64, _P, _I64, _I32, _P, _P, _SZ, _P]),
    "mt_backward_pooled_workspace_bytes": (_SZ, [_P, _I64, _I64]),
    "mt_backward_adam_pooled": (_I32, [_P, _P, _I64, _P, _I64, _I32, _P, _P, _P, _P, _SZ, _P]),
    "mt_backward_adam": (_I32, [_P, _P, _I64, _P, _I32, _P, _P, _P, _SZ, _P]),
    "mt_shard_group_create": (_I32, [_P, _I32, _P]),
    "mt_shard_group_destroy": (_I32, [_P]),
    "mt_shard_workspace_bytes": (_SZ, [_P, _P]),
    "mt_shard_lookup": (_I32, [_P, _P, _P, _P, _P, _I32, _I32, _P, _P, _P, _SZ, _P]),
    "mt_shard_backward_adam": (_I32, [_P, _P, _P, _I32, _P, _P, _P, _SZ, _P]),
    "mt_plan_merge": (_I32, [_P, _I32, ctypes.c_double, _P, _P, _P]),
    "mt_lookup_grouped_workspace_bytes": (_SZ, [_I64, _I32]),
    "mt_lookup_grouped": (_I32, [_P, _I32, _P, _P, _I64, _P, _I32, _I32, _P, _P, _P, _P, _SZ, _P]),
    "mt_backward_grouped_workspace_bytes": (_SZ, [_P, _I32, _P]),
    "mt_backward_adam_grouped": (_I32, [_P, _I32, _P, _P, _P, _I32, _P, _P, _P, _SZ, _P]),
    "mt_erase_workspace_bytes": (_SZ, [_I64]),
    "mt_erase": (_I32, [_P, _P, _I64, _P, _P, _SZ, _P]),
    "mt_compact_workspace_bytes": (_SZ, [_P]),
    "mt_compact": (_I32, [_P, _P, _SZ, _P, _P]),
    "mt_stats": (_I32, [_P, _P, _P]),
    "mt_export": (_I32, [_P, _P, _P, _I64, _P, _P]),
    "mt_read_rows": (_I32, [_P, _P, _I64, _P, _P, _P, _P]),
    "mt_import_workspace_bytes": (_SZ, [_I64]),
    "mt_import": (_I32, [_P, _P, _I64, _P, _P, _P, _P, _SZ, _P]),
    "mt_get_adam_state": (_I32, [_P, _P, _P, _P, _P]),
    "mt_set_adam_state": (_I32, [_P, _I64, ctypes.c_double, ctypes.c_double, _P]),
    "mt_get_error": (_I32, [_P, _P, _I32, _P]),
    "mt_step": (_I64, [_P]),
    "mt_profile_enable": (_I32, [_I32]),
    "mt_profile_report": (_I32, [_P, _I32, _P, _I32]),
    "mt_kernel_launches": (_I64, []),
}

class _FeatureSpec(ctypes.Structure):
    _fields_ = [("dim", ctypes.c_uint32), ("row_dtype", ctypes.c_uint32), ("capacity", ctypes.c_int64)]


class _Placement(ctypes.Structure):
    _fields_ = [("group", ctypes.c_int32), ("table_id", ctypes.c_uint8), ("pad", ctypes.c_uint8 * 3)]


class _MergeGroup(ctypes.Structure):
    _fields_ = [("dim", ctypes.c_uint32), ("row_dtype", ctypes.c_uint32), ("log2_slots", ctypes.c_uint32),
                ("num_features", ctypes.c_int32), ("capacity", ctypes.c_int64)]


class _KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 40), ("launches", ctypes.c_int64), ("total_ms", ctypes.c_double)]


_lib = None


def profile_enable(on: bool = True) -> None:
    """Per-kernel CUDA-event timing for every table of the process (off by default)."""
    _check(load_library().mt_profile_enable(int(bool(on))), "mt_profile_enable")


def profile_report(reset: bool = True) -> dict:
    """{kernel name: (launches, total ms)} accumulated since the last reset; synchronises the events."""
    L = load_library()
    cap = 64
    buf = (_KernelTime * cap)()
    cnt = ctypes.c_int()
    _check(L.mt_profile_report(buf, cap, ctypes.byref(cnt), int(bool(reset))), "mt_profile_report")
    return {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms)) for i in range(min(cnt.value, cap))}


def kernel_launches() -> int:
    """Kernels launched by the library so far in this process."""
    return int(load_library().mt_kernel_launches())


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libmt.so (built by ``build_lib.build()``); raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library not built: {p} is missing (run update_merged_table_gb300.build_lib.build())")
    L = ctypes.CDLL(p)
    for name, (res, args) in ABI_FUNCTIONS.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    if L.mt_abi_version() != ABI_VERSION:
        raise RuntimeError("libmt.so ABI version mismatch")
    if path is None:
        _lib = L
    return L


def _strerror(code: int) -> str:
    try:
        return load_library().mt_strerror(code).decode()
    except Exception:  # pragma: no cover
        return "?"


def _check(rc: int, what: str):
    if rc != MT_OK:
        raise MTError(rc, what)


def _torch():
    import torch
    return torch


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


@dataclasses.dataclass
class LookupResult:
    """Device outputs of one lookup (capacity n; the first U entries are valid)."""
    unique_keys: "object"   # int64 [n] (bit pattern of the uint64 merged keys)
    inverse: "object"       # int32 [n]
    counts: "object"        # int32 [n]
    unique_rows: "object"   # int32 [n]
    num_unique: "object"    # int64 [1]
    rows: "object" = None   # [n, dim] row dtype, or None
    n: int = 0
    ranks: "object" = None  # int32 [n] or None: rank of each position among its key's positions

    def as_struct(self) -> _Result:
        return _Result(_ptr(self.unique_keys), _ptr(self.inverse), _ptr(self.counts), _ptr(self.unique_rows),
                       _ptr(self.num_unique), _ptr(self.ranks))

    @property
    def U(self) -> int:
        return int(self.num_unique.item())


class Table:
    """A merged dynamic embedding table held in one device arena.

    Args mirror ``mt_config``: ``log2_slots`` (M = 2^n slots), ``dim``,
    ``row_dtype`` ("f32" or "bf16"), ``probe_step`` (odd S), seeds,
    ``init_scale`` (0 = 1/sqrt(dim)), ``max_probes`` (0 = M), ``num_rows``
    (0 = M).
    """

    def __init__(self, log2_slots: int, dim: int, row_dtype: str = "f32", probe_step: int = 1, hash_seed: int = 0,
                 init_seed: int = 0, init_scale: float = 0.0, max_probes: int = 0, num_rows: int = 0,
                 device=None, stream=None, flags: int = 0):
        torch = _torch()
        self.lib = load_library()
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        dt = {"f32": MT_F32, "bf16": MT_BF16}[row_dtype]
        self.row_dtype = row_dtype
        self.torch_row_dtype = torch.float32 if dt == MT_F32 else torch.bfloat16
        self.cfg = _Config(log2_slots, dim, dt, max_probes, probe_step, hash_seed, init_seed, init_scale, flags,
                           num_rows)
        nbytes = self.lib.mt_table_bytes(ctypes.byref(self.cfg))
        if nbytes == 0:
            raise MTError(MT_EINVAL, "mt_table_bytes")
        self.arena = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        self.h = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            _check(self.lib.mt_table_create(ctypes.byref(self.cfg), self.arena.data_ptr(), nbytes, _stream(stream),
                                            ctypes.byref(self.h)), "mt_table_create")
        # device memory the table uses: row segments (the arena holds the first), the key store, the slot
        # array when compaction moved it out of the key store, and a spare slot array for the next compaction
        self._row_bufs = [self.arena]
        self._keystore = self.arena
        self._slots_buf = None
        self._spare = None
        out = _Config()
        _check(self.lib.mt_table_config(self.h, ctypes.byref(out)), "mt_table_config")
        self.cfg = out
        self.dim = dim
        self.log2_slots = log2_slots
        self._ws = {}

    def __del__(self):
        h = getattr(self, "h", None)
        if h and h.value:
            try:
                self.lib.mt_table_destroy(h)
            except Exception:  # pragma: no cover
                pass
            self.h = None

    @property
    def config(self) -> dict:
        c = self.cfg
        return {f: getattr(c, f) for f, _ in c._fields_}

    def _workspace(self, kind: str, nbytes: int):
        torch = _torch()
        buf = self._ws.get(kind)
        if buf is None or buf.numel() < nbytes:
            if torch.cuda.is_current_stream_capturing():
                # graphs captured earlier hold the old buffer's address, and a later capture may return the
                # freed buffer to the driver: they would replay on unmapped memory
                raise RuntimeError(f"the {kind} workspace would have to grow during CUDA graph capture; call "
                                   "reserve_workspaces() with the largest batch before capturing")
            buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device)
            self._ws[kind] = buf
        return buf

    def new_result(self, n: int, gather: bool = True, ranks: bool = True) -> LookupResult:
        """Result buffers for a batch of n IDs.  ranks=True lets the backward skip re-grouping positions."""
        torch = _torch()
        dev = self.device
        return LookupResult(
            unique_keys=torch.empty(max(n, 1), dtype=torch.int64, device=dev),
            inverse=torch.empty(max(n, 1), dtype=torch.int32, device=dev),
            counts=torch.empty(max(n, 1), dtype=torch.int32, device=dev),
            unique_rows=torch.empty(max(n, 1), dtype=torch.int32, device=dev),
            num_unique=torch.empty(1, dtype=torch.int64, device=dev),
            rows=torch.empty((n, self.dim), dtype=self.torch_row_dtype, device=dev) if gather else None,
            n=n,
            ranks=torch.empty(max(n, 1), dtype=torch.int32, device=dev) if ranks else None)

    def lookup(self, ids, feat_offsets=None, table_ids=None, insert_missing: bool = True, gather: bool = True,
               result: LookupResult | None = None, stream=None) -> LookupResult:
        """Encode, deduplicate, find/insert and gather one batch.

        ids: int64 CUDA tensor [n].  feat_offsets: host sequence of F+1 int64
        (None = one feature).  table_ids: host sequence of F uint8 (None = 0).
        """
        torch = _torch()
        if ids.dtype != torch.int64 or not ids.is_cuda or not ids.is_contiguous():
            raise TypeError("ids must be a contiguous int64 CUDA tensor")
        n = ids.numel()
        res = result if result is not None else self.new_result(n, gather)
        if res.n != n:
            raise ValueError("result capacity differs from the batch size")
        F = 1
        fo_p = ti_p = None
        if feat_offsets is not None:
            fo = np.ascontiguousarray(feat_offsets, dtype=np.int64)
            F = fo.size - 1
            fo_p = fo.ctypes.data_as(ctypes.c_void_p)
        if table_ids is not None:
            ti = np.ascontiguousarray(table_ids, dtype=np.uint8)
            if feat_offsets is None and ti.size != 1:
                raise ValueError("table_ids without feat_offsets must have one entry")
            ti_p = ti.ctypes.data_as(ctypes.c_void_p)
        wsb = self.lib.mt_lookup_workspace_bytes(self.h, n)
        ws = self._workspace("lookup", wsb)
        st = res.as_struct()
        _check(self.lib.mt_lookup(self.h, ids.data_ptr() if n else None, n, fo_p, ti_p, F, int(bool(insert_missing)),
                                  _ptr(res.rows) if (gather and n) else None, ctypes.byref(st), ws.data_ptr(),
                                  ws.numel(), _stream(stream)), "mt_lookup")
        return res

    def backward_adam(self, res: LookupResult, grads, lr: float = 1e-3, beta1: float = 0.9, beta2: float = 0.999,
                      eps: float = 1e-8, want_gsum: bool = False, stream=None):
        """Per-unique gradient sum and one sparse Adam step; returns gsum [n, dim] fp32 if asked."""
        torch = _torch()
        n = res.n
        if grads.shape != (n, self.dim) or not grads.is_cuda or not grads.is_contiguous():
            raise ValueError("grads must be a contiguous CUDA tensor [n, dim]")
        gd = {torch.float32: MT_F32, torch.bfloat16: MT_BF16}.get(grads.dtype)
        if gd is None:
            raise TypeError("grads must be float32 or bfloat16")
        gsum = torch.empty((max(n, 1), self.dim), dtype=torch.float32, device=self.device) if want_gsum else None
        hp = _Adam(lr, beta1, beta2, eps)
        wsb = self.lib.mt_backward_workspace_bytes(self.h, n)
        ws = self._workspace("backward", wsb)
        st = res.as_struct()
        _check(self.lib.mt_backward_adam(self.h, ctypes.byref(st), n, grads.data_ptr() if n else None, gd,
                                         ctypes.byref(hp), _ptr(gsum), ws.data_ptr(), ws.numel(), _stream(stream)),
               "mt_backward_adam")
        return gsum

    def pool_forward(self, res: LookupResult, bag_offsets, mode: str = "sum", out=None, stream=None):
        """Pooled rows fp32 [B, dim] of the lookup `res`: per bag of positions
        [bag_offsets[b], bag_offsets[b+1]) the sum or the mean of its rows.
        bag_offsets: int64 CUDA tensor [B + 1]."""
        torch = _torch()
        bo = self._bag_offsets(bag_offsets)
        B = bo.numel() - 1
        m = {"sum": POOL_SUM, "mean": POOL_MEAN}[mode]
        if out is None:
            out = torch.empty((max(B, 1), self.dim), dtype=torch.float32, device=self.device)
        ws = self._workspace("pool", self.lib.mt_pool_workspace_bytes(self.h, B))
        st = res.as_struct()
        _check(self.lib.mt_pool_forward(self.h, ctypes.byref(st), res.n, bo.data_ptr(), B, m, out.data_ptr(),
                                        ws.data_ptr(), ws.numel(), _stream(stream)), "mt_pool_forward")
        return out[:B]

    def backward_adam_pooled(self, res: LookupResult, bag_offsets, dpooled, mode: str = "sum", lr: float = 1e-3,
                             beta1: float = 0.9, beta2: float = 0.999, eps: float = 1e-8, want_gsum: bool = False,
                             stream=None):
        """Backward of pool_forward (bag gradients dpooled fp32 [B, dim]) and one sparse Adam step."""
        torch = _torch()
        bo = self._bag_offsets(bag_offsets)
        B = bo.numel() - 1
        m = {"sum": POOL_SUM, "mean": POOL_MEAN}[mode]
        if dpooled.shape != (B, self.dim) or dpooled.dtype != torch.float32 or not dpooled.is_cuda \
                or not dpooled.is_contiguous():
            raise ValueError("dpooled must be a contiguous fp32 CUDA tensor [B, dim]")
        n = res.n
        gsum = torch.empty((max(n, 1), self.dim), dtype=torch.float32, device=self.device) if want_gsum else None
        hp = _Adam(lr, beta1, beta2, eps)
        ws = self._workspace("backward_pooled", self.lib.mt_backward_pooled_workspace_bytes(self.h, n, B))
        st = res.as_struct()
        _check(self.lib.mt_backward_adam_pooled(self.h, ctypes.byref(st), n, bo.data_ptr(), B, m,
                                                dpooled.data_ptr() if B else None, ctypes.byref(hp), _ptr(gsum),
                                                ws.data_ptr(), ws.numel(), _stream(stream)),
               "mt_backward_adam_pooled")
        return gsum

    def reserve_workspaces(self, n: int, num_bags: int = 0, n_erase: int = 0):
        """Allocate every workspace a batch of n IDs (num_bags pooled bags, n_erase keys to erase) needs, so
        that later calls (for instance under CUDA graph capture) allocate nothing."""
        self._workspace("lookup", self.lib.mt_lookup_workspace_bytes(self.h, n))
        self._workspace("backward", self.lib.mt_backward_workspace_bytes(self.h, n))
        if n_erase:
            self._workspace("erase", self.lib.mt_erase_workspace_bytes(n_erase))
        if num_bags:
            self._workspace("pool", self.lib.mt_pool_workspace_bytes(self.h, num_bags))
            self._workspace("backward_pooled", self.lib.mt_backward_pooled_workspace_bytes(self.h, n, num_bags))

    def _bag_offsets(self, bag_offsets):
        torch = _torch()
        if not torch.is_tensor(bag_offsets):
            bag_offsets = torch.as_tensor(np.ascontiguousarray(bag_offsets, dtype=np.int64)).to(self.device)
        if bag_offsets.dtype != torch.int64 or not bag_offsets.is_cuda or not bag_offsets.is_contiguous() \
                or bag_offsets.dim() != 1 or bag_offsets.numel() < 1:
            raise TypeError("bag_offsets must be a contiguous 1-D int64 CUDA tensor [B + 1]")
        return bag_offsets

    def grow(self, log2_slots: int, num_rows: int = 0, stream=None):
        """Capacity expansion to 2^log2_slots slots and num_rows rows (0 = one per slot): a new key store
        is built and the added rows come as a new row segment; no row moves."""
        torch = _torch()
        c = _Config(log2_slots, self.cfg.dim, self.cfg.row_dtype, 0, self.cfg.probe_step, self.cfg.hash_seed,
                    self.cfg.init_seed, self.cfg.init_scale, self.cfg.flags, num_rows)
        ks_bytes = self.lib.mt_keystore_bytes(ctypes.byref(c))
        if ks_bytes == 0:
            raise MTError(MT_EINVAL, "mt_keystore_bytes")
        new_rows = (num_rows or (1 << log2_slots)) - self.cfg.num_rows
        ks = torch.empty(ks_bytes, dtype=torch.uint8, device=self.device)
        rows = None
        if new_rows > 0:
            rows = torch.empty(self.lib.mt_rows_bytes(ctypes.byref(c), new_rows), dtype=torch.uint8,
                               device=self.device)
        _check(self.lib.mt_table_grow(self.h, ctypes.byref(c), ks.data_ptr(), ks_bytes,
                                      rows.data_ptr() if rows is not None else None,
                                      rows.numel() if rows is not None else 0, _stream(stream)), "mt_table_grow")
        self._keystore = ks  # the old key store is released with its last reference (the arena stays: rows)
        self._slots_buf = None
        self._spare = None
        if rows is not None:
            self._row_bufs.append(rows)
        out = _Config()
        _check(self.lib.mt_table_config(self.h, ctypes.byref(out)), "mt_table_config")
        self.cfg = out
        self.log2_slots = log2_slots

    def compact(self, stream=None):
        """Rebuild the key store's slots without tombstones into a spare slot array, which becomes the
        table's (rows and keys unchanged); the slot array used before becomes the next spare."""
        torch = _torch()
        need = self.lib.mt_compact_workspace_bytes(self.h)
        spare = self._spare
        if spare is None or spare.numel() < need:
            spare = torch.empty(need, dtype=torch.uint8, device=self.device)
        released = ctypes.c_void_p()
        _check(self.lib.mt_compact(self.h, spare.data_ptr(), spare.numel(), ctypes.byref(released),
                                   _stream(stream)), "mt_compact")
        old = released.value
        holder = None
        for buf in (self._slots_buf, self._keystore):
            if buf is not None and buf.data_ptr() <= old < buf.data_ptr() + buf.numel():
                holder = buf[old - buf.data_ptr(): old - buf.data_ptr() + need]
                break
        self._slots_buf = spare
        self._spare = holder

    def erase(self, keys, want_found: bool = True, stream=None):
        """Delete merged keys (int64 CUDA tensor holding the uint64 bit patterns)."""
        torch = _torch()
        if keys.dtype != torch.int64 or not keys.is_cuda or not keys.is_contiguous():
            raise TypeError("keys must be a contiguous int64 CUDA tensor")
        n = keys.numel()
        found = torch.empty(max(n, 1), dtype=torch.uint8, device=self.device) if want_found else None
        ws = self._workspace("erase", self.lib.mt_erase_workspace_bytes(n))
        _check(self.lib.mt_erase(self.h, keys.data_ptr() if n else None, n, _ptr(found), ws.data_ptr(), ws.numel(),
                                 _stream(stream)), "mt_erase")
        return found[:n] if want_found else None

    def stats(self, stream=None) -> dict:
        s = _Stats()
        _check(self.lib.mt_stats(self.h, ctypes.byref(s), _stream(stream)), "mt_stats")
        out = {f: getattr(s, f) for f, _ in s._fields_ if f not in ("probe_hist", "reserved")}
        out["probe_hist"] = np.array(list(s.probe_hist), dtype=np.int64)
        return out

    def export(self, stream=None):
        """(keys int64 [live], rows int32 [live]) of every live key, in no particular order."""
        torch = _torch()
        cap = int(self.stats(stream)["live"])
        keys = torch.empty(max(cap, 1), dtype=torch.int64, device=self.device)
        rows = torch.empty(max(cap, 1), dtype=torch.int32, device=self.device)
        cnt = ctypes.c_int64()
        _check(self.lib.mt_export(self.h, keys.data_ptr(), rows.data_ptr(), cap, ctypes.byref(cnt), _stream(stream)),
               "mt_export")
        c = min(int(cnt.value), cap)
        return keys[:c], rows[:c]

    def read_rows(self, rows, stream=None):
        """(emb, m, v) as fp32 [n, dim] for int32 CUDA row indices (-1 gives zeros)."""
        torch = _torch()
        n = rows.numel()
        emb = torch.empty((max(n, 1), self.dim), dtype=torch.float32, device=self.device)
        m = torch.empty_like(emb)
        v = torch.empty_like(emb)
        _check(self.lib.mt_read_rows(self.h, rows.data_ptr() if n else None, n, emb.data_ptr(), m.data_ptr(),
                                     v.data_ptr(), _stream(stream)), "mt_read_rows")
        return emb[:n], m[:n], v[:n]

    def import_rows(self, keys, emb, m, v, stream=None):
        """Checkpoint restore: find or insert each merged key (int64 CUDA tensor of the
        uint64 bit patterns, distinct) and write its row from fp32 [n, dim] emb, m, v."""
        torch = _torch()
        n = keys.numel()
        if keys.dtype != torch.int64 or not keys.is_cuda or not keys.is_contiguous():
            raise TypeError("keys must be a contiguous int64 CUDA tensor")
        for x in (emb, m, v):
            if x.shape != (n, self.dim) or x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
                raise ValueError("emb, m, v must be contiguous fp32 CUDA tensors [n, dim]")
        if n and torch.unique(keys).numel() != n:
            raise ValueError("keys must be distinct")
        ws = self._workspace("import", self.lib.mt_import_workspace_bytes(n))
        _check(self.lib.mt_import(self.h, keys.data_ptr() if n else None, n, emb.data_ptr() if n else None,
                                  m.data_ptr() if n else None, v.data_ptr() if n else None, ws.data_ptr(),
                                  ws.numel(), _stream(stream)), "mt_import")

    def adam_state(self, stream=None):
        """(steps taken, beta1^t, beta2^t) of the table's Adam accumulators."""
        st, b1, b2 = ctypes.c_int64(), ctypes.c_double(), ctypes.c_double()
        _check(self.lib.mt_get_adam_state(self.h, ctypes.byref(st), ctypes.byref(b1), ctypes.byref(b2),
                                          _stream(stream)), "mt_get_adam_state")
        return int(st.value), float(b1.value), float(b2.value)

    def set_adam_state(self, step: int, b1pow: float, b2pow: float, stream=None):
        _check(self.lib.mt_set_adam_state(self.h, step, b1pow, b2pow, _stream(stream)), "mt_set_adam_state")

    def error(self, clear: bool = False, stream=None) -> int:
        e = ctypes.c_int32()
        _check(self.lib.mt_get_error(self.h, ctypes.byref(e), int(bool(clear)), _stream(stream)), "mt_get_error")
        return int(e.value)

    @property
    def step(self) -> int:
        return int(self.lib.mt_step(self.h))


class ShardGroup:
    """G tables as the shards of one logical table, driven as G logical ranks on one GPU
    (``mt_shard_lookup`` / ``mt_shard_backward_adam``): each rank deduplicates its own batch, sends its
    unique keys to their owners, the owners deduplicate again and serve the rows, and the rows come back."""

    def __init__(self, shards):
        self.lib = load_library()
        self.shards = list(shards)
        self.G = len(self.shards)
        arr = (ctypes.c_void_p * self.G)(*[t.h.value for t in self.shards])
        self.h = ctypes.c_void_p()
        _check(self.lib.mt_shard_group_create(arr, self.G, ctypes.byref(self.h)), "mt_shard_group_create")
        self.dim = self.shards[0].dim
        self.device = self.shards[0].device
        self._ws = None
        self._last = None

    def __del__(self):
        h = getattr(self, "h", None)
        if h and h.value:
            try:
                self.lib.mt_shard_group_destroy(h)
            except Exception:  # pragma: no cover
                pass
            self.h = None

    def lookup(self, ids, feat_offsets=None, table_ids=None, insert_missing: bool = True, gather: bool = True,
               ranks: bool = True, stream=None):
        """ids: G int64 CUDA tensors; feat_offsets: G host sequences of F+1 (or None).  Returns G LookupResults
        (rows per rank; unique_rows are -1, the rows live in the owners' shards)."""
        torch = _torch()
        G = self.G
        if len(ids) != G:
            raise ValueError("one ID tensor per rank")
        ns = np.array([int(x.numel()) for x in ids], dtype=np.int64)
        for x in ids:
            if x.dtype != torch.int64 or not x.is_cuda or not x.is_contiguous():
                raise TypeError("ids must be contiguous int64 CUDA tensors")
        res = [self.shards[r].new_result(int(ns[r]), gather=gather, ranks=ranks) for r in range(G)]
        F = 1
        fo_p = ti_p = None
        if feat_offsets is not None:
            fo = np.ascontiguousarray(np.concatenate([np.asarray(f, np.int64) for f in feat_offsets]), np.int64)
            F = fo.size // G - 1
            fo_p = fo.ctypes.data_as(ctypes.c_void_p)
        if table_ids is not None:
            ti = np.ascontiguousarray(table_ids, dtype=np.uint8)
            ti_p = ti.ctypes.data_as(ctypes.c_void_p)
        wsb = self.lib.mt_shard_workspace_bytes(self.h, ns.ctypes.data_as(ctypes.c_void_p))
        if self._ws is None or self._ws.numel() < wsb:
            self._ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device=self.device)
        ids_p = (ctypes.c_void_p * G)(*[x.data_ptr() if x.numel() else None for x in ids])
        out_p = (ctypes.c_void_p * G)(*[(r.rows.data_ptr() if (gather and r.n) else None) for r in res])
        st = (_Result * G)(*[r.as_struct() for r in res])
        _check(self.lib.mt_shard_lookup(self.h, ids_p, ns.ctypes.data_as(ctypes.c_void_p), fo_p, ti_p, F,
                                        int(bool(insert_missing)), out_p, st, self._ws.data_ptr(), self._ws.numel(),
                                        _stream(stream)), "mt_shard_lookup")
        self._last = res
        return res

    def backward_adam(self, res, grads, lr: float = 1e-3, beta1: float = 0.9, beta2: float = 0.999,
                      eps: float = 1e-8, want_gsum: bool = False, stream=None):
        """grads: G CUDA tensors [n_r, dim] (fp32 or bf16).  Returns per-rank fp32 sums [U_r, dim] over all
        ranks if asked."""
        torch = _torch()
        G = self.G
        gd = {torch.float32: MT_F32, torch.bfloat16: MT_BF16}.get(grads[0].dtype)
        if gd is None or any(g.dtype != grads[0].dtype for g in grads):
            raise TypeError("grads must all be float32 or all bfloat16")
        for r in range(G):
            if grads[r].shape != (res[r].n, self.dim) or not grads[r].is_cuda or not grads[r].is_contiguous():
                raise ValueError("grads[r] must be a contiguous CUDA tensor [n_r, dim]")
        gsum = None
        gs_p = None
        if want_gsum:
            gsum = [torch.empty((max(int(r.U), 1), self.dim), dtype=torch.float32, device=self.device) for r in res]
            gs_p = (ctypes.c_void_p * G)(*[g.data_ptr() for g in gsum])
        hp = _Adam(lr, beta1, beta2, eps)
        g_p = (ctypes.c_void_p * G)(*[g.data_ptr() if g.numel() else None for g in grads])
        st = (_Result * G)(*[r.as_struct() for r in res])
        _check(self.lib.mt_shard_backward_adam(self.h, st, g_p, gd, ctypes.byref(hp), gs_p, self._ws.data_ptr(),
                                               self._ws.numel(), _stream(stream)), "mt_shard_backward_adam")
        return gsum


def plan_merge(features, max_load: float = 0.5):
    """Automatic table merging (``mt_plan_merge``).  features: sequence of (dim, "f32"|"bf16", capacity).
    Returns (placement, groups): placement[f] = (group, table_id); groups[g] = dict(dim, row_dtype,
    log2_slots, num_features, capacity)."""
    L = load_library()
    F = len(features)
    specs = (_FeatureSpec * max(F, 1))(*[_FeatureSpec(d, {"f32": MT_F32, "bf16": MT_BF16}[t], c)
                                        for d, t, c in features])
    pl = (_Placement * max(F, 1))()
    gr = (_MergeGroup * max(F, 1))()
    G = ctypes.c_int()
    _check(L.mt_plan_merge(specs, F, float(max_load), pl, gr, ctypes.byref(G)), "mt_plan_merge")
    placement = [(int(pl[f].group), int(pl[f].table_id)) for f in range(F)]
    groups = [dict(dim=int(gr[g].dim), row_dtype="f32" if gr[g].row_dtype == MT_F32 else "bf16",
                   log2_slots=int(gr[g].log2_slots), num_features=int(gr[g].num_features),
                   capacity=int(gr[g].capacity)) for g in range(G.value)]
    return placement, groups


class MergedTables:
    """The merged tables of a plan (``plan_merge``) and the lookup that routes a batch's feature segments
    to them (``mt_lookup_grouped``); the backward runs every merged table's step (``mt_backward_adam_grouped``)."""

    def __init__(self, features, max_load: float = 0.5, device=None, **table_kwargs):
        self.lib = load_library()
        self.placement, self.groups = plan_merge(features, max_load)
        self.tables = [Table(g["log2_slots"], g["dim"], row_dtype=g["row_dtype"], device=device, **table_kwargs)
                       for g in self.groups]
        self.device = self.tables[0].device
        self._pl = (_Placement * len(self.placement))(*[_Placement(g, t) for g, t in self.placement])
        self._ws = {}

    def group_sizes(self, feat_offsets):
        """IDs each merged table receives from a batch with these feature offsets."""
        fo = np.asarray(feat_offsets, dtype=np.int64)
        sizes = [0] * len(self.tables)
        for f, (g, _) in enumerate(self.placement):
            sizes[g] += int(fo[f + 1] - fo[f])
        return sizes

    def lookup(self, ids, feat_offsets, insert_missing: bool = True, gather: bool = True, stream=None):
        """ids: int64 CUDA tensor [n]; feat_offsets: host sequence of F+1.  Returns one LookupResult per
        merged table (its IDs are the batch's segments of its features, in feature order)."""
        torch = _torch()
        fo = np.ascontiguousarray(feat_offsets, dtype=np.int64)
        F = fo.size - 1
        if F != len(self.placement):
            raise ValueError("one segment per planned feature")
        n = int(ids.numel())
        sizes = self.group_sizes(fo)
        res = [t.new_result(sz, gather=gather) for t, sz in zip(self.tables, sizes)]
        G = len(self.tables)
        ws = self._workspace("lookup", self.lib.mt_lookup_grouped_workspace_bytes(n, F))
        tabs = (ctypes.c_void_p * G)(*[t.h.value for t in self.tables])
        outs = (ctypes.c_void_p * G)(*[(r.rows.data_ptr() if (gather and r.n) else None) for r in res])
        st = (_Result * G)(*[r.as_struct() for r in res])
        gn = np.zeros(G, dtype=np.int64)
        _check(self.lib.mt_lookup_grouped(tabs, G, self._pl, ids.data_ptr() if n else None, n,
                                          fo.ctypes.data_as(ctypes.c_void_p), F, int(bool(insert_missing)), outs, st,
                                          gn.ctypes.data_as(ctypes.c_void_p), ws.data_ptr(), ws.numel(),
                                          _stream(stream)), "mt_lookup_grouped")
        if list(gn) != sizes:
            raise RuntimeError("group sizes disagree with the plan")
        return res

    def _workspace(self, kind: str, nbytes: int):
        torch = _torch()
        buf = self._ws.get(kind)
        if buf is None or buf.numel() < nbytes:
            if torch.cuda.is_current_stream_capturing():
                raise RuntimeError(f"the grouped {kind} workspace would have to grow during CUDA graph capture; "
                                   "run one eager step with the largest batch before capturing")
            buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device)
            self._ws[kind] = buf
        return buf

    def backward_adam(self, results, grads, lr: float = 1e-3, beta1: float = 0.9, beta2: float = 0.999,
                      eps: float = 1e-8, want_gsum: bool = False, stream=None):
        """grads: one CUDA tensor [n_g, dim_g] per merged table, all float32 or all bfloat16
        (``mt_backward_adam_grouped``: the tables' backward steps run side by side).  Returns one gradient-sum
        tensor (or None) per table."""
        torch = _torch()
        G = len(self.tables)
        if len(results) != G or len(grads) != G:
            raise ValueError("one lookup result and one gradient tensor per merged table")
        gd = {torch.float32: MT_F32, torch.bfloat16: MT_BF16}.get(grads[0].dtype)
        if gd is None or any(g.dtype != grads[0].dtype for g in grads):
            raise TypeError("grads must all be float32 or all bfloat16")
        for t, r, g in zip(self.tables, results, grads):
            if g.shape != (r.n, t.dim) or not g.is_cuda or not g.is_contiguous():
                raise ValueError("grads[g] must be a contiguous CUDA tensor [n_g, dim_g]")
        gsums = [torch.empty((max(r.n, 1), t.dim), dtype=torch.float32, device=self.device) if want_gsum else None
                 for t, r in zip(self.tables, results)]
        tabs = (ctypes.c_void_p * G)(*[t.h.value for t in self.tables])
        gn = np.asarray([r.n for r in results], dtype=np.int64)
        ws = self._workspace("backward", self.lib.mt_backward_grouped_workspace_bytes(
            tabs, G, gn.ctypes.data_as(ctypes.c_void_p)))
        st = (_Result * G)(*[r.as_struct() for r in results])
        gp = (ctypes.c_void_p * G)(*[(g.data_ptr() if r.n else None) for g, r in zip(grads, results)])
        gs = (ctypes.c_void_p * G)(*[_ptr(x) for x in gsums]) if want_gsum else None
        hp = _Adam(lr, beta1, beta2, eps)
        _check(self.lib.mt_backward_adam_grouped(tabs, G, st, gn.ctypes.data_as(ctypes.c_void_p), gp, gd,
                                                 ctypes.byref(hp), gs, ws.data_ptr(), ws.numel(), _stream(stream)),
               "mt_backward_adam_grouped")
        return gsums
