"""Benchmark of the merged dynamic embedding table hot path on GB300.

One step = one lookup (encode, two-stage dedup, find/insert, gather) plus one
backward (per-unique gradient sum + sparse Adam) over one batch, plus the
erase of that step's deletions for the online-churn workload.  The default
workload (``--config 3``) is the GRM jagged-sequence batch: 2048 users with
lognormal(5, 1) sequence lengths capped at 3000, 4 ID features per token
(Zipf(1.1) over 1e6 IDs each, merged by table id), M = 2^24 slots, dim 64
bf16 rows, fp32 Adam state, bf16 grads.  A run is the cold step 0, warm-up
steps on it, then K timed steps on fresh seeds 1..K, so every timed step
inserts the keys it brings that the table has not seen.  Synthetic, seeded
inputs; every step's inputs and outputs exceed the 126 MB L2, so no flush is
needed between steps.  ``--config 1, 2, 4, 5`` time the single-table,
merged-tables, large-table and online-churn workloads the same way.

Prints one JSON line.  ``--impl reference`` times the CPU oracle on a bounded
sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from update_merged_table_gb300 import workloads as W  # noqa: E402

METRIC = "unique+lookup+gather IDs/s and backward+Adam IDs/s; % of GB300 HBM roofline"
UNIT = "IDs/s"
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

FRESH_CAP = 64  # distinct fresh-seed steps held on the device; longer runs cycle through them


class Workload:
    """Table shape and the step sequence of one workload.

    A run is a cold step 0 (seed 0: on an empty or prefilled table it inserts
    its keys), warm-up steps, and timed steps 1, 2, ... on fresh seeds, so the
    timed steps insert whatever keys they bring that the table has not seen.
    """

    def __init__(self, cfg: int, users: int = 2048, log2_slots: int | None = None):
        self.cfg = cfg
        self.users = users
        self.prefill_ids = None
        self.churn = None
        if cfg == 1:
            self.name = "single table: M=2^16, dim 16 fp32, 4096 IDs Zipf(1.1) over 1e5"
            self.log2, self.dim, self.row, self.grad = 16, 16, "f32", "f32"
        elif cfg == 2:
            self.name = ("merged tables: 8 features (vocab 1e4..1e6, Zipf s 0.8..1.3) in one M=2^22 table, "
                         "dim 32 fp32, 65536 IDs")
            self.log2, self.dim, self.row, self.grad = 22, 32, "f32", "f32"
        elif cfg == 3:
            self.log2, self.dim, self.row, self.grad = 24, 64, "bf16", "bf16"
            self.name = ("GRM jagged sequences: 2048 users, lognormal(5,1) lengths capped at 3000, 4 ID features, "
                         "M=2^24, dim 64 bf16")
        elif cfg == 4:
            self.name = ("large table: M=2^26, dim 128 fp32, prefilled to load 0.7, 2^20 IDs Zipf(1.05) over a "
                         "2^32 key space")
            self.log2, self.dim, self.row, self.grad = 26, 128, "f32", "f32"
            self.prefill_ids = lambda: W.large_table_prefill_ids(int(0.7 * (1 << 26)))
        elif cfg == 5:
            self.name = ("online churn: M=2^24, dim 64 fp32, 2^23 prefilled keys, 2^18 IDs per step with 10% new, "
                         "erase of 2^16 live keys per step")
            self.log2, self.dim, self.row, self.grad = 24, 64, "f32", "f32"
            self.churn = W.ChurnStream(0)
            self.prefill_ids = self.churn.prefill_ids
            self._sample_churn = W.ChurnStream(0)
            self._sample_next = 0
        else:
            raise ValueError("config must be 1..5")
        if log2_slots is not None:
            self.log2 = log2_slots
        if cfg == 3 and (users != 2048 or self.log2 != 24):
            self.name = (f"GRM jagged sequences (reduced): {users} users, lognormal(5,1) lengths capped at 3000, "
                         f"4 ID features, M=2^{self.log2}, dim 64 bf16")

    def batch(self, seed: int):
        """(batch, None) of seed `seed` (configs 1-4; the churn stream is sequential, see `steps`)."""
        if self.cfg == 1:
            return W.single_table_batch(seed), None
        if self.cfg == 2:
            return W.merged_batch(seed), None
        if self.cfg == 3:
            return W.jagged_batch(seed, users=self.users), None
        if self.cfg == 4:
            return W.large_table_batch(seed), None
        raise ValueError("the churn workload draws its steps in order: use steps()")

    def steps(self, first: int, count: int):
        """(batch, erase ids or None) of steps first .. first+count-1.  For the churn workload
        the stream is sequential, so successive calls must continue where the last one ended."""
        if self.cfg == 5:
            return [self.churn.step(k) for k in range(first, first + count)]
        return [self.batch(k) for k in range(first, first + count)]

    def sample_batch(self, k: int):
        """A bounded slice of step k of the same workload for the CPU oracle (k = 0, 1, 2, ...)."""
        if self.cfg == 2:
            return W.merged_batch(k, per_table=2048)
        if self.cfg == 3:
            return W.jagged_batch(k, users=256)
        if self.cfg == 4:
            return W.large_table_batch(k, n=1 << 17)
        if self.cfg == 5:
            b, _ = self._sample_churn.step(self._sample_next)
            self._sample_next += 1
            return W.single_feature(b.ids[: 1 << 16])
        return W.single_table_batch(k)

    @property
    def row_bytes(self):
        return self.dim * (2 if self.row == "bf16" else 4)

    @property
    def grad_bytes(self):
        return self.dim * (2 if self.grad == "bf16" else 4)


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(ids_local: float, secs_local: float, group=None):
    """Whole-job totals over ranks: sum of IDs processed, max of elapsed seconds."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized():
        return ids_local, secs_local
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([ids_local], dtype=torch.float64, device=dev)
    s = torch.tensor([secs_local], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    dist.all_reduce(s, op=dist.ReduceOp.MAX, group=group)
    return float(t.item()), float(s.item())


def measured_hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            for k in ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs"):
                if k in d and d[k]:
                    return float(d[k]), "measured"
            for k, v in d.items():
                if "hbm" in k.lower() and isinstance(v, (int, float)):
                    return float(v), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def _parse_cpulist(text: str) -> set:
    cpus = set()
    for part in text.strip().split(","):
        if not part:
            continue
        a, _, b = part.partition("-")
        cpus.update(range(int(a), int(b or a) + 1))
    return cpus


def numa_cpus_for_gpu(pci_bus_id: str, sysfs: str = "/sys") -> tuple[set, str]:
    """CPUs to run on for the GPU at `pci_bus_id`, and how they were chosen.

    In order: the device's own local_cpulist; the CPUs of its numa_node; and,
    when that node has no CPUs (a GPU-memory node) or none is given, the
    CPU-bearing node nearest to it by the node distance table (else node 0).
    """
    bus = pci_bus_id.lower()
    dom, _, rest = bus.partition(":")
    cands = [bus, dom[-4:].zfill(4) + ":" + rest, dom.zfill(8) + ":" + rest]  # sysfs uses a 4-digit domain
    nodes_dir = os.path.join(sysfs, "devices", "system", "node")

    def node_cpus(n: int) -> set:
        p = os.path.join(nodes_dir, f"node{n}", "cpulist")
        return _parse_cpulist(open(p).read()) if os.path.exists(p) else set()

    for cand in cands:
        dev_dir = os.path.join(sysfs, "bus", "pci", "devices", cand)
        p = os.path.join(dev_dir, "local_cpulist")
        if os.path.exists(p):
            cpus = _parse_cpulist(open(p).read())
            if cpus:
                return cpus, "local_cpulist"
        p = os.path.join(dev_dir, "numa_node")
        if os.path.exists(p):
            node = int(open(p).read().strip())
            if node >= 0:
                cpus = node_cpus(node)
                if cpus:
                    return cpus, f"numa_node {node}"
                dpath = os.path.join(nodes_dir, f"node{node}", "distance")
                if os.path.exists(dpath):
                    dist = [int(x) for x in open(dpath).read().split()]
                    order = sorted(range(len(dist)), key=lambda k: dist[k])
                    for k in order:
                        cpus = node_cpus(k)
                        if cpus:
                            return cpus, f"node {k}, nearest CPU node to GPU node {node}"
    cpus = node_cpus(0)
    return cpus, "node 0 (no NUMA information for the GPU)" if cpus else "unbound"


def gpu_pci_bus_id(dev_index: int):
    """PCI bus id of the GPU torch calls `dev_index`: from torch's device properties where they carry it,
    else from nvidia-smi, matched by the device UUID."""
    import torch
    props = torch.cuda.get_device_properties(dev_index)
    for attr in ("pci_bus_id",):
        v = getattr(props, attr, None)
        if isinstance(v, str) and ":" in v:
            return v
    dom, bus, devn = (getattr(props, a, None) for a in ("pci_domain_id", "pci_bus_id", "pci_device_id"))
    if all(isinstance(x, int) for x in (dom, bus, devn)):
        return f"{dom:08x}:{bus:02x}:{devn:02x}.0"
    uuid = str(getattr(props, "uuid", "") or "")
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=uuid,pci.bus_id", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=20).stdout
    except Exception:
        return None
    rows = [tuple(x.strip() for x in line.split(",")) for line in out.splitlines() if "," in line]
    for u, b in rows:
        if uuid and uuid.replace("GPU-", "") in u:
            return b
    return rows[dev_index][1] if dev_index < len(rows) else None


def bind_to_gpu_numa_node(dev_index: int) -> str:
    """Run on the CPUs next to the GPU so pinned host buffers land in its NUMA node."""
    try:
        bus = gpu_pci_bus_id(dev_index)
        if bus is None:
            return "unbound (no PCI bus id for the GPU)"
        cpus, how = numa_cpus_for_gpu(bus)
        avail = os.sched_getaffinity(0)
        cpus &= avail
        if cpus:
            os.sched_setaffinity(0, cpus)
            return f"cpus {min(cpus)}-{max(cpus)} ({len(cpus)}; {how})"
    except Exception as e:  # pragma: no cover
        return f"unbound ({type(e).__name__})"
    return "unbound"


def kernel_source(kernel: str):
    """The CUDA source file that defines `kernel`, or None."""
    import re
    csrc = os.path.join(ROOT, "update_merged_table_gb300", "csrc")
    pat = re.compile(r"__global__[^;{]*\b" + re.escape(kernel) + r"\s*\(")
    for f in sorted(os.listdir(csrc)):
        if f.endswith(".cu") and pat.search(open(os.path.join(csrc, f)).read()):
            return os.path.join(csrc, f)
    return None


def source_digest(kernel: str | None = None) -> str:
    """Digest of the sources a kernel's counters depend on: the shared headers and the file that defines the
    kernel (every CUDA source when kernel is None).  Counters taken on other sources do not apply."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "update_merged_table_gb300", "csrc")
    names = sorted(f for f in os.listdir(csrc) if f.endswith(".cuh"))
    if kernel is None:
        names += sorted(f for f in os.listdir(csrc) if f.endswith(".cu"))
    else:
        src = kernel_source(kernel)
        if src is None:
            return "none"
        names.append(os.path.basename(src))
    for f in names:
        h.update(f.encode())
        h.update(open(os.path.join(csrc, f), "rb").read())
    h.update(open(os.path.join(ROOT, "include", "mt.h"), "rb").read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str):
    """(DRAM bytes per ID of `kernel`, capture note) from the committed ncu summary, or
    (None, reason) when there is none or it was taken on other sources of that kernel."""
    tpath = os.path.join(ROOT, "profiles", "kernel_traffic.txt")
    if not os.path.exists(tpath):
        return None, "no committed ncu summary"
    per_id = {}
    for line in open(tpath):
        f = line.split()
        if len(f) == 3 and not line.startswith("#"):
            per_id[f[0]] = (float(f[1]), f[2])
    if kernel not in per_id:
        return None, f"no counters for {kernel}"
    value, digest = per_id[kernel]
    if digest != source_digest(kernel):
        return None, f"the committed ncu counters of {kernel} were taken on other sources"
    return value, "profiles/kernel_traffic.txt"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (getattr(self, "out", "") or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)), "reasons": sorted(reasons),
                "samples": len(sm)}


def batch_stats(b):
    """Unique keys, heavy uniques (more than 32 positions) and their positions, from the batch itself."""
    f = np.searchsorted(b.feat_offsets, np.arange(b.n), side="right") - 1
    keys = (b.table_ids[f].astype(np.uint64) << np.uint64(56)) | b.ids.astype(np.uint64)
    _, cnt = np.unique(keys, return_counts=True)
    heavy = cnt > 32
    return int(cnt.size), int(heavy.sum()), int(cnt[heavy].sum())


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------

def _device_grads(torch, dev, dtype, seed: int, n: int, dim: int):
    """N(0, 1) gradients [n, dim] drawn on the device from a seeded generator."""
    g = torch.Generator(device=dev)
    g.manual_seed(500_000 + seed)
    return torch.randn((max(n, 1), dim), generator=g, device=dev, dtype=torch.float32)[:n].to(dtype)


def _prefill(torch, tab, wl, dev):
    if wl.prefill_ids is not None:  # untimed: the resident key set of a steady state
        pre = wl.prefill_ids()
        for s0 in range(0, pre.size, 1 << 22):
            tab.lookup(torch.from_numpy(pre[s0:s0 + (1 << 22)]).to(dev), gather=False)


def e2e_run(args, dev, stream, tdt):
    """The same step sequence through the public API with HOST buffers, on a table of its own: a cold
    step, warm-up steps, then K fresh steps, each copying its IDs and gradients from pinned host memory
    (step j + 1's copies on a copy stream while step j computes), running its calls (captured as a CUDA
    graph before timing) and reading its unique count back."""
    import torch
    import update_merged_table_gb300 as mt
    wl = Workload(args.config, args.users, args.log2_slots)
    tab = mt.Table(wl.log2, wl.dim, row_dtype=wl.row, device=dev)
    _prefill(torch, tab, wl, dev)
    ke = min(args.steps, FRESH_CAP)
    seq = wl.steps(0, 1 + ke)
    (cold, _), steps = seq[0], seq[1:]
    cold_ids = torch.from_numpy(cold.ids).to(dev)
    cold_g = _device_grads(torch, dev, tdt[wl.grad], 0, cold.n, wl.dim)
    for _ in range(1 + args.warmup):
        r = tab.lookup(cold_ids, cold.feat_offsets, cold.table_ids)
        tab.backward_adam(r, cold_g)
    del r, cold_ids, cold_g
    nmax = max(b.n for b, _ in steps)
    host = []
    for j, (b, er) in enumerate(steps):
        ids_h = torch.from_numpy(b.ids).pin_memory()
        g_h = torch.empty((b.n, wl.dim), dtype=tdt[wl.grad], pin_memory=True)
        g_h.copy_(_device_grads(torch, dev, tdt[wl.grad], 1 + j, b.n, wl.dim))
        er_h = torch.from_numpy(er.astype(np.int64)).pin_memory() if er is not None else None
        host.append((b, ids_h, g_h, er_h))
    slots = []
    for _ in range(2):
        big = tab.new_result(nmax, gather=True)
        slots.append(dict(ids=torch.empty(nmax, dtype=torch.int64, device=dev),
                          grads=torch.empty((nmax, wl.dim), dtype=tdt[wl.grad], device=dev),
                          erase=torch.empty(max(1, max((h[3].numel() for h in host if h[3] is not None),
                                                       default=1)), dtype=torch.int64, device=dev),
                          big=big, u_h=torch.empty(1, dtype=torch.int64).pin_memory()))
    copy_stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize(dev)
    # the link alone: one step's copies, timed on the copy stream
    la, lb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    b0, ids0, g0, _ = host[0]
    with torch.cuda.stream(copy_stream):
        la.record(copy_stream)
        slots[0]["ids"][:b0.n].copy_(ids0, non_blocking=True)
        slots[0]["grads"][:b0.n].copy_(g0, non_blocking=True)
        lb.record(copy_stream)
    torch.cuda.synchronize(dev)
    link_gbs = (ids0.numel() * 8 + g0.numel() * g0.element_size()) / (la.elapsed_time(lb) / 1e3) / 1e9

    # each step's public-API calls (lookup, backward with Adam, erase) captured once as a CUDA graph on its
    # slot's device buffers, as a training loop would run them: per step the timed loop then issues the copies
    # from pinned host memory, one graph replay and the read-back, so the host's own per-call overhead does
    # not sit between the copies
    tab.reserve_workspaces(nmax, n_erase=max((h[3].numel() for h in host if h[3] is not None), default=0))
    torch.cuda.synchronize(dev)
    graphs = []
    for j, (b, ids_h, g_h, er_h) in enumerate(host):
        s = slots[j % 2]
        big = s["big"]
        res = mt.LookupResult(big.unique_keys[:b.n], big.inverse[:b.n], big.counts[:b.n], big.unique_rows[:b.n],
                              big.num_unique, big.rows[:b.n], b.n, big.ranks[:b.n])
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            tab.lookup(s["ids"][:b.n], b.feat_offsets, b.table_ids, result=res)
            tab.backward_adam(res, s["grads"][:b.n])
            if er_h is not None:
                tab.erase(s["erase"][:er_h.numel()], want_found=False)
        graphs.append((gr, res))
    torch.cuda.synchronize(dev)

    used = [None, None]
    landed = [None, None]

    def issue_copy(j):
        k = j % 2
        b, ids_h, g_h, er_h = host[j]
        with torch.cuda.stream(copy_stream):
            if used[k] is not None:
                copy_stream.wait_event(used[k])
            slots[k]["ids"][:b.n].copy_(ids_h, non_blocking=True)
            slots[k]["grads"][:b.n].copy_(g_h, non_blocking=True)
            if er_h is not None:
                slots[k]["erase"][:er_h.numel()].copy_(er_h, non_blocking=True)
            landed[k] = torch.cuda.Event()
            landed[k].record(copy_stream)

    h2d = d2h = ids_done = 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_stream.wait_event(e0)
    issue_copy(0)
    for j in range(ke):
        if j + 1 < ke:
            issue_copy(j + 1)
        k = j % 2
        b, ids_h, g_h, er_h = host[j]
        stream.wait_event(landed[k])
        s = slots[k]
        gr, res = graphs[j]
        gr.replay()  # on `stream`, the current stream
        s["u_h"].copy_(res.num_unique, non_blocking=True)
        used[k] = torch.cuda.Event()
        used[k].record(stream)
        h2d += ids_h.numel() * 8 + g_h.numel() * g_h.element_size() + (er_h.numel() * 8 if er_h is not None else 0)
        d2h += 8
        ids_done += b.n
    e1.record(stream)
    torch.cuda.synchronize(dev)
    secs = e0.elapsed_time(e1) / 1e3
    if tab.error() != 0:
        raise RuntimeError(f"device error {tab.error()} in the end-to-end run")
    tot, mx = aggregate(float(ids_done), secs)
    out = {"value": tot / mx, "unit": UNIT, "h2d_bytes_per_step": h2d // ke, "d2h_bytes_per_step": d2h // ke,
           "steps": ke, "h2d_GB/s_effective": h2d / secs / 1e9, "h2d_GB/s_link": link_gbs,
           "what": "mt_lookup + mt_backward_adam through the Python binding, each step's calls captured as a "
                   "CUDA graph before timing; inputs copied from pinned host memory inside the timed region (one "
                   "step ahead, on a copy stream); the unique count read back each step; a table of its own "
                   "running the same cold, warm-up and fresh steps"}
    del tab, host, slots, graphs
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return out


def jagged_bag_offsets(b) -> np.ndarray:
    """Bags of a feature-major jagged batch: feature f of user u covers positions f*T + [uo[u], uo[u+1])."""
    T = int(b.user_offsets[-1])
    F = b.feat_offsets.size - 1
    return np.concatenate([f * T + b.user_offsets[:-1] for f in range(F)] + [[F * T]]).astype(np.int64)


def shard_run(args, wl, dev, stream, tdt):
    """Sharded two-stage deduplication: G logical ranks on one GPU, each with its own jagged batch and one shard
    table (the keys it owns).  A step is mt_shard_lookup (stage-1 unique per rank, owner partition, exchange,
    stage-2 unique + find/insert + gather at the owners, rows back, expand) and mt_shard_backward_adam (per-rank
    sums to the owners, owner sums, Adam).  The lookup reads the exchange sizes on the host, as a variable
    all-to-all does, so the step runs eagerly (no graph)."""
    import torch
    import update_merged_table_gb300 as mt
    G = args.shard
    log2 = wl.log2 - 1  # the shards share the keys of G batches
    shards = [mt.Table(log2, wl.dim, row_dtype=wl.row, hash_seed=r, device=dev) for r in range(G)]
    grp = mt.ShardGroup(shards)
    steps = min(args.steps, 8)
    nstep = args.warmup + steps
    batches = [[wl.batch(2000 + j * G + r)[0] for r in range(G)] for j in range(nstep)]
    ids = [[torch.from_numpy(b.ids).to(dev) for b in row] for row in batches]
    grads = [[_device_grads(torch, dev, tdt[wl.grad], 3000 + j * G + r, b.n, wl.dim) for r, b in enumerate(row)]
             for j, row in enumerate(batches)]
    stats = [[batch_stats(b) for b in row] for row in batches]

    def step(j):
        row = batches[j]
        res = grp.lookup(ids[j], [b.feat_offsets for b in row], row[0].table_ids)
        ev_m.record(stream)
        grp.backward_adam(res, grads[j])

    for j in range(args.warmup):
        ev_m = torch.cuda.Event(enable_timing=True)
        step(j)
    torch.cuda.synchronize(dev)
    live0 = sum(s.stats()["live"] for s in shards)
    fwd_ms = bwd_ms = 0.0
    for j in range(args.warmup, nstep):
        e0, ev_m, e1 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e0.record(stream)
        step(j)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        fwd_ms += e0.elapsed_time(ev_m)
        bwd_ms += ev_m.elapsed_time(e1)
    live1 = sum(s.stats()["live"] for s in shards)
    if any(s.error() != 0 for s in shards):
        raise RuntimeError("device error in the sharded leg")
    N = sum(b.n for j in range(args.warmup, nstep) for b in batches[j]) / steps
    U = sum(st[0] for j in range(args.warmup, nstep) for st in stats[j]) / steps  # per-rank uniques, summed
    new_keys = max(0.0, (live1 - live0) / steps)
    B, Gb, d = wl.row_bytes, wl.grad_bytes, wl.dim
    # the compulsory bytes of G ranks each with its own batch (the exchange's own traffic is not counted)
    fwd_bytes = 8 * N + 4 * N + U * (8 + 16) + U * B + N * B + new_keys * (16 + B + 8 * d)
    bwd_bytes = N * Gb + 4 * N + U * (4 + 2 * B + 16 * d)
    peak, _ = measured_hbm_peak()
    f_s, b_s = fwd_ms / steps / 1e3, bwd_ms / steps / 1e3
    return {"G": G, "steps": steps, "ids_per_step": N, "rank_uniques_per_step": U, "new_keys_per_step": new_keys,
            "ids_per_s": N / (f_s + b_s), "fwd_ms": f_s * 1e3, "bwd_ms": b_s * 1e3,
            "roofline_fwd": {"bytes_per_step": fwd_bytes, "achieved": fwd_bytes / f_s / 1e9,
                             "frac": fwd_bytes / f_s / 1e9 / peak},
            "roofline_bwd": {"bytes_per_step": bwd_bytes, "achieved": bwd_bytes / b_s / 1e9,
                             "frac": bwd_bytes / b_s / 1e9 / peak},
            "what": "mt_shard_lookup + mt_shard_backward_adam over G logical ranks on one GPU (each a full jagged "
                    "batch of its own), eager: the lookup reads the exchange sizes on the host"}


def merged_run(args, dev, stream):
    """Automatic table merging with mixed row shapes: the 8 features of the merged-tables workload (vocab 1e4 to
    1e6, Zipf 0.8 to 1.3), 2^17 IDs each, given row dims 16, 16, 16, 32, 32, 32, 64, 64 (fp32); the planner puts
    them into three merged tables.  A step is mt_lookup_grouped (every feature segment routed to its table) and
    mt_backward_adam_grouped (each merged table's backward and Adam), the tables side by side on side streams,
    replayed as CUDA graphs on fresh batches."""
    import torch
    import update_merged_table_gb300 as mt
    dims = [16, 16, 16, 32, 32, 32, 64, 64]
    per = 1 << 17
    features = [(dims[k], "f32", W.merged_vocab(k)) for k in range(len(dims))]
    mtabs = mt.MergedTables(features, max_load=0.5, device=dev)
    steps = min(args.steps, 8)
    nstep = 1 + args.warmup + steps
    batches = [W.merged_batch(4000 + j, per_table=per) for j in range(nstep)]
    ids = [torch.from_numpy(b.ids).to(dev) for b in batches]
    sizes = mtabs.group_sizes(batches[0].feat_offsets)
    grads = [[_device_grads(torch, dev, torch.float32, 5000 + 10 * j + g, sizes[g], mtabs.groups[g]["dim"])
              for g in range(len(sizes))] for j in range(nstep)]

    def fwd(j):
        return mtabs.lookup(ids[j], batches[j].feat_offsets)

    for j in range(1 + args.warmup):  # cold step and warm-up, eager (they also size the grouped workspaces)
        mtabs.backward_adam(fwd(j), grads[j])
    torch.cuda.synchronize(dev)
    live0 = [t.stats()["live"] for t in mtabs.tables]
    graphs = []
    for j in range(1 + args.warmup, nstep):
        gf, gb = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(gf, stream=stream):
            res = fwd(j)
        with torch.cuda.graph(gb, stream=stream):
            mtabs.backward_adam(res, grads[j])
        graphs.append((gf, gb))
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in graphs]
    for (gf, gb), (a, m_, z) in zip(graphs, ev):
        a.record(stream)
        gf.replay()
        m_.record(stream)
        gb.replay()
        z.record(stream)
    torch.cuda.synchronize(dev)
    f_s = sum(a.elapsed_time(m_) for a, m_, _ in ev) / 1e3 / steps
    b_s = sum(m_.elapsed_time(z) for _, m_, z in ev) / 1e3 / steps
    live1 = [t.stats()["live"] for t in mtabs.tables]
    if any(t.error() != 0 for t in mtabs.tables):
        raise RuntimeError("device error in the merged-tables leg")
    N = float(sum(sizes))
    # per merged table: its IDs, uniques and row bytes (the same compulsory bytes as the single-table step)
    fwd_bytes = bwd_bytes = 0.0
    fo = batches[-1].feat_offsets
    for g, grp in enumerate(mtabs.groups):
        B = grp["dim"] * 4
        d = grp["dim"]
        segs = [f for f, (gg, _) in enumerate(mtabs.placement) if gg == g]
        keys = np.concatenate([(np.uint64(mtabs.placement[f][1]) << np.uint64(56)) |
                               batches[-1].ids[fo[f]:fo[f + 1]].astype(np.uint64) for f in segs])
        Ng, Ug = float(keys.size), float(np.unique(keys).size)
        new_g = max(0.0, (live1[g] - live0[g]) / steps)
        fwd_bytes += 12 * Ng + Ug * (24 + B) + Ng * B + new_g * (16 + B + 8 * d)
        bwd_bytes += Ng * B + 4 * Ng + Ug * (4 + 2 * B + 16 * d)
    new_keys = max(0.0, (sum(live1) - sum(live0)) / steps)
    peak, _ = measured_hbm_peak()
    return {"tables": [(g["dim"], g["row_dtype"], g["num_features"], g["log2_slots"]) for g in mtabs.groups],
            "ids_per_step": N, "new_keys_per_step": new_keys, "steps": steps,
            "ids_per_s": N / (f_s + b_s), "fwd_ms": f_s * 1e3, "bwd_ms": b_s * 1e3,
            "roofline_fwd": {"bytes_per_step": fwd_bytes, "frac": fwd_bytes / f_s / 1e9 / peak},
            "roofline_bwd": {"bytes_per_step": bwd_bytes, "frac": bwd_bytes / b_s / 1e9 / peak},
            "what": "mt_lookup_grouped over the planner's three merged tables (dims 16, 32, 64) + "
                    "mt_backward_adam_grouped, the tables side by side on side streams, CUDA graphs, fresh batches"}


def queue_ahead(torch, stream, steps: int):
    """Keep the GPU busy for about 2 ms (+ 0.5 ms per step) before an eager pass with per-kernel events, so that
    the host enqueues the pass's launches ahead of the GPU: a kernel's start event and the kernel then run back
    to back, and no host launch latency is counted as kernel time."""
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(2.0e6 * (2.0 + 0.5 * steps)))  # cycles at about 2 GHz


def pooled_run(args, tab, wl, dev, stream, first_seed: int):
    """Mean-pooled jagged bags: each step is a lookup without the per-position gather, the pooled forward
    (mt_pool_forward) and the pooled backward + Adam (mt_backward_adam_pooled), on fresh batches, replayed as
    CUDA graphs with events between the two halves."""
    import torch
    import update_merged_table_gb300 as mt
    steps = min(args.steps, 8)
    seq = wl.steps(first_seed, steps + 1)  # the last batch: one eager pass for the per-kernel device times
    entries = []
    for j, (b, _) in enumerate(seq):
        U, _, _ = batch_stats(b)
        bo = jagged_bag_offsets(b)
        Bg = bo.size - 1
        e = dict(batch=b, U=U, Bg=Bg, ids=torch.from_numpy(b.ids).to(dev), bo=torch.from_numpy(bo).to(dev),
                 res=tab.new_result(b.n, gather=False),
                 dp=_device_grads(torch, dev, torch.float32, 700_000 + first_seed + j, Bg, wl.dim))
        e["out"] = torch.empty((Bg, wl.dim), dtype=torch.float32, device=dev)
        entries.append(e)

    def fwd(e):
        b = e["batch"]
        tab.lookup(e["ids"], b.feat_offsets, b.table_ids, gather=False, result=e["res"])
        tab.pool_forward(e["res"], e["bo"], mode="mean", out=e["out"])

    def bwd(e):
        tab.backward_adam_pooled(e["res"], e["bo"], e["dp"], mode="mean")

    # workspaces sized before capture (a capture must not allocate them)
    tab.reserve_workspaces(max(e["batch"].n for e in entries), max(e["Bg"] for e in entries))
    prof_entry = entries.pop()
    torch.cuda.synchronize(dev)
    graphs = []
    for e in entries:
        gf, gb = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(gf, stream=stream):
            fwd(e)
        with torch.cuda.graph(gb, stream=stream):
            bwd(e)
        graphs.append((gf, gb))
    st0 = tab.stats()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in entries]
    for (gf, gb), (a, m_, z) in zip(graphs, ev):
        a.record(stream)
        gf.replay()
        m_.record(stream)
        gb.replay()
        z.record(stream)
    torch.cuda.synchronize(dev)
    fwd_s = sum(a.elapsed_time(m_) for a, m_, _ in ev) / 1e3 / steps
    bwd_s = sum(m_.elapsed_time(z) for _, m_, z in ev) / 1e3 / steps
    new_keys = max(0.0, (tab.stats()["live"] - st0["live"]) / steps)
    mt.profile_enable(True)
    mt.profile_report(reset=True)
    queue_ahead(torch, stream, 1)
    fwd(prof_entry)
    bwd(prof_entry)
    torch.cuda.synchronize(dev)
    prof = mt.profile_report(reset=True)
    mt.profile_enable(False)
    N = sum(e["batch"].n for e in entries) / steps
    U = sum(e["U"] for e in entries) / steps
    Bg = sum(e["Bg"] for e in entries) / steps
    B, d = wl.row_bytes, wl.dim
    fwd_bytes = 12 * N + 24 * U + new_keys * (16 + B + 8 * d) + 4 * N + U * B + 8 * (Bg + 1) + 4 * d * Bg
    bwd_bytes = 4 * N + 4 * d * Bg + U * (4 + 2 * B + 16 * d)
    peak, _ = measured_hbm_peak()
    return {"mode": "mean", "steps": steps, "bags_per_step": Bg, "ids_per_step": N, "new_keys_per_step": new_keys,
            "fwd_ids_per_s": N / fwd_s, "bwd_ids_per_s": N / bwd_s,
            "roofline_fwd": {"bytes_per_step": fwd_bytes, "ms_per_step": fwd_s * 1e3,
                             "achieved": fwd_bytes / fwd_s / 1e9, "frac": fwd_bytes / fwd_s / 1e9 / peak},
            "roofline_bwd": {"bytes_per_step": bwd_bytes, "ms_per_step": bwd_s * 1e3,
                             "achieved": bwd_bytes / bwd_s / 1e9, "frac": bwd_bytes / bwd_s / 1e9 / peak},
            "kernels_us": {k: round(1e3 * v[1] / v[0], 2) for k, v in prof.items()},
            "what": "lookup without the per-position gather + mean pooling of each (user, feature) bag; backward "
                    "of the pooling folded into the per-unique reduction + Adam (no per-position gradient rows)"}


def run_ours(args):
    import torch
    import update_merged_table_gb300 as mt
    from update_merged_table_gb300 import build_lib

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    numa = bind_to_gpu_numa_node(dev.index)
    build_lib.build()
    mt.load_library()
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16}

    # -------- end to end through the public API with host buffers (its own table, before any capture) ----
    e2e = e2e_run(args, dev, stream, tdt) if args.e2e else None

    wl = Workload(args.config, args.users, args.log2_slots)
    tab = mt.Table(wl.log2, wl.dim, row_dtype=wl.row, device=dev)
    _prefill(torch, tab, wl, dev)
    B, G = wl.row_bytes, wl.grad_bytes
    K = args.steps
    kf = min(K, FRESH_CAP)
    nprof = min(K, 8)
    seq = wl.steps(0, 1 + kf + nprof)  # cold step 0, the timed fresh steps, then the profiling steps
    (cold, _), timed, prof_steps = seq[0], seq[1:1 + kf], seq[1 + kf:]

    def entry(j, b, er):
        U, H, NH = batch_stats(b)
        e = dict(batch=b, U=U, H=H, NH=NH, erase=None, n_erase=0)
        e["ids_d"] = torch.from_numpy(b.ids).to(dev)
        e["grads_d"] = _device_grads(torch, dev, tdt[wl.grad], j, b.n, wl.dim)
        e["res"] = tab.new_result(b.n, gather=True, ranks=bool(args.ranks))
        if er is not None:
            e["erase"] = torch.from_numpy(er.astype(np.int64)).to(dev)
            e["n_erase"] = er.size
        return e

    pool = [entry(1 + j, b, er) for j, (b, er) in enumerate(timed)]
    prof_pool = [entry(1 + kf + j, b, er) for j, (b, er) in enumerate(prof_steps)]

    def fwd_call(e):
        b = e["batch"]
        tab.lookup(e["ids_d"], b.feat_offsets, b.table_ids, result=e["res"])

    def bwd_call(e):
        tab.backward_adam(e["res"], e["grads_d"])
        if e["erase"] is not None:
            tab.erase(e["erase"], want_found=False)

    # the cold step (seed 0; on an empty table every key is new) -- timed on its own, untimed in the run
    cold_ids = torch.from_numpy(cold.ids).to(dev)
    cold_g = _device_grads(torch, dev, tdt[wl.grad], 0, cold.n, wl.dim)
    live_before = int(tab.stats()["live"])
    torch.cuda.synchronize(dev)
    c0, c1, c2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    c0.record(stream)
    cres = tab.lookup(cold_ids, cold.feat_offsets, cold.table_ids)
    c1.record(stream)
    tab.backward_adam(cres, cold_g)
    c2.record(stream)
    torch.cuda.synchronize(dev)
    cold_stats = {"ids": cold.n, "new_keys": int(tab.stats()["live"]) - live_before, "lookup_ms": c0.elapsed_time(c1),
                  "backward_ms": c1.elapsed_time(c2), "note": "step 0, the first call: includes lazy set-up"}
    # warm-up: the cold batch again (its keys are resident now; no erase)
    for _ in range(args.warmup):
        cres = tab.lookup(cold_ids, cold.feat_offsets, cold.table_ids, result=cres)
        tab.backward_adam(cres, cold_g)
    torch.cuda.synchronize(dev)
    del cres, cold_ids, cold_g

    graphs = None
    launches_per_step = None
    if args.graph:
        # every workspace sized for the largest batch first: a capture must not replace a buffer that graphs
        # captured before it still use
        tab.reserve_workspaces(max(e["batch"].n for e in pool + prof_pool),
                               n_erase=max(e["n_erase"] for e in pool + prof_pool))
        torch.cuda.synchronize(dev)
        graphs = []
        l0 = mt.kernel_launches()
        for e in pool:
            gf, gb = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
            with torch.cuda.graph(gf, stream=stream):
                fwd_call(e)
            with torch.cuda.graph(gb, stream=stream):
                bwd_call(e)
            graphs.append((gf, gb))
        torch.cuda.synchronize(dev)
        launches_per_step = (mt.kernel_launches() - l0) / len(pool)

    def run_fwd(j):
        if graphs is not None:
            graphs[j % kf][0].replay()
        else:
            fwd_call(pool[j % kf])

    def run_bwd(j):
        if graphs is not None:
            graphs[j % kf][1].replay()
        else:
            bwd_call(pool[j % kf])

    # -------- timed region: K steps on fresh batches, inputs resident in HBM --------
    st0 = tab.stats()
    n_ids = sum(pool[j % kf]["batch"].n for j in range(K))
    launches0 = mt.kernel_launches()
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_m = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clk:
        ev0.record(stream)
        for j in range(K):
            ev_a[j].record(stream)
            run_fwd(j)
            ev_m[j].record(stream)
            run_bwd(j)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    if ws > 1:
        dist.barrier()
    secs = ev0.elapsed_time(ev1) / 1e3
    fwd_ms = sum(ev_a[j].elapsed_time(ev_m[j]) for j in range(K))
    bwd_ms = sum(ev_m[j].elapsed_time(ev_a[j + 1] if j + 1 < K else ev1) for j in range(K))
    launches = mt.kernel_launches() - launches0
    if launches_per_step is not None:  # graph replays launch the captured kernels
        launches = int(round(launches_per_step * K))
    st1 = tab.stats()
    erased = sum(pool[j % kf]["n_erase"] for j in range(K))  # every erase key of the stream is live
    n_new_per_step = max(0.0, (st1["live"] - st0["live"] + erased) / K)
    tot_ids, tot_secs = aggregate(float(n_ids), secs)

    # -------- per-kernel device times: an eager pass over further fresh steps --------
    pst0 = tab.stats()
    mt.profile_enable(True)
    mt.profile_report(reset=True)
    queue_ahead(torch, stream, len(prof_pool))
    for e in prof_pool:
        fwd_call(e)
        bwd_call(e)
    torch.cuda.synchronize(dev)
    prof = mt.profile_report(reset=True)
    mt.profile_enable(False)
    pst1 = tab.stats()
    p_erased = sum(e["n_erase"] for e in prof_pool)
    p_new = max(0.0, (pst1["live"] - pst0["live"] + p_erased) / len(prof_pool))

    # algorithmic bytes per step (the timed steps' own batches; new keys from the table's growth)
    def mean(key, entries):
        return sum(e[key] for e in entries) / len(entries)

    N_avg = sum(pool[j % kf]["batch"].n for j in range(K)) / K
    U_avg = sum(pool[j % kf]["U"] for j in range(K)) / K
    fwd_bytes = (8 * N_avg + 4 * N_avg + U_avg * (8 + 16) + U_avg * B + N_avg * B
                 + n_new_per_step * (16 + B + 8 * wl.dim))
    bwd_bytes = N_avg * G + 4 * N_avg + U_avg * (4 + 2 * B + 16 * wl.dim)
    row_rw = 2 * B + 16 * wl.dim  # emb, m, v read and written
    pN = sum(e["batch"].n for e in prof_pool) / len(prof_pool)
    pU, pH, pNH = mean("U", prof_pool), mean("H", prof_pool), mean("NH", prof_pool)
    kernel_bytes = {  # algorithmic bytes per launch of the kernels that move the bulk
        "k_bw_heavy_reduce": pNH * (G + 4) + pH * row_rw,
        "k_bw_light_reduce": (pN - pNH) * (G + 4) + (pU - pH) * (row_rw + 16),
        "k_gather": pN * B + pU * B + 4 * pN,
    }
    peak, peak_kind = measured_hbm_peak()
    tot_k = sum(v[1] for v in prof.values()) or 1.0
    dom = max((k for k in prof if k in kernel_bytes), key=lambda k: prof[k][1])
    dom_ms = prof[dom][1] / prof[dom][0]
    achieved = kernel_bytes[dom] / (dom_ms / 1e3) / 1e9
    per_id, traffic_note = committed_traffic(dom) if args.config == 3 else (None, "counters cover the jagged workload")
    traffic = per_id * pN if per_id is not None else None

    # -------- pooled jagged bags (sum/mean of each user's rows per feature) on further fresh steps --------
    pooled = pooled_run(args, tab, wl, dev, stream, 1 + kf + nprof) if (args.config == 3 and args.pooled) else None

    # -------- sharded two-stage dedup: G logical ranks, each with a batch and a shard table of its own --------
    sharded = shard_run(args, wl, dev, stream, tdt) if (args.config == 3 and args.shard > 1 and ws == 1) else None

    # -------- automatic table merging with mixed row shapes: the grouped lookup over the planner's tables --------
    merged = merged_run(args, dev, stream) if (args.config == 3 and args.merged and ws == 1) else None

    # -------- tombstone compaction of the key store (one call, outside the step) --------
    comp = None
    if ws == 1:
        st_before = tab.stats()
        tab.compact()  # first call allocates its workspace
        torch.cuda.synchronize(dev)
        cc0, cc1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        mt.profile_enable(True)
        mt.profile_report(reset=True)
        cc0.record(stream)
        tab.compact()
        cc1.record(stream)
        torch.cuda.synchronize(dev)
        cp = mt.profile_report(reset=True)
        mt.profile_enable(False)
        c_ms = cc0.elapsed_time(cc1)
        k_ms = cp["k_compact_rebuild"][1] if "k_compact_rebuild" in cp else None
        M = 1 << wl.log2
        comp = {"ms": c_ms, "kernel_ms": k_ms, "slots": M, "live": int(st_before["live"]),
                "algorithmic_GB/s": 32.0 * M / (c_ms / 1e3) / 1e9,  # read every old slot, write every new one
                "note": "mt_compact (one call: clear the spare slot array, re-insert the live keys into it, swap); "
                        "kernel_ms is the re-insert kernel alone"}

    # -------- occupancy statistics: one scan of the key store (the kernel's own device time) --------
    stats_leg = None
    if ws == 1:
        tab.stats()
        mt.profile_enable(True)
        mt.profile_report(reset=True)
        tab.stats()
        sp = mt.profile_report(reset=True)
        mt.profile_enable(False)
        if "k_stats" in sp:
            s_ms = sp["k_stats"][1] / sp["k_stats"][0]
            M = 1 << wl.log2
            stats_leg = {"kernel_ms": s_ms, "slots": M, "algorithmic_GB/s": 16.0 * M / (s_ms / 1e3) / 1e9,
                         "frac": 16.0 * M / (s_ms / 1e3) / 1e9 / peak,
                         "note": "mt_stats: one read of every 16-byte slot (live, tombstones, probe-index histogram)"}

    # -------- capacity expansion: twice the slots, rows unchanged (one call, after everything else) --------
    grow = None
    if ws == 1 and args.grow:
        st_before = tab.stats()
        M_old = 1 << wl.log2
        torch.cuda.synchronize(dev)
        mt.profile_enable(True)
        mt.profile_report(reset=True)
        g0 = time.perf_counter()
        tab.grow(wl.log2 + 1, num_rows=tab.cfg.num_rows)  # synchronises
        g_ms = (time.perf_counter() - g0) * 1e3
        gp = mt.profile_report(reset=True)
        mt.profile_enable(False)
        grow = {"ms_host_timed": g_ms, "kernels_ms": {k: v[1] for k, v in gp.items()},
                "slots_before": M_old, "slots_after": 2 * M_old,
                "live": int(st_before["live"]),
                "rows_moved": 0, "row_bytes_in_table": int(tab.cfg.num_rows) * (B + 8 * wl.dim),
                "key_store_GB/s": (16.0 * M_old + 16.0 * 2 * M_old) / (g_ms / 1e3) / 1e9,
                "note": "mt_table_grow: a new key store (old slots read, new slots cleared and filled); the rows "
                        "stay in place, so the cost follows the slot count, not the row pool; ms_host_timed includes "
                        "allocating the new key store and row segment"}
        if tab.stats()["live"] != st_before["live"]:
            raise RuntimeError("capacity expansion lost keys")

    err = tab.error()
    if err != 0:
        raise RuntimeError(f"device error {err} during the benchmark")

    fwd_s, bwd_s = fwd_ms / K / 1e3, bwd_ms / K / 1e3
    line = {
        "metric": METRIC, "value": tot_ids / tot_secs, "unit": UNIT, "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": 1e3 * tot_secs / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.row, "data": "synthetic",
        "config": {"workload": wl.name, "ids_per_step": N_avg, "unique_per_step": U_avg,
                   "new_keys_per_step": n_new_per_step, "fresh_steps": kf,
                   "steps_cycle_fresh_batches": K > kf,
                   "step_sequence": (f"cold step 0 (seed 0) untimed, {args.warmup} warm-up steps on it, then timed "
                                     f"steps 1..{K} on fresh seeds" + (f" (cycling {kf} batches)" if K > kf else "")),
                   "cuda_graph": bool(args.graph), "lookup_ranks": bool(args.ranks),
                   "l2": ("inputs larger than L2 (ids+grads+out ~0.5 GB per step), no flush" if args.config == 3
                          else "fresh batches every step; see the workload's sizes"),
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU", "host_binding": numa,
                   "direction_timing": "CUDA events between the lookup and backward graph replays of each step"},
        "fwd_ids_per_s": N_avg / fwd_s, "bwd_ids_per_s": N_avg / bwd_s,
        "roofline_fwd": {"bytes_per_step": fwd_bytes, "ms_per_step": fwd_s * 1e3, "achieved": fwd_bytes / fwd_s / 1e9,
                         "peak": peak, "unit": "GB/s", "frac": fwd_bytes / fwd_s / 1e9 / peak},
        "roofline_bwd": {"bytes_per_step": bwd_bytes, "ms_per_step": bwd_s * 1e3, "achieved": bwd_bytes / bwd_s / 1e9,
                         "peak": peak, "unit": "GB/s", "frac": bwd_bytes / bwd_s / 1e9 / peak},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_kind, "traffic": traffic,
                     "traffic_source": traffic_note,
                     "algorithmic_bytes_per_launch": kernel_bytes[dom], "avg_launch_ms": dom_ms,
                     "time_share": prof[dom][1] / tot_k},
        "kernel_rooflines": {k: {"GB/s": kernel_bytes[k] / (prof[k][1] / prof[k][0] / 1e3) / 1e9,
                                 "frac": kernel_bytes[k] / (prof[k][1] / prof[k][0] / 1e3) / 1e9 / peak}
                             for k in kernel_bytes if k in prof},
        "kernels": {k: {"launches": v[0], "avg_us": 1e3 * v[1] / v[0], "share": v[1] / tot_k} for k, v in prof.items()},
        "kernel_pass": f"eager, CUDA events around each launch, {len(prof_pool)} further fresh steps "
                       f"({p_new:.0f} new keys per step)",
        "cold_step": cold_stats,
        "pooled": pooled,
        "sharded": sharded,
        "merged": merged,
        "compaction": comp,
        "stats": stats_leg,
        "grow": grow,
        "e2e": e2e,
        "gpu_launches": int(launches),
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(Workload(args.config, args.users, args.log2_slots), args.cpu_seconds)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the oracle on the host cores (reported baseline / reference arm)
# ---------------------------------------------------------------------------

class OracleSteps:
    """The oracle (single-threaded C++) on bounded samples of the workload: a
    smaller batch of the same distributions per step (for the jagged workload
    the first 256 users), starting with one untimed cold step."""

    def __init__(self, wl: Workload):
        import oracle
        self.oracle = oracle
        self.wl = wl
        self.ref = oracle.Table(wl.log2, wl.dim, row_dtype=oracle.BF16 if wl.row == "bf16" else oracle.F32)
        self.k = 0
        self.step()  # cold step

    def _grads(self, seed, n):
        import torch
        g = W.grads_normal(seed, n, self.wl.dim)
        if self.wl.grad == "bf16":
            return torch.from_numpy(g).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16), self.oracle.BF16
        return g, self.oracle.F32

    def step(self):
        """One lookup + backward on the next sample batch; returns (IDs, seconds of oracle time)."""
        b = self.wl.sample_batch(self.k)
        g, gd = self._grads(self.k + 500_000, b.n)
        t0 = time.perf_counter()
        self.ref.lookup(b.ids, b.feat_offsets, b.table_ids)
        self.ref.backward_adam(g, grad_dtype=gd)
        dt = time.perf_counter() - t0
        self.k += 1
        return b.n, dt


def cpu_baseline(wl: Workload, budget_s: float):
    """Oracle lookup+backward IDs/s: steps on bounded samples until about
    `budget_s` seconds of oracle time have been spent."""
    runner = OracleSteps(wl)
    ids_done, t_total, steps = 0, 0.0, 0
    while t_total < budget_s and steps < 10_000:
        n, dt = runner.step()
        ids_done += n
        t_total += dt
        steps += 1
    return {"value": ids_done / t_total, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{steps} steps of a reduced batch (avg {ids_done // max(1, steps)} IDs/step) of the same "
                      f"workload after one untimed cold step; single-threaded C++ oracle, {t_total:.1f} s"}


def run_reference(args):
    """The reference arm: the oracle as it stands, W untimed warm-up steps and
    then K timed steps, each a bounded sample of the workload (a time cap
    ends the timed steps early if K of them would take too long; the line
    says how many ran)."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    wl = Workload(args.config, args.users, args.log2_slots)
    runner = OracleSteps(wl)
    for _ in range(args.warmup):
        runner.step()
    ids_done, t_total, steps = 0, 0.0, 0
    while steps < args.steps and t_total < args.ref_seconds:
        n, dt = runner.step()
        ids_done += n
        t_total += dt
        steps += 1
    value = ids_done / t_total
    sample = (f"{steps} timed steps (of {args.steps} asked; cap {args.ref_seconds:.0f} s) of a reduced batch "
              f"(avg {ids_done // max(1, steps)} IDs/step) of the same workload after one cold and {args.warmup} "
              f"warm-up steps; single-threaded C++ oracle, {t_total:.1f} s")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * t_total / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name + " (bounded sample per step, see cpu_baseline.sample)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=3, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--e2e", type=int, default=1, help="also time the step through host buffers (its own table)")
    ap.add_argument("--pooled", type=int, default=1, help="also time the pooled jagged-bag step (jagged workload)")
    ap.add_argument("--grow", type=int, default=1, help="also time one capacity expansion at the end")
    ap.add_argument("--merged", type=int, default=1,
                    help="also time the grouped lookup over planner-merged tables of dims 16/32/64 (with config 3)")
    ap.add_argument("--shard", type=int, default=2,
                    help="also time the sharded two-stage dedup with this many logical ranks (jagged workload; 0: no)")
    ap.add_argument("--ranks", type=int, default=1,
                    help="1: the lookup also returns per-position ranks (the backward groups positions with them); "
                         "0: the backward groups positions itself")
    ap.add_argument("--graph", type=int, default=1, help="replay each step as a captured CUDA graph")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-seconds", type=float, default=150.0,
                    help="--impl reference: cap on the timed oracle seconds")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--users", type=int, default=2048, help="users per jagged batch (smaller cases for profiling)")
    ap.add_argument("--log2-slots", type=int, default=None)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
