"""Benchmark of the merged dynamic embedding table hot path on GB300.

One step = one lookup (encode, two-stage dedup, find/insert, gather) plus one
backward (per-unique gradient sum + sparse Adam) over one batch, plus the
erase of that step's deletions for the online-churn workload.  The default
workload (``--config 3``) is the GRM jagged-sequence batch: 2048 users with
lognormal(5, 1) sequence lengths capped at 3000, 4 ID features per token
(Zipf(1.1) over 1e6 IDs each, merged by table id), M = 2^24 slots, dim 64
bf16 rows, fp32 Adam state, bf16 grads.  Synthetic, seeded inputs; every
step's inputs and outputs exceed the 126 MB L2, so no flush is needed between
steps.  ``--config 1, 2, 4, 5`` time the single-table, merged-tables,
large-table and online-churn workloads the same way.

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

class Workload:
    """Table shape, batch generator and (for the oracle sample) a smaller batch generator."""

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
                         "erase of 2^16 keys per step")
            self.log2, self.dim, self.row, self.grad = 24, 64, "f32", "f32"
            self.churn = W.ChurnStream(0)
            self.prefill_ids = self.churn.prefill_ids
        else:
            raise ValueError("config must be 1..5")
        if log2_slots is not None:
            self.log2 = log2_slots
        if cfg == 3 and (users != 2048 or self.log2 != 24):
            self.name = (f"GRM jagged sequences (reduced): {users} users, lognormal(5,1) lengths capped at 3000, "
                         f"4 ID features, M=2^{self.log2}, dim 64 bf16")

    def batch(self, seed: int):
        """(batch, erase ids or None) of step `seed`."""
        if self.cfg == 1:
            return W.single_table_batch(seed), None
        if self.cfg == 2:
            return W.merged_batch(seed), None
        if self.cfg == 3:
            return W.jagged_batch(seed, users=self.users), None
        if self.cfg == 4:
            return W.large_table_batch(seed), None
        return self.churn.step(seed)

    def sample_batch(self, seed: int):
        """A bounded slice of the same workload for the CPU oracle."""
        if self.cfg == 2:
            return W.merged_batch(seed, per_table=2048)
        if self.cfg == 3:
            return W.jagged_batch(seed, users=256)
        if self.cfg == 4:
            return W.large_table_batch(seed, n=1 << 17)
        if self.cfg == 5:
            b, _ = self.churn.step(seed)
            return W.single_feature(b.ids[: 1 << 16])
        return W.single_table_batch(seed)

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


def bind_to_gpu_numa_node(dev_index: int) -> str:
    """Run on the CPUs next to the GPU so pinned host buffers land in its NUMA node."""
    try:
        import torch
        bus = torch.cuda.get_device_properties(dev_index).pci_bus_id.lower()
        for cand in (bus, "0000" + bus[4:] if len(bus) > 4 else bus):
            path = f"/sys/bus/pci/devices/{cand}/local_cpulist"
            if os.path.exists(path):
                cpus = set()
                for part in open(path).read().strip().split(","):
                    a, _, b = part.partition("-")
                    cpus.update(range(int(a), int(b or a) + 1))
                if cpus:
                    os.sched_setaffinity(0, cpus)
                    return f"cpus {min(cpus)}-{max(cpus)}"
    except Exception:
        pass
    return "unbound"


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

    wl = Workload(args.config, args.users, args.log2_slots)
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16}
    tab = mt.Table(wl.log2, wl.dim, row_dtype=wl.row, device=dev)
    if wl.prefill_ids is not None:  # untimed: the resident key set of a steady state
        pre = wl.prefill_ids()
        for s0 in range(0, pre.size, 1 << 22):
            tab.lookup(torch.from_numpy(pre[s0:s0 + (1 << 22)]).to(dev), gather=False)
        del pre
    B, G = wl.row_bytes, wl.grad_bytes

    pool = []
    for k in range(args.pool):
        b, er = wl.batch(1 + k + 1000 * rank)
        U, H, NH = batch_stats(b)
        g = torch.from_numpy(W.grads_normal(1 + k + 500_000 + 1000 * rank, b.n, wl.dim)).to(tdt[wl.grad])
        e = dict(batch=b, grads=g, U=U, H=H, NH=NH, erase=None)
        e["ids_d"] = torch.from_numpy(b.ids).to(dev)
        e["grads_d"] = g.to(dev)
        e["res"] = tab.new_result(b.n, gather=True)
        if er is not None:
            e["erase"] = torch.from_numpy(er.astype(np.int64)).to(dev)
        e["ids_h"] = torch.from_numpy(b.ids).pin_memory()
        e["grads_h"] = g.pin_memory()
        e["u_h"] = torch.empty(1, dtype=torch.int64).pin_memory()
        pool.append(e)

    def step(e):
        b = e["batch"]
        tab.lookup(e["ids_d"], b.feat_offsets, b.table_ids, result=e["res"])
        tab.backward_adam(e["res"], e["grads_d"])
        if e["erase"] is not None:
            tab.erase(e["erase"], want_found=False)

    # the cold step (a batch on the table as prefilled; for the jagged workload every key is new) -- untimed
    cold, _ = wl.batch(1000 * rank + 999)
    cold_ids = torch.from_numpy(cold.ids).to(dev)
    cold_g = torch.from_numpy(W.grads_normal(7, cold.n, wl.dim)).to(tdt[wl.grad]).to(dev)
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
                  "backward_ms": c1.elapsed_time(c2), "note": "first step after set-up, includes lazy set-up"}
    del cres, cold_ids, cold_g
    for j in range(args.warmup):
        step(pool[j % len(pool)])
    torch.cuda.synchronize(dev)

    # -------- end to end through the public API with host buffers --------
    # (measured before any graph is captured: the eager API is what a caller
    # feeding host buffers uses)
    # Every step copies its IDs and gradients from pinned host memory and reads
    # its unique count back; the copies of step j + 1 run on a copy stream
    # while step j computes (the pool entry's device buffers are rewritten only
    # after the step that last used them has finished).
    e2e_steps = min(args.steps, 4 * len(pool))
    h2d = d2h = 0
    ev2, ev3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_ids = 0
    copy_stream = torch.cuda.Stream(device=dev)
    P = len(pool)
    used = [None] * P    # event after the step that last used entry k's device buffers
    landed = [None] * P  # event after entry k's inputs reached the device

    def issue_copy(j):
        k = j % P
        e = pool[k]
        with torch.cuda.stream(copy_stream):
            if used[k] is not None:
                copy_stream.wait_event(used[k])
            e["ids_d"].copy_(e["ids_h"], non_blocking=True)
            e["grads_d"].copy_(e["grads_h"], non_blocking=True)
            landed[k] = torch.cuda.Event()
            landed[k].record(copy_stream)

    torch.cuda.synchronize(dev)
    ev2.record(stream)
    copy_stream.wait_event(ev2)
    issue_copy(0)
    for j in range(e2e_steps):
        if j + 1 < e2e_steps:
            issue_copy(j + 1)
        k = j % P
        e = pool[k]
        stream.wait_event(landed[k])
        step(e)
        e["u_h"].copy_(e["res"].num_unique, non_blocking=True)
        used[k] = torch.cuda.Event()
        used[k].record(stream)
        h2d += e["ids_h"].numel() * 8 + e["grads_h"].numel() * e["grads_h"].element_size()
        d2h += 8
        e2e_ids += e["batch"].n
    ev3.record(stream)
    torch.cuda.synchronize(dev)
    e2e_secs = ev2.elapsed_time(ev3) / 1e3
    e2e_tot, e2e_max = aggregate(float(e2e_ids), e2e_secs)

    graphs = None
    launches_per_step = None
    if args.graph:
        graphs = []
        c0 = mt.kernel_launches()
        for e in pool:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(e)
            graphs.append(g)
        torch.cuda.synchronize(dev)
        launches_per_step = (mt.kernel_launches() - c0) / len(pool)

        def run(j):
            graphs[j % len(pool)].replay()
    else:
        def run(j):
            step(pool[j % len(pool)])

    # -------- timed region: K steps, inputs resident in HBM --------
    live0 = tab.stats()["live"]
    n_ids = sum(pool[j % len(pool)]["batch"].n for j in range(args.steps))
    launches0 = mt.kernel_launches()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clk:
        ev0.record(stream)
        for j in range(args.steps):
            run(j)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    if ws > 1:
        dist.barrier()
    secs = ev0.elapsed_time(ev1) / 1e3
    launches = mt.kernel_launches() - launches0
    if launches_per_step is not None:  # graph replays launch the captured kernels
        launches = int(round(launches_per_step * args.steps))
    live1 = tab.stats()["live"]
    tot_ids, tot_secs = aggregate(float(n_ids), secs)

    # -------- per-direction and per-kernel device times (separate pass) --------
    # The lookup and the backward are timed the way the step runs: as CUDA
    # graph replays when the step is replayed from a graph, else eagerly.
    def fwd_call(e):
        tab.lookup(e["ids_d"], e["batch"].feat_offsets, e["batch"].table_ids, result=e["res"])

    def bwd_call(e):
        tab.backward_adam(e["res"], e["grads_d"])

    if args.graph:
        dir_graphs = []
        for e in pool:
            gf, gb = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
            with torch.cuda.graph(gf, stream=stream):
                fwd_call(e)
            with torch.cuda.graph(gb, stream=stream):
                bwd_call(e)
            dir_graphs.append((gf, gb))
        torch.cuda.synchronize(dev)
    fwd_ms = bwd_ms = 0.0
    npass = min(args.steps, 4 * len(pool))
    pass_ids = pass_U = pass_H = pass_NH = 0
    evs = []
    for j in range(npass):
        e = pool[j % len(pool)]
        a, m_, z = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        a.record(stream)
        if args.graph:
            dir_graphs[j % len(pool)][0].replay()
        else:
            fwd_call(e)
        m_.record(stream)
        if args.graph:
            dir_graphs[j % len(pool)][1].replay()
        else:
            bwd_call(e)
        z.record(stream)
        if e["erase"] is not None:
            tab.erase(e["erase"], want_found=False)
        evs.append((a, m_, z))
        pass_ids += e["batch"].n
        pass_U += e["U"]
        pass_H += e["H"]
        pass_NH += e["NH"]
    torch.cuda.synchronize(dev)
    for a, m_, z in evs:
        fwd_ms += a.elapsed_time(m_)
        bwd_ms += m_.elapsed_time(z)
    mt.profile_enable(True)
    mt.profile_report(reset=True)
    for j in range(npass):
        step(pool[j % len(pool)])
    torch.cuda.synchronize(dev)
    prof = mt.profile_report(reset=True)
    mt.profile_enable(False)

    # algorithmic bytes (new keys counted from the live-key growth of the timed steps)
    n_new_per_step = max(0.0, (live1 - live0) / max(1, args.steps))
    N_avg = pass_ids / npass
    U_avg = pass_U / npass
    H_avg, NH_avg = pass_H / npass, pass_NH / npass
    fwd_bytes = (8 * N_avg + 4 * N_avg + U_avg * (8 + 16) + U_avg * B + N_avg * B
                 + n_new_per_step * (16 + B + 8 * wl.dim))
    bwd_bytes = N_avg * G + 4 * N_avg + U_avg * (4 + 2 * B + 16 * wl.dim)
    row_rw = 2 * B + 16 * wl.dim  # emb, m, v read and written
    kernel_bytes = {  # algorithmic bytes per launch of the kernels that move the bulk
        "k_bw_heavy_reduce": NH_avg * (G + 4) + H_avg * row_rw,
        "k_bw_light_reduce": (N_avg - NH_avg) * (G + 4) + (U_avg - H_avg) * (row_rw + 16),
        "k_gather": N_avg * B + U_avg * B + 4 * N_avg,
    }
    peak, peak_kind = measured_hbm_peak()
    tot_k = sum(v[1] for v in prof.values()) or 1.0
    dom = max((k for k in prof if k in kernel_bytes), key=lambda k: prof[k][1])
    dom_ms = prof[dom][1] / prof[dom][0]
    achieved = kernel_bytes[dom] / (dom_ms / 1e3) / 1e9
    traffic = None  # DRAM bytes per launch from the committed ncu summary, scaled by the IDs of a launch
    tpath = os.path.join(ROOT, "profiles", "kernel_traffic.txt")
    if args.config == 3 and os.path.exists(tpath):
        for line in open(tpath):
            f = line.split()
            if len(f) == 2 and f[0] == dom:
                traffic = float(f[1]) * N_avg

    # -------- tombstone compaction of the key store (one call, untimed in the step) --------
    comp = None
    if ws == 1:
        st_before = tab.stats()
        tab.compact()  # first call allocates its workspace
        torch.cuda.synchronize(dev)
        cc0, cc1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        cc0.record(stream)
        tab.compact()
        cc1.record(stream)
        torch.cuda.synchronize(dev)
        c_ms = cc0.elapsed_time(cc1)
        M = 1 << wl.log2
        comp = {"ms": c_ms, "slots": M, "live": int(st_before["live"]),
                "algorithmic_GB/s": 32.0 * M / (c_ms / 1e3) / 1e9,  # read every old slot, write every new one
                "moved_GB/s": 80.0 * M / (c_ms / 1e3) / 1e9,  # + clear the fresh array, copy it back
                "note": "mt_compact: live keys re-inserted into a fresh slot array that replaces the table's"}

    err = tab.error()
    if err != 0:
        raise RuntimeError(f"device error {err} during the benchmark")

    line = {
        "metric": METRIC, "value": tot_ids / tot_secs, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * tot_secs / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.row, "data": "synthetic",
        "config": {"workload": wl.name, "ids_per_step": N_avg, "unique_per_step": U_avg,
                   "new_keys_per_step": n_new_per_step, "batch_pool": len(pool), "cuda_graph": bool(args.graph),
                   "l2": ("inputs larger than L2 (ids+grads+out ~0.5 GB per step), no flush" if args.config == 3
                          else "batch pool cycled; see the workload's sizes"),
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU", "host_binding": numa,
                   "direction_timing": "graph replays" if args.graph else "eager"},
        "fwd_ids_per_s": pass_ids / (fwd_ms / 1e3), "bwd_ids_per_s": pass_ids / (bwd_ms / 1e3),
        "kernel_rooflines": {k: {"GB/s": kernel_bytes[k] / (prof[k][1] / prof[k][0] / 1e3) / 1e9,
                                 "frac": kernel_bytes[k] / (prof[k][1] / prof[k][0] / 1e3) / 1e9 / peak}
                             for k in kernel_bytes if k in prof},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_kind, "traffic": traffic,
                     "algorithmic_bytes_per_launch": kernel_bytes[dom], "avg_launch_ms": dom_ms,
                     "time_share": prof[dom][1] / tot_k},
        "roofline_fwd": {"bytes_per_step": fwd_bytes, "achieved": fwd_bytes / (fwd_ms / npass / 1e3) / 1e9,
                         "frac": fwd_bytes / (fwd_ms / npass / 1e3) / 1e9 / peak},
        "roofline_bwd": {"bytes_per_step": bwd_bytes, "achieved": bwd_bytes / (bwd_ms / npass / 1e3) / 1e9,
                         "frac": bwd_bytes / (bwd_ms / npass / 1e3) / 1e9 / peak},
        "kernels": {k: {"launches": v[0], "avg_us": 1e3 * v[1] / v[0], "share": v[1] / tot_k} for k, v in prof.items()},
        "cold_step": cold_stats,
        "compaction": comp,
        "e2e": {"value": e2e_tot / e2e_max, "unit": UNIT, "h2d_bytes_per_step": h2d // e2e_steps,
                "d2h_bytes_per_step": d2h // e2e_steps},
        "gpu_launches": int(launches),
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
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
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=3, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--pool", type=int, default=8, help="distinct pre-generated batches cycled through")
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
