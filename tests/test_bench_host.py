"""The benchmark's host-side pieces on CPU: every workload builds batches of
the sizes it states, its bounded oracle sample is smaller than the timed
batch, and the batch statistics behind the algorithmic bytes (uniques, heavy
uniques and their positions) match a plain count."""
import collections

import numpy as np
import pytest

import bench


def plain_stats(b):
    f = np.searchsorted(b.feat_offsets, np.arange(b.n), side="right") - 1
    keys = [(int(b.table_ids[f[i]]) << 56) | int(b.ids[i]) for i in range(b.n)]
    cnt = collections.Counter(keys)
    heavy = [c for c in cnt.values() if c > 32]
    return len(cnt), len(heavy), sum(heavy)


@pytest.mark.parametrize("cfg, n", [(1, 4096), (2, 65536), (4, 1 << 20)])
def test_workload_batch_sizes(cfg, n):
    wl = bench.Workload(cfg)
    b, er = wl.batch(1)
    assert b.n == n and er is None
    assert b.feat_offsets[0] == 0 and b.feat_offsets[-1] == b.n and np.all(np.diff(b.feat_offsets) >= 0)
    s = wl.sample_batch(1)
    assert 0 < s.n <= b.n


def test_jagged_workload_and_reduced_name():
    wl = bench.Workload(3, users=64, log2_slots=18)
    b, er = wl.batch(2)
    assert er is None and b.table_ids.tolist() == [0, 1, 2, 3]
    assert b.n == b.feat_offsets[-1] and b.n % 4 == 0  # four features per token
    assert "reduced" in wl.name and wl.log2 == 18 and wl.row == "bf16" and wl.grad == "bf16"


def test_batch_stats_match_a_plain_count():
    wl = bench.Workload(2)
    b, _ = wl.batch(3)
    assert bench.batch_stats(b) == plain_stats(b)
    wl3 = bench.Workload(3, users=48)
    b3, _ = wl3.batch(0)
    assert bench.batch_stats(b3) == plain_stats(b3)


def test_row_and_grad_bytes():
    wl = bench.Workload(3)
    assert wl.row_bytes == 128 and wl.grad_bytes == 128
    wl4 = bench.Workload(4)
    assert wl4.row_bytes == 512 and wl4.grad_bytes == 512


def test_churn_steps_are_sequential():
    wl = bench.Workload(5)
    wl.churn = bench.W.ChurnStream(0, hot=1 << 12, n=1 << 10, erase=1 << 8)
    a = wl.steps(0, 2)
    b = wl.steps(2, 1)
    assert len(a) == 2 and len(b) == 1 and all(er is not None and er.size == 1 << 8 for _, er in a + b)
    with pytest.raises(ValueError):
        wl.steps(7, 1)
    with pytest.raises(ValueError):
        wl.batch(1)


def _fake_sysfs(tmp_path, bus, local=None, node=None, nodes=None, distance=None):
    d = tmp_path / "bus" / "pci" / "devices" / bus
    d.mkdir(parents=True)
    if local is not None:
        (d / "local_cpulist").write_text(local + "\n")
    if node is not None:
        (d / "numa_node").write_text(f"{node}\n")
    for k, cpus in (nodes or {}).items():
        nd = tmp_path / "devices" / "system" / "node" / f"node{k}"
        nd.mkdir(parents=True)
        (nd / "cpulist").write_text(cpus + "\n")
        if distance and k in distance:
            (nd / "distance").write_text(" ".join(map(str, distance[k])) + "\n")
    return str(tmp_path)


def test_numa_binding_prefers_local_cpulist(tmp_path):
    root = _fake_sysfs(tmp_path, "0000:01:00.0", local="0-3,8")
    cpus, how = bench.numa_cpus_for_gpu("00000000:01:00.0", root)
    assert cpus == {0, 1, 2, 3, 8} and how == "local_cpulist"


def test_numa_binding_from_numa_node(tmp_path):
    root = _fake_sysfs(tmp_path, "0009:01:00.0", node=1, nodes={0: "0-71", 1: "72-143"})
    cpus, how = bench.numa_cpus_for_gpu("0009:01:00.0", root)
    assert cpus == set(range(72, 144)) and how == "numa_node 1"


def test_numa_binding_gpu_memory_node_takes_nearest_cpu_node(tmp_path):
    # the GPU's node holds memory only (no CPUs): the CPU node at the smallest distance is chosen
    root = _fake_sysfs(tmp_path, "0009:01:00.0", node=4, nodes={0: "0-71", 1: "72-143", 4: ""},
                       distance={4: [80, 40, 80, 80, 10]})
    cpus, how = bench.numa_cpus_for_gpu("0009:01:00.0", root)
    assert cpus == set(range(72, 144)) and "nearest" in how


def test_kernel_sources_and_traffic_digests(tmp_path, monkeypatch):
    """Every kernel named in the committed traffic file is found in its own source file, and counters whose
    recorded digest differs from the sources' are not used."""
    import os
    assert os.path.basename(bench.kernel_source("k_bw_light_reduce")) == "mt_backward.cu"
    assert os.path.basename(bench.kernel_source("k_claim")) == "mt_lookup.cu"
    assert bench.kernel_source("no_such_kernel") is None
    assert bench.source_digest("k_claim") != bench.source_digest("k_bw_light_reduce")
    # a traffic file with one current and one stale entry
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "kernel_traffic.txt").write_text(
        "# comment\n"
        f"k_bw_light_reduce 250.0 {bench.source_digest('k_bw_light_reduce')}\n"
        "k_gather 97.0 0000000000000000\n")
    src = tmp_path / "update_merged_table_gb300"
    src.symlink_to(os.path.join(bench.ROOT, "update_merged_table_gb300"))
    (tmp_path / "include").symlink_to(os.path.join(bench.ROOT, "include"))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.committed_traffic("k_bw_light_reduce") == (250.0, "profiles/kernel_traffic.txt")
    value, why = bench.committed_traffic("k_gather")
    assert value is None and "other sources" in why
    value, why = bench.committed_traffic("k_expand")
    assert value is None and "no counters" in why
