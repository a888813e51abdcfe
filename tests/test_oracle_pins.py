"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test names what the oracle is checked against: a hand-worked golden, a
closed form, brute force, or an independent library routine (numpy's Philox,
torch's bf16 rounding, torch.index_add_, torch.optim.Adam).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# Theorem 1 (MTGenRec): h_t = (h0 + t*S) mod 2^n covers all 2^n slots iff S is odd
# ---------------------------------------------------------------------------

def test_theorem1_golden_orbits():
    g = _golden("theorem1_orbits.json")
    for key, n in (("M8", 3), ("M16", 4)):
        M = 1 << n
        for S, want in zip(g[key]["S"], g[key]["distinct"]):
            sim = oracle.Simulator(n, S if S else M, max_probes=M)  # S = 0 is passed as M (== 0 mod M)
            seq = sim.sequence(5 % M, M)
            assert len(set(seq.tolist())) == want, (M, S)


@pytest.mark.parametrize("n", list(range(1, 13)))
def test_theorem1_brute_force(n):
    """Every S in [0, 2^n): the orbit is all of M exactly when S is odd; its size is M/gcd(S, M)."""
    M = 1 << n
    rng = np.random.default_rng(n)
    for S in range(M):
        sim = oracle.Simulator(n, S + M, max_probes=M)  # S + M: same residue, never rejected as zero
        h0 = int(rng.integers(0, M))
        seq = sim.sequence(h0, M)
        distinct = np.unique(seq).size
        assert distinct == M // math.gcd(S, M)
        assert (distinct == M) == (S % 2 == 1)
        assert seq[0] == h0


def test_theorem1_trivial_table():
    sim = oracle.Simulator(0, 1, max_probes=1)
    assert sim.sequence(0, 1).tolist() == [0]


def test_even_step_rejected():
    with pytest.raises(ValueError):
        oracle.Table(8, 4, probe_step=2)
    oracle.Table(8, 4, probe_step=3)


# ---------------------------------------------------------------------------
# Unique + inverse (first occurrence)
# ---------------------------------------------------------------------------

def test_unique_golden():
    g = _golden("unique_small.json")
    keys, valid = oracle.encode(g["ids"], g["feat_offsets"], g["table_ids"])
    assert valid.all()
    assert [hex(int(k)) for k in keys] == [hex(int(x, 16)) for x in g["keys"]]
    uniq, inv, cnt = oracle.unique(keys)
    assert [int(k) for k in uniq] == [int(x, 16) for x in g["unique"]]
    assert inv.tolist() == g["inverse"]
    assert cnt.tolist() == g["counts"]
    t = oracle.Table(6, 4)
    r = t.lookup(g["ids"], g["feat_offsets"], g["table_ids"])
    assert [int(k) for k in r["unique"]] == [int(x, 16) for x in g["unique"]]
    assert r["inverse"].tolist() == g["inverse"] and r["counts"].tolist() == g["counts"]


def _brute_unique(keys):
    uniq, inv = [], []
    for k in keys:
        if k not in uniq:
            uniq.append(k)
        inv.append(uniq.index(k))
    return uniq, inv


@pytest.mark.parametrize("seed", range(20))
def test_unique_vs_brute_force_and_sort(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(0, 200))
    keys = rng.integers(0, max(1, n // 3 + 1), size=n).astype(np.uint64) * np.uint64(0x0101010101)
    bu, bi = _brute_unique(keys.tolist())
    u1, i1, c1 = oracle.unique(keys)
    u2, i2, _ = oracle.unique(keys, method="sort")
    assert u1.tolist() == bu and i1.tolist() == bi
    assert u2.tolist() == bu and i2.tolist() == bi
    assert c1.tolist() == [bi.count(u) for u in range(len(bu))]


def test_unique_large_invariants():
    rng = np.random.default_rng(7)
    keys = rng.integers(0, 5000, size=100_000).astype(np.uint64)
    u, inv, cnt = oracle.unique(keys)
    u2, inv2, _ = oracle.unique(keys, method="sort")
    assert np.array_equal(u, u2) and np.array_equal(inv, inv2)
    assert np.array_equal(u[inv], keys)                      # uniq[inverse[i]] == key[i]
    assert np.unique(u).size == u.size                       # distinct
    first = np.array([np.argmax(keys == k) for k in u[:50]])
    assert np.all(np.diff(first) > 0)                        # first positions increase
    assert cnt.sum() == keys.size
    assert np.array_equal(cnt, np.bincount(inv, minlength=u.size))


def test_encode_rejects_out_of_range():
    ids = [0, -1, (1 << 56) - 1, 1 << 56, 5]
    keys, valid = oracle.encode(ids, [0, 3, 5], [7, 255])
    assert valid.tolist() == [True, False, True, False, False]
    assert int(keys[0]) == 7 << 56
    assert int(keys[2]) == (7 << 56) | ((1 << 56) - 1)
    t = oracle.Table(6, 4)
    r = t.lookup(ids, [0, 3, 5], [7, 255])
    assert r["inverse"].tolist()[1] == -1 and t.error == -4
    assert np.all(r["rows"][1] == 0)


# ---------------------------------------------------------------------------
# Row initialisation: Philox4x64-10 pinned to numpy.random.Philox
# ---------------------------------------------------------------------------

def _numpy_philox_block(ctr, key):
    """Philox4x64-10 block at counter `ctr` from numpy's independent implementation.

    numpy's bit generator adds one to its 256-bit counter (with carry) before
    each block, so it is started one below `ctr`.
    """
    c = [int(x) for x in ctr]
    for i in range(4):          # c - 1 with borrow
        if c[i]:
            c[i] -= 1
            break
        c[i] = 2**64 - 1
    bg = np.random.Philox(key=np.array(key, dtype=np.uint64), counter=np.array(c, dtype=np.uint64))
    return bg.random_raw(4)


def test_philox_matches_numpy():
    rng = np.random.default_rng(11)
    for _ in range(200):
        ctr = [int(x) for x in rng.integers(1, 2**63, size=4, dtype=np.uint64)]
        key = [int(x) for x in rng.integers(0, 2**63, size=2, dtype=np.uint64)]
        want = _numpy_philox_block(ctr, key)
        got = oracle.philox4x64_10(ctr, key)
        assert np.array_equal(got, want)


def test_init_row_from_numpy_philox():
    rng = np.random.default_rng(3)
    for dim, dtype in ((16, oracle.F32), (24, oracle.F32), (64, oracle.BF16)):
        scale = oracle.default_init_scale(dim)
        for key in [0, 1, 0x0300000000012345, int(rng.integers(0, 2**56))]:
            seed = int(rng.integers(0, 2**63))
            want = np.zeros(dim, np.float32)
            for j in range(dim):
                w = int(_numpy_philox_block([j // 8, 0, 0, 0], [key, seed])[(j // 2) % 4])
                q = (w >> 40) if j % 2 == 0 else ((w >> 16) & 0xFFFFFF)
                unit = np.float32((2 * q - (1 << 24)) / float(1 << 24))
                want[j] = np.float32(unit * np.float32(scale))
            if dtype == oracle.BF16:
                want = torch.from_numpy(want).to(torch.bfloat16).float().numpy()
            got = oracle.init_row(key, seed, scale, dim, dtype)
            assert np.array_equal(got, want), (dim, key)


def test_init_uniformity():
    """Initial values are uniform on [-scale, scale): chi-square over 16 bins."""
    dim = 64
    scale = oracle.default_init_scale(dim)
    vals = np.concatenate([oracle.init_row(k, 99, scale, dim) for k in range(2000)]) / scale
    assert vals.min() >= -1.0 and vals.max() < 1.0
    hist, _ = np.histogram(vals, bins=16, range=(-1, 1))
    exp = vals.size / 16
    chi2 = ((hist - exp) ** 2 / exp).sum()
    assert chi2 < 40.0  # 15 dof, p ~ 5e-4


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32),
                        (rng.integers(0, 2**16, 2000).astype(np.uint32) << 16 | 0x8000).view(np.float32),
                        np.array([0.0, -0.0, 1.0, 3.0e38, -1e-40], np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([oracle.bf16_bits(float(v)) for v in x], np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], want[~nan])
    # NaN payloads differ between implementations; both must stay NaN
    assert np.all((got[nan] & 0x7F80) == 0x7F80) and np.all((got[nan] & 0x7F) != 0)


# ---------------------------------------------------------------------------
# Gradient reduction and Adam
# ---------------------------------------------------------------------------

def _lookup_batch(t, ids):
    return t.lookup(np.asarray(ids, np.int64))


def test_gsum_matches_index_add():
    rng = np.random.default_rng(1)
    ids = rng.integers(0, 300, size=5000)
    t = oracle.Table(12, 16)
    r = _lookup_batch(t, ids)
    g = rng.standard_normal((ids.size, 16)).astype(np.float32)
    gsum = t.backward_adam(g, want_gsum=True)
    ref = torch.zeros(r["U"], 16, dtype=torch.float64)
    ref.index_add_(0, torch.from_numpy(r["inverse"].astype(np.int64)), torch.from_numpy(g).double())
    assert np.array_equal(gsum, ref.float().numpy())


def test_gsum_bf16_grads():
    rng = np.random.default_rng(2)
    ids = rng.integers(0, 50, size=800)
    t = oracle.Table(10, 8, row_dtype=oracle.BF16)
    r = _lookup_batch(t, ids)
    gb = torch.from_numpy(rng.standard_normal((ids.size, 8)).astype(np.float32)).to(torch.bfloat16)
    gsum = t.backward_adam(gb.view(torch.int16).numpy().view(np.uint16), grad_dtype=oracle.BF16, want_gsum=True)
    ref = torch.zeros(r["U"], 8, dtype=torch.float64)
    ref.index_add_(0, torch.from_numpy(r["inverse"].astype(np.int64)), gb.double())
    assert np.array_equal(gsum, ref.float().numpy())


def test_adam_golden_t1():
    g = _golden("adam_t1.json")
    for c in g["cases"]:
        t = oracle.Table(4, 4)
        key = 1
        t.lookup([key])
        e0 = t.get_row(key)[0]
        # shift so the row's first element starts at w0: apply the step to a known row by
        # comparing deltas (w1 - w0 is what the closed form fixes)
        grads = np.zeros((1, 4), np.float32)
        grads[0, 0] = c["g"]
        t.backward_adam(grads, lr=g["lr"], beta1=g["beta1"], beta2=g["beta2"], eps=g["eps"])
        e1, m1, v1 = t.get_row(key)
        want_delta = c["w1"] - c["w0"]
        assert abs((float(e1[0]) - float(e0[0])) - want_delta) <= 1e-6 + 1e-5 * abs(want_delta)
        assert abs(m1[0] - c["m1"]) <= 1e-5 * abs(c["m1"]) + 1e-30
        assert abs(v1[0] - c["v1"]) <= 1e-5 * abs(c["v1"]) + 1e-30
        assert np.array_equal(e1[1:], e0[1:])  # zero gradient, zero moments: no move


def test_adam_closed_form_t1():
    """At t = 1 from m = v = 0: w1 = w0 - lr * g / (|g| + eps), evaluated in float64."""
    rng = np.random.default_rng(4)
    ids = rng.integers(0, 100, size=2000)
    t = oracle.Table(10, 16)
    r = _lookup_batch(t, ids)
    w0 = np.stack([t.get_row(k)[0] for k in r["unique"]]).astype(np.float64)
    g = rng.standard_normal((ids.size, 16)).astype(np.float32)
    gsum = t.backward_adam(g, want_gsum=True).astype(np.float64)
    w1 = np.stack([t.get_row(k)[0] for k in r["unique"]]).astype(np.float64)
    want = w0 - 1e-3 * gsum / (np.abs(gsum) + 1e-8)
    np.testing.assert_allclose(w1, want, rtol=1e-5, atol=1e-6)


def test_adam_matches_torch_optim_over_steps():
    rng = np.random.default_rng(6)
    ids = rng.integers(0, 40, size=400)
    dim = 8
    t = oracle.Table(8, dim)
    r = _lookup_batch(t, ids)
    W = torch.tensor(np.stack([t.get_row(k)[0] for k in r["unique"]]), dtype=torch.float64, requires_grad=True)
    opt = torch.optim.Adam([W], lr=1e-3, betas=(0.9, 0.999), eps=1e-8, foreach=False)
    for step in range(5):
        if step:
            _lookup_batch(t, ids)
        g = rng.standard_normal((ids.size, dim)).astype(np.float32)
        gsum = t.backward_adam(g, want_gsum=True)
        W.grad = torch.from_numpy(gsum.astype(np.float64))
        opt.step()
    got = np.stack([t.get_row(k)[0] for k in r["unique"]])
    np.testing.assert_allclose(got, W.detach().numpy(), rtol=1e-5, atol=1e-6)
    assert t.step == 5


def test_adam_lazy_rows_and_global_step():
    """Rows absent from a batch are not moved; the step counter advances once per call."""
    t = oracle.Table(8, 4)
    t.lookup([1, 2])
    t.backward_adam(np.ones((2, 4), np.float32))
    row2 = t.get_row(2)[0].copy()
    t.lookup([1])
    t.backward_adam(np.ones((1, 4), np.float32))
    e2, m2, _ = t.get_row(2)
    assert np.array_equal(e2, row2)
    np.testing.assert_allclose(m2, 0.1, rtol=1e-6)          # one update
    _, m1, _ = t.get_row(1)
    np.testing.assert_allclose(m1, 0.9 * 0.1 + 0.1, rtol=1e-6)  # two updates
    assert t.step == 2


# ---------------------------------------------------------------------------
# Table: presence against a dict under random insert/erase scripts
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(5))
def test_table_presence_script(seed):
    rng = np.random.default_rng(seed)
    t = oracle.Table(10, 4, simulate=True, probe_step=int(rng.integers(0, 512)) * 2 + 1)
    ref = set()
    for _ in range(40):
        ids = rng.integers(0, 300, size=int(rng.integers(1, 60)))
        r = t.lookup(ids, insert_missing=bool(rng.integers(0, 2)) or len(ref) == 0)
        if r["present"].all():
            ref.update(int(k) for k in r["unique"])
        else:
            for k, p in zip(r["unique"], r["present"]):
                assert p == (int(k) in ref)
        er = rng.integers(0, 300, size=int(rng.integers(0, 30))).astype(np.uint64)
        found = t.erase(er)
        for k, f in zip(er, found):
            assert f == (int(k) in ref) or int(k) in set(int(x) for x in er[: list(er).index(k)])
        for k in er:
            ref.discard(int(k))
        assert t.live == len(ref)
        assert set(int(k) for k in t.live_keys()) == ref
        st = t.sim_stats()
        assert st["live"] == len(ref)
        assert t.error == 0


def test_erase_duplicates_all_report_found():
    t = oracle.Table(8, 4)
    t.lookup([5, 6])
    assert t.erase(np.array([5, 5, 7, 6], np.uint64)).tolist() == [True, True, False, True]
    assert t.live == 0


def test_reinsert_after_erase_restarts_from_init():
    t = oracle.Table(8, 4, init_seed=9)
    t.lookup([5])
    e0 = t.get_row(5)[0].copy()
    t.backward_adam(np.ones((1, 4), np.float32))
    assert not np.array_equal(t.get_row(5)[0], e0)
    t.erase(np.array([5], np.uint64))
    r = t.lookup([5])
    assert np.array_equal(r["rows"][0], e0)
    assert np.all(t.get_row(5)[1] == 0)


def test_row_pool_exhaustion_latches_full():
    t = oracle.Table(8, 4, num_rows=3)
    r = t.lookup([1, 2, 3, 4, 5])
    assert r["present"].tolist() == [True, True, True, False, False]
    assert t.error == -3
    assert np.all(r["rows"][3:] == 0)


# ---------------------------------------------------------------------------
# Shadow simulator: linear probing after relabelling slots by S^-1
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("S", [1, 3, 0x9E3779B97F4A7C15 % 4096 | 1])
def test_insert_only_occupancy_is_order_independent(S):
    """Insert-only probing with a fixed odd S is linear probing on relabelled slots, so the set of
    occupied slots and the total displacement do not depend on the insertion order."""
    rng = np.random.default_rng(S)
    n = 12
    keys = rng.choice(2**40, size=int(0.8 * (1 << n)), replace=False)
    base = None
    for trial in range(4):
        sim = oracle.Simulator(n, S, hash_seed=17)
        for k in rng.permutation(keys):
            assert sim.insert(int(k)) == 0
        occ, D = sim.occupancy()
        if base is None:
            base = (occ, D)
        else:
            assert np.array_equal(occ, base[0]) and D == base[1]


def test_probe_index_relation():
    """slot(key) = (h0 + t*S) mod M for the recorded probe index t, so t = (slot - h0) * S^-1 mod M."""
    n, S, seed = 10, 77, 5
    M = 1 << n
    sim = oracle.Simulator(n, S, hash_seed=seed)
    rng = np.random.default_rng(0)
    keys = rng.choice(2**50, size=700, replace=False)
    for k in keys:
        sim.insert(int(k))
    Sinv = pow(S, -1, M)
    for k in keys[:200]:
        s = sim.find(int(k))
        t = sim.placed(int(k))
        h0 = oracle.home_slot(int(k), seed, n)
        assert s == (h0 + t * S) % M
        assert t == ((s - h0) * Sinv) % M


def test_tombstone_reuse_and_chain():
    """An erased key leaves a tombstone that find passes over and insert reuses."""
    n = 4
    sim = oracle.Simulator(n, 1, hash_seed=0)
    # collect keys with the same home slot
    h = {}
    for k in range(5000):
        h.setdefault(oracle.home_slot(k, 0, n), []).append(k)
    a, b, c = next(v for v in h.values() if len(v) >= 3)[:3]
    for k in (a, b, c):
        sim.insert(k)
    assert sim.placed(a) == 0 and sim.placed(b) == 1 and sim.placed(c) == 2
    sim.erase(b)
    assert sim.find(c) >= 0          # passes over the tombstone
    d = next(k for k in h[oracle.home_slot(a, 0, n)] if k not in (a, b, c))
    sim.insert(d)
    assert sim.placed(d) == 1        # reuses it
    occ, _ = sim.occupancy()
    assert (occ == 2).sum() == 0


# ---------------------------------------------------------------------------
# Adam: the folded form against the textbook form over many steps
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("row_dtype", [oracle.F32, oracle.BF16])
def test_adam_folded_form_matches_textbook_form(row_dtype):
    """The oracle applies w -= step_size * m / (sqrt(v) * inv_sqrt_bc2 + eps) with the bias corrections folded
    into per-step scalars and beta powers kept as running products.  Kingma & Ba's textbook form,
    m_hat = m / (1 - b1^t), v_hat = v / (1 - b2^t), w -= lr * m_hat / (sqrt(v_hat) + eps), written here in
    float32 numpy with pow() for the beta powers, must agree over 30 steps: fp32 rows to 1e-5 relative,
    bf16 rows (stored rounded each step, as the table does) to one bf16 ulp."""
    from numerics import bf16_ulp_distance
    rng = np.random.default_rng(12)
    dim, keys = 16, np.arange(20, dtype=np.int64)
    t = oracle.Table(8, dim, row_dtype=row_dtype)
    t.lookup(keys)
    w = np.stack([t.get_row(int(k))[0] for k in keys]).astype(np.float32)
    m = np.zeros_like(w)
    v = np.zeros_like(w)
    lr, b1, b2, eps = np.float32(1e-3), np.float32(0.9), np.float32(0.999), np.float32(1e-8)
    for step in range(1, 31):
        t.lookup(keys)
        g = rng.standard_normal((keys.size, dim)).astype(np.float32)
        t.backward_adam(g)
        m = b1 * m + (np.float32(1) - b1) * g
        v = b2 * v + (np.float32(1) - b2) * g * g
        m_hat = m / np.float32(1.0 - 0.9 ** step)
        v_hat = v / np.float32(1.0 - 0.999 ** step)
        w = w - lr * m_hat / (np.sqrt(v_hat) + eps)
        if row_dtype == oracle.BF16:
            w = torch.from_numpy(w).to(torch.bfloat16).float().numpy()
    got = np.stack([t.get_row(int(k))[0] for k in keys])
    if row_dtype == oracle.BF16:
        assert bf16_ulp_distance(got, w).max() <= 1
    else:
        np.testing.assert_allclose(got, w, rtol=1e-5, atol=1e-6)


# ---------------------------------------------------------------------------
# Pooled bags
# ---------------------------------------------------------------------------

def _pool_case(seed, dim=8, n=3000, vocab=400):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, vocab, size=n)
    cuts = np.sort(rng.choice(np.arange(1, n), size=40, replace=False))
    bo = np.concatenate([[0], cuts, [n]]).astype(np.int64)
    bo = np.insert(bo, 5, bo[5])  # an empty bag
    t = oracle.Table(12, dim)
    r = t.lookup(ids)
    return t, r, bo, rng


@pytest.mark.parametrize("mode", [0, 1])
def test_pool_forward_matches_numpy_segment_sum(mode):
    """Sum (mode 0) and mean (mode 1) of each bag's gathered rows, against numpy's reduceat in float64."""
    t, r, bo, _ = _pool_case(3)  # bags cover every position, one of them is empty
    got = t.pool_forward(bo, mode)
    lens = np.diff(bo)
    full = lens > 0
    seg = np.add.reduceat(r["rows"].astype(np.float64), bo[:-1][full], axis=0)  # contiguous bags up to n
    if mode == 1:
        seg = seg / lens[full][:, None]
    assert np.array_equal(got[full], seg.astype(np.float32))
    assert not got[~full].any()


def test_pool_forward_partial_cover_and_bad_offsets():
    t, r, _, _ = _pool_case(4)
    bo = np.array([100, 100, 300, 301], np.int64)  # positions before 100 and from 301 on are in no bag
    got = t.pool_forward(bo)
    assert not got[0].any()
    assert np.array_equal(got[1], r["rows"][100:300].astype(np.float64).sum(0).astype(np.float32))
    assert np.array_equal(got[2], r["rows"][300])
    with pytest.raises(ValueError):
        t.pool_forward(np.array([0, 20, 10], np.int64))
    with pytest.raises(ValueError):
        t.pool_forward(np.array([0, 5000], np.int64))


@pytest.mark.parametrize("mode", [0, 1])
def test_pool_backward_equals_expanded_backward(mode):
    """The pooled backward equals the plain backward fed the bag gradient at every position of the bag (times
    fp32(1/len) for the mean); its gradient sums equal torch's index_add_ of those expanded rows."""
    t1, r, bo, rng = _pool_case(5, dim=8)
    t2, _, _, _ = _pool_case(5, dim=8)
    B = bo.size - 1
    dp = rng.standard_normal((B, 8)).astype(np.float32)
    gs1 = t1.backward_adam_pooled(bo, dp, mode=mode, want_gsum=True)
    lens = np.diff(bo)
    scale = np.where(lens > 0, np.float32(1) / np.maximum(lens, 1).astype(np.float32), np.float32(1))
    per_bag = dp * scale[:, None] if mode == 1 else dp
    expanded = np.repeat(per_bag.astype(np.float32), lens, axis=0)
    gs2 = t2.backward_adam(expanded, want_gsum=True)
    assert np.array_equal(gs1, gs2)
    ref = torch.zeros(r["U"], 8, dtype=torch.float64)
    ref.index_add_(0, torch.from_numpy(r["inverse"].astype(np.int64)), torch.from_numpy(expanded).double())
    assert np.array_equal(gs1, ref.float().numpy())
    for k in r["unique"][:50]:
        a, b_ = t1.get_row(int(k)), t2.get_row(int(k))
        assert all(np.array_equal(x, y) for x, y in zip(a, b_))


def test_reciprocal_of_bag_length_is_correctly_rounded():
    """The mean's scale fp32(1/len), taken from the double quotient, equals IEEE's correctly rounded fp32
    division 1/len for every length up to 10^5 (no double-rounding case), so the CUDA side may use the
    correctly rounded fp32 reciprocal."""
    lens = np.arange(1, 100_001, dtype=np.float64)
    via_double = (1.0 / lens).astype(np.float32)
    direct = np.float32(1) / lens.astype(np.float32)
    assert np.array_equal(via_double, direct)
