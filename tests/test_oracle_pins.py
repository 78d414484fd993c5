"""Pins for the fp64 oracle: each check compares it with something other than itself.

The oracle computes grouped-query softmax attention over a block-table page layout, split states and their exact
merge, and the compact worklist ("PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM Serving on
Commodity GPUs", gist.science technical summary, "Methodologie" 1). The pages print no worked example, so the pins
are: the exact fp16 widening (numpy), dense attention written with numpy/scipy on the gathered contiguous KV, a
pure-Python brute force, closed forms, invariances and hand-derived worklists.
"""

import math

import numpy as np
import pytest
from scipy.special import softmax

import oracle
from workloads import make_trace, normal_fp16, rng_for


def _random_problem(seed, lens, Hq=8, Hkv=2, d=128, ps=16, extra_pages=7):
    """Small paged problem with a shuffled pool; every page holds distinct fp16 N(0,1) data."""
    r = rng_for(seed, 99)
    lens = np.asarray(lens, dtype=np.int32)
    P = (lens.astype(np.int64) + ps - 1) // ps
    num_pages = int(P.sum()) + extra_pages
    max_pages = max(int(P.max()), 1)
    perm = r.permutation(num_pages)
    bt = np.full((len(lens), max_pages), -1, dtype=np.int32)
    nxt = 0
    for b, p in enumerate(P):
        bt[b, :p] = perm[nxt:nxt + p]
        nxt += p
    q = normal_fp16(r, (len(lens), Hq, d))
    k = normal_fp16(r, (num_pages, ps, Hkv, d))
    v = normal_fp16(r, (num_pages, ps, Hkv, d))
    return q, k, v, bt, lens


def _dense_numpy(q, k, v, bt, lens, scale):
    """Gather each row's KV into contiguous [L, d] arrays with numpy indexing, then softmax(Kq*scale) @ V."""
    B, Hq, d = q.shape
    ps, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Hq, d))
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        j = np.arange(L)
        phys = bt[b, j // ps]
        for hq in range(Hq):
            K = k[phys, j % ps, hq // G].astype(np.float64)
            V = v[phys, j % ps, hq // G].astype(np.float64)
            w = softmax(K @ q[b, hq].astype(np.float64) * scale)
            out[b, hq] = w @ V
    return out


def test_half_widening_exhaustive():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.half_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


@pytest.mark.parametrize("seed,lens,Hq,Hkv", [
    (0, [512], 32, 8),
    (1, [1, 15, 16, 17, 100], 8, 2),
    (2, [33, 0, 250], 4, 4),
    (3, [64, 70], 16, 1),
])
def test_matches_dense_numpy(seed, lens, Hq, Hkv):
    q, k, v, bt, lens = _random_problem(seed, lens, Hq=Hq, Hkv=Hkv)
    scale = 1.0 / math.sqrt(q.shape[2])
    ours = oracle.attention(q, k, v, bt, lens, scale)
    ref = _dense_numpy(q, k, v, bt, lens, scale)
    assert np.max(np.abs(ours - ref)) < 1e-12


def test_tiny_workload_matches_dense_numpy():
    tr = make_trace("tiny", 3)
    kp, vp = tr.host_pools()
    q, bt, sl = tr.q(0), tr.block_table(0), tr.seq_lens(0)
    ours = oracle.attention(q, kp, vp, bt, sl)
    ref = _dense_numpy(q, kp, vp, bt, sl, 1.0 / math.sqrt(128))
    assert np.max(np.abs(ours - ref)) < 1e-12


def test_brute_force_pure_python():
    # d = 4, page size 4, two rows, pure-Python loops over the block table
    for d, lens in ((4, [7, 13]), (128, [5, 9])):
        q, k, v, bt, lens = _random_problem(11 + d, lens, Hq=4, Hkv=2, d=d, ps=4)
        scale = 1.0 / math.sqrt(d)
        ours = oracle.attention(q, k, v, bt, lens, scale)
        for b in range(len(lens)):
            for hq in range(4):
                hkv = hq // 2
                s = []
                for j in range(int(lens[b])):
                    phys = int(bt[b][j // 4])
                    s.append(sum(float(q[b, hq, i]) * float(k[phys, j % 4, hkv, i]) for i in range(d)) * scale)
                mx = max(s)
                e = [math.exp(x - mx) for x in s]
                z = sum(e)
                for i in range(d):
                    ref = sum(e[j] * float(v[int(bt[b][j // 4]), j % 4, hkv, i]) for j in range(len(s))) / z
                    assert abs(ours[b, hq, i] - ref) < 1e-12


def test_closed_forms():
    q, k, v, bt, lens = _random_problem(5, [1, 40, 40, 40], Hq=8, Hkv=2)
    G = 4
    # L = 1: the output is v_0 exactly
    out = oracle.attention(q, k, v, bt, lens)
    for hq in range(8):
        assert np.array_equal(out[0, hq], v[bt[0, 0], 0, hq // G].astype(np.float64))
    # q = 0: uniform weights, output is the mean of the row's values
    q0 = q.copy()
    q0[1] = 0
    out = oracle.attention(q0, k, v, bt, lens)
    j = np.arange(40)
    for hq in range(8):
        mean = v[bt[1, j // 16], j % 16, hq // G].astype(np.float64).mean(axis=0)
        assert np.max(np.abs(out[1, hq] - mean)) < 1e-13
    # all keys equal: uniform weights again
    k2 = k.copy()
    for jj in range(40):
        k2[bt[2, jj // 16], jj % 16] = k[bt[2, 0], 0]
    out = oracle.attention(q, k2, v, bt, lens)
    for hq in range(8):
        mean = v[bt[2, j // 16], j % 16, hq // G].astype(np.float64).mean(axis=0)
        assert np.max(np.abs(out[2, hq] - mean)) < 1e-13
    # one key aligned with q and large: the output is that token's value
    k3 = k.copy()
    hot = 27
    for hkv in range(2):
        qd = q[3, hkv * G].astype(np.float64)
        k3[bt[3, hot // 16], hot % 16, hkv] = (40.0 * qd / np.linalg.norm(qd) * 11.3).astype(np.float16)
    out = oracle.attention(q, k3, v, bt, lens)
    for hkv in range(2):
        assert np.max(np.abs(out[3, hkv * G] - v[bt[3, hot // 16], hot % 16, hkv])) < 1e-9
    # all values one: the weights sum to one
    ones = np.ones_like(v)
    out = oracle.attention(q, k, ones, bt, lens)
    assert np.max(np.abs(out - 1.0)) < 1e-13


def test_page_permutation_invariance_bit_exact():
    q, k, v, bt, lens = _random_problem(7, [100, 17, 64], Hq=8, Hkv=2, extra_pages=20)
    ref = oracle.attention(q, k, v, bt, lens)
    r = rng_for(7, 1234)
    perm = r.permutation(k.shape[0])  # new physical id of old page i is perm[i]
    k2 = np.empty_like(k)
    v2 = np.empty_like(v)
    k2[perm] = k
    v2[perm] = v
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    out = oracle.attention(q, k2, v2, bt2, lens)
    assert np.array_equal(out, ref)


@pytest.mark.parametrize("chunk_pages", [1, 2, 3, 4, 8, 64])
def test_split_merge_invariance(chunk_pages):
    q, k, v, bt, lens = _random_problem(8, [1, 16, 17, 250, 513], Hq=8, Hkv=2)
    ref = oracle.attention(q, k, v, bt, lens)
    ps = 16
    for b in range(len(lens)):
        L = int(lens[b])
        P = -(-L // ps)
        S = -(-P // chunk_pages)
        ranges = [(s * chunk_pages * ps, min((s + 1) * chunk_pages * ps, L)) for s in range(S)]
        ranges += [(L, L)]  # a trailing empty split holds the neutral state
        for hq in (0, 5):
            m, l, acc = oracle.split_states(q, k, v, bt, lens, b, hq, ranges)
            assert m[-1] == -np.inf and l[-1] == 0 and not acc[-1].any()
            out = oracle.merge(m, l, acc)
            assert np.max(np.abs(out - ref[b, hq])) < 1e-12
            perm = rng_for(b, hq).permutation(len(ranges))
            out2 = oracle.merge(m[perm], l[perm], acc[perm])
            assert np.max(np.abs(out2 - ref[b, hq])) < 1e-12


def test_merge_closed_form_two_states():
    # two states with known (m, l, acc): the merge is sum exp(m_s - M) acc_s / sum exp(m_s - M) l_s
    m = np.array([0.5, 2.0])
    l = np.array([3.0, 1.5])
    acc = np.array([[1.0, -2.0], [4.0, 0.5]])
    w = np.exp(m - 2.0)
    ref = (w[:, None] * acc).sum(0) / (w * l).sum()
    assert np.max(np.abs(oracle.merge(m, l, acc) - ref)) < 1e-15
    assert not oracle.merge(np.array([-np.inf]), np.array([0.0]), np.zeros((1, 2))).any()


def test_worklist_hand_derived():
    # L = 1, 16, 17 tokens -> 1, 1, 2 pages
    got = oracle.worklist([1, 16, 17], 16, 2, 1)
    want = [(0, 0, 0, 0, 1), (0, 1, 0, 0, 1), (1, 0, 0, 0, 1), (1, 1, 0, 0, 1),
            (2, 0, 0, 0, 1), (2, 0, 1, 1, 2), (2, 1, 0, 0, 1), (2, 1, 1, 1, 2)]
    assert [tuple(t) for t in got] == want
    got = oracle.worklist([1, 16, 17], 16, 2, 2)
    want = [(0, 0, 0, 0, 1), (0, 1, 0, 0, 1), (1, 0, 0, 0, 1), (1, 1, 0, 0, 1), (2, 0, 0, 0, 2), (2, 1, 0, 0, 2)]
    assert [tuple(t) for t in got] == want
    # an empty row has no tasks; 33 tokens = 3 pages = splits [0,2) and [2,3)
    got = oracle.worklist([0, 33], 16, 1, 2)
    assert [tuple(t) for t in got] == [(1, 0, 0, 0, 2), (1, 0, 1, 2, 3)]
    assert len(oracle.worklist([0, 0], 16, 8, 4)) == 0


def test_worklist_count_closed_form():
    r = rng_for(0, 77)
    for c in (1, 3, 8, 32):
        lens = r.integers(0, 5000, size=37)
        n = len(oracle.worklist(lens, 16, 8, c))
        assert n == sum(8 * math.ceil(math.ceil(int(L) / 16) / c) for L in lens)


def test_worklist_tasks_tile_every_page_once():
    lens = np.array([1, 15, 16, 17, 31, 32, 33, 1000, 4097])
    for c in (1, 2, 5, 64):
        tasks = oracle.worklist(lens, 16, 3, c)
        for b, L in enumerate(lens):
            P = -(-int(L) // 16)
            for h in range(3):
                mine = tasks[(tasks[:, 0] == b) & (tasks[:, 1] == h)]
                covered = np.concatenate([np.arange(t[3], t[4]) for t in mine])
                assert np.array_equal(covered, np.arange(P))
                assert np.array_equal(mine[:, 2], np.arange(len(mine)))
                assert (mine[:, 4] - mine[:, 3] >= 1).all() and (mine[:, 4] - mine[:, 3] <= c).all()
