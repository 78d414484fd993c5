"""The seeded input generators: determinism, shapes, distributions and the page-allocation rule."""

import numpy as np
import pytest

from workloads import CONFIGS, make_trace, normal_fp16, rng_for, zipf_lengths


def test_normal_fp16_moments_and_determinism():
    a = normal_fp16(rng_for(1, 2), (1 << 20,))
    b = normal_fp16(rng_for(1, 2), (1 << 20,))
    assert a.dtype == np.float16 and np.array_equal(a.view(np.uint16), b.view(np.uint16))
    x = a.astype(np.float64)
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1.0) < 5e-3
    assert np.isfinite(x).all() and np.abs(x).max() < 4.5


def test_zipf_truncated():
    k = zipf_lengths(rng_for(0, 1), 200000) // 256
    assert k.min() >= 1 and k.max() <= 128
    p = np.arange(1, 129, dtype=np.float64) ** -1.1
    p /= p.sum()
    assert abs((k == 1).mean() - p[0]) < 0.01
    assert abs(k.mean() - (np.arange(1, 129) * p).sum()) < 0.3


@pytest.mark.parametrize("name", ["tiny", "b1_bucketed", "b8_bimodal", "b8_uniform", "b8_zipf", "b4_bimodal"])
def test_trace_structure(name):
    for seed in (0, 5):
        tr = make_trace(name, seed)
        cfg = CONFIGS[name]
        assert tr.batch == cfg.batch and tr.steps == cfg.steps
        s0 = tr.seq_lens(0)
        if name == "tiny":
            assert list(s0) == [512] and tr.num_pages == 64
        if name == "b1_bucketed":
            assert int(s0[0]) in (4096, 8192, 16384, 32768)
        if name in ("b8_bimodal", "b4_bimodal"):
            h = tr.batch // 2
            assert ((256 <= s0[:h]) & (s0[:h] <= 1024)).all()
            assert ((16384 <= s0[h:]) & (s0[h:] <= 32768)).all()
        if name == "b8_uniform":
            assert ((1024 <= s0) & (s0 <= 32768)).all()
        if name == "b8_zipf":
            assert (s0 % 256 == 0).all() and ((256 <= s0) & (s0 <= 32768)).all()
        # pages are distinct, inside the pool, and exactly cover every row at every step
        assert len(np.unique(tr.used_pages)) == len(tr.used_pages)
        assert tr.used_pages.min() >= 0 and tr.used_pages.max() < tr.num_pages
        for t in (0, tr.steps - 1):
            bt = tr.block_table(t)
            P = tr.pages(t)
            for b in range(tr.batch):
                assert (bt[b, :P[b]] >= 0).all() and (bt[b, P[b]:] == -1).all()
        # a new page appears exactly when a row's newest token opens one
        for t in range(1, tr.steps):
            opened = tr.pages(t) - tr.pages(t - 1)
            assert np.array_equal(opened, ((tr.seq_lens(t) - 1) % 16 == 0).astype(int))


def test_stress_lengths():
    tr = make_trace("stress", 0, steps=1)
    L = tr.seq_lens(0)
    assert tr.batch == 64 and L.min() >= 512 and L.max() <= 131072
    assert tr.num_pages == min(1 << 20, int(np.ceil(1.25 * tr.pages(0).sum())))


def test_valid_slots_match_lengths():
    tr = make_trace("b8_zipf", 3, steps=20)
    for t in (0, 7, 19):
        vs = tr.valid_slots(t)
        for b in range(tr.batch):
            assert vs[tr.page_row == b].sum() == tr.seq_lens(t)[b]
