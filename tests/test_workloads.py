"""The seeded input generator produces what the workload recipes state (no GPU)."""
import numpy as np
import pytest

import workloads as W


def _check_common(wl, steps):
    for s in range(steps):
        tk = wl.top_k_tokens(s)
        S = wl.seq_lens(s)
        for r in range(wl.R):
            v = tk[r][tk[r] >= 0]
            assert len(np.unique(v)) == len(v), "duplicate token in a top-k row"
            assert np.all(v < S[r])
            assert len(v) == min(wl.K, int(S[r]))
    hcl = wl.host_cache_locs
    valid = hcl[hcl >= 0]
    assert len(np.unique(valid)) == len(valid) and valid.max() < wl.host_rows
    for r in range(wl.R):
        assert np.all(hcl[r, : wl.seq_max[r]] >= 0)
    dbl = wl.device_buffer_locs
    assert len(np.unique(dbl)) == dbl.size and dbl.max() < wl.device_rows


def test_deterministic():
    a, b = W.make("tiny", seed=3), W.make("tiny", seed=3)
    for s in range(4):
        assert np.array_equal(a.top_k_tokens(s), b.top_k_tokens(s))
    assert np.array_equal(a.rows(0, 1, [5, 6]), b.rows(0, 1, [5, 6]))
    c = W.make("tiny", seed=4)
    assert not np.array_equal(a.top_k_tokens(1), c.top_k_tokens(1))
    # rows differ by layer, request and token
    r = a.rows(0, 0, [1, 2])
    assert not np.array_equal(r[0], r[1])
    assert not np.array_equal(a.rows(0, 0, [1]), a.rows(0, 1, [1]))


def test_tiny_recipe():
    wl = W.make("tiny")
    _check_common(wl, wl.steps)
    for s in range(1, wl.steps):
        prev, cur = wl.top_k_tokens(s - 1), wl.top_k_tokens(s)
        S = wl.seq_lens(s)
        for r in range(wl.R):
            assert S[r] - 1 in cur[r]
            reused = len(set(cur[r].tolist()) & set(prev[r].tolist()) - {-1})
            assert reused >= int(np.floor(0.7 * wl.K))


def test_dsa_recipe_small():
    wl = W.make("dsa", requests=2, steps=3)
    _check_common(wl, 3)
    for s in range(3):
        S = wl.seq_lens(s)
        for r in range(wl.R):
            assert set(range(S[r] - 64, S[r])) <= set(wl.top_k_tokens(s)[r].tolist())
    prev, cur = wl.top_k_tokens(1), wl.top_k_tokens(2)
    assert len(set(cur[0].tolist()) & set(prev[0].tolist())) >= 1843


def test_mixed_recipe_small():
    wl = W.make("mixed1m", requests=2, steps=2, seq0=(40000, 40000))
    _check_common(wl, 2)
    for s in range(2):
        tk = wl.top_k_tokens(s)
        for r in range(wl.R):
            res = [t for t in tk[r] if t >= 0 and wl.resident_row(r, t) >= 0]
            assert len(res) == int(np.floor(0.2 * wl.K))
    # resident rows lie beyond the hot region and never collide
    rp = wl.resident_pages
    pages = rp[rp >= 0]
    assert len(np.unique(pages)) == len(pages)
    assert pages.min() * wl.ps >= wl.R * (wl.H + 1)
    assert (pages.max() + 1) * wl.ps <= wl.device_rows


def test_indexshare_seq_lengths():
    wl = W.make("indexshare", requests=8, steps=1)
    assert np.all(wl.seq0 >= 32768) and np.all(wl.seq0 <= 65536)
    _check_common(wl, 1)


@pytest.mark.parametrize("h,f", [(2048, 0.5), (6144, 0.99)])
def test_sweep_points(h, f):
    wl = W.make(f"sweep_h{h}_f{f}", requests=2, steps=2)
    assert wl.H == h and wl.cfg.reuse == f and wl.B == 1152
    _check_common(wl, 2)


def test_pool_fill_matches_rows():
    wl = W.make("tiny")
    pool = np.zeros(wl.host_rows * wl.B, dtype=np.uint8)
    wl.fill_host_pool(0, pool, 2)
    for r, t in [(0, 0), (0, 8000), (1, 50)]:
        h = wl.host_cache_locs[r, t]
        assert np.array_equal(pool[h * wl.B:(h + 1) * wl.B], wl.rows(0, r, [t])[0])
