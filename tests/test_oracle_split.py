"""Pins of the oracle's leader/follower split (no GPU needed).

* resolving the leader layers only and gathering the followers from the recorded plan
  gives, step after step, exactly what the fused step gives (slot maps, row tables and
  every layer's pool), for several splits of the layer group;
* the plan is the step's misses: recomputed here from the hot set before the step (valid,
  non-resident, non-newest top-k tokens no slot holds, in top-k order), with the rows the
  step wrote for them;
* a leader-only resolve leaves the follower layers' rows untouched.
"""
import numpy as np
import pytest

from harness import OracleSim, device_pool_model, host_pools_for, poison_host_newest
from test_oracle_pins import small_workload


def _split_sim(wl):
    sim = OracleSim(wl, host_pools=host_pools_for(wl))
    plan = sim.orc.new_plan(wl.R)
    return sim, plan


def _resolve_split(sim, step, copy_layers, plan, gathers):
    wl = sim.wl
    err = sim.orc.resolve(wl.top_k_tokens(step), wl.seq_lens(step), wl.host_cache_locs, wl.device_buffer_locs,
                          sim.tokens, sim.stamps, sim.clock, wl.resident_pages, sim.out, sim.miss, sim.host,
                          sim.dev, copy_layers=copy_layers, plan=plan)
    for first, n in gathers:
        err |= sim.orc.gather(plan, wl.host_cache_locs, first, n, sim.host, sim.dev)
    return err


SPLITS = [(1, [(1, 2)]), (1, [(1, 1), (2, 1)]), (2, [(2, 1)]), (0, [(0, 3)])]


@pytest.mark.parametrize("copy_layers,gathers", SPLITS, ids=[f"leader{c}" for c, _ in SPLITS])
def test_split_equals_fused(copy_layers, gathers):
    wl = small_workload("indexshare_small", seed=4)
    assert wl.L == 3
    fused = OracleSim(wl, host_pools=host_pools_for(wl))
    split, plan = _split_sim(wl)
    for step in range(wl.steps):
        for sim in (fused, split):
            sim.write_newest(step)
            poison_host_newest(wl, step, sim.host)
        ef = fused.resolve(step)
        es = _resolve_split(split, step, copy_layers, plan, gathers)
        ef |= fused.backup(step)
        es |= split.backup(step)
        assert ef == es
        for name in ("out", "miss", "tokens", "stamps", "clock"):
            assert np.array_equal(getattr(fused, name), getattr(split, name)), f"step {step}: {name}"
        for layer in range(wl.L):
            assert np.array_equal(fused.dev[layer], split.dev[layer]), f"step {step}: layer {layer} pool"


@pytest.mark.parametrize("name", ["dsa_small", "mixed_small", "indexshare_small"])
def test_plan_is_the_steps_misses(name):
    wl = small_workload(name, seed=2)
    sim, plan = _split_sim(wl)
    checked = 0
    for step in range(wl.steps):
        sim.write_newest(step)
        hot = [set(sim.tokens[r][sim.tokens[r] >= 0].tolist()) for r in range(wl.R)]
        _resolve_split(sim, step, wl.L, plan, [])
        tk, S = wl.top_k_tokens(step), wl.seq_lens(step)
        assert np.array_equal(plan.count, sim.miss)
        for r in range(wl.R):
            if S[r] <= wl.H:
                assert plan.count[r] == 0
                continue
            seen, expect = set(), []
            for i, t in enumerate(tk[r]):
                t = int(t)
                if t < 0 or t >= S[r] or t in seen:
                    continue
                seen.add(t)
                if t == S[r] - 1:
                    continue
                if wl.resident_pages is not None and wl.resident_pages[r, t // wl.ps] >= 0:
                    continue
                if t not in hot[r]:
                    expect.append((t, int(sim.out[r, i])))
            m = int(plan.count[r])
            assert m == len(expect)
            got = list(zip(plan.tokens[r, :m].tolist(), plan.dst[r, :m].tolist()))
            assert got == expect, f"step {step} request {r}"
            checked += m
    assert checked > 0


def test_leader_only_leaves_followers():
    wl = small_workload("indexshare_small", seed=6)
    sim, plan = _split_sim(wl)
    for step in range(3):
        sim.write_newest(step)
        before = [p.copy() for p in sim.dev]
        _resolve_split(sim, step, 1, plan, [])
        B = wl.B
        moved = 0
        for r in range(wl.R):
            for j in range(int(plan.count[r])):
                d = int(plan.dst[r, j])
                if d < 0:
                    continue
                moved += 1
                for layer in range(1, wl.L):
                    assert np.array_equal(sim.dev[layer][d * B:(d + 1) * B], before[layer][d * B:(d + 1) * B])
                t = int(plan.tokens[r, j])
                assert np.array_equal(sim.dev[0][d * B:(d + 1) * B], wl.rows(0, r, [t])[0])
        assert moved > 0
        # then the followers, and every layer holds the token's bytes
        sim.orc.gather(plan, wl.host_cache_locs, 1, wl.L - 1, sim.host, sim.dev)
        for r in range(wl.R):
            for j in range(int(plan.count[r])):
                d, t = int(plan.dst[r, j]), int(plan.tokens[r, j])
                for layer in range(wl.L):
                    assert np.array_equal(sim.dev[layer][d * B:(d + 1) * B], wl.rows(layer, r, [t])[0])
