"""Pins of the oracle's hot-slot invalidation (no GPU needed).

* a hand-worked example (tests/golden/invalidate_h6.json),
* the two formulations agree: clearing the host rows of a token set equals clearing
  the tokens, when every (request, token) has its own host row,
* after an invalidation the next resolve misses exactly on the cleared tokens it looks
  up, and copies their current rows (the resolve's own invariants hold).
"""
import json
import os

import numpy as np
import pytest

import oracle
from harness import OracleSim
from test_oracle_pins import small_workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_invalidate_golden():
    g = json.load(open(os.path.join(GOLDEN, "invalidate_h6.json")))
    H, MC = g["hot_slots"], g["max_context"]
    orc = oracle.Oracle(4, H, 8, 1, MC, 2 * MC + 2, 64)
    hcl = (2 * np.arange(MC, dtype=np.int32) + 1).reshape(1, MC)
    for c in g["cases"]:
        tok = np.array([g["tokens"]], dtype=np.int32)
        st = np.array([g["stamps"]], dtype=np.int32)
        S = np.array([c["seq_len"]], dtype=np.int32)
        if c["kind"] == "tokens":
            clear = np.array(c["clear"], dtype=np.int32)
            err = orc.invalidate_tokens(S, np.array([0, clear.size], dtype=np.int32), clear, tok, st)
        else:
            err = orc.invalidate_host_rows(S, hcl, np.array(c["rows"], dtype=np.int32), tok, st)
        assert tok[0].tolist() == c["tokens"], c["why"]
        assert st[0].tolist() == c["stamps"], c["why"]
        assert err == c["err"], c["why"]


def _warm_sim(name, steps=6, seed=3):
    wl = small_workload(name, seed)
    sim = OracleSim(wl)
    for s in range(steps):
        sim.step(s)
    return wl, sim


def _pick(rng, wl, sim, frac=0.3):
    """Per request, a random subset of the held tokens plus some tokens no slot holds."""
    offs, toks = [0], []
    for r in range(wl.R):
        held = sim.tokens[r][sim.tokens[r] >= 0]
        k = int(frac * held.size)
        pick = list(rng.choice(held, size=k, replace=False)) if k else []
        pick += list(rng.integers(0, wl.max_context, size=3))
        toks += pick
        offs.append(len(toks))
    return np.array(offs, dtype=np.int32), np.array(toks, dtype=np.int32)


FORMS = ["tiny", "dsa_small", "mixed_small", "indexshare_small"]


@pytest.mark.parametrize("name", FORMS)
def test_token_and_host_row_forms_agree(name):
    wl, sim = _warm_sim(name)
    rng = np.random.default_rng(11)
    offs, toks = _pick(rng, wl, sim)
    S = wl.seq_lens(6)
    a_tok, a_st = sim.tokens.copy(), sim.stamps.copy()
    ea = sim.orc.invalidate_tokens(S, offs, toks, a_tok, a_st)
    rows = []
    for r in range(wl.R):
        for t in toks[offs[r]:offs[r + 1]]:
            if 0 <= t < S[r] - 1:
                rows.append(wl.host_cache_locs[r, t])
    rows = np.unique(np.array(rows, dtype=np.int32))
    # every (request, token) owns its host row, so the row set names exactly those tokens
    assert np.unique(wl.host_cache_locs[wl.host_cache_locs >= 0]).size == int((wl.host_cache_locs >= 0).sum())
    b_tok, b_st = sim.tokens.copy(), sim.stamps.copy()
    eb = sim.orc.invalidate_host_rows(S, wl.host_cache_locs, rows, b_tok, b_st)
    assert ea == eb
    assert np.array_equal(a_tok, b_tok) and np.array_equal(a_st, b_st)


@pytest.mark.parametrize("name", FORMS)
def test_next_resolve_refetches_cleared_tokens(name):
    wl, sim = _warm_sim(name)
    rng = np.random.default_rng(5)
    offs, toks = _pick(rng, wl, sim, frac=0.5)
    step = 6
    S = wl.seq_lens(step)
    before = sim.tokens.copy()
    sim.orc.invalidate_tokens(S, offs, toks, sim.tokens, sim.stamps)
    cleared = [set(before[r][(before[r] >= 0) & (sim.tokens[r] < 0)].tolist()) for r in range(wl.R)]
    # the step looks up some cleared tokens: they must miss and come back with their bytes
    tk = wl.top_k_tokens(step).copy()
    for r in range(wl.R):
        c = sorted(cleared[r])[:4]
        if c and S[r] > wl.H:
            keep = [t for t in tk[r] if t not in c][: wl.K - len(c)]
            tk[r, :len(keep) + len(c)] = np.array(keep + c, dtype=np.int32)
    hot = [set(sim.tokens[r][sim.tokens[r] >= 0].tolist()) for r in range(wl.R)]
    sim.write_newest(step)
    sim.resolve(step, top_k=tk)
    checked = 0
    for r in range(wl.R):
        if S[r] <= wl.H:
            continue
        res = set()
        if wl.resident_pages is not None:
            res = {int(t) for t in tk[r] if t >= 0 and wl.resident_pages[r, t // wl.ps] >= 0}
        look = {int(t) for t in tk[r] if 0 <= t < S[r] - 1} - res
        assert int(sim.miss[r]) == len(look - hot[r])
        for i, t in enumerate(tk[r]):
            if int(t) in cleared[r] and int(t) in look:
                row = int(sim.out[r, i])
                assert row >= 0
                checked += 1
                for layer in range(wl.L):
                    assert np.array_equal(sim.dev_row(layer, row), wl.rows(layer, r, [int(t)])[0])
    assert checked > 0, "no cleared token was looked up: the case proves nothing"
