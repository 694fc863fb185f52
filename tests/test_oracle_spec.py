"""Pins of the oracle's speculative batches (no GPU needed).

* a hand-worked batch sequence (tests/golden/spec_h3_k1_q2.json),
* a one-query batch is a plain decode step (resolve and backup, step after step),
* replayable plans: with H >= (Q + 1) * K no verify step overwrites a row an earlier step
  of the same batch resolved, so every step's rows still hold their tokens' bytes when the
  batch ends -- and with a smaller buffer the same check finds an overwrite,
* the speculative backup makes the accepted positions' host rows exact.
"""
import json
import os

import numpy as np
import pytest

import oracle
import workloads as W
from harness import OracleSim, device_pool_model, host_pools_for, poison_host_newest
from test_oracle_pins import small_workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_spec_golden():
    g = json.load(open(os.path.join(GOLDEN, "spec_h3_k1_q2.json")))
    H, K, Q = g["hot_slots"], g["top_k"], g["num_queries"]
    MC = 32
    orc = oracle.Oracle(K, H, 8, 1, MC, MC, 64)
    dbl = np.array([g["device_buffer_locs"]], dtype=np.int32)
    hcl = np.arange(MC, dtype=np.int32).reshape(1, MC)
    host = [np.zeros(MC * 8, np.uint8)]
    dev = [np.zeros(64 * 8, np.uint8)]
    tok = np.full((1, H), -1, np.int32)
    st = np.zeros((1, H), np.int32)
    clk = np.zeros(1, np.int32)
    for b in g["batches"]:
        tk = np.array(b["top_k"], dtype=np.int32).reshape(Q, 1, K)
        out = np.zeros((Q, 1, K), np.int32)
        miss = np.zeros((Q, 1), np.int32)
        err = orc.resolve_spec(tk, np.array([b["committed"]], np.int32), hcl, dbl, tok, st, clk, None, out, miss,
                               host, dev)
        assert err == 0, b["why"]
        assert out.reshape(Q, K).tolist() == b["out"], b["why"]
        assert miss.reshape(Q, 1).tolist() == b["miss"], b["why"]
        assert tok[0].tolist() == b["tokens"] and st[0].tolist() == b["stamps"], b["why"]
        assert int(clk[0]) == b["clock"], b["why"]


@pytest.mark.parametrize("name", ["tiny", "dsa_small", "mixed_small", "indexshare_small"])
def test_one_query_batch_is_a_plain_step(name):
    wl = small_workload(name, seed=9)
    plain = OracleSim(wl, host_pools=host_pools_for(wl))
    spec = OracleSim(wl, host_pools=[p.copy() for p in plain.host])  # rows no token maps to are unset
    for step in range(wl.steps):
        for sim in (plain, spec):
            sim.write_newest(step)
            poison_host_newest(wl, step, sim.host)
        ep = plain.resolve(step)
        S = wl.seq_lens(step)
        out = np.zeros((1, wl.R, wl.K), np.int32)
        miss = np.zeros((1, wl.R), np.int32)
        es = spec.orc.resolve_spec(wl.top_k_tokens(step)[None], S - 1, wl.host_cache_locs, wl.device_buffer_locs,
                                   spec.tokens, spec.stamps, spec.clock, wl.resident_pages, out, miss, spec.host,
                                   spec.dev)
        spec.out[:], spec.miss[:] = out[0], miss[0]
        if wl.cfg.backup:
            ep |= plain.backup(step)
            es |= spec.orc.backup_spec(1, S - 1, np.ones(wl.R, np.int32), wl.host_cache_locs, wl.device_buffer_locs,
                                       wl.resident_pages, spec.host, spec.dev)
        assert ep == es
        for a in ("out", "miss", "tokens", "stamps", "clock"):
            assert np.array_equal(getattr(plain, a), getattr(spec, a)), f"step {step}: {a}"
        for layer in range(wl.L):
            assert np.array_equal(plain.dev[layer], spec.dev[layer]) and np.array_equal(plain.host[layer],
                                                                                         spec.host[layer])


class SpecRun:
    """Speculative batches over a workload's request layout: Q verify steps per batch, a
    seeded accepted count per request, top-k rows reusing the previous batch's tokens."""

    def __init__(self, wl, Q, seed, hot_slots=None):
        self.wl, self.Q = wl, Q
        self.H = wl.H if hot_slots is None else hot_slots
        self.rng = np.random.default_rng(seed)
        # a buffer of H slots + Q reserved rows per request, in device rows after the
        # workload's own (resident pages keep their rows)
        self.device_rows = wl.device_rows + wl.R * (self.H + Q)
        self.orc = oracle.Oracle(wl.K, self.H, wl.B, wl.L, wl.max_context, wl.host_rows, self.device_rows, wl.ps,
                                 wl.max_pages)
        self.host = host_pools_for(wl)
        self.dev = [np.concatenate([p, np.zeros(wl.R * (self.H + Q) * wl.B, np.uint8)])
                    for p in device_pool_model(wl)]
        self.dbl = (wl.device_rows + np.arange(wl.R * (self.H + Q), dtype=np.int64)).reshape(wl.R, self.H + Q)
        self.dbl = self.dbl.astype(np.int32)
        self.tok = np.where(np.arange(self.H)[None, :] < np.minimum(wl.seq0[:, None] - 1, self.H),
                            np.arange(self.H)[None, :], -1).astype(np.int32)
        self.tok[wl.seq0 > self.H] = -1
        # requests that fit the buffer hold token t in slot t: write those rows
        for r in range(wl.R):
            n = min(int(wl.seq0[r]) - 1, self.H)
            if n <= 0 or wl.seq0[r] > self.H:
                continue
            for layer in range(wl.L):
                rows = wl.rows(layer, r, list(range(n)))
                for t in range(n):
                    d = int(self.dbl[r, t])
                    self.dev[layer][d * wl.B:(d + 1) * wl.B] = rows[t]
        self.st = np.zeros((wl.R, self.H), np.int32)
        self.clk = np.zeros(wl.R, np.int32)
        self.S0 = wl.seq0.astype(np.int32) - 1
        self.prev = [np.zeros(0, np.int32) for _ in range(wl.R)]

    def row_of(self, r, t, j):
        wl = self.wl
        if wl.resident_pages is not None and wl.resident_pages[r, t // wl.ps] >= 0:
            return int(wl.resident_pages[r, t // wl.ps]) * wl.ps + t % wl.ps
        return int(self.dbl[r, t] if t + 1 <= self.H else self.dbl[r, self.H + j])

    def forward(self):
        """What the forward pass does before a batch: write its Q new positions' rows to their
        device rows; their host rows are not valid yet (poisoned). Returns the writes as
        (request, token, device row, host row)."""
        wl, writes = self.wl, []
        for r in range(wl.R):
            for j in range(self.Q):
                t = int(self.S0[r]) + j
                row = self.row_of(r, t, j)
                h = int(wl.host_cache_locs[r, t])
                writes.append((r, t, row, h))
                for layer in range(wl.L):
                    self.dev[layer][row * wl.B:(row + 1) * wl.B] = wl.rows(layer, r, [t])[0]
                    self.host[layer][h * wl.B:(h + 1) * wl.B] = 0xEE
        return writes

    def topk(self):
        """Q seeded top-k rows: 70 % of the previous batch's last row (still in range), the
        rest fresh, every verify step over its own length S0 + q + 1."""
        wl, Q, K = self.wl, self.Q, self.wl.K
        tk = np.full((Q, wl.R, K), -1, np.int32)
        for q in range(Q):
            for r in range(wl.R):
                S = int(self.S0[r]) + q + 1
                keep = self.prev[r][self.prev[r] < S]
                keep = self.rng.permutation(keep)[: int(0.7 * K)]
                pool = np.setdiff1d(np.arange(S, dtype=np.int32), keep)
                fresh = self.rng.choice(pool, size=min(K - keep.size, pool.size), replace=False)
                row = np.concatenate([keep, fresh]).astype(np.int32)
                tk[q, r, : row.size] = self.rng.permutation(row)
        return tk

    def resolve(self, tk):
        wl, Q = self.wl, self.Q
        out = np.zeros((Q, wl.R, wl.K), np.int32)
        miss = np.zeros((Q, wl.R), np.int32)
        err = self.orc.resolve_spec(tk, self.S0, wl.host_cache_locs, self.dbl, self.tok, self.st, self.clk,
                                    wl.resident_pages, out, miss, self.host, self.dev)
        for r in range(wl.R):
            self.prev[r] = tk[Q - 1, r][tk[Q - 1, r] >= 0]
        return out, miss, err

    def resolve_split(self, tk, copy_layers):
        """The batch with only layers [0, copy_layers) copied by the verify steps, each step's
        miss plan recorded, then every step's plan gathered for the follower layers, in step
        order. Returns (out, miss, err, plan)."""
        wl, Q = self.wl, self.Q
        out = np.zeros((Q, wl.R, wl.K), np.int32)
        miss = np.zeros((Q, wl.R), np.int32)
        plan = self.orc.new_spec_plan(Q, wl.R)
        err = self.orc.resolve_spec(tk, self.S0, wl.host_cache_locs, self.dbl, self.tok, self.st, self.clk,
                                    wl.resident_pages, out, miss, self.host, self.dev, copy_layers=copy_layers,
                                    plan=plan)
        if copy_layers < wl.L:
            for q in range(Q):
                err |= self.orc.gather(self.orc.step_plan(plan, q), wl.host_cache_locs, copy_layers,
                                       wl.L - copy_layers, self.host, self.dev)
        for r in range(wl.R):
            self.prev[r] = tk[Q - 1, r][tk[Q - 1, r] >= 0]
        return out, miss, err, plan

    def batch(self):
        self.forward()
        tk = self.topk()
        out, miss, err = self.resolve(tk)
        return tk, out, miss, err

    def accept(self, acc=None, check=True):
        wl = self.wl
        if acc is None:
            acc = self.rng.integers(1, self.Q + 1, size=wl.R).astype(np.int32)
        S0 = self.S0.copy()
        err = self.orc.backup_spec(self.Q, S0, acc, wl.host_cache_locs, self.dbl, wl.resident_pages,
                                   self.host, self.dev)
        if check:
            for r in range(wl.R):
                for j in range(int(acc[r])):
                    t = int(S0[r]) + j
                    h = int(wl.host_cache_locs[r, t])
                    for layer in range(wl.L):
                        assert np.array_equal(self.host[layer][h * wl.B:(h + 1) * wl.B], wl.rows(layer, r, [t])[0])
        self.S0 = self.S0 + acc
        return acc, S0, err


def _spec_workload(name, steps=40):
    """A small workload with room for `steps` accepted positions per request (default: six
    batches of up to four)."""
    from test_oracle_pins import SMALL
    kw = dict(SMALL[name])
    base = kw.pop("base", name)
    kw["steps"] = steps
    return W.make(base, 12, **kw)


def _overwrites(run, tk, out):
    """(q, request, entry) whose row no longer holds its token's bytes after the batch."""
    wl, bad = run.wl, []
    for q in range(run.Q):
        for r in range(wl.R):
            for i, t in enumerate(tk[q, r]):
                if t < 0 or out[q, r, i] < 0:
                    continue
                row = int(out[q, r, i])
                if not np.array_equal(run.dev[0][row * wl.B:(row + 1) * wl.B], wl.rows(0, r, [int(t)])[0]):
                    bad.append((q, r, i))
    return bad


@pytest.mark.parametrize("name,Q", [("dsa_small", 4), ("mixed_small", 3), ("indexshare_small", 2)])
def test_replayable_plans(name, Q):
    wl = _spec_workload(name)
    run = SpecRun(wl, Q, seed=3, hot_slots=(Q + 1) * wl.K)
    for _ in range(6):
        tk, out, miss, err = run.batch()
        assert err == 0
        assert not _overwrites(run, tk, out), "a verify step reused a row an earlier step of its batch resolved"
        assert run.accept()[2] == 0


def test_too_small_a_buffer_breaks_replay():
    wl = _spec_workload("dsa_small")
    Q = 4
    run = SpecRun(wl, Q, seed=3, hot_slots=Q * wl.K // 2)
    found = False
    for _ in range(6):
        tk, out, miss, err = run.batch()
        found = found or bool(_overwrites(run, tk, out))
        run.accept()
    assert found, "with H < (Q + 1) * K some verify step should reuse an earlier step's row"


@pytest.mark.parametrize("copy_layers", [0, 1, 3])
def test_leader_batch_and_step_gathers_equal_the_full_batch(copy_layers):
    """IndexShare under MTP: verify steps that copy only the leader layers and record their own
    plans, then each step's plan replayed for the followers in step order, leave every layer's
    pool, the row tables, the miss counts and the slot state exactly as the full batch does;
    each step's plan holds as many misses as its miss count."""
    wl = _spec_workload("indexshare_small")
    assert wl.L == 3
    Q = 2
    full = SpecRun(wl, Q, seed=3, hot_slots=(Q + 1) * wl.K)
    split = SpecRun(wl, Q, seed=3, hot_slots=(Q + 1) * wl.K)
    for b in range(6):
        full.forward()
        split.forward()
        tk = full.topk()
        assert np.array_equal(tk, split.topk())
        out_f, miss_f, err_f = full.resolve(tk)
        out_s, miss_s, err_s, plan = split.resolve_split(tk, copy_layers)
        assert err_f == err_s == 0
        assert np.array_equal(out_f, out_s) and np.array_equal(miss_f, miss_s)
        assert np.array_equal(plan.count, miss_s), f"batch {b}: plan counts"
        assert int(miss_s.sum()) > 0
        for name in ("tok", "st", "clk"):
            assert np.array_equal(getattr(full, name), getattr(split, name)), f"batch {b}: {name}"
        for layer in range(wl.L):
            assert np.array_equal(full.dev[layer], split.dev[layer]), f"batch {b}: layer {layer} pool"
        acc = full.rng.integers(1, Q + 1, size=wl.R).astype(np.int32)
        split.rng.integers(1, Q + 1, size=wl.R)
        assert full.accept(acc.copy())[2] == 0
        assert split.accept(acc.copy())[2] == 0


def test_step_gathers_out_of_step_order_can_differ():
    """The follower replay must follow step order: replaying the steps' plans backwards leaves
    some follower row with a later step's token overwritten by an earlier step's, once a slot
    is reused within a batch (a buffer too small to keep every step's rows)."""
    wl = _spec_workload("indexshare_small")
    Q = 4
    runs = [SpecRun(wl, Q, seed=3, hot_slots=Q * wl.K // 2) for _ in range(2)]
    differs = False
    for b in range(6):
        for run in runs:
            run.forward()
        tk = runs[0].topk()
        runs[1].topk()
        plans = []
        for run in runs:
            out = np.zeros((Q, wl.R, wl.K), np.int32)
            miss = np.zeros((Q, wl.R), np.int32)
            plan = run.orc.new_spec_plan(Q, wl.R)
            run.orc.resolve_spec(tk, run.S0, wl.host_cache_locs, run.dbl, run.tok, run.st, run.clk,
                                 wl.resident_pages, out, miss, run.host, run.dev, copy_layers=1, plan=plan)
            plans.append(plan)
        for q in range(Q):
            runs[0].orc.gather(runs[0].orc.step_plan(plans[0], q), wl.host_cache_locs, 1, wl.L - 1,
                               runs[0].host, runs[0].dev)
        for q in reversed(range(Q)):
            runs[1].orc.gather(runs[1].orc.step_plan(plans[1], q), wl.host_cache_locs, 1, wl.L - 1,
                               runs[1].host, runs[1].dev)
        differs = differs or any(not np.array_equal(runs[0].dev[l], runs[1].dev[l]) for l in range(1, wl.L))
        acc = runs[0].rng.integers(1, Q + 1, size=wl.R).astype(np.int32)
        runs[1].rng.integers(1, Q + 1, size=wl.R)
        for run in runs:
            run.accept(acc.copy(), check=False)
    assert differs
