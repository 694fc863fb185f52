"""Pins of the CPU oracle to things other than itself (no GPU needed).

* a hand-traced example of the policy (tests/golden/hand_trace_h4_k3.json),
* brute-force enumeration of every victim assignment on tiny inputs, with its own
  history-based notion of "least recently used" (no stamps),
* reduction to textbook LRU (collections.OrderedDict) at top_k = 1,
* the pages' invariants on multi-step seeded runs (injective slot map, occupancy,
  exact row bytes, misses = |top-k minus hot set|, eager backup restores the host row),
* special cases (fast path identity, fast->slow transition, full reuse, padding),
* the page-printed sizing arithmetic (tests/golden/pages_arithmetic.json).
"""
import collections
import itertools
import json
import os

import numpy as np
import pytest

import oracle
import workloads as W
from harness import OracleSim, host_newest_ok

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _single_request_oracle(H, K, B=8, host_rows=64, max_context=64, device_rows=None, L=1):
    device_rows = device_rows if device_rows is not None else 200
    return oracle.Oracle(K, H, B, L, max_context, host_rows, device_rows)


class OneRequest:
    """A single request driven directly through the oracle (host row of t is t)."""

    def __init__(self, H, K, dbl=None, B=8, max_context=64, L=1, device_rows=200):
        self.H, self.K, self.B, self.L = H, K, B, L
        self.orc = oracle.Oracle(K, H, B, L, max_context, max_context, device_rows)
        self.dbl = np.asarray(dbl if dbl is not None else np.arange(H + 1), dtype=np.int32).reshape(1, H + 1)
        self.hcl = np.arange(max_context, dtype=np.int32).reshape(1, max_context)
        self.tokens = np.full((1, H), -1, dtype=np.int32)
        self.stamps = np.zeros((1, H), dtype=np.int32)
        self.clock = np.zeros(1, dtype=np.int32)
        self.host = [np.arange(max_context * B, dtype=np.uint32).astype(np.uint8) + np.uint8(17 * l)
                     for l in range(L)]
        self.dev = [np.zeros(device_rows * B, dtype=np.uint8) for _ in range(L)]
        self.out = np.zeros((1, K), dtype=np.int32)
        self.miss = np.zeros(1, dtype=np.int32)

    def step(self, seq_len, topk, hcl=None):
        tk = np.asarray(topk, dtype=np.int32).reshape(1, self.K)
        err = self.orc.resolve(tk, np.array([seq_len], dtype=np.int32), self.hcl if hcl is None else hcl,
                               self.dbl, self.tokens, self.stamps, self.clock, None, self.out, self.miss,
                               self.host, self.dev)
        return self.out[0].copy(), int(self.miss[0]), err


# ---------------------------------------------------------------------------------------
def test_hand_trace():
    g = json.load(open(os.path.join(GOLDEN, "hand_trace_h4_k3.json")))
    q = OneRequest(g["hot_slots"], g["top_k"], dbl=g["device_buffer_locs"])
    for st in g["steps"]:
        out, miss, err = q.step(st["seq_len"], st["top_k"])
        assert out.tolist() == st["out"], st["why"]
        assert miss == st["miss"] and err == st["err"], st["why"]
        assert q.tokens[0].tolist() == st["tokens"], st["why"]
        assert q.stamps[0].tolist() == st["stamps"], st["why"]
        assert int(q.clock[0]) == st["clock"]


def test_duplicate_holders_golden():
    """A slot map holding two tokens twice, worked by hand from the resolve kernel's phases 2
    and 3 ("vLLM Hybrid HiSparse source implementation analysis", 7.2): a looked-up token's
    lowest holder serves it, its other holder stays evictable, and ages out like any slot."""
    g = json.load(open(os.path.join(GOLDEN, "duplicate_holders_h5_k2.json")))
    q = OneRequest(g["hot_slots"], g["top_k"], dbl=g["device_buffer_locs"])
    q.tokens[0, :] = g["initial"]["tokens"]
    q.stamps[0, :] = g["initial"]["stamps"]
    q.clock[0] = g["initial"]["clock"]
    for st in g["steps"]:
        out, miss, err = q.step(st["seq_len"], st["top_k"])
        assert out.tolist() == st["out"], st["why"]
        assert miss == st["miss"] and err == st["err"], st["why"]
        assert q.tokens[0].tolist() == st["tokens"], st["why"]
        assert q.stamps[0].tolist() == st["stamps"], st["why"]
        assert int(q.clock[0]) == st["clock"]


def test_page_first_layout_changes_only_addresses():
    """Every layer's bytes of a token in one host row ("Hierarchical Sparse Attention" (Alibaba
    Tair KVCache), 2.4.4, page_first): the same steps give the same row tables, slot state,
    flags and device pools as one host pool per layer, and after every backup host row h of
    layer l in the shared pool holds exactly layer l's row h of the layer-first pools."""
    wl_a = small_workload("indexshare_small")
    wl_b = W.make("indexshare", 0, host_layout="page_first", **{k: v for k, v in SMALL["indexshare_small"].items()
                                                                   if k != "base"})
    a, b = OracleSim(wl_a), OracleSim(wl_b)
    assert wl_b.host_row_stride == wl_b.L * wl_b.B and len(b.host_bases) == 1
    for step in range(wl_a.steps):
        assert a.step(step) == b.step(step) == 0
        for name in ("out", "miss", "tokens", "stamps", "clock"):
            np.testing.assert_array_equal(getattr(a, name), getattr(b, name), err_msg=f"step {step}: {name}")
        for layer in range(wl_a.L):
            assert np.array_equal(a.dev[layer], b.dev[layer]), f"step {step}: device pool {layer}"
        shared = b.host_bases[0].reshape(wl_b.host_rows, wl_b.L, wl_b.B)
        for layer in range(wl_a.L):
            assert np.array_equal(shared[:, layer, :], a.host[layer].reshape(wl_a.host_rows, wl_a.B)), \
                f"step {step}: host layer {layer}"


def test_pages_arithmetic():
    g = json.load(open(os.path.join(GOLDEN, "pages_arithmetic.json")))
    row = g["fp8_mla_row"]
    assert row["nope"] + row["scales"] + row["rope"] == row["total"] == W.CONFIGS["dsa"].row_bytes
    hb = g["hot_buffer_60_layers"]
    got = oracle.hot_bytes_per_request(hb["top_k"], hb["n_spec"], hb["row_bytes"], hb["layers"])
    assert abs(got / 2**20 - hb["printed_mib"]) / hb["printed_mib"] < hb["rel_tol"]
    rs = g["region_stride_mtp3"]
    assert oracle.hot_bytes_per_request(2048, rs["n_spec"], 656, 1) / \
        oracle.hot_bytes_per_request(2048, 0, 656, 1) == rs["ratio_to_no_spec"]
    # the fp8 MLA generator lays the row out as the page describes: scales are finite fp32
    wl = W.make("dsa", requests=1, steps=1)
    r = wl.rows(0, 0, [3])[0]
    sc = r[512:528].view(np.float32)
    assert np.all(sc >= 2.0**-8) and np.all(sc < 1.0)
    assert not np.any((r[:512] & 0x7F) == 0x7F)  # no e4m3 NaN codes


# ---------------------------------------------------------------------------------------
# brute force
def brute_force_step(slots, last_use, seq_len, topk, step_no):
    """Independent formulation of one slow-path call on one request.

    slots[s] = token or None; last_use[s] = call number of the slot's last fill/hit (None
    if never used). Returns (out_slots per entry (-1 none, 'N' newest), misses, new slots,
    new last_use). Victims are found by enumerating every injective assignment of the
    misses to non-hit slots and keeping those that respect "least recently used first,
    never-used before used, lower slot on ties, earlier miss gets the more preferred slot".
    """
    H = len(slots)
    out = []
    seen = set()
    lookups = []
    for i, t in enumerate(topk):
        if t < 0 or t >= seq_len or t in seen:
            out.append(-1)
            continue
        seen.add(t)
        if t == seq_len - 1:
            out.append("N")
            continue
        out.append(None)
        lookups.append(i)
    hit_slots = set()
    misses = []
    for i in lookups:
        holders = [s for s in range(H) if slots[s] == topk[i]]
        if holders:
            out[i] = holders[0]
            hit_slots.add(holders[0])
        else:
            misses.append(i)

    def pref(s):  # smaller = evicted first
        return (0, 0, s) if slots[s] is None else (1, last_use[s], s)

    cands = [s for s in range(H) if s not in hit_slots]
    survivors = []
    for assign in itertools.permutations(cands, len(misses)):
        chosen = set(assign)
        ok = all(pref(b) > pref(a) for a in chosen for b in cands if b not in chosen)
        ok = ok and all(pref(assign[j]) < pref(assign[j + 1]) for j in range(len(assign) - 1))
        if ok:
            survivors.append(assign)
    assert len(survivors) == 1, "the victim rule must single out one assignment"
    new_slots, new_last = list(slots), list(last_use)
    for s in hit_slots:
        new_last[s] = step_no
    for j, i in enumerate(misses):
        s = survivors[0][j]
        new_slots[s] = topk[i]
        new_last[s] = step_no
        out[i] = s
    return out, len(misses), new_slots, new_last


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_tiny(seed):
    rng = np.random.default_rng(1000 + seed)
    for trial in range(40):
        H = int(rng.integers(1, 7))
        K = int(rng.integers(1, min(3, H) + 1))
        seq = int(rng.integers(H + 1, 13))
        dbl = rng.permutation(50)[: H + 1] + 10
        q = OneRequest(H, K, dbl=dbl, max_context=32)
        slots, last = [None] * H, [None] * H
        for step_no in range(1, int(rng.integers(2, 7)) + 1):
            S = seq + step_no - 1
            topk = [int(x) if rng.random() > 0.1 else -1 for x in rng.integers(0, S, size=K)]
            out, miss, err = q.step(S, topk)
            want, wmiss, slots, last = brute_force_step(slots, last, S, topk, step_no)
            exp_out = [int(dbl[H]) if w == "N" else (-1 if w == -1 else int(dbl[w])) for w in want]
            assert out.tolist() == exp_out
            assert miss == wmiss
            assert q.tokens[0].tolist() == [-1 if s is None else s for s in slots]
            assert q.stamps[0].tolist() == [0 if u is None else u for u in last]
            assert int(q.clock[0]) == step_no
            dup = len([t for t in topk if 0 <= t < S]) != len({t for t in topk if 0 <= t < S})
            assert err == (oracle.ERR_DUP if dup else 0)


# ---------------------------------------------------------------------------------------
# textbook LRU
@pytest.mark.parametrize("H", [1, 2, 3, 5, 8])
def test_textbook_lru_k1(H):
    rng = np.random.default_rng(H)
    S = 60
    q = OneRequest(H, 1, dbl=np.arange(H + 1), max_context=64)
    lru = collections.OrderedDict()  # token -> frame
    for step in range(400):
        t = int(rng.integers(0, 2 * H + 3))
        out, miss, err = q.step(S, [t])
        if t in lru:
            lru.move_to_end(t)
            want_frame, want_miss = lru[t], 0
        else:
            if len(lru) < H:
                free = sorted(set(range(H)) - set(lru.values()))
                frame = free[0]
            else:
                _, frame = lru.popitem(last=False)
            lru[t] = frame
            want_frame, want_miss = frame, 1
        assert (int(out[0]), miss, err) == (want_frame, want_miss, 0)
    # frame contents agree at the end
    want = [-1] * H
    for tok, fr in lru.items():
        want[fr] = tok
    assert q.tokens[0].tolist() == want


# ---------------------------------------------------------------------------------------
# invariants on seeded multi-step runs
SMALL = {
    "tiny": dict(),
    "dsa_small": dict(base="dsa", requests=3, top_k=256, hot_slots=512, steps=8, seq0=(6000, 9000, 300)),
    "mixed_small": dict(base="mixed1m", requests=2, top_k=128, hot_slots=256, steps=8, seq0=(20000, 9000),
                        resident_tail_pages=16),
    "indexshare_small": dict(base="indexshare", requests=4, top_k=64, hot_slots=128, steps=8, layers=3,
                             seq_range=(1000, 3000)),
    "sweep_small": dict(base="sweep", requests=2, top_k=128, hot_slots=128, steps=6, seq0=(5000, 5000),
                        reuse=0.5),
}


def small_workload(name, seed=0):
    kw = dict(SMALL[name])
    base = kw.pop("base", name)
    return W.make(base, seed, **kw)


@pytest.mark.parametrize("name", list(SMALL))
def test_invariants(name):
    wl = small_workload(name)
    sim = OracleSim(wl)
    for step in range(wl.steps):
        S = wl.seq_lens(step)
        tk = wl.top_k_tokens(step)
        before = sim.tokens.copy()
        clock_before = sim.clock.copy()
        err = sim.step(step)
        assert err == 0
        assert host_newest_ok(wl, step, sim.host)
        for r in range(wl.R):
            s_len = int(S[r])
            valid = [int(t) for t in tk[r] if 0 <= t < s_len]
            fast = s_len <= wl.H
            tok = sim.tokens[r]
            held = tok[tok >= 0]
            assert len(np.unique(held)) == len(held), "a token is held by two slots"
            assert len(held) <= wl.H
            if fast:
                assert sim.clock[r] == clock_before[r]
                assert int(sim.miss[r]) == 0
            else:
                c = int(sim.clock[r])
                assert c == clock_before[r] + 1
                assert np.all(sim.stamps[r] <= c) and np.all(sim.stamps[r] >= 0)
                nonres = [t for t in valid if wl.resident_row(r, t) < 0 and t != s_len - 1]
                prev = set(before[r][before[r] >= 0].tolist())
                assert int(sim.miss[r]) == len([t for t in nonres if t not in prev])
                for t in nonres:  # every looked-up token is now held, stamped with c
                    s = int(np.nonzero(tok == t)[0][0])
                    assert sim.stamps[r][s] == c
            # every resolved row holds the exact bytes of its token, in every layer
            rows = []
            for i, t in enumerate(tk[r]):
                o = int(sim.out[r, i])
                if t < 0:
                    assert o == -1
                    continue
                assert o >= 0
                rows.append(o)
                for layer in range(wl.L):
                    assert np.array_equal(sim.dev_row(layer, o), wl.rows(layer, r, [int(t)])[0])
            assert len(set(rows)) == len(rows), "two entries share a physical row"


# ---------------------------------------------------------------------------------------
# special cases
def test_fast_path_identity_and_transition():
    H, K = 8, 3
    dbl = np.arange(H + 1) * 3 + 5
    q = OneRequest(H, K, dbl=dbl, max_context=32, device_rows=64)
    for s in range(5):  # caller initialisation: slot s holds token s
        q.tokens[0, s] = s
    for S in range(6, H + 1):  # fast path: identity, newest slot recorded, no clock
        out, miss, err = q.step(S, [S - 1, 0, S - 3])
        assert out.tolist() == [dbl[S - 1], dbl[0], dbl[S - 3]]
        assert (miss, err, int(q.clock[0])) == (0, 0, 0)
        assert q.tokens[0, S - 1] == S - 1
    assert q.tokens[0].tolist() == list(range(H))
    # first slow-path call: all stamps are 0, so evictions go in ascending slot order
    out, miss, err = q.step(H + 1, [H, 1, 2])  # newest, and two hits on the identity slots
    assert miss == 0 and err == 0 and int(q.clock[0]) == 1
    assert out.tolist() == [dbl[H], dbl[1], dbl[2]]
    out, miss, err = q.step(H + 2, [H, H + 1, 3])  # H is no longer newest and is host-only
    assert miss == 1
    # victims among unhit slots with stamp 0: lowest is slot 0 (slots 1, 2 stamped 1; 3 hit now)
    assert out.tolist() == [dbl[0], dbl[H], dbl[3]]
    assert q.tokens[0, 0] == H


def test_first_step_takes_free_slots_in_order():
    H, K = 16, 6
    q = OneRequest(H, K, max_context=64)
    out, miss, err = q.step(40, [30, 7, 39, 12, -1, 2])
    assert miss == 4 and err == 0
    assert out.tolist() == [0, 1, H, 2, -1, 3]


def test_full_reuse_gives_zero_misses_after_warmup():
    H, K = 16, 8
    q = OneRequest(H, K, max_context=64)
    base = [3, 9, 11, 20, 21, 2, 5]
    for step in range(5):
        S = 40 + step
        out, miss, err = q.step(S, base + [S - 1])
        assert miss == (len(base) if step == 0 else 0)


def test_all_padding_changes_nothing_but_the_clock():
    q = OneRequest(8, 4, max_context=64)
    q.step(30, [1, 2, 3, 29])
    tok, st = q.tokens.copy(), q.stamps.copy()
    out, miss, err = q.step(31, [-1, -1, -1, -1])
    assert out.tolist() == [-1] * 4 and miss == 0 and err == 0
    assert np.array_equal(tok, q.tokens) and np.array_equal(st, q.stamps) and int(q.clock[0]) == 2


def test_resident_first():
    """A resident token resolves in place even when a hot slot also holds it."""
    H, K, ps = 4, 2, 4
    orc = oracle.Oracle(K, H, 8, 1, 32, 32, 100, page_size=ps, max_pages=8)
    dbl = np.arange(H + 1, dtype=np.int32).reshape(1, -1)
    tokens = np.array([[5, -1, -1, -1]], dtype=np.int32)
    stamps = np.array([[1, 0, 0, 0]], dtype=np.int32)
    clock = np.array([1], dtype=np.int32)
    rp = np.full((1, 8), -1, dtype=np.int32)
    rp[0, 1] = 20  # tokens 4..7 resident at rows 80..83
    out = np.zeros((1, K), dtype=np.int32)
    miss = np.zeros(1, dtype=np.int32)
    host = [np.zeros(32 * 8, np.uint8)]
    dev = [np.zeros(100 * 8, np.uint8)]
    err = orc.resolve(np.array([[5, 9]], np.int32), np.array([12], np.int32),
                      np.arange(32, dtype=np.int32).reshape(1, -1), dbl, tokens, stamps, clock, rp, out,
                      miss, host, dev)
    assert err == 0 and out.tolist() == [[81, 1]] and int(miss[0]) == 1
    # slot 0 (token 5) was not hit; the free slot 1 took token 9
    assert tokens.tolist() == [[5, 9, -1, -1]] and stamps.tolist() == [[1, 2, 0, 0]]


# ---------------------------------------------------------------------------------------
# tripwires and invalid input
def test_error_paths():
    H, K = 4, 3
    q = OneRequest(H, K, max_context=32, device_rows=64)
    q.step(20, [1, 2, 3])
    # corrupt: slot 0 stamp in the future, slot 1 token beyond the sequence
    q.stamps[0, 0] = 99
    q.tokens[0, 1] = 25
    out, miss, err = q.step(21, [1, 2, 3])
    assert err == oracle.ERR_STATE
    assert miss == 2  # tokens 1 and 2 re-miss; slots 0 and 1 were reset to free
    assert q.tokens[0].tolist()[:3] == [1, 2, 3]
    # duplicate holders of a looked-up token: the lowest slot wins, flagged
    q.tokens[0, 3] = 3
    out, miss, err = q.step(22, [3, -1, -1])
    assert err == oracle.ERR_STATE and out[0] == 2 and miss == 0
    # host row out of range: destination zeroed
    hcl = q.hcl.copy()
    hcl[0, 9] = 10**6
    q.dev[0][:] = 0xEE
    out, miss, err = q.step(23, [9, -1, -1], hcl=hcl)
    assert err == oracle.ERR_HOSTROW and miss == 1
    assert np.all(q.dev[0][out[0] * q.B:(out[0] + 1) * q.B] == 0)
    # device row out of range: output -1, nothing written, state still updated
    q.dbl[0, :] = [0, 1, 2, 3, 1000]
    out, miss, err = q.step(24, [23, -1, -1])
    assert err == oracle.ERR_DEVROW and out[0] == -1
    # seq_len beyond max_context: request skipped
    out, miss, err = q.step(33, [1, 2, 3])
    assert err == oracle.ERR_SEQLEN and out.tolist() == [-1, -1, -1]


def test_slot_holding_the_newest_token_is_corrupt():
    """The newest token lives in the reserved row, so a slot claiming it is stale state."""
    q = OneRequest(4, 2, max_context=32)
    q.step(20, [1, 2])
    q.tokens[0, 2] = 20
    out, miss, err = q.step(21, [20, 1])
    assert err == oracle.ERR_STATE and miss == 0
    assert out.tolist() == [4, 0] and q.tokens[0].tolist() == [1, 2, -1, -1]


def test_backup_locations():
    """Backup reads the resident row, the fast-path slot or the reserved slot H."""
    wl = small_workload("mixed_small")
    sim = OracleSim(wl)
    sim.step(0)
    assert host_newest_ok(wl, 0, sim.host)
    wl2 = small_workload("dsa_small")  # request 2 (seq 300 <= H 512) is on the fast path
    sim2 = OracleSim(wl2)
    for s in range(3):
        sim2.step(s)
        assert host_newest_ok(wl2, s, sim2.host)


def run_all_pins() -> int:
    """Run every pin above in-process; returns the number that failed (used on purpose-
    broken oracle builds by test_oracle_mutants)."""
    checks = [test_hand_trace, test_duplicate_holders_golden, test_page_first_layout_changes_only_addresses,
              test_pages_arithmetic, test_fast_path_identity_and_transition,
              test_first_step_takes_free_slots_in_order, test_full_reuse_gives_zero_misses_after_warmup,
              test_all_padding_changes_nothing_but_the_clock, test_resident_first, test_error_paths,
              test_slot_holding_the_newest_token_is_corrupt, test_backup_locations]
    checks += [lambda s=s: test_brute_force_tiny(s) for s in range(2)]
    checks += [lambda h=h: test_textbook_lru_k1(h) for h in (2, 5)]
    checks += [lambda n=n: test_invariants(n) for n in ("tiny", "mixed_small")]
    import test_oracle_invalidate as inv
    checks += [inv.test_invalidate_golden]
    checks += [lambda n=n: inv.test_token_and_host_row_forms_agree(n) for n in ("tiny", "mixed_small")]
    checks += [lambda n=n: inv.test_next_resolve_refetches_cleared_tokens(n) for n in ("tiny", "dsa_small")]
    import test_oracle_split as sp
    checks += [lambda c=c, gs=gs: sp.test_split_equals_fused(c, gs) for c, gs in sp.SPLITS[:2]]
    checks += [lambda n=n: sp.test_plan_is_the_steps_misses(n) for n in ("dsa_small", "indexshare_small")]
    checks += [sp.test_leader_only_leaves_followers]
    import test_oracle_spec as spec
    checks += [spec.test_spec_golden, lambda: spec.test_one_query_batch_is_a_plain_step("tiny"),
               lambda: spec.test_replayable_plans("dsa_small", 4),
               lambda: spec.test_leader_batch_and_step_gathers_equal_the_full_batch(1)]
    failed = 0
    for c in checks:
        try:
            c()
        except Exception:  # noqa: BLE001 - any failure counts
            failed += 1
    return failed
