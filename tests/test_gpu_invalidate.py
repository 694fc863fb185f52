"""GPU parity of hot-slot invalidation (hs_invalidate_tokens, hs_invalidate_host_rows)
against the CPU oracle, bit-exact: slot maps, stamps and flags after each invalidation,
then further decode steps on both sides, which must refetch the cleared tokens (the
kernels also keep the token->slot hints in step, which only affects speed)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import workloads as W  # noqa: E402
from harness import host_newest_ok, poison_host_newest  # noqa: E402
from test_gpu_parity import _gpu, compare_pools, compare_step  # noqa: E402

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _clear_lists(rng, wl, tokens, S, frac=0.3, extra=5):
    """Per request: some held tokens, some tokens no slot holds, padding, out-of-range."""
    offs, toks = [0], []
    for r in range(wl.R):
        held = tokens[r][tokens[r] >= 0]
        k = int(frac * held.size)
        pick = list(rng.choice(held, size=k, replace=False)) if k else []
        pick += list(rng.integers(0, max(1, int(S[r])), size=extra)) + [-1, int(S[r]) + 3, int(S[r]) - 1]
        rng.shuffle(pick)
        toks += pick
        offs.append(len(toks))
    return np.array(offs, dtype=np.int32), np.array(toks, dtype=np.int32)


def _rows_of(wl, offs, toks, S):
    rows = []
    for r in range(wl.R):
        for t in toks[offs[r]:offs[r + 1]]:
            if 0 <= t < S[r] - 1:
                rows.append(wl.host_cache_locs[r, t])
    return np.unique(np.array(rows + [10 ** 9 - 7], dtype=np.int32))  # plus a row nobody has


def _compare_state(gpu, orc, what):
    import hierarchical_sparse_attention_gb300 as hs
    np.testing.assert_array_equal(gpu.tok.cpu().numpy(), orc.tokens, err_msg=f"{what}: device_buffer_tokens")
    np.testing.assert_array_equal(gpu.st.cpu().numpy(), orc.stamps, err_msg=f"{what}: lru_slots")
    np.testing.assert_array_equal(gpu.clk.cpu().numpy(), orc.clock, err_msg=f"{what}: lru_clock")
    return hs.hs_get_error(gpu.h, clear=True)


def run_with_invalidation(wl, every=3, seed=0):
    import hierarchical_sparse_attention_gb300 as hs
    gh = _gpu()
    orc, gpu = gh.make_pair(wl)
    rng = np.random.default_rng(seed)
    try:
        for step in range(wl.steps):
            gpu.write_newest(step)
            orc.write_newest(step)
            poison_host_newest(wl, step, gpu.host)
            poison_host_newest(wl, step, orc.host)
            gpu.upload(step)
            gpu.resolve()
            gpu.backup()
            torch.cuda.synchronize()
            assert host_newest_ok(wl, step, gpu.host)
            oerr = orc.resolve(step) | orc.backup(step)
            gerr = compare_step(gpu, orc, f"{wl.cfg.name} step {step}")
            assert gerr == oerr, f"step {step}: flags gpu {gerr} oracle {oerr}"
            if step % every != every - 1:
                continue
            S = wl.seq_lens(step)
            offs, toks = _clear_lists(rng, wl, orc.tokens, S)
            if (step // every) % 2 == 0:
                hs.hs_invalidate_tokens(gpu.h, wl.R, _dev(S), _dev(offs), _dev(toks), gpu.tok, gpu.st)
                oerr = orc.orc.invalidate_tokens(S, offs, toks, orc.tokens, orc.stamps)
                kind = "tokens"
            else:
                rows = _rows_of(wl, offs, toks, S)
                hs.hs_invalidate_host_rows(gpu.h, wl.R, _dev(S), gpu.hcl, _dev(rows), rows.size, gpu.tok, gpu.st)
                oerr = orc.orc.invalidate_host_rows(S, wl.host_cache_locs, rows, orc.tokens, orc.stamps)
                kind = "host rows"
            gerr = _compare_state(gpu, orc, f"{wl.cfg.name} after step {step}, invalidate by {kind}")
            assert gerr == oerr, f"invalidate by {kind}: flags gpu {gerr} oracle {oerr}"
        compare_pools(gpu, orc, f"{wl.cfg.name} end")
        gh.final_host_check(orc, gpu, f"{wl.cfg.name} end")
    finally:
        gh.close_pair(gpu)


def test_invalidate_tiny():
    run_with_invalidation(W.make("tiny", 0))


def test_invalidate_dsa_small():
    run_with_invalidation(W.make("dsa", 1, requests=3, top_k=256, hot_slots=512, steps=10,
                                 seq0=(6000, 9000, 300)))


def test_invalidate_mixed_residency():
    run_with_invalidation(W.make("mixed1m", 2, requests=2, top_k=128, hot_slots=256, steps=9,
                                 seq0=(20000, 9000), resident_tail_pages=16))


def test_invalidate_indexshare_layers():
    run_with_invalidation(W.make("indexshare", 3, requests=4, top_k=64, hot_slots=128, steps=9, layers=3,
                                 seq_range=(1000, 3000)))


def _synthetic_state(rng, R, H, S, clock):
    """A seeded slot map: distinct tokens below S - 1 (a fifth of the slots free), stamps <= clock."""
    tok = np.full((R, H), -1, dtype=np.int32)
    st = np.zeros((R, H), dtype=np.int32)
    for r in range(R):
        n = min(H, max(0, int(S[r]) - 1))
        held = rng.choice(int(S[r]) - 1, size=n, replace=False).astype(np.int32) if n else np.zeros(0, np.int32)
        keep = rng.random(n) < 0.8
        slots = rng.permutation(H)[:n]
        tok[r, slots[keep]] = held[keep]
        st[r, slots[keep]] = rng.integers(1, clock + 1, size=int(keep.sum()))
    return tok, st


@pytest.mark.parametrize("form", ["tokens", "host_rows"])
def test_invalidate_dsa_full_size(form):
    """The dsa decode shape (32 requests, 4096 slots, seq 131072) on a seeded state, one CTA
    per request as in every call."""
    import hierarchical_sparse_attention_gb300 as hs
    _gpu()
    wl = W.make("dsa", 0, steps=2)
    rng = np.random.default_rng(21)
    S = wl.seq_lens(0)
    tok, st = _synthetic_state(rng, wl.R, wl.H, S, clock=50)
    offs, toks = _clear_lists(rng, wl, tok, S, frac=0.25, extra=50)
    orc = oracle.Oracle(wl.K, wl.H, wl.B, wl.L, wl.max_context, wl.host_rows, wl.device_rows)
    o_tok, o_st = tok.copy(), st.copy()
    cfg = hs.make_config(wl.R, wl.K, wl.H, wl.B, wl.L, wl.ps, wl.max_context, wl.max_pages)
    ws = torch.zeros(hs.hs_workspace_bytes(cfg), dtype=torch.uint8, device="cuda")
    hostp = [np.zeros(wl.host_rows * wl.B, dtype=np.uint8)]
    for p in hostp:
        hs.hs_host_register(p)
    devp = [torch.zeros(wl.device_rows * wl.B, dtype=torch.uint8, device="cuda")]
    h = hs.hs_create(cfg, hostp, devp, wl.host_rows, wl.device_rows, ws)
    try:
        g_tok, g_st = _dev(tok), _dev(st)
        if form == "tokens":
            hs.hs_invalidate_tokens(h, wl.R, _dev(S), _dev(offs), _dev(toks), g_tok, g_st)
            oerr = orc.invalidate_tokens(S, offs, toks, o_tok, o_st)
        else:
            rows = _rows_of(wl, offs, toks, S)
            assert rows.size > 8192  # the binary search runs on the unstaged list here
            hs.hs_invalidate_host_rows(h, wl.R, _dev(S), _dev(wl.host_cache_locs), _dev(rows), rows.size,
                                       g_tok, g_st)
            oerr = orc.invalidate_host_rows(S, wl.host_cache_locs, rows, o_tok, o_st)
        gerr = hs.hs_get_error(h, clear=True)
        assert gerr == oerr
        assert int((o_tok != tok).sum()) > 1000  # a real amount of clearing happened
        np.testing.assert_array_equal(g_tok.cpu().numpy(), o_tok)
        np.testing.assert_array_equal(g_st.cpu().numpy(), o_st)
    finally:
        hs.hs_destroy(h)
        for p in hostp:
            hs.hs_host_unregister(p)


def test_invalidate_edge_cases():
    """Long clear lists (several hash passes), a bad seq_len, an unsorted row list, empty lists."""
    import hierarchical_sparse_attention_gb300 as hs
    gh = _gpu()
    wl = W.make("tiny", 4)
    orc, gpu = gh.make_pair(wl)
    rng = np.random.default_rng(8)
    try:
        for step in range(6):
            gpu.write_newest(step)
            orc.write_newest(step)
            gpu.upload(step)
            gpu.resolve()
            gpu.backup()
            orc.resolve(step)
            orc.backup(step)
        torch.cuda.synchronize()
        hs.hs_get_error(gpu.h, clear=True)
        S = wl.seq_lens(5).copy()
        # 1. request 0 clears 12,000 entries (three passes of the token hash), request 1 none
        big = rng.integers(-2, int(S[0]) + 5, size=12000).astype(np.int32)
        held = orc.tokens[0][orc.tokens[0] >= 0]
        big[rng.choice(big.size, size=held.size // 2, replace=False)] = held[: held.size // 2]
        offs = np.array([0, big.size, big.size], dtype=np.int32)
        hs.hs_invalidate_tokens(gpu.h, wl.R, _dev(S), _dev(offs), _dev(big), gpu.tok, gpu.st)
        oerr = orc.orc.invalidate_tokens(S, offs, big, orc.tokens, orc.stamps)
        assert _compare_state(gpu, orc, "12,000 tokens") == oerr
        # 2. a seq_len above max_context: the request is skipped and flagged on both sides
        bad = S.copy()
        bad[0] = wl.max_context + 1
        offs = np.array([0, 3, 3], dtype=np.int32)
        toks = orc.tokens[0][orc.tokens[0] >= 0][:3].copy()
        hs.hs_invalidate_tokens(gpu.h, wl.R, _dev(bad), _dev(offs), _dev(toks), gpu.tok, gpu.st)
        oerr = orc.orc.invalidate_tokens(bad, offs, toks, orc.tokens, orc.stamps)
        assert oerr == oracle.ERR_SEQLEN and _compare_state(gpu, orc, "bad seq_len") == oerr
        # 3. an unsorted row list of at most 8192 rows: the kernel clears nothing and flags it
        rows = np.unique(wl.host_cache_locs[0, orc.tokens[0][orc.tokens[0] >= 0]])[::-1].copy()
        assert rows.size >= 2
        before = (gpu.tok.clone(), gpu.st.clone())
        hs.hs_invalidate_host_rows(gpu.h, wl.R, _dev(S), gpu.hcl, _dev(rows), rows.size, gpu.tok, gpu.st)
        assert hs.hs_get_error(gpu.h, clear=True) == hs.HS_FLAG_ORDER
        assert torch.equal(gpu.tok, before[0]) and torch.equal(gpu.st, before[1])
        # 4. empty lists change nothing
        hs.hs_invalidate_tokens(gpu.h, wl.R, _dev(S), _dev(np.zeros(3, np.int32)), _dev(np.zeros(1, np.int32)),
                                gpu.tok, gpu.st)
        hs.hs_invalidate_host_rows(gpu.h, wl.R, _dev(S), gpu.hcl, _dev(np.zeros(1, np.int32)), 0, gpu.tok, gpu.st)
        assert _compare_state(gpu, orc, "empty lists") == 0
        # 5. the next steps refetch what was cleared, bit-exact
        for step in range(6, 10):
            gpu.write_newest(step)
            orc.write_newest(step)
            poison_host_newest(wl, step, gpu.host)
            poison_host_newest(wl, step, orc.host)
            gpu.upload(step)
            gpu.resolve()
            gpu.backup()
            torch.cuda.synchronize()
            oerr = orc.resolve(step) | orc.backup(step)
            assert compare_step(gpu, orc, f"after edge cases, step {step}") == oerr
        compare_pools(gpu, orc, "after edge cases")
        gh.final_host_check(orc, gpu, "after edge cases")
    finally:
        gh.close_pair(gpu)
