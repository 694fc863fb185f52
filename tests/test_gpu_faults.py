"""Tripwires, invalid inputs and API misuse on the GPU, against the oracle.

Faults are planted in the input data on the host (corrupt slot state, out-of-range
tokens and rows, repeated tokens, oversize seq_len); the kernels must flag them in the
error word and behave exactly as the oracle does. Nothing here can fault the GPU: every
planted value is caught by the kernels' own range checks before it is used as an index.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads as W  # noqa: E402
from harness import OracleSim, poison_host_newest  # noqa: E402,F401

pytestmark = pytest.mark.gpu
ERR = dict(TOKEN=1, DUP=2, STATE=4, HOSTROW=8, DEVROW=16, SEQLEN=32)


def _make_pair(requests=4, layers=1):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gpu_harness import make_pair
    seq0 = (6000, 7000, 8000, 300) + (5000,) * (requests - 4)
    wl = W.make("dsa", requests=requests, top_k=256, hot_slots=512, steps=12, seq0=seq0, layers=layers)
    orc, gpu = make_pair(wl)
    return wl, orc, gpu


def _done(orc, gpu, what):
    """Both runs' host pools agree at the end (the GPU's written only by its backups), and no
    guard around the GPU's pools or workspace changed."""
    from gpu_harness import close_pair, final_host_check
    try:
        final_host_check(orc, gpu, what)
    finally:
        close_pair(gpu)


@pytest.fixture
def pair():
    wl, orc, gpu = _make_pair()
    yield wl, orc, gpu
    _done(orc, gpu, "faults")


@pytest.fixture(params=["copy_ctas", "no_copy_ctas"])
def pair_any(request):
    """The 4-request shape (copy CTAs beside each resolve CTA), and 160 requests x 2 layers,
    which leave no SM for copy CTAs: the resolve records its plan, the plan is grouped by
    host region, and a gather copies both layers."""
    import hierarchical_sparse_attention_gb300 as hs
    wl, orc, gpu = _make_pair(*((4, 1) if request.param == "copy_ctas" else (160, 2)))
    assert (hs.hs_launch_shape(gpu.h)[0] == 0) == (request.param == "no_copy_ctas")
    yield wl, orc, gpu
    _done(orc, gpu, f"faults ({request.param})")


def step_both(wl, orc, gpu, step, tk=None, sl=None, hcl=None, dbl=None):
    import hierarchical_sparse_attention_gb300 as hs
    gpu.write_newest(step)
    orc.write_newest(step)
    poison_host_newest(wl, step, orc.host)
    poison_host_newest(wl, step, gpu.host)
    tk = wl.top_k_tokens(step) if tk is None else tk
    sl = wl.seq_lens(step) if sl is None else sl
    gpu.upload(step, top_k=tk, seq_lens=sl)
    saved = (gpu.hcl, gpu.dbl)
    if hcl is not None:
        gpu.hcl = torch.from_numpy(hcl).cuda()
    if dbl is not None:
        gpu.dbl = torch.from_numpy(dbl).cuda()
    gpu.resolve()
    gpu.backup()
    torch.cuda.synchronize()
    gpu.hcl, gpu.dbl = saved
    oerr = orc.resolve(step, top_k=tk, seq_lens=sl, host_cache_locs=hcl, device_buffer_locs=dbl)
    if hcl is None and dbl is None:
        oerr |= orc.backup(step, seq_lens=sl)
    else:
        oerr |= orc.orc.backup(sl, wl.host_cache_locs if hcl is None else hcl,
                               wl.device_buffer_locs if dbl is None else dbl, wl.resident_pages, orc.host, orc.dev)
    g = gpu.state()
    for k, o in (("out", orc.out), ("miss", orc.miss), ("tokens", orc.tokens), ("stamps", orc.stamps),
                 ("clock", orc.clock)):
        np.testing.assert_array_equal(g[k], o, err_msg=f"step {step}: {k}")
    gerr = hs.hs_get_error(gpu.h, clear=True)
    assert gerr == oerr
    for layer in range(wl.L):
        assert np.array_equal(gpu.dev[layer].cpu().numpy(), orc.dev[layer]), "device pools differ"
    return gerr


def warm(wl, orc, gpu, n=3):
    for s in range(n):
        assert step_both(wl, orc, gpu, s) == 0


def set_both(gpu, orc, name, r, s, v):
    getattr(orc, name)[r, s] = v
    t = gpu.tok if name == "tokens" else gpu.st
    t[r, s] = v


def test_corrupt_slot_state(pair):
    wl, orc, gpu = pair
    warm(wl, orc, gpu)
    set_both(gpu, orc, "stamps", 0, 5, 10**6)  # stamp from the future
    set_both(gpu, orc, "stamps", 1, 7, -3)  # negative stamp
    set_both(gpu, orc, "tokens", 1, 9, 10**7)  # token beyond the sequence
    set_both(gpu, orc, "tokens", 2, 11, -9)  # token below -1
    # two slots hold the same token that this step looks up
    tk = wl.top_k_tokens(3)
    held = orc.tokens[2]
    S = int(wl.seq_lens(3)[2])
    t = next(int(x) for x in tk[2] if x >= 0 and x != S - 1 and x in set(held.tolist()))
    s0 = int(np.nonzero(held == t)[0][0])
    other = next(s for s in range(wl.H) if s != s0 and orc.tokens[2, s] >= 0)
    set_both(gpu, orc, "tokens", 2, other, t)
    err = step_both(wl, orc, gpu, 3)
    assert err == ERR["STATE"]
    for s in range(4, 8):
        assert step_both(wl, orc, gpu, s) in (0, ERR["STATE"])


def test_bad_and_repeated_tokens(pair):
    wl, orc, gpu = pair
    warm(wl, orc, gpu)
    tk = wl.top_k_tokens(3).copy()
    S = wl.seq_lens(3)
    tk[0, 0] = S[0] + 17  # beyond the sequence
    tk[1, 3] = tk[1, 4]  # repeated token
    tk[2, :] = -1  # all padding
    err = step_both(wl, orc, gpu, 3, tk=tk)
    assert err == ERR["TOKEN"] | ERR["DUP"]


def test_host_row_out_of_range_zero_fills(pair_any):
    wl, orc, gpu = pair_any
    warm(wl, orc, gpu)
    tk = wl.top_k_tokens(3)
    hcl = wl.host_cache_locs.copy()
    S = wl.seq_lens(3)
    for r in range(3):  # a token of each long request that is not in its hot set
        held = set(orc.tokens[r].tolist())
        t = next(int(x) for x in tk[r] if x >= 0 and x != S[r] - 1 and int(x) not in held)
        hcl[r, t] = wl.host_rows + 5 if r != 1 else -4
    err = step_both(wl, orc, gpu, 3, hcl=hcl)
    assert err == ERR["HOSTROW"]


def test_device_row_out_of_range(pair_any):
    wl, orc, gpu = pair_any
    warm(wl, orc, gpu)
    dbl = wl.device_buffer_locs.copy()
    dbl[0, wl.H] = wl.device_rows + 3  # reserved newest row of a long request
    dbl[1, 17] = -2  # a hot slot
    dbl[3, 5] = 1 << 30  # a fast-path slot
    err = step_both(wl, orc, gpu, 3, dbl=dbl)
    assert err & ERR["DEVROW"]


def test_seq_len_beyond_max_context(pair):
    wl, orc, gpu = pair
    warm(wl, orc, gpu)
    sl = wl.seq_lens(3).copy()
    sl[1] = wl.max_context + 1
    err = step_both(wl, orc, gpu, 3, sl=sl)
    assert err == ERR["SEQLEN"]


def test_api_misuse():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import hierarchical_sparse_attention_gb300 as hs
    cfg = hs.make_config(2, 64, 128, 576, 1, 0, 1024, 0)
    dev = torch.zeros(1000 * 576, dtype=torch.uint8, device="cuda")
    ws = torch.zeros(hs.hs_workspace_bytes(cfg), dtype=torch.uint8, device="cuda")
    import mmap
    raw = mmap.mmap(-1, 1000 * 576, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
    host = np.frombuffer(raw, dtype=np.uint8)
    with pytest.raises(hs.HsError) as e:  # host pool not registered
        hs.hs_create(cfg, [host], [dev], 1000, 1000, ws)
    assert e.value.status == hs.HS_ERR_INVALID_ARG
    hs.hs_host_register(host)
    try:
        with pytest.raises(hs.HsError) as e:  # device pool given as host memory
            hs.hs_create(cfg, [host], [host], 1000, 1000, ws)
        assert e.value.status == hs.HS_ERR_INVALID_ARG
        with pytest.raises(hs.HsError) as e:  # workspace on the host
            hs.hs_create(cfg, [host], [dev], 1000, 1000, host)
        assert e.value.status == hs.HS_ERR_INVALID_ARG
        with pytest.raises(hs.HsError) as e:  # more rows than int32 tables can address
            hs.hs_create(cfg, [host], [dev], 1 << 33, 1000, ws)
        assert e.value.status == hs.HS_ERR_INVALID_ARG
        big = hs.make_config(2, 4096, 16384, 576, 1, 0, 1024, 0)  # shared memory does not fit
        with pytest.raises(hs.HsError) as e:
            hs.hs_create(big, [host], [dev], 1000, 1000, ws)
        assert e.value.status == hs.HS_ERR_INVALID_CONFIG
        short = hs.make_config(2, 64, 128, 576, 1, 0, 1024, 0, 500)  # host rows closer than a row
        with pytest.raises(hs.HsError) as e:
            hs.hs_create(short, [host], [dev], 1000, 1000, ws)
        assert e.value.status == hs.HS_ERR_INVALID_CONFIG
        h = hs.hs_create(cfg, [host], [dev], 1000, 1000, ws)
        i32 = lambda *s: torch.zeros(s, dtype=torch.int32, device="cuda")  # noqa: E731
        tk, sl, hcl, dbl = i32(2, 64), i32(2), i32(2, 1024), i32(2, 129)
        tok, st, clk, out, miss = i32(2, 128), i32(2, 128), i32(2), i32(2, 64), i32(2)
        with pytest.raises(hs.HsError) as e:  # more requests than configured
            hs.hs_resolve(h, 3, tk, sl, hcl, dbl, tok, st, clk, None, out, miss)
        assert e.value.status == hs.HS_ERR_INVALID_ARG
        with pytest.raises(hs.HsError) as e:  # missing table
            hs.hs_resolve(h, 2, tk, sl, None, dbl, tok, st, clk, None, out, miss)
        assert e.value.status == hs.HS_ERR_INVALID_ARG
        with pytest.raises(hs.HsError) as e:  # resident pages without a page size
            hs.hs_resolve(h, 2, tk, sl, hcl, dbl, tok, st, clk, i32(2, 4), out, miss)
        assert e.value.status == hs.HS_ERR_INVALID_ARG
        out.fill_(123)
        hs.hs_resolve(h, 0, tk, sl, hcl, dbl, tok, st, clk, None, out, miss)  # empty batch: no-op
        hs.hs_backup(h, 0, sl, hcl, dbl, None)
        torch.cuda.synchronize()
        assert int(out.min()) == 123 and int(out.max()) == 123
        assert hs.hs_get_error(h) == 0
        hs.hs_destroy(h)
    finally:
        hs.hs_host_unregister(host)


def test_partial_batch_leaves_other_requests_alone(pair):
    wl, orc, gpu = pair
    warm(wl, orc, gpu)
    before = gpu.state()
    gpu.write_newest(3)
    gpu.upload(3)
    gpu.resolve(num_requests=2)
    torch.cuda.synchronize()
    after = gpu.state()
    for k in ("tokens", "stamps", "clock"):
        np.testing.assert_array_equal(after[k][2:], before[k][2:])
    np.testing.assert_array_equal(after["out"][2:], before["out"][2:])


def test_two_handles_with_different_shared_memory_sizes():
    """Creating a smaller handle after a larger one must not break the larger one's launches."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gpu_harness import close_pair, make_pair
    big = W.make("dsa", requests=2, top_k=2048, hot_slots=6144, steps=2, seq0=(20000, 30000))
    small = W.make("tiny", steps=2)
    ob, gb = make_pair(big)
    osm, gs = make_pair(small)  # created second, needs less shared memory
    try:
        for s in range(2):
            for wl, o, g in ((big, ob, gb), (small, osm, gs)):
                g.write_newest(s)
                o.write_newest(s)
                g.upload(s)
                g.resolve()
                g.backup()
                torch.cuda.synchronize()
                o.resolve(s)
                o.backup(s)
                np.testing.assert_array_equal(g.state()["out"], o.out)
                np.testing.assert_array_equal(g.state()["stamps"], o.stamps)
    finally:
        close_pair(gb)
        close_pair(gs)


def test_stale_or_garbage_hints_do_not_change_results(pair):
    """The residency bitmap in the workspace only starts transfers early: overwriting it (and
    the plan after it) with garbage, or resetting a request's state behind its back, leaves
    every result exact."""
    wl, orc, gpu = pair
    warm(wl, orc, gpu)
    g = torch.Generator(device="cpu").manual_seed(7)
    junk = torch.randint(-32768, 32767, (gpu.ws.numel() // 2 - 128,), generator=g, dtype=torch.int16)
    gpu.ws.view(torch.int16)[128:].copy_(junk)  # keep the 256-byte header, scramble the bitmap
    assert step_both(wl, orc, gpu, 3) == 0
    # request 0 starts over with an empty buffer; its bits still describe the old contents
    for name in ("tokens", "stamps"):
        getattr(orc, name)[0, :] = -1 if name == "tokens" else 0
    orc.clock[0] = 0
    gpu.tok[0].fill_(-1)
    gpu.st[0].fill_(0)
    gpu.clk[0] = 0
    for s in range(4, 8):
        assert step_both(wl, orc, gpu, s) == 0


def bitmap_words(wl):
    """The residency bitmap region of the workspace, as hs.h lays it out after the header."""
    words = (wl.max_context + 127) // 128 * 4
    return words, 256, wl.R * words


def test_reset_hints_after_state_change(pair):
    """hs_reset_hints clears the residency bitmap (every bit 0, as hs_create leaves it) in
    stream order; later steps stay exact and set the bits of the tokens they place again."""
    import hierarchical_sparse_attention_gb300 as hs
    wl, orc, gpu = pair
    warm(wl, orc, gpu)
    words, off, n = bitmap_words(wl)
    bits = gpu.ws[off: off + 4 * n].view(torch.int32)
    assert int((bits != 0).sum().item()) > 0  # the warm steps set bits
    bits.fill_(0x5A5A5A5A)
    hs.hs_reset_hints(gpu.h)
    torch.cuda.synchronize()
    assert bool((bits == 0).all().item())
    for s in range(3, 6):
        assert step_both(wl, orc, gpu, s) == 0
    assert int((bits != 0).sum().item()) > 0


def test_bitmap_matches_slot_map(pair):
    """While the kernels alone change the state, a set bit always names a token its request
    holds (a miss is never predicted to hit), and every held token of the last step's top-k
    has its bit set (placed misses, hits, and predicted misses that hit). Tokens of the
    starting state that no step touched yet may still be clear: those only cost speed."""
    wl, orc, gpu = pair
    warm(wl, orc, gpu)
    last = 5
    for s in range(3, last + 1):
        assert step_both(wl, orc, gpu, s) == 0
    words, off, n = bitmap_words(wl)
    bits = gpu.ws[off: off + 4 * n].view(torch.int32).cpu().numpy().view(np.uint32).reshape(wl.R, words)
    tok = gpu.tok.cpu().numpy()
    seq = gpu.sl.cpu().numpy()
    topk = wl.top_k_tokens(last)
    for r in range(wl.R):
        got = ((bits[r][:, None] >> np.arange(32, dtype=np.uint32)) & 1).astype(bool).reshape(-1)[:seq[r]]
        held = np.zeros(seq[r], dtype=bool)
        held[tok[r][tok[r] >= 0]] = True
        if seq[r] <= wl.H:  # fast path: slot t holds token t for every committed t
            np.testing.assert_array_equal(got, held)
            continue
        assert not (got & ~held).any(), f"request {r}: a set bit names a token no slot holds"
        mine = topk[r][(topk[r] >= 0) & (topk[r] < seq[r] - 1)]
        mine = mine[held[mine]]
        assert mine.size > 0 and got[mine].all(), f"request {r}: a held top-k token has a clear bit"
