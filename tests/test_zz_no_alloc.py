"""hs_resolve_noalloc through the C ABI, on two decode steps in a row, against the CPU oracle
and against the handle-based hs_resolve.

hs_resolve_noalloc serves callers that cannot allocate device memory -- engines whose
device memory is fully planned before decoding, plugins living inside another
framework's allocator, processes that must not call cudaMalloc on the decode path. It
needs no hs_create workspace: the library keeps that scratch in its own device array.
Its results must be exactly the oracle's and those of hs_resolve on the same inputs (all
comparisons here are bit-exact, like the rest of the parity tests), in each launch shape:
copy CTAs beside the resolve CTAs, none (the resolve CTA copies its own rows), and the
largest top_k. This file is collected last so a run that stops at the first failure has run
everything else first.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu

SHAPES = {
    # request 3 takes the fast path; 6 requests leave room for copy CTAs
    "copy_ctas": dict(name="dsa", requests=6, top_k=256, hot_slots=512, steps=2, layers=2,
                      seq0=(6000, 7000, 8000, 300, 9000, 10000)),
    # 160 requests leave no SM for copy CTAs: each resolve CTA copies its own misses
    "no_copy_ctas": dict(name="indexshare", requests=160, top_k=64, hot_slots=128, steps=2, layers=2,
                         seq_range=(1000, 3000)),
    # the largest top_k: the top-k hash half full
    "top_k_4096": dict(name="dsa", requests=2, top_k=4096, hot_slots=4096, steps=2, layers=1,
                       seq0=(200000, 9000)),
}


@pytest.mark.parametrize("shape", list(SHAPES))
def test_noalloc_matches_oracle_and_hs_resolve_on_two_steps(shape):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import hierarchical_sparse_attention_gb300 as hs
    from gpu_harness import close_pair, final_host_check, make_pair

    kw = dict(SHAPES[shape])
    wl = W.make(kw.pop("name"), 17, **kw)
    orc, ref = make_pair(wl)  # the oracle with its own host pools; hs_resolve with its workspace
    try:
        if shape == "no_copy_ctas":
            assert hs.hs_launch_shape(ref.h)[0] == 0
        elif shape == "copy_ctas":
            assert hs.hs_launch_shape(ref.h)[0] > 0
        # the no-allocation call's own device pools and state, on the same pinned host pools
        dev = [torch.empty_like(p).copy_(p) for p in ref.dev]
        tok0, st0, clk0 = wl.initial_state()
        tok, st, clk = (torch.from_numpy(x).cuda() for x in (tok0, st0, clk0))
        out = torch.full((wl.R, wl.K), -7, dtype=torch.int32, device="cuda")
        miss = torch.full((wl.R,), -7, dtype=torch.int32, device="cuda")
        flags = torch.full((1,), 0x7777, dtype=torch.int32, device="cuda")
        for step in range(2):
            ref.write_newest(step)
            orc.write_newest(step)
            for layer in range(wl.L):  # the same newest-token rows into the second pool
                dev[layer].copy_(ref.dev[layer])
            ref.upload(step)
            hs.hs_resolve_noalloc(ref.cfg, ref.host, dev, wl.host_rows, wl.device_rows, wl.R, ref.tk, ref.sl,
                                  ref.hcl, ref.dbl, tok, st, clk, None, out, miss, flags)
            ref.resolve()
            torch.cuda.synchronize()
            oerr = orc.resolve(step)
            want = ref.state()
            for name, got, o in (("out_rows", out, orc.out), ("miss_counts", miss, orc.miss),
                                 ("slot map", tok, orc.tokens), ("stamps", st, orc.stamps),
                                 ("clock", clk, orc.clock)):
                np.testing.assert_array_equal(got.cpu().numpy(), o, err_msg=f"{shape} step {step}: {name} vs oracle")
            for name, got in (("out", out), ("miss", miss), ("tokens", tok), ("stamps", st), ("clock", clk)):
                np.testing.assert_array_equal(got.cpu().numpy(), want[name],
                                              err_msg=f"{shape} step {step}: {name} vs hs_resolve")
            for layer in range(wl.L):
                assert np.array_equal(dev[layer].cpu().numpy(), orc.dev[layer]), \
                    f"{shape} step {step}: device pool layer {layer} vs oracle"
                assert torch.equal(dev[layer], ref.dev[layer]), f"{shape} step {step}: device pool layer {layer}"
            assert int(flags.item()) == hs.hs_get_error(ref.h, clear=True) == oerr == 0
            assert int(want["miss"].max()) > 0  # the steps did move rows
        final_host_check(orc, ref, f"{shape}")  # no backup ran: the host pools were only read
    finally:
        close_pair(ref)


def test_noalloc_rejects_more_layers_than_its_scratch_holds():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import hierarchical_sparse_attention_gb300 as hs
    cfg = hs.make_config(1, 8, 16, 64, hs.HS_NOALLOC_MAX_LAYERS + 1, 0, 64, 0)
    z = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(hs.HsError) as e:
        hs.hs_resolve_noalloc(cfg, [z] * 9, [z] * 9, 64, 64, 1, z, z, z, z, z, z, z, None, z, z, None)
    assert e.value.status == hs.HS_ERR_INVALID_CONFIG
