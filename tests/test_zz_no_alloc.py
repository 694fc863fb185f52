"""hs_resolve_noalloc against hs_resolve, through the C ABI, on two decode steps in a row.

hs_resolve_noalloc serves callers that cannot allocate device memory -- engines whose
device memory is fully planned before decoding, plugins living inside another
framework's allocator, processes that must not call cudaMalloc on the decode path. It
needs no hs_create workspace: the library keeps that scratch in its own device array.
Its results must be exactly those of the handle-based hs_resolve (all comparisons here
are bit-exact, like the rest of the parity tests). This file is collected last so a run
that stops at the first failure has run everything else first.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu


def test_noalloc_matches_hs_resolve_on_two_steps():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import hierarchical_sparse_attention_gb300 as hs
    from gpu_harness import GpuSim, host_pools
    from harness import device_pool_model

    wl = W.make("dsa", requests=6, top_k=256, hot_slots=512, steps=2, layers=2,
                seq0=(6000, 7000, 8000, 300, 9000, 10000))  # request 3 takes the fast path
    host = host_pools(wl)
    init = device_pool_model(wl)
    ref = GpuSim(wl, host, init)  # the existing entry point, with its workspace
    try:
        dev = [torch.from_numpy(m.copy()).cuda() for m in init]
        tok0, st0, clk0 = wl.initial_state()
        tok, st, clk = (torch.from_numpy(x).cuda() for x in (tok0, st0, clk0))
        out = torch.full((wl.R, wl.K), -7, dtype=torch.int32, device="cuda")
        miss = torch.full((wl.R,), -7, dtype=torch.int32, device="cuda")
        flags = torch.full((1,), 0x7777, dtype=torch.int32, device="cuda")
        for step in range(2):
            ref.write_newest(step)
            for layer in range(wl.L):  # the same newest-token rows into the second pool
                dev[layer].copy_(ref.dev[layer])
            ref.upload(step)
            ref.resolve()
            hs.hs_resolve_noalloc(ref.cfg, host, dev, wl.host_rows, wl.device_rows, wl.R, ref.tk, ref.sl, ref.hcl,
                                  ref.dbl, tok, st, clk, None, out, miss, flags)
            torch.cuda.synchronize()
            want = ref.state()
            np.testing.assert_array_equal(out.cpu().numpy(), want["out"], err_msg=f"step {step}: out_rows")
            np.testing.assert_array_equal(miss.cpu().numpy(), want["miss"], err_msg=f"step {step}: miss_counts")
            np.testing.assert_array_equal(tok.cpu().numpy(), want["tokens"], err_msg=f"step {step}: slot map")
            np.testing.assert_array_equal(st.cpu().numpy(), want["stamps"], err_msg=f"step {step}: stamps")
            np.testing.assert_array_equal(clk.cpu().numpy(), want["clock"], err_msg=f"step {step}: clock")
            for layer in range(wl.L):
                assert torch.equal(dev[layer], ref.dev[layer]), f"step {step}: device pool layer {layer}"
            assert int(flags.item()) == hs.hs_get_error(ref.h, clear=True) == 0
            assert int(want["miss"][:3].min()) > 0  # the steps did move rows
    finally:
        ref.close()


def test_noalloc_rejects_more_layers_than_its_scratch_holds():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import hierarchical_sparse_attention_gb300 as hs
    cfg = hs.make_config(1, 8, 16, 64, hs.HS_NOALLOC_MAX_LAYERS + 1, 0, 64, 0)
    z = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(hs.HsError) as e:
        hs.hs_resolve_noalloc(cfg, [z] * 9, [z] * 9, 64, 64, 1, z, z, z, z, z, z, z, None, z, z, None)
    assert e.value.status == hs.HS_ERR_INVALID_CONFIG
