"""GPU parity of the synthetic consumer (hs_sparse_mla_decode: sparse-MLA decode attention over
the resolver's row table, on the tcgen05 tensor cores) against the oracle.

Two comparisons per output:
* tight: against the oracle's formula evaluated in the kernel's precision (q and RoPE converted
  from bf16 to fp16, the scale rounded to fp16 and each latent code times it rounded to fp16,
  P rounded to fp16 before the product). The kernel rounds P against each block's running
  maximum, the model against the final one, so the two roundings of a weight may differ by
  2^-10 (relative): |d o| <= 2^-10 * max|v_j - o| <= 2^-9 * max|latent|; with fp32
  accumulation and exp2 on top, the test allows 3e-3 * max|latent| per element;
* rigorous: against the exact oracle (float64), a first-order bound of the fp16 rounding with
  U = 2^-10 (two fp16 roundings in each latent value, one in each weight):
  |d o_i| <= 2 * max_j |v_ji| * (3 U + 4 E), E = max_j sm_scale * U * sum_d |q_d v_jd|
  (score error from rounding v; the factor 2 covers second-order terms), and |d lse| <= 2 E + 4 U.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads as W  # noqa: E402
from oracle import sparse_mla as M  # noqa: E402

pytestmark = pytest.mark.gpu
U = 2.0 ** -10


def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import hierarchical_sparse_attention_gb300 as hs
    return hs


def _f16(x):
    """Round to the nearest fp16 (ties to even), as the kernel's conversions do."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def model(q_bits, pool, out_rows, sm_scale):
    """The oracle's formula in the kernel's precision (see the module docstring)."""
    R, Hq, _ = q_bits.shape
    q = _f16(M.bf16_decode(q_bits))
    o = np.zeros((R, Hq, M.D_LATENT))
    for r in range(R):
        rows = out_rows[r][out_rows[r] >= 0].astype(np.int64)
        if rows.size == 0:
            continue
        raw = pool.reshape(-1, M.ROW_BYTES)[rows]
        sc = raw[:, 512:528].copy().view("<f4")
        lat = _f16(M.e4m3_decode(raw[:, :512]) * np.repeat(_f16(sc), 128, axis=1))
        rope = _f16(M.bf16_decode(raw[:, 528:].copy().view("<u2")))
        s = sm_scale * (q[r, :, :512] @ lat.T + q[r, :, 512:] @ rope.T)
        p = _f16(np.exp(s - s.max(1, keepdims=True)))
        o[r] = (p @ lat) / p.sum(1, keepdims=True)
    return o


def make_case(seed, R, Hq, K, pool_rows, masked=0.1, bad_rows=0):
    wl = W.make("dsa", seed, requests=R, top_k=min(K, 2048), steps=2)
    rng = np.random.default_rng(seed)
    toks = rng.integers(0, 100000, size=pool_rows)
    pool = np.concatenate([wl.rows(0, 0, [int(t)]) for t in toks]).reshape(-1).astype(np.uint8)
    out_rows = rng.integers(0, pool_rows, size=(R, K)).astype(np.int32)
    out_rows[rng.random((R, K)) < masked] = -1
    if bad_rows:
        out_rows[0, :bad_rows] = pool_rows + 5  # outside the pool: counted as -1
    q = wl.queries_bf16(0, Hq)
    # a scale that gives the synthetic scores about unit spread (uniform e4m3 codes make raw
    # scores of order 1e3)
    lat, rope = M.dequant_rows(pool, np.arange(min(pool_rows, 64)))
    qq = M.bf16_decode(q[0])
    raw = qq[:, :512] @ lat.T + qq[:, 512:] @ rope.T
    sm_scale = float(np.float32(1.0 / raw.std()))
    return q, pool, out_rows, sm_scale


def run_gpu(hs, q, pool, out_rows, sm_scale, splits):
    R, Hq, _ = q.shape
    K = out_rows.shape[1]
    d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()  # noqa: E731
    g_q, g_pool, g_rows = d(q.view(np.int16)), d(pool), d(out_rows)
    o = torch.full((R, Hq, 512), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((R, Hq), float("nan"), dtype=torch.float32, device="cuda")
    wsb = hs.hs_sparse_mla_workspace_bytes(R, Hq, splits)
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hs.hs_sparse_mla_decode(R, Hq, K, splits, g_q, g_pool, pool.size // 656, g_rows, sm_scale, o, lse, ws, wsb, err)
    torch.cuda.synchronize()
    return o.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), int(err.item())


def check(q, pool, out_rows, sm_scale, go, glse, what):
    ro = out_rows.copy()
    ro[(ro < 0) | (ro >= pool.size // 656)] = -1
    o, lse = M.sparse_mla_decode(q, pool, ro, sm_scale)
    mo = model(q, pool, ro, sm_scale)
    qf = M.bf16_decode(q)
    for r in range(q.shape[0]):
        rows = ro[r][ro[r] >= 0].astype(np.int64)
        if rows.size == 0:
            assert np.all(go[r] == 0) and np.all(np.isneginf(glse[r])), f"{what}: empty request {r}"
            continue
        lat, _ = M.dequant_rows(pool, rows)
        vmax = np.abs(lat).max(0)  # per value dim
        E = sm_scale * U * (np.abs(qf[r, :, :512]) @ np.abs(lat).T).max(1)  # per head
        tight = np.abs(go[r] - mo[r]).max()
        assert tight <= 3e-3 * np.abs(lat).max(), f"{what}: request {r} differs from the precision model by {tight}"
        bound = 2 * vmax[None, :] * (3 * U + 4 * E[:, None])
        assert np.all(np.abs(go[r] - o[r]) <= bound + 1e-6), f"{what}: request {r} outside the rounding bound"
        assert np.all(np.abs(glse[r] - lse[r]) <= 2 * E + 4 * U), f"{what}: request {r} lse"


@pytest.mark.parametrize("R,Hq,K,splits", [(2, 128, 256, 1), (3, 128, 2048, 2), (2, 64, 100, 1), (1, 16, 333, 4),
                                           (4, 128, 1024, 4),
                                           (2, 128, 600, 16),  # the most splits: two blocks each
                                           (2, 128, 5, 16),    # most splits hold no row at all
                                           (2, 48, 300, 2),    # two splits, heads not a multiple of 32
                                           (3, 16, 1, 2),      # two splits, the second empty
                                           (64, 128, 512, 2)])  # two splits, more requests than four-CTA clusters fit at once
def test_sparse_mla_matches_oracle(R, Hq, K, splits):
    hs = _gpu()
    q, pool, out_rows, sm = make_case(R * 7 + K, R, Hq, K, pool_rows=3000)
    go, glse, err = run_gpu(hs, q, pool, out_rows, sm, splits)
    assert err == 0
    check(q, pool, out_rows, sm, go, glse, f"R{R} H{Hq} K{K} splits{splits}")


def test_sparse_mla_masked_and_out_of_pool_rows():
    hs = _gpu()
    q, pool, out_rows, sm = make_case(5, 3, 128, 200, pool_rows=500, masked=0.5, bad_rows=17)
    out_rows[2, :] = -1  # a request with no valid row: o = 0, lse = -inf
    go, glse, err = run_gpu(hs, q, pool, out_rows, sm, 2)
    assert err == 0
    check(q, pool, out_rows, sm, go, glse, "masked")


def test_sparse_mla_reads_the_resolvers_rows():
    """The consumer over the row table and device pool a decode step of the resolver left."""
    hs = _gpu()
    from gpu_harness import close_pair, make_pair
    from harness import poison_host_newest
    wl = W.make("dsa", 3, requests=3, top_k=512, hot_slots=1024, steps=4, seq0=(6000, 9000, 700))
    orc, gpu = make_pair(wl)
    try:
        for step in range(wl.steps):
            gpu.write_newest(step)
            orc.write_newest(step)
            poison_host_newest(wl, step, gpu.host)
            poison_host_newest(wl, step, orc.host)
            gpu.upload(step)
            gpu.resolve()
            gpu.backup()
            orc.resolve(step)
            orc.backup(step)
        torch.cuda.synchronize()
        assert np.array_equal(gpu.out.cpu().numpy(), orc.out)
        q = wl.queries_bf16(wl.steps, 128)
        pool = orc.dev[0]
        lat, rope = M.dequant_rows(pool, orc.out[0][orc.out[0] >= 0][:64])
        qq = M.bf16_decode(q[0])
        sm = float(np.float32(1.0 / (qq[:, :512] @ lat.T + qq[:, 512:] @ rope.T).std()))
        R, Hq, K = wl.R, 128, wl.K
        o = torch.zeros((R, Hq, 512), dtype=torch.float32, device="cuda")
        lse = torch.zeros((R, Hq), dtype=torch.float32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        wsb = hs.hs_sparse_mla_workspace_bytes(R, Hq, 2)
        ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
        hs.hs_sparse_mla_decode(R, Hq, K, 2, torch.from_numpy(q.view(np.int16)).cuda(), gpu.dev[0], wl.device_rows,
                                gpu.out, sm, o, lse, ws, wsb, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        check(q, pool, orc.out, sm, o.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
              "after the resolver")
    finally:
        close_pair(gpu)


def _distinct_rows_case(seed, R, Hq, K, pool_rows, sm_scale=None):
    """R requests of K distinct valid rows each from a pool of fp8 MLA rows (as a resolved
    step gives them: every entry a row, no two alike), seeded N(0, 1) queries."""
    wl = W.make("dsa", seed, requests=R, top_k=min(K, 2048), steps=2)
    rng = np.random.default_rng(seed)
    pool = wl.rows(0, 0, rng.integers(0, 1 << 20, size=pool_rows).astype(np.int32)).reshape(-1)
    out_rows = np.stack([rng.choice(pool_rows, size=K, replace=False) for _ in range(R)]).astype(np.int32)
    q = wl.queries_bf16(0, Hq)
    if sm_scale is None:
        lat, rope = M.dequant_rows(pool, np.arange(64))
        qq = M.bf16_decode(q[0])
        sm_scale = float(np.float32(1.0 / (qq[:, :512] @ lat.T + qq[:, 512:] @ rope.T).std()))
    return q, pool, out_rows, sm_scale


def test_sparse_mla_bench_shape_one_split():
    """The shape the consumer is timed at: 32 requests x 128 heads x 2,048 rows in one split,
    i.e. 32 blocks of 64 rows per CTA through the three-tile ring, with the staged row table
    at its 2,048-entry limit; the bench's sm_scale 1/1400 and the tests' unit-spread scale."""
    hs = _gpu()
    for sm in (1.0 / 1400, None):
        q, pool, out_rows, scale = _distinct_rows_case(31, 32, 128, 2048, pool_rows=32 * 2048 + 4096, sm_scale=sm)
        go, glse, err = run_gpu(hs, q, pool, out_rows, scale, 1)
        assert err == 0
        check(q, pool, out_rows, scale, go, glse, f"32 x 128 x 2048, 1 split, sm_scale {scale:.3g}")


def test_sparse_mla_bench_shape_two_splits():
    """The same shape in two splits of 1,024 rows: the split pairs of a request run as one
    four-CTA cluster and merge inside the kernel."""
    hs = _gpu()
    assert hs.hs_sparse_mla_launches(32, 128, 2) == 1  # merged inside the kernel: no second launch
    q, pool, out_rows, scale = _distinct_rows_case(33, 32, 128, 2048, pool_rows=32 * 2048 + 4096, sm_scale=1.0 / 1400)
    go, glse, err = run_gpu(hs, q, pool, out_rows, scale, 2)
    assert err == 0
    check(q, pool, out_rows, scale, go, glse, "32 x 128 x 2048, 2 splits")


def test_sparse_mla_top_k_4096_one_split():
    """4,096 rows in one split: more than the staged row table holds, so the producers read
    the split's rows from global memory; 64 blocks per CTA."""
    hs = _gpu()
    q, pool, out_rows, sm = _distinct_rows_case(32, 4, 128, 4096, pool_rows=20000)
    out_rows[1, ::7] = -1  # masked entries spread over the table
    go, glse, err = run_gpu(hs, q, pool, out_rows, sm, 1)
    assert err == 0
    check(q, pool, out_rows, sm, go, glse, "top_k 4096, 1 split")


_CAPTURE_SCRIPT = r"""
import sys
import numpy as np
import torch
sys.path[:0] = [sys.argv[1], sys.argv[2]]
import test_gpu_sparse_mla as T
import hierarchical_sparse_attention_gb300 as hs
R, Hq, K, splits = 4, 128, 700, 2
q, pool, out_rows, sm = T.make_case(11, R, Hq, K, pool_rows=3000)
d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
g_q, g_pool, g_rows = d(q.view(np.int16)), d(pool), d(out_rows)
wsb = hs.hs_sparse_mla_workspace_bytes(R, Hq, splits)
res = []
for mode in ("graph", "eager"):
    o = torch.full((R, Hq, 512), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((R, Hq), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = (R, Hq, K, splits, g_q, g_pool, pool.size // 656, g_rows, sm, o, lse, ws, wsb, err)
    torch.cuda.synchronize()
    if mode == "graph":
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            hs.hs_sparse_mla_decode(*args, stream=s)
        g.replay()
    else:
        hs.hs_sparse_mla_decode(*args)
    torch.cuda.synchronize()
    res.append((o.cpu(), lse.cpu(), int(err.item())))
(go, gl, ge), (eo, el, ee) = res
assert ge == 0 and ee == 0, (ge, ee)
assert torch.equal(go, eo) and torch.equal(gl, el), "graph replay differs from the eager call"
print("ok")
"""


def test_sparse_mla_first_call_inside_a_graph_capture():
    """The process's first consumer call is made while a stream is being captured (the launch
    shape is chosen then): the replayed graph gives the eager call's outputs bit for bit."""
    _gpu()
    import os
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    root = os.path.dirname(here)
    p = subprocess.run([sys.executable, "-c", _CAPTURE_SCRIPT, here, root], cwd=root, capture_output=True, text=True,
                       timeout=300)
    assert p.returncode == 0 and p.stdout.strip().endswith("ok"), p.stdout[-2000:] + p.stderr[-2000:]


def test_sparse_mla_in_kernel_merge_matches_the_merge_kernel():
    """Two splits over the same 32 requests, once as the first 32 of 64 (more four-CTA clusters
    than fit at once: two-CTA pairs and the merge kernel) and once alone (four-CTA clusters
    merging inside the kernel): the same partial outputs, merged with the same arithmetic, so
    the outputs agree to rounding."""
    hs = _gpu()
    assert hs.hs_sparse_mla_launches(64, 128, 2) == 2  # 256 CTAs in clusters of four: the merge kernel
    q, pool, out_rows, sm = _distinct_rows_case(34, 64, 128, 512, pool_rows=40000)
    o64, l64, e64 = run_gpu(hs, q, pool, out_rows, sm, 2)
    o32, l32, e32 = run_gpu(hs, q[:32], pool, out_rows[:32], sm, 2)
    assert e64 == 0 and e32 == 0
    scale = float(np.abs(o64[:32]).max())
    assert np.abs(o32 - o64[:32]).max() <= 1e-6 * scale, "in-kernel merge differs from the merge kernel"
    assert np.abs(l32 - l64[:32]).max() <= 1e-6
    check(q[:32], pool, out_rows[:32], sm, o32, l32, "32 x 128 x 512, 2 splits, merged inside")
