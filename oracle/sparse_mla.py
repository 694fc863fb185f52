"""CPU ORACLE of a sparse-MLA decode attention over the resolver's row table -- TEST
INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline leg may import it; the library never does. Plain numpy in float64; a matmul
and an exp are the only library steps.

Sources (page title, section):
  "vLLM Hybrid HiSparse source implementation analysis", 7.3 (the resolver's output is a
    table of physical rows; the sparse attention kernel reads the pool's flat view through
    it) and 9 (an fp8 sparse-MLA row is 656 B: 512 B of e4m3 latent ("NoPE"), 16 B of scales,
    128 B of RoPE).
  "HiSparse: Turbocharging Sparse Attention with Hierarchical Memory" and the decode launch
    line in the same page: decode attention only over the top-k positions, through the
    sparse MLA backend.

What it computes, per request r and query head h, over the valid entries j of out_rows[r]
(-1 entries are left out):
  latent_j[d] = e4m3(code_j[d]) * scale_j[d // 128]    d < 512   (the row's first 512 B,
                                                                  then 4 fp32 scales)
  rope_j[e]   = bf16(rope_j[e])                         e < 64    (the row's last 128 B)
  s[h, j]     = sm_scale * (q[h, :512] . latent_j + q[h, 512:] . rope_j)
  p[h, :]     = softmax_j(s[h, :]),  o[h, :] = sum_j p[h, j] latent_j,  lse[h] = log sum_j exp s
With no valid entry, o = 0 and lse = -inf. (MLA decode with the absorbed projection: keys
are the 576-dim rows, values their 512-dim latent part.)

Parity pins (tests/test_oracle_sparse_mla.py): e4m3 decode of the format's landmark codes,
attention closed forms (one row, uniform scores, duplicated rows, masking, permutation, one
dominant row), and the log-sum-exp merge of two disjoint parts of a row set into the whole.
"""
from __future__ import annotations

import numpy as np

ROW_BYTES = 656
D_LATENT, D_ROPE = 512, 64
D_QK = D_LATENT + D_ROPE
SCALE_BLOCK = 128


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """OCP FP8 E4M3: sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is
    subnormal (m / 8 * 2^-6); the all-ones exponent with mantissa 7 is NaN (no infinity)."""
    c = codes.astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = np.where((e == 0xF) & (m == 7), np.nan, val)
    return sign * val


def bf16_decode(bits: np.ndarray) -> np.ndarray:
    """bfloat16 = the top 16 bits of an IEEE float32."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def dequant_rows(pool: np.ndarray, rows: np.ndarray):
    """(latent [n, 512], rope [n, 64]) of the given rows of a flat fp8 MLA pool."""
    raw = pool.reshape(-1, ROW_BYTES)[rows]
    codes = raw[:, :D_LATENT]
    scales = raw[:, D_LATENT:D_LATENT + 16].copy().view("<f4").astype(np.float64)  # [n, 4]
    rope = bf16_decode(raw[:, D_LATENT + 16:].copy().view("<u2"))
    latent = e4m3_decode(codes) * np.repeat(scales, SCALE_BLOCK, axis=1)
    return latent, rope


def sparse_mla_decode(q_bits: np.ndarray, pool: np.ndarray, out_rows: np.ndarray, sm_scale: float):
    """q_bits [R, Hq, 576] bfloat16 bit patterns (uint16), pool: flat uint8 fp8 MLA rows,
    out_rows [R, K] (row or -1). Returns (o [R, Hq, 512], lse [R, Hq]) in float64."""
    R, Hq, _ = q_bits.shape
    q = bf16_decode(q_bits)
    o = np.zeros((R, Hq, D_LATENT))
    lse = np.full((R, Hq), -np.inf)
    for r in range(R):
        rows = out_rows[r][out_rows[r] >= 0].astype(np.int64)
        if rows.size == 0:
            continue
        latent, rope = dequant_rows(pool, rows)
        s = sm_scale * (q[r, :, :D_LATENT] @ latent.T + q[r, :, D_LATENT:] @ rope.T)  # [Hq, n]
        smax = s.max(axis=1, keepdims=True)
        e = np.exp(s - smax)
        z = e.sum(axis=1, keepdims=True)
        o[r] = (e / z) @ latent
        lse[r] = (smax + np.log(z))[:, 0]
    return o, lse
