"""Pins of the sparse-MLA decode oracle (no GPU): e4m3 landmark codes from the format's
definition, and closed forms of softmax attention."""
import numpy as np
import pytest

from oracle import sparse_mla as M


def test_e4m3_landmarks():
    # 1.0, 2.0, the largest normal 448, the smallest normal 2^-6, the smallest subnormal 2^-9,
    # the largest subnormal 7/8 * 2^-6, negative one, zero, negative zero, and NaN
    codes = np.array([0x38, 0x40, 0x7E, 0x08, 0x01, 0x07, 0xB8, 0x00, 0x80, 0x7F, 0xFF], np.uint8)
    v = M.e4m3_decode(codes)
    assert v[:9].tolist() == [1.0, 2.0, 448.0, 2.0 ** -6, 2.0 ** -9, 7 / 8 * 2.0 ** -6, -1.0, 0.0, 0.0]
    assert np.isnan(v[9]) and np.isnan(v[10])
    # every non-NaN code round-trips through its value's sign, exponent and mantissa
    all_codes = np.arange(256, dtype=np.uint8)
    vals = M.e4m3_decode(all_codes)
    finite = ~np.isnan(vals)
    assert finite.sum() == 254 and np.unique(np.abs(vals[finite])).size == 127  # +0 and -0 share 0


def _rows(rng, n):
    """n fp8 MLA rows of 656 B from the format: codes, 4 fp32 scales, 64 bf16."""
    raw = np.zeros((n, M.ROW_BYTES), np.uint8)
    codes = rng.integers(0, 256, size=(n, 512)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] -= 1
    raw[:, :512] = codes
    raw[:, 512:528] = rng.uniform(2 ** -8, 1, size=(n, 4)).astype("<f4").view(np.uint8)
    rope = (rng.standard_normal((n, 64)).astype(np.float32).view(np.uint32) >> 16).astype("<u2")
    raw[:, 528:] = rope.view(np.uint8)
    return raw.reshape(-1)


def _q(rng, R, Hq):
    return (rng.standard_normal((R, Hq, M.D_QK)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_dequant_layout():
    rng = np.random.default_rng(1)
    pool = _rows(rng, 3)
    latent, rope = M.dequant_rows(pool, np.array([2, 0]))
    raw = pool.reshape(3, -1)
    sc = raw[2, 512:528].copy().view("<f4")
    assert latent[0, 130] == M.e4m3_decode(raw[2, 130:131])[0] * sc[1]  # element 130 uses scale 1
    assert rope[1, 3] == M.bf16_decode(raw[0, 528 + 6:528 + 8].copy().view("<u2"))[0]


def test_single_row_returns_its_latent():
    rng = np.random.default_rng(2)
    pool = _rows(rng, 5)
    q = _q(rng, 1, 4)
    o, lse = M.sparse_mla_decode(q, pool, np.array([[-1, 3, -1]], np.int32), 0.01)
    latent, rope = M.dequant_rows(pool, np.array([3]))
    assert np.allclose(o[0], latent[0][None, :], rtol=0, atol=1e-12)
    qq = M.bf16_decode(q)[0]
    s = 0.01 * (qq[:, :512] @ latent[0] + qq[:, 512:] @ rope[0])
    assert np.allclose(lse[0], s, rtol=0, atol=1e-9)


def test_zero_query_averages_the_rows():
    rng = np.random.default_rng(3)
    pool = _rows(rng, 6)
    q = np.zeros((1, 2, M.D_QK), np.uint16)
    rows = np.array([[0, 5, 2, -1]], np.int32)
    o, lse = M.sparse_mla_decode(q, pool, rows, 0.3)
    latent, _ = M.dequant_rows(pool, np.array([0, 5, 2]))
    assert np.allclose(o[0], latent.mean(0)[None, :], atol=1e-9)
    assert np.allclose(lse[0], np.log(3.0))


def test_duplicated_row_and_permutation_and_masking():
    rng = np.random.default_rng(4)
    pool = _rows(rng, 8)
    q = _q(rng, 1, 3)
    sm = 1.0 / 4000
    o1, l1 = M.sparse_mla_decode(q, pool, np.array([[1, 4, 6]], np.int32), sm)
    o2, l2 = M.sparse_mla_decode(q, pool, np.array([[6, -1, 1, 4, -1]], np.int32), sm)
    assert np.allclose(o1, o2, atol=1e-12) and np.allclose(l1, l2, atol=1e-12)
    # every row twice: the same distribution, log-sum-exp up by log 2
    o3, l3 = M.sparse_mla_decode(q, pool, np.array([[1, 4, 6, 1, 4, 6]], np.int32), sm)
    assert np.allclose(o1, o3, atol=1e-9) and np.allclose(l3, l1 + np.log(2.0), atol=1e-9)


def test_empty_row_table():
    rng = np.random.default_rng(5)
    pool = _rows(rng, 2)
    o, lse = M.sparse_mla_decode(_q(rng, 2, 2), pool, np.full((2, 3), -1, np.int32), 0.1)
    assert not o.any() and np.all(np.isneginf(lse))


def test_dominant_row():
    """One score far above the rest: the output is that row's latent."""
    rng = np.random.default_rng(6)
    pool = _rows(rng, 4)
    latent, rope = M.dequant_rows(pool, np.arange(4))
    # a query aligned with row 2's latent and scaled up: row 2 dominates the softmax
    qf = np.zeros((1, 1, M.D_QK), np.float32)
    qf[0, 0, :512] = latent[2] / np.abs(latent[2]).max()
    q = (qf.view(np.uint32) >> 16).astype(np.uint16)
    o, _ = M.sparse_mla_decode(q, pool, np.array([[0, 1, 2, 3]], np.int32), 1.0)
    assert np.allclose(o[0, 0], latent[2], rtol=1e-6, atol=1e-6)


def test_disjoint_halves_merge_by_log_sum_exp():
    """Attention over a row set equals the log-sum-exp merge of attention over any two disjoint
    parts of it (the identity the split kernels and their merge rely on): a slip in the oracle's
    normalisation or its lse (a missing log z, a sum over the wrong axis) breaks it."""
    rng = np.random.default_rng(7)
    pool = _rows(rng, 40)
    q = _q(rng, 2, 5)
    sm = 1.0 / 900
    rows = rng.permutation(40)[:24].astype(np.int32).reshape(2, 12)
    o, lse = M.sparse_mla_decode(q, pool, rows, sm)
    oa, la = M.sparse_mla_decode(q, pool, rows[:, :5], sm)
    ob, lb = M.sparse_mla_decode(q, pool, rows[:, 5:], sm)
    lm = np.logaddexp(la, lb)
    om = np.exp(la - lm)[..., None] * oa + np.exp(lb - lm)[..., None] * ob
    assert np.allclose(lse, lm, rtol=0, atol=1e-9)
    assert np.allclose(o, om, rtol=0, atol=1e-9 * np.abs(o).max())
