"""Pins for the oracle's RMSNorm -> q8_1 producer (CPU only).

RMSNorm against a library rms_norm in f64 and closed forms; the q8_1 quantizer against closed
forms, the half-away tie rule, a brute-force argmin over all 255 codes, and its invariants.
"""
import numpy as np
import pytest
import torch

from quantized_decode_memq_gb300 import synth


def _lib_rmsnorm(x, w, eps):
    xt = torch.from_numpy(np.asarray(x, np.float64))
    wt = torch.from_numpy(np.asarray(w, np.float64))
    return torch.nn.functional.rms_norm(xt, (xt.shape[-1],), weight=wt, eps=eps).numpy()


@pytest.mark.parametrize("rows,ncols", [(1, 32), (3, 64), (2, 4096), (5, 1536)])
def test_rmsnorm_vs_library(oracle, rows, ncols):
    x, w = synth.activation_rows(ncols, rows)
    eps = np.float32(1e-6)
    z = oracle.rmsnorm(x, w, float(eps))
    ref = _lib_rmsnorm(x, w, float(eps))
    np.testing.assert_allclose(z, ref, rtol=1e-13, atol=0)


def test_rmsnorm_closed_forms(oracle):
    # constant row, unit weight, eps = 0 -> z = sign(c)
    for c in (3.0, -0.25, 1e-3):
        x = np.full((1, 64), c, np.float32)
        z = oracle.rmsnorm(x, np.ones(64, np.float32), 0.0)
        np.testing.assert_allclose(z, np.sign(c), rtol=1e-15)
    # alternating +-a with weight k: mean(x^2) = a^2, z = +-a*k/sqrt(a^2 + eps)
    a, k, eps = 2.0, 0.5, np.float32(1e-6)
    x = np.tile(np.array([a, -a], np.float32), 16)[None, :]
    z = oracle.rmsnorm(x, np.full(32, k, np.float32), float(eps))
    expect = np.tile([a * k, -a * k], 16) / np.sqrt(a * a + float(eps))
    np.testing.assert_allclose(z[0], expect, rtol=1e-15)
    # eps enters under the root: x = 0 row gives z = 0 (no division by zero)
    z0 = oracle.rmsnorm(np.zeros((1, 32), np.float32), np.ones(32, np.float32), 1e-6)
    assert np.all(z0 == 0)


def test_rmsnorm_rows_independent(oracle):
    x, w = synth.activation_rows(256, 4)
    z_all = oracle.rmsnorm(x, w)
    for r in range(4):
        np.testing.assert_array_equal(oracle.rmsnorm(x[r:r + 1], w)[0], z_all[r])


def test_quantize_constant_row(oracle):
    z = np.full((1, 64), -1.0)
    d, qs, ratio = oracle.quantize_q8_1(z)
    assert np.all(d == np.float32(1.0 / 127.0))
    assert np.all(qs == -127)


def test_quantize_ties_half_away(oracle):
    # amax = 127 * 2^-3 gives d = 2^-3 exactly, so z/d is exact and hits .5 ties on purpose
    blk = np.zeros(32)
    blk[0] = 127 * 0.125
    vals = [2.5, -2.5, 0.5, -0.5, 1.4999999, 126.5, -3.5, 0.0]
    blk[1:1 + len(vals)] = np.array(vals) * 0.125
    d, qs, ratio = oracle.quantize_q8_1(blk[None, :])
    assert d[0, 0] == np.float32(0.125)
    assert qs[0, 0] == 127
    assert qs[0, 1:1 + len(vals)].tolist() == [3, -3, 1, -1, 1, 127, -4, 0]


def test_quantize_zero_block(oracle):
    z = np.zeros((2, 64))
    z[1, 40] = 5.0
    d, qs, _ = oracle.quantize_q8_1(z)
    assert d[0, 0] == 0 and d[0, 1] == 0 and d[1, 0] == 0
    assert np.all(qs[0] == 0) and np.all(qs[1, :32] == 0)
    assert qs[1, 40] == 127


def test_quantize_bruteforce_argmin(oracle):
    """qs is the code k in [-127, 127] nearest to z/d (ties away from zero), found by trying
    every code -- an enumeration, not a call of a rounding function."""
    x, w = synth.activation_rows(128, 2)
    z = oracle.rmsnorm(x, w)
    d, qs, _ = oracle.quantize_q8_1(z)
    ks = np.arange(-127, 128, dtype=np.float64)
    for r in range(2):
        for i in range(128):
            dd = float(d[r, i // 32])
            err = np.abs(z[r, i] - ks * dd)
            best = np.flatnonzero(err <= err.min() * (1 + 1e-15) + 1e-300)
            k = ks[best[np.argmax(np.abs(ks[best]))]]  # tie -> larger magnitude
            assert qs[r, i] == k


@pytest.mark.parametrize("ncols", [1536, 4096, 8192])
def test_quantize_invariants_page_inputs(oracle, ncols):
    x, w = synth.activation_rows(ncols, 1)
    z, d, qs, ratio = oracle.rmsnorm_q8_1(x, w)
    zb = z.reshape(-1, 32)
    qb = qs.reshape(-1, 32).astype(np.int64)
    db = d.reshape(-1).astype(np.float64)
    assert np.all(np.abs(qb) <= 127)
    amax_idx = np.argmax(np.abs(zb), axis=1)
    rows = np.arange(zb.shape[0])
    assert np.all(np.abs(qb[rows, amax_idx]) == 127)
    assert np.all(np.sign(qb[rows, amax_idx]) == np.sign(zb[rows, amax_idx]))
    assert np.all(np.abs(zb - db[:, None] * qb) <= db[:, None] * (0.5 + 1e-12))
    # d is amax/127 stored as f32
    assert np.array_equal(d.reshape(-1), (np.abs(zb).max(axis=1) / 127.0).astype(np.float32))
    np.testing.assert_array_equal(ratio.reshape(-1, 32), zb / db[:, None])
