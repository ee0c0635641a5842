"""Pins for the oracle's three GEMVs (CPU only).

Each container is dequantized here with library decoders (torch float8_e4m3fn, numpy float16)
and contracted with a library matmul; the oracle must match to f64 rounding.  Identities that
hold exactly (one-hot activations, sign flips, zero weights, a constant block grid equal to a
per-tensor scale, and E4M3/Q8_0 encodings of the same small integers) pin the rest.
"""
import numpy as np
import pytest
import torch

from quantized_decode_memq_gb300 import synth


def _act(oracle, m, in_f, seed=7):
    x = synth.uniform_pm4(seed, m * in_f).reshape(m, in_f)
    w = synth.uniform_pm4(seed + 1, in_f)
    _, d, qs, _ = oracle.rmsnorm_q8_1(x, w)
    return qs, d


def _x_deq(qs, d):
    m, in_f = qs.shape
    return np.repeat(d.astype(np.float64), 32, axis=1) * qs.astype(np.float64)


def _e4m3_lib(wbytes):
    t = torch.from_numpy(np.ascontiguousarray(wbytes)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def _q8_0_lib(wbytes, in_f):
    out_f = wbytes.shape[0]
    blk = wbytes.reshape(out_f, in_f // 32, 34)
    dw = np.ascontiguousarray(blk[:, :, 0:2]).view(np.float16)[:, :, 0].astype(np.float64)
    q = np.ascontiguousarray(blk[:, :, 2:]).view(np.int8).astype(np.float64)
    return (dw[:, :, None] * q).reshape(out_f, in_f)


def _close(y, ref, s, rel=1e-12):
    assert y.shape == ref.shape
    assert np.all(np.abs(y - ref) <= rel * s + 1e-300), np.max(np.abs(y - ref) / s)


SHAPES = [(32, 64, 1), (37, 96, 3), (130, 160, 8), (5, 4096 + 32, 2)]


@pytest.mark.parametrize("out_f,in_f,m", SHAPES)
def test_e4m3_vs_library_matmul(oracle, out_f, in_f, m):
    w = synth.e4m3_bytes(11, out_f, in_f)
    qs, d = _act(oracle, m, in_f)
    scale = 2.0 ** -4
    y, s = oracle.gemv_e4m3(w, scale, qs, d)
    ref = _x_deq(qs, d) @ (scale * _e4m3_lib(w)).T
    _close(y, ref, s)
    sref = np.abs(_x_deq(qs, d)) @ np.abs(scale * _e4m3_lib(w)).T
    np.testing.assert_allclose(s, sref, rtol=1e-12)


@pytest.mark.parametrize("out_f,in_f,m", SHAPES)
def test_blk128_vs_library_matmul(oracle, out_f, in_f, m):
    w = synth.e4m3_bytes(12, out_f, in_f)
    grid = synth.grid_log2_uniform(13, out_f, in_f)
    qs, d = _act(oracle, m, in_f)
    y, s = oracle.gemv_e4m3_blk128(w, grid, qs, d)
    g = np.repeat(np.repeat(grid.astype(np.float64), 128, axis=0), 128, axis=1)[:out_f, :in_f]
    ref = _x_deq(qs, d) @ (g * _e4m3_lib(w)).T
    _close(y, ref, s)


@pytest.mark.parametrize("out_f,in_f,m", SHAPES)
def test_q8_0_vs_library_matmul(oracle, out_f, in_f, m):
    w = synth.q8_0_bytes(14, out_f, in_f)
    qs, d = _act(oracle, m, in_f)
    y, s = oracle.gemv_q8_0(w, in_f, qs, d)
    ref = _x_deq(qs, d) @ _q8_0_lib(w, in_f).T
    _close(y, ref, s)


def test_page_generators_vs_library(oracle):
    out_f, in_f = 48, 256
    qs, d = _act(oracle, 1, in_f)
    w = synth.lcg_e4m3(out_f, in_f)
    y, s = oracle.gemv_e4m3(w, 0.0625, qs, d)
    _close(y, _x_deq(qs, d) @ (0.0625 * _e4m3_lib(w)).T, s)
    grid = synth.lcg_blk_grid(out_f, in_f)
    y, s = oracle.gemv_e4m3_blk128(w, grid, qs, d)
    g = np.repeat(np.repeat(grid.astype(np.float64), 128, 0), 128, 1)[:out_f, :in_f]
    _close(y, _x_deq(qs, d) @ (g * _e4m3_lib(w)).T, s)
    wq = synth.lcg_q8_0(out_f, in_f)  # includes qs = -128
    assert (wq.reshape(-1, 34)[:, 2:].view(np.int8) == -128).any()
    y, s = oracle.gemv_q8_0(wq, in_f, qs, d)
    _close(y, _x_deq(qs, d) @ _q8_0_lib(wq, in_f).T, s)


def test_one_hot_activation(oracle):
    out_f, in_f = 40, 128
    w = synth.e4m3_bytes(21, out_f, in_f)
    grid = synth.grid_log2_uniform(22, out_f, in_f)
    wq = synth.q8_0_bytes(23, out_f, in_f)
    col = 77
    qs = np.zeros((1, in_f), np.int8)
    qs[0, col] = -5
    d = np.full((1, in_f // 32), 0.25, np.float32)
    tab = oracle.e4m3_table()
    y, _ = oracle.gemv_e4m3(w, 0.5, qs, d)
    np.testing.assert_array_equal(y[0], 0.5 * tab[w[:, col]] * (0.25 * -5))
    y, _ = oracle.gemv_e4m3_blk128(w, grid, qs, d)
    np.testing.assert_array_equal(y[0], grid[np.arange(out_f) // 128, col // 128]
                                  .astype(np.float64) * tab[w[:, col]] * (0.25 * -5))
    y, _ = oracle.gemv_q8_0(wq, in_f, qs, d)
    blk = wq.reshape(out_f, in_f // 32, 34)[:, col // 32]
    dw = oracle.f16_decode(blk[:, 0].astype(np.uint16) | (blk[:, 1].astype(np.uint16) << 8))
    qw = blk[:, 2 + col % 32].view(np.int8).astype(np.float64)
    np.testing.assert_array_equal(y[0], dw * qw * (0.25 * -5))


def test_sign_flip_and_zero(oracle):
    out_f, in_f, m = 33, 192, 4
    w = synth.e4m3_bytes(31, out_f, in_f)
    grid = synth.grid_log2_uniform(32, out_f, in_f)
    qs, d = _act(oracle, m, in_f)
    y, _ = oracle.gemv_e4m3(w, 1.0, qs, d)
    yn, _ = oracle.gemv_e4m3(w ^ 0x80, 1.0, qs, d)
    np.testing.assert_array_equal(yn, -y)
    y, _ = oracle.gemv_e4m3_blk128(w, grid, qs, d)
    yn, _ = oracle.gemv_e4m3_blk128(w ^ 0x80, grid, qs, d)
    np.testing.assert_array_equal(yn, -y)
    # negating the activation negates y
    yq, _ = oracle.gemv_e4m3(w, 1.0, -qs, d)
    y1, _ = oracle.gemv_e4m3(w, 1.0, qs, d)
    np.testing.assert_array_equal(yq, -y1)
    z, _ = oracle.gemv_e4m3(np.zeros_like(w), 1.0, qs, d)
    assert np.all(z == 0)
    wq = synth.q8_0_bytes(33, out_f, in_f)
    wq.reshape(-1, 34)[:, 2:] = 0
    z, _ = oracle.gemv_q8_0(wq, in_f, qs, d)
    assert np.all(z == 0)


def test_constant_grid_equals_per_tensor(oracle):
    out_f, in_f, m = 200, 300 - 300 % 32, 2
    w = synth.e4m3_bytes(41, out_f, in_f)
    qs, d = _act(oracle, m, in_f)
    g = np.full(((out_f + 127) // 128, (in_f + 127) // 128), 0.375, np.float32)
    yb, _ = oracle.gemv_e4m3_blk128(w, g, qs, d)
    ye, _ = oracle.gemv_e4m3(w, 0.375, qs, d)
    np.testing.assert_array_equal(yb, ye)


def test_grid_tile_indexing(oracle):
    """Each (128-row, 128-col) tile of the grid scales exactly its own tile of W: scaling one
    grid entry by 2 changes only the rows of its row tile, by exactly that tile's part."""
    out_f, in_f = 260, 4096 + 32
    w = synth.e4m3_bytes(51, out_f, in_f)
    grid = synth.grid_log2_uniform(52, out_f, in_f)
    qs, d = _act(oracle, 1, in_f)
    y0, _ = oracle.gemv_e4m3_blk128(w, grid, qs, d)
    g2 = grid.copy()
    g2[2, 32] *= 2  # the partial edge tile (rows 256..259, cols 4096..4127)
    y1, _ = oracle.gemv_e4m3_blk128(w, g2, qs, d)
    assert np.array_equal(y0[0, :256], y1[0, :256])
    tab = oracle.e4m3_table()
    xd = _x_deq(qs, d)[0]
    part = (grid[2, 32] * tab[w[256:, 4096:]] * xd[4096:]).sum(axis=1)
    np.testing.assert_allclose(y1[0, 256:] - y0[0, 256:], part, rtol=1e-9, atol=1e-12)


def test_cross_container_identity(oracle):
    """Weights k * 2^-j with |k| <= 16 are exact in E4M3 and in Q8_0 (scale 2^-j, qs = k), so
    the two oracles give identical results."""
    out_f, in_f, m, j = 24, 256, 3, 5
    rng = np.random.default_rng(5)
    k = rng.integers(-16, 17, size=(out_f, in_f))
    tab = oracle.e4m3_table()
    lookup = {}
    for c in range(256):
        if not np.isnan(tab[c]):
            lookup.setdefault(tab[c], c)
    w8 = np.vectorize(lambda v: lookup[v * 2.0 ** -j])(k).astype(np.uint8)
    assert np.array_equal(tab[w8], k * 2.0 ** -j)
    nb = in_f // 32
    blocks = np.zeros((out_f * nb, 34), np.uint8)
    blocks[:, 0:2] = np.array([2.0 ** -j], np.float16).view(np.uint8)
    blocks[:, 2:] = k.reshape(out_f * nb, 32).astype(np.int8).view(np.uint8)
    wq = blocks.reshape(out_f, nb * 34)
    qs, d = _act(oracle, m, in_f)
    ye, _ = oracle.gemv_e4m3(w8, 1.0, qs, d)
    yq, _ = oracle.gemv_q8_0(wq, in_f, qs, d)
    np.testing.assert_array_equal(ye, yq)


def test_row_sampling_matches_full(oracle):
    out_f, in_f, m = 50, 128, 2
    w = synth.e4m3_bytes(61, out_f, in_f)
    qs, d = _act(oracle, m, in_f)
    y, s = oracle.gemv_e4m3(w, 1.0, qs, d)
    rows = np.array([49, 0, 17, 17])
    ys, ss = oracle.gemv_e4m3(w, 1.0, qs, d, rows=rows)
    np.testing.assert_array_equal(ys, y[:, rows])
    np.testing.assert_array_equal(ss, s[:, rows])
