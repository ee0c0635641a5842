"""Pins of the oracle's next-row functions: the silu(gate)*up -> q8_1 producer (q8_fuse_gate.rs,
`main`, the expert-ff site) and the E4M3 -> Q8_0 load-time repack (gemv_e4m3_bench.rs, module
doc "QUESTION", "ARM B'").  Each is checked against something other than itself: library
routines (scipy's logistic function, numpy's float16 conversion, torch's float8 decode), closed
forms and identities, and brute force over every Q8_0 code."""
import numpy as np
import pytest
import torch

from quantized_decode_memq_gb300 import synth


# ----------------------------------------------------------------------------------- silu
def test_silu_identity_and_zero(oracle):
    x = synth.uniform_pm4(0x5110, 4096).astype(np.float32) * np.float32(4)
    one = np.ones_like(x)
    zp = oracle.silu_mul(x, one)[0]
    zn = oracle.silu_mul(-x, one)[0]
    # silu(x) - silu(-x) = x * (sigma(x) + sigma(-x)) = x
    np.testing.assert_allclose(zp - zn, x.astype(np.float64), rtol=1e-14, atol=1e-300)
    assert oracle.silu_mul(np.zeros(32, np.float32), np.ones(32, np.float32))[0].tolist() == [0.0] * 32


def test_silu_against_library_logistic(oracle):
    scipy_special = pytest.importorskip("scipy.special")
    g = synth.uniform_pm4(0x5111, 8192).astype(np.float32) * np.float32(8)
    u = synth.uniform_pm4(0x5112, 8192).astype(np.float32)
    ref = g.astype(np.float64) * scipy_special.expit(g.astype(np.float64)) * u.astype(np.float64)
    np.testing.assert_allclose(oracle.silu_mul(g, u)[0], ref, rtol=1e-14, atol=1e-300)
    # saturation: silu(-1000) = -0, silu(1000) = 1000
    z = oracle.silu_mul(np.array([-1000.0, 1000.0] + [0.0] * 30, np.float32), np.ones(32, np.float32))[0]
    assert z[0] == 0.0 and z[1] == 1000.0


def test_silu_producer_quantizes_its_z(oracle):
    g = synth.uniform_pm4(0x5113, 2 * 1536).reshape(2, 1536)
    u = synth.uniform_pm4(0x5114, 2 * 1536).reshape(2, 1536)
    z, d, qs, ratio = oracle.silu_mul_q8_1(g, u)
    d2, qs2, _ = oracle.quantize_q8_1(oracle.silu_mul(g, u))
    assert np.array_equal(d, d2) and np.array_equal(qs, qs2)
    blocks = np.abs(z).reshape(2, -1, 32)
    assert np.all(np.abs(qs) <= 127)
    amax_pos = blocks.argmax(axis=2)
    q = np.abs(qs.reshape(2, -1, 32))
    assert np.all(np.take_along_axis(q, amax_pos[..., None], 2) == 127)


# ----------------------------------------------------------------------------------- f16
def test_f16_rounding_matches_numpy_on_every_value_and_midpoint(oracle):
    h = np.arange(0, 0x7C00, dtype=np.uint16)          # every finite non-negative f16
    v = h.view(np.float16).astype(np.float64)
    mids = (v[:-1] + v[1:]) / 2                          # exact ties between neighbours
    cases = np.concatenate([v, mids, -mids[::97], [65519.0, 65520.0, 70000.0, 2.0 ** -26]])
    with np.errstate(over="ignore"):
        expect = cases.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.f16_bits(cases), expect)


def test_f16_rounding_random_f32(oracle):
    rng = np.random.default_rng(7)
    v = (2.0 ** rng.uniform(-30, 16, 20000)).astype(np.float32).astype(np.float64)
    v *= np.where(rng.random(v.size) < 0.5, -1.0, 1.0)
    assert np.array_equal(oracle.f16_bits(v), v.astype(np.float16).view(np.uint16))


# ----------------------------------------------------------------------------------- repack
def dequant_e4m3(w, aux, grid):
    """Library decode (torch float8_e4m3fn -> f32) times the scale, in f32."""
    wf = torch.from_numpy(w).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    out_f, in_f = w.shape
    if grid:
        s = np.repeat(np.repeat(aux, 128, 0), 128, 1)[:out_f, :in_f].astype(np.float32)
    else:
        s = np.float32(aux[0])
    return (wf * s).astype(np.float32)     # one f32 rounding per product


def unpack_q8_0(slab, in_f):
    out_f = slab.shape[0]
    b = slab.reshape(out_f, in_f // 32, 34)
    d16 = b[..., :2].copy().view(np.float16)[..., 0]
    qs = b[..., 2:].view(np.int8)
    return d16, qs


@pytest.mark.parametrize("grid", [False, True])
def test_repack_codes_are_the_nearest(oracle, grid):
    out_f, in_f = 130, 4096 + 32
    w = synth.e4m3_bytes(0x5201 + grid, out_f, in_f)
    aux = synth.grid_log2_uniform(0x5203, out_f, in_f) if grid else np.array([2.0 ** -4], np.float32)
    slab, d = oracle.repack_q8_0(w, aux, grid)
    d16, qs = unpack_q8_0(slab, in_f)
    W = dequant_e4m3(w, aux, grid).reshape(out_f, in_f // 32, 32).astype(np.float64)
    amax = np.abs(W).max(axis=2)
    # the f16 scale is the library rounding of amax / 127 (taken in f32)
    dd = (amax.astype(np.float32) / np.float32(127)).astype(np.float32)
    assert np.array_equal(d, dd)
    assert np.array_equal(d16.view(np.uint16), dd.astype(np.float16).view(np.uint16))
    # every code is the nearest multiple of d among all 255 codes (brute force), except where the
    # exact quotient W/d lies within the f32 rounding of W/d (2^-23 relative) of a .5 tie: the
    # codes are decided on the f32 quotient, which may land on the tie and round away from zero
    k = np.arange(-127, 128, dtype=np.float64)
    d64 = dd.astype(np.float64)[..., None]
    best = np.empty_like(W)
    for r0 in range(0, out_f, 8):  # in row chunks: the full [rows, blocks, 32, 255] is 1.1 GB
        err = np.abs(W[r0:r0 + 8, ..., None] - k * d64[r0:r0 + 8, ..., None])
        best[r0:r0 + 8] = err.min(axis=3)
    mine = np.abs(W - qs.astype(np.float64) * d64)
    t = np.divide(W, d64, out=np.zeros_like(W), where=d64 != 0)
    near_tie = np.abs(np.abs(t - np.trunc(t)) - 0.5) <= 2.0 ** -23 * np.abs(t)
    nearest = mine <= best + 1e-12 * np.abs(W).max()
    assert np.all(nearest | (near_tie & (np.abs(qs - t) <= 0.5 + 2.0 ** -23 * np.abs(t))))
    # exact ties are common (E4M3 values are coarse, so W / amax is often a simple fraction);
    # with a non-power-of-two scale the f32 roundings of W and d turn some of them into near
    # ties that the f32 quotient still lands on -- codes off the nearest one come only from
    # those, well under 1% of the codes
    exact_tie = np.abs(np.abs(t - np.trunc(t)) - 0.5) == 0
    assert (near_tie & ~exact_tie & ~nearest).sum() < 1e-2 * t.size
    # the rounding rule at the ties the f32 quotient lands on: half away from zero
    t32 = np.divide(W.astype(np.float32), dd[..., None], out=np.zeros(W.shape, np.float32),
                    where=dd[..., None] != 0).astype(np.float64)
    tie = np.abs(t32 - np.trunc(t32)) == 0.5
    assert tie.sum() > 0
    assert np.array_equal(qs[tie].astype(np.float64), np.trunc(t32[tie]) + np.sign(t32[tie]))
    # invariants: |qs| <= 127 and the block's largest |W| maps to +-127
    assert np.all(np.abs(qs.astype(np.int32)) <= 127)
    pos = np.abs(W).argmax(axis=2)
    assert np.all(np.abs(np.take_along_axis(qs.astype(np.int32), pos[..., None], 2)) == 127)


def test_repack_constant_and_zero_blocks(oracle):
    w = np.zeros((2, 64), np.uint8)
    w[0, :32] = 0x38       # 1.0
    w[0, 32:] = 0xB8 ^ 0x00  # -1.0
    slab, d = oracle.repack_q8_0(w, np.array([0.25], np.float32), False)
    d16, qs = unpack_q8_0(slab, 64)
    assert np.all(qs[0, 0] == 127) and np.all(qs[0, 1] == -127)
    assert d16[0, 0] == np.float16(np.float32(0.25) / np.float32(127))
    assert np.all(qs[1] == 0) and np.all(d16[1].astype(np.float32) == 0)


@pytest.mark.parametrize("grid", [False, True])
def test_repacked_gemv_within_quantization_bound(oracle, grid):
    """The Q8_0 GEMV of the repacked slab against the block-128 / E4M3 GEMV of the source: each
    weight moves by at most d/2 + 127*|d16 - d| (code rounding, then f16 rounding of d)."""
    out_f, in_f = 96, 2048
    w = synth.e4m3_bytes(0x5205, out_f, in_f)
    aux = synth.grid_log2_uniform(0x5206, out_f, in_f) if grid else np.array([2.0 ** -3], np.float32)
    slab, d = oracle.repack_q8_0(w, aux, grid)
    d16, _ = unpack_q8_0(slab, in_f)
    x = synth.uniform_pm4(0x5207, 2 * in_f).reshape(2, in_f)
    _, dx, qx, _ = oracle.rmsnorm_q8_1(x, synth.uniform_pm4(0x5208, in_f))
    y8, _ = oracle.gemv_q8_0(slab, in_f, qx, dx)
    if grid:
        ye, _ = oracle.gemv_e4m3_blk128(w, aux, qx, dx)
    else:
        ye, _ = oracle.gemv_e4m3(w, float(aux[0]), qx, dx)
    eps_w = (d.astype(np.float64) / 2 + 127 * np.abs(d16.astype(np.float64) - d))   # [out_f, nb]
    X = (qx.astype(np.float64) * np.repeat(dx, 32, 1)).reshape(2, in_f // 32, 32)
    bound = np.abs(X).sum(axis=2) @ eps_w.T                                         # [2, out_f]
    # + the f32 rounding of each dequantized weight (|W| * 2^-24) on the E4M3 side
    assert np.all(np.abs(y8 - ye) <= bound * (1 + 1e-9) + 1e-6 * np.abs(ye).max())
