"""Shared checks for the GPU parity tests: CUDA path (through the C ABI) vs the f64 oracle."""
from __future__ import annotations

import numpy as np
import torch

# GEMV tolerance: |y - y_oracle| <= GEMV_TOL * sum_i |W_i X_i|  (both sides fed the same q8_1).
GEMV_TOL = 2e-5
# z tolerance: relative 1e-6 with an absolute floor of one f32 ulp of the row's largest |z|.
Z_REL = 1e-6
# qs may differ by 1 only when z/d lies within this distance of a .5 rounding boundary.
QS_WINDOW = 1e-5


def to_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def check_gemv(y_gpu: torch.Tensor, y_ref: np.ndarray, s_ref: np.ndarray, rows=None,
               tol=GEMV_TOL):
    y = y_gpu.double().cpu().numpy()
    if rows is not None:
        y = y[:, rows]
    assert y.shape == y_ref.shape, (y.shape, y_ref.shape)
    assert np.all(np.isfinite(y))
    err = np.abs(y - y_ref)
    bound = tol * s_ref
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{bad.sum()} GEMV outputs outside {tol}*S; worst ratio "
            f"{(err / np.maximum(s_ref, 1e-300)).max():.3e}; first {idx.tolist()}")
    return float((err / np.maximum(s_ref, 1e-300)).max())


def check_producer(oracle, x: np.ndarray, w: np.ndarray, eps: float, z_gpu, qs_gpu, d_gpu,
                   rows=None):
    """Checks the GPU producer on the given rows (all rows when None).

    1. z within Z_REL of the oracle's f64 z (with a one-ulp-of-row-max floor).
    2. Self-consistency, decided at the kernel's inputs: the oracle's quantizer applied to the
       GPU's own z gives bit-identical d, and identical qs except +-1 where z/d lies within
       QS_WINDOW of a .5 boundary.
    3. Against the full f64 chain: d within Z_REL; qs equal except +-1 near a boundary, where
       "near" widens by the propagated z tolerance (127 * 2 * Z_REL relative).
    Returns the number of qs codes that differ from the full-chain oracle.
    """
    if rows is not None:
        x = x[rows]
    z_ref, d_ref, qs_ref, ratio_ref = oracle.rmsnorm_q8_1(x, w, eps)
    return check_q8_1(oracle, z_ref, d_ref, qs_ref, ratio_ref, z_gpu, qs_gpu, d_gpu, rows)


def check_q8_1(oracle, z_ref, d_ref, qs_ref, ratio_ref, z_gpu, qs_gpu, d_gpu, rows=None):
    """The q8_1 checks of check_producer against an oracle z (f64) and its quantization."""
    z_g = None if z_gpu is None else z_gpu.cpu().numpy().astype(np.float64)
    qs_g = qs_gpu.cpu().numpy()
    d_g = d_gpu.cpu().numpy()
    if rows is not None:
        z_g = None if z_g is None else z_g[rows]
        qs_g = qs_g[rows]
        d_g = d_g[rows]

    if z_g is not None:
        floor = np.abs(z_ref).max(axis=1, keepdims=True) * 2.0 ** -24
        zerr = np.abs(z_g - z_ref)
        assert np.all(zerr <= Z_REL * np.abs(z_ref) + floor), (
            f"z error up to {(zerr / np.maximum(np.abs(z_ref), 1e-30)).max():.3e} relative")
        # 2. self-consistency on the GPU's own z
        d_s, qs_s, ratio_s = oracle.quantize_q8_1(z_g)
        assert np.array_equal(d_g.view(np.uint32), d_s.view(np.uint32)), "d not bit-exact"
        diff = qs_g.astype(np.int32) - qs_s.astype(np.int32)
        near = np.abs(np.abs(ratio_s - np.trunc(ratio_s)) - 0.5) <= QS_WINDOW
        assert np.all(np.abs(diff) <= 1)
        assert np.all((diff == 0) | near), f"{np.sum((diff != 0) & ~near)} qs codes off"

    # 3. the full chain
    np.testing.assert_allclose(d_g, d_ref, rtol=Z_REL, atol=0)
    diff = qs_g.astype(np.int32) - qs_ref.astype(np.int32)
    frac = np.abs(np.abs(ratio_ref - np.trunc(ratio_ref)) - 0.5)
    near = frac <= QS_WINDOW + 2.5e-6 * np.abs(ratio_ref)
    assert np.all(np.abs(diff) <= 1)
    assert np.all((diff == 0) | near), f"{np.sum((diff != 0) & ~near)} qs codes off"
    assert np.all(np.abs(qs_g.astype(np.int32)) <= 127)
    return int(np.sum(diff != 0))


def sample_rows(out_f: int, n: int = 192, seed: int = 0) -> np.ndarray:
    """Rows for sampled full-size checks: both ends plus seeded random rows."""
    if out_f <= n:
        return np.arange(out_f)
    rng = np.random.default_rng(seed)
    ends = np.r_[np.arange(32), np.arange(out_f - 32, out_f)]
    mid = rng.choice(out_f, size=n - 64, replace=False)
    return np.unique(np.r_[ends, mid])
