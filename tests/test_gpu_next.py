"""GPU parity of the next-row entry points against the oracle.

memq_silu_mul_q8_1 (the silu(gate) * up -> q8_1 producer of q8_fuse_gate.rs, `main`): z within
1e-6 relative of the f64 oracle, qs / d checked as for the RMSNorm producer (self-consistent on
the GPU's own z, and against the full f64 chain within the rounding window).

memq_repack_e4m3[_blk128]_q8_0 (the load-time E4M3 -> Q8_0 slab of gemv_e4m3_bench.rs,
"QUESTION"): every output byte equal to the oracle's (the conversion is defined in IEEE f32, so
it is bit-reproducible), and the slab feeds memq_gemv_q8_0 like any Q8_0 weight.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import check_gemv, check_q8_1, sample_rows, to_dev
from quantized_decode_memq_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def memq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_decode_memq_gb300 import build
    build.build()
    import quantized_decode_memq_gb300 as m
    return m


def gate_up(rows, ncols, seed):
    g = synth.uniform_pm4(seed, rows * ncols).reshape(rows, ncols) * np.float32(2.0)
    u = synth.uniform_pm4(seed + 1, rows * ncols).reshape(rows, ncols)
    return g.astype(np.float32), u.astype(np.float32)


@pytest.mark.parametrize("rows,ncols", [(1, 32), (1, 1536), (8, 1536), (3, 4096 + 32), (64, 8192),
                                        (1000, 1536)])
def test_silu_mul_q8_1_parity(memq, oracle, rows, ncols):
    g, u = gate_up(rows, ncols, 0x7100 + rows + ncols)
    z, qs, d = memq.memq_silu_mul_q8_1(to_dev(g), to_dev(u))
    torch.cuda.synchronize()
    check_q8_1(oracle, *oracle.silu_mul_q8_1(g, u), z, qs, d)
    assert memq.memq_device_fault() == 0


def test_silu_mul_q8_1_saturation_and_zero_blocks(memq, oracle):
    g = np.zeros((2, 64), np.float32)
    u = np.ones((2, 64), np.float32)
    g[0, :32] = np.linspace(-120, 120, 32, dtype=np.float32)   # exp overflow / underflow
    z, qs, d = memq.memq_silu_mul_q8_1(to_dev(g), to_dev(u))
    torch.cuda.synchronize()
    check_q8_1(oracle, *oracle.silu_mul_q8_1(g, u), z, qs, d)
    assert torch.all(d[1] == 0) and torch.all(qs[1] == 0) and torch.all(d[0, 1] == 0)


def test_silu_mul_q8_1_without_z(memq, oracle):
    g, u = gate_up(4, 1536, 0x7200)
    _, qs, d = memq.memq_silu_mul_q8_1(to_dev(g), to_dev(u), want_z=False)
    torch.cuda.synchronize()
    check_q8_1(oracle, *oracle.silu_mul_q8_1(g, u), None, qs, d)


def aux_for(grid, out_f, in_f, seed):
    if grid:
        return synth.grid_log2_uniform(seed, out_f, in_f)
    return np.array([2.0 ** -4], np.float32)


def gpu_repack(memq, w, aux, grid):
    fn = memq.memq_repack_e4m3_blk128_q8_0 if grid else memq.memq_repack_e4m3_q8_0
    out = fn(to_dev(w), to_dev(aux))
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("grid", [False, True])
@pytest.mark.parametrize("out_f,in_f", [(1, 32), (37, 96), (130, 4096 + 32), (1000, 2560),
                                        (257, 1024 + 256)])
def test_repack_bit_exact(memq, oracle, grid, out_f, in_f):
    w = synth.e4m3_bytes(0x7300 + out_f + grid, out_f, in_f)
    aux = aux_for(grid, out_f, in_f, 0x7301 + in_f)
    out = gpu_repack(memq, w, aux, grid)
    ref, _ = oracle.repack_q8_0(w, aux, grid)
    got = out.cpu().numpy()
    assert np.array_equal(got, ref), f"{np.sum(got != ref)} bytes differ"


@pytest.mark.parametrize("grid", [False, True])
def test_repack_full_size_bit_exact_and_gemv(memq, oracle, grid):
    """17408 x 5120: the whole slab bit-exact; then memq_gemv_q8_0 on the GPU slab against the
    oracle's Q8_0 GEMV of the same bytes (sampled rows)."""
    out_f, in_f = 17408, 5120
    w = synth.e4m3_bytes(0x7400 + grid, out_f, in_f)
    aux = aux_for(grid, out_f, in_f, 0x7401)
    out = gpu_repack(memq, w, aux, grid)
    ref, _ = oracle.repack_q8_0(w, aux, grid)
    assert np.array_equal(out.cpu().numpy(), ref)
    x = synth.uniform_pm4(0x7402, in_f).reshape(1, in_f)
    _, d, qs, _ = oracle.rmsnorm_q8_1(x, synth.uniform_pm4(0x7403, in_f))
    y = memq.memq_gemv_q8_0(out, to_dev(qs), to_dev(d))
    torch.cuda.synchronize()
    rows = sample_rows(out_f, 128, seed=grid)
    y_ref, s_ref = oracle.gemv_q8_0(ref, in_f, qs, d, rows=rows)
    check_gemv(y, y_ref, s_ref, rows=rows)
    assert memq.memq_device_fault() == 0


def test_repack_zero_rows_and_constant_blocks(memq, oracle):
    w = np.zeros((3, 64), np.uint8)
    w[0, :32] = 0x38      # +1.0
    w[0, 32:] = 0xB8      # -1.0
    w[2, :] = 0x80        # -0.0
    aux = np.array([0.25], np.float32)
    got = gpu_repack(memq, w, aux, False).cpu().numpy()
    ref, _ = oracle.repack_q8_0(w, aux, False)
    assert np.array_equal(got, ref)
    assert memq.memq_repack_e4m3_q8_0(torch.empty((0, 64), dtype=torch.uint8, device="cuda"),
                                      to_dev(aux)).shape == (0, 68)
