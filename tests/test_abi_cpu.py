"""The C ABI library on the CPU: it loads, exports every entry point the headers declare, and
rejects bad arguments before touching CUDA.  No compute call is made here."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from quantized_decode_memq_gb300 import build
    try:
        build.build()
    except RuntimeError as e:  # no nvcc on this machine
        pytest.skip(str(e))
    import quantized_decode_memq_gb300 as m
    return m.lib()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(memq_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("memq_rmsnorm_q8_1", "memq_gemv_e4m3", "memq_gemv_e4m3_blk128",
                     "memq_gemv_q8_0", "memq_rmsnorm_q8_1_gemv_e4m3",
                     "memq_rmsnorm_q8_1_gemv_e4m3_blk128", "memq_rmsnorm_q8_1_gemv_q8_0",
                     "memq_gemv_e4m3_group", "memq_gemv_e4m3_blk128_group",
                     "memq_gemv_q8_0_group", "memq_silu_mul_q8_1", "memq_repack_e4m3_q8_0",
                     "memq_repack_e4m3_blk128_q8_0", "memq_mla_absorb_q",
                     "memq_mla_decompress_v", "memq_mla_attn_gathered",
                     "memq_decode_step_host", "memq_status_string", "memq_device_fault",
                     "memq_version"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    import quantized_decode_memq_gb300 as m
    assert m.memq_status_string(0) == "ok"
    for s in m.Status:
        assert m.memq_status_string(int(s))
    assert m.memq_status_string(99) == "unknown memq status"
    assert m.memq_version() >> 16 == 1


def test_validation_rejects_before_any_cuda_call(lib):
    import quantized_decode_memq_gb300 as m
    P = ctypes.c_void_p
    fake = P(0x1000)  # never dereferenced: every call below fails validation first
    assert lib.memq_gemv_e4m3(None, fake, fake, fake, fake, 4, 64, 1, None) == m.Status.ERR_NULL
    assert lib.memq_gemv_e4m3(fake, fake, fake, fake, fake, 4, 64, 0, None) == m.Status.ERR_M_RANGE
    assert lib.memq_gemv_e4m3_blk128(fake, fake, fake, fake, fake, 4, 40, 1, None) == m.Status.ERR_SHAPE
    assert lib.memq_gemv_q8_0(fake, fake, fake, fake, -3, 64, 1, None) == m.Status.ERR_SHAPE
    assert lib.memq_gemv_q8_0(fake, fake, P(0x1002), fake, 4, 64, 1, None) == m.Status.ERR_ALIGN
    assert lib.memq_rmsnorm_q8_1(fake, fake, None, fake, fake, 33, 1, 1e-6, None) == m.Status.ERR_SHAPE
    assert lib.memq_rmsnorm_q8_1(fake, None, None, fake, fake, 64, 1, 1e-6, None) == m.Status.ERR_NULL
    assert lib.memq_rmsnorm_q8_1(P(0x1004), fake, None, fake, fake, 64, 1, 1e-6, None) == m.Status.ERR_ALIGN
    # empty problems are valid no-ops and launch nothing, even with NULL pointers
    assert lib.memq_rmsnorm_q8_1(None, None, None, None, None, 64, 0, 1e-6, None) == m.Status.OK
    assert lib.memq_gemv_q8_0(None, None, None, None, 0, 64, 1, None) == m.Status.OK
    assert lib.memq_device_fault(None, None) == m.Status.ERR_NULL
    # fused decode step: validation before any launch
    assert lib.memq_rmsnorm_q8_1_gemv_q8_0(None, fake, 1e-6, fake, fake, fake, None, fake, 4, 64, 1, None) == m.Status.ERR_NULL
    assert lib.memq_rmsnorm_q8_1_gemv_e4m3(fake, fake, 1e-6, fake, fake, fake, fake, None, fake, 4, 64, 9, None) == m.Status.ERR_M_RANGE
    assert lib.memq_rmsnorm_q8_1_gemv_e4m3_blk128(fake, fake, -1.0, fake, fake, fake, fake, None, fake, 4, 64, 1, None) == m.Status.ERR_SHAPE
    # host-buffer decode step: the same checks, plus the container and the host pointers, all
    # before any copy
    host_args = [fake, fake, 1e-6, fake, fake, fake, fake, None, fake, fake, 4, 64]
    assert lib.memq_decode_step_host(3, fake, *host_args, 1, None) == m.Status.ERR_SHAPE
    assert lib.memq_decode_step_host(-1, fake, *host_args, 1, None) == m.Status.ERR_SHAPE
    assert lib.memq_decode_step_host(0, None, *host_args, 1, None) == m.Status.ERR_NULL
    assert lib.memq_decode_step_host(2, fake, *host_args, 0, None) == m.Status.ERR_M_RANGE
    assert lib.memq_decode_step_host(1, fake, P(0x1004), *host_args[1:], 1, None) == m.Status.ERR_ALIGN
    no_y_host = host_args[:9] + [None] + host_args[10:]
    assert lib.memq_decode_step_host(2, fake, *no_y_host, 1, None) == m.Status.ERR_NULL
    assert lib.memq_rmsnorm_q8_1_gemv_q8_0(fake, fake, 1e-6, fake, fake, fake, None, fake, 4, 65536, 1, None) == m.Status.ERR_SHAPE
    assert lib.memq_rmsnorm_q8_1_gemv_q8_0(P(0x1004), fake, 1e-6, fake, fake, fake, None, fake, 4, 64, 1, None) == m.Status.ERR_ALIGN
    # grouped GEMVs: the count and the host arrays are checked first
    VP2 = ctypes.c_void_p * 2
    I2 = ctypes.c_int64 * 2
    ws, ys = VP2(0x1000, 0x1000), VP2(0x1000, 0x1000)
    assert lib.memq_gemv_e4m3_group(0, ws, ws, ys, I2(4, 4), fake, fake, 64, 1, None) == m.Status.ERR_SHAPE
    assert lib.memq_gemv_e4m3_blk128_group(5, ws, ws, ys, I2(4, 4), fake, fake, 64, 1, None) == m.Status.ERR_SHAPE
    assert lib.memq_gemv_q8_0_group(2, None, ys, I2(4, 4), fake, fake, 256, 1, None) == m.Status.ERR_NULL
    assert lib.memq_gemv_e4m3_group(2, ws, ws, ys, I2(4, 0), fake, fake, 64, 1, None) == m.Status.ERR_SHAPE
    assert lib.memq_gemv_e4m3_group(2, ws, ws, ys, I2(4, 4), fake, fake, 64, 9, None) == m.Status.ERR_M_RANGE
    # silu(gate) * up -> q8_1 producer
    assert lib.memq_silu_mul_q8_1(fake, fake, None, fake, fake, 48, 1, None) == m.Status.ERR_SHAPE
    assert lib.memq_silu_mul_q8_1(None, fake, None, fake, fake, 64, 1, None) == m.Status.ERR_NULL
    assert lib.memq_silu_mul_q8_1(fake, P(0x1008), None, fake, fake, 64, 1, None) == m.Status.ERR_ALIGN
    assert lib.memq_silu_mul_q8_1(None, None, None, None, None, 64, 0, None) == m.Status.OK
    # E4M3 -> Q8_0 repack
    assert lib.memq_repack_e4m3_q8_0(fake, fake, fake, 4, 40, None) == m.Status.ERR_SHAPE
    assert lib.memq_repack_e4m3_blk128_q8_0(fake, None, fake, 4, 64, None) == m.Status.ERR_NULL
    assert lib.memq_repack_e4m3_q8_0(fake, fake, P(0x1002), 4, 64, None) == m.Status.ERR_ALIGN
    assert lib.memq_repack_e4m3_q8_0(None, None, None, 0, 64, None) == m.Status.OK
    # MLA decode attention kernels: (.., t, nh, d_nope | d_v, kv_rank, split, stream)
    assert lib.memq_mla_absorb_q(fake, fake, fake, 0, 64, 256, 512, 0, None) == m.Status.ERR_M_RANGE
    assert lib.memq_mla_absorb_q(fake, fake, fake, 9, 64, 256, 512, 0, None) == m.Status.ERR_M_RANGE
    assert lib.memq_mla_absorb_q(fake, fake, fake, 1, 64, 200, 512, 0, None) == m.Status.ERR_SHAPE
    assert lib.memq_mla_absorb_q(fake, fake, fake, 1, 64, 2048, 512, 0, None) == m.Status.ERR_SHAPE
    assert lib.memq_mla_absorb_q(fake, fake, fake, 1, 64, 256, 512, -1, None) == m.Status.ERR_SHAPE
    assert lib.memq_mla_absorb_q(fake, None, fake, 1, 64, 256, 512, 0, None) == m.Status.ERR_NULL
    assert lib.memq_mla_absorb_q(P(0x1004), fake, fake, 1, 64, 256, 512, 0, None) == m.Status.ERR_ALIGN
    assert lib.memq_mla_decompress_v(fake, fake, fake, 1, 64, 256, 500, 0, None) == m.Status.ERR_SHAPE
    assert lib.memq_mla_decompress_v(fake, fake, fake, 1, 0, 256, 512, 0, None) == m.Status.ERR_SHAPE
    assert lib.memq_mla_decompress_v(fake, fake, P(0x1002), 1, 64, 256, 512, 0, None) == m.Status.ERR_ALIGN
    #   (q_lat, q_pe, cache, idx, out, nh, kv_rank, d_rope, t, n_slots, scale, split, stream)
    attn = lib.memq_mla_attn_gathered
    assert attn(fake, None, fake, fake, fake, 64, 512, 0, 9, 2048, 0.04, 0, None) == m.Status.ERR_M_RANGE
    assert attn(fake, None, fake, fake, fake, 64, 512, 0, 1, 0, 0.04, 0, None) == m.Status.ERR_SHAPE
    assert attn(fake, None, fake, fake, fake, 64, 384 + 1, 0, 1, 16, 0.04, 0, None) == m.Status.ERR_SHAPE
    assert attn(fake, fake, fake, fake, fake, 64, 512, 129, 1, 16, 0.04, 0, None) == m.Status.ERR_SHAPE
    assert attn(fake, None, fake, fake, fake, 64, 512, 0, 1, 16, 0.04, 3, None) == m.Status.ERR_SHAPE
    assert attn(fake, None, fake, fake, fake, 64, 512, 0, 1, 16, float("inf"), 0, None) == m.Status.ERR_SHAPE
    assert attn(fake, None, fake, fake, fake, 64, 512, 64, 1, 16, 0.04, 0, None) == m.Status.ERR_NULL
    assert attn(fake, None, fake, None, fake, 64, 512, 0, 1, 16, 0.04, 0, None) == m.Status.ERR_NULL
    assert attn(fake, None, P(0x1004), fake, fake, 64, 512, 0, 1, 16, 0.04, 0, None) == m.Status.ERR_ALIGN
    assert attn(fake, None, fake, P(0x1002), fake, 64, 512, 0, 1, 16, 0.04, 0, None) == m.Status.ERR_ALIGN


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import quantized_decode_memq_gb300._binding as b
    monkeypatch.setattr(b, "_lib", None)
    monkeypatch.setattr(b, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        b.lib()
