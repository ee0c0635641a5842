"""memq for GB300: the m <= 8 quantized decode chain as hand-written sm_103a CUDA kernels.

The compute lives in ``libmemq.so`` behind the C ABI of ``include/memq.h``; this module is a
thin ctypes binding with the same entry-point names.  It only checks and marshals arguments
(torch CUDA tensors -> device pointers, the current torch stream -> ``cudaStream_t``) and
raises on a nonzero status.  There is no CPU fallback: if the library is missing every call
raises.

Stage 1 -- ``memq_rmsnorm_q8_1``: q8_fuse_gate.rs (memra-engine 0.125.0), the fused
``rms_norm_zq8_f32`` producer.  Stage 2 -- ``memq_gemv_e4m3``, ``memq_gemv_e4m3_blk128``,
``memq_gemv_q8_0``: gemv_e4m3_bench.rs, the E4M3 / block-128 / Q8_0 arms.  The fused decode
step ``memq_rmsnorm_q8_1_gemv_*`` runs both stages in one launch, and
``memq_decode_step_host`` runs it for host-resident rows (copy in, fused step, copy out, wait)
in one native call.  Around them:
``memq_silu_mul_q8_1`` (the silu(gate) * up -> q8_1 producer named in q8_fuse_gate.rs, ``main``)
and ``memq_repack_e4m3[_blk128]_q8_0`` (gemv_e4m3_bench.rs, "QUESTION": E4M3 weights converted to
Q8_0 once at load).  The MLA decode attention kernels ``memq_mla_absorb_q``,
``memq_mla_attn_gathered`` and ``memq_mla_decompress_v``: mla_decode_arm_gate.rs (module doc).
"""
from __future__ import annotations

from ._binding import (  # noqa: F401
    MAX_GROUP,
    MAX_M,
    MAX_NCOLS,
    Container,
    MemqError,
    Status,
    lib,
    lib_path,
    memq_decode_step_host,
    memq_device_fault,
    memq_gemv_e4m3,
    memq_gemv_e4m3_blk128,
    memq_gemv_e4m3_blk128_group,
    memq_gemv_e4m3_group,
    memq_gemv_q8_0,
    memq_gemv_q8_0_group,
    memq_mla_absorb_q,
    memq_mla_attn_gathered,
    memq_mla_decompress_v,
    memq_rmsnorm_q8_1,
    memq_rmsnorm_q8_1_gemv_e4m3,
    memq_rmsnorm_q8_1_gemv_e4m3_blk128,
    memq_rmsnorm_q8_1_gemv_q8_0,
    memq_repack_e4m3_blk128_q8_0,
    memq_repack_e4m3_q8_0,
    memq_silu_mul_q8_1,
    memq_status_string,
    memq_version,
)
