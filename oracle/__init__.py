"""f64 CPU oracle of the quantized decode chain -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import this package.  The product path (``quantized_decode_memq_gb300``) never
imports, links or runs it, and this package imports nothing from the product path.

The arithmetic lives in ``memq_oracle.c`` (plain C, f64, straight loops in definition order);
this module only compiles it with gcc and marshals numpy arrays through ctypes.  Each function
cites the passage of the memra-engine 0.125.0 source pages it follows:

* ``rmsnorm`` / ``quantize_q8_1`` / ``rmsnorm_q8_1`` -- q8_fuse_gate.rs, module doc and
  ``run_shape`` (the ``rms_norm`` -> ``quantize_q8_1`` chain and the fused
  ``rms_norm_zq8_f32`` producer).
* ``gemv_e4m3`` / ``gemv_e4m3_blk128`` / ``gemv_q8_0`` -- gemv_e4m3_bench.rs, module doc
  ("THE COMPARISON", "THE BLOCK-128 ARM") and ``synth_e4m3`` / ``synth_blk_grid`` /
  ``synth_q8_0`` for the container layouts.

Every function is pinned by a CPU test against something other than itself (closed forms,
invariants, library decoders and a library matmul on small shapes); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "memq_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmemq_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile memq_oracle.c with gcc (-O2, no fast-math) into oracle/_build/."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-fno-fast-math", "-ffp-contract=off",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # MEMQ_ORACLE_LIB lets the mutation tests load a deliberately broken copy.
            override = os.environ.get("MEMQ_ORACLE_LIB")
            lib = ctypes.CDLL(override if override else build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            lib.memq_oracle_e4m3.restype = ctypes.c_double
            lib.memq_oracle_e4m3.argtypes = [ctypes.c_uint8]
            lib.memq_oracle_f16.restype = ctypes.c_double
            lib.memq_oracle_f16.argtypes = [ctypes.c_uint16]
            lib.memq_oracle_e4m3_table.argtypes = [P]
            lib.memq_oracle_f16_decode.argtypes = [P, I64, P]
            lib.memq_oracle_rmsnorm.argtypes = [P, P, I64, I64, ctypes.c_float, P]
            lib.memq_oracle_quantize_q8_1.argtypes = [P, I64, I64, P, P, P]
            lib.memq_oracle_gemv_e4m3.argtypes = [P, ctypes.c_float, P, P, I64, I64,
                                                  ctypes.c_int, P, I64, P, P]
            lib.memq_oracle_gemv_e4m3_blk128.argtypes = [P, P, P, P, I64, I64, ctypes.c_int,
                                                         P, I64, P, P]
            lib.memq_oracle_gemv_q8_0.argtypes = [P, P, P, I64, I64, ctypes.c_int, P, I64,
                                                  P, P]
            lib.memq_oracle_mla_head_gemv.argtypes = [P, P, ctypes.c_int, ctypes.c_int,
                                                      ctypes.c_int, ctypes.c_int, P, P]
            lib.memq_oracle_mla_attn_gathered.argtypes = [P, P, P, P] + [ctypes.c_int] * 5 + [
                ctypes.c_float, P, P, P]
            lib.memq_oracle_silu_mul.argtypes = [P, P, I64, P]
            lib.memq_oracle_f16_bits.argtypes = [ctypes.c_double]
            lib.memq_oracle_f16_bits.restype = ctypes.c_uint16
            lib.memq_oracle_repack_q8_0.argtypes = [P, P, ctypes.c_int, I64, I64, P, P]
            for name in ("memq_oracle_e4m3_table", "memq_oracle_f16_decode",
                         "memq_oracle_rmsnorm", "memq_oracle_quantize_q8_1",
                         "memq_oracle_gemv_e4m3", "memq_oracle_gemv_e4m3_blk128",
                         "memq_oracle_gemv_q8_0", "memq_oracle_silu_mul",
                         "memq_oracle_repack_q8_0", "memq_oracle_mla_head_gemv",
                         "memq_oracle_mla_attn_gathered"):
                getattr(lib, name).restype = None
            _lib = lib
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# ------------------------------------------------------------------------------------------
# Decoders
# ------------------------------------------------------------------------------------------

def e4m3_table() -> np.ndarray:
    """f64 value of every E4M3 code 0..255 (NaN at 0x7F and 0xFF)."""
    out = np.empty(256, np.float64)
    _load().memq_oracle_e4m3_table(_ptr(out))
    return out


def e4m3(code: int) -> float:
    return _load().memq_oracle_e4m3(int(code) & 0xFF)


def f16_decode(bits: np.ndarray) -> np.ndarray:
    """f64 value of IEEE binary16 bit patterns."""
    b = _c(bits, np.uint16).ravel()
    out = np.empty(b.size, np.float64)
    _load().memq_oracle_f16_decode(_ptr(b), b.size, _ptr(out))
    return out.reshape(np.shape(bits))


# ------------------------------------------------------------------------------------------
# Stage 1
# ------------------------------------------------------------------------------------------

def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """z = x * 1/sqrt(mean(x^2) + eps) * w per row, in f64.  x: [rows, ncols] f32."""
    x = _c(np.atleast_2d(x), np.float32)
    w = _c(w, np.float32)
    rows, ncols = x.shape
    assert w.shape == (ncols,)
    z = np.empty((rows, ncols), np.float64)
    _load().memq_oracle_rmsnorm(_ptr(x), _ptr(w), rows, ncols, ctypes.c_float(eps), _ptr(z))
    return z


def quantize_q8_1(z: np.ndarray):
    """Per 32-block: d = f32(amax/127), qs = round-half-away(z/d) (0 when d == 0).

    Returns (d f32 [rows, ncols/32], qs int8 [rows, ncols], ratio f64 [rows, ncols] = z/d).
    """
    z = _c(np.atleast_2d(z), np.float64)
    rows, ncols = z.shape
    assert ncols % 32 == 0
    d = np.empty((rows, ncols // 32), np.float32)
    qs = np.empty((rows, ncols), np.int8)
    ratio = np.empty((rows, ncols), np.float64)
    _load().memq_oracle_quantize_q8_1(_ptr(z), rows, ncols, _ptr(d), _ptr(qs), _ptr(ratio))
    return d, qs, ratio


def rmsnorm_q8_1(x: np.ndarray, w: np.ndarray, eps: float = 1e-6):
    """The whole producer: returns (z f64, d f32, qs int8, ratio f64)."""
    z = rmsnorm(x, w, eps)
    d, qs, ratio = quantize_q8_1(z)
    return z, d, qs, ratio


# ------------------------------------------------------------------------------------------
# Stage 2
# ------------------------------------------------------------------------------------------

def _rows_arg(rows, out_f):
    if rows is None:
        return None, out_f
    r = _c(rows, np.int64).ravel()
    assert r.size == 0 or (r.min() >= 0 and r.max() < out_f)
    return r, r.size


def _act_args(qs, d, in_f):
    qs = _c(np.atleast_2d(qs), np.int8)
    d = _c(np.atleast_2d(d), np.float32)
    m = qs.shape[0]
    assert qs.shape == (m, in_f) and d.shape == (m, in_f // 32)
    return qs, d, m


def _finish(fn, w, mid_args, qs, d, out_f, in_f, m, rows):
    r, n = _rows_arg(rows, out_f)
    y = np.empty((m, n), np.float64)
    s = np.empty((m, n), np.float64)
    fn(_ptr(w), *mid_args, _ptr(qs), _ptr(d), out_f, in_f, m,
       None if r is None else _ptr(r), n, _ptr(y), _ptr(s))
    return y, s


def gemv_e4m3(w: np.ndarray, scale: float, qs, d, rows=None):
    """y[j, t] = sum_i scale*e4m3(w[r_t, i]) * d[j, i//32]*qs[j, i]; returns (y, sum|.|)."""
    w = _c(w, np.uint8)
    out_f, in_f = w.shape
    qs, d, m = _act_args(qs, d, in_f)
    return _finish(_load().memq_oracle_gemv_e4m3, w, (ctypes.c_float(scale),), qs, d,
                   out_f, in_f, m, rows)


def gemv_e4m3_blk128(w: np.ndarray, grid: np.ndarray, qs, d, rows=None):
    """As gemv_e4m3 with W = grid[r//128, i//128] * e4m3(w[r, i])."""
    w = _c(w, np.uint8)
    out_f, in_f = w.shape
    grid = _c(grid, np.float32)
    assert grid.shape == ((out_f + 127) // 128, (in_f + 127) // 128)
    qs, d, m = _act_args(qs, d, in_f)
    return _finish(_load().memq_oracle_gemv_e4m3_blk128, w, (_ptr(grid),), qs, d,
                   out_f, in_f, m, rows)


def gemv_q8_0(w: np.ndarray, in_f: int, qs, d, rows=None):
    """ggml block_q8_0 weights (uint8 [out_f, in_f/32*34]); W = f16(d_blk) * qs_blk."""
    w = _c(w, np.uint8)
    out_f = w.shape[0]
    assert w.shape == (out_f, in_f // 32 * 34)
    qs, d, m = _act_args(qs, d, in_f)
    return _finish(_load().memq_oracle_gemv_q8_0, w, (), qs, d, out_f, in_f, m, rows)


# ------------------------------------------------------------------------------------------
# Next rows: the silu(gate)*up -> q8_1 producer and the E4M3 -> Q8_0 repack
# ------------------------------------------------------------------------------------------

def silu_mul(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """z = silu(g) * u = g / (1 + exp(-g)) * u in f64 (g, u: f32, same shape)."""
    g = _c(np.atleast_2d(g), np.float32)
    u = _c(np.atleast_2d(u), np.float32)
    assert g.shape == u.shape
    z = np.empty(g.shape, np.float64)
    _load().memq_oracle_silu_mul(_ptr(g), _ptr(u), g.size, _ptr(z))
    return z


def silu_mul_q8_1(g: np.ndarray, u: np.ndarray):
    """The whole silu producer: returns (z f64, d f32, qs int8, ratio f64)."""
    z = silu_mul(g, u)
    d, qs, ratio = quantize_q8_1(z)
    return z, d, qs, ratio


def f16_bits(v) -> np.ndarray:
    """IEEE binary16 bits of f64 values, round to nearest even (scalar or array)."""
    a = np.asarray(v, np.float64)
    f = _load().memq_oracle_f16_bits
    return np.array([f(float(x)) for x in a.reshape(-1)], np.uint16).reshape(a.shape)


def repack_q8_0(w: np.ndarray, aux: np.ndarray, grid: bool):
    """E4M3 weights -> Q8_0 slab (uint8 [out_f, in_f/32*34]) and the f32 d of every block.

    aux: the per-tensor scale (grid=False, shape (1,)) or the block-128 grid (grid=True)."""
    w = _c(w, np.uint8)
    out_f, in_f = w.shape
    aux = _c(aux, np.float32)
    if grid:
        assert aux.shape == ((out_f + 127) // 128, (in_f + 127) // 128)
    out = np.empty((out_f, in_f // 32 * 34), np.uint8)
    d = np.empty((out_f, in_f // 32), np.float32)
    _load().memq_oracle_repack_q8_0(_ptr(w), _ptr(aux), int(grid), out_f, in_f, _ptr(out),
                                    _ptr(d))
    return out, d


# ------------------------------------------------------------------------------------------
# t <= 8 MLA decode attention (mla_decode_arm_gate.rs)
# ------------------------------------------------------------------------------------------

def mla_head_gemv(x: np.ndarray, w: np.ndarray):
    """out[t,h,i] = sum_k x[t,h,k] * w[h,i,k]; x f32 [t,nh,cols], w f32 [nh,rows,cols].

    Returns (out f64 [t,nh,rows], sabs f64 [t,nh,rows] = sum |terms|)."""
    x = _c(x, np.float32)
    w = _c(w, np.float32)
    t, nh, cols = x.shape
    assert w.shape[0] == nh and w.shape[2] == cols
    rows = w.shape[1]
    out = np.empty((t, nh, rows), np.float64)
    sabs = np.empty((t, nh, rows), np.float64)
    _load().memq_oracle_mla_head_gemv(_ptr(x), _ptr(w), t, nh, rows, cols, _ptr(out), _ptr(sabs))
    return out, sabs


def mla_absorb_q(q_nope, wk_b):
    """absorb_q: q_nope [t,nh,d_nope], wk_b [nh,kv_rank,d_nope] -> [t,nh,kv_rank]."""
    return mla_head_gemv(q_nope, wk_b)


def mla_decompress_v(o_lat, wv_b):
    """decompress_v: o_lat [t,nh,kv_rank], wv_b [nh,d_v,kv_rank] -> [t,nh,d_v]."""
    return mla_head_gemv(o_lat, wv_b)


def mla_attn_gathered(q_lat, q_pe, cache, idx, scale: float, d_rope: int = 0, scores=False):
    """q_lat [t,nh,kv_rank], q_pe [t,nh,d_rope], cache [kv, kv_rank+d_rope], idx int32
    [t,n_slots] -> (out f64 [t,nh,kv_rank], cabs f64 = max_j |c_j[r]|[, scores f64])."""
    q_lat = _c(q_lat, np.float32)
    t, nh, kv_rank = q_lat.shape
    q_pe = _c(q_pe if q_pe is not None and q_pe.size else np.zeros((t, nh, max(d_rope, 1)), np.float32), np.float32)
    cache = _c(cache, np.float32)
    idx = _c(idx, np.int32)
    n_slots = idx.shape[1]
    out = np.empty((t, nh, kv_rank), np.float64)
    cabs = np.empty((t, nh, kv_rank), np.float64)
    sc = np.empty((t, nh, n_slots), np.float64) if scores else None
    _load().memq_oracle_mla_attn_gathered(_ptr(q_lat), _ptr(q_pe), _ptr(cache), _ptr(idx), nh,
                                          kv_rank, d_rope, t, n_slots, ctypes.c_float(scale),
                                          _ptr(out), _ptr(cabs), None if sc is None else _ptr(sc))
    return (out, cabs, sc) if scores else (out, cabs)
