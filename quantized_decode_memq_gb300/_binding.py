"""ctypes binding of libmemq.so (argument marshalling only; all compute is in the kernels)."""
from __future__ import annotations

import ctypes
import enum
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_build", "libmemq.so")
_lock = threading.Lock()
_lib = None

MAX_M = 8
MAX_NCOLS = 32768
MAX_GROUP = 4


class Status(enum.IntEnum):
    OK = 0
    ERR_NULL = 1
    ERR_SHAPE = 2
    ERR_ALIGN = 3
    ERR_M_RANGE = 4
    ERR_LAUNCH = 5
    ERR_DEVICE = 6


class Container(enum.IntEnum):
    E4M3 = 0
    E4M3_BLK128 = 1
    Q8_0 = 2


class MemqError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: memq status {status} ({memq_status_string(status)})")


def lib_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """Load libmemq.so; raise (never fall back) if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"libmemq.so is missing at {_LIB_PATH}: build it with "
                    "quantized_decode_memq_gb300.build.build() (there is no CPU fallback)")
            L = ctypes.CDLL(_LIB_PATH)
            P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            L.memq_rmsnorm_q8_1.argtypes = [P, P, P, P, P, I64, I64, ctypes.c_float, P]
            L.memq_gemv_e4m3.argtypes = [P, P, P, P, P, I64, I64, I32, P]
            L.memq_gemv_e4m3_blk128.argtypes = [P, P, P, P, P, I64, I64, I32, P]
            L.memq_gemv_q8_0.argtypes = [P, P, P, P, I64, I64, I32, P]
            L.memq_rmsnorm_q8_1_gemv_e4m3.argtypes = [P, P, ctypes.c_float, P, P, P, P, P, P,
                                                      I64, I64, I32, P]
            L.memq_rmsnorm_q8_1_gemv_e4m3_blk128.argtypes = [P, P, ctypes.c_float, P, P, P, P,
                                                             P, P, I64, I64, I32, P]
            L.memq_rmsnorm_q8_1_gemv_q8_0.argtypes = [P, P, ctypes.c_float, P, P, P, P, P, I64,
                                                      I64, I32, P]
            PP = ctypes.POINTER(ctypes.c_void_p)
            PI64 = ctypes.POINTER(ctypes.c_int64)
            L.memq_gemv_e4m3_group.argtypes = [I32, PP, PP, PP, PI64, P, P, I64, I32, P]
            L.memq_gemv_e4m3_blk128_group.argtypes = [I32, PP, PP, PP, PI64, P, P, I64, I32, P]
            L.memq_gemv_q8_0_group.argtypes = [I32, PP, PP, PI64, P, P, I64, I32, P]
            L.memq_silu_mul_q8_1.argtypes = [P, P, P, P, P, I64, I64, P]
            L.memq_repack_e4m3_q8_0.argtypes = [P, P, P, I64, I64, P]
            L.memq_repack_e4m3_blk128_q8_0.argtypes = [P, P, P, I64, I64, P]
            L.memq_mla_absorb_q.argtypes = [P, P, P, I32, I32, I32, I32, I32, P]
            L.memq_mla_decompress_v.argtypes = [P, P, P, I32, I32, I32, I32, I32, P]
            L.memq_mla_attn_gathered.argtypes = [P, P, P, P, P, I32, I32, I32, I32, I32,
                                                 ctypes.c_float, I32, P]
            L.memq_decode_step_host.argtypes = [I32, P, P, P, ctypes.c_float, P, P, P, P, P, P,
                                                P, I64, I64, I32, P]
            L.memq_device_fault.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
            L.memq_status_string.argtypes = [I32]
            L.memq_status_string.restype = ctypes.c_char_p
            L.memq_version.argtypes = []
            for name in ("memq_rmsnorm_q8_1", "memq_gemv_e4m3", "memq_gemv_e4m3_blk128",
                         "memq_gemv_q8_0", "memq_rmsnorm_q8_1_gemv_e4m3",
                         "memq_rmsnorm_q8_1_gemv_e4m3_blk128", "memq_rmsnorm_q8_1_gemv_q8_0",
                         "memq_gemv_e4m3_group", "memq_gemv_e4m3_blk128_group",
                         "memq_gemv_q8_0_group", "memq_silu_mul_q8_1", "memq_repack_e4m3_q8_0",
                         "memq_repack_e4m3_blk128_q8_0", "memq_decode_step_host",
                         "memq_device_fault", "memq_version"):
                getattr(L, name).restype = ctypes.c_int
            _lib = L
    return _lib


def memq_status_string(status: int) -> str:
    return lib().memq_status_string(int(status)).decode()


def memq_version() -> int:
    return lib().memq_version()


# The current stream as a raw cudaStream_t: torch's C binding returns the pointer directly
# (~0.2 us), where torch.cuda.current_stream() builds a Stream object (~3 us per call).
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_cur_device = getattr(torch._C, "_cuda_getDevice", None)


def _stream(stream):
    if stream is None:
        if _raw_stream is not None and _cur_device is not None:
            return _raw_stream(_cur_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check(fn: str, rc: int):
    if rc != 0:
        raise MemqError(fn, rc)


def _cuda(name: str, t: torch.Tensor, dtype, shape=None):
    # one combined test on the common path; the specific error only when it fails
    if (isinstance(t, torch.Tensor) and t.dtype is dtype and t.is_cuda and t.is_contiguous()
            and (shape is None or t.shape == shape)):
        return t
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t


def memq_rmsnorm_q8_1(x: torch.Tensor, w: torch.Tensor, eps: float = 1e-6, *, z=None, qs=None,
                      d=None, want_z: bool = True, stream=None):
    """Fused RMSNorm -> q8_1.  x: f32 [rows, ncols], w: f32 [ncols].

    Returns (z f32 [rows, ncols] or None, qs int8 [rows, ncols], d f32 [rows, ncols/32]).
    Output tensors may be passed in (z/qs/d) to avoid allocation.
    """
    x2 = x if x.dim() == 2 else x.reshape(1, -1)
    _cuda("x", x2, torch.float32)
    rows, ncols = x2.shape
    _cuda("w", w, torch.float32, (ncols,))
    if qs is None:
        qs = torch.empty((rows, ncols), dtype=torch.int8, device=x.device)
    if d is None:
        d = torch.empty((rows, ncols // 32), dtype=torch.float32, device=x.device)
    if z is None and want_z:
        z = torch.empty((rows, ncols), dtype=torch.float32, device=x.device)
    _cuda("qs", qs, torch.int8, (rows, ncols))
    _cuda("d", d, torch.float32, (rows, ncols // 32))
    if z is not None:
        _cuda("z", z, torch.float32, (rows, ncols))
    rc = lib().memq_rmsnorm_q8_1(_ptr(x2), _ptr(w), _ptr(z), _ptr(qs), _ptr(d), ncols, rows,
                                 ctypes.c_float(eps), _stream(stream))
    _check("memq_rmsnorm_q8_1", rc)
    return z, qs, d


def _act(qs, d, in_f):
    qs2 = qs if qs.dim() == 2 else qs.reshape(1, -1)
    _cuda("qs", qs2, torch.int8)
    m = qs2.shape[0]
    if qs2.shape[1] != in_f:
        raise ValueError(f"qs has {qs2.shape[1]} columns, expected in_f={in_f}")
    d2 = d if d.dim() == 2 else d.reshape(1, -1)
    _cuda("d", d2, torch.float32, (m, in_f // 32))
    return qs2, d2, m


def _out(y, m, out_f, device):
    if y is None:
        y = torch.empty((m, out_f), dtype=torch.float32, device=device)
    _cuda("y", y, torch.float32, (m, out_f))
    return y


def memq_gemv_e4m3(w: torch.Tensor, w_scale: torch.Tensor, qs: torch.Tensor, d: torch.Tensor, *,
                   y=None, stream=None):
    """y[m, out_f] = scale * e4m3(w) . (d*qs).  w: uint8 [out_f, in_f]; w_scale: f32 [1]."""
    _cuda("w", w, torch.uint8)
    out_f, in_f = w.shape
    _cuda("w_scale", w_scale, torch.float32, (1,))
    qs2, d2, m = _act(qs, d, in_f)
    y = _out(y, m, out_f, w.device)
    rc = lib().memq_gemv_e4m3(_ptr(w), _ptr(w_scale), _ptr(qs2), _ptr(d2), _ptr(y), out_f, in_f,
                              m, _stream(stream))
    _check("memq_gemv_e4m3", rc)
    return y


def memq_gemv_e4m3_blk128(w: torch.Tensor, grid: torch.Tensor, qs: torch.Tensor, d: torch.Tensor,
                          *, y=None, stream=None):
    """y = (grid (x) e4m3(w)) . (d*qs); grid: f32 [ceil(out_f/128), ceil(in_f/128)]."""
    _cuda("w", w, torch.uint8)
    out_f, in_f = w.shape
    _cuda("grid", grid, torch.float32, ((out_f + 127) // 128, (in_f + 127) // 128))
    qs2, d2, m = _act(qs, d, in_f)
    y = _out(y, m, out_f, w.device)
    rc = lib().memq_gemv_e4m3_blk128(_ptr(w), _ptr(grid), _ptr(qs2), _ptr(d2), _ptr(y), out_f,
                                     in_f, m, _stream(stream))
    _check("memq_gemv_e4m3_blk128", rc)
    return y


def memq_gemv_q8_0(w: torch.Tensor, qs: torch.Tensor, d: torch.Tensor, *, y=None, stream=None):
    """y = W_q8_0 . (d*qs); w: uint8 [out_f, in_f/32*34] (ggml block_q8_0 rows)."""
    _cuda("w", w, torch.uint8)
    out_f, row_bytes = w.shape
    if row_bytes % 34 != 0:
        raise ValueError("Q8_0 rows must be a whole number of 34-byte blocks")
    in_f = row_bytes // 34 * 32
    qs2, d2, m = _act(qs, d, in_f)
    y = _out(y, m, out_f, w.device)
    rc = lib().memq_gemv_q8_0(_ptr(w), _ptr(qs2), _ptr(d2), _ptr(y), out_f, in_f, m,
                              _stream(stream))
    _check("memq_gemv_q8_0", rc)
    return y


def _fused_outputs(x2, m, in_f, out_f, qs, d, z, y, want_z):
    dev = x2.device
    if qs is None:
        qs = torch.empty((m, in_f), dtype=torch.int8, device=dev)
    if d is None:
        d = torch.empty((m, in_f // 32), dtype=torch.float32, device=dev)
    if z is None and want_z:
        z = torch.empty((m, in_f), dtype=torch.float32, device=dev)
    _cuda("qs", qs, torch.int8, (m, in_f))
    _cuda("d", d, torch.float32, (m, in_f // 32))
    if z is not None:
        _cuda("z", z, torch.float32, (m, in_f))
    y = _out(y, m, out_f, dev)
    return qs, d, z, y


def _fused_in(x, wn, in_f):
    x2 = x if x.dim() == 2 else x.reshape(1, -1)
    _cuda("x", x2, torch.float32)
    if x2.shape[1] != in_f:
        raise ValueError(f"x has {x2.shape[1]} columns, expected in_f={in_f}")
    _cuda("wn", wn, torch.float32, (in_f,))
    return x2, x2.shape[0]


def memq_rmsnorm_q8_1_gemv_e4m3(x, wn, w, w_scale, eps: float = 1e-6, *, qs=None, d=None, z=None,
                                y=None, want_z: bool = False, stream=None):
    """Fused decode step, E4M3 weights.  Returns (y, qs, d, z)."""
    _cuda("w", w, torch.uint8)
    out_f, in_f = w.shape
    _cuda("w_scale", w_scale, torch.float32, (1,))
    x2, m = _fused_in(x, wn, in_f)
    qs, d, z, y = _fused_outputs(x2, m, in_f, out_f, qs, d, z, y, want_z)
    rc = lib().memq_rmsnorm_q8_1_gemv_e4m3(_ptr(x2), _ptr(wn), ctypes.c_float(eps), _ptr(w),
                                           _ptr(w_scale), _ptr(qs), _ptr(d), _ptr(z), _ptr(y),
                                           out_f, in_f, m, _stream(stream))
    _check("memq_rmsnorm_q8_1_gemv_e4m3", rc)
    return y, qs, d, z


def memq_rmsnorm_q8_1_gemv_e4m3_blk128(x, wn, w, grid, eps: float = 1e-6, *, qs=None, d=None,
                                       z=None, y=None, want_z: bool = False, stream=None):
    """Fused decode step, block-128 E4M3 weights.  Returns (y, qs, d, z)."""
    _cuda("w", w, torch.uint8)
    out_f, in_f = w.shape
    _cuda("grid", grid, torch.float32, ((out_f + 127) // 128, (in_f + 127) // 128))
    x2, m = _fused_in(x, wn, in_f)
    qs, d, z, y = _fused_outputs(x2, m, in_f, out_f, qs, d, z, y, want_z)
    rc = lib().memq_rmsnorm_q8_1_gemv_e4m3_blk128(_ptr(x2), _ptr(wn), ctypes.c_float(eps), _ptr(w),
                                                  _ptr(grid), _ptr(qs), _ptr(d), _ptr(z), _ptr(y),
                                                  out_f, in_f, m, _stream(stream))
    _check("memq_rmsnorm_q8_1_gemv_e4m3_blk128", rc)
    return y, qs, d, z


def memq_rmsnorm_q8_1_gemv_q8_0(x, wn, w, eps: float = 1e-6, *, qs=None, d=None, z=None, y=None,
                                want_z: bool = False, stream=None):
    """Fused decode step, Q8_0 weights.  Returns (y, qs, d, z)."""
    _cuda("w", w, torch.uint8)
    out_f, row_bytes = w.shape
    if row_bytes % 34 != 0:
        raise ValueError("Q8_0 rows must be a whole number of 34-byte blocks")
    in_f = row_bytes // 34 * 32
    x2, m = _fused_in(x, wn, in_f)
    qs, d, z, y = _fused_outputs(x2, m, in_f, out_f, qs, d, z, y, want_z)
    rc = lib().memq_rmsnorm_q8_1_gemv_q8_0(_ptr(x2), _ptr(wn), ctypes.c_float(eps), _ptr(w),
                                           _ptr(qs), _ptr(d), _ptr(z), _ptr(y), out_f, in_f, m,
                                           _stream(stream))
    _check("memq_rmsnorm_q8_1_gemv_q8_0", rc)
    return y, qs, d, z


def _host(name: str, t: torch.Tensor, shape):
    if (isinstance(t, torch.Tensor) and t.dtype is torch.float32 and not t.is_cuda
            and t.is_contiguous() and t.shape == shape):
        return t
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.device.type != "cpu":
        raise ValueError(f"{name} must be a host (CPU) tensor, got {t.device}")
    if t.dtype is not torch.float32 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous float32 tensor")
    raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def memq_decode_step_host(container, x_host, x_dev, wn, w, aux, y_host, eps: float = 1e-6, *,
                          qs, d, y_dev, z=None, stream=None):
    """Decode step with the activation rows and the result in host memory, in one native call:
    x_host -> x_dev, the fused step on the device buffers, y_dev -> y_host, then a wait for the
    stream.
    `container` is a Container; x_host / y_host are contiguous float32 CPU tensors (pinned for
    the asynchronous copy), every other buffer a preallocated CUDA tensor.  Returns y_host."""
    container = int(container)
    if container not in (0, 1, 2):
        raise ValueError(f"container must be a Container, got {container}")
    _cuda("w", w, torch.uint8)
    out_f, row_bytes = w.shape
    if container == Container.Q8_0:
        if row_bytes % 34 != 0:
            raise ValueError("Q8_0 rows must be a whole number of 34-byte blocks")
        in_f = row_bytes // 34 * 32
    else:
        in_f = row_bytes
        shape = (1,) if container == Container.E4M3 else ((out_f + 127) // 128, (in_f + 127) // 128)
        _cuda("aux", aux, torch.float32, shape)
    x2, m = _fused_in(x_dev, wn, in_f)
    _host("x_host", x_host if x_host.dim() == 2 else x_host.reshape(1, -1), (m, in_f))
    _host("y_host", y_host, (m, out_f))
    _cuda("qs", qs, torch.int8, (m, in_f))
    _cuda("d", d, torch.float32, (m, in_f // 32))
    _cuda("y_dev", y_dev, torch.float32, (m, out_f))
    if z is not None:
        _cuda("z", z, torch.float32, (m, in_f))
    rc = lib().memq_decode_step_host(container, _ptr(x_host), _ptr(x2), _ptr(wn),
                                     ctypes.c_float(eps), _ptr(w),
                                     None if container == Container.Q8_0 else _ptr(aux),
                                     _ptr(qs), _ptr(d), _ptr(z), _ptr(y_dev), _ptr(y_host),
                                     out_f, in_f, m, _stream(stream))
    _check("memq_decode_step_host", rc)
    return y_host


def memq_device_fault(stream=None) -> int:
    """Synchronize the stream, then read and clear the device fault word (0 = none)."""
    v = ctypes.c_uint32(0)
    rc = lib().memq_device_fault(_stream(stream), ctypes.byref(v))
    _check("memq_device_fault", rc)
    return int(v.value)


def memq_silu_mul_q8_1(gate: torch.Tensor, up: torch.Tensor, *, z=None, qs=None, d=None,
                       want_z: bool = True, stream=None):
    """silu(gate) * up -> q8_1.  gate, up: f32 [rows, ncols] (or [ncols]).

    Returns (z f32 [rows, ncols] or None, qs int8 [rows, ncols], d f32 [rows, ncols/32])."""
    g2 = gate if gate.dim() == 2 else gate.reshape(1, -1)
    u2 = up if up.dim() == 2 else up.reshape(1, -1)
    _cuda("gate", g2, torch.float32)
    rows, ncols = g2.shape
    _cuda("up", u2, torch.float32, (rows, ncols))
    if qs is None:
        qs = torch.empty((rows, ncols), dtype=torch.int8, device=g2.device)
    if d is None:
        d = torch.empty((rows, ncols // 32), dtype=torch.float32, device=g2.device)
    if z is None and want_z:
        z = torch.empty((rows, ncols), dtype=torch.float32, device=g2.device)
    _cuda("qs", qs, torch.int8, (rows, ncols))
    _cuda("d", d, torch.float32, (rows, ncols // 32))
    if z is not None:
        _cuda("z", z, torch.float32, (rows, ncols))
    rc = lib().memq_silu_mul_q8_1(_ptr(g2), _ptr(u2), _ptr(z), _ptr(qs), _ptr(d), ncols, rows,
                                  _stream(stream))
    _check("memq_silu_mul_q8_1", rc)
    return z, qs, d


def _repack(fn: str, w, aux, aux_shape, out, stream):
    _cuda("w", w, torch.uint8)
    out_f, in_f = w.shape
    _cuda("scale" if aux_shape == (1,) else "grid", aux, torch.float32, aux_shape)
    if out is None:
        out = torch.empty((out_f, in_f // 32 * 34), dtype=torch.uint8, device=w.device)
    _cuda("out", out, torch.uint8, (out_f, in_f // 32 * 34))
    rc = getattr(lib(), fn)(_ptr(w), _ptr(aux), _ptr(out), out_f, in_f, _stream(stream))
    _check(fn, rc)
    return out


def memq_repack_e4m3_q8_0(w: torch.Tensor, w_scale: torch.Tensor, *, out=None, stream=None):
    """E4M3 [out_f, in_f] with a per-tensor scale -> Q8_0 slab uint8 [out_f, in_f/32*34]."""
    return _repack("memq_repack_e4m3_q8_0", w, w_scale, (1,), out, stream)


def memq_repack_e4m3_blk128_q8_0(w: torch.Tensor, grid: torch.Tensor, *, out=None, stream=None):
    """E4M3 [out_f, in_f] with a block-128 grid -> Q8_0 slab uint8 [out_f, in_f/32*34]."""
    out_f, in_f = w.shape
    return _repack("memq_repack_e4m3_blk128_q8_0", w, grid,
                   ((out_f + 127) // 128, (in_f + 127) // 128), out, stream)


def _group(fn: str, ws, auxs, qs, d, ys, stream, aux_shape):
    count = len(ws)
    if not 1 <= count <= MAX_GROUP:
        raise ValueError(f"{fn}: 1 to {MAX_GROUP} matrices, got {count}")
    in_f = ws[0].shape[1] if ws[0].dim() == 2 else None
    for i, w in enumerate(ws):
        _cuda(f"w[{i}]", w, torch.uint8)
    qs2, d2, m = _act(qs, d, in_f)
    outs = []
    for i, w in enumerate(ws):
        out_f = w.shape[0]
        if auxs is not None:
            _cuda(f"aux[{i}]", auxs[i], torch.float32, aux_shape(out_f, in_f))
        y = None if ys is None else ys[i]
        outs.append(_out(y, m, out_f, w.device))
    VP = ctypes.c_void_p * count
    wp = VP(*[w.data_ptr() for w in ws])
    yp = VP(*[y.data_ptr() for y in outs])
    of = (ctypes.c_int64 * count)(*[w.shape[0] for w in ws])
    args = [count, wp]
    if auxs is not None:
        args.append(VP(*[a.data_ptr() for a in auxs]))
    args += [yp, of, _ptr(qs2), _ptr(d2), in_f, m, _stream(stream)]
    _check(fn, getattr(lib(), fn)(*args))
    return outs


def memq_gemv_e4m3_group(ws, w_scales, qs, d, *, ys=None, stream=None):
    """Several E4M3 GEMVs sharing one activation, one launch.  Returns [y_i]."""
    return _group("memq_gemv_e4m3_group", ws, w_scales, qs, d, ys, stream, lambda o, i: (1,))


def memq_gemv_e4m3_blk128_group(ws, grids, qs, d, *, ys=None, stream=None):
    """Several block-128 E4M3 GEMVs sharing one activation, one launch.  Returns [y_i]."""
    return _group("memq_gemv_e4m3_blk128_group", ws, grids, qs, d, ys, stream,
                  lambda o, i: ((o + 127) // 128, (i + 127) // 128))


def memq_gemv_q8_0_group(ws, qs, d, *, in_f=None, ys=None, stream=None):
    """Several Q8_0 GEMVs sharing one activation, one launch.  ws: uint8 [out_f, in_f/32*34]."""
    return _group_q8(ws, qs, d, in_f, ys, stream)


def _group_q8(ws, qs, d, in_f, ys, stream):
    count = len(ws)
    if not 1 <= count <= MAX_GROUP:
        raise ValueError(f"memq_gemv_q8_0_group: 1 to {MAX_GROUP} matrices, got {count}")
    for i, w in enumerate(ws):
        _cuda(f"w[{i}]", w, torch.uint8)
    if in_f is None:
        in_f = ws[0].shape[1] // 34 * 32
    qs2, d2, m = _act(qs, d, in_f)
    outs = [_out(None if ys is None else ys[i], m, w.shape[0], w.device) for i, w in enumerate(ws)]
    VP = ctypes.c_void_p * count
    rc = lib().memq_gemv_q8_0_group(count, VP(*[w.data_ptr() for w in ws]),
                                    VP(*[y.data_ptr() for y in outs]),
                                    (ctypes.c_int64 * count)(*[w.shape[0] for w in ws]),
                                    _ptr(qs2), _ptr(d2), in_f, m, _stream(stream))
    _check("memq_gemv_q8_0_group", rc)
    return outs


def _head_gemv(fn: str, x, w, out, split, stream):
    _cuda("x", x, torch.float32)
    _cuda("w", w, torch.float32)
    if x.dim() != 3 or w.dim() != 3:
        raise ValueError(f"{fn}: x must be [t, nh, k] and w [nh, n, k]")
    t, nh, k = x.shape
    n = w.shape[1]
    if tuple(w.shape) != (nh, n, k):
        raise ValueError(f"{fn}: w has shape {tuple(w.shape)}, expected ({nh}, n, {k})")
    if out is None:
        out = torch.empty((t, nh, n), dtype=torch.float32, device=x.device)
    _cuda("out", out, torch.float32, (t, nh, n))
    # absorb_q takes (d_nope, kv_rank) = (k, n); decompress_v takes (d_v, kv_rank) = (n, k)
    dims = (k, n) if fn == "memq_mla_absorb_q" else (n, k)
    rc = getattr(lib(), fn)(_ptr(x), _ptr(w), _ptr(out), t, nh, *dims, split, _stream(stream))
    _check(fn, rc)
    return out


def memq_mla_absorb_q(q_nope: torch.Tensor, wk_b: torch.Tensor, *, out=None, split: int = 0,
                      stream=None):
    """out[t, h, r] = sum_d q_nope[t, h, d] * wk_b[h, r, d].  q_nope f32 [t, nh, d_nope],
    wk_b f32 [nh, kv_rank, d_nope] -> f32 [t, nh, kv_rank]."""
    return _head_gemv("memq_mla_absorb_q", q_nope, wk_b, out, split, stream)


def memq_mla_decompress_v(o_lat: torch.Tensor, wv_b: torch.Tensor, *, out=None, split: int = 0,
                          stream=None):
    """out[t, h, v] = sum_r o_lat[t, h, r] * wv_b[h, v, r].  o_lat f32 [t, nh, kv_rank],
    wv_b f32 [nh, d_v, kv_rank] -> f32 [t, nh, d_v]."""
    return _head_gemv("memq_mla_decompress_v", o_lat, wv_b, out, split, stream)


def memq_mla_attn_gathered(q_lat: torch.Tensor, q_pe, cache: torch.Tensor, idx: torch.Tensor,
                           scale: float, *, out=None, split: int = 0, stream=None):
    """Softmax attention of each (t, h) query over its gathered cache rows.

    q_lat f32 [t, nh, kv_rank]; q_pe f32 [t, nh, d_rope] or None (d_rope 0);
    cache f32 [pool, kv_rank + d_rope]; idx int32 [t, n_slots] -> f32 [t, nh, kv_rank]."""
    _cuda("q_lat", q_lat, torch.float32)
    if q_lat.dim() != 3:
        raise ValueError("memq_mla_attn_gathered: q_lat must be [t, nh, kv_rank]")
    t, nh, kv_rank = q_lat.shape
    _cuda("cache", cache, torch.float32)
    if cache.dim() != 2:
        raise ValueError("memq_mla_attn_gathered: cache must be [pool, kv_rank + d_rope]")
    d_rope = cache.shape[1] - kv_rank
    if q_pe is not None:
        _cuda("q_pe", q_pe, torch.float32, (t, nh, d_rope))
    elif d_rope != 0:
        raise ValueError("memq_mla_attn_gathered: q_pe is required when d_rope > 0")
    _cuda("idx", idx, torch.int32)
    if idx.dim() != 2 or idx.shape[0] != t:
        raise ValueError(f"memq_mla_attn_gathered: idx must be [{t}, n_slots]")
    n_slots = idx.shape[1]
    if out is None:
        out = torch.empty((t, nh, kv_rank), dtype=torch.float32, device=q_lat.device)
    _cuda("out", out, torch.float32, (t, nh, kv_rank))
    rc = lib().memq_mla_attn_gathered(_ptr(q_lat), _ptr(q_pe), _ptr(cache), _ptr(idx), _ptr(out),
                                      nh, kv_rank, d_rope, t, n_slots, float(scale), split,
                                      _stream(stream))
    _check("memq_mla_attn_gathered", rc)
    return out
