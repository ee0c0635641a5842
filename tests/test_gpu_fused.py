"""GPU parity of the fused decode step (memq_rmsnorm_q8_1_gemv_*) against the f64 oracle.

The q8_1 activation the call publishes (qs, d, z) is checked like the standalone producer;
y is checked against the oracle GEMV fed those same bytes (|y - y_ref| <= 2e-5 * S).
"""
import numpy as np
import pytest
import torch

from gpu_helpers import check_gemv, check_producer, sample_rows, to_dev
from quantized_decode_memq_gb300 import synth

pytestmark = pytest.mark.gpu

EPS = float(np.float32(1e-6))
KINDS = ("e4m3", "blk", "q8_0")


@pytest.fixture(scope="module")
def memq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_decode_memq_gb300 import build
    build.build()
    import quantized_decode_memq_gb300 as m
    return m


def weights(kind, out_f, in_f, seed):
    if kind == "q8_0":
        return synth.q8_0_bytes(seed, out_f, in_f), None
    w = synth.e4m3_bytes(seed, out_f, in_f)
    if kind == "blk":
        return w, synth.grid_log2_uniform(seed + 7, out_f, in_f)
    return w, np.array([2.0 ** -4], np.float32)


def fused(memq, kind, x, wn, w, aux, wd=None):
    xd, wnd = to_dev(x), to_dev(wn)
    wd = to_dev(w) if wd is None else wd
    if kind == "q8_0":
        out = memq.memq_rmsnorm_q8_1_gemv_q8_0(xd, wnd, wd, EPS, want_z=True)
    elif kind == "blk":
        out = memq.memq_rmsnorm_q8_1_gemv_e4m3_blk128(xd, wnd, wd, to_dev(aux), EPS, want_z=True)
    else:
        out = memq.memq_rmsnorm_q8_1_gemv_e4m3(xd, wnd, wd, to_dev(aux), EPS, want_z=True)
    torch.cuda.synchronize()
    return out


def ref(oracle, kind, w, aux, qs, d, in_f, rows=None):
    if kind == "q8_0":
        return oracle.gemv_q8_0(w, in_f, qs, d, rows=rows)
    if kind == "blk":
        return oracle.gemv_e4m3_blk128(w, aux, qs, d, rows=rows)
    return oracle.gemv_e4m3(w, float(aux[0]), qs, d, rows=rows)


def run_case(memq, oracle, kind, out_f, in_f, m, seed, rows=None, page=True):
    x, wn = synth.activation_rows(in_f, m, page_streams=page)
    w, aux = weights(kind, out_f, in_f, seed)
    y, qs, d, z = fused(memq, kind, x, wn, w, aux)
    check_producer(oracle, x, wn, EPS, z, qs, d)
    qs_h, d_h = qs.cpu().numpy(), d.cpu().numpy()
    check_gemv(y, *ref(oracle, kind, w, aux, qs_h, d_h, in_f, rows=rows), rows=rows)
    assert memq.memq_device_fault() == 0


@pytest.mark.parametrize("kind", KINDS)
# in_f / 32 divisible by 8 runs the clustered prologue (8 CTAs share the RMSNorm -> q8_1);
# 96 and 1056 (3 and 33 blocks) take the per-CTA prologue.
@pytest.mark.parametrize("out_f,in_f,m", [(4096, 4096, 1), (1024, 4096, 1), (37, 256, 1),
                                          (257, 1024 + 256, 3), (777, 5120, 8), (5120, 5120, 2),
                                          (300, 17408, 1), (3, 512, 2), (129, 96, 1),
                                          (500, 1024 + 32, 4)])
def test_fused_parity(memq, oracle, kind, out_f, in_f, m):
    rows = sample_rows(out_f, 128, seed=out_f + m) if out_f > 1024 else None
    run_case(memq, oracle, kind, out_f, in_f, m, seed=out_f + in_f + m, rows=rows)


@pytest.mark.parametrize("kind", KINDS)
def test_fused_17408x5120(memq, oracle, kind):
    run_case(memq, oracle, kind, 17408, 5120, 1, seed=0x51ED0003, rows=sample_rows(17408))


def test_fused_fallback_paths(memq, oracle):
    """Q8_0 rows of 129 blocks and E4M3 weights at an odd address take the two-launch path."""
    run_case(memq, oracle, "q8_0", 50, 4096 + 32, 2, seed=3)
    in_f, out_f = 1024, 64
    x, wn = synth.activation_rows(in_f, 1)
    w8 = synth.e4m3_bytes(4, out_f, in_f)
    buf = torch.zeros(w8.size + 16, dtype=torch.uint8, device="cuda")
    buf[3:3 + w8.size] = to_dev(w8.reshape(-1))
    wv = buf[3:3 + w8.size].view(out_f, in_f)
    aux = np.array([0.5], np.float32)
    y, qs, d, z = fused(memq, "e4m3", x, wn, w8, aux, wd=wv)
    check_producer(oracle, x, wn, EPS, z, qs, d)
    check_gemv(y, *oracle.gemv_e4m3(w8, 0.5, qs.cpu().numpy(), d.cpu().numpy()))


def test_fused_out_f_zero_still_produces_activation(memq, oracle):
    L = memq.lib()
    in_f = 512
    x, wn = synth.activation_rows(in_f, 2)
    xd, wnd = to_dev(x), to_dev(wn)
    qs = torch.zeros((2, in_f), dtype=torch.int8, device="cuda")
    d = torch.zeros((2, in_f // 32), dtype=torch.float32, device="cuda")
    z = torch.zeros((2, in_f), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = L.memq_rmsnorm_q8_1_gemv_q8_0(xd.data_ptr(), wnd.data_ptr(), EPS, None, qs.data_ptr(),
                                       d.data_ptr(), z.data_ptr(), None, 0, in_f, 2, s)
    assert rc == 0
    torch.cuda.synchronize()
    check_producer(oracle, x, wn, EPS, z, qs, d)


def test_fused_matches_split_chain(memq, oracle):
    """The fused step and producer + GEMV agree within the GEMV tolerance on the same inputs."""
    out_f, in_f = 2048, 4096
    x, wn = synth.activation_rows(in_f, 1)
    for kind in KINDS:
        w, aux = weights(kind, out_f, in_f, 9)
        y_f, qs_f, d_f, _ = fused(memq, kind, x, wn, w, aux)
        _, qs_s, d_s = memq.memq_rmsnorm_q8_1(to_dev(x), to_dev(wn), EPS)
        if kind == "q8_0":
            y_s = memq.memq_gemv_q8_0(to_dev(w), qs_s, d_s)
        elif kind == "blk":
            y_s = memq.memq_gemv_e4m3_blk128(to_dev(w), to_dev(aux), qs_s, d_s)
        else:
            y_s = memq.memq_gemv_e4m3(to_dev(w), to_dev(aux), qs_s, d_s)
        torch.cuda.synchronize()
        _, s_ref = ref(oracle, kind, w, aux, qs_f.cpu().numpy(), d_f.cpu().numpy(), in_f)
        diff = (y_f.double() - y_s.double()).abs().cpu().numpy()
        # both are within 2e-5*S of the oracle on their own activation; the activations differ
        # at most in rare +-1 codes next to a .5 boundary
        assert np.all(diff <= 1e-4 * s_ref)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("out_f,in_f,m,pinned", [(4096, 4096, 1, True), (777, 5120, 3, False),
                                                 (5120, 5120, 8, True)])
def test_decode_step_host_matches_fused(memq, oracle, kind, out_f, in_f, m, pinned):
    """memq_decode_step_host: x from host memory, the fused step, y back to host memory, in one
    call.  y_host, qs, d and z equal those of memq_rmsnorm_q8_1_gemv_* on the same device inputs
    bit for bit, with page-locked and with pageable host buffers, on two calls in a row; y is
    within the GEMV tolerance of the oracle."""
    x, wn = synth.activation_rows(in_f, m)
    w, aux = weights(kind, out_f, in_f, out_f + m)
    wd, wnd = to_dev(w), to_dev(wn)
    auxd = None if aux is None else to_dev(aux)
    y_ref, qs_ref, d_ref, z_ref = fused(memq, kind, x, wn, w, aux, wd=wd)
    container = {"e4m3": memq.Container.E4M3, "blk": memq.Container.E4M3_BLK128,
                 "q8_0": memq.Container.Q8_0}[kind]
    x_host = torch.from_numpy(x.copy())
    y_host = torch.full((m, out_f), float("nan"))
    if pinned:
        x_host, y_host = x_host.pin_memory(), y_host.pin_memory()
    x_dev = torch.empty((m, in_f), dtype=torch.float32, device="cuda")
    qs = torch.empty((m, in_f), dtype=torch.int8, device="cuda")
    d = torch.empty((m, in_f // 32), dtype=torch.float32, device="cuda")
    z = torch.empty((m, in_f), dtype=torch.float32, device="cuda")
    y_dev = torch.empty((m, out_f), dtype=torch.float32, device="cuda")
    for _ in range(2):
        out = memq.memq_decode_step_host(container, x_host, x_dev, wnd, wd, auxd, y_host, EPS,
                                         qs=qs, d=d, y_dev=y_dev, z=z)
        assert out is y_host
        # the call has waited: y_host is final without a synchronize
        assert torch.equal(y_host, y_ref.cpu())
        assert torch.equal(x_dev.cpu(), x_host)
        assert torch.equal(qs.cpu(), qs_ref.cpu()) and torch.equal(d.cpu(), d_ref.cpu())
        assert torch.equal(z.cpu(), z_ref.cpu())
        y_host.fill_(float("nan"))
    memq.memq_decode_step_host(container, x_host, x_dev, wnd, wd, auxd, y_host, EPS, qs=qs, d=d,
                               y_dev=y_dev)
    rows = sample_rows(out_f, 64, seed=m) if out_f > 1024 else None
    check_gemv(y_host, *ref(oracle, kind, w, aux, qs.cpu().numpy(), d.cpu().numpy(), in_f,
                            rows=rows), rows=rows)
    assert memq.memq_device_fault() == 0


def test_decode_step_host_rejects_before_copying(memq):
    """A bad argument returns its status and leaves every buffer untouched."""
    L = memq.lib()
    in_f, out_f = 512, 64
    x_host = torch.ones((1, in_f)).pin_memory()
    x_dev = torch.zeros((1, in_f), dtype=torch.float32, device="cuda")
    wn = torch.ones(in_f, dtype=torch.float32, device="cuda")
    w = torch.zeros((out_f, in_f // 32 * 34), dtype=torch.uint8, device="cuda")
    qs = torch.zeros((1, in_f), dtype=torch.int8, device="cuda")
    d = torch.zeros((1, in_f // 32), dtype=torch.float32, device="cuda")
    y_dev = torch.zeros((1, out_f), dtype=torch.float32, device="cuda")
    y_host = torch.zeros((1, out_f)).pin_memory()
    s = torch.cuda.current_stream().cuda_stream
    args = [x_host.data_ptr(), x_dev.data_ptr(), wn.data_ptr(), EPS, w.data_ptr(), None,
            qs.data_ptr(), d.data_ptr(), None, y_dev.data_ptr(), y_host.data_ptr(), out_f, in_f]
    assert L.memq_decode_step_host(5, *args, 1, s) == memq.Status.ERR_SHAPE
    assert L.memq_decode_step_host(int(memq.Container.Q8_0), *args, 9, s) == memq.Status.ERR_M_RANGE
    assert L.memq_decode_step_host(int(memq.Container.E4M3), *args, 1, s) == memq.Status.ERR_NULL
    torch.cuda.synchronize()
    assert not x_dev.any() and not y_dev.any() and not y_host.any()


def test_decode_step_host_out_f_zero(memq, oracle):
    """out_f == 0: the call copies x in, produces the q8_1 activation (as the producer alone
    would) and waits; w and y_host may be NULL."""
    L = memq.lib()
    in_f, m = 1024, 2
    x, wn = synth.activation_rows(in_f, m)
    x_host = torch.from_numpy(x.copy()).pin_memory()
    x_dev = torch.zeros((m, in_f), dtype=torch.float32, device="cuda")
    wnd = to_dev(wn)
    qs = torch.zeros((m, in_f), dtype=torch.int8, device="cuda")
    d = torch.zeros((m, in_f // 32), dtype=torch.float32, device="cuda")
    z = torch.zeros((m, in_f), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = L.memq_decode_step_host(int(memq.Container.Q8_0), x_host.data_ptr(), x_dev.data_ptr(),
                                 wnd.data_ptr(), EPS, None, None, qs.data_ptr(), d.data_ptr(),
                                 z.data_ptr(), None, None, 0, in_f, m, s)
    assert rc == 0
    assert torch.equal(x_dev.cpu(), x_host)
    check_producer(oracle, x, wn, EPS, z, qs, d)
