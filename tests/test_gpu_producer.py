"""GPU parity of memq_rmsnorm_q8_1 (through the C ABI) against the f64 oracle."""
import numpy as np
import pytest
import torch

from gpu_helpers import check_producer, to_dev
from quantized_decode_memq_gb300 import synth

pytestmark = pytest.mark.gpu

EPS = float(np.float32(1e-6))


@pytest.fixture(scope="module")
def memq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_decode_memq_gb300 import build
    build.build()
    import quantized_decode_memq_gb300 as m
    return m


def run(memq, x, w, eps=EPS, want_z=True):
    xd, wd = to_dev(x), to_dev(w)
    z, qs, d = memq.memq_rmsnorm_q8_1(xd, wd, eps, want_z=want_z)
    torch.cuda.synchronize()
    return z, qs, d


# The PR1 reference shape (one row of 4096, page generators and seeds) and the producer sweep
# widths 1536 / 4096 / 8192 at 1 and 8 rows, plus the decode-stack widths 5120 and 17408.
@pytest.mark.parametrize("ncols,rows", [(4096, 1), (1536, 1), (8192, 1), (1536, 8), (4096, 8),
                                        (8192, 8), (5120, 1), (17408, 1), (5120, 8)])
def test_producer_page_inputs(memq, oracle, ncols, rows):
    x, w = synth.activation_rows(ncols, rows)
    z, qs, d = run(memq, x, w)
    check_producer(oracle, x, w, EPS, z, qs, d)


@pytest.mark.parametrize("ncols,rows", [(1536, 64), (4096, 64), (8192, 64), (1536, 4096),
                                        (4096, 4096), (8192, 4096)])
def test_producer_sweep_sampled(memq, oracle, ncols, rows):
    x, w = synth.activation_rows(ncols, rows, page_streams=False)
    z, qs, d = run(memq, x, w)
    sel = np.unique(np.r_[0, rows - 1, np.random.default_rng(ncols).choice(rows, 24)])
    check_producer(oracle, x, w, EPS, z, qs, d, rows=sel)


@pytest.mark.parametrize("ncols", [32, 64, 96, 160, 1056, 2080, 8224, 16416, 32768])
def test_producer_ragged_widths(memq, oracle, ncols):
    """Widths that leave partial thread slices (ragged last iteration) at every V."""
    x, w = synth.activation_rows(ncols, 3, page_streams=False)
    z, qs, d = run(memq, x, w)
    check_producer(oracle, x, w, EPS, z, qs, d)


def test_producer_without_z_matches(memq):
    x, w = synth.activation_rows(4096, 4)
    z, qs, d = run(memq, x, w, want_z=True)
    z2, qs2, d2 = run(memq, x, w, want_z=False)
    assert z2 is None
    assert torch.equal(qs, qs2) and torch.equal(d.view(torch.int32), d2.view(torch.int32))


def test_producer_degenerate_blocks(memq, oracle):
    """Zero blocks (d = 0, qs = 0), a constant row (qs = +-127) and single spikes."""
    ncols = 256
    x = np.zeros((4, ncols), np.float32)
    x[1, :] = -2.5
    x[2, 37] = 3.0
    x[3, :] = np.where(np.arange(ncols) % 2 == 0, 1.0, -1.0).astype(np.float32)
    x[3, 64:96] = 0.0
    w = np.ones(ncols, np.float32)
    z, qs, d = run(memq, x, w)
    q = qs.cpu().numpy()
    dd = d.cpu().numpy()
    assert np.all(q[0] == 0) and np.all(dd[0] == 0)
    assert np.all(q[1] == -127)
    assert q[2, 37] == 127 and np.count_nonzero(q[2]) == 1
    assert np.all(dd[3, 2] == 0) and np.all(q[3, 64:96] == 0)
    check_producer(oracle, x, w, EPS, z, qs, d)


def test_producer_eps_zero_and_large(memq, oracle):
    x, w = synth.activation_rows(512, 2, page_streams=False)
    for eps in (0.0, 1.0, 100.0):
        z, qs, d = run(memq, x, w, eps=eps)
        check_producer(oracle, x, w, eps, z, qs, d)


def test_producer_rows_zero_is_noop(memq):
    x = torch.empty((0, 128), dtype=torch.float32, device="cuda")
    w = torch.ones(128, dtype=torch.float32, device="cuda")
    z, qs, d = memq.memq_rmsnorm_q8_1(x, w)
    assert qs.shape == (0, 128)


def test_producer_argument_errors(memq):
    L = memq.lib()
    x = torch.zeros((2, 64), dtype=torch.float32, device="cuda")
    w = torch.ones(64, dtype=torch.float32, device="cuda")
    qs = torch.full((2, 64), 7, dtype=torch.int8, device="cuda")
    d = torch.zeros((2, 2), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    args = [x.data_ptr(), w.data_ptr(), None, qs.data_ptr(), d.data_ptr()]
    assert L.memq_rmsnorm_q8_1(None, *args[1:], 64, 2, 1e-6, s) == memq.Status.ERR_NULL
    assert L.memq_rmsnorm_q8_1(*args, 48, 2, 1e-6, s) == memq.Status.ERR_SHAPE
    assert L.memq_rmsnorm_q8_1(*args, 0, 2, 1e-6, s) == memq.Status.ERR_SHAPE
    assert L.memq_rmsnorm_q8_1(*args, 65536, 2, 1e-6, s) == memq.Status.ERR_SHAPE
    assert L.memq_rmsnorm_q8_1(*args, 64, -1, 1e-6, s) == memq.Status.ERR_SHAPE
    assert L.memq_rmsnorm_q8_1(*args, 64, 2, -1.0, s) == memq.Status.ERR_SHAPE
    assert L.memq_rmsnorm_q8_1(x.data_ptr() + 4, *args[1:], 64, 1, 1e-6, s) == memq.Status.ERR_ALIGN
    torch.cuda.synchronize()
    assert torch.all(qs == 7)  # nothing was written


def test_producer_on_side_stream(memq, oracle):
    x, w = synth.activation_rows(4096, 2)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        xd, wd = to_dev(x), to_dev(w)
        z, qs, d = memq.memq_rmsnorm_q8_1(xd, wd, EPS, stream=st)
    st.synchronize()
    check_producer(oracle, x, w, EPS, z, qs, d)
