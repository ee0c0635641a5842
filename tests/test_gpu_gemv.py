"""GPU parity of the three GEMVs (through the C ABI) against the f64 oracle.

Both sides are fed the same q8_1 bytes (the oracle's own quantization of seeded activations,
uploaded), so the only difference under test is the GEMV arithmetic: |y - y_ref| <= 2e-5 * S,
S = sum_i |W_i X_i|.  Full-size shapes are checked on sampled rows.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import check_gemv, sample_rows, to_dev
from quantized_decode_memq_gb300 import synth

pytestmark = pytest.mark.gpu

KINDS = ("e4m3", "blk", "q8_0")


@pytest.fixture(scope="module")
def memq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_decode_memq_gb300 import build
    build.build()
    import quantized_decode_memq_gb300 as m
    return m


def act(oracle, m, in_f, seed=101):
    """q8_1 activation rows from the oracle's producer on uniform [-4, 4) inputs."""
    x = synth.uniform_pm4(seed, m * in_f).reshape(m, in_f)
    w = synth.uniform_pm4(seed + 1, in_f)
    _, d, qs, _ = oracle.rmsnorm_q8_1(x, w)
    return qs, d


def weights(kind, out_f, in_f, seed):
    if kind == "q8_0":
        return synth.q8_0_bytes(seed, out_f, in_f), None
    w = synth.e4m3_bytes(seed, out_f, in_f)
    if kind == "blk":
        return w, synth.grid_log2_uniform(seed + 7, out_f, in_f)
    return w, np.array([2.0 ** -4], np.float32)


def gpu_gemv(memq, kind, w, aux, qs, d, y=None):
    wd, qd, dd = to_dev(w), to_dev(qs), to_dev(d)
    if kind == "q8_0":
        y = memq.memq_gemv_q8_0(wd, qd, dd, y=y)
    elif kind == "blk":
        y = memq.memq_gemv_e4m3_blk128(wd, to_dev(aux), qd, dd, y=y)
    else:
        y = memq.memq_gemv_e4m3(wd, to_dev(aux), qd, dd, y=y)
    torch.cuda.synchronize()
    return y


def ref_gemv(oracle, kind, w, aux, qs, d, in_f, rows=None):
    if kind == "q8_0":
        return oracle.gemv_q8_0(w, in_f, qs, d, rows=rows)
    if kind == "blk":
        return oracle.gemv_e4m3_blk128(w, aux, qs, d, rows=rows)
    return oracle.gemv_e4m3(w, float(aux[0]), qs, d, rows=rows)


def compare(memq, oracle, kind, out_f, in_f, m, seed=1, rows=None):
    w, aux = weights(kind, out_f, in_f, seed)
    qs, d = act(oracle, m, in_f, seed + 100)
    y = gpu_gemv(memq, kind, w, aux, qs, d)
    y_ref, s_ref = ref_gemv(oracle, kind, w, aux, qs, d, in_f, rows=rows)
    return check_gemv(y, y_ref, s_ref, rows=rows)


# Small shapes spanning several tiles / chunks with ragged tails: out_f not a multiple of the
# tile rows, in_f not a multiple of the chunk, K slices of unequal width, partial 128-tiles.
SMALL = [(1, 32), (3, 256), (37, 96), (130, 4096 + 32), (257, 1024 + 256), (1000, 2048 + 512)]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("out_f,in_f", SMALL)
@pytest.mark.parametrize("m", [1, 2, 5, 8])
def test_gemv_small(memq, oracle, kind, out_f, in_f, m):
    compare(memq, oracle, kind, out_f, in_f, m, seed=out_f + in_f + m)


def test_pr1_reference_shape(memq, oracle):
    """PR1: producer (one row of 4096, page xorshift inputs) then E4M3 1024 x 4096 from the
    page LCG generator with per-tensor scale 2^-4."""
    x, w = synth.activation_rows(4096, 1)
    _, qs_g, d_g = memq.memq_rmsnorm_q8_1(to_dev(x), to_dev(w))
    wq = synth.lcg_e4m3(1024, 4096)
    scale = np.array([2.0 ** -4], np.float32)
    y = memq.memq_gemv_e4m3(to_dev(wq), to_dev(scale), qs_g, d_g)
    torch.cuda.synchronize()
    qs, d = qs_g.cpu().numpy(), d_g.cpu().numpy()
    y_ref, s_ref = oracle.gemv_e4m3(wq, 2.0 ** -4, qs, d)
    check_gemv(y, y_ref, s_ref)


def test_q8_0_4096_square(memq, oracle):
    """Q8_0 4096 x 4096, m = 1: qs U[-127, 127], f16 scales in [2^-10, 2^-6], activation from
    the GPU producer on uniform [-4, 4)."""
    x, w = synth.activation_rows(4096, 1)
    _, qs_g, d_g = memq.memq_rmsnorm_q8_1(to_dev(x), to_dev(w))
    wq = synth.q8_0_bytes(0x51ED0002, 4096, 4096)
    y = memq.memq_gemv_q8_0(to_dev(wq), qs_g, d_g)
    torch.cuda.synchronize()
    y_ref, s_ref = oracle.gemv_q8_0(wq, 4096, qs_g.cpu().numpy(), d_g.cpu().numpy())
    check_gemv(y, y_ref, s_ref)


@pytest.mark.parametrize("kind", KINDS)
def test_17408x5120_three_arms(memq, oracle, kind):
    rows = sample_rows(17408)
    compare(memq, oracle, kind, 17408, 5120, 1, seed=0x51ED0003, rows=rows)


@pytest.mark.parametrize("kind", ["blk", "q8_0"])
@pytest.mark.parametrize("out_f,in_f", [(5120, 5120), (1024, 5120), (17408, 5120),
                                        (5120, 17408)])
@pytest.mark.parametrize("m", [1, 2, 4, 8])
def test_m_sweep_shapes(memq, oracle, kind, out_f, in_f, m):
    rows = sample_rows(out_f, 96, seed=out_f + m)
    compare(memq, oracle, kind, out_f, in_f, m, seed=out_f * 7 + in_f + m, rows=rows)


@pytest.mark.parametrize("kind", KINDS)
def test_m_batched_bit_parity(memq, oracle, kind):
    """Row j of an m-row call equals a smaller call on activation row j, bit for bit, within one
    code path: E4M3 / block-128 always run on the tensor cores (m = 8 vs m = 1); Q8_0 runs dp4a
    for m <= 2 (m = 2 vs m = 1) and the tensor cores from m = 6 on any shape (m = 8 vs m = 6).
    Across the two Q8_0 paths the block sums are the same exact integers but are added in
    another order, so m = 8 vs m = 1 agree within the GEMV tolerance instead."""
    out_f, in_f = 777, 5120
    w, aux = weights(kind, out_f, in_f, 5)
    qs, d = act(oracle, 8, in_f, 55)
    y8 = gpu_gemv(memq, kind, w, aux, qs, d)
    for j in (0, 3, 5):
        if kind == "q8_0":
            sel = [j] + [(j + i) % 8 for i in range(3, 8)]
            y6 = gpu_gemv(memq, kind, w, aux, qs[sel], d[sel])
            assert torch.equal(y8[j].view(torch.int32), y6[0].view(torch.int32))
            y2 = gpu_gemv(memq, kind, w, aux, qs[[j, (j + 4) % 8]], d[[j, (j + 4) % 8]])
            y1 = gpu_gemv(memq, kind, w, aux, qs[j:j + 1], d[j:j + 1])
            assert torch.equal(y2[0].view(torch.int32), y1[0].view(torch.int32))
            y_ref, s_ref = ref_gemv(oracle, kind, w, aux, qs[j:j + 1], d[j:j + 1], in_f)
            check_gemv(y8[j:j + 1], y_ref, s_ref)
        else:
            y1 = gpu_gemv(memq, kind, w, aux, qs[j:j + 1], d[j:j + 1])
            assert torch.equal(y8[j].view(torch.int32), y1[0].view(torch.int32))


@pytest.mark.parametrize("kind", KINDS)
def test_m_batched_bit_parity_across_kernels(memq, oracle, kind):
    """Rows of an m-batched call equal a smaller call on those activation rows, bit for bit,
    where the two calls run different kernels.  E4M3 / block-128: 5120 x 5120 at m = 8 runs the
    K-outer kernel (11-row CTAs, the activation streamed with the weights) and at m = 1 the
    tile kernel; 5120 x 17408 runs K-outer at m = 4 and m = 1.  Q8_0 (tensor-core path, K-outer):
    5120 x 5120 m = 8 against m = 4, 5120 x 17408 m = 4 against m = 3."""
    cases = ((5120, 5120, 8, 1), (5120, 17408, 4, 1))
    if kind == "q8_0":
        cases = ((5120, 5120, 8, 4), (5120, 17408, 4, 3))
    for out_f, in_f, mb, ms in cases:
        w, aux = weights(kind, out_f, in_f, 21)
        qs, d = act(oracle, mb, in_f, 77)
        yb = gpu_gemv(memq, kind, w, aux, qs, d)
        for j in (0, mb - 1):
            sel = [(j + i) % mb for i in range(ms)]
            ys = gpu_gemv(memq, kind, w, aux, qs[sel], d[sel])
            assert torch.equal(yb[j].view(torch.int32), ys[0].view(torch.int32)), (out_f, in_f, j)


def test_page_generators(memq, oracle):
    """The pages' own generators: LCG E4M3 (no NaN), the discrete 2^-6..2^-2 grid, and the
    fixed-scale Q8_0 whose qs cover the full int8 range including -128."""
    out_f, in_f = 300, 2048
    qs, d = act(oracle, 2, in_f, 9)
    w8 = synth.lcg_e4m3(out_f, in_f)
    y = gpu_gemv(memq, "e4m3", w8, np.array([1.0], np.float32), qs, d)
    check_gemv(y, *oracle.gemv_e4m3(w8, 1.0, qs, d))
    grid = synth.lcg_blk_grid(out_f, in_f)
    y = gpu_gemv(memq, "blk", w8, grid, qs, d)
    check_gemv(y, *oracle.gemv_e4m3_blk128(w8, grid, qs, d))
    wq = synth.lcg_q8_0(out_f, in_f)
    y = gpu_gemv(memq, "q8_0", wq, None, qs, d)
    check_gemv(y, *oracle.gemv_q8_0(wq, in_f, qs, d))


def test_activation_with_minus_128(memq, oracle):
    """q8_1 never emits -128, but the GEMVs accept the full int8 range in the activation."""
    out_f, in_f = 64, 512
    qs = synth.lcg_q8_0(2, in_f).reshape(-1, 34)[:, 2:].view(np.int8).reshape(2, in_f)
    assert (qs == -128).any()
    d = np.full((2, in_f // 32), 0.01, np.float32)
    for kind in KINDS:
        w, aux = weights(kind, out_f, in_f, 3)
        y = gpu_gemv(memq, kind, w, aux, qs, d)
        check_gemv(y, *ref_gemv(oracle, kind, w, aux, qs, d, in_f))


def test_zero_weights_and_zero_activation_blocks(memq, oracle):
    out_f, in_f = 96, 1024
    qs, d = act(oracle, 3, in_f, 12)
    d[:, 5:9] = 0.0
    qs[:, 160:288] = 0
    for kind in KINDS:
        w, aux = weights(kind, out_f, in_f, 4)
        w = w.copy()
        w[:10] = 0
        y = gpu_gemv(memq, kind, w, aux, qs, d)
        assert torch.all(y[:, :10] == 0)
        check_gemv(y, *ref_gemv(oracle, kind, w, aux, qs, d, in_f))


def test_nan_weight_code_propagates(memq, oracle):
    out_f, in_f = 16, 256
    qs, d = act(oracle, 1, in_f, 13)
    w, aux = weights("e4m3", out_f, in_f, 6)
    w = w.copy()
    w[3, 17] = 0x7F
    w[9, 200] = 0xFF
    y = gpu_gemv(memq, "e4m3", w, aux, qs, d).cpu().numpy()
    assert np.isnan(y[0, 3]) and np.isnan(y[0, 9])
    assert np.isfinite(np.delete(y[0], [3, 9])).all()


def test_generic_path_unaligned_and_odd_q8_0(memq, oracle):
    """Inputs the stream kernel does not take go through the generic kernel, same contract."""
    out_f, in_f, m = 50, 4096 + 32, 3
    qs, d = act(oracle, m, in_f, 14)
    # Q8_0 rows of 129 blocks are not 16-byte aligned
    wq = synth.q8_0_bytes(15, out_f, in_f)
    y = gpu_gemv(memq, "q8_0", wq, None, qs, d)
    check_gemv(y, *oracle.gemv_q8_0(wq, in_f, qs, d))
    # E4M3 weights at an odd device address
    w8 = synth.e4m3_bytes(16, out_f, in_f)
    buf = torch.zeros(w8.size + 16, dtype=torch.uint8, device="cuda")
    buf[1:1 + w8.size] = to_dev(w8.reshape(-1))
    wv = buf[1:1 + w8.size].view(out_f, in_f)
    y = memq.memq_gemv_e4m3(wv, to_dev(np.array([0.5], np.float32)), to_dev(qs), to_dev(d))
    torch.cuda.synchronize()
    check_gemv(y, *oracle.gemv_e4m3(w8, 0.5, qs, d))


def test_widest_activation(memq, oracle):
    """m = 8 x in_f = 32768 (the activation is read from L2, not staged)."""
    out_f, in_f, m = 40, 32768, 8
    qs, d = act(oracle, m, in_f, 17)
    for kind in KINDS:
        w, aux = weights(kind, out_f, in_f, 18)
        y = gpu_gemv(memq, kind, w, aux, qs, d)
        check_gemv(y, *ref_gemv(oracle, kind, w, aux, qs, d, in_f))


def test_out_f_zero_and_y_untouched_on_error(memq):
    L = memq.lib()
    s = torch.cuda.current_stream().cuda_stream
    w = torch.zeros((4, 64), dtype=torch.uint8, device="cuda")
    sc = torch.ones(1, dtype=torch.float32, device="cuda")
    qs = torch.zeros((1, 64), dtype=torch.int8, device="cuda")
    d = torch.ones((1, 2), dtype=torch.float32, device="cuda")
    y = torch.full((1, 4), 3.0, dtype=torch.float32, device="cuda")
    p = [w.data_ptr(), sc.data_ptr(), qs.data_ptr(), d.data_ptr(), y.data_ptr()]
    assert L.memq_gemv_e4m3(*p, 0, 64, 1, s) == memq.Status.OK
    assert L.memq_gemv_e4m3(*p, 4, 64, 0, s) == memq.Status.ERR_M_RANGE
    assert L.memq_gemv_e4m3(*p, 4, 64, 9, s) == memq.Status.ERR_M_RANGE
    assert L.memq_gemv_e4m3(*p, 4, 48, 1, s) == memq.Status.ERR_SHAPE
    assert L.memq_gemv_e4m3(*p, -1, 64, 1, s) == memq.Status.ERR_SHAPE
    assert L.memq_gemv_e4m3(None, *p[1:], 4, 64, 1, s) == memq.Status.ERR_NULL
    assert L.memq_gemv_e4m3(p[0], None, *p[2:], 4, 64, 1, s) == memq.Status.ERR_NULL
    assert L.memq_gemv_e4m3_blk128(p[0], None, *p[2:], 4, 64, 1, s) == memq.Status.ERR_NULL
    assert L.memq_gemv_q8_0(p[0], p[2], p[3] + 2, p[4], 4, 64, 1, s) == memq.Status.ERR_ALIGN
    torch.cuda.synchronize()
    assert torch.all(y == 3.0)


def test_repeat_calls_deterministic_and_no_fault(memq, oracle):
    out_f, in_f = 2048, 4096
    qs, d = act(oracle, 4, in_f, 19)
    for kind in KINDS:
        w, aux = weights(kind, out_f, in_f, 20)
        a = gpu_gemv(memq, kind, w, aux, qs, d)
        b = gpu_gemv(memq, kind, w, aux, qs, d)
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert memq.memq_device_fault() == 0


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("m", [1, 8])
def test_graph_back_to_back_launches(memq, oracle, kind, m):
    """Six GEMVs captured in one CUDA graph and replayed twice, as the benchmark times them:
    consecutive launches overlap (each releases the next at entry).  Every launch has its own
    weights and output; each output is checked on sampled rows."""
    out_f, in_f, n = 17408, 5120, 6
    qs, d = act(oracle, m, in_f, 77)
    qs_d, d_d = to_dev(qs), to_dev(d)
    ws = [weights(kind, out_f, in_f, 900 + i) for i in range(n)]
    wd = [(to_dev(w), None if aux is None else to_dev(aux)) for w, aux in ws]
    ys = [torch.full((m, out_f), float("nan"), device="cuda") for _ in range(n)]
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())

    def launch(i):
        w, aux = wd[i]
        if kind == "q8_0":
            memq.memq_gemv_q8_0(w, qs_d, d_d, y=ys[i])
        elif kind == "blk":
            memq.memq_gemv_e4m3_blk128(w, aux, qs_d, d_d, y=ys[i])
        else:
            memq.memq_gemv_e4m3(w, aux, qs_d, d_d, y=ys[i])

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        for i in range(n):
            launch(i)
    with torch.cuda.stream(st):
        g.replay()
        g.replay()
    st.synchronize()
    assert memq.memq_device_fault() == 0
    rows = sample_rows(out_f, 64, seed=m)
    for i, (w, aux) in enumerate(ws):
        y_ref, s_ref = ref_gemv(oracle, kind, w, aux, qs, d, in_f, rows=rows)
        check_gemv(ys[i], y_ref, s_ref, rows=rows)


@pytest.mark.parametrize("out_f", [17408, 12288])
def test_q8_0_dp4a_two_ctas_m3(memq, oracle, out_f):
    """Q8_0 at m = 3 on >= 9728 rows runs dp4a on two CTAs per SM (the tensor cores take over
    from m = 4 there): sampled rows within the GEMV tolerance of the oracle, and each row of the
    m = 3 call equal bit for bit to the m = 1 call on that activation row (dp4a at both m; its
    per-(row, token) arithmetic does not depend on m)."""
    in_f, m = 5120, 3
    w, aux = weights("q8_0", out_f, in_f, 31)
    qs, d = act(oracle, m, in_f, 91)
    y3 = gpu_gemv(memq, "q8_0", w, aux, qs, d)
    rows = sample_rows(out_f, 96, seed=out_f)
    y_ref, s_ref = ref_gemv(oracle, "q8_0", w, aux, qs, d, in_f, rows=rows)
    check_gemv(y3, y_ref, s_ref, rows=rows)
    for j in range(m):
        y1 = gpu_gemv(memq, "q8_0", w, aux, qs[j:j + 1], d[j:j + 1])
        assert torch.equal(y3[j].view(torch.int32), y1[0].view(torch.int32)), j
