"""GPU parity of the grouped GEMVs (several weight matrices sharing one activation, one launch).

Every output of a group equals the single-matrix call on the same matrix bit for bit (a row's
arithmetic does not depend on which CTA streams it), and matches the oracle within the GEMV
tolerance on sampled rows.  m in {1, 2, 8}: there a single Q8_0 call and the group take the same
code path (dp4a up to m = 2, the tensor cores from m = 6).
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


def weights(kind, out_f, in_f, seed):
    if kind == "q8_0":
        return synth.q8_0_bytes(seed, out_f, in_f), None
    w = synth.e4m3_bytes(seed, out_f, in_f)
    if kind == "blk":
        return w, synth.grid_log2_uniform(seed + 1, out_f, in_f)
    return w, np.array([2.0 ** -(3 + seed % 3)], np.float32)


def single(memq, kind, w, aux, qs, d):
    if kind == "q8_0":
        return memq.memq_gemv_q8_0(w, qs, d)
    if kind == "blk":
        return memq.memq_gemv_e4m3_blk128(w, aux, qs, d)
    return memq.memq_gemv_e4m3(w, aux, qs, d)


def group(memq, kind, ws, auxs, qs, d):
    if kind == "q8_0":
        return memq.memq_gemv_q8_0_group(ws, qs, d)
    if kind == "blk":
        return memq.memq_gemv_e4m3_blk128_group(ws, auxs, qs, d)
    return memq.memq_gemv_e4m3_group(ws, auxs, qs, d)


def ref(oracle, kind, w, aux, qs, d, in_f, rows):
    if kind == "q8_0":
        return oracle.gemv_q8_0(w, in_f, qs, d, rows=rows)
    if kind == "blk":
        return oracle.gemv_e4m3_blk128(w, aux, qs, d, rows=rows)
    return oracle.gemv_e4m3(w, float(aux[0]), qs, d, rows=rows)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("m", [1, 2, 8])
@pytest.mark.parametrize("shapes,in_f", [((6144, 5120), 5120), ((17408, 17408), 5120),
                                         ((37, 130, 1000), 1024 + 256), ((5120, 33, 700, 1), 2048),
                                         ((5120, 5120), 17408)])
def test_group_equals_single_calls_and_oracle(memq, oracle, kind, m, shapes, in_f):
    x = synth.uniform_pm4(0x7700 + m, m * in_f).reshape(m, in_f)
    _, d, qs, _ = oracle.rmsnorm_q8_1(x, synth.uniform_pm4(0x7701, in_f))
    host = [weights(kind, o, in_f, 0x7710 + 3 * i) for i, o in enumerate(shapes)]
    ws = [to_dev(w) for w, _ in host]
    auxs = None if kind == "q8_0" else [to_dev(a) for _, a in host]
    qd, dd = to_dev(qs), to_dev(d)
    ys = group(memq, kind, ws, auxs, qd, dd)
    torch.cuda.synchronize()
    assert memq.memq_device_fault() == 0
    for i, (w, aux) in enumerate(host):
        y1 = single(memq, kind, ws[i], None if auxs is None else auxs[i], qd, dd)
        torch.cuda.synchronize()
        assert torch.equal(ys[i].view(torch.int32), y1.view(torch.int32)), f"matrix {i}"
        rows = sample_rows(shapes[i], 64, seed=i) if shapes[i] > 2048 else None
        check_gemv(ys[i], *ref(oracle, kind, w, aux, qs, d, in_f, rows), rows=rows)


def test_group_in_a_graph_back_to_back(memq, oracle):
    """Grouped launches replayed from a CUDA graph, alternating with single ones."""
    in_f = 5120
    x = synth.uniform_pm4(0x7800, in_f).reshape(1, in_f)
    _, d, qs, _ = oracle.rmsnorm_q8_1(x, synth.uniform_pm4(0x7801, in_f))
    host = [weights("blk", o, in_f, 0x7810 + i) for i, o in enumerate((17408, 17408, 5120))]
    ws = [to_dev(w) for w, _ in host]
    gs = [to_dev(g) for _, g in host]
    qd, dd = to_dev(qs), to_dev(d)
    ys = [torch.full((1, o), float("nan"), device="cuda") for o in (17408, 17408, 5120)]
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        for _ in range(3):
            memq.memq_gemv_e4m3_blk128_group(ws[:2], gs[:2], qd, dd, ys=ys[:2])
            memq.memq_gemv_e4m3_blk128(ws[2], gs[2], qd, dd, y=ys[2])
    with torch.cuda.stream(st):
        g.replay()
    st.synchronize()
    assert memq.memq_device_fault() == 0
    for i, (w, grid) in enumerate(host):
        rows = sample_rows(w.shape[0], 64, seed=i)
        check_gemv(ys[i], *oracle.gemv_e4m3_blk128(w, grid, qs, d, rows=rows), rows=rows)
