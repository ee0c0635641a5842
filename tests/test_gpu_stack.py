"""GPU parity of the decode chain layered like a transformer block, teacher-forced per stage.

Each layer: RMSNorm -> q8_1 on the 5120-wide input; block-128 E4M3 GEMVs 5120->6144 and
5120->5120 on it; RMSNorm -> q8_1 of the 5120 output; GEMVs 5120->17408 (gate, up) on that;
RMSNorm -> q8_1 of the 17408 up output; GEMV 17408->5120, whose output feeds the next layer.
All launches go back to back on one stream, as in a decode step.  Each stage is then checked
against the oracle fed the GPU's own inputs to that stage (the previous stage's GPU output), so
one stage's rounding never counts against the next.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import check_gemv, check_producer, sample_rows, to_dev
from quantized_decode_memq_gb300 import synth

pytestmark = pytest.mark.gpu

EPS = float(np.float32(1e-6))
SHAPES = ((6144, 5120), (5120, 5120), (17408, 5120), (17408, 5120), (5120, 17408))
# (norm input, GEMVs fed by that norm): norm k reads the output of GEMV SRC[k]
NORMS = ((None, (0, 1)), (1, (2, 3)), (3, (4,)))


@pytest.fixture(scope="module")
def memq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_decode_memq_gb300 import build
    build.build()
    import quantized_decode_memq_gb300 as m
    return m


def test_two_layer_chain_teacher_forced(memq, oracle):
    layers = 2
    w = [[synth.e4m3_bytes(0x5A00 + 8 * l + k, o, i) for k, (o, i) in enumerate(SHAPES)]
         for l in range(layers)]
    g = [[synth.grid_log2_uniform(0x5B00 + 8 * l + k, o, i) for k, (o, i) in enumerate(SHAPES)]
         for l in range(layers)]
    wn = [synth.uniform_pm4(0x5C00 + k, n) for k, n in enumerate((5120, 5120, 17408))]
    x0, _ = synth.activation_rows(5120, 1)
    wd = [[to_dev(a) for a in row] for row in w]
    gd = [[to_dev(a) for a in row] for row in g]
    wnd = [to_dev(a) for a in wn]

    # run every layer back to back, keeping each stage's output for the checks
    outs = []
    x = to_dev(x0)
    for l in range(layers):
        ys, acts, ins = [None] * 5, [], []
        for k, (src, gemvs) in enumerate(NORMS):
            inp = x if src is None else ys[src]
            ins.append(inp)
            z, qs, d = memq.memq_rmsnorm_q8_1(inp, wnd[k], EPS)
            acts.append((z, qs, d))
            for j in gemvs:
                ys[j] = memq.memq_gemv_e4m3_blk128(wd[l][j], gd[l][j], qs, d)
        outs.append((ins, acts, ys))
        x = ys[4]
    torch.cuda.synchronize()
    assert memq.memq_device_fault() == 0

    for l, (ins, acts, ys) in enumerate(outs):
        for k, (src, gemvs) in enumerate(NORMS):
            xin = ins[k].cpu().numpy().reshape(1, -1)
            assert np.all(np.isfinite(xin))
            z, qs, d = acts[k]
            check_producer(oracle, xin, wn[k], EPS, z, qs, d)
            qs_h, d_h = qs.cpu().numpy(), d.cpu().numpy()
            for j in gemvs:
                rows = sample_rows(SHAPES[j][0], 128, seed=l * 8 + j)
                y_ref, s_ref = oracle.gemv_e4m3_blk128(w[l][j], g[l][j], qs_h, d_h, rows=rows)
                check_gemv(ys[j], y_ref, s_ref, rows=rows)


def test_repeated_gemv_to_norm_handoff(memq, oracle):
    """A GEMV followed at once by the RMSNorm of its output, 40 times, launched back to back.

    Every launch releases its successor at entry, so each RMSNorm starts while the GEMV before
    it is still finishing; it must read the GEMV's final output.  Each z is checked against the
    oracle on the GEMV output as read back afterwards (both widths of the producer kernel)."""
    reps = 40
    w_up = to_dev(synth.e4m3_bytes(0x5D00, 17408, 5120))
    g_up = to_dev(synth.grid_log2_uniform(0x5D01, 17408, 5120))
    w_dn = to_dev(synth.e4m3_bytes(0x5D02, 5120, 17408))
    g_dn = to_dev(synth.grid_log2_uniform(0x5D03, 5120, 17408))
    wn_up = synth.uniform_pm4(0x5D04, 17408)
    wn_dn = synth.uniform_pm4(0x5D05, 5120)
    wn_up_d, wn_dn_d = to_dev(wn_up), to_dev(wn_dn)
    x0, _ = synth.activation_rows(5120, 1)
    _, qs, d = memq.memq_rmsnorm_q8_1(to_dev(x0), wn_dn_d, EPS)
    keep = []
    for _ in range(reps):
        y_up = memq.memq_gemv_e4m3_blk128(w_up, g_up, qs, d)
        z1, qs1, d1 = memq.memq_rmsnorm_q8_1(y_up, wn_up_d, EPS)
        y_dn = memq.memq_gemv_e4m3_blk128(w_dn, g_dn, qs1, d1)
        z2, qs, d = memq.memq_rmsnorm_q8_1(y_dn, wn_dn_d, EPS)
        keep.append((y_up, z1, qs1, d1, y_dn, z2, qs, d))
    torch.cuda.synchronize()
    assert memq.memq_device_fault() == 0
    for y_up, z1, qs1, d1, y_dn, z2, qs2, d2 in keep:
        check_producer(oracle, y_up.cpu().numpy(), wn_up, EPS, z1, qs1, d1)
        check_producer(oracle, y_dn.cpu().numpy(), wn_dn, EPS, z2, qs2, d2)


def test_stack48_teacher_forced_layers(memq, oracle):
    """One token through the 48-layer block-128 stack (each layer its own device copy of the
    weights, 15.6 GB), launched back to back; layers 0, 23 and 47 are checked stage by stage
    against the oracle fed the GPU's own inputs to each stage (teacher forcing), GEMVs on
    sampled rows.  The end state after 48 re-quantizations is not compared with an oracle run
    of its own (rounding flips compound); it is only required to be finite."""
    layers, check = 48, (0, 23, 47)
    w = [synth.e4m3_bytes(0x5E00 + k, o, i) for k, (o, i) in enumerate(SHAPES)]
    g = [synth.grid_log2_uniform(0x5F00 + k, o, i) for k, (o, i) in enumerate(SHAPES)]
    wn = [synth.uniform_pm4(0x6000 + k, n) for k, n in enumerate((5120, 5120, 17408))]
    x0, _ = synth.activation_rows(5120, 1)
    base_w, base_g = [to_dev(a) for a in w], [to_dev(a) for a in g]
    wd = [[t.clone() for t in base_w] for _ in range(layers)]
    gd = [[t.clone() for t in base_g] for _ in range(layers)]
    wnd = [to_dev(a) for a in wn]
    keep = {}
    x = to_dev(x0)
    for l in range(layers):
        ys, acts, ins = [None] * 5, [], []
        for k, (src, gemvs) in enumerate(NORMS):
            inp = x if src is None else ys[src]
            ins.append(inp)
            z, qs, d = memq.memq_rmsnorm_q8_1(inp, wnd[k], EPS)
            acts.append((z, qs, d))
            for j in gemvs:
                ys[j] = memq.memq_gemv_e4m3_blk128(wd[l][j], gd[l][j], qs, d)
        if l in check:
            keep[l] = (ins, acts, ys)
        x = ys[4]
    torch.cuda.synchronize()
    assert memq.memq_device_fault() == 0
    assert torch.isfinite(x).all()
    del wd, gd
    for l in check:
        ins, acts, ys = keep[l]
        for k, (src, gemvs) in enumerate(NORMS):
            xin = ins[k].cpu().numpy().reshape(1, -1)
            assert np.all(np.isfinite(xin))
            z, qs, d = acts[k]
            check_producer(oracle, xin, wn[k], EPS, z, qs, d)
            qs_h, d_h = qs.cpu().numpy(), d.cpu().numpy()
            for j in gemvs:
                rows = sample_rows(SHAPES[j][0], 96, seed=100 * l + j)
                y_ref, s_ref = oracle.gemv_e4m3_blk128(w[j], g[j], qs_h, d_h, rows=rows)
                check_gemv(ys[j], y_ref, s_ref, rows=rows)
