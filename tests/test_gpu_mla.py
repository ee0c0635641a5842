"""GPU parity of the MLA decode attention kernels against the oracle.

mla_decode_arm_gate.rs (module doc and `main`): absorb_q, decompress_v and attn_gathered at
the page's geometry (64 heads, kv_rank 512, d_nope = d_v = 256, d_rope 0, 2048 gathered slots,
t in {1, 2, 4, 8}, pools of kv cached rows), plus ragged shapes and the rope path.  Two checks:

1. Against the f64 oracle, within bounds derived from the f32 arithmetic of each kernel:
   - absorb_q / decompress_v: a dot of k products, each lane summing k/32 of them in order and a
     5-level tree over the lanes: |err| <= (k/32 + 5 + 1) * 2^-24 * sum |terms|.  The test uses
     the GEMV tolerance 2e-5 * sum |terms|, above that bound for k <= 1024.
   - attn_gathered: attn_bound() below.
2. The page's BIT-IDENTITY gate: every split gives the same output bits as split 1.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import GEMV_TOL, to_dev
from quantized_decode_memq_gb300 import synth

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


@pytest.fixture(scope="module")
def memq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_decode_memq_gb300 import build
    build.build()
    import quantized_decode_memq_gb300 as m
    return m


def check_head(y_gpu, ref, sabs):
    y = y_gpu.double().cpu().numpy()
    assert y.shape == ref.shape
    err = np.abs(y - ref)
    assert np.all(err <= GEMV_TOL * sabs), f"worst {(err / np.maximum(sabs, 1e-300)).max():.3e}"


def assert_bits_equal(a: torch.Tensor, b: torch.Tensor, what: str):
    av = a.cpu().numpy().view(np.uint32)
    bv = b.cpu().numpy().view(np.uint32)
    assert np.array_equal(av, bv), f"{what}: {np.sum(av != bv)} of {av.size} outputs differ"


# --------------------------------------------------------------------------- absorb / decompress
@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_absorb_q_page_geometry(memq, oracle, t):
    q, w = synth.mla_absorb_inputs(t)
    dq, dw = to_dev(q), to_dev(w)
    base = memq.memq_mla_absorb_q(dq, dw, split=1)
    torch.cuda.synchronize()
    ref, sabs = oracle.mla_absorb_q(q, w)
    check_head(base, ref, sabs)
    for split in (2, 4, 8, 0, 7):
        assert_bits_equal(memq.memq_mla_absorb_q(dq, dw, split=split), base, f"split {split}")


@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_decompress_v_page_geometry(memq, oracle, t):
    o, w = synth.mla_decompress_inputs(t)
    do, dw = to_dev(o), to_dev(w)
    base = memq.memq_mla_decompress_v(do, dw, split=1)
    torch.cuda.synchronize()
    ref, sabs = oracle.mla_decompress_v(o, w)
    check_head(base, ref, sabs)
    for split in (2, 4, 8, 0, 5):
        assert_bits_equal(memq.memq_mla_decompress_v(do, dw, split=split), base, f"split {split}")


@pytest.mark.parametrize("t,nh,rows,cols", [(1, 1, 1, 128), (3, 5, 37, 128), (8, 3, 129, 1024),
                                            (2, 7, 300, 384 + 128)])
def test_head_gemv_ragged(memq, oracle, t, nh, rows, cols):
    x = synth.uniform_pm4(0x8100 + rows, t * nh * cols).reshape(t, nh, cols)
    w = synth.uniform_pm4(0x8101 + cols, nh * rows * cols).reshape(nh, rows, cols)
    dx, dw = to_dev(x), to_dev(w)
    base = memq.memq_mla_absorb_q(dx, dw, split=1)
    torch.cuda.synchronize()
    ref, sabs = oracle.mla_head_gemv(x, w)
    check_head(base, ref, sabs)
    for split in (2, 3, rows, rows + 5):
        assert_bits_equal(memq.memq_mla_absorb_q(dx, dw, split=split), base, f"split {split}")
    # decompress_v is the same contraction with the roles of the names swapped
    assert_bits_equal(memq.memq_mla_decompress_v(dx, dw, split=2), base, "decompress_v")


# --------------------------------------------------------------------------- attn_gathered
def tensor_core_attn(t, kv_rank, d_rope):
    """attn_gathered takes its tensor-core kernel (3xTF32) for t >= 2, d_rope == 0 and
    kv_rank <= 512."""
    return t >= 2 and d_rope == 0 and kv_rank <= 512


def attn_bound(q_lat, q_pe, cache, idx, scale, cabs):
    """Per-output bound on |out_gpu - out_oracle| for attn_gathered's f32 arithmetic.

    A score s_j = scale * (q . c_j) is a lane chain of kv_rank/32 + ceil(d_rope/32) fmas, a
    5-level tree and one multiply: |e_j| <= (kv_rank/32 + ceil(d_rope/32) + 6) u scale S_j with
    S_j = sum |q_i c_ji|.  A weight exp(s_j - m) then carries relative error at most
    3 E + (chunks + 2)(3u + u R)  (E = max e_j, R = 2 max |s_j| bounds |s_j - m|: the score
    error, the shared running max, each subtraction, expf's 2-ulp error, and one rescale factor
    per staged chunk).  A relative weight error delta moves the normalised output by at most
    2 delta max_j |c_j[r]|; the numerator and denominator sums (at most per + chunks + 8 roundings
    each, in a part and the 8-way merge) add 2 gamma max_j |c_j[r]|, gamma = (per + chunks + 10) u.

    Tensor-core kernel (3xTF32): a product x y is hi_x hi_y + hi_x lo_y + lo_x hi_y with hi the
    TF32 truncation (exact) and lo = x - hi taken by the MMA at TF32 precision, so it carries
    |lo_x lo_y| + the truncation of both lo parts <= 3 2^-20 |x y| = 48 u |x y|.  Every MMA is
    counted as adding its 8 products to the running sum one rounding at a time (the hardware
    order is not specified), so a score is a chain of at most 3 kv_rank / 8 additions (one warp's
    K slice in three terms), 2 for the chain combine, 8 for the warp partials and the scale:
    k_ops = 48 + 3 kv_rank / 8 + 11.  The output sums likewise: 48 u per product and three terms
    per row, gamma = (48 + 3 per + chunks + 10) u.
    """
    t, nh, kv_rank = q_lat.shape
    n_slots = idx.shape[1]
    d_rope = cache.shape[1] - kv_rank
    per = -(-(-(-n_slots // 8)) // 16) * 16
    chunks = -(-per // 16)
    tc = tensor_core_attn(t, kv_rank, d_rope)
    k_ops = 48 + 3 * kv_rank / 8 + 11 if tc else kv_rank / 32 + -(-d_rope // 32) + 6
    bound = np.empty((t, nh), np.float64)
    for tt in range(t):
        c = np.abs(cache[idx[tt]].astype(np.float64))               # [n_slots, row]
        q = np.abs(q_lat[tt].astype(np.float64))                     # [nh, kv_rank]
        s_abs = q @ c[:, :kv_rank].T
        if d_rope:
            s_abs += np.abs(q_pe[tt].astype(np.float64)) @ c[:, kv_rank:].T
        s_abs *= scale
        e = k_ops * U * s_abs.max(axis=1)
        r = 2.0 * s_abs.max(axis=1)
        delta = 3.0 * e + (chunks + 2) * (3.0 * U + U * r)
        gamma = ((48 + 3 * per) if tc else per) * U + (chunks + 10) * U
        bound[tt] = 2.0 * delta + 2.0 * gamma
    return bound[:, :, None] * cabs


def run_attn(memq, oracle, q_lat, q_pe, cache, idx, scale, splits=(2, 4, 8, 0)):
    dq = to_dev(q_lat)
    dpe = None if q_pe is None else to_dev(q_pe)
    dc, di = to_dev(cache), to_dev(idx)
    base = memq.memq_mla_attn_gathered(dq, dpe, dc, di, scale, split=1)
    torch.cuda.synchronize()
    d_rope = cache.shape[1] - q_lat.shape[2]
    ref, cabs = oracle.mla_attn_gathered(q_lat, q_pe, cache, idx, scale, d_rope=d_rope)
    got = base.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref)
    bound = attn_bound(q_lat, q_pe, cache, idx, scale, cabs)
    assert np.all(err <= bound), f"worst err/bound {(err / bound).max():.3f}"
    for split in splits:
        out = memq.memq_mla_attn_gathered(dq, dpe, dc, di, scale, split=split)
        assert_bits_equal(out, base, f"split {split}")
    assert memq.memq_device_fault() == 0
    return float((err / np.maximum(cabs, 1e-300)).max())


@pytest.mark.parametrize("t,kv", [(1, 2048), (2, 2048), (4, 32768), (8, 32768)])
def test_attn_gathered_page_geometry(memq, oracle, t, kv):
    q_lat, q_pe, cache, idx = synth.mla_attn_inputs(t, kv)
    run_attn(memq, oracle, q_lat, q_pe, cache, idx, synth.MLA_SCALE)


@pytest.mark.parametrize("t,nh,kv_rank,d_rope,kv,n_slots", [
    (1, 1, 128, 0, 40, 1),          # one slot: the output is that row
    (3, 5, 128, 64, 300, 37),       # rope path, partial chunks, empty slot parts
    (2, 9, 256, 3, 100, 130),       # rows not float4-aligned (row length 259)
    (1, 64, 512, 0, 4096, 2048),    # pool larger than the gather
    (2, 6, 1024, 128, 500, 333),    # the largest row the kernel takes
    (8, 2, 256, 32, 64, 2048),      # indices repeat (gather wider than the pool)
    (2, 5, 128, 0, 300, 37),        # tensor cores: partial head group, partial chunks, empty parts
    (4, 9, 256, 0, 100, 130),       # tensor cores: 9 heads (groups of 8 + 1), ragged slots
    (3, 64, 512, 0, 64, 2048),      # tensor cores: indices repeat
])
def test_attn_gathered_ragged(memq, oracle, t, nh, kv_rank, d_rope, kv, n_slots):
    q_lat, q_pe, cache, idx = synth.mla_attn_inputs(t, kv, nh=nh, kv_rank=kv_rank, d_rope=d_rope,
                                                     n_slots=n_slots)
    run_attn(memq, oracle, q_lat, q_pe, cache, idx, 1.0 / np.sqrt(kv_rank + d_rope))


@pytest.mark.parametrize("d_rope", [0, 32])
def test_attn_gathered_one_slot_is_the_row(memq, d_rope):
    """A single gathered slot has softmax weight 1: the output is the gathered row.  Exactly with
    the f32 kernel (d_rope = 32); with the tensor-core kernel (d_rope = 0) the weight-1 product is
    hi + (x - hi) at TF32 precision, so each element is the row's within 2^-20 relative."""
    q_lat, q_pe, cache, idx = synth.mla_attn_inputs(2, 50, nh=3, kv_rank=256, d_rope=d_rope,
                                                     n_slots=1)
    dpe = None if q_pe is None else to_dev(q_pe)
    out = memq.memq_mla_attn_gathered(to_dev(q_lat), dpe, to_dev(cache), to_dev(idx), 0.1)
    got = out.cpu().numpy()
    for tt in range(2):
        for h in range(3):
            row = cache[idx[tt, 0], :256]
            if tensor_core_attn(2, 256, d_rope):
                assert np.all(np.abs(got[tt, h].astype(np.float64) - row) <= 2.0 ** -20 * np.abs(row))
            else:
                assert np.array_equal(got[tt, h], row)


@pytest.mark.parametrize("t", [1, 2])
def test_attn_gathered_sharp_softmax(memq, oracle, t):
    """Scale 4: scores near 512 spread over tens of units, so the softmax concentrates on a few
    slots and the running max changes between chunks (t = 1 f32 kernel, t = 2 tensor cores)."""
    q_lat, _, cache, idx = synth.mla_attn_inputs(t, 2048, nh=8)
    run_attn(memq, oracle, q_lat, None, cache, idx, 4.0)


def test_head_gemv_hand_off_between_overlapping_launches(memq):
    """decompress_v's output [t, 64, 256] is absorb_q's input: launched back to back, absorb_q's
    weight stream overlaps the end of decompress_v (programmatic dependent launch) and its
    consumers must still read the finished x.  20 chains on fresh inputs, each bit-identical to
    the same two calls separated by a device synchronize."""
    t = 4
    _, wk = synth.mla_absorb_inputs(t)
    _, wv = synth.mla_decompress_inputs(t)
    dwk, dwv = to_dev(wk), to_dev(wv)
    o_all = [to_dev(synth.mla_randf(t * 64 * 512, 0x8200 + i).reshape(t, 64, 512)) for i in range(20)]
    mid = torch.empty((t, 64, 256), dtype=torch.float32, device="cuda")
    outs = []
    for o in o_all:  # back to back on one stream, one shared intermediate buffer
        memq.memq_mla_decompress_v(o, dwv, out=mid)
        outs.append(memq.memq_mla_absorb_q(mid, dwk))
    torch.cuda.synchronize()
    for o, got in zip(o_all, outs):
        m2 = memq.memq_mla_decompress_v(o, dwv)
        torch.cuda.synchronize()
        ref = memq.memq_mla_absorb_q(m2, dwk)
        torch.cuda.synchronize()
        assert_bits_equal(got, ref, "chained absorb_q")
    assert memq.memq_device_fault() == 0


def test_mla_kernels_in_a_cuda_graph(memq):
    """The three kernels captured in one CUDA graph and replayed give the eager outputs."""
    t = 2
    q, wk = synth.mla_absorb_inputs(t)
    o, wv = synth.mla_decompress_inputs(t)
    q_lat, _, cache, idx = synth.mla_attn_inputs(t, 4096)
    dq, dwk, do, dwv = to_dev(q), to_dev(wk), to_dev(o), to_dev(wv)
    dql, dc, di = to_dev(q_lat), to_dev(cache), to_dev(idx)
    outs = [torch.empty((t, 64, 512), dtype=torch.float32, device="cuda"),
            torch.empty((t, 64, 256), dtype=torch.float32, device="cuda"),
            torch.empty((t, 64, 512), dtype=torch.float32, device="cuda")]

    def run():
        memq.memq_mla_absorb_q(dq, dwk, out=outs[0])
        memq.memq_mla_decompress_v(do, dwv, out=outs[1])
        memq.memq_mla_attn_gathered(dql, None, dc, di, synth.MLA_SCALE, out=outs[2])

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        run()
        s.synchronize()
        eager = [x.clone() for x in outs]
        for x in outs:
            x.zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            run()
        g.replay()
        g.replay()
    s.synchronize()
    for a, b in zip(outs, eager):
        assert_bits_equal(a, b, "graph replay")


@pytest.mark.parametrize("which", ["absorb", "decompress"])
def test_head_gemv_stage_reuse_repeatable(memq, which):
    """A stage of the weight ring is released only after its weights have been used: released
    earlier, the next bulk copy could overwrite loads still in flight and change a few outputs
    from one launch to the next.  40 launches over several splits, each bit-identical to split 1."""
    t = 8
    x, w = synth.mla_absorb_inputs(t) if which == "absorb" else synth.mla_decompress_inputs(t)
    fn = memq.memq_mla_absorb_q if which == "absorb" else memq.memq_mla_decompress_v
    dx, dw = to_dev(x), to_dev(w)
    base = fn(dx, dw, split=1)
    outs = [fn(dx, dw, split=s) for s in (7, 3, 0, 5) * 10]
    torch.cuda.synchronize()
    for k, got in enumerate(outs):
        assert_bits_equal(got, base, f"launch {k}")


def test_mla_chain_hand_offs(memq):
    """absorb_q -> attn_gathered -> decompress_v back to back (each kernel's output is the next
    one's input, every launch overlapping its predecessor's end through programmatic dependent
    launch): 10 chains on fresh queries, each bit-identical to the same three calls separated by
    device synchronizes."""
    t = 2
    _, wk = synth.mla_absorb_inputs(t)
    _, wv = synth.mla_decompress_inputs(t)
    _, _, cache, idx = synth.mla_attn_inputs(t, 32768)
    dwk, dwv, dc, di = to_dev(wk), to_dev(wv), to_dev(cache), to_dev(idx)
    qs = [to_dev(synth.mla_randf(t * 64 * 256, 0x8300 + i).reshape(t, 64, 256)) for i in range(10)]
    q_lat = torch.empty((t, 64, 512), dtype=torch.float32, device="cuda")
    o_lat = torch.empty((t, 64, 512), dtype=torch.float32, device="cuda")
    outs = []
    for q in qs:
        memq.memq_mla_absorb_q(q, dwk, out=q_lat)
        memq.memq_mla_attn_gathered(q_lat, None, dc, di, synth.MLA_SCALE, out=o_lat)
        outs.append(memq.memq_mla_decompress_v(o_lat, dwv))
    torch.cuda.synchronize()
    for q, got in zip(qs, outs):
        a = memq.memq_mla_absorb_q(q, dwk)
        torch.cuda.synchronize()
        b = memq.memq_mla_attn_gathered(a, None, dc, di, synth.MLA_SCALE)
        torch.cuda.synchronize()
        ref = memq.memq_mla_decompress_v(b, dwv)
        torch.cuda.synchronize()
        assert_bits_equal(got, ref, "chained MLA step")
    assert memq.memq_device_fault() == 0
