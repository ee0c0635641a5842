"""Pins of the oracle's MLA decode attention (mla_decode_arm_gate.rs: absorb_q, decompress_v,
attn_gathered; geometry 64 heads, kv_rank 512, d_nope = d_v = 256, d_rope 0, 2048 gathered
slots).  Checked against library routines (numpy einsum, scipy softmax) on independently
computed operands, closed forms (identical rows, a single slot, shift invariance) and the
page generators' own properties."""
import numpy as np
import pytest

from quantized_decode_memq_gb300 import synth


def test_page_generators_match_their_definition():
    def seq(n, seed):
        s = (seed | 1) & ((1 << 64) - 1)
        out = []
        for _ in range(n):
            s = (s * 6364136223846793005 + 1442695040888963407) & ((1 << 64) - 1)
            out.append(s >> 33)
        return np.array(out, np.uint64)
    hi = seq(20000, 0xB2000005)
    f = synth.mla_randf(20000, 0xB2000005)
    expect = hi.astype(np.uint32).astype(np.float32) / np.float32(2147483648.0) - np.float32(1.0)
    assert np.array_equal(f, expect)
    assert f.min() >= -1.0 and f.max() < 0.0
    hi8 = seq(20000, 0xB2000008)
    assert np.array_equal(synth.mla_randidx(20000, 0xB2000008, 32768), (hi8 % 32768).astype(np.int32))


@pytest.mark.parametrize("t,nh,rows,cols", [(1, 3, 16, 32), (8, 4, 40, 96), (2, 64, 512, 256)])
def test_head_gemv_against_einsum(oracle, t, nh, rows, cols):
    x = synth.mla_randf(t * nh * cols, 0x100 + t).reshape(t, nh, cols) * np.float32(3)
    x[..., ::3] *= -1
    w = synth.mla_randf(nh * rows * cols, 0x200 + rows).reshape(nh, rows, cols)
    w[:, ::2] *= -1
    out, sabs = oracle.mla_head_gemv(x, w)
    ref = np.einsum("thk,hik->thi", x.astype(np.float64), w.astype(np.float64))
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(sabs, np.einsum("thk,hik->thi", np.abs(x).astype(np.float64),
                                               np.abs(w).astype(np.float64)), rtol=1e-13)
    # head h uses w[h] only: zero one head's weights
    w2 = w.copy()
    w2[1 % nh] = 0
    out2, _ = oracle.mla_head_gemv(x, w2)
    assert np.all(out2[:, 1 % nh] == 0)


def attn_ref(q_lat, cache, idx, scale):
    """softmax(scale * q . c_j) applied to the gathered rows, with a library softmax."""
    scipy_special = pytest.importorskip("scipy.special")
    c = cache[idx].astype(np.float64)                                  # [t, n_slots, kv_rank]
    s = scale * np.einsum("thr,tjr->thj", q_lat.astype(np.float64), c)
    p = scipy_special.softmax(s, axis=2)
    return np.einsum("thj,tjr->thr", p, c)


def test_attn_gathered_against_library_softmax(oracle):
    t, nh, kv_rank, kv, n_slots = 2, 5, 64, 300, 96
    q = synth.mla_randf(t * nh * kv_rank, 0x301).reshape(t, nh, kv_rank) * np.float32(4)
    q[..., 1::2] *= -1
    cache = synth.mla_randf(kv * kv_rank, 0x302).reshape(kv, kv_rank)
    cache[::3] *= -2
    idx = synth.mla_randidx(t * n_slots, 0x303, kv).reshape(t, n_slots)
    scale = 1.0 / 8.0
    out, cabs = oracle.mla_attn_gathered(q, None, cache, idx, scale)
    np.testing.assert_allclose(out, attn_ref(q, cache, idx, np.float32(scale)), rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(cabs, np.abs(cache[idx].astype(np.float64)).max(axis=1)[:, None, :].repeat(nh, 1))


def test_attn_closed_forms(oracle):
    kv_rank = 32
    cache = synth.mla_randf(10 * kv_rank, 0x304).reshape(10, kv_rank)
    q = synth.mla_randf(2 * kv_rank, 0x305).reshape(1, 2, kv_rank)
    # identical gathered rows: the output is that row, whatever the scores
    out, _ = oracle.mla_attn_gathered(q, None, cache, np.full((1, 7), 4, np.int32), 0.3)
    np.testing.assert_allclose(out[0], np.repeat(cache[4:5].astype(np.float64), 2, 0), rtol=1e-15)
    # a single slot: weight 1
    out, _ = oracle.mla_attn_gathered(q, None, cache, np.array([[6]], np.int32), 5.0)
    np.testing.assert_allclose(out[0, 0], cache[6].astype(np.float64), rtol=1e-15)
    # scale 0: the plain mean of the gathered rows
    idx = np.array([[0, 1, 2, 3]], np.int32)
    out, _ = oracle.mla_attn_gathered(q, None, cache, idx, 0.0)
    np.testing.assert_allclose(out[0, 1], cache[:4].astype(np.float64).mean(0), rtol=1e-14)
    # scores are scale * q . c
    _, _, sc = oracle.mla_attn_gathered(q, None, cache, idx, 0.25, scores=True)
    np.testing.assert_allclose(sc[0], 0.25 * q[0].astype(np.float64) @ cache[:4].astype(np.float64).T,
                               rtol=1e-14)


def test_attn_rope_term(oracle):
    """With d_rope > 0 the score adds q_pe . c[kv_rank:]: equal to a NoPE problem whose query and
    rows are the concatenations."""
    t, nh, kv_rank, d_rope, kv = 1, 2, 16, 8, 12
    q = synth.mla_randf(t * nh * kv_rank, 0x306).reshape(t, nh, kv_rank)
    qp = synth.mla_randf(t * nh * d_rope, 0x307).reshape(t, nh, d_rope)
    cache = synth.mla_randf(kv * (kv_rank + d_rope), 0x308).reshape(kv, kv_rank + d_rope)
    idx = synth.mla_randidx(t * 9, 0x309, kv).reshape(t, 9)
    out, _ = oracle.mla_attn_gathered(q, qp, cache, idx, 0.5, d_rope=d_rope)
    full, _ = oracle.mla_attn_gathered(np.concatenate([q, qp], 2), None, cache, idx, 0.5)
    np.testing.assert_allclose(out, full[..., :kv_rank], rtol=1e-14)
