"""Properties of the seeded input generators (CPU only)."""
import numpy as np

from quantized_decode_memq_gb300 import synth


def _lcg_ref(seed, n):
    s, out = seed, []
    for _ in range(n):
        s = (s * 1664525 + 1013904223) & 0xFFFFFFFF
        out.append(s)
    return out


def test_lcg_jump_ahead_matches_sequential():
    n = (1 << 16) * 2 + 123  # crosses two jump-ahead blocks
    fast = synth._lcg_states(0x12345678, n)
    ref = _lcg_ref(0x12345678, n)
    assert fast.tolist() == ref


def test_page_e4m3_never_nan_and_sign_balanced():
    w = synth.lcg_e4m3(64, 4096)
    assert not np.any((w & 0x7F) == 0x7F)
    assert 0.45 < (w >> 7).mean() < 0.55


def test_page_q8_0_layout():
    w = synth.lcg_q8_0(8, 256)
    blk = w.reshape(-1, 34)
    assert np.all(blk[:, 0] == 0x00) and np.all(blk[:, 1] == 0x14)


def test_xorshift_range_and_no_zero_for_page_seeds():
    for ncols in (1536, 4096, 5120, 8192, 17408):
        x, w = synth.activation_rows(ncols, 1)
        for v in (x, w):
            assert v.dtype == np.float32
            assert v.min() >= -4.0 and v.max() < 4.0
            assert np.all(v != 0)  # keeps amax > 0 on every 32-block


def test_splitmix_counter_based():
    a = synth.splitmix64(99, 1000)
    b = synth.splitmix64(99, 500, start=500)
    assert np.array_equal(a[500:], b)
    # first output of splitmix64 seeded with 0 (Vigna's splitmix64.c reference output)
    assert int(synth.splitmix64(0, 1)[0]) == 0xE220A8397B1DCDAF


def test_workload_distributions():
    w = synth.e4m3_bytes(3, 100, 512)
    assert not np.any((w & 0x7F) == 0x7F)
    g = synth.grid_log2_uniform(4, 17408, 5120)
    assert g.shape == (136, 40)
    assert g.min() >= 2.0 ** -6 and g.max() <= 2.0 ** -2
    q = synth.q8_0_bytes(5, 64, 512).reshape(-1, 34)
    qs = q[:, 2:].view(np.int8)
    assert qs.min() == -127 and qs.max() == 127
    dw = np.ascontiguousarray(q[:, 0:2]).view(np.float16).astype(np.float64)
    assert dw.min() >= 2.0 ** -10 and dw.max() <= 2.0 ** -6
