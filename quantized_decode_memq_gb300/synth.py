"""Seeded synthetic inputs for the quantized decode chain.

This module is the one piece shared by the CUDA path's tests/bench and by the oracle's tests: it
draws random bytes and floats and lays them out in the three weight containers.  It holds none
of the chain's arithmetic (no normalisation, no quantisation, no dot products, no decoding).

Generators taken from the memra-engine 0.125.0 source pages, kept bit-exact:

* ``xorshift64_f32`` -- q8_fuse_gate.rs, ``Xorshift64`` (shifts 13, 7, 17; state seeded with
  ``seed | 1``; ``next_f32`` maps the top 24 bits to ``(u/2^24 - 0.5) * 8``, i.e. [-4, 4)) and the
  per-width seeds of ``run_shape``.
* ``lcg_e4m3`` -- gemv_e4m3_bench.rs, ``synth_e4m3`` (LCG 1664525/1013904223 from 0x12345678;
  magnitude ``(s>>16)&0x7F`` with the NaN magnitude 0x7F replaced by 0x30, sign ``(s>>8)&1``).
* ``lcg_blk_grid`` -- gemv_e4m3_bench.rs, ``synth_blk_grid`` (2^(-6 + (s>>20) % 5)).
* ``lcg_q8_0`` -- gemv_e4m3_bench.rs, ``synth_q8_0`` (fixed f16 scale 0x1400, qs = s>>24).

* ``mla_randf`` / ``mla_randidx`` -- mla_decode_arm_gate.rs, ``randf`` / ``randidx`` (64-bit LCG with
  Knuth's MMIX constants from ``seed | 1``; ``randf`` maps ``(s >> 33) as u32 as f32`` by dividing by
  ``u32::MAX as f32 / 2`` and subtracting 1 in f32 -- (s >> 33) has 31 bits, so the values lie in
  [-1, 0); ``randidx`` is ``(s >> 33) % max``).

For sizes where a sequential generator is too slow in Python, and for the distributions the
workload descriptions give without naming a generator, a counter-based SplitMix64
(Steele, Lea & Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014; the
constants of Vigna's splitmix64.c) gives value i = mix64(seed + (i+1) * 0x9E3779B97F4A7C15).
"""
from __future__ import annotations

import numpy as np

MASK64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15

# Per-width seeds of q8_fuse_gate.rs `run_shape`.
SEED_X = 0x9E3779B97F4A7C15
SEED_W = 0xD1B54A32D192ED03


# ------------------------------------------------------------------------------------------
# Page generators (bit-exact)
# ------------------------------------------------------------------------------------------

def xorshift64_f32(seed: int, n: int) -> np.ndarray:
    """n draws of q8_fuse_gate.rs `Xorshift64::next_f32` from `Xorshift64::new(seed)`."""
    s = (seed | 1) & MASK64
    out = np.empty(n, np.float32)
    for k in range(n):
        s ^= (s << 13) & MASK64
        s ^= s >> 7
        s ^= (s << 17) & MASK64
        out[k] = np.float32(s >> 40)
    # (bits as f32) / 2^24 - 0.5, times 8: every step is exact in f32 for 24-bit integers.
    out /= np.float32(1 << 24)
    out -= np.float32(0.5)
    out *= np.float32(8.0)
    return out


def _lcg_states(seed: int, n: int) -> np.ndarray:
    """States s_1..s_n of s <- s*1664525 + 1013904223 (mod 2^32), vectorised by jump-ahead."""
    a, c = 1664525, 1013904223
    blk = min(n, 1 << 16)
    first = np.empty(blk, np.uint64)
    s = seed & 0xFFFFFFFF
    for k in range(blk):
        s = (s * a + c) & 0xFFFFFFFF
        first[k] = s
    if blk == n:
        return first.astype(np.uint32)
    # Affine map of `blk` steps: s -> A*s + C (mod 2^32).
    A, C = 1, 0
    for _ in range(blk):
        A, C = (A * a) & 0xFFFFFFFF, (C * a + c) & 0xFFFFFFFF
    out = np.empty(n, np.uint32)
    cur = first
    pos = 0
    A64, C64 = np.uint64(A), np.uint64(C)
    m32 = np.uint64(0xFFFFFFFF)
    while pos < n:
        take = min(blk, n - pos)
        out[pos:pos + take] = cur[:take].astype(np.uint32)
        pos += take
        cur = (cur * A64 + C64) & m32
    return out


def lcg_e4m3(out_f: int, in_f: int, seed: int = 0x12345678) -> np.ndarray:
    """gemv_e4m3_bench.rs `synth_e4m3`: uint8 [out_f, in_f], never a NaN code."""
    s = _lcg_states(seed, out_f * in_f)
    mag = ((s >> 16) & 0x7F).astype(np.uint8)
    mag[mag == 0x7F] = 0x30
    sign = (((s >> 8) & 1) << 7).astype(np.uint8)
    return (mag | sign).reshape(out_f, in_f)


def lcg_blk_grid(out_f: int, in_f: int, seed: int = 0x5BF03635) -> np.ndarray:
    """gemv_e4m3_bench.rs `synth_blk_grid`: f32 [ceil(out_f/128), ceil(in_f/128)]."""
    rows, cols = -(-out_f // 128), -(-in_f // 128)
    s = _lcg_states(seed, rows * cols)
    e = -6 + ((s >> 20) % 5).astype(np.int64)
    return np.ldexp(np.ones(rows * cols, np.float32), e).astype(np.float32).reshape(rows, cols)


def lcg_q8_0(out_f: int, in_f: int, seed: int = 0x9E3779B9) -> np.ndarray:
    """gemv_e4m3_bench.rs `synth_q8_0`: uint8 [out_f, in_f/32*34]; f16 scale bytes 00 14
    (2^-10), then 32 bytes (s>>24) -- so qs spans the full int8 range including -128."""
    nb = in_f // 32
    s = _lcg_states(seed, out_f * nb * 32)
    blocks = np.empty((out_f * nb, 34), np.uint8)
    blocks[:, 0] = 0x00
    blocks[:, 1] = 0x14
    blocks[:, 2:] = (s >> 24).astype(np.uint8).reshape(out_f * nb, 32)
    return blocks.reshape(out_f, nb * 34)


# ------------------------------------------------------------------------------------------
# Counter-based generator and the workload distributions
# ------------------------------------------------------------------------------------------

def splitmix64(seed: int, n: int, start: int = 0) -> np.ndarray:
    """u64 values mix64(seed + (start+i+1)*GOLDEN), i < n."""
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & MASK64) + i * np.uint64(GOLDEN)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        z = z ^ (z >> np.uint64(31))
    return z


def uniform_pm4(seed: int, n: int, start: int = 0) -> np.ndarray:
    """f32 uniform on [-4, 4) with the `next_f32` mapping, fed by splitmix64 bits."""
    bits = (splitmix64(seed, n, start) >> np.uint64(40)).astype(np.float32)
    return ((bits / np.float32(1 << 24)) - np.float32(0.5)) * np.float32(8.0)


def e4m3_bytes(seed: int, out_f: int, in_f: int) -> np.ndarray:
    """Uniform random E4M3 bytes with both NaN codes (0x7F, 0xFF) replaced by 0x30|sign."""
    b = (splitmix64(seed, out_f * in_f) >> np.uint64(56)).astype(np.uint8)
    nan = (b & 0x7F) == 0x7F
    b[nan] = (b[nan] & 0x80) | 0x30
    return b.reshape(out_f, in_f)


def grid_log2_uniform(seed: int, out_f: int, in_f: int, lo: float = -6.0,
                      hi: float = -2.0) -> np.ndarray:
    """f32 block-128 grid with log2 uniform on [lo, hi): f32(2^(lo + (hi-lo)*u))."""
    rows, cols = -(-out_f // 128), -(-in_f // 128)
    u = (splitmix64(seed, rows * cols) >> np.uint64(11)).astype(np.float64) / float(1 << 53)
    return np.exp2(lo + (hi - lo) * u).astype(np.float32).reshape(rows, cols)


def q8_0_bytes(seed: int, out_f: int, in_f: int, qlo: int = -127, qhi: int = 127,
               dlo: float = 2.0 ** -10, dhi: float = 2.0 ** -6) -> np.ndarray:
    """block_q8_0 rows: qs uniform integers in [qlo, qhi], scale f16(uniform [dlo, dhi))."""
    nb = in_f // 32
    nblk = out_f * nb
    r = splitmix64(seed, nblk * 33)
    span = np.uint64(qhi - qlo + 1)
    q = ((r[:nblk * 32] >> np.uint64(32)) * span >> np.uint64(32)).astype(np.int64) + qlo
    u = (r[nblk * 32:] >> np.uint64(11)).astype(np.float64) / float(1 << 53)
    dval = (dlo + (dhi - dlo) * u).astype(np.float16)
    blocks = np.empty((nblk, 34), np.uint8)
    blocks[:, 0:2] = dval.view(np.uint8).reshape(nblk, 2)
    blocks[:, 2:] = q.astype(np.int8).view(np.uint8).reshape(nblk, 32)
    return blocks.reshape(out_f, nb * 34)


def activation_rows(ncols: int, rows: int, page_streams: bool = True, seed_x: int = SEED_X,
                    seed_w: int = SEED_W):
    """(x [rows, ncols] f32, w [ncols] f32) uniform on [-4, 4).

    With ``page_streams`` the q8_fuse_gate.rs generators and seeds are used (x continues one
    xorshift stream across rows); otherwise splitmix64 with the same seeds (large sweeps).
    """
    if page_streams:
        x = xorshift64_f32(seed_x ^ ncols, rows * ncols).reshape(rows, ncols)
        w = xorshift64_f32(seed_w ^ ncols, ncols)
    else:
        x = uniform_pm4(seed_x ^ ncols, rows * ncols).reshape(rows, ncols)
        w = uniform_pm4(seed_w ^ ncols, ncols)
    return x, w


# ------------------------------------------------------------------------------------------
# mla_decode_arm_gate.rs generators (64-bit LCG, MMIX constants), bit-exact, vectorised by
# jump-ahead like _lcg_states.
# ------------------------------------------------------------------------------------------
_MMIX_A = 6364136223846793005
_MMIX_C = 1442695040888963407


def _mmix_states(seed: int, n: int) -> np.ndarray:
    """States s_1..s_n of s <- s*A + C (mod 2^64) from s_0 = seed | 1."""
    blk = min(n, 1 << 14)
    first = np.empty(blk, np.uint64)
    s = (seed | 1) & MASK64
    for k in range(blk):
        s = (s * _MMIX_A + _MMIX_C) & MASK64
        first[k] = s
    if blk == n:
        return first
    A, C = 1, 0
    for _ in range(blk):
        A, C = (A * _MMIX_A) & MASK64, (C * _MMIX_A + _MMIX_C) & MASK64
    out = np.empty(n, np.uint64)
    cur = first
    pos = 0
    with np.errstate(over="ignore"):
        while pos < n:
            take = min(blk, n - pos)
            out[pos:pos + take] = cur[:take]
            pos += take
            cur = cur * np.uint64(A) + np.uint64(C)
    return out


def mla_randf(n: int, seed: int) -> np.ndarray:
    """mla_decode_arm_gate.rs ``randf(n, seed)``: f32 in [-1, 0)."""
    hi = (_mmix_states(seed, n) >> np.uint64(33)).astype(np.uint32)
    return hi.astype(np.float32) / np.float32(np.float32(4294967295.0) / np.float32(2.0)) - np.float32(1.0)


def mla_randidx(n: int, seed: int, max_excl: int) -> np.ndarray:
    """mla_decode_arm_gate.rs ``randidx(n, seed, max_excl)``: int32 in [0, max_excl)."""
    hi = (_mmix_states(seed, n) >> np.uint64(33)).astype(np.uint32)
    return (hi % np.uint32(max_excl)).astype(np.int32)


# ---------------------------------------------------------------------------------------------
# MLA decode attention inputs, as mla_decode_arm_gate.rs (`main`) draws them: every array from
# randf with the page's per-array seed xor'd with t (and with the pool depth kv for the cache
# and the gather indices); n_slots = min(2048, kv).
# ---------------------------------------------------------------------------------------------
MLA_NH, MLA_KV_RANK, MLA_D_NOPE, MLA_D_V, MLA_N_SLOTS = 64, 512, 256, 256, 2048
MLA_SCALE = float(np.float32(1.0) / np.float32(23.323808))


def mla_absorb_inputs(t: int, nh: int = MLA_NH, kv_rank: int = MLA_KV_RANK,
                      d_nope: int = MLA_D_NOPE):
    """(q_nope f32 [t, nh, d_nope], wk_b f32 [nh, kv_rank, d_nope])."""
    q = mla_randf(t * nh * d_nope, 0xB2000001 ^ t).reshape(t, nh, d_nope)
    w = mla_randf(nh * kv_rank * d_nope, 0xB2000002 ^ t).reshape(nh, kv_rank, d_nope)
    return q, w


def mla_decompress_inputs(t: int, nh: int = MLA_NH, kv_rank: int = MLA_KV_RANK,
                          d_v: int = MLA_D_V):
    """(o_lat f32 [t, nh, kv_rank], wv_b f32 [nh, d_v, kv_rank])."""
    o = mla_randf(t * nh * kv_rank, 0xB2000003 ^ t).reshape(t, nh, kv_rank)
    w = mla_randf(nh * d_v * kv_rank, 0xB2000004 ^ t).reshape(nh, d_v, kv_rank)
    return o, w


def mla_attn_inputs(t: int, kv: int, nh: int = MLA_NH, kv_rank: int = MLA_KV_RANK,
                    d_rope: int = 0, n_slots: int | None = None):
    """(q_lat [t, nh, kv_rank], q_pe [t, nh, d_rope] or None, cache [kv, kv_rank + d_rope],
    idx int32 [t, n_slots]); n_slots defaults to min(2048, kv)."""
    if n_slots is None:
        n_slots = min(MLA_N_SLOTS, kv)
    q_lat = mla_randf(t * nh * kv_rank, 0xB2000005 ^ t).reshape(t, nh, kv_rank)
    q_pe = (mla_randf(t * nh * d_rope, 0xB2000006 ^ t).reshape(t, nh, d_rope)
            if d_rope else None)
    cache = mla_randf(kv * (kv_rank + d_rope), 0xB2000007 ^ kv).reshape(kv, kv_rank + d_rope)
    idx = mla_randidx(t * n_slots, 0xB2000008 ^ t ^ kv, kv).reshape(t, n_slots)
    return q_lat, q_pe, cache, idx
