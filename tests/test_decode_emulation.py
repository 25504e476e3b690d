"""CPU emulation of the GPU's in-register MXFP4 -> BF16 decode, and of the
single kernel's group-32 INT4 -> FP16 decode.

The CUDA kernels decode repacked 32-bit words with byte permutes (PRMT) and a
BF16 multiply (mx_decode.cuh).  This test emulates those exact bit operations
in Python for every code and sign pattern and compares the result with the
E2M1 table printed on the page (tests/golden/e2m1_table.txt) times 2^(e-127).
The repack bit layout it emulates is the one documented in mx_decode.cuh.
"""
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e2m1_table.txt")

MAG_HI_0, MAG_HI_1 = 0x3F3F3F00, 0x40404040
MAG_LO_0, MAG_LO_1 = 0xC0800000, 0xC0804000


def table():
    t = {}
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if line:
            c, v = line.split()
            t[int(c)] = float(v)
    return t


def prmt(a, b, sel):
    src = [(a >> (8 * i)) & 0xFF for i in range(4)] + [(b >> (8 * i)) & 0xFF for i in range(4)]
    d = 0
    for i in range(4):
        n = (sel >> (4 * i)) & 0xF
        byte = src[n & 7]
        if n & 8:
            byte = 0xFF if byte & 0x80 else 0x00
        d |= byte << (8 * i)
    return d


def sign_bit(i):
    return 8 * i + 7 if i < 4 else 8 * (i - 4) + 3


def repack_word(codes8):
    w = 0
    for i, c in enumerate(codes8):
        w |= (c & 7) << (4 * i)
        w |= (c >> 3) << sign_bit(i)
    return w


def bf16_bits_value(b):
    return struct.unpack("<f", struct.pack("<I", (b & 0xFFFF) << 16))[0]


def to_bf16_exact(x):
    """x must be exactly representable in BF16 (possibly subnormal)."""
    f = np.float32(x)
    assert float(f) == x or (x != 0 and math.isinf(float(f)))
    b = int(f.view(np.uint32))
    assert b & 0xFFFF == 0, x
    return b >> 16


def bf16x2_mul(a, b):
    out = 0
    for half in range(2):
        x = bf16_bits_value(a >> (16 * half))
        y = bf16_bits_value(b >> (16 * half))
        p = x * y
        out |= to_bf16_exact(p) << (16 * half)
    return out


def e8m0_to_bf16x2(e):
    b = (e << 7) if e else 0x0040
    return b | (b << 16)


def decode_word(w, s2):
    m = w & 0x77777777
    mh = m >> 16
    h0 = prmt(MAG_HI_0, MAG_HI_1, m)
    l0 = prmt(MAG_LO_0, MAG_LO_1, m)
    h1 = prmt(MAG_HI_0, MAG_HI_1, mh)
    l1 = prmt(MAG_LO_0, MAG_LO_1, mh)
    h0 |= w & 0x80808080
    h1 |= ((w << 4) & 0xFFFFFFFF) & 0x80808080
    return [bf16x2_mul(prmt(l0, h0, 0x5140), s2), bf16x2_mul(prmt(l0, h0, 0x7362), s2),
            bf16x2_mul(prmt(l1, h1, 0x5140), s2), bf16x2_mul(prmt(l1, h1, 0x7362), s2)]


def unpack(outs):
    vals = []
    for r in outs:
        vals.append(bf16_bits_value(r))
        vals.append(bf16_bits_value(r >> 16))
    return vals


def expect(code, e, tab):
    v = Fraction(tab[code]) * Fraction(2) ** (e - 127)
    return math.copysign(float(v), tab[code]) if v == 0 else float(v)


@pytest.mark.parametrize("e", [0, 1, 2, 64, 120, 126, 127, 128, 130, 200, 252])
def test_every_code_in_every_position(e):
    tab = table()
    s2 = e8m0_to_bf16x2(e)
    rng = np.random.default_rng(e)
    words = [list(range(i, i + 8)) for i in (0, 8)]          # all 16 codes, each position
    words += [[(c + s) % 16 for c in range(8)] for s in range(16)]
    words += [rng.integers(0, 16, 8).tolist() for _ in range(50)]
    for codes in words:
        got = unpack(decode_word(repack_word(codes), s2))
        for i, c in enumerate(codes):
            want = expect(c, e, tab)
            assert got[i] == want and math.copysign(1, got[i]) == math.copysign(1, want), (e, codes, i)


def decode_word_frag(w, sa, sb):
    m = w & 0x77777777
    mh = m >> 16
    h0 = prmt(MAG_HI_0, MAG_HI_1, m)
    l0 = prmt(MAG_LO_0, MAG_LO_1, m)
    h1 = prmt(MAG_HI_0, MAG_HI_1, mh)
    l1 = prmt(MAG_LO_0, MAG_LO_1, mh)
    h0 |= w & 0x80808080
    h1 |= ((w << 4) & 0xFFFFFFFF) & 0x80808080
    return [bf16x2_mul(prmt(l0, h0, 0x5140), sa), bf16x2_mul(prmt(l0, h0, 0x7362), sb),
            bf16x2_mul(prmt(l1, h1, 0x5140), sa), bf16x2_mul(prmt(l1, h1, 0x7362), sb)]


def test_fragment_word_maps_to_mma_a_registers():
    """A FRAG-layout word holds, for lane (g, q) and K step j, the elements
    (g, 2q), (g, 2q+1), (g+8, 2q), (g+8, 2q+1), (g, 2q+8), (g, 2q+9), (g+8, 2q+8),
    (g+8, 2q+9) of the 16x16 A tile; the decode must yield the m16n8k16 A
    registers a0 = rows g / k 2q..2q+1, a1 = rows g+8, a2 = rows g / k+8, a3 =
    rows g+8 / k+8, each row with its own block scale."""
    tab = table()
    rng = np.random.default_rng(7)
    for trial in range(200):
        tile = rng.integers(0, 16, (16, 16))
        ea, eb = int(rng.integers(100, 150)), int(rng.integers(100, 150))
        g, q = int(rng.integers(0, 8)), int(rng.integers(0, 4))
        codes = [tile[g, 2 * q], tile[g, 2 * q + 1], tile[g + 8, 2 * q], tile[g + 8, 2 * q + 1],
                 tile[g, 2 * q + 8], tile[g, 2 * q + 9], tile[g + 8, 2 * q + 8], tile[g + 8, 2 * q + 9]]
        regs = decode_word_frag(repack_word([int(c) for c in codes]), e8m0_to_bf16x2(ea), e8m0_to_bf16x2(eb))
        want = [(g, 2 * q, ea), (g + 8, 2 * q, eb), (g, 2 * q + 8, ea), (g + 8, 2 * q + 8, eb)]
        for reg, (row, col, e) in zip(regs, want):
            lo, hi = bf16_bits_value(reg), bf16_bits_value(reg >> 16)
            assert lo == expect(int(tile[row, col]), e, tab)
            assert hi == expect(int(tile[row, col + 1]), e, tab)


# ------------------------------------------------------------------ group-32 INT4 (single kernel)
# The FRAG_F16 INT4 word holds the A fragment's element pair p in nibbles p
# (first element) and p + 4 (second); the kernel turns a pair into FP16 q - z
# with a shift, a mask, an OR with 0x6400 (FP16 1024) in both halves and one
# FP16x2 subtraction of 1024 + z.  Emulated here with numpy's float16, which
# rounds like the hardware's round-to-nearest subtraction.

def i4_repack_word(first, second):
    w = 0
    for p in range(4):
        w |= first[p] << (4 * p) | second[p] << (4 * p + 16)
    return w


def decode_i4_pair(w, p, z):
    v = ((w >> (4 * p)) & 0x000F000F) | 0x64006400
    halves = np.array([v & 0xFFFF, v >> 16], np.uint16).view(np.float16)
    m = np.array([0x6400 + z, 0x6400 + z], np.uint16).view(np.float16)
    return (halves - m).astype(np.float64)


def test_i4_pair_decode_is_exact_for_every_code_and_zero_point():
    for z in range(16):
        for q0 in range(16):
            for q1 in range(16):
                w = i4_repack_word([q0, 0, 0, 0], [q1, 0, 0, 0])
                got = decode_i4_pair(w, 0, z)
                assert got[0] == q0 - z and got[1] == q1 - z, (q0, q1, z)


def test_i4_fragment_word_maps_pairs_to_registers():
    rng = np.random.default_rng(3)
    for _ in range(200):
        first = rng.integers(0, 16, 4).tolist()
        second = rng.integers(0, 16, 4).tolist()
        za, zb = int(rng.integers(0, 16)), int(rng.integers(0, 16))
        w = i4_repack_word(first, second)
        for p in range(4):
            z = zb if p & 1 else za       # pairs 1 and 3 belong to row g + 8
            got = decode_i4_pair(w, p, z)
            assert got[0] == first[p] - z and got[1] == second[p] - z


# ------------------------------------------------------------------ group-32 INT4 (tensor-core GEMMs)
# The TILE_I4 decoder turns s (q - z) into two FP16 values: s' = s * 2^-b_row in
# FP16 (b_row = floor(log2 max|s|) - 11 over the row, so s' < 2^12), qz = q - z
# as above, hi = fp16(qz * s') and lo = fp16(qz * s' - hi) from a fused
# multiply-add, which rounds once from the exact value.  Emulated with numpy:
# the exact product and residual in float64, each rounded once to float16.

def i4_hilo(qz, s_prime):
    prod = float(qz) * float(s_prime)             # exact: 4 x 11 significant bits
    hi = np.float16(prod)
    lo = np.float16(prod - float(hi))             # one rounding of the exact residual
    return hi, lo, prod


def test_i4_hi_lo_split_is_exact_for_normal_scales():
    rng = np.random.default_rng(5)
    # FP16 scales s' across the normal range below 2^12, including the extremes
    sp = [np.float16(2.0 ** -14), np.float16(4095.0), np.float16(1.0), np.float16(0.3)]
    sp += [np.float16(v) for v in np.exp2(rng.uniform(-14, 12, 400)) * rng.choice([-1, 1], 400)]
    for s in sp:
        assert np.isfinite(s) and abs(float(s)) >= 2.0 ** -14
        for qz in range(-15, 16):
            hi, lo, prod = i4_hilo(qz, s)
            assert float(hi) + float(lo) == prod, (qz, float(s))
            assert abs(float(hi)) <= 15 * 4096


def test_i4_row_base_keeps_scales_exact_and_weights_finite():
    rng = np.random.default_rng(6)
    for _ in range(300):
        top = int(rng.integers(-24, 16))           # exponent of the row's largest FP16 scale
        s_max = np.float16(np.exp2(top) * rng.uniform(1.0, 1.999))
        if not np.isfinite(s_max) or s_max == 0:
            continue
        b = int(np.floor(np.log2(float(s_max)))) - 11
        for d in range(0, 25):                      # groups up to 2^-24 below the row's largest
            s = np.float16(float(s_max) * 2.0 ** -d * rng.uniform(0.5, 1.0))
            if s == 0:
                continue
            sp = np.float16(float(s) * 2.0 ** -b)   # exact unless it falls below the FP16 normal range
            if abs(float(sp)) >= 2.0 ** -14:
                assert float(sp) == float(s) * 2.0 ** -b
            assert abs(float(sp)) < 4096.0
            hi, lo, prod = i4_hilo(15, sp)
            assert np.isfinite(hi) and abs(float(hi)) <= 15 * 4096
