// mx_decode.cuh -- in-register decode of the library's repacked MXFP4 words
// into BF16 pairs, used by the GEMM kernels.
//
// A decoded weight is v(c) * 2^(e-127) ("DeepSeek-V4-Flash on a four-GPU
// Ampere workstation", section "MXFP4 is not NVFP4, and the difference matters
// on Ampere"): 4-bit E2M1 code c, E8M0 exponent e shared by 32 consecutive
// values.  The product is exact in BF16 (v has at most 2 significant bits, the
// power of two only moves the exponent) for every e in [0, 254] unless it
// overflows, so decoding to BF16 adds no error.
//
// Repacked word (32 bits, 8 consecutive elements e_0..e_7 of a row):
//   nibble i, bits 0..2  : the magnitude index of e_i (position in the list
//                          0, 0.5, 1, 1.5, 2, 3, 4, 6)
//   nibble 2j+1, bit 3   : sign of e_j      (j = 0..3)  -> word bit 8j+7
//   nibble 2j,   bit 3   : sign of e_{4+j}  (j = 0..3)  -> word bit 8j+3
// so that byte j of a PRMT table lookup on nibbles 0..3 (resp. 4..7) takes its
// sign with a single mask (resp. shift + mask).  The repack kernel writes
// exactly this layout (see repack_kernel in layout.cu).
#pragma once

#include <stdint.h>

namespace moe {

// BF16 bytes of the 8 magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6 (0x0000, 0x3F00,
// 0x3F80, 0x3FC0, 0x4000, 0x4040, 0x4080, 0x40C0), split into high and low
// bytes and packed as two 4-byte tables each for PRMT.
constexpr uint32_t MAG_HI_0 = 0x3F3F3F00u;  // magnitudes 0..3, high bytes
constexpr uint32_t MAG_HI_1 = 0x40404040u;  // magnitudes 4..7, high bytes
constexpr uint32_t MAG_LO_0 = 0xC0800000u;  // magnitudes 0..3, low bytes
constexpr uint32_t MAG_LO_1 = 0xC0804000u;  // magnitudes 4..7, low bytes

__host__ __device__ constexpr uint32_t repacked_sign_bit(int i)
{
    // word bit holding the sign of element i of the word
    return i < 4 ? 8 * i + 7 : 8 * (i - 4) + 3;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// BF16 pair {2^(e-127), 2^(e-127)}; e = 0 gives the BF16 subnormal 2^-127.
__device__ __forceinline__ uint32_t e8m0_to_bf16x2(uint32_t e)
{
    uint32_t b = e ? (e << 7) : 0x0040u;
    return b | (b << 16);
}

// Decode one repacked word (8 elements) into 4 BF16 pairs out[0..3]
// ((e0,e1), (e2,e3), (e4,e5), (e6,e7), lower element in the low half), each
// multiplied by the block scale pair s2.
__device__ __forceinline__ void decode_word(uint32_t w, uint32_t s2, uint32_t out[4])
{
    const uint32_t m = w & 0x77777777u;
    const uint32_t mh = m >> 16;
    uint32_t h0 = prmt(MAG_HI_0, MAG_HI_1, m);
    uint32_t l0 = prmt(MAG_LO_0, MAG_LO_1, m);
    uint32_t h1 = prmt(MAG_HI_0, MAG_HI_1, mh);
    uint32_t l1 = prmt(MAG_LO_0, MAG_LO_1, mh);
    h0 |= w & 0x80808080u;
    h1 |= (w << 4) & 0x80808080u;
    out[0] = bf16x2_mul(prmt(l0, h0, 0x5140u), s2);
    out[1] = bf16x2_mul(prmt(l0, h0, 0x7362u), s2);
    out[2] = bf16x2_mul(prmt(l1, h1, 0x5140u), s2);
    out[3] = bf16x2_mul(prmt(l1, h1, 0x7362u), s2);
}

// The same for a warp-level MMA A fragment word (FRAG layout): pairs 0 and 2
// belong to row g and take scale sa, pairs 1 and 3 to row g+8 and take sb.
__device__ __forceinline__ void decode_word_frag(uint32_t w, uint32_t sa, uint32_t sb, uint32_t out[4])
{
    const uint32_t m = w & 0x77777777u;
    const uint32_t mh = m >> 16;
    uint32_t h0 = prmt(MAG_HI_0, MAG_HI_1, m);
    uint32_t l0 = prmt(MAG_LO_0, MAG_LO_1, m);
    uint32_t h1 = prmt(MAG_HI_0, MAG_HI_1, mh);
    uint32_t l1 = prmt(MAG_LO_0, MAG_LO_1, mh);
    h0 |= w & 0x80808080u;
    h1 |= (w << 4) & 0x80808080u;
    out[0] = bf16x2_mul(prmt(l0, h0, 0x5140u), sa);
    out[1] = bf16x2_mul(prmt(l0, h0, 0x7362u), sb);
    out[2] = bf16x2_mul(prmt(l1, h1, 0x5140u), sa);
    out[3] = bf16x2_mul(prmt(l1, h1, 0x7362u), sb);
}

}  // namespace moe
