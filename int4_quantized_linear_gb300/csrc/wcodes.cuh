// wcodes.cuh -- integer weight codes to the e4m3 operand bytes the tensor-core kernels read.
// Every function turns the packed codes of one checkpoint word into bytes whose e4m3 values are
// exact multiples of 2^-9, so the fp8 MMA computes the integer dot product exactly (up to its
// fp32 accumulation).  Checked on every code in every position against the e4m3 decode.
#pragma once
#include <stdint.h>

namespace w4a8 {
namespace tci {

// Eight int4 codes of one word (k = 8i..8i+7, low nibble first) -> the eight codes as bytes,
// low byte first, in two words: each byte read as e4m3 is c * 2^-9.
__device__ __forceinline__ uint2 i4x8_to_bytes(uint32_t w)
{
    const uint32_t ev = w & 0x0F0F0F0Fu;          // codes 0, 2, 4, 6
    const uint32_t od = (w >> 4) & 0x0F0F0F0Fu;   // codes 1, 3, 5, 7
    return make_uint2(__byte_perm(ev, od, 0x5140), __byte_perm(ev, od, 0x7362));
}

constexpr uint32_t E4M3_MINUS_2POW_M6 = 0x88u;  // sign 1, exponent field 1, mantissa 0: -2^-6

// Bits 0, 2, 4 and 6 of b (the others clear) -> 0xFF or 0x00 in bytes 0..3.  The multiply by
// 1 + 2^6 + 2^12 + 2^18 puts bit 2j at bit 8j; the other copies land on even positions that are
// not multiples of 8 (where two coincide the carry stops one bit higher, still off 8j), and the
// mask keeps bits 8j only.
__device__ __forceinline__ uint32_t spread_even_bits(uint32_t b)
{
    return ((b * 0x00041041u) & 0x01010101u) * 0xFFu;
}

// Eight int5 codes: the nibbles of word w and the fifth bits of plane byte hb (bit j for code j)
// -> the e4m3 bytes of (c - 16) * 2^-9, low byte first: the nibble where the fifth bit is set,
// 0x90 - nibble where it is clear (no byte borrows: 0x90 > 15).
__device__ __forceinline__ uint2 i5x8_to_signed_bytes(uint32_t w, uint32_t hb)
{
    const uint32_t ev = w & 0x0F0F0F0Fu, od = (w >> 4) & 0x0F0F0F0Fu;
    const uint32_t he = spread_even_bits(hb & 0x55u), ho = spread_even_bits((hb >> 1) & 0x55u);
    const uint32_t e = (ev & he) | ((0x90909090u - ev) & ~he);
    const uint32_t o = (od & ho) | ((0x90909090u - od) & ~ho);
    return make_uint2(__byte_perm(e, o, 0x5140), __byte_perm(e, o, 0x7362));
}

// Byte permute with the PTX sign-replicate mode: byte j of the result is byte (s_j & 7) of the
// eight bytes {b:a} (a holds bytes 0-3), or, when bit 3 of the selector nibble s_j is set, 0xFF
// or 0x00 after the top bit of that byte.  Only the low 16 bits of s are read.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t s)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(s));
    return d;
}

// Four int4 codes c (the nibbles in the low 16 bits of w; wx = w ^ 0x88888888) -> the e4m3 bytes
// of (c - 8) * 2^-9: c - 8 itself for c >= 8 (0x00-0x07), sign | (8 - c) = 0x88 - c below.  Two
// table lookups give both candidates (the selector's bit 3 picks the replicate mode, which
// leaves 0xFF or 0x00 where the other candidate applies); bit 6, set only in 0xFF, picks.
__device__ __forceinline__ uint32_t i4x4_to_signed_bytes(uint32_t w, uint32_t wx)
{
    const uint32_t neg = prmt(0x85868788u, 0x81828384u, w);   // c < 8: 0x88 - c; c >= 8: 0xFF
    const uint32_t pos = prmt(0x03020100u, 0x07060504u, wx);  // c >= 8: c - 8;  c < 8: 0x00
    const uint32_t sel = prmt(neg << 1, 0u, 0xBA98u);          // 0xFF in the bytes where c >= 8
    return (pos & sel) | (neg & ~sel);
}

// Eight int4 codes of one word -> the e4m3 bytes of (c - 8) * 2^-9, low byte first.
__device__ __forceinline__ uint2 i4x8_to_signed_bytes(uint32_t w)
{
    const uint32_t wx = w ^ 0x88888888u;
    return make_uint2(i4x4_to_signed_bytes(w, wx), i4x4_to_signed_bytes(w >> 16, wx >> 16));
}

}  // namespace tci
}  // namespace w4a8
