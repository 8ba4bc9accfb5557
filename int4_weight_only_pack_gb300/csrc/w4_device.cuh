// Device helpers shared by the decode and prefill kernels: streaming loads of
// the packed weight and the nibble -> fp16 unpack (see include/w4.h for the
// layout).
#pragma once

#include <stdint.h>

namespace w4 {

__device__ __forceinline__ uint4 ld_stream16(const uint8_t* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld_stream4(const uint8_t* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// (v & mask) | magic in one LOP3.
__device__ __forceinline__ uint32_t and_or(uint32_t v, uint32_t mask, uint32_t magic) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(v), "r"(mask), "r"(magic));
    return r;
}

// Eight nibbles u (offset binary) of lane (r, c) -> four f16x2 registers
// holding q = u - 8: a[0] = rows r, k 4c..4c+1; a[1] = row r+8, same k;
// a[2] = row r, k 4c+2..4c+3; a[3] = row r+8, same k.  In this order they are
// an m16n8k16 A fragment (see include/w4.h for the k relabelling).
__device__ __forceinline__ void unpack_word(uint32_t v, uint32_t (&a)[4]) {
    const uint32_t lo_mask = 0x000F000Fu, hi_mask = 0x00F000F0u, magic = 0x64006400u;
    const uint32_t v8 = v >> 8;
    const uint32_t t0 = and_or(v, lo_mask, magic);   // 1024 + u  (nibbles 0, 4)
    const uint32_t t1 = and_or(v, hi_mask, magic);   // 1024 + 16u (nibbles 1, 5)
    const uint32_t t2 = and_or(v8, lo_mask, magic);  // nibbles 2, 6
    const uint32_t t3 = and_or(v8, hi_mask, magic);  // nibbles 3, 7
    const uint32_t k1032 = 0x64086408u;              // 1032
    const uint32_t k1_16 = 0x2C002C00u;              // 1/16
    const uint32_t km72 = 0xD480D480u;               // -72
    asm("sub.f16x2 %0, %1, %2;" : "=r"(a[0]) : "r"(t0), "r"(k1032));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(a[1]) : "r"(t1), "r"(k1_16), "r"(km72));
    asm("sub.f16x2 %0, %1, %2;" : "=r"(a[2]) : "r"(t2), "r"(k1032));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(a[3]) : "r"(t3), "r"(k1_16), "r"(km72));
}

// Eight nibbles u of lane (r, c) -> four f16x2 registers holding u itself
// as fp16 subnormals: a[0] = u * 2^-24 of row r, k 4c..4c+1; a[1] = u * 2^-20
// (16u * 2^-24) of row r+8; a[2], a[3] the same for k 4c+2..4c+3.  Every
// value is exact; the caller rescales rows r and r+8 by 2^24 and 2^20 and
// subtracts 8 * sum(x) to turn u into q = u - 8.
__device__ __forceinline__ void unpack_word_biased(uint32_t v, uint32_t (&a)[4]) {
    const uint32_t v8 = v >> 8;
    a[0] = v & 0x000F000Fu;
    a[1] = v & 0x00F000F0u;
    a[2] = v8 & 0x000F000Fu;
    a[3] = v8 & 0x00F000F0u;
}

}  // namespace w4
