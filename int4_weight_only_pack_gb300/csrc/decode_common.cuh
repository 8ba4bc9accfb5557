// Consumer-side building blocks shared by the single-projection decode kernel
// (gemv.cu) and the persistent decode-step kernel (step.cu): staging x in
// shared memory, the per-tile multiply-accumulate, and the fixed-order
// reduction of a block's per-warp partials.
//
// Arithmetic of one tile (16 rows x 128 K, one scale group per row): the
// nibbles u enter the tensor core as exact fp16 subnormals (u * 2^-24 for rows
// r, u * 2^-20 for rows r + 8), x as fp16; mma.sync m16n8k16 multiplies
// exactly and sums in FP32 (two independent chains).  The group's partial
//     sum_k x*q = 2^24 * D - 8 * sum_k x        (2^20 for rows r + 8)
// is then scaled by the group's FP32 scale and added in FP32.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tc_ptx.cuh"
#include "w4_device.cuh"
#include "w4_internal.cuh"

namespace w4 {
namespace dec {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kChunk = 8;  // tiles per ring slot: one per consumer warp

__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// Activation types: binary16 (the pages' FP16 activations) or bfloat16.
enum : int { kActF16 = 0, kActBF16 = 1, kActI8 = 2 };  // kActI8: binary16 x quantised to INT8 (Path A)

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// First MMA of a chain: C = 0.
__device__ __forceinline__ void mma16816_zero(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
}

__device__ __forceinline__ void mma16816_bf(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma16816_bf_zero(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
}

// What changes with the activation type: how x pairs widen to FP32, how a
// result rounds, how a nibble word becomes MMA A registers, the MMA itself,
// and the constants that turn the MMA sum D into the group partial:
//   sum_k x * q = kLo * D - kBias * sum_k x      (kHi for rows r + 8)
//  * binary16: nibbles as exact subnormals u * 2^-24 (rows r) and u * 2^-20
//    (rows r + 8), 5 integer ops per word; kLo = 2^24, kHi = 2^20, kBias = 8.
//  * bfloat16: x is rescaled per (group, token) by a power of two 2^e that
//    puts the group's largest |x| in [2^14, 2^15), rounded to binary16 in
//    shared memory when it is staged, and then takes the binary16 path (the
//    5-op unpack; a bfloat16 unpack needs 7 ops per word, since a bfloat16
//    subnormal product would fall below FP32's normal range: that cost the
//    28-layer one-token step 1129 against 908 us).  Every x within 2^-28 of
//    its group's largest magnitude converts exactly (binary16 holds 11
//    significant bits to bfloat16's 8); smaller ones round to a multiple of
//    2^-24 * 2^-e, at most 2^-40 of the group's largest |x| away.  The group
//    partial is c' * D + d with c' = 2^(24-e) (2^(20-e) for rows r + 8) and
//    d = -8 * sum_k x, the FP32 sum of the bfloat16 values as given (equal to
//    -8 * 2^-e * sum_k x' wherever the conversion is exact; forming it before
//    the conversion took the 28-layer one-token step from 974 to 963 us), both
//    per (group, token) from the staging.
template <int ACT>
struct ActOps;
template <>
struct ActOps<kActF16> {
    static constexpr float kLo = 16777216.f, kHi = 1048576.f, kBias = 8.f;
    static constexpr bool kScaled = false;
    __device__ static __forceinline__ float2 to_float2(uint32_t v) {
        return __half22float2(*reinterpret_cast<const __half2*>(&v));
    }
    __device__ static __forceinline__ uint16_t round(float v) { return __half_as_ushort(__float2half_rn(v)); }
    __device__ static __forceinline__ void unpack(uint32_t v, uint32_t (&a)[4]) { unpack_word_biased(v, a); }
    __device__ static __forceinline__ void mma(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                               bool first) {
        if (first)
            mma16816_zero(c, a, b0, b1);
        else
            mma16816(c, a, b0, b1);
    }
};
template <>
struct ActOps<kActBF16> : ActOps<kActF16> {
    static constexpr bool kScaled = true;  // x staged as rescaled binary16 (above)
    // the staged input's pairs (before rescaling)
    __device__ static __forceinline__ float2 to_float2(uint32_t v) {
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
    }
    __device__ static __forceinline__ uint16_t round(float v) {
        return __bfloat16_as_ushort(__float2bfloat16_rn(v));
    }
};

template <>
struct ActOps<kActI8> {
    static constexpr bool kScaled = false;
    __device__ static __forceinline__ uint16_t round(float v) { return __half_as_ushort(__float2half_rn(v)); }
};

// Shared-memory bytes of an x slice of Gs groups for MP padded tokens, and of
// its per-group sums: xsum[gl * xsum_stride(MP) + m] (the stride is even so
// that a lane reads its token pair as one float2; eight floats of slack cover
// the reads of lanes whose MMA columns are padding and never written).  Both
// sizes are multiples of 16 bytes, so what follows them stays 16-byte aligned.
__host__ __device__ constexpr int x_bytes(int MP, int Gs) { return MP * Gs * 256; }
__host__ __device__ constexpr int xsum_stride(int MP) { return MP < 2 ? 2 : MP; }
// Rescaled binary16 x (bfloat16 input): per group d for tokens m at
// xsum[gl * xsum_gstride + m] and c' at + xsum_cofs (at one token the pair
// (d, c') fills the slot of the token and its padding neighbour).
__host__ __device__ constexpr int xsum_gstride(int MP, bool scaled) {
    return scaled && MP > 1 ? 2 * xsum_stride(MP) : xsum_stride(MP);
}
__host__ __device__ constexpr int xsum_cofs(int MP) { return MP > 1 ? xsum_stride(MP) : 1; }
__host__ __device__ constexpr int xsum_bytes(int MP, int Gs, bool scaled = false) {
    return ((Gs * xsum_gstride(MP, scaled) + 8 + 16) * 4 + 15) & ~15;  // + 16 floats: per-token scales (INT8 path)
}

// The power of two 2^e of a (group, token) of rescaled x, from the largest
// magnitude amax: e = 14 - floor(log2 amax), so that amax * 2^e lies in
// [2^14, 2^15), clamped to [-103, 126] (zero groups take 126; |x| must stay
// below 2^116).  Returns 2^e; c1 = 2^(24-e), the group's c' for rows r.
__device__ __forceinline__ float x_scale_of(float amax, float& c1) {
    const int E = (__float_as_int(amax) >> 23) & 0xFF;  // biased exponent of amax (0 for zero)
    const int e = min(126, max(-103, 141 - E));
    c1 = __int_as_float((151 - e) << 23);
    return __int_as_float((127 + e) << 23);
}
__device__ __forceinline__ uint32_t to_half2_bits(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Sum x over every group gl < Gs and token m < M into xsum[gl *
// xsum_stride(MP) + m], each lane adding the four values at word offsets
// word(gl, m) and word(gl, m) + 1 (the layout's fragment positions of lane
// class (lane >> 1) & 3, k16 step 2 * (lane >> 3) + (lane & 1)), then a
// butterfly over the warp: the same order, so the same bits, whatever the
// layout.  Warp w takes groups w, w + NW, ...; several groups' reductions are
// interleaved, and no index is divided by the run-time token count.
template <int MP, int NW, int ACT, typename Word>
__device__ __forceinline__ void sum_groups(uint32_t* xs, float* xsum, int M, int Gs, int warp, int lane,
                                           Word&& word) {
    // groups reduced together: two per warp with 16 warps (a K = 3584 slice has
    // 28 groups: four per warp left half of them empty, and the one-token
    // step took 911 us against 901 with two, 1010 against 986 at two tokens,
    // 962 against 938 with bfloat16 x), four with fewer warps
    constexpr int kBatch = NW >= 16 ? 2 : 4;
    constexpr bool kScaled = ActOps<ACT>::kScaled;
    constexpr int kG = xsum_gstride(MP, kScaled);
    for (int g0 = warp; g0 < Gs; g0 += NW * kBatch) {
        for (int m = 0; m < M; ++m) {
            float sum[kBatch], c1[kBatch];
            if constexpr (kScaled) {
                // rescale each group by its power of two and round to binary16 in place: the four
                // groups' maxima first (their butterflies interleaved), then the conversions
                // (the largest magnitude as an integer warp reduction of the bfloat16 magnitude bits, which
                // order like the values: one redux per group instead of a five-step shuffle butterfly)
                float2 f[kBatch][2];
                uint32_t mag[kBatch];
#pragma unroll
                for (int b = 0; b < kBatch; ++b) {
                    const int gl = g0 + b * NW;
                    uint32_t w0 = 0, w1 = 0;
                    if (gl < Gs) {
                        const uint32_t* src = xs + word(gl, m);
                        w0 = src[0];
                        w1 = src[1];
                    }
                    f[b][0] = ActOps<ACT>::to_float2(w0);
                    f[b][1] = ActOps<ACT>::to_float2(w1);
                    mag[b] = max(max(w0 & 0x7FFFu, (w0 >> 16) & 0x7FFFu), max(w1 & 0x7FFFu, (w1 >> 16) & 0x7FFFu));
                }
#pragma unroll
                for (int b = 0; b < kBatch; ++b) mag[b] = __reduce_max_sync(0xFFFFFFFFu, mag[b]);
#pragma unroll
                for (int b = 0; b < kBatch; ++b) {
                    const int gl = g0 + b * NW;
                    const float sc = x_scale_of(__uint_as_float(mag[b] << 16), c1[b]);
                    const uint32_t h0 = to_half2_bits(f[b][0].x * sc, f[b][0].y * sc);
                    const uint32_t h1 = to_half2_bits(f[b][1].x * sc, f[b][1].y * sc);
                    sum[b] = 0.f;
                    if (gl < Gs) {
                        uint32_t* dst = xs + word(gl, m);
                        dst[0] = h0;
                        dst[1] = h1;
                        // the bias term from the bfloat16 values themselves (no wait on the conversion)
                        sum[b] = (f[b][0].x + f[b][0].y) + (f[b][1].x + f[b][1].y);
                    }
                }
            } else {
#pragma unroll
                for (int b = 0; b < kBatch; ++b) {
                    const int gl = g0 + b * NW;
                    sum[b] = 0.f;
                    if (gl < Gs) {
                        const uint32_t* src = xs + word(gl, m);
                        const float2 f0 = ActOps<ACT>::to_float2(src[0]);
                        const float2 f1 = ActOps<ACT>::to_float2(src[1]);
                        sum[b] = (f0.x + f0.y) + (f1.x + f1.y);
                    }
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                for (int b = 0; b < kBatch; ++b) sum[b] += __shfl_xor_sync(0xFFFFFFFFu, sum[b], off);
            if (lane == 0)
#pragma unroll
                for (int b = 0; b < kBatch; ++b)
                    if (g0 + b * NW < Gs) {
                        if constexpr (kScaled) {  // d = -8 * sum of x, c' = 2^(24-e)
                            xsum[(g0 + b * NW) * kG + m] = -8.f * sum[b];
                            xsum[(g0 + b * NW) * kG + xsum_cofs(MP) + m] = c1[b];
                        } else {
                            xsum[(g0 + b * NW) * kG + m] = sum[b];
                        }
                    }
        }
    }
}

// Sum x over every group gl < Gs and token m < M of a natural-order slice
// (token rows of row_w words) into xsum[gl * xsum_stride(MP) + m]: eight
// threads per (group, token) pair, each adding its 16 consecutive values in a
// fixed order, then a three-step butterfly over the eight.  The work is spread
// over every thread whatever M is (a warp per pair left most lanes of a
// butterfly idle at 8 and 16 tokens).
template <int MP, int NCONS, int ACT>
__device__ __forceinline__ void sum_groups_nat(uint32_t* xs, float* xsum, int M, int Gs, int row_w) {
    constexpr bool kScaled = ActOps<ACT>::kScaled;
    constexpr int kG = xsum_gstride(MP, kScaled);
    const int tid = threadIdx.x, sub = tid & 7;
    const int pairs = Gs * M;
    constexpr int kStep = NCONS / 8;  // pairs per pass
    // pair p = gl * M + m, walked without dividing by M: (gl, m) advance together
    int gl = 0, m = tid >> 3;
    while (m >= M) {
        m -= M;
        ++gl;
    }
    // every lane runs every pass (the butterflies need the whole warp); lanes past the end add nothing
    for (int base = 0; base < pairs; base += kStep) {
        const bool live = base + (tid >> 3) < pairs;
        float sum = 0.f, c1 = 0.f;
        uint4* src = reinterpret_cast<uint4*>(xs + m * row_w + gl * 64 + sub * 8);
        uint4 a = make_uint4(0, 0, 0, 0), b = a;
        if (live) {
            a = src[0];
            b = src[1];
        }
        uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        if (live) {  // the sum of x as given (for rescaled x, before the rescale)
            float t[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float2 f = ActOps<ACT>::to_float2(w[k]);
                t[k] = f.x + f.y;
            }
            sum = ((t[0] + t[1]) + (t[2] + t[3])) + ((t[4] + t[5]) + (t[6] + t[7]));
        }
        if constexpr (kScaled) {
            // rescale by the (group, token)'s power of two and round to binary16 in place
            float amax = 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float2 f = ActOps<ACT>::to_float2(w[k]);
                amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
            const float sc = x_scale_of(amax, c1);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float2 f = ActOps<ACT>::to_float2(w[k]);
                w[k] = to_half2_bits(f.x * sc, f.y * sc);
            }
            if (live) {
                src[0] = make_uint4(w[0], w[1], w[2], w[3]);
                src[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
        }
        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 4);
        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
        if (live && sub == 0) {
            if constexpr (kScaled) {  // d = -8 * sum of x, c' = 2^(24-e)
                xsum[gl * kG + m] = -8.f * sum;
                xsum[gl * kG + xsum_cofs(MP) + m] = c1;
            } else {
                xsum[gl * kG + m] = sum;
            }
        }
        m += kStep;
        while (m >= M) {
            m -= M;
            ++gl;
        }
    }
}

// Stage x[0:M, 128*g_lo : 128*(g_lo+Gs)) (fp16 pairs; row stride K/2 words)
// into `xs` in fragment order -- word (gl, q, m, c, e) at
// gl*MP*64 + q*MP*16 + (m*4 + c)*4 + e holds k16 step 2q + (e >> 1) of group
// gl, k 4c + 2(e & 1) .. +1 -- with rows M..MP-1 zero, and the sum of x over
// every group and token m < M into xsum[gl*xsum_stride(MP) + m].  Every
// 8-byte piece (the b0, b1 words of one lane class and k16 step) is copied
// from global memory straight into its fragment slot by a cp.async, all
// issued before any is waited for: one memory round trip whatever the slice
// size (synchronous loads, eight in flight per thread, took 2.6-4 us per
// decode-kernel launch).  Called by the NCONS threads tid < NCONS; returns
// with them synchronised.  x must be 8-byte aligned.
template <int MP, int NCONS, int ACT = kActF16>
__device__ __forceinline__ void stage_x_async(const uint32_t* x, int M, int K, int g_lo, int Gs, uint32_t* xs,
                                              float* xsum) {
    constexpr int kWarps = NCONS / 32;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int per_row = Gs * 64;
    const uint32_t* xg = x + (size_t)g_lo * 64;
    const int kp = K / 2;
    const uint32_t xs_s = tc::smem_addr(xs);
    // 8-byte pieces: k 4c .. 4c+3 of one k16 step (its b0 and b1 words)
    const int per_row8 = per_row / 2;
    for (int m = 0; m < MP; ++m) {
        for (int r = tid; r < per_row8; r += NCONS) {
            const int gl = r >> 5, kq = r & 31;
            const int j = kq >> 2, c = kq & 3;
            const int dst = gl * (MP * 64) + (j >> 1) * (MP * 16) + (m * 4 + c) * 4 + (j & 1) * 2;
            if (m < M)
                asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(xs_s + 4u * dst),
                             "l"(xg + (size_t)m * kp + 2 * r)
                             : "memory");
            else
                *reinterpret_cast<uint2*>(xs + dst) = make_uint2(0, 0);
        }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    tc::named_barrier(1, NCONS);
    const int q = lane >> 3, c = (lane >> 1) & 3, e = (lane & 1) * 2;
    sum_groups<MP, kWarps, ACT>(xs, xsum, M, Gs, warp, lane, [&](int gl, int m) {
        return gl * (MP * 64) + q * (MP * 16) + (m * 4 + c) * 4 + e;
    });
    tc::named_barrier(1, NCONS);
}

// Natural-order x slice (the step kernel from 4 tokens on): token m's Gs*128
// values are contiguous at byte m * x_row_bytes(Gs); rows are padded by 32
// bytes so that the 8-byte fragment loads of 8 tokens (a half warp's) fall in
// distinct banks.  One bulk copy per token row fills it.
__host__ __device__ constexpr int x_row_bytes(int Gs) { return Gs * 256 + 32; }
__host__ __device__ constexpr int x_bytes_nat(int MP, int Gs) { return MP * x_row_bytes(Gs); }

// Stage x[0:M, 128*g_lo : 128*(g_lo+Gs)) into `xs` in natural order (one bulk
// copy per token row, completing on the mbarrier `bar`, whose phase `phase`
// this staging completes), zero the rows of padded tokens M..MP-1, and write
// the sum of x over every group and token m < M into xsum[gl*xsum_stride(MP)
// + m] -- each lane adding the same four values in the same order as with the
// fragment layout, so the sums are the same bits.  Called by all NCONS
// threads; returns with them synchronised; false if the copies did not land
// within the wait's bound.  x must be 16-byte aligned and K a multiple of 128.
template <int MP, int NCONS, int ACT = kActF16>
__device__ __forceinline__ bool stage_x_bulk(const uint32_t* x, int M, int K, int g_lo, int Gs, uint32_t* xs,
                                             float* xsum, uint32_t bar, uint32_t phase) {
    const int tid = threadIdx.x;
    const int row = x_row_bytes(Gs), row_w = row / 4;
    if constexpr (MP >= 16) {
        // lane m issues token row m's copy, lane 0 having posted the bytes to expect first (at 16
        // tokens this took the step from 1792 to 1766 us; at 4 and 8 tokens one thread issuing
        // every row measured faster, 1125 against 1134 and 1208 against 1219 us)
        if (tid < 32) {
            if (tid == 0) tc::mbar_arrive_expect_tx(bar, (uint32_t)(M * Gs * 256));
            __syncwarp();
            if (tid < M)
                tc::bulk_load(tc::smem_addr(xs) + (uint32_t)(tid * row), x + (size_t)tid * (K / 2) + (size_t)g_lo * 64,
                              (uint32_t)(Gs * 256), bar);
        }
    } else if (tid == 0) {
        tc::mbar_arrive_expect_tx(bar, (uint32_t)(M * Gs * 256));
        const uint32_t xs_s = tc::smem_addr(xs);
        for (int m = 0; m < M; ++m)
            tc::bulk_load(xs_s + (uint32_t)(m * row), x + (size_t)m * (K / 2) + (size_t)g_lo * 64, (uint32_t)(Gs * 256),
                          bar);
    }
    for (int i = tid; i < (MP - M) * Gs * 64; i += NCONS) {
        const int m = M + i / (Gs * 64), w = i - (m - M) * (Gs * 64);
        xs[m * row_w + w] = 0;
    }
    const bool ok = tc::mbar_wait(bar, phase);
    sum_groups_nat<MP, NCONS, ACT>(xs, xsum, M, Gs, row_w);
    tc::named_barrier(1, NCONS);
    return ok;
}

// Predicated shared-memory loads: lanes whose predicate is false issue no
// access (and cost no bandwidth) and keep the register's previous contents.
__device__ __forceinline__ void lds128_if(uint4& v, uint32_t a, uint32_t pred) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n @p ld.shared.v4.u32 {%0,%1,%2,%3}, [%5];\n}\n"
        : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)
        : "r"(pred), "r"(a));
}
__device__ __forceinline__ void lds64f_if(float2& v, uint32_t a, uint32_t pred) {
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %2, 0;\n @p ld.shared.v2.f32 {%0,%1}, [%3];\n}\n"
                 : "+f"(v.x), "+f"(v.y)
                 : "r"(pred), "r"(a));
}
__device__ __forceinline__ void lds64_if(uint32_t& lo, uint32_t& hi, uint32_t a, uint32_t pred) {
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %2, 0;\n @p ld.shared.v2.u32 {%0,%1}, [%3];\n}\n"
                 : "+r"(lo), "+r"(hi)
                 : "r"(pred), "r"(a));
}

// Per-lane state of the tile multiply-accumulate.
//
// Lane L = 4*tok + cl4 holds the B fragment of MMA column tok (a token) and
// the accumulators of tokens nt*8 + 2*cl4 + {0, 1}.  Only lanes of real
// (padded) tokens, tok < MP, load x fragments and only lanes whose first
// token is real load group sums: the other lanes' MMA columns are never
// written out, so whatever their registers hold is harmless, and the loads
// they skip are shared-memory bandwidth saved.
template <int MP, int ACT = kActF16>
struct TileMac {
    using Ops = ActOps<ACT>;
    static constexpr int NT = (MP + 7) / 8;  // n8 token tiles of the MMA
    static constexpr int NE = MP == 1 ? 1 : 2;  // tokens per lane that can be real (token 2*cl4 + 1 >= MP=1)
    uint32_t xfrag;                          // this lane's B-fragment words of group 0
    uint32_t xsum;                           // this lane's token pair's sums of group 0
    uint32_t xl, sl;                         // load predicates: x fragments, group sums
    uint4 xv[4][NT];                         // x fragments of up to four tiles
    float2 X[4][NT];                         // group sums (rescaled x: d) of up to four tiles
    float2 C[Ops::kScaled && MP > 1 ? 4 : 1][NT];  // rescaled x, two or more tokens: c' of the token pair
    int xrow = 0;                            // natural x layout: bytes per token row

    __device__ __forceinline__ TileMac(uint32_t x_smem, uint32_t xsum_smem, int lane, int /*Gs*/ = 0) {
        const int tok = lane >> 2, cl4 = lane & 3;
        xfrag = x_smem + (uint32_t)(((tok % MP) * 4 + cl4) * 16);
        xsum = xsum_smem + (uint32_t)(2 * cl4 * 4);
        xl = tok < MP;
        sl = 2 * cl4 < MP || MP >= 8;
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                xv[n][nt] = make_uint4(0, 0, 0, 0);
                X[n][nt] = make_float2(0.f, 0.f);
            }
#pragma unroll
        for (int n = 0; n < (Ops::kScaled && MP > 1 ? 4 : 1); ++n)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) C[n][nt] = make_float2(0.f, 0.f);
    }

    // Read x from the natural layout of stage_x_bulk (rows of row_bytes)
    // instead of the fragment layout: run_tiles<NTL, true>.
    __device__ __forceinline__ void set_natural(uint32_t x_smem, int lane, int row_bytes) {
        const int tok = lane >> 2, cl4 = lane & 3;
        xrow = row_bytes;
        xfrag = x_smem + (uint32_t)((tok % MP) * row_bytes + cl4 * 8);
    }

    // acc += s * sum_{k in group} x * q for NTL consecutive tiles at ta, ta +
    // 1056, ... (groups gl, gl + 1, ... of one band), their MMA chains
    // interleaved; the tiles are added to acc in order.  Per tile and row:
    //     acc += s * (kLo * D - kBias * sum_k x)      (kHi for rows r + 8)
    // NAT: x in the natural layout (two 8-byte loads per pair of k16 steps:
    // the same registers as the fragment layout's one 16-byte load).
    template <int NTL, bool NAT = false>
    __device__ __forceinline__ void run_tiles(uint32_t ta, int gl, int lane, float (&acc)[NT][4]) {
        uint32_t wd[NTL][8], sc[NTL];
#pragma unroll
        for (int n = 0; n < NTL; ++n) {
            const uint32_t tn = ta + (uint32_t)(n * kTileBytes);
            const uint4 lo = lds128(tn + 16 * lane), hi = lds128(tn + 512 + 16 * lane);
            wd[n][0] = lo.x, wd[n][1] = lo.y, wd[n][2] = lo.z, wd[n][3] = lo.w;
            wd[n][4] = hi.x, wd[n][5] = hi.y, wd[n][6] = hi.z, wd[n][7] = hi.w;
            sc[n] = lds32(tn + kScaleOffset + 4 * (lane >> 2));
            constexpr int kG = xsum_gstride(MP, Ops::kScaled);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                lds64f_if(X[n][nt], xsum + (uint32_t)(((gl + n) * kG + nt * 8) * 4), sl);
                if constexpr (Ops::kScaled && MP > 1)
                    lds64f_if(C[n][nt], xsum + (uint32_t)(((gl + n) * kG + xsum_cofs(MP) + nt * 8) * 4), sl);
            }
        }
        const uint32_t xa0 = NAT ? xfrag + (uint32_t)gl * 256 : xfrag + (uint32_t)gl * (MP * 256);
        float pe[NTL][NT][4], po[NTL][NT][4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // k16 steps 2q (even chain) and 2q + 1 (odd chain)
#pragma unroll
            for (int n = 0; n < NTL; ++n) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    if constexpr (NAT) {
                        const uint32_t a = xa0 + (uint32_t)(n * 256 + q * 64 + nt * 8 * xrow);
                        lds64_if(xv[n][nt].x, xv[n][nt].y, a, xl);
                        lds64_if(xv[n][nt].z, xv[n][nt].w, a + 32, xl);
                    } else {
                        lds128_if(xv[n][nt], xa0 + (uint32_t)(n * MP * 256 + q * MP * 64 + nt * 512), xl);
                    }
                }
                uint32_t a[4], b[4];
                Ops::unpack(wd[n][2 * q], a);
                Ops::unpack(wd[n][2 * q + 1], b);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint4 v = xv[n][nt];
                    Ops::mma(pe[n][nt], a, v.x, v.y, q == 0);
                    Ops::mma(po[n][nt], b, v.z, v.w, q == 0);
                }
            }
        }
#pragma unroll
        for (int n = 0; n < NTL; ++n) {
            const float2 s = __half22float2(*reinterpret_cast<const __half2*>(&sc[n]));  // rows r, r + 8
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int e = 0; e < NE; ++e) {
                    if constexpr (Ops::kScaled) {
                        // d and c' of the token: at one token the pair (d, c') of the group's slot
                        const float d = e ? X[n][nt].y : X[n][nt].x;
                        const float c1 = MP == 1 ? X[n][nt].y : (e ? C[n % (MP > 1 ? 4 : 1)][nt].y
                                                                   : C[n % (MP > 1 ? 4 : 1)][nt].x);
                        acc[nt][e] = fmaf(s.x, fmaf(c1, pe[n][nt][e] + po[n][nt][e], d), acc[nt][e]);
                        acc[nt][2 + e] =
                            fmaf(s.y, fmaf(c1 * 0.0625f, pe[n][nt][2 + e] + po[n][nt][2 + e], d), acc[nt][2 + e]);
                    } else {
                        const float mbx = -Ops::kBias * (e ? X[n][nt].y : X[n][nt].x);
                        acc[nt][e] = fmaf(s.x, fmaf(Ops::kLo, pe[n][nt][e] + po[n][nt][e], mbx), acc[nt][e]);
                        acc[nt][2 + e] =
                            fmaf(s.y, fmaf(Ops::kHi, pe[n][nt][2 + e] + po[n][nt][2 + e], mbx), acc[nt][2 + e]);
                    }
                }
            }
        }
    }

    // One tile.
    __device__ __forceinline__ void run(uint32_t ta, int gl, int lane, float (&acc)[NT][4]) {
        run_tiles<1>(ta, gl, lane, acc);
    }
};

// Shared-memory floats of one buffer of per-warp block partials:
// [warp][band][nt][lane][4].
__host__ __device__ constexpr int red_floats(int BB, int NT, int warps = kConsumerWarps) {
    return warps * BB * NT * 128;
}

// Fixed-order sum over the consumer warps of the block partials for the
// outputs t = tid + i * kConsumers < nb*16*M (t = m * nb*16 + band row);
// NaN where !ok.
template <int NT, int NCONS = kConsumers>
__device__ __forceinline__ void block_sums(const float* red, int BB, int nb, int M, bool ok, float (&v)[4]) {
    constexpr int kConsumers = NCONS, kConsumerWarps = NCONS / 32;
    const int Tout = nb * 16 * M;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = threadIdx.x + i * kConsumers;
        v[i] = 0.f;
        if (t < Tout) {
            const int m = t / (nb * 16), rl = t - m * (nb * 16);
            const int bb = rl >> 4, rr = rl & 15;
            const int nt = m >> 3, col = m & 7;
            const int ln = (rr & 7) * 4 + (col >> 1), r = (rr >> 3) * 2 + (col & 1);
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) sum += red[((w * BB + bb) * NT + nt) * 128 + ln * 4 + r];
            v[i] = ok ? sum : __int_as_float(0x7FC00000);
        }
    }
}

// ---- Path A: INT8 activations ----------------------------------------------------
// Per-token symmetric quantisation in IEEE binary32 (round-to-nearest
// division, then round half to even): sx = max_k |x| / 127,
// xq = rne(x / sx) clamped to +-127.  The CTA reads the whole row for the
// maximum and quantises its K slice into shared memory as bytes in the order
// the nibble bytes come out of a packed word ((v & 0x0F0F0F0F) gives k 4c+0,
// 4c+2, 4c+1, 4c+3 of rows r; (v >> 4) the same of rows r + 8): word
// ((gl*MP + m)*4 + c)*8 + j holds k16 step j of lane class c.  Per group and
// token the integer sum of xq goes to xsum[gl*xsum_stride(MP) + m] (as int)
// and sx to xsum[Gs*xsum_stride(MP) + 8 + m].
template <int MP, int NCONS>
__device__ __forceinline__ void stage_x_q8(const uint32_t* x, int M, int K, int g_lo, int Gs, uint32_t* xs,
                                           float* xsum, float* red /* NCONS / 32 * MP floats of scratch */) {
    constexpr int kWarps = NCONS / 32;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kp = K / 2;
    float* sxs = xsum + Gs * xsum_stride(MP) + 8;
    int* isum = reinterpret_cast<int*>(xsum);
    for (int m = 0; m < M; ++m) {
        float mx = 0.f;
        for (int i = tid; i < kp; i += NCONS) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(x + (size_t)m * kp + i));
            mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
        if (lane == 0) red[warp * MP + m] = mx;
    }
    tc::named_barrier(1, NCONS);
    if (tid < MP) {
        float mx = 0.f;
        if (tid < M)
            for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, red[w * MP + tid]);
        sxs[tid] = __fdiv_rn(mx, 127.f);
    }
    tc::named_barrier(1, NCONS);
    // quantise the slice: one thread per (token, group, k16 step, lane class)
    const uint32_t* xg = x + (size_t)g_lo * 64;
    for (int idx = tid; idx < MP * Gs * 32; idx += NCONS) {
        const int m = idx / (Gs * 32), rest = idx - m * (Gs * 32);
        const int gl = rest >> 5, jc = rest & 31, j = jc >> 2, c = jc & 3;
        uint32_t word = 0;
        if (m < M) {
            const float sc = sxs[m];
            const int k0 = gl * 128 + 16 * j + 4 * c;  // within the slice
            const uint32_t w01 = xg[(size_t)m * kp + k0 / 2], w23 = xg[(size_t)m * kp + k0 / 2 + 1];
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w01));
            const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&w23));
            const float v[4] = {a.x, b.x, a.y, b.y};  // k 4c+0, 4c+2, 4c+1, 4c+3
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                int qv = 0;
                if (sc > 0.f) qv = max(-127, min(127, __float2int_rn(__fdiv_rn(v[e], sc))));
                word |= (uint32_t)(qv & 0xFF) << (8 * e);
            }
        }
        xs[((gl * MP + m) * 4 + c) * 8 + j] = word;
    }
    tc::named_barrier(1, NCONS);
    // integer sum of xq per group and token
    for (int idx = warp; idx < Gs * MP; idx += kWarps) {
        const int gl = idx / MP, m = idx - gl * MP;
        const uint32_t w = xs[((gl * MP + m) * 4 + (lane >> 3)) * 8 + (lane & 7)];
        int sum = (int)(int8_t)(w & 0xFF) + (int)(int8_t)((w >> 8) & 0xFF) + (int)(int8_t)((w >> 16) & 0xFF) +
                  (int)(int8_t)(w >> 24);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
        if (lane == 0) isum[gl * xsum_stride(MP) + m] = sum;
    }
    tc::named_barrier(1, NCONS);
}

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Path A tile multiply-accumulate: per lane, for rows r and r + 8 and every
// token, exact integer dot products of the nibbles u (unsigned bytes) with
// xq (signed bytes) over the lane's 32 k of the group (dp4a); the four lanes
// of a row quad add theirs (shuffles), and each lane keeps the tokens its MMA
// fragment position owns, so the reduction and finishing code is the one of
// the tensor-core path:
//     acc += s * sx * (sum_k u*xq - 8 * sum_k xq)
template <int MP>
struct TileMac<MP, kActI8> {
    static constexpr int NT = (MP + 7) / 8;
    uint32_t xq_base, xsum_base, sx_base;
    int gs_stride;

    __device__ __forceinline__ TileMac(uint32_t x_smem, uint32_t xsum_smem, int lane, int Gs) {
        const int c = lane & 3;
        xq_base = x_smem + (uint32_t)(c * 8 * 4);
        xsum_base = xsum_smem;
        sx_base = xsum_smem + (uint32_t)((Gs * xsum_stride(MP) + 8) * 4);
        gs_stride = Gs;
    }

    template <int NTL, bool NAT = false>  // NAT: unused (Path A keeps its own x layout)
    __device__ __forceinline__ void run_tiles(uint32_t ta, int gl, int lane, float (&acc)[NT][4]) {
#pragma unroll
        for (int n = 0; n < NTL; ++n) run(ta + (uint32_t)(n * kTileBytes), gl + n, lane, acc);
    }

    __device__ __forceinline__ void run(uint32_t ta, int gl, int lane, float (&acc)[NT][4]) {
        const uint4 lo4 = lds128(ta + 16 * lane), hi4 = lds128(ta + 512 + 16 * lane);
        const uint32_t sc = lds32(ta + kScaleOffset + 4 * (lane >> 2));
        const uint32_t wd[8] = {lo4.x, lo4.y, lo4.z, lo4.w, hi4.x, hi4.y, hi4.z, hi4.w};
        uint32_t lo[8], hi[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            lo[j] = wd[j] & 0x0F0F0F0Fu;
            hi[j] = (wd[j] >> 4) & 0x0F0F0F0Fu;
        }
        const float2 s = __half22float2(*reinterpret_cast<const __half2*>(&sc));  // rows r, r + 8
        const int cl4 = lane & 3;
        const int* isum = reinterpret_cast<const int*>(__cvta_shared_to_generic(xsum_base));
        const float* sx = reinterpret_cast<const float*>(__cvta_shared_to_generic(sx_base));
#pragma unroll
        for (int m = 0; m < MP; ++m) {
            const uint32_t xa = xq_base + (uint32_t)((gl * MP + m) * 4 * 8 * 4);
            const uint4 x0 = lds128(xa), x1 = lds128(xa + 16);
            const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            int ar = 0, ar8 = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                ar = dp4a_us(lo[j], xw[j], ar);
                ar8 = dp4a_us(hi[j], xw[j], ar8);
            }
            ar += __shfl_xor_sync(0xFFFFFFFFu, ar, 1);
            ar8 += __shfl_xor_sync(0xFFFFFFFFu, ar8, 1);
            ar += __shfl_xor_sync(0xFFFFFFFFu, ar, 2);
            ar8 += __shfl_xor_sync(0xFFFFFFFFu, ar8, 2);
            // the lane whose fragment position holds token m keeps it
            const int nt = m >> 3, e = m & 1;
            if (((m & 7) >> 1) == cl4) {
                const int b8 = 8 * isum[gl * xsum_stride(MP) + m];
                const float f = sx[m];
                acc[nt][e] = fmaf(s.x * f, (float)(ar - b8), acc[nt][e]);
                acc[nt][2 + e] = fmaf(s.y * f, (float)(ar8 - b8), acc[nt][2 + e]);
            }
        }
    }
};

}  // namespace dec
}  // namespace w4
