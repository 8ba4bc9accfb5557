// Offline repack of (q, scales) into the tile layout the decode and prefill
// kernels read, and its inverse.  The layout is specified in include/w4.h.
//
// The pages call their layout "ValueShuffle": INT4 nibbles interleaved even
// with odd so that the byte-permute datapath unpacks them cheaply ("Building a
// Custom LLM Inference Runtime ...", "The .nanoqwen File Format and Safety
// Protocols").  Here the shuffle is chosen so that one 32-bit word per lane
// and k16-step becomes, after two masks and one shift, the four f16x2
// registers of an m16n8k16 tensor-core A fragment; the tile's 16 scales sit
// right behind its nibbles so one stream carries both.
#include <cstdlib>
#include <cstring>
#include <vector>

#include "w4_internal.cuh"

namespace w4 {

// Nibble i (0..7) of the word owned by lane L = 4r + c at k16-step j holds the
// element at (row within band, k within group):
//   row = r + 8 * (i & 1),  k = 16 j + 4 c + 2 * ((i >> 1) & 1) + (i >> 2).
__host__ __device__ inline int nib_row(int L, int i) { return (L >> 2) + 8 * (i & 1); }
__host__ __device__ inline int nib_k(int L, int j, int i) {
    return 16 * j + 4 * (L & 3) + 2 * ((i >> 1) & 1) + (i >> 2);
}
// Byte offset of that word inside its tile.
__host__ __device__ inline int word_offset(int L, int j) { return (j >> 2) * 512 + 16 * L + 4 * (j & 3); }

// Source row of packed row n.  glu_I = 0: the identity.  glu_I = I > 0: the
// source is a stacked [gate (I rows); up (I rows)] weight and 16-row band b
// takes gate rows 8b .. 8b+7 then up rows 8b .. 8b+7, so rows r and r + 8 of
// every band are a (gate, up) pair.
__host__ __device__ inline int64_t src_row(int64_t n, int64_t glu_I) {
    if (glu_I == 0) return n;
    const int64_t b = n >> 4, r = n & 15;
    return r < 8 ? 8 * b + r : glu_I + 8 * b + (r - 8);
}

static bool q_in_range(const int8_t* q, size_t n) {
    for (size_t i = 0; i < n; ++i)
        if (q[i] < -8 || q[i] > 7) return false;
    return true;
}

static w4_status check_shape(int64_t N, int64_t K) {
    if (N < 1 || K < kGroupK || K % kGroupK != 0) {
        set_error("shape N=%lld K=%lld: need N >= 1 and K a positive multiple of 128", (long long)N,
                  (long long)K);
        return W4_ERR_SHAPE;
    }
    return W4_OK;
}

static void pack_host_impl(const int8_t* q, const uint16_t* s, int64_t N, int64_t K, uint8_t* dst,
                           int64_t glu_I = 0) {
    const int64_t G = num_groups(K), B = num_bands(N);
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t g = 0; g < G; ++g) {
            uint8_t* tile = dst + (b * G + g) * kTileBytes;
            for (int L = 0; L < 32; ++L) {
                for (int j = 0; j < 8; ++j) {
                    uint32_t word = 0;
                    for (int i = 0; i < 8; ++i) {
                        const int64_t n = b * kBandRows + nib_row(L, i);
                        const int64_t k = g * kGroupK + nib_k(L, j, i);
                        const uint32_t u = n < N ? (uint32_t)(q[src_row(n, glu_I) * K + k] + 8) : 8u;
                        word |= u << (4 * i);
                    }
                    memcpy(tile + word_offset(L, j), &word, 4);  // little-endian hosts only
                }
            }
            for (int p = 0; p < 8; ++p) {
                const int64_t n0 = b * kBandRows + p, n1 = n0 + 8;
                const uint32_t lo = n0 < N ? s[src_row(n0, glu_I) * G + g] : 0u;
                const uint32_t hi = n1 < N ? s[src_row(n1, glu_I) * G + g] : 0u;
                const uint32_t word = lo | (hi << 16);
                memcpy(tile + kScaleOffset + 4 * p, &word, 4);
            }
        }
    }
}

static void unpack_host_impl(const uint8_t* src, int64_t N, int64_t K, int8_t* q, uint16_t* s) {
    const int64_t G = num_groups(K), B = num_bands(N);
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t g = 0; g < G; ++g) {
            const uint8_t* tile = src + (b * G + g) * kTileBytes;
            for (int L = 0; L < 32; ++L) {
                for (int j = 0; j < 8; ++j) {
                    uint32_t word;
                    memcpy(&word, tile + word_offset(L, j), 4);
                    for (int i = 0; i < 8; ++i) {
                        const int64_t n = b * kBandRows + nib_row(L, i);
                        if (n >= N) continue;
                        const int64_t k = g * kGroupK + nib_k(L, j, i);
                        q[n * K + k] = (int8_t)((int)((word >> (4 * i)) & 15u) - 8);
                    }
                }
            }
            for (int p = 0; p < 8; ++p) {
                uint32_t word;
                memcpy(&word, tile + kScaleOffset + 4 * p, 4);
                const int64_t n0 = b * kBandRows + p, n1 = n0 + 8;
                if (n0 < N) s[n0 * G + g] = (uint16_t)(word & 0xFFFFu);
                if (n1 < N) s[n1 * G + g] = (uint16_t)(word >> 16);
            }
        }
    }
}

// One CTA per tile, one thread per 32-bit nibble word; threads 0..7 also
// write the tile's scale words.
__global__ void __launch_bounds__(256) pack_kernel(const int8_t* __restrict__ q,
                                                   const uint16_t* __restrict__ s, int64_t N, int64_t K,
                                                   uint8_t* __restrict__ dst, unsigned* bad, int64_t glu_I) {
    const int64_t G = K / kGroupK;
    const int64_t t = blockIdx.x;
    const int64_t b = t / G, g = t % G;
    const int L = threadIdx.x >> 3, j = threadIdx.x & 7;
    uint32_t word = 0;
    bool ok = true;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t n = b * kBandRows + nib_row(L, i);
        int v = 0;
        if (n < N) v = q[src_row(n, glu_I) * K + g * kGroupK + nib_k(L, j, i)];
        ok &= (v >= -8 && v <= 7);
        word |= (uint32_t)((v + 8) & 15) << (4 * i);
    }
    uint8_t* tile = dst + t * kTileBytes;
    *reinterpret_cast<uint32_t*>(tile + word_offset(L, j)) = word;
    if (threadIdx.x < 8) {
        const int p = threadIdx.x;
        const int64_t n0 = b * kBandRows + p, n1 = n0 + 8;
        const uint32_t lo = n0 < N ? s[src_row(n0, glu_I) * G + g] : 0u;
        const uint32_t hi = n1 < N ? s[src_row(n1, glu_I) * G + g] : 0u;
        *reinterpret_cast<uint32_t*>(tile + kScaleOffset + 4 * p) = lo | (hi << 16);
    }
    if (!ok) atomicOr(bad, 1u);
}

__global__ void __launch_bounds__(256) unpack_kernel(const uint8_t* __restrict__ src, int64_t N, int64_t K,
                                                     int8_t* __restrict__ q, uint16_t* __restrict__ s) {
    const int64_t G = K / kGroupK;
    const int64_t t = blockIdx.x;
    const int64_t b = t / G, g = t % G;
    const int L = threadIdx.x >> 3, j = threadIdx.x & 7;
    const uint8_t* tile = src + t * kTileBytes;
    const uint32_t word = *reinterpret_cast<const uint32_t*>(tile + word_offset(L, j));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t n = b * kBandRows + nib_row(L, i);
        if (n < N) q[n * K + g * kGroupK + nib_k(L, j, i)] = (int8_t)((int)((word >> (4 * i)) & 15u) - 8);
    }
    if (threadIdx.x < 8) {
        const int p = threadIdx.x;
        const uint32_t word_s = *reinterpret_cast<const uint32_t*>(tile + kScaleOffset + 4 * p);
        const int64_t n0 = b * kBandRows + p, n1 = n0 + 8;
        if (n0 < N) s[n0 * G + g] = (uint16_t)(word_s & 0xFFFFu);
        if (n1 < N) s[n1 * G + g] = (uint16_t)(word_s >> 16);
    }
}

}  // namespace w4

using namespace w4;

extern "C" size_t w4_packed_bytes(int64_t N, int64_t K) {
    if (N < 1 || K < kGroupK || K % kGroupK != 0) return 0;
    return (size_t)(num_bands(N) * num_groups(K)) * kTileBytes;
}

extern "C" w4_status w4_weight_view(const void* packed_dev, int64_t N, int64_t K, w4_weight* out) {
    clear_error();
    if (!out || !packed_dev) {
        set_error("NULL argument");
        return W4_ERR_ARG;
    }
    w4_status st = check_shape(N, K);
    if (st != W4_OK) return st;
    if (!aligned16(packed_dev)) {
        set_error("packed pointer not 16-byte aligned");
        return W4_ERR_ALIGN;
    }
    out->data = packed_dev;
    out->N = N;
    out->K = K;
    out->magic = W4_PACK_MAGIC;
    out->version = W4_PACK_VERSION;
    return W4_OK;
}

extern "C" w4_status w4_pack_host(const int8_t* q, const uint16_t* scales, int64_t N, int64_t K, void* dst,
                                  size_t dst_bytes) {
    clear_error();
    w4_status st = check_shape(N, K);
    if (st != W4_OK) return st;
    if (!q || !scales || !dst) {
        set_error("NULL argument");
        return W4_ERR_ARG;
    }
    if (dst_bytes < w4_packed_bytes(N, K)) {
        set_error("dst_bytes %zu < %zu", dst_bytes, w4_packed_bytes(N, K));
        return W4_ERR_ARG;
    }
    if (!q_in_range(q, (size_t)(N * K))) {
        set_error("q outside [-8, 7]");
        return W4_ERR_RANGE;
    }
    pack_host_impl(q, scales, N, K, static_cast<uint8_t*>(dst));
    return W4_OK;
}

extern "C" w4_status w4_unpack_host(const void* packed, int64_t N, int64_t K, int8_t* q, uint16_t* scales) {
    clear_error();
    w4_status st = check_shape(N, K);
    if (st != W4_OK) return st;
    if (!packed || !q || !scales) {
        set_error("NULL argument");
        return W4_ERR_ARG;
    }
    unpack_host_impl(static_cast<const uint8_t*>(packed), N, K, q, scales);
    return W4_OK;
}

static w4_status pack_impl(const int8_t* q, const uint16_t* scales, int64_t N, int64_t K, void* dst_dev,
                           size_t dst_bytes, int src_on_device, void* stream, w4_weight* out, int64_t glu_I) {
    w4_status st = check_shape(N, K);
    if (st != W4_OK) return st;
    if (!q || !scales || !dst_dev || (src_on_device != 0 && src_on_device != 1)) {
        set_error("NULL argument or bad src_on_device flag");
        return W4_ERR_ARG;
    }
    if (!aligned16(dst_dev)) {
        set_error("dst_dev not 16-byte aligned");
        return W4_ERR_ALIGN;
    }
    const size_t need = w4_packed_bytes(N, K);
    if (dst_bytes < need) {
        set_error("dst_bytes %zu < %zu", dst_bytes, need);
        return W4_ERR_ARG;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!src_on_device) {
        if (!q_in_range(q, (size_t)(N * K))) {
            set_error("q outside [-8, 7]");
            return W4_ERR_RANGE;
        }
        std::vector<uint8_t> host(need);
        pack_host_impl(q, scales, N, K, host.data(), glu_I);
        W4_CUDA_TRY(cudaMemcpyAsync(dst_dev, host.data(), need, cudaMemcpyHostToDevice, s));
        W4_CUDA_TRY(cudaStreamSynchronize(s));
    } else {
        unsigned* bad = nullptr;
        W4_CUDA_TRY(cudaMalloc(&bad, sizeof(unsigned)));
        unsigned h_bad = 0;
        cudaError_t e = cudaMemsetAsync(bad, 0, sizeof(unsigned), s);
        const int64_t tiles = num_bands(N) * num_groups(K);
        if (e == cudaSuccess) {
            pack_kernel<<<(unsigned)tiles, 256, 0, s>>>(q, scales, N, K, static_cast<uint8_t*>(dst_dev), bad, glu_I);
            e = cudaGetLastError();
        }
        if (e == cudaSuccess) e = cudaMemcpyAsync(&h_bad, bad, sizeof(unsigned), cudaMemcpyDeviceToHost, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        cudaFree(bad);
        if (e != cudaSuccess) return cuda_fail(e, "device pack");
        if (h_bad) {
            set_error("q outside [-8, 7]");
            return W4_ERR_RANGE;
        }
    }
    if (out) {
        out->data = dst_dev;
        out->N = N;
        out->K = K;
        out->magic = W4_PACK_MAGIC;
        out->version = W4_PACK_VERSION;
    }
    return W4_OK;
}

extern "C" w4_status w4_pack(const int8_t* q, const uint16_t* scales, int64_t N, int64_t K, void* dst_dev,
                             size_t dst_bytes, int src_on_device, void* stream, w4_weight* out) {
    clear_error();
    return pack_impl(q, scales, N, K, dst_dev, dst_bytes, src_on_device, stream, out, 0);
}

extern "C" w4_status w4_pack_glu(const int8_t* q, const uint16_t* scales, int64_t I, int64_t K, void* dst_dev,
                                 size_t dst_bytes, int src_on_device, void* stream, w4_weight* out) {
    clear_error();
    if (I < 8 || I % 8 != 0) {
        set_error("gated weight: I=%lld rows per half must be a positive multiple of 8", (long long)I);
        return W4_ERR_SHAPE;
    }
    return pack_impl(q, scales, 2 * I, K, dst_dev, dst_bytes, src_on_device, stream, out, I);
}

extern "C" w4_status w4_unpack(const w4_weight* w, int8_t* q, uint16_t* scales, int dst_on_device, void* stream) {
    clear_error();
    w4_status st = check_weight(w);
    if (st != W4_OK) return st;
    if (!q || !scales || (dst_on_device != 0 && dst_on_device != 1)) {
        set_error("NULL argument or bad dst_on_device flag");
        return W4_ERR_ARG;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t bytes = w4_packed_bytes(w->N, w->K);
    if (dst_on_device) {
        const int64_t tiles = num_bands(w->N) * num_groups(w->K);
        unpack_kernel<<<(unsigned)tiles, 256, 0, s>>>(static_cast<const uint8_t*>(w->data), w->N, w->K, q, scales);
        W4_CUDA_TRY(cudaGetLastError());
        W4_CUDA_TRY(cudaStreamSynchronize(s));
    } else {
        std::vector<uint8_t> host(bytes);
        W4_CUDA_TRY(cudaMemcpyAsync(host.data(), w->data, bytes, cudaMemcpyDeviceToHost, s));
        W4_CUDA_TRY(cudaStreamSynchronize(s));
        unpack_host_impl(host.data(), w->N, w->K, q, scales);
    }
    return W4_OK;
}
