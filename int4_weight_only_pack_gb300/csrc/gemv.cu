// Decode projection y[M, N] = x[M, K] . W^T for 1 <= M <= 16 on sm_103a.
//
// What it computes is the pages' W4A16 projection: symmetric INT4 weights in
// groups of 128 with one FP16 scale each, FP16 activations ("Building a Custom
// LLM Inference Runtime ...", "Technical Specifications and Hardware Alignment"
// and "The INT8 vs. FP16 Activation Trade-off", Path B).  The pages' own kernel
// is an sm_90 GEMV with prmt-based unpacking; this one is designed for GB300:
//
//  * HBM-bound: every packed byte is read exactly once with 16-byte
//    non-coherent streaming loads (ld.global.nc.L1::no_allocate), and all of a
//    warp's first `D` tile groups are requested before the kernel waits on the
//    previous grid (programmatic dependent launch), so the weight stream of
//    consecutive projections overlaps.
//  * Unpacking: one 32-bit word per lane and k16-step holds eight nibbles; two
//    LOP3 masks with the fp16 exponent pattern 0x6400 (and the same after a
//    shift by 8) give 1024 + u and 1024 + 16u, and one f16x2 subtract or FMA
//    turns them into q exactly.  The four registers are an m16n8k16 A fragment.
//  * MACs: mma.sync m16n8k16 (FP16 x FP16 products are exact, FP32
//    accumulation) per 128-wide group; the group's FP32 partial is then scaled
//    by the group's FP16 scale and added in FP32.  x is the B operand, tokens
//    padded to 8 (NT = 1) or 16 (NT = 2).
//  * x is staged once per CTA in shared memory in fragment order (four 16-byte
//    LDS per lane per group, conflict-free).
//  * Reductions: fixed-order sums over the CTA's 8 warps in shared memory; when
//    K is split across a thread-block cluster, fixed-order sums over the
//    cluster's CTAs through distributed shared memory.  No atomics, no global
//    scratch: results are bit-identical run to run.
#include <cooperative_groups.h>
#include <cuda_fp16.h>

#include <mutex>
#include <set>
#include <utility>

#include "w4_device.cuh"
#include "w4_internal.cuh"

namespace cg = cooperative_groups;

namespace w4 {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxSmem = 200 * 1024;

struct GemvParams {
    const uint32_t* x;  // fp16 pairs, [M, K/2]
    const uint8_t* w;   // packed tiles
    uint16_t* y;        // fp16 [M, N]
    int M, N, K, G, bands;
};

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Shared memory: x slice in fragment order, then the per-warp partials, then
// the CTA partial read by the cluster.
__host__ __device__ inline int smem_x_bytes(int M, int gpc) { return M * gpc * 256; }
__host__ __device__ inline int smem_red_bytes(int BB, int NT) { return kWarps * BB * NT * 4 * 32 * 4; }
__host__ __device__ inline int smem_part_bytes(int BB, int M) { return BB * 16 * M * 4; }

template <int NT, int BB, int D>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(GemvParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = gridDim.y, split = blockIdx.y;
    const int g_lo = (int)(((long long)p.G * split) / S);
    const int g_hi = (int)(((long long)p.G * (split + 1)) / S);
    const int ng = g_hi - g_lo;
    const int gpc = (p.G + S - 1) / S;
    const int my_n = (ng - warp + kWarps - 1) / kWarps;  // my groups: warp, warp + 8, ...
    const int band0 = blockIdx.x * BB;
    const int M = p.M;

    const uint8_t* tile0[BB];
    bool bvalid[BB];
#pragma unroll
    for (int bb = 0; bb < BB; ++bb) {
        bvalid[bb] = band0 + bb < p.bands;
        tile0[bb] = p.w + ((size_t)(band0 + bb) * p.G + g_lo + warp) * kTileBytes;
    }
    const size_t step = (size_t)kWarps * kTileBytes;

    uint4 wlo[D][BB], whi[D][BB];
    uint32_t wsc[D][BB];
#pragma unroll
    for (int d = 0; d < D; ++d) {
#pragma unroll
        for (int bb = 0; bb < BB; ++bb) {
            wlo[d][bb] = make_uint4(0, 0, 0, 0);
            whi[d][bb] = make_uint4(0, 0, 0, 0);
            wsc[d][bb] = 0;
            if (d < my_n && bvalid[bb]) {
                const uint8_t* t = tile0[bb] + d * step;
                wlo[d][bb] = ld_stream16(t + 16 * lane);
                whi[d][bb] = ld_stream16(t + 512 + 16 * lane);
                wsc[d][bb] = ld_stream4(t + kScaleOffset + 4 * (lane >> 2));
            }
        }
    }

    // x may be produced by the previous kernel on the stream: read it only now.
    pdl_wait();
    pdl_launch_dependents();

    uint32_t* xs = reinterpret_cast<uint32_t*>(smem);
    {
        const int per_row = ng * 64;  // fp16 pairs of this split's K range
        const uint32_t* xg = p.x + (size_t)g_lo * 64;
        const int kp = p.K / 2;
        for (int idx = threadIdx.x; idx < M * per_row; idx += kThreads) {
            const int m = idx / per_row, r = idx - m * per_row;
            const uint32_t v = __ldcg(xg + (size_t)m * kp + r);
            // pair kk2 of the group = k 2*kk2, 2*kk2+1; lane class c owns
            // k 4c..4c+3 of each k16 step (the lower pair is b0, the upper b1)
            const int gl = r >> 6, kk2 = r & 63;
            const int j = kk2 >> 3, c = (kk2 >> 1) & 3, hi = kk2 & 1;
            xs[gl * (M * 64) + (j >> 1) * (M * 16) + (m * 4 + c) * 4 + (j & 1) * 2 + hi] = v;
        }
    }
    __syncthreads();

    float acc[BB][NT][4];
#pragma unroll
    for (int bb = 0; bb < BB; ++bb)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[bb][nt][r] = 0.f;

    const uint4* xs4 = reinterpret_cast<const uint4*>(smem);
    const int tok = lane >> 2, cl4 = lane & 3;

    for (int i0 = 0; i0 < my_n; i0 += D) {
#pragma unroll
        for (int d = 0; d < D; ++d) {
            const int i = i0 + d;
            if (i < my_n) {
                const int gl = warp + kWarps * i;
                uint4 xb[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int m = nt * 8 + tok;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        xb[nt][q] = (m < M) ? xs4[gl * (M * 16) + q * (M * 4) + m * 4 + cl4] : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int bb = 0; bb < BB; ++bb) {
                    float part[NT][4];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int r = 0; r < 4; ++r) part[nt][r] = 0.f;
                    const uint32_t wd[8] = {wlo[d][bb].x, wlo[d][bb].y, wlo[d][bb].z, wlo[d][bb].w,
                                            whi[d][bb].x, whi[d][bb].y, whi[d][bb].z, whi[d][bb].w};
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint32_t a[4];
                        unpack_word(wd[j], a);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const uint4& v = xb[nt][j >> 1];
                            mma16816(part[nt], a, (j & 1) ? v.z : v.x, (j & 1) ? v.w : v.y);
                        }
                    }
                    const float2 sf = __half22float2(*reinterpret_cast<const __half2*>(&wsc[d][bb]));
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        acc[bb][nt][0] = fmaf(sf.x, part[nt][0], acc[bb][nt][0]);
                        acc[bb][nt][1] = fmaf(sf.x, part[nt][1], acc[bb][nt][1]);
                        acc[bb][nt][2] = fmaf(sf.y, part[nt][2], acc[bb][nt][2]);
                        acc[bb][nt][3] = fmaf(sf.y, part[nt][3], acc[bb][nt][3]);
                    }
                }
                if (i + D < my_n) {
#pragma unroll
                    for (int bb = 0; bb < BB; ++bb) {
                        if (bvalid[bb]) {
                            const uint8_t* t = tile0[bb] + (size_t)(i + D) * step;
                            wlo[d][bb] = ld_stream16(t + 16 * lane);
                            whi[d][bb] = ld_stream16(t + 512 + 16 * lane);
                            wsc[d][bb] = ld_stream4(t + kScaleOffset + 4 * (lane >> 2));
                        }
                    }
                }
            }
        }
    }

    // ---- fixed-order reduction over the CTA's warps -------------------------
    float* red = reinterpret_cast<float*>(smem + smem_x_bytes(M, gpc));
#pragma unroll
    for (int bb = 0; bb < BB; ++bb)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int r = 0; r < 4; ++r) red[(((warp * BB + bb) * NT + nt) * 4 + r) * 32 + lane] = acc[bb][nt][r];
    __syncthreads();

    const int T = BB * 16 * M;  // outputs of this CTA: [m][band row]
    float* cta_part = red + kWarps * BB * NT * 4 * 32;
    for (int t = threadIdx.x; t < T; t += kThreads) {
        const int m = t / (BB * 16), rl = t - m * (BB * 16);
        const int bb = rl >> 4, rr = rl & 15;
        const int nt = m >> 3, col = m & 7;
        const int ln = (rr & 7) * 4 + (col >> 1), r = (rr >> 3) * 2 + (col & 1);
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) sum += red[(((w * BB + bb) * NT + nt) * 4 + r) * 32 + ln];
        if (S == 1) {
            const int n = (band0 + bb) * 16 + rr;
            if (n < p.N) p.y[(size_t)m * p.N + n] = __half_as_ushort(__float2half_rn(sum));
        } else {
            cta_part[t] = sum;
        }
    }

    // ---- fixed-order reduction over the cluster's K splits (DSMEM) ----------
    if (S > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        const int rank = (int)cluster.block_rank();
        const int t0 = T * rank / S, t1 = T * (rank + 1) / S;
        for (int t = t0 + threadIdx.x; t < t1; t += kThreads) {
            float sum = 0.f;
            for (int s = 0; s < S; ++s) sum += cluster.map_shared_rank(cta_part, s)[t];
            const int m = t / (BB * 16), rl = t - m * (BB * 16);
            const int n = (band0 + (rl >> 4)) * 16 + (rl & 15);
            if (n < p.N) p.y[(size_t)m * p.N + n] = __half_as_ushort(__float2half_rn(sum));
        }
        cluster.sync();  // keep this CTA's shared memory alive until every rank has read it
    }
}

// ---- host side -------------------------------------------------------------
using KernelFn = void (*)(GemvParams);

template <int NT, int BB, int D>
static KernelFn kernel_ptr() {
    return gemv_kernel<NT, BB, D>;
}

static KernelFn pick_kernel(int NT, int BB, int D) {
#define W4_CASE(nt, bb, d) \
    if (NT == nt && BB == bb && D == d) return kernel_ptr<nt, bb, d>();
    W4_CASE(1, 1, 1) W4_CASE(1, 1, 2) W4_CASE(1, 1, 4)
    W4_CASE(1, 2, 1) W4_CASE(1, 2, 2) W4_CASE(1, 2, 4)
    W4_CASE(1, 4, 1) W4_CASE(1, 4, 2)
    W4_CASE(2, 1, 1) W4_CASE(2, 1, 2) W4_CASE(2, 1, 4)
    W4_CASE(2, 2, 1) W4_CASE(2, 2, 2)
    W4_CASE(2, 4, 1)
#undef W4_CASE
    return nullptr;
}

static int gemv_smem_bytes(int M, int G, int BB, int S) {
    const int NT = M <= 8 ? 1 : 2;
    const int gpc = (G + S - 1) / S;
    return smem_x_bytes(M, gpc) + smem_red_bytes(BB, NT) + smem_part_bytes(BB, M);
}

void default_gemv_config(int M, int64_t N, int64_t K, w4_gemv_config* c) {
    const int64_t bands = num_bands(N);
    const int G = (int)num_groups(K);
    c->bands_per_cta = M <= 2 ? 1 : (M <= 8 ? 2 : 4);
    c->depth = c->bands_per_cta == 1 ? 4 : (c->bands_per_cta == 2 ? 2 : 1);
    const int64_t ctas = (bands + c->bands_per_cta - 1) / c->bands_per_cta;
    int S = 1;
    while (S < 8 && 2 * S <= G &&
           (gemv_smem_bytes(M, G, c->bands_per_cta, S) > 64 * 1024 || ctas * S < 228))
        S *= 2;
    c->splits = S;
    c->pdl = 1;
}

// Raise a kernel's dynamic shared-memory limit once per (device, kernel).  Not
// a stream operation, so it is done before any capture begins (sequence
// creation prepares every launch first).
static w4_status allow_large_smem(KernelFn fn) {
    static std::mutex mu;
    static std::set<std::pair<int, KernelFn>> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lock(mu);
    if (done.count({dev, fn})) return W4_OK;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    done.insert({dev, fn});
    return W4_OK;
}

// Validate a launch shape and prepare its kernel without launching it.
w4_status prepare_gemv(const w4_weight* w, int M, const w4_gemv_config& c) {
    const int NT = M <= 8 ? 1 : 2;
    KernelFn fn = pick_kernel(NT, c.bands_per_cta, c.depth);
    if (!fn) return W4_ERR_UNSUPPORTED;
    const int smem = gemv_smem_bytes(M, (int)num_groups(w->K), c.bands_per_cta, c.splits);
    if (smem > 48 * 1024 && smem <= kMaxSmem) return allow_large_smem(fn);
    return W4_OK;
}

// Launch with an explicit shape; every argument already validated.
w4_status launch_gemv(const void* x, const w4_weight* w, void* y, int M, const w4_gemv_config& c,
                      cudaStream_t stream) {
    const int NT = M <= 8 ? 1 : 2;
    KernelFn fn = pick_kernel(NT, c.bands_per_cta, c.depth);
    if (!fn || c.splits < 1 || c.splits > 8 || c.splits > w->K / kGroupK) {
        set_error("no decode kernel for M=%d bands_per_cta=%d depth=%d splits=%d", M, c.bands_per_cta, c.depth,
                  c.splits);
        return W4_ERR_UNSUPPORTED;
    }
    const int G = (int)num_groups(w->K);
    const int smem = gemv_smem_bytes(M, G, c.bands_per_cta, c.splits);
    if (smem > kMaxSmem) {
        set_error("decode kernel needs %d bytes of shared memory (max %d); use more splits", smem, kMaxSmem);
        return W4_ERR_UNSUPPORTED;
    }
    if (w->N > (int64_t)0x7FFFFFF0 || w->K > (int64_t)0x7FFFFFF0) {
        set_error("N or K too large");
        return W4_ERR_SHAPE;
    }
    if (smem > 48 * 1024) {
        w4_status st = allow_large_smem(fn);
        if (st != W4_OK) return st;
    }
    GemvParams p;
    p.x = static_cast<const uint32_t*>(x);
    p.w = static_cast<const uint8_t*>(w->data);
    p.y = static_cast<uint16_t*>(y);
    p.M = M;
    p.N = (int)w->N;
    p.K = (int)w->K;
    p.G = G;
    p.bands = (int)num_bands(w->N);

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((p.bands + c.bands_per_cta - 1) / c.bands_per_cta), (unsigned)c.splits, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (c.splits > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = 1;
        attrs[na].val.clusterDim.y = (unsigned)c.splits;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    if (c.pdl != 0) {
        attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = (unsigned)na;
    cudaError_t e = cudaLaunchKernelEx(&cfg, fn, p);
    if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelEx(decode)");
    return W4_OK;
}

w4_status check_gemv_args(const void* x, const w4_weight* w, const void* y, int M) {
    w4_status st = check_weight(w);
    if (st != W4_OK) return st;
    if (!x || !y) {
        set_error("x or y is NULL");
        return W4_ERR_ARG;
    }
    if (M < 1 || M > 16) {
        set_error("M=%d: the decode kernel takes 1 <= M <= 16", M);
        return W4_ERR_SHAPE;
    }
    if (!aligned16(x) || !aligned16(y)) {
        set_error("x or y not 16-byte aligned");
        return W4_ERR_ALIGN;
    }
    return W4_OK;
}

}  // namespace w4

using namespace w4;

extern "C" w4_status w4a16_gemv_default_config(int M, int64_t N, int64_t K, w4_gemv_config* out) {
    clear_error();
    if (!out) {
        set_error("NULL argument");
        return W4_ERR_ARG;
    }
    if (M < 1 || M > 16 || N < 1 || K < kGroupK || K % kGroupK != 0) {
        set_error("bad shape M=%d N=%lld K=%lld", M, (long long)N, (long long)K);
        return W4_ERR_SHAPE;
    }
    default_gemv_config(M, N, K, out);
    return W4_OK;
}

extern "C" w4_status w4a16_gemv(const void* x, const w4_weight* w, void* y, int M, void* workspace,
                                size_t workspace_bytes, void* stream) {
    (void)workspace;
    (void)workspace_bytes;
    clear_error();
    w4_status st = check_gemv_args(x, w, y, M);
    if (st != W4_OK) return st;
    w4_gemv_config c;
    default_gemv_config(M, w->N, w->K, &c);
    return launch_gemv(x, w, y, M, c, static_cast<cudaStream_t>(stream));
}

extern "C" w4_status w4a16_gemv_config(const void* x, const w4_weight* w, void* y, int M,
                                       const w4_gemv_config* cfg, void* stream) {
    clear_error();
    w4_status st = check_gemv_args(x, w, y, M);
    if (st != W4_OK) return st;
    w4_gemv_config c;
    default_gemv_config(M, w->N, w->K, &c);
    if (cfg) {
        if (cfg->bands_per_cta) c.bands_per_cta = cfg->bands_per_cta;
        if (cfg->splits) c.splits = cfg->splits;
        if (cfg->depth) c.depth = cfg->depth;
        if (cfg->pdl >= 0) c.pdl = cfg->pdl;
    }
    return launch_gemv(x, w, y, M, c, static_cast<cudaStream_t>(stream));
}
