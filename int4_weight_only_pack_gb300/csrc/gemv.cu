// Decode projection y[M, N] = x[M, K] . W^T for 1 <= M <= 16 on sm_103a.
//
// What it computes is the pages' W4A16 projection: symmetric INT4 weights in
// groups of 128 with one FP16 scale each, FP16 activations ("Building a Custom
// LLM Inference Runtime ...", "Technical Specifications and Hardware Alignment"
// and "The INT8 vs. FP16 Activation Trade-off", Path B).  The pages' own kernel
// is an sm_90 GEMV with prmt-based unpacking; this one is designed for GB300:
//
//  * HBM-bound streaming.  One persistent CTA per SM (a cluster of `splits`
//    CTAs when K is split).  Its producer lane streams the CTA's packed tiles,
//    in order, into a ring of shared-memory slots with 1-D bulk copies
//    (cp.async.bulk, one 1056-byte tile per slot, completion on the slot's
//    mbarrier).  The producer starts before the kernel waits on the previous
//    grid (programmatic dependent launch), so a projection's weights are in
//    flight while its predecessor drains; every CTA lets its dependents launch
//    at once, so the next projection's CTAs can do the same.
//  * Eight consumer warps take the ring's tiles round-robin.  Unpacking: one
//    32-bit word per lane and k16 step holds eight nibbles; two LOP3 masks
//    with the fp16 exponent pattern 0x6400 (and the same after a shift by 8)
//    give 1024 + u and 1024 + 16u, and one f16x2 subtract or FMA turns them
//    into q exactly: an m16n8k16 A fragment.
//  * MACs: mma.sync m16n8k16 (FP16 x FP16 products are exact, FP32
//    accumulation) per 128-wide group; the group's FP32 partial is scaled by
//    the group's FP32 scale and added in FP32.  x is the B operand (tokens
//    padded to 8 or 16), staged once per CTA in shared memory in fragment
//    order after the wait on the previous grid.
//  * Work unit: a block of `bands_per_cta` 16-row bands over the CTA's K range.
//    Per block, the warps' partials are summed in fixed order in shared
//    memory; with a K split, every non-leader CTA of the cluster stores its
//    block partial into the leader's shared memory and arrives on the leader's
//    mbarrier, and the leader adds them in rank order.  No atomics, no global
//    scratch: bit-identical results run to run.
//  * Every wait is bounded (about a second); a timeout writes NaN into the
//    block's outputs instead of hanging.
#include <cuda_fp16.h>

#include <mutex>
#include <set>
#include <utility>

#include "tc_ptx.cuh"
#include "w4_device.cuh"
#include "w4_internal.cuh"

namespace w4 {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kMaxSmem = 220 * 1024;
constexpr int kDefaultRing = 48;
constexpr int kMaxRing = 96;

// SM count of the current device (looked up once per device).
static int sm_count() {
    static std::mutex mu;
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 152;
        cache[dev] = n;
    }
    return cache[dev];
}

struct GemvParams {
    const uint32_t* x;  // fp16 pairs, [M, K/2]
    const uint8_t* w;   // packed tiles
    uint16_t* y;        // fp16 [M, N]
    int M, N, K, G, bands;
    int nblocks;        // ceil(bands / BB)
    int ring;           // ring slots
};

// Shared-memory carve-up, identical on host and device.
struct SmemLayout {
    int bar, x, red, cpart, total;
    __host__ __device__ SmemLayout(int ring, int M, int gpc, int BB, int NT, int S) {
        bar = ring * kTileBytes;                                        // ring of tile slots first
        x = (bar + (2 * ring + 4) * 8 + 15) & ~15;                      // full/empty per slot, cfull[2], cempty[2]
        red = x + M * gpc * 256;                                        // x slice in fragment order
        cpart = red + 2 * kConsumerWarps * BB * NT * 4 * 32 * 4;        // per-warp block partials, 2 buffers
        total = cpart + 2 * (S > 1 ? S - 1 : 0) * BB * 16 * M * 4;      // leader's receive buffers
    }
};

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

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

template <int NT, int BB>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(GemvParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int S = gridDim.y, rank = blockIdx.y;  // cluster (1, S, 1): rank = K split
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g_lo = (int)(((long long)p.G * rank) / S);
    const int g_hi = (int)(((long long)p.G * (rank + 1)) / S);
    const int Gs = g_hi - g_lo;
    const int gpc = (p.G + S - 1) / S;
    const int M = p.M, ring = p.ring;
    const SmemLayout L(ring, M, gpc, BB, NT, S);
    const uint32_t sbase = tc::smem_addr(smem);
    const uint32_t full0 = sbase + L.bar, empty0 = full0 + 8 * ring, cfull0 = empty0 + 8 * ring,
                   cempty0 = cfull0 + 16;

    if (threadIdx.x == 0) {
        for (int s = 0; s < ring; ++s) {
            tc::mbar_init(full0 + 8 * s, 1);
            tc::mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(cfull0 + 8 * b, S > 1 ? S - 1 : 1);
            tc::mbar_init(cempty0 + 8 * b, 1);
        }
        tc::mbar_init_fence();
    }
    __syncthreads();
    if (S > 1) tc::cluster_sync_all();  // every CTA's barriers exist before any remote access
    // The next kernel on the stream may start now: it only streams its own
    // weights until it, too, waits for this grid to finish.
    pdl_launch_dependents();

    const int P = gridDim.x;
    if (warp == kConsumerWarps) {
        // ---- producer: stream this CTA's tiles into the ring ------------------
        if (lane == 0) {
            int seq = 0;
            bool ok = true;
            for (int blk = blockIdx.x; blk < p.nblocks && ok; blk += P) {
                const int band0 = blk * BB;
                const int T = min(BB, p.bands - band0) * Gs;
                for (int t = 0; t < T; ++t, ++seq) {
                    const int slot = seq % ring, use = seq / ring;
                    if (use > 0 && !tc::mbar_wait(empty0 + 8 * slot, (use - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    const int bb = t / Gs, g = g_lo + (t - bb * Gs);
                    const uint8_t* src = p.w + ((size_t)(band0 + bb) * p.G + g) * kTileBytes;
                    tc::mbar_arrive_expect_tx(full0 + 8 * slot, kTileBytes);
                    tc::bulk_load(sbase + slot * kTileBytes, src, kTileBytes, full0 + 8 * slot);
                }
            }
            // every copy has landed before the CTA may exit
            for (int sq = seq - 1; sq >= 0 && sq >= seq - ring; --sq)
                tc::mbar_wait(full0 + 8 * (sq % ring), (sq / ring) & 1);
        }
        __syncwarp();
    } else {
        // ---- consumers -----------------------------------------------------------
        // x may be produced by the previous kernel on the stream: read it only now.
        pdl_wait();
        uint32_t* xs = reinterpret_cast<uint32_t*>(smem + L.x);
        {
            const int per_row = Gs * 64;  // fp16 pairs of this split's K range
            const uint32_t* xg = p.x + (size_t)g_lo * 64;
            const int kp = p.K / 2;
            for (int idx = threadIdx.x; idx < M * per_row; idx += kConsumers) {
                const int m = idx / per_row, r = idx - m * per_row;
                const uint32_t v = __ldcg(xg + (size_t)m * kp + r);
                // pair kk2 of the group = k 2*kk2, 2*kk2+1; lane class c owns
                // k 4c..4c+3 of each k16 step (the lower pair is b0, the upper b1)
                const int gl = r >> 6, kk2 = r & 63;
                const int j = kk2 >> 3, c = (kk2 >> 1) & 3, hi = kk2 & 1;
                xs[gl * (M * 64) + (j >> 1) * (M * 16) + (m * 4 + c) * 4 + (j & 1) * 2 + hi] = v;
            }
        }
        tc::named_barrier(1, kConsumers);

        const uint4* xs4 = reinterpret_cast<const uint4*>(smem + L.x);
        const int tok = lane >> 2, cl4 = lane & 3;
        float* red_base = reinterpret_cast<float*>(smem + L.red);
        const int red_buf = kConsumerWarps * BB * NT * 4 * 32;
        const int part_buf = (S > 1 ? S - 1 : 0) * BB * 16 * M;
        int seq = 0, kblk = 0;
        for (int blk = blockIdx.x; blk < p.nblocks; blk += P, ++kblk) {
            const int band0 = blk * BB;
            const int nb = min(BB, p.bands - band0);
            const int T = nb * Gs;
            bool ok = true;
            float acc[BB][NT][4];
#pragma unroll
            for (int bb = 0; bb < BB; ++bb)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int r = 0; r < 4; ++r) acc[bb][nt][r] = 0.f;

            for (int t = warp; t < T; t += kConsumerWarps) {
                const int sq = seq + t;
                const int slot = sq % ring;
                if (!tc::mbar_wait(full0 + 8 * slot, (sq / ring) & 1)) {
                    ok = false;
                    break;
                }
                const uint32_t ta = sbase + slot * kTileBytes;
                const uint4 lo = lds128(ta + 16 * lane), hi = lds128(ta + 512 + 16 * lane);
                const uint32_t sc = lds32(ta + kScaleOffset + 4 * (lane >> 2));
                const int bb = t / Gs, gl = t - bb * Gs;
                uint4 xb[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int m = nt * 8 + tok;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        xb[nt][q] = (m < M) ? xs4[gl * (M * 16) + q * (M * 4) + m * 4 + cl4] : make_uint4(0, 0, 0, 0);
                }
                float part[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int r = 0; r < 4; ++r) part[nt][r] = 0.f;
                const uint32_t wd[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
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
                // the tile's words are consumed: hand the slot back
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(empty0 + 8 * slot);
                const float2 sf = __half22float2(*reinterpret_cast<const __half2*>(&sc));
#pragma unroll
                for (int b2 = 0; b2 < BB; ++b2) {
                    if (b2 == bb) {
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            acc[b2][nt][0] = fmaf(sf.x, part[nt][0], acc[b2][nt][0]);
                            acc[b2][nt][1] = fmaf(sf.x, part[nt][1], acc[b2][nt][1]);
                            acc[b2][nt][2] = fmaf(sf.y, part[nt][2], acc[b2][nt][2]);
                            acc[b2][nt][3] = fmaf(sf.y, part[nt][3], acc[b2][nt][3]);
                        }
                    }
                }
            }
            seq += T;

            // ---- fixed-order reduction of the block over the warps --------------
            float* red = red_base + (kblk & 1) * red_buf;
#pragma unroll
            for (int bb = 0; bb < BB; ++bb)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int r = 0; r < 4; ++r)
                        red[(((warp * BB + bb) * NT + nt) * 4 + r) * 32 + lane] = ok ? acc[bb][nt][r] : __int_as_float(0x7FC00000);
            tc::named_barrier(1, kConsumers);
            const int Tout = nb * 16 * M;  // outputs of this block: [m][band row]
            float v[4];                    // <= 4 outputs per thread (BB * 16 * 16 <= 1024)
            int cnt = 0;
            for (int t = threadIdx.x; t < Tout; t += kConsumers, ++cnt) {
                const int m = t / (nb * 16), rl = t - m * (nb * 16);
                const int bb = rl >> 4, rr = rl & 15;
                const int nt = m >> 3, col = m & 7;
                const int ln = (rr & 7) * 4 + (col >> 1), r = (rr >> 3) * 2 + (col & 1);
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) sum += red[(((w * BB + bb) * NT + nt) * 4 + r) * 32 + ln];
                v[cnt & 3] = sum;
                if (S == 1) {
                    const int n = band0 * 16 + rl;
                    if (n < p.N) p.y[(size_t)m * p.N + n] = __half_as_ushort(__float2half_rn(sum));
                }
            }
            if (S > 1) {
                const int buf = kblk & 1;
                const uint32_t use = (uint32_t)(kblk >> 1);
                float* cpart = reinterpret_cast<float*>(smem + L.cpart) + buf * part_buf;
                if (rank != 0) {
                    // wait until the leader has read this buffer's previous contents
                    bool got = tc::mbar_wait_cluster(cempty0 + 8 * buf, (use & 1) ^ 1);
                    const uint32_t remote = tc::map_rank(tc::smem_addr(cpart), 0) + (uint32_t)(rank - 1) * BB * 16 * M * 4;
                    cnt = 0;
                    for (int t = threadIdx.x; t < Tout; t += kConsumers, ++cnt)
                        tc::st_cluster_f32(remote + 4u * t, got ? v[cnt & 3] : __int_as_float(0x7FC00000));
                    tc::fence_acq_rel_cluster();
                    tc::named_barrier(1, kConsumers);
                    if (threadIdx.x == 0) tc::mbar_arrive_remote(tc::map_rank(cfull0 + 8 * buf, 0));
                } else {
                    const bool got = tc::mbar_wait_cluster(cfull0 + 8 * buf, use & 1);
                    cnt = 0;
                    for (int t = threadIdx.x; t < Tout; t += kConsumers, ++cnt) {
                        float sum = v[cnt & 3];
                        for (int r2 = 1; r2 < S; ++r2) sum += cpart[(r2 - 1) * BB * 16 * M + t];
                        if (!got) sum = __int_as_float(0x7FC00000);
                        const int m = t / (nb * 16), rl = t - m * (nb * 16);
                        const int n = band0 * 16 + rl;
                        if (n < p.N) p.y[(size_t)m * p.N + n] = __half_as_ushort(__float2half_rn(sum));
                    }
                    tc::named_barrier(1, kConsumers);
                    if (threadIdx.x == 0)
                        for (int r2 = 1; r2 < S; ++r2) tc::mbar_arrive_remote(tc::map_rank(cempty0 + 8 * buf, r2));
                }
            }
        }
    }
    // leave no remote access pending: the leader's last arrivals land before
    // any CTA of the cluster exits
    if (S > 1) tc::cluster_sync_all();
}

// ---- host side -------------------------------------------------------------
using KernelFn = void (*)(GemvParams);

template <int NT, int BB>
static KernelFn kernel_ptr() {
    return gemv_kernel<NT, BB>;
}

static KernelFn pick_kernel(int NT, int BB) {
    if (NT == 1 && BB == 1) return kernel_ptr<1, 1>();
    if (NT == 1 && BB == 2) return kernel_ptr<1, 2>();
    if (NT == 1 && BB == 4) return kernel_ptr<1, 4>();
    if (NT == 2 && BB == 1) return kernel_ptr<2, 1>();
    if (NT == 2 && BB == 2) return kernel_ptr<2, 2>();
    if (NT == 2 && BB == 4) return kernel_ptr<2, 4>();
    return nullptr;
}

static int gemv_smem_bytes(int M, int G, int BB, int S, int ring) {
    const int NT = M <= 8 ? 1 : 2;
    return SmemLayout(ring, M, (G + S - 1) / S, BB, NT, S).total;
}

// Critical-path tiles per consumer warp of a launch shape (lower is better):
// waves of blocks over the persistent clusters x tiles per warp per block.
static double shape_cost(int64_t bands, int G, int BB, int S, int sms) {
    const int64_t nblocks = (bands + BB - 1) / BB;
    const int64_t clusters = sms / S;
    const int64_t P = nblocks < clusters ? nblocks : clusters;
    const int64_t waves = (nblocks + P - 1) / P;
    const int Gs = (G + S - 1) / S;
    return (double)waves * (double)((BB * Gs + kConsumerWarps - 1) / kConsumerWarps) * (S > 1 ? 1.05 : 1.0);
}

void default_gemv_config(int M, int64_t N, int64_t K, w4_gemv_config* c) {
    const int64_t bands = num_bands(N);
    const int G = (int)num_groups(K);
    const int sms = sm_count();
    double best = 1e30;
    c->bands_per_cta = 1;
    c->splits = 8;
    for (int S = 1; S <= 8; S *= 2) {
        if (S > G) break;
        for (int BB = 1; BB <= 4; BB *= 2) {
            if (gemv_smem_bytes(M, G, BB, S, kDefaultRing) > 128 * 1024) continue;
            const double cost = shape_cost(bands, G, BB, S, sms);
            if (cost < best - 1e-9) {
                best = cost;
                c->bands_per_cta = BB;
                c->splits = S;
            }
        }
    }
    c->depth = kDefaultRing;
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
    if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    done.insert({dev, fn});
    return W4_OK;
}

static w4_status resolve(const w4_weight* w, int M, const w4_gemv_config& c, KernelFn* fn, int* smem) {
    const int NT = M <= 8 ? 1 : 2;
    *fn = pick_kernel(NT, c.bands_per_cta);
    const int G = (int)num_groups(w->K);
    if (!*fn || c.splits < 1 || c.splits > 8 || c.splits > G || c.depth < 2 || c.depth > kMaxRing) {
        set_error("no decode kernel for M=%d bands_per_cta=%d splits=%d depth=%d", M, c.bands_per_cta, c.splits,
                  c.depth);
        return W4_ERR_UNSUPPORTED;
    }
    *smem = gemv_smem_bytes(M, G, c.bands_per_cta, c.splits, c.depth);
    if (*smem > kMaxSmem) {
        set_error("decode kernel needs %d bytes of shared memory (max %d); use more splits", *smem, kMaxSmem);
        return W4_ERR_UNSUPPORTED;
    }
    if (w->N > (int64_t)0x7FFFFFF0 || w->K > (int64_t)0x7FFFFFF0) {
        set_error("N or K too large");
        return W4_ERR_SHAPE;
    }
    return W4_OK;
}

// Validate a launch shape and prepare its kernel without launching it.
w4_status prepare_gemv(const w4_weight* w, int M, const w4_gemv_config& c) {
    KernelFn fn;
    int smem;
    w4_status st = resolve(w, M, c, &fn, &smem);
    if (st != W4_OK) return st;
    return allow_large_smem(fn);
}

// Launch with an explicit shape; every argument already validated.
w4_status launch_gemv(const void* x, const w4_weight* w, void* y, int M, const w4_gemv_config& c,
                      cudaStream_t stream) {
    KernelFn fn;
    int smem;
    w4_status st = resolve(w, M, c, &fn, &smem);
    if (st != W4_OK) return st;
    st = allow_large_smem(fn);
    if (st != W4_OK) return st;
    GemvParams p;
    p.x = static_cast<const uint32_t*>(x);
    p.w = static_cast<const uint8_t*>(w->data);
    p.y = static_cast<uint16_t*>(y);
    p.M = M;
    p.N = (int)w->N;
    p.K = (int)w->K;
    p.G = (int)num_groups(w->K);
    p.bands = (int)num_bands(w->N);
    p.nblocks = (p.bands + c.bands_per_cta - 1) / c.bands_per_cta;
    p.ring = c.depth;
    const int clusters = sm_count() / c.splits;
    const int P = p.nblocks < clusters ? p.nblocks : clusters;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)P, (unsigned)c.splits, 1);
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
