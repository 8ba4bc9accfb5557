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
//    (cp.async.bulk; a slot holds 8 consecutive tiles, copied as one or two
//    contiguous runs, completion on the slot's mbarrier).  The producer starts before the kernel waits on the previous
//    grid (programmatic dependent launch), so a projection's weights are in
//    flight while its predecessor drains; every CTA lets its dependents launch
//    at once, so the next projection's CTAs can do the same.
//  * Eight consumer warps consume every slot in order, warp w taking the
//    slot's tile w, and all eight hand the slot back.  Unpacking: one
//    32-bit word per lane and k16 step holds eight offset-binary nibbles u;
//    two masks (0x000F000F and 0x00F000F0, and the same after a shift by 8)
//    leave four f16x2 registers whose halves are u itself as exact fp16
//    subnormals, u * 2^-24 (rows r) and u * 2^-20 (rows r + 8): an m16n8k16
//    A fragment with no floating-point conversion (5 integer ops per word).
//  * MACs: mma.sync m16n8k16 (FP16 x FP16 products are exact, FP32
//    accumulation) per 128-wide group gives D = sum_k x * u * 2^-24 (2^-20);
//    the group's exact partial sum_k x * q = 2^24 * D - 8 * sum_k x (2^20
//    for rows r + 8) is scaled by the group's FP32 scale and added in FP32.
//    x is the B operand (tokens padded to 8 or 16), staged once per CTA in
//    shared memory in fragment order after the wait on the previous grid,
//    with its per-group sums sum_k x computed once at staging.
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

#include "decode_common.cuh"

namespace w4 {

using dec::kChunk;
using dec::kConsumers;
using dec::kConsumerWarps;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kMaxSmem = 220 * 1024;
constexpr int kDefaultRing = 64;
constexpr int kMaxRing = 96;

struct GemvParams {
    const uint32_t* x;  // fp16 pairs, [M, K/2]
    const uint8_t* w;   // packed tiles
    uint16_t* y;        // fp16 [M, N]
    int M, N, K, G, bands;
    int BB;             // bands per work block
    int nblocks;        // ceil(bands / BB)
    int ring;           // ring slots
    int early_trigger;  // let dependents launch at once instead of after the loads are issued
};

// Shared-memory carve-up, identical on host and device.
struct SmemLayout {
    int bar, x, xsum, red, cpart, total;
    __host__ __device__ SmemLayout(int ring, int MP, int gpc, int BB, int NT, int S, int M) {
        bar = ring * kTileBytes;                                 // ring of 8-tile slots first
        x = (bar + (2 * (ring / kChunk) + 4) * 8 + 15) & ~15;    // full/empty per slot, cfull[2], cempty[2]
        xsum = x + dec::x_bytes(MP, gpc);                        // x slice in fragment order
        red = xsum + dec::xsum_bytes(MP, gpc);                   // per group and token: sum of x
        cpart = red + 2 * dec::red_floats(BB, NT) * 4;           // per-warp block partials, 2 buffers
        total = cpart + 2 * (S > 1 ? S - 1 : 0) * BB * 16 * M * 4;  // leader's receive buffers
    }
};

// MP: token count padded to 1, 2, 4, 8 or 16 (x rows beyond M are zero).
template <int MP>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(GemvParams p) {
    constexpr int NT = (MP + 7) / 8;  // n8 token tiles of the MMA
    extern __shared__ __align__(128) uint8_t smem[];
    const int S = gridDim.y, rank = blockIdx.y;  // cluster (1, S, 1): rank = K split
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g_lo = (int)(((long long)p.G * rank) / S);
    const int g_hi = (int)(((long long)p.G * (rank + 1)) / S);
    const int Gs = g_hi - g_lo;
    const int gpc = (p.G + S - 1) / S;
    const int M = p.M, BB = p.BB, nslots = p.ring / kChunk;
    const SmemLayout L(p.ring, MP, gpc, BB, NT, S, M);
    const uint32_t sbase = tc::smem_addr(smem);
    const uint32_t full0 = sbase + L.bar, empty0 = full0 + 8 * nslots, cfull0 = empty0 + 8 * nslots,
                   cempty0 = cfull0 + 16;

    if (threadIdx.x == 0) {
        for (int s = 0; s < nslots; ++s) {
            tc::mbar_init(full0 + 8 * s, 1);
            tc::mbar_init(empty0 + 8 * s, kConsumerWarps);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(cfull0 + 8 * b, S > 1 ? S - 1 : 1);
            tc::mbar_init(cempty0 + 8 * b, 1);
        }
        tc::mbar_init_fence();
    }
    __syncthreads();
    if (S > 1) tc::cluster_sync_all();  // every CTA's barriers exist before any remote access
    if (p.early_trigger) pdl_launch_dependents();

    const int P = gridDim.x;
    if (warp == kConsumerWarps) {
        // ---- producer: stream this CTA's tiles, 8 per chunk slot -----------------
        if (lane == 0) {
            int slot = 0;
            uint32_t use = 0, issued = 0;
            bool ok = true;
            for (int blk = blockIdx.x; blk < p.nblocks && ok; blk += P) {
                const int band0 = blk * BB;
                const int T = min(BB, p.bands - band0) * Gs;
                int bb = 0, gl = 0;  // position of tile t0 within the block
                for (int t0 = 0; t0 < T; t0 += kChunk) {
                    if (use > 0 && !tc::mbar_wait(empty0 + 8 * slot, (use - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    const int n = min(kChunk, T - t0);
                    const uint32_t bar = full0 + 8 * slot;
                    tc::mbar_arrive_expect_tx(bar, (uint32_t)n * kTileBytes);
                    // copy tiles t0 .. t0+n-1 as runs that stay inside one band's K range
                    uint32_t dst = sbase + (uint32_t)slot * (kChunk * kTileBytes);
                    for (int left = n; left > 0;) {
                        const int run = min(left, Gs - gl);
                        const uint8_t* src = p.w + ((size_t)(band0 + bb) * p.G + g_lo + gl) * kTileBytes;
                        tc::bulk_load(dst, src, (uint32_t)run * kTileBytes, bar);
                        dst += run * kTileBytes;
                        left -= run;
                        gl += run;
                        if (gl == Gs) {
                            gl = 0;
                            ++bb;
                        }
                    }
                    ++issued;
                    if (++slot == nslots) {
                        slot = 0;
                        ++use;
                    }
                }
            }
            // Everything this CTA reads is in flight: the next kernel on the
            // stream may start (it streams its own weights until it, too,
            // waits for this grid to finish).
            pdl_launch_dependents();
            // every copy has landed before the CTA may exit: wait for the
            // latest phase of each slot that was filled
            for (uint32_t k = 0; k < (uint32_t)nslots && k < issued; ++k) {
                const uint32_t c = issued - 1 - k;
                tc::mbar_wait(full0 + 8 * (c % nslots), (c / nslots) & 1);
            }
        }
        __syncwarp();
    } else {
        // ---- consumers -----------------------------------------------------------
        // x may be produced by the previous kernel on the stream: read it only now.
        pdl_wait();
        dec::stage_x_async<MP, dec::kConsumers>(p.x, M, p.K, g_lo, Gs, reinterpret_cast<uint32_t*>(smem + L.x),
                                                reinterpret_cast<float*>(smem + L.xsum));
        // everything this CTA's consumers read from the previous grid is read
        pdl_launch_dependents();

        dec::TileMac<MP> mac(sbase + L.x, sbase + L.xsum, lane);
        float* red_base = reinterpret_cast<float*>(smem + L.red);
        const int red_buf = dec::red_floats(BB, NT);
        const int part_buf = (S > 1 ? S - 1 : 0) * BB * 16 * M;
        int slot = 0;
        uint32_t use = 0;
        int kblk = 0;
        bool ok = true;
        for (int blk = blockIdx.x; blk < p.nblocks; blk += P, ++kblk) {
            const int band0 = blk * BB;
            const int nb = min(BB, p.bands - band0);
            const int T = nb * Gs;
            const bool blk_ok0 = ok;
            // this warp's partial of band cur_bb; bands it has no tile of stay 0
            float* red = red_base + (kblk & 1) * red_buf;
            float4* myred = reinterpret_cast<float4*>(red) + warp * BB * NT * 32 + lane;
            for (int i = 0; i < BB * NT; ++i) myred[i * 32] = make_float4(0.f, 0.f, 0.f, 0.f);
            float acc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int r = 0; r < 4; ++r) acc[nt][r] = 0.f;
            int cur_bb = 0, band_end = Gs;

            for (int t0 = 0; t0 < T; t0 += kChunk) {
                if (ok && !tc::mbar_wait(full0 + 8 * slot, use & 1)) ok = false;
                const int t = t0 + warp;  // this warp's tile in the chunk
                if (ok && t < T) {
                    while (t >= band_end) {  // entering a new band: park the finished one
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            myred[(cur_bb * NT + nt) * 32] = make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                            for (int r = 0; r < 4; ++r) acc[nt][r] = 0.f;
                        ++cur_bb;
                        band_end += Gs;
                    }
                    mac.run(sbase + (uint32_t)slot * (kChunk * kTileBytes) + (uint32_t)warp * kTileBytes,
                            t - cur_bb * Gs, lane, acc);
                }
                // the chunk is consumed by this warp (its words are in registers
                // and used): hand the slot back
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(empty0 + 8 * slot);
                if (++slot == nslots) {
                    slot = 0;
                    ++use;
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                myred[(cur_bb * NT + nt) * 32] = make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);

            // ---- fixed-order reduction of the block over the warps --------------
            tc::named_barrier(1, kConsumers);
            const int Tout = nb * 16 * M;  // outputs of this block: [m][band row]
            float v[4];
            dec::block_sums<NT>(red, BB, nb, M, blk_ok0 && ok, v);
            if (S == 1) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int t = threadIdx.x + i * kConsumers;
                    if (t < Tout) {
                        const int m = t / (nb * 16), rl = t - m * (nb * 16);
                        const int n = band0 * 16 + rl;
                        if (n < p.N) p.y[(size_t)m * p.N + n] = __half_as_ushort(__float2half_rn(v[i]));
                    }
                }
            } else {
                const int buf = kblk & 1;
                const uint32_t cuse = (uint32_t)(kblk >> 1);
                float* cpart = reinterpret_cast<float*>(smem + L.cpart) + buf * part_buf;
                if (rank != 0) {
                    // wait until the leader has read this buffer's previous contents
                    const bool got = tc::mbar_wait_cluster(cempty0 + 8 * buf, (cuse & 1) ^ 1);
                    const uint32_t remote =
                        tc::map_rank(tc::smem_addr(cpart), 0) + (uint32_t)(rank - 1) * BB * 16 * M * 4;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int t = threadIdx.x + i * kConsumers;
                        if (t < Tout) tc::st_cluster_f32(remote + 4u * t, got ? v[i] : __int_as_float(0x7FC00000));
                    }
                    tc::fence_acq_rel_cluster();
                    tc::named_barrier(1, kConsumers);
                    if (threadIdx.x == 0) tc::mbar_arrive_remote(tc::map_rank(cfull0 + 8 * buf, 0));
                } else {
                    const bool got = tc::mbar_wait_cluster(cfull0 + 8 * buf, cuse & 1);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int t = threadIdx.x + i * kConsumers;
                        if (t < Tout) {
                            float sum = v[i];
                            for (int r2 = 1; r2 < S; ++r2) sum += cpart[(r2 - 1) * BB * 16 * M + t];
                            if (!got) sum = __int_as_float(0x7FC00000);
                            const int m = t / (nb * 16), rl = t - m * (nb * 16);
                            const int n = band0 * 16 + rl;
                            if (n < p.N) p.y[(size_t)m * p.N + n] = __half_as_ushort(__float2half_rn(sum));
                        }
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

static int padded_tokens(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : 16; }

static KernelFn pick_kernel(int M) {
    switch (padded_tokens(M)) {
        case 1: return gemv_kernel<1>;
        case 2: return gemv_kernel<2>;
        case 4: return gemv_kernel<4>;
        case 8: return gemv_kernel<8>;
        default: return gemv_kernel<16>;
    }
}

static int gemv_smem_bytes(int M, int G, int BB, int S, int ring) {
    const int MP = padded_tokens(M);
    return SmemLayout(ring, MP, (G + S - 1) / S, BB, (MP + 7) / 8, S, M).total;
}

// Critical-path tiles per consumer warp of a launch shape (lower is better):
// waves of blocks over the persistent clusters x tiles per warp per block.
static double shape_cost(int64_t bands, int G, int BB, int S, int slots) {
    const int64_t nblocks = (bands + BB - 1) / BB;
    const int64_t clusters = slots / S;
    const int64_t P = nblocks < clusters ? nblocks : clusters;
    const int64_t waves = (nblocks + P - 1) / P;
    const int Gs = (G + S - 1) / S;
    return (double)waves * (double)((BB * Gs + kConsumerWarps - 1) / kConsumerWarps) * (S > 1 ? 1.05 : 1.0);
}

// Launch shapes measured best on GB300 (sweeps over bands per CTA, splits,
// ring depth and CTAs per SM) for the Qwen2.5-7B projection shapes, at one
// token and at 9-16 tokens.
struct TunedShape {
    int64_t N, K;
    int m_lo, m_hi;
    w4_gemv_config c;  // bands_per_cta, splits, depth, pdl, ctas_per_sm
};
static const TunedShape kTuned[] = {
    {4608, 3584, 1, 1, {2, 1, 48, 1, 2}},   {3584, 3584, 1, 1, {2, 1, 48, 1, 1}},
    {37888, 3584, 1, 1, {4, 1, 64, 1, 2}},  {3584, 18944, 1, 1, {4, 4, 48, 1, 2}},
    {4608, 3584, 9, 16, {4, 2, 64, 1, 1}},  {3584, 3584, 9, 16, {2, 4, 32, 1, 1}},
    {37888, 3584, 9, 16, {4, 2, 48, 1, 1}}, {3584, 18944, 9, 16, {2, 8, 64, 1, 1}},
};

void default_gemv_config(int M, int64_t N, int64_t K, w4_gemv_config* c) {
    const int64_t bands = num_bands(N);
    const int G = (int)num_groups(K);
    const int sms = device_sm_count();
    for (const TunedShape& t : kTuned)
        if (t.N == N && t.K == K && M >= t.m_lo && M <= t.m_hi &&
            gemv_smem_bytes(M, G, t.c.bands_per_cta, t.c.splits, t.c.depth) <=
                (t.c.ctas_per_sm == 2 ? 110 * 1024 : kMaxSmem)) {
            *c = t.c;
            return;
        }
    double best = 1e30;
    c->bands_per_cta = 1;
    c->splits = 8;
    for (int S = 1; S <= 8; S *= 2) {
        if (S > G) break;
        for (int BB = 1; BB <= 4; BB *= 2) {
            if (gemv_smem_bytes(M, G, BB, S, kDefaultRing) > 110 * 1024) continue;  // two CTAs per SM
            const double cost = shape_cost(bands, G, BB, S, 2 * sms);
            if (cost < best - 1e-9) {
                best = cost;
                c->bands_per_cta = BB;
                c->splits = S;
            }
        }
    }
    c->depth = kDefaultRing;
    c->pdl = 1;
    c->ctas_per_sm = 2;
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
    *fn = (c.bands_per_cta == 1 || c.bands_per_cta == 2 || c.bands_per_cta == 4) ? pick_kernel(M) : nullptr;
    const int G = (int)num_groups(w->K);
    if (!*fn || c.splits < 1 || c.splits > 8 || c.splits > G || c.depth < kChunk || c.depth > kMaxRing ||
        c.depth % kChunk != 0 || c.ctas_per_sm < 1 || c.ctas_per_sm > 2) {
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
    p.BB = c.bands_per_cta;
    p.nblocks = (p.bands + c.bands_per_cta - 1) / c.bands_per_cta;
    p.ring = c.depth;
    p.early_trigger = c.pdl == 2 ? 1 : 0;
    const int clusters = c.ctas_per_sm * device_sm_count() / c.splits;
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
        if (cfg->ctas_per_sm) c.ctas_per_sm = cfg->ctas_per_sm;
    }
    return launch_gemv(x, w, y, M, c, static_cast<cudaStream_t>(stream));
}
