// Persistent decode-step kernel: the whole chain of projections of a decode
// step (28 layers x qkv, o, gate_up, down) in one cooperative launch.
//
// Why: the pages' runtime reached its decode speed by capturing the step in
// a CUDA graph ("Building a Custom LLM Inference Runtime ...", "The Impact of
// CUDA Graphs").  On GB300 each separate projection kernel still pays a ramp
// up (first bytes in flight), a drain (the last CTA) and a grid completion at
// every boundary; over 112 projections of 1 to 10 microseconds of streaming
// that is most of the step.  Here one persistent grid (two CTAs per SM)
// streams the weights of every projection back to back:
//
//  * The producer lane of each CTA walks the projections in order and streams
//    the tiles of its work blocks into a shared-memory ring (cp.async.bulk,
//    8 tiles per slot) without ever waiting on the dependency chain: weights
//    do not depend on activations, so the ring fills with the next
//    projection's weights while the consumers finish the current one.
//  * Consumers of projection i wait until every CTA has finished projection
//    i - 1 (a completion counter in the workspace, read with acquire
//    semantics), then stage x_i and compute exactly as the single-projection
//    kernel does (same tile arithmetic, same fixed-order block reduction).
//    This honours the data dependency of a real decode step, where x_i is
//    computed from y_(i-1).
//  * A K split (when a projection has too few bands to balance) writes FP32
//    block partials to the workspace; the CTA whose arrival completes a block
//    adds the partials in split order (deterministic) and writes y.
//  * Counters reset themselves (the last arriver of a block, the last CTA of
//    the step), so the launch can be replayed from a graph.
//  * Every wait is bounded (about a second); a timeout sets the status word
//    and the CTA moves on instead of hanging.
#include <cooperative_groups.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "decode_common.cuh"
#include "step_launch.h"

namespace w4 {

struct StepOp {
    const uint8_t* w;
    const uint32_t* x;
    uint16_t* y;
    float* part;    // K split: partials [nblocks][S][BB*16*M]
    unsigned* cnt;  // K split: arrivals per block
    int N, K, G, bands;
    int S, BB, nblocks;
    int pad;
};

namespace {

constexpr int kWarps = 16;              // consumer warps
constexpr int kCons = kWarps * 32;      // consumer threads
constexpr int kSlot = kWarps;           // tiles per ring slot: one per consumer warp
constexpr int kThreads = kCons + 32;    // + one producer warp
constexpr int kQueue = 32;              // block-queue entries
constexpr int kSmemBudget = 225 * 1024; // one CTA per SM

struct StepSmem {
    int ring, nslots, bar, queue, flag, x, xsum, red, total;
    __host__ __device__ StepSmem(int ring_tiles, int MP, int gpc_max, int bb_max) {
        ring = ring_tiles;
        nslots = ring_tiles / kSlot;
        bar = ring_tiles * kTileBytes;                        // ring of 16-tile slots first
        queue = bar + (2 * nslots + 2 * kQueue) * 8;          // full/empty per slot, queue full/empty
        flag = queue + kQueue * 4;
        x = (flag + 16 + 127) & ~127;
        xsum = x + dec::x_bytes(MP, gpc_max);
        red = xsum + dec::xsum_bytes(gpc_max);
        total = red + 2 * dec::red_floats(bb_max, (MP + 7) / 8, kWarps) * 4;
    }
};

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// The share of projection `o` that CTA c takes without contention: blocks
// g, g + cps, ... (g = c / S) up to floor(nblocks / cps) of them; the rest are
// handed out by the per-split counter.
__device__ __forceinline__ int static_blocks(const StepOp& o, int cps) { return o.nblocks / cps; }

template <int MP>
__global__ void __launch_bounds__(kThreads, 1) step_kernel(StepParams p) {
    constexpr int NT = (MP + 7) / 8;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NC = gridDim.x, c = blockIdx.x;
    const int M = p.M;
    const StepSmem L(p.ring, MP, p.gpc_max, p.bb_max);
    const int nslots = L.nslots;
    const uint32_t sbase = tc::smem_addr(smem);
    const uint32_t full0 = sbase + L.bar, empty0 = full0 + 8 * nslots, qfull0 = empty0 + 8 * nslots,
                   qempty0 = qfull0 + 8 * kQueue;
    volatile int* queue = reinterpret_cast<volatile int*>(smem + L.queue);
    volatile int* flag = reinterpret_cast<volatile int*>(smem + L.flag);

    if (threadIdx.x == 0) {
        for (int s = 0; s < nslots; ++s) {
            tc::mbar_init(full0 + 8 * s, 1);
            tc::mbar_init(empty0 + 8 * s, kWarps);
        }
        for (int q = 0; q < kQueue; ++q) {
            tc::mbar_init(qfull0 + 8 * q, 1);
            tc::mbar_init(qempty0 + 8 * q, 1);
        }
        tc::mbar_init_fence();
    }
    __syncthreads();

    if (warp == kWarps) {
        // ---- producer: pick blocks, publish them, stream their tiles ---------------
        if (lane == 0) {
            int slot = 0, qs = 0;
            uint32_t use = 0, quse = 0, issued = 0;
            bool ok = true;
            for (int i = 0; i < p.nops && ok; ++i) {
                const StepOp o = p.ops[i];
                const int r = c % o.S, cps = NC / o.S, g = c / o.S;
                const int g_lo = (int)(((long long)o.G * r) / o.S);
                const int Gs = (int)(((long long)o.G * (r + 1)) / o.S) - g_lo;
                const int nstatic = static_blocks(o, cps);
                for (int k = 0; ok; ++k) {
                    int blk = k < nstatic ? g + k * cps
                                          : nstatic * cps + (int)atomicAdd(p.sched + i * 8 + r, 1u);
                    if (blk >= o.nblocks) blk = -1;
                    if (quse > 0 && !tc::mbar_wait(qempty0 + 8 * qs, (quse - 1) & 1)) {
                        atomicOr(p.status, 1);
                        ok = false;
                        break;
                    }
                    queue[qs] = blk;
                    tc::mbar_arrive(qfull0 + 8 * qs);  // release: the entry is visible to the waiters
                    if (++qs == kQueue) {
                        qs = 0;
                        ++quse;
                    }
                    if (blk < 0) break;
                    const int band0 = blk * o.BB;
                    const int T = min(o.BB, o.bands - band0) * Gs;
                    int bb = 0, gl = 0;
                    for (int t0 = 0; t0 < T; t0 += kSlot) {
                        if (use > 0 && !tc::mbar_wait(empty0 + 8 * slot, (use - 1) & 1)) {
                            atomicOr(p.status, 1);
                            ok = false;
                            break;
                        }
                        const int n = min(kSlot, T - t0);
                        const uint32_t bar = full0 + 8 * slot;
                        tc::mbar_arrive_expect_tx(bar, (uint32_t)n * kTileBytes);
                        uint32_t dst = sbase + (uint32_t)slot * (kSlot * kTileBytes);
                        for (int left = n; left > 0;) {
                            const int run = min(left, Gs - gl);
                            const uint8_t* src = o.w + ((size_t)(band0 + bb) * o.G + g_lo + gl) * kTileBytes;
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
            }
            for (uint32_t k = 0; k < (uint32_t)nslots && k < issued; ++k) {
                const uint32_t cc = issued - 1 - k;
                tc::mbar_wait(full0 + 8 * (cc % nslots), (cc / nslots) & 1);
            }
        }
        __syncwarp();
    } else {
        // ---- consumers ----------------------------------------------------------------
        int slot = 0, qs = 0;
        uint32_t use = 0, quse = 0;
        int kblk = 0;
        bool ok = true;
        uint32_t* xs = reinterpret_cast<uint32_t*>(smem + L.x);
        float* xsum = reinterpret_cast<float*>(smem + L.xsum);
        float* red_base = reinterpret_cast<float*>(smem + L.red);
        for (int i = 0; i < p.nops; ++i) {
            const StepOp o = p.ops[i];
            const int r = c % o.S;
            const int g_lo = (int)(((long long)o.G * r) / o.S);
            const int Gs = (int)(((long long)o.G * (r + 1)) / o.S) - g_lo;
            const int BB = o.BB;
            if (i > 0) {
                // x_i may be computed from y_(i-1): wait until every CTA is done with it
                if (threadIdx.x == 0) {
                    const long long t0 = clock64();
                    while (ld_acquire(p.done + (i - 1)) < (unsigned)NC) {
                        if (clock64() - t0 > (1ll << 31)) {
                            atomicOr(p.status, 2);
                            break;
                        }
                    }
                }
                tc::named_barrier(1, kCons);
            }
            dec::stage_x_async<MP, kCons>(o.x, M, o.K, g_lo, Gs, xs, xsum);
            dec::TileMac<MP> mac(sbase + L.x, sbase + L.xsum, lane);
            const int red_buf = dec::red_floats(BB, NT, kWarps);

            while (true) {
                if (!tc::mbar_wait(qfull0 + 8 * qs, quse & 1)) {
                    atomicOr(p.status, 8);
                    ok = false;
                }
                const int blk = ok ? queue[qs] : -1;
                if (blk < 0) {
                    tc::named_barrier(1, kCons);  // everyone has read the entry
                    if (threadIdx.x == 0) tc::mbar_arrive(qempty0 + 8 * qs);
                    if (++qs == kQueue) {
                        qs = 0;
                        ++quse;
                    }
                    break;
                }
                const int band0 = blk * BB;
                const int nb = min(BB, o.bands - band0);
                const int T = nb * Gs;
                const bool blk_ok0 = ok;
                float* red = red_base + (kblk & 1) * red_buf;
                float4* myred = reinterpret_cast<float4*>(red) + warp * BB * NT * 32 + lane;
                for (int q = 0; q < BB * NT; ++q) myred[q * 32] = make_float4(0.f, 0.f, 0.f, 0.f);
                float acc[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
                int cur_bb = 0, band_end = Gs;
                for (int t0 = 0; t0 < T; t0 += kSlot) {
                    if (ok && !tc::mbar_wait(full0 + 8 * slot, use & 1)) {
                        atomicOr(p.status, 4);
                        ok = false;
                    }
                    const int t = t0 + warp;
                    if (ok && t < T) {
                        while (t >= band_end) {
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
                                myred[(cur_bb * NT + nt) * 32] =
                                    make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                                for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
                            ++cur_bb;
                            band_end += Gs;
                        }
                        mac.run(sbase + (uint32_t)slot * (kSlot * kTileBytes) + (uint32_t)warp * kTileBytes,
                                t - cur_bb * Gs, lane, acc);
                    }
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
                tc::named_barrier(1, kCons);
                // every consumer has read this block's queue entry: free it
                if (threadIdx.x == 0) tc::mbar_arrive(qempty0 + 8 * qs);
                if (++qs == kQueue) {
                    qs = 0;
                    ++quse;
                }
                const int Tout = nb * 16 * M;
                float v[4];
                dec::block_sums<NT, kCons>(red, BB, nb, M, blk_ok0 && ok, v);
                if (o.S == 1) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int t = threadIdx.x + q * kCons;
                        if (t < Tout) {
                            const int m = t / (nb * 16), rl = t - m * (nb * 16);
                            const int n = band0 * 16 + rl;
                            if (n < o.N) o.y[(size_t)m * o.N + n] = __half_as_ushort(__float2half_rn(v[q]));
                        }
                    }
                } else {
                    // K split: publish this split's partial; the last arrival adds all
                    // splits in order and writes y
                    const int pb = BB * 16 * M;
                    float* mine = o.part + ((size_t)blk * o.S + r) * pb;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int t = threadIdx.x + q * kCons;
                        if (t < Tout) mine[t] = v[q];
                    }
                    __threadfence();
                    tc::named_barrier(1, kCons);
                    if (threadIdx.x == 0) *flag = (atomicAdd(o.cnt + blk, 1u) == (unsigned)(o.S - 1));
                    tc::named_barrier(1, kCons);
                    if (*flag) {
                        __threadfence();
                        const float* base = o.part + (size_t)blk * o.S * pb;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int t = threadIdx.x + q * kCons;
                            if (t < Tout) {
                                float sum = 0.f;
                                for (int s2 = 0; s2 < o.S; ++s2) sum += __ldcg(base + (size_t)s2 * pb + t);
                                const int m = t / (nb * 16), rl = t - m * (nb * 16);
                                const int n = band0 * 16 + rl;
                                if (n < o.N) o.y[(size_t)m * o.N + n] = __half_as_ushort(__float2half_rn(sum));
                            }
                        }
                        if (threadIdx.x == 0) o.cnt[blk] = 0;  // ready for the next step
                    }
                }
                ++kblk;
            }
            // this CTA is done with projection i: its y (and partials) are visible
            __threadfence();
            tc::named_barrier(1, kCons);
            if (threadIdx.x == 0) atomicAdd(p.done + i, 1u);
        }
        // the last CTA out resets the counters for the next step
        if (threadIdx.x == 0) {
            __threadfence();
            if (atomicAdd(p.exit_cnt, 1u) == (unsigned)(NC - 1)) {
                for (int i = 0; i < p.nops; ++i) p.done[i] = 0;
                for (int i = 0; i < 8 * p.nops; ++i) p.sched[i] = 0;
                *p.exit_cnt = 0;
                __threadfence();
            }
        }
    }
}

StepFn step_fn(int MP) {
    switch (MP) {
        case 1: return step_kernel<1>;
        case 2: return step_kernel<2>;
        case 4: return step_kernel<4>;
        case 8: return step_kernel<8>;
        default: return step_kernel<16>;
    }
}

int padded(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : 16; }

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

}  // namespace

// ---- host-side plan ---------------------------------------------------------------
struct StepPlan {
    int MP = 1, NC = 0, gpc_max = 1, bb_max = 1, ring = 0, smem = 0;
    std::vector<StepOp> ops;  // device pointers filled against a workspace base
    size_t table_off = 0, done_off = 0, exit_off = 0, status_off = 0, sched_off = 0, total = 0;
    std::vector<size_t> cnt_off, part_off;
};

// Per projection: one band per block (the block queue balances the tail) and
// the smallest K split (dividing NC) whose x slice fits 48 KB; the ring takes
// the rest of the shared memory.  Lays out the workspace.
static void plan_step(const w4_weight* w, int n, int M, int NC, StepPlan* pl) {
    pl->MP = padded(M);
    pl->NC = NC;
    pl->ops.assign(n, StepOp{});
    pl->cnt_off.assign(n, 0);
    pl->part_off.assign(n, 0);
    std::vector<int> S_of(n);
    for (int i = 0; i < n; ++i) {
        const int G = (int)(w[i].K / kGroupK);
        int S = 1;
        while (S < 8 && 2 * S <= G && NC % (2 * S) == 0 &&
               dec::x_bytes(pl->MP, (G + S - 1) / S) + dec::xsum_bytes((G + S - 1) / S) > 48 * 1024)
            S *= 2;
        S_of[i] = S;
        pl->gpc_max = std::max(pl->gpc_max, (G + S - 1) / S);
    }
    pl->bb_max = 1;
    int ring = 192;
    while (ring > kSlot && StepSmem(ring, pl->MP, pl->gpc_max, pl->bb_max).total > kSmemBudget) ring -= kSlot;
    pl->ring = ring;
    pl->smem = StepSmem(ring, pl->MP, pl->gpc_max, pl->bb_max).total;
    size_t off = 0;
    pl->table_off = off;
    off = align_up(off + sizeof(StepOp) * n);
    pl->done_off = off;
    off = align_up(off + sizeof(unsigned) * n);
    pl->sched_off = off;
    off = align_up(off + sizeof(unsigned) * 8 * n);
    pl->exit_off = off;
    pl->status_off = off + 16;
    off = align_up(off + 32);
    for (int i = 0; i < n; ++i) {
        StepOp& o = pl->ops[i];
        o.N = (int)w[i].N;
        o.K = (int)w[i].K;
        o.G = (int)(w[i].K / kGroupK);
        o.bands = (int)num_bands(w[i].N);
        o.S = S_of[i];
        o.BB = 1;
        o.nblocks = o.bands;
        if (o.S > 1) {
            pl->cnt_off[i] = off;
            off = align_up(off + sizeof(unsigned) * o.nblocks);
            pl->part_off[i] = off;
            off = align_up(off + sizeof(float) * (size_t)o.nblocks * o.S * o.BB * 16 * M);
        }
    }
    pl->total = off;
}

static int sm_count_now() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        return 152;
    return sms;
}

// One resident CTA per SM, or 0 if the kernel cannot be resident.
static int step_grid(int MP, int smem) {
    int per_sm = 0;
    StepFn fn = step_fn(MP);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, smem) != cudaSuccess) return 0;
    return per_sm >= 1 ? sm_count_now() : 0;
}

size_t step_workspace_bytes(const w4_weight* w, int n, int M) {
    StepPlan pl;
    plan_step(w, n, M, sm_count_now(), &pl);
    return pl.total;
}

w4_status step_prepare(const w4_weight* w, const void* const* x, void* const* y, int n, int M, void* ws,
                       size_t ws_bytes, cudaStream_t stream, StepLaunch* out) {
    const int MP = padded(M);
    StepPlan pl;
    plan_step(w, n, M, sm_count_now(), &pl);
    const int NC = step_grid(MP, pl.smem);
    if (NC <= 0 || NC != pl.NC || pl.ring < 2 * kSlot) {
        set_error("the persistent step kernel cannot be resident (shared memory %d bytes, ring %d tiles)",
                  pl.smem, pl.ring);
        return W4_ERR_UNSUPPORTED;
    }
    if (!ws || ws_bytes < pl.total) {
        set_error("step workspace of %zu bytes needed (got %zu)", pl.total, ws_bytes);
        return W4_ERR_WORKSPACE;
    }
    if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) {
        set_error("step workspace must be 256-byte aligned");
        return W4_ERR_ALIGN;
    }
    char* base = static_cast<char*>(ws);
    for (int i = 0; i < n; ++i) {
        StepOp& o = pl.ops[i];
        o.w = static_cast<const uint8_t*>(w[i].data);
        o.x = static_cast<const uint32_t*>(x[i]);
        o.y = static_cast<uint16_t*>(y[i]);
        o.cnt = o.S > 1 ? reinterpret_cast<unsigned*>(base + pl.cnt_off[i]) : nullptr;
        o.part = o.S > 1 ? reinterpret_cast<float*>(base + pl.part_off[i]) : nullptr;
    }
    W4_CUDA_TRY(cudaMemsetAsync(ws, 0, pl.total, stream));
    W4_CUDA_TRY(cudaMemcpyAsync(base + pl.table_off, pl.ops.data(), sizeof(StepOp) * n, cudaMemcpyHostToDevice,
                                stream));
    W4_CUDA_TRY(cudaStreamSynchronize(stream));
    out->fn = step_fn(MP);
    out->NC = NC;
    out->smem = pl.smem;
    StepParams& p = out->params;
    p.ops = reinterpret_cast<const StepOp*>(base + pl.table_off);
    p.nops = n;
    p.M = M;
    p.done = reinterpret_cast<unsigned*>(base + pl.done_off);
    p.exit_cnt = reinterpret_cast<unsigned*>(base + pl.exit_off);
    p.sched = reinterpret_cast<unsigned*>(base + pl.sched_off);
    p.status = reinterpret_cast<int*>(base + pl.status_off);
    p.gpc_max = pl.gpc_max;
    p.bb_max = pl.bb_max;
    p.ring = pl.ring;
    return W4_OK;
}

int step_status(const StepLaunch& s) {
    int v = 0;
    if (cudaMemcpy(&v, s.params.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
    return v;
}

w4_status step_launch(const StepLaunch& s, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)s.NC, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);  // 16 consumer warps + the producer warp
    cfg.dynamicSmemBytes = (size_t)s.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeCooperative;
    attr.val.cooperative = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, s.fn, s.params);
    if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelEx(step)");
    return W4_OK;
}

}  // namespace w4
