// Persistent decode-step kernel: the whole chain of projections of a decode
// step (28 layers x qkv, o, gate_up, down) in one cooperative launch.
//
// Why: the pages' runtime reached its decode speed by capturing the step in
// a CUDA graph ("Building a Custom LLM Inference Runtime ...", "The Impact of
// CUDA Graphs").  On GB300 each separate projection kernel still pays a ramp
// up (first bytes in flight), a drain (the last CTA) and a grid completion at
// every boundary; over 112 projections of 1 to 10 microseconds of streaming
// that is most of the step.  Here one persistent grid (one CTA per SM)
// streams the weights of every projection back to back.
//
// Work split.  Projection i is cut into units: (16-row band, K split) pairs.
// The CTAs of K split r (c % S == r) share its bands in contiguous runs, and
// the tiles of a CTA's run (band-major, then group) are cut into 16 equal
// contiguous ranges, one per warp.  So every warp streams one contiguous run
// of tiles per projection and sums its bands in registers:
//
//  * Each warp owns a ring of R slots of up to 4 tiles in shared memory and
//    issues its own bulk copies (one cp.async.bulk and one mbarrier per slot;
//    a slot never crosses the end of a band's run of tiles).  Its copy
//    cursor walks its ranges of all projections in order and never waits on
//    the dependency chain (weights do not depend on activations), so while a
//    warp waits for projection i's input, the copies of its next tiles,
//    of projection i+1 onwards, are already in flight.  A slot is refilled
//    as soon as the warp has consumed it: no cross-warp handshake per tile.
//  * Before projection i the CTA waits until every CTA has finished
//    projection i - 1 (a completion counter, read with acquire semantics),
//    then stages x_i: x_i may be computed from y_(i-1) in a real decode step.
//  * A band whose tiles all fall in one warp's range is finished by that warp
//    straight from its accumulators.  A band cut between warps is parked in
//    shared memory by each and summed, in warp order, by one warp after a CTA
//    barrier.  A band split in K (S > 1) goes through FP32 partials in the
//    workspace; below 8 tokens the arrival that completes the band adds the
//    S partials in split order and writes y, from 8 tokens on every CTA adds
//    up an equal share of the bands once all partials are in (kOpTwoPhase).
//    Every sum has a fixed order, so results are identical from run to run.
//  * Counters reset themselves (the last arrival of a band, the last CTA of
//    the step), so the launch can be replayed from a graph.
//  * Every wait is bounded (about a second); a timeout sets the status word,
//    the warp stops issuing copies and, before it exits, waits (bounded
//    again) for the copies it still has in flight.
#include <algorithm>
#include <climits>
#include <cstring>
#include <vector>

#include "decode_common.cuh"
#include "step_launch.h"

namespace w4 {

struct StepOp {
    const uint8_t* w;
    const uint32_t* x;
    uint16_t* y;
    float* part;    // K split: partials [bands][S][16*M]
    unsigned* cnt;  // K split: arrivals per band
    int N, K, G, bands;
    int16_t S;      // K splits
    int16_t flags;  // W4_OP_* of the projection
    int cps;        // CTAs per split (grid / S)
};
static_assert(sizeof(StepOp) == 64, "one projection record");

// The kernel's only parameter: the projection table travels in the launch's
// parameter space (read through the constant cache; at most 32 KB).
struct StepArgs {
    int nops, M;
    unsigned* done;      // [nops] CTAs finished with each projection
    unsigned* exit_cnt;  // CTAs finished with the step
    int* status;         // set non-zero when a wait gives up
    int gpc_max;         // largest x slice (groups): shared-memory sizing
    int ring;            // ring slots per warp; at 16 tokens also the parked partials per warp in bits
                         // 16-31 (2, or 3 with the finishing scratch): one field keeps the table's offset
    StepOp ops[kMaxStepOps];
};
static_assert(sizeof(StepArgs) <= 32000, "kernel parameter space");

namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kSmemBudget = 227 * 1024;  // one CTA per SM
constexpr int kSlotTiles = 4;            // tiles per ring slot (one bulk copy)
constexpr int kMaxRing = 32;             // slots per warp (one mbarrier per lane at most)
constexpr int kSplitPenalty = 64;        // tiles: the cost of combining K-split partials (~2 us of streaming),
                                         // plus 4 per split
constexpr int kMaxCtaTiles = 1 << 22;    // per-CTA tiles of one projection (float division below)
// From 8 tokens on, a K-split projection is finished in two phases: every CTA
// stores its FP32 partials with plain stores and counts itself on the
// projection's counter; once all have, each CTA adds up an equal share of the
// bands (split order) and writes y.  One more grid-wide wait per projection,
// but no fence and atomic per band, and no CTA left holding the combines of
// whichever bands it happened to complete last.
constexpr int16_t kOpTwoPhase = 0x4000;  // internal flag bit of StepOp::flags
constexpr int kTwoPhaseMinMP = 8;
// x slice + its group sums: small for one or two tokens so that the rings keep
// three slots per warp; 60 KB from 3 tokens on, where a K = 3584 projection
// needs no K split up to 8 tokens and two at 16 (the partials cost far more
// than the shallower ring: the 8-token step went 1883 -> 1643 us).  Where a
// plan with this slice cannot keep two ring slots per warp (a long projection
// table, or 16 tokens with a gated projection's finishing scratch), the
// fallback budget is used instead.
__host__ __device__ constexpr int x_budget(int MP) { return MP <= 2 ? 20 * 1024 : 60 * 1024; }
__host__ __device__ constexpr int x_budget_fallback(int MP) { return MP <= 2 ? 20 * 1024 : MP <= 8 ? 60 * 1024 : 40 * 1024; }

// x slice bytes: the fragment layout up to two tokens, from four on the
// natural layout that one bulk copy per token row fills (see stage_x_bulk:
// the larger slices staged by many 8-byte copies took 2.5 us at 4 tokens;
// step 1212 -> 1190 us at 4 tokens, 1645 -> 1565 at 8, 3420 -> 3336 at 16;
// unchanged at 1, 2 us slower at 2)
__host__ __device__ constexpr bool step_x_natural(int MP) { return MP >= 4; }
__host__ __device__ constexpr int step_x_bytes(int MP, int Gs) {
    return step_x_natural(MP) ? dec::x_bytes_nat(MP, Gs) : dec::x_bytes(MP, Gs);
}

struct StepSmem {
    int R, bar, xbar, geo, x, xsum, park, total;
    __host__ __device__ StepSmem(int R_, int MP, int gpc_max, int nops, int shares, bool scaled) {
        R = R_;
        bar = kWarps * R * kSlotTiles * kTileBytes;  // rings first: warp w's at w*R*4*1056
        xbar = bar + kWarps * R * 8;                 // x staging (natural layout only)
        geo = xbar + (step_x_natural(MP) ? 16 : 0);
        x = (geo + nops * 16 + 127) & ~127;
        xsum = x + step_x_bytes(MP, gpc_max);
        park = xsum + dec::xsum_bytes(MP, gpc_max, scaled);
        total = park + kWarps * shares * 16 * MP * 4;  // two parked shares (+ a finishing scratch) per warp
    }
};

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// This CTA's share of one projection, computed once per launch.
struct Geo {
    int g_lo, Gs;  // the K split's group range
    int ub, nu;    // the CTA's first band and band count
    int r;         // K split
    float inv_gs;  // 1 / Gs
    __device__ __forceinline__ int Tc() const { return nu * Gs; }
};
__device__ __forceinline__ void put_geo(uint4* tab, const StepOp& o, int c) {
    const int S = o.S, g = c / S, r = c - g * S;
    const int g_lo = o.G * r / S, Gs = o.G * (r + 1) / S - g_lo;
    const int ub = o.bands * g / o.cps, nu = o.bands * (g + 1) / o.cps - ub;
    *tab = make_uint4((uint32_t)g_lo | ((uint32_t)Gs << 16), (uint32_t)ub | ((uint32_t)nu << 16), (uint32_t)r,
                      __float_as_uint(1.0f / (float)Gs));
}
__device__ __forceinline__ Geo get_geo(const uint4* tab) {
    const uint4 v = *tab;
    Geo q;
    q.g_lo = (int)(v.x & 0xFFFF);
    q.Gs = (int)(v.x >> 16);
    q.ub = (int)(v.y & 0xFFFF);
    q.nu = (int)(v.y >> 16);
    q.r = (int)v.z;
    q.inv_gs = __uint_as_float(v.w);
    return q;
}
__device__ __forceinline__ int warp_lo(int Tc, int w) { return Tc * w / kWarps; }
// t / d for 0 <= t < 2^22, with inv = 1/d: the float estimate is off by at most one.
__device__ __forceinline__ int div_small(int t, int d, float inv) {
    int q = __float2int_rz((float)t * inv);
    const int rem = t - q * d;
    if (rem < 0) --q;
    else if (rem >= d) ++q;
    return q;
}

// The copy cursor of one warp: the next chunk of its ranges, over all projections.
struct Cursor {
    int i, t, t1, gl, Gs, G;
    const uint8_t* src;
    uint64_t policy;  // weights are read once: first out of L2

    __device__ __forceinline__ void seek(const StepArgs& a, const uint4* geo, int w) {
        for (; i < a.nops; ++i) {
            const Geo q = get_geo(geo + i);
            const int t0 = warp_lo(q.Tc(), w), te = warp_lo(q.Tc(), w + 1);
            if (t0 < te) {
                const int u = div_small(t0, q.Gs, q.inv_gs);
                t = t0;
                t1 = te;
                Gs = q.Gs;
                G = a.ops[i].G;
                gl = t0 - u * q.Gs;
                src = a.ops[i].w + ((size_t)(q.ub + u) * G + q.g_lo + gl) * kTileBytes;
                return;
            }
        }
    }
    // Copy the cursor's next chunk -- up to 4 tiles, not past the end of the
    // band's run nor of the range -- into dst (lane 0), completing on bar;
    // advance.  False (nothing issued) at the end of the stream.
    __device__ __forceinline__ bool issue(const StepArgs& a, const uint4* geo, int w, int lane, uint32_t dst,
                                          uint32_t bar) {
        if (i >= a.nops) return false;
        const int n = min(kSlotTiles, min(Gs - gl, t1 - t));
        if (lane == 0) {
            tc::mbar_arrive_expect_tx(bar, (uint32_t)(n * kTileBytes));
            tc::bulk_load_hint(dst, src, (uint32_t)(n * kTileBytes), bar, policy);
        }
        src += (size_t)n * kTileBytes;
        gl += n;
        if (gl == Gs) {
            gl = 0;
            src += (size_t)(G - Gs) * kTileBytes;
        }
        t += n;
        if (t == t1) {
            ++i;
            seek(a, geo, w);
        }
        return true;
    }
};

// The outputs a lane holds in MMA fragment layout: rows g8 and g8 + 8 of the
// band, tokens nt*8 + 2*(lane%4) + {0, 1}; f(row, m, value) for m < M.
template <int MP, typename F>
__device__ __forceinline__ void for_frag(const float (&acc)[(MP + 7) / 8][4], int lane, int M, F&& f) {
    constexpr int NT = (MP + 7) / 8;
    const int g8 = lane >> 2, cl4 = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int m0 = nt * 8 + 2 * cl4;
        if (m0 < M) {
            f(g8, m0, acc[nt][0]);
            f(g8 + 8, m0, acc[nt][2]);
        }
        if (m0 + 1 < M) {
            f(g8, m0 + 1, acc[nt][1]);
            f(g8 + 8, m0 + 1, acc[nt][3]);
        }
    }
}

// The final FP32 sums of band `band` of a K-split projection: publish this
// split's partial; the arrival that completes the band adds the S partials in
// split order and hands each sum to emit(row, m, sum).  False for every other
// arrival.  For 8 or more (padded) tokens the adding warp walks the band's
// outputs in lane-strided batches of kCombineOut and issues every load of a
// batch (kCombineOut outputs x up to 8 splits) before adding any: one output
// and one split at a time, each load is a dependent L2 round trip, which at
// 16 tokens (8 outputs per lane) made this the longest stretch of a
// projection.  At one token each lane issues its output's split loads at
// once; at 2 and 4 tokens the plain loop measured faster.
constexpr int kCombineOut = 4;
template <int MP, typename V, typename E>
__device__ __forceinline__ bool combine_splits(const StepOp& o, int band, int r, int M, int lane, V&& visit,
                                               E&& emit) {
    const int pb = 16 * M;
    float* mine = o.part + ((size_t)band * o.S + r) * pb;
    visit([&](int row, int m, float v) { mine[row * M + m] = v; });
    // the warp's stores are ordered before lane 0's fence by the warp barrier
    __syncwarp();
    unsigned last = 0;
    if (lane == 0) {
        __threadfence();
        last = atomicAdd(o.cnt + band, 1u) == (unsigned)(o.S - 1);
        if (last) __threadfence();
    }
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    if (!last) return false;
    const float* base = o.part + (size_t)band * o.S * pb;
    if constexpr (MP == 1) {
        // one token: at most one output per lane; every split's load in flight at once
        // (4 splits for down: 939 against 944 us per step; slower at 2 and 4 tokens)
        visit([&](int row, int m, float) {
            const float* pp = base + row * M + m;
            float sum = 0.f;
            for (int s = 0; s < o.S; s += 8) {
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = (s + e < o.S) ? __ldcg(pp + (size_t)(s + e) * pb) : 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (s + e < o.S) sum += v[e];  // only real splits: 0 + -0 would flip a zero's sign
            }
            emit(row, m, sum);
        });
    } else if constexpr (MP < 8) {
        visit([&](int row, int m, float) {
            const float* pp = base + row * M + m;
            float sum = 0.f;
            int s = 0;
            for (; s + 8 <= o.S; s += 8) {
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = __ldcg(pp + (size_t)(s + e) * pb);
#pragma unroll
                for (int e = 0; e < 8; ++e) sum += v[e];
            }
            for (; s < o.S; ++s) sum += __ldcg(pp + (size_t)s * pb);
            emit(row, m, sum);
        });
    } else {
    // (row, token) of output idx = row * M + m without an integer division: idx < 256, so the float
    // quotient, truncated, is exact
    const float inv_m = 1.f / (float)M;
    for (int o0 = 0; o0 < pb; o0 += 32 * kCombineOut) {
        float sum[kCombineOut];
#pragma unroll
        for (int j = 0; j < kCombineOut; ++j) sum[j] = 0.f;
        for (int s = 0; s < o.S; s += 8) {
            float v[kCombineOut][8];
#pragma unroll
            for (int j = 0; j < kCombineOut; ++j) {
                const int idx = o0 + 32 * j + lane;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    v[j][e] = (idx < pb && s + e < o.S) ? __ldcg(base + (size_t)(s + e) * pb + idx) : 0.f;
            }
#pragma unroll
            for (int j = 0; j < kCombineOut; ++j)
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (s + e < o.S) sum[j] += v[j][e];  // only real splits: 0 + -0 would flip a zero's sign
        }
#pragma unroll
        for (int j = 0; j < kCombineOut; ++j) {
            const int idx = o0 + 32 * j + lane;
            if (idx < pb) {
                const int row = __float2int_rz(((float)idx + 0.5f) * inv_m);
                emit(row, idx - row * M, sum[j]);
            }
        }
    }
    }
    if (lane == 0) o.cnt[band] = 0;  // ready for the next replay
    return true;
}

// Finish band `band` of projection o from per-lane outputs (visit(f) calls
// f(row, m, value) for each output this lane holds; every output of the band
// is held by exactly one lane of the warp).  Plain projection: the sums go to
// y.  Gated projection (W4_OP_SWIGLU): rows r and r + 8 of the band are gate
// and up row 8*band + r; the sums go to this warp's scratch and y (I = N/2
// columns) gets silu(gate) * up.
template <int ACT, int MPT, typename V>
__device__ __forceinline__ void finish_band(const StepOp& o, int band, int r, int M, int lane, V&& visit,
                                            float* scratch, int MP) {
    using Ops = dec::ActOps<ACT>;
    const int n0 = band * 16;
    if (o.flags & kOpTwoPhase) {
        float* mine = o.part + ((size_t)band * o.S + r) * (16 * M);
        visit([&](int row, int m, float v) { mine[row * M + m] = v; });
        return;
    }
    if (!(o.flags & W4_OP_SWIGLU)) {
        auto to_y = [&](int row, int m, float v) {
            if (n0 + row < o.N) o.y[(size_t)m * o.N + n0 + row] = Ops::round(v);
        };
        if (o.S == 1)
            visit(to_y);
        else
            combine_splits<MPT>(o, band, r, M, lane, visit, to_y);
        return;
    }
    auto to_scratch = [&](int row, int m, float v) { scratch[row * MP + m] = v; };
    if (o.S == 1)
        visit(to_scratch);
    else if (!combine_splits<MPT>(o, band, r, M, lane, visit, to_scratch))
        return;
    __syncwarp();
    const int I = o.N / 2;
    for (int oi = lane; oi < 8 * MPT; oi += 32) {
        const int rr = oi / MPT, m = oi % MPT;  // MPT is a power of two: shifts
        if (m >= M) continue;
        const float g = scratch[rr * MP + m], u = scratch[(rr + 8) * MP + m];
        const int n = band * 8 + rr;
        if (n < I) o.y[(size_t)m * I + n] = Ops::round(g / (1.f + expf(-g)) * u);
    }
    __syncwarp();
}

// Second phase of a two-phase projection: CTA c of NC adds up the partials of
// bands [bands*c/NC, bands*(c+1)/NC), each output over its S splits in split
// order, and writes y (a gated projection: silu(gate) * up of rows r and
// r + 8 of each band).  Every thread takes outputs strided by the block, with
// the loads of up to eight splits of an output in flight at once (batching
// eight outputs per thread as well measured slower: 16 tokens 1813 -> 1930
// us per step).
template <int MP, int ACT, bool GATED>
__device__ __forceinline__ void combine_share_of(const StepOp& o, int b0, int total, int M) {
    using Ops = dec::ActOps<ACT>;
    constexpr int kLogMP = MP == 1 ? 0 : MP == 2 ? 1 : MP == 4 ? 2 : MP == 8 ? 3 : 4;
    constexpr int sh = (GATED ? 3 : 4) + kLogMP;  // outputs per band: (8 or 16 rows) x MP
    const int pb = 16 * M, S = o.S;
    for (int idx = threadIdx.x; idx < total; idx += kThreads) {
        const int rem = idx & ((1 << sh) - 1), band = b0 + (idx >> sh);
        const int row = rem >> kLogMP, m = rem & (MP - 1);
        if (m >= M) continue;
        const float* pp = o.part + (size_t)band * S * pb + row * M + m;
        float g = 0.f, u = 0.f;
        for (int s0 = 0; s0 < S; s0 += 8) {
            float v[8], w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                v[e] = s0 + e < S ? __ldcg(pp + (size_t)(s0 + e) * pb) : 0.f;
                if constexpr (GATED) w[e] = s0 + e < S ? __ldcg(pp + (size_t)(s0 + e) * pb + 8 * M) : 0.f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (s0 + e < S) {  // the first split starts the sum: 0 + -0 would flip a zero's sign
                    g = s0 + e == 0 ? v[e] : g + v[e];
                    if constexpr (GATED) u = s0 + e == 0 ? w[e] : u + w[e];
                }
        }
        if constexpr (!GATED) {
            const int n = band * 16 + row;
            if (n < o.N) o.y[(size_t)m * o.N + n] = Ops::round(g);
        } else {
            const int I = o.N / 2, n = band * 8 + row;
            if (n < I) o.y[(size_t)m * I + n] = Ops::round(g / (1.f + expf(-g)) * u);
        }
    }
}
// The same for two splits of a plain projection: every output's two loads,
// for up to eight outputs per thread, in flight at once (at 16 tokens a
// CTA's share of gate_up is about 4000 outputs: eight per thread).
template <int MP, int ACT>
__device__ __forceinline__ void combine_share_two(const StepOp& o, int b0, int total, int M) {
    using Ops = dec::ActOps<ACT>;
    constexpr int kLogMP = MP == 1 ? 0 : MP == 2 ? 1 : MP == 4 ? 2 : MP == 8 ? 3 : 4;
    constexpr int sh = 4 + kLogMP, kOut = 8;
    const int pb = 16 * M;
    for (int r0 = threadIdx.x; r0 < total; r0 += kThreads * kOut) {
        float v0[kOut], v1[kOut];
#pragma unroll
        for (int j = 0; j < kOut; ++j) {
            const int idx = r0 + j * kThreads, rem = idx & ((1 << sh) - 1);
            const int row = rem >> kLogMP, m = rem & (MP - 1);
            const float* pp = o.part + (size_t)(b0 + (idx >> sh)) * 2 * pb + row * M + m;
            const bool live = idx < total && m < M;
            v0[j] = live ? __ldcg(pp) : 0.f;
            v1[j] = live ? __ldcg(pp + pb) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < kOut; ++j) {
            const int idx = r0 + j * kThreads, rem = idx & ((1 << sh) - 1);
            const int row = rem >> kLogMP, m = rem & (MP - 1), n = (b0 + (idx >> sh)) * 16 + row;
            if (idx < total && m < M && n < o.N) o.y[(size_t)m * o.N + n] = Ops::round(v0[j] + v1[j]);
        }
    }
}
template <int MP, int ACT>
__device__ __forceinline__ void combine_share(const StepOp& o, int c, int NC, int M) {
    constexpr int kLogMP = MP == 1 ? 0 : MP == 2 ? 1 : MP == 4 ? 2 : MP == 8 ? 3 : 4;
    const int b0 = (int)((long long)o.bands * c / NC), b1 = (int)((long long)o.bands * (c + 1) / NC);
    if (o.S == 2 && !(o.flags & W4_OP_SWIGLU))
        combine_share_two<MP, ACT>(o, b0, (b1 - b0) << (4 + kLogMP), M);
    else if (o.flags & W4_OP_SWIGLU)
        combine_share_of<MP, ACT, true>(o, b0, (b1 - b0) << (3 + kLogMP), M);
    else
        combine_share_of<MP, ACT, false>(o, b0, (b1 - b0) << (4 + kLogMP), M);
}

template <int MP, int ACT>
__global__ void __launch_bounds__(kThreads, 1) step_kernel(const __grid_constant__ StepArgs a) {
    constexpr int NT = (MP + 7) / 8;
    constexpr int PB = 16 * MP;  // floats of one parked band partial
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NC = gridDim.x, c = blockIdx.x, M = a.M, nops = a.nops;
    // parked shares: 3 below 16 tokens, else from the table
    const int PS = MP >= 16 ? (a.ring >> 16) : 3;
    const StepSmem L(MP >= 16 ? (a.ring & 0xFFFF) : a.ring, MP, a.gpc_max, nops, PS, dec::ActOps<ACT>::kScaled);
    const int R = L.R;
    const uint32_t sbase = tc::smem_addr(smem);
    const uint32_t ring_w = sbase + (uint32_t)(warp * R * kSlotTiles * kTileBytes);
    const uint32_t bar_w = sbase + (uint32_t)(L.bar + warp * R * 8);
    uint4* geo = reinterpret_cast<uint4*>(smem + L.geo);
    uint32_t* xs = reinterpret_cast<uint32_t*>(smem + L.x);
    float* xsum = reinterpret_cast<float*>(smem + L.xsum);
    float* park = reinterpret_cast<float*>(smem + L.park);
    float* park_w = park + warp * PS * PB;
    float* scratch_w = park_w + 2 * PB;

    for (int i = threadIdx.x; i < nops; i += kThreads) put_geo(geo + i, a.ops[i], c);
    // x slices are small and read by every CTA of a split: keep the next one
    // warm in L2 (as it is when x has just been written)
    auto prefetch_x = [&](int i) {
        if (i < nops) {
            const Geo q = get_geo(geo + i);
            const StepOp& o = a.ops[i];
            if (q.nu > 0)
                for (int m = 0; m < M; ++m)
                    tc::prefetch_l2(o.x + (size_t)m * (o.K / 2) + (size_t)q.g_lo * 64, (uint32_t)(q.Gs * 256));
        }
    };
    if (lane < R) tc::mbar_init(bar_w + 8 * lane, 1);
    // x slices from four tokens on: natural layout, one bulk copy per token row
    constexpr bool kNat = step_x_natural(MP) && ACT != dec::kActI8;
    const uint32_t xbar = sbase + (uint32_t)L.xbar;
    uint32_t xphase = 0;
    if (kNat && threadIdx.x == 0) tc::mbar_init(xbar, 1);
    tc::mbar_init_fence();
    __syncthreads();
    if (threadIdx.x == 0) prefetch_x(0);

    // fill this warp's ring
    Cursor cur;
    cur.i = 0;
    cur.policy = tc::policy_evict_first();
    cur.seek(a, geo, warp);
    int inflight = 0;
    for (int s = 0; s < R; ++s) {
        if (!cur.issue(a, geo, warp, lane, ring_w + (uint32_t)(s * kSlotTiles * kTileBytes), bar_w + 8 * s)) break;
        ++inflight;
    }
    int slot = 0;           // next slot to consume
    uint32_t phase = 0;     // its expected completion parity
    bool ok = true;

    for (int i = 0; i < nops; ++i) {
        const StepOp& o = a.ops[i];
        if (threadIdx.x == 32) prefetch_x(i + 1);
        if (i > 0) {
            // x_i may be computed from y_(i-1): wait until every CTA is done with it
            if (threadIdx.x == 0) {
                const long long t0 = clock64();
                while (ld_acquire(a.done + (i - 1)) < (unsigned)NC) {
                    if (clock64() - t0 > (1ll << 31)) {
                        atomicOr(a.status, 2);
                        break;
                    }
                }
            }
            __syncthreads();
        }
        const Geo q = get_geo(geo + i);
        if (q.nu > 0) {
            if constexpr (ACT == dec::kActI8)
                dec::stage_x_q8<MP, kThreads>(o.x, M, o.K, q.g_lo, q.Gs, xs, xsum, park);  // parks are free now
            else if constexpr (!kNat)
                dec::stage_x_async<MP, kThreads, ACT>(o.x, M, o.K, q.g_lo, q.Gs, xs, xsum);
            else {
                if (!dec::stage_x_bulk<MP, kThreads, ACT>(o.x, M, o.K, q.g_lo, q.Gs, xs, xsum, xbar, xphase) &&
                    threadIdx.x == 0)
                    atomicOr(a.status, 8);
                xphase ^= 1;
            }
            dec::TileMac<MP, ACT> mac(sbase + L.x, sbase + L.xsum, lane, q.Gs);
            if constexpr (kNat) mac.set_natural(sbase + L.x, lane, dec::x_row_bytes(q.Gs));
            const int Tc = q.Tc();
            const int t0 = warp_lo(Tc, warp), t1 = warp_lo(Tc, warp + 1);
            const int u_first = div_small(t0, q.Gs, q.inv_gs);
            int t = t0, gl = t0 - u_first * q.Gs, u = u_first;
            float acc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
            while (t < t1) {
                const int n = min(kSlotTiles, min(q.Gs - gl, t1 - t));  // the chunk the cursor copied
                if (ok) {
                    const uint32_t ta = ring_w + (uint32_t)(slot * kSlotTiles * kTileBytes), bar = bar_w + 8 * slot;
                    const bool got = tc::mbar_wait(bar, phase);
                    if (__all_sync(0xFFFFFFFFu, got)) {
                        --inflight;
                        static_assert(kSlotTiles == 4, "chunk cases below");
                        // register budget: at most two tiles at once (16 tokens; 4 tokens of rescaled x)
                        if constexpr (MP >= 16 || (MP == 4 && dec::ActOps<ACT>::kScaled)) {
                            if (n >= 2) mac.template run_tiles<2, kNat>(ta, gl, lane, acc);
                            if (n == 4) mac.template run_tiles<2, kNat>(ta + 2 * kTileBytes, gl + 2, lane, acc);
                            if (n & 1)
                                mac.template run_tiles<1, kNat>(ta + (uint32_t)((n - 1) * kTileBytes), gl + n - 1,
                                                                lane, acc);
                        } else {
                            if (n == 4) mac.template run_tiles<4, kNat>(ta, gl, lane, acc);
                            else if (n == 3) mac.template run_tiles<3, kNat>(ta, gl, lane, acc);
                            else if (n == 2) mac.template run_tiles<2, kNat>(ta, gl, lane, acc);
                            else mac.template run_tiles<1, kNat>(ta, gl, lane, acc);
                        }
                        __syncwarp();  // every lane is done reading the slot
                        if (cur.issue(a, geo, warp, lane, ta, bar)) ++inflight;
                        if (++slot == R) {
                            slot = 0;
                            phase ^= 1;
                        }
                    } else {
                        if (lane == 0) atomicOr(a.status, 4);
                        ok = false;
                    }
                }
                t += n;
                gl += n;
                if (gl == q.Gs || t == t1) {
                    const int us = u * q.Gs;
                    if (us >= t0 && us + q.Gs <= t1) {
                        // the whole band is this warp's: finish it from the accumulators
                        finish_band<ACT, MP>(o, q.ub + u, q.r, M, lane, [&](auto&& f) { for_frag<MP>(acc, lane, M, f); },
                                         scratch_w, MP);
                    } else {
                        // cut between warps: park this warp's share
                        float* dst = park_w + (u == u_first ? 0 : PB);
                        for_frag<MP>(acc, lane, M, [&](int row, int m, float v) { dst[row * MP + m] = v; });
                    }
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
                    ++u;
                    gl = 0;
                }
            }
            __syncthreads();
            const int bs = u_first * q.Gs, be = bs + q.Gs;
            const bool two = o.flags & kOpTwoPhase;
            if (MP >= 8 && (two || (o.S == 1 && !(o.flags & W4_OP_SWIGLU)))) {
                // a plain band cut between warps is added up, in warp order, by every warp whose range
                // begins inside it, each taking every nh-th batch of 32 outputs (the others are idle here;
                // measured slower below 8 tokens, where a band has at most 64 outputs)
                if (t0 < t1 && !(bs == t0 && be <= t1)) {
                    int hidx = 0, nh = 0, wa = 0;
#pragma unroll
                    for (int w2 = 0; w2 < kWarps; ++w2) {
                        const int lo = warp_lo(Tc, w2), hi = warp_lo(Tc, w2 + 1);
                        if (lo < hi && lo >= bs && lo < be) {
                            hidx += w2 < warp;
                            ++nh;
                        }
                        if (lo < hi && lo <= bs) wa = w2;  // the warp holding the band's first tile
                    }
                    for (int oi = lane + 32 * hidx; oi < 16 * MP; oi += 32 * nh) {
                        const int row = oi / MP, m = oi % MP;  // MP is a power of two: shifts
                        if (m >= M) continue;
                        float sum = 0.f;
                        for (int w2 = wa; w2 < kWarps; ++w2) {
                            const int lo = warp_lo(Tc, w2), hi = warp_lo(Tc, w2 + 1);
                            if (lo >= be) break;
                            if (lo < hi) sum += park[(w2 * PS + (lo >= bs ? 0 : 1)) * PB + row * MP + m];
                        }
                        if (two) {
                            o.part[((size_t)(q.ub + u_first) * o.S + q.r) * (16 * M) + row * M + m] = sum;
                        } else {
                            const int n0 = (q.ub + u_first) * 16;
                            if (n0 + row < o.N) o.y[(size_t)m * o.N + n0 + row] = dec::ActOps<ACT>::round(sum);
                        }
                    }
                }
            } else if (warp > 0 && t0 < Tc && t0 != bs && warp_lo(Tc, warp - 1) <= bs) {
                // a split or gated band cut between warps is added up, in warp order, by the lowest warp
                // whose range starts strictly inside it (warp - 1 then holds the band's first tile)
                finish_band<ACT, MP>(o, q.ub + u_first, q.r, M, lane, [&](auto&& f) {
                    // outputs strided by the padded token count (a power of two: no division)
                    for (int oi = lane; oi < 16 * MP; oi += 32) {
                        const int row = oi / MP, m = oi % MP;
                        if (m >= M) continue;
                        float sum = 0.f;
                        for (int w2 = warp - 1; w2 < kWarps; ++w2) {
                            const int lo = warp_lo(Tc, w2), hi = warp_lo(Tc, w2 + 1);
                            if (lo >= be) break;
                            if (lo < hi) sum += park[(w2 * PS + (lo >= bs ? 0 : 1)) * PB + row * MP + m];
                        }
                        f(row, m, sum);
                    }
                }, scratch_w, MP);
            }
        }
        // this CTA is done with projection i: the barrier orders every
        // thread's y stores before thread 0's fence, which makes them visible
        // before the completion count
        __syncthreads();
        if (MP >= kTwoPhaseMinMP && (o.flags & kOpTwoPhase)) {
            // the same for the partials, then wait for every CTA's and add up this CTA's share
            if (threadIdx.x == 0) {
                asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(o.cnt) : "memory");
                const long long t0 = clock64();
                while (ld_acquire(o.cnt) < (unsigned)NC) {
                    if (clock64() - t0 > (1ll << 31)) {
                        atomicOr(a.status, 16);
                        break;
                    }
                }
            }
            __syncthreads();
            combine_share<MP, ACT>(o, c, NC, M);
            __syncthreads();
        }
        if (threadIdx.x == 0)
            asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(a.done + i) : "memory");
    }

    // copies still in flight after a timeout
    for (; inflight > 0; --inflight) {
        if (!tc::mbar_wait(bar_w + 8 * slot, phase)) break;
        if (++slot == R) {
            slot = 0;
            phase ^= 1;
        }
    }

    // the last CTA out resets the counters for the next step
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(a.exit_cnt, 1u) == (unsigned)(NC - 1)) {
            for (int i = 0; i < nops; ++i) {
                a.done[i] = 0;
                if (a.ops[i].flags & kOpTwoPhase) *a.ops[i].cnt = 0;
            }
            *a.exit_cnt = 0;
            __threadfence();
        }
    }
}

using StepKernel = void (*)(StepArgs);

template <int ACT>
StepKernel step_fn_act(int MP) {
    switch (MP) {
        case 1: return step_kernel<1, ACT>;
        case 2: return step_kernel<2, ACT>;
        case 4: return step_kernel<4, ACT>;
        case 8: return step_kernel<8, ACT>;
        default: return step_kernel<16, ACT>;
    }
}
StepKernel step_fn(int MP, int act) {
    if (act == dec::kActBF16) return step_fn_act<dec::kActBF16>(MP);
    if (act == dec::kActI8) return step_fn_act<dec::kActI8>(MP);
    return step_fn_act<dec::kActF16>(MP);
}

int padded(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : 16; }

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

}  // namespace

// ---- host-side plan ---------------------------------------------------------------
struct StepPlan {
    int MP = 1, NC = 0, gpc_max = 1, R = 0, smem = 0, shares = 2;
    std::vector<StepOp> ops;  // device pointers filled against a workspace base
    size_t done_off = 0, exit_off = 0, status_off = 0, total = 0;
    std::vector<size_t> cnt_off, part_off;
};

// K split of one projection: S divides NC (the CTAs of a split are c % S),
// the x slice fits its budget, and the largest per-CTA share of tiles (plus a
// fixed cost for combining partials when S > 1, plus the x slice's staging
// for up to 4 tokens) is smallest.  0 if no split fits.
static int choose_split(int bands, int G, int MP, int NC, int budget, bool scaled) {
    int best = 0;
    long best_cost = LONG_MAX;
    for (int S = 1; S <= std::min(G, NC); ++S) {
        if (NC % S) continue;
        const int Gs = (G + S - 1) / S;
        if (step_x_bytes(MP, Gs) + dec::xsum_bytes(MP, Gs, scaled) > budget) continue;
        const int cps = NC / S;
        // up to 4 tokens, staging the x slice (an L2 round trip plus ~3 tile-times per KB
        // under load) is counted too; from 8 tokens on, more splits cost more in partials
        // than they save in staging, and the plain count measured better
        const long x_cost = MP <= 4 ? 3L * (step_x_bytes(MP, Gs) + dec::xsum_bytes(MP, Gs, scaled)) / 1024 : 0;
        const long cost = (long)((bands + cps - 1) / cps) * Gs + (S > 1 ? kSplitPenalty + 4 * S : 0) + x_cost;
        if (cost < best_cost) {
            best_cost = cost;
            best = S;
        }
    }
    return best;
}

// Splits, shared-memory sizing (the rings take what the rest leaves) and the
// workspace layout for x slices of at most `budget` bytes and `shares` parked
// partials per warp.  False if some projection cannot be planned.
static bool plan_step_with(const w4_weight* w, int n, int M, int NC, int budget, int shares, bool scaled,
                           StepPlan* pl) {
    pl->MP = padded(M);
    pl->shares = shares;
    pl->NC = NC;
    pl->ops.assign(n, StepOp{});
    pl->cnt_off.assign(n, 0);
    pl->part_off.assign(n, 0);
    pl->gpc_max = 1;
    bool fits = NC > 0 && n <= kMaxStepOps;
    for (int i = 0; i < n && fits; ++i) {
        StepOp& o = pl->ops[i];
        o.N = (int)w[i].N;
        o.K = (int)w[i].K;
        o.G = (int)(w[i].K / kGroupK);
        o.bands = (int)num_bands(w[i].N);
        o.S = choose_split(o.bands, o.G, pl->MP, NC, budget, scaled);
        if (o.S == 0) {
            fits = false;
            o.S = 1;
        }
        o.cps = NC / o.S;
        // 16-bit fields of the per-CTA share table, 32-bit share arithmetic
        const long long cta_tiles = (long long)((o.bands + o.cps - 1) / o.cps) * ((o.G + o.S - 1) / o.S);
        if (o.bands >= 65536 || o.G >= 65536 || (long long)o.bands * NC >= INT_MAX ||
            (long long)o.G * o.S >= INT_MAX || cta_tiles >= kMaxCtaTiles)
            fits = false;
        pl->gpc_max = std::max(pl->gpc_max, (o.G + o.S - 1) / o.S);
    }
    const int fixed = StepSmem(0, pl->MP, pl->gpc_max, n, shares, scaled).total;
    pl->R = std::min(kMaxRing, (kSmemBudget - fixed) / (kWarps * (kSlotTiles * kTileBytes + 8)));
    while (pl->R > 0 && StepSmem(pl->R, pl->MP, pl->gpc_max, n, shares, scaled).total > kSmemBudget) --pl->R;
    pl->smem = StepSmem(pl->R, pl->MP, pl->gpc_max, n, shares, scaled).total;
    size_t off = 0;
    pl->done_off = off;
    off = align_up(off + sizeof(unsigned) * n);
    pl->exit_off = off;
    pl->status_off = off + 16;
    off = align_up(off + 32);
    for (int i = 0; i < n; ++i) {
        const StepOp& o = pl->ops[i];
        if (o.S > 1) {
            pl->cnt_off[i] = off;
            off = align_up(off + sizeof(unsigned) * o.bands);
            pl->part_off[i] = off;
            off = align_up(off + sizeof(float) * (size_t)o.bands * o.S * 16 * M);
        }
    }
    pl->total = off;
    return fits && pl->R >= 2;
}

// The plan with the large x budget, or, if that cannot keep two ring slots
// per warp, with the fallback budget.  The finishing scratch (a third parked
// share per warp) is left out only at 16 tokens without a gated projection,
// where the 16 KB it frees lets a 60 KB x slice (2 K splits instead of 4)
// keep two ring slots: 3689 -> 3418 us.  Below 16 tokens the kernel keeps
// three shares as a constant (its code is unchanged there: a run-time share
// count or ring mask measured 4-35 us slower at 1-8 tokens).
static bool plan_step(const w4_weight* w, int n, int M, int NC, bool gated, int act, StepPlan* pl) {
    const int MP = padded(M), shares = (gated || MP < 16) ? 3 : 2;
    const bool scaled = act == dec::kActBF16;  // x staged as rescaled binary16: a second float per group sum
    if (plan_step_with(w, n, M, NC, x_budget(MP), shares, scaled, pl)) return true;
    return x_budget_fallback(MP) != x_budget(MP) &&
           plan_step_with(w, n, M, NC, x_budget_fallback(MP), shares, scaled, pl);
}

// One resident CTA per SM, or 0 if the kernel cannot be resident.
static int step_grid(int MP, int act, int smem) {
    int per_sm = 0;
    StepKernel fn = step_fn(MP, act);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, smem) != cudaSuccess) return 0;
    return per_sm >= 1 ? device_sm_count() : 0;
}

// Enough for the sequence with or without gated projections and for every
// activation type (the plans can differ in their splits).
size_t step_workspace_bytes(const w4_weight* w, int n, int M) {
    size_t most = 0;
    for (int act : {(int)dec::kActF16, (int)dec::kActBF16, (int)dec::kActI8})
        for (bool gated : {false, true}) {
            StepPlan pl;
            plan_step(w, n, M, device_sm_count(), gated, act, &pl);
            most = std::max(most, pl.total);
        }
    return most;
}

void step_splits(const w4_weight* w, int n, int M, int act, bool gated, int* splits) {
    StepPlan pl;
    plan_step(w, n, M, device_sm_count(), gated, act, &pl);
    for (int i = 0; i < n; ++i) splits[i] = pl.ops[i].S;
}

w4_status step_prepare(const w4_weight* w, const void* const* x, void* const* y, const uint32_t* op_flags, int n,
                       int M, int act, void* ws, size_t ws_bytes, cudaStream_t stream, StepLaunch* out) {
    const int MP = padded(M);
    bool gated = false;
    for (int i = 0; i < n && op_flags; ++i) gated = gated || (op_flags[i] & W4_OP_SWIGLU);
    StepPlan pl;
    if (!plan_step(w, n, M, device_sm_count(), gated, act, &pl)) {
        set_error("the persistent step kernel cannot take this sequence (%d projections; at most %d, and each "
                  "must fit its shared-memory and index limits)",
                  n, kMaxStepOps);
        return W4_ERR_UNSUPPORTED;
    }
    const int NC = step_grid(MP, act, pl.smem);
    if (NC <= 0 || NC != pl.NC) {
        set_error("the persistent step kernel cannot be resident (shared memory %d bytes)", pl.smem);
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
        o.flags = (int16_t)(op_flags ? op_flags[i] : 0u);
        if (o.S > 1 && pl.MP >= kTwoPhaseMinMP) o.flags |= kOpTwoPhase;
        o.w = static_cast<const uint8_t*>(w[i].data);
        o.x = static_cast<const uint32_t*>(x[i]);
        o.y = static_cast<uint16_t*>(y[i]);
        o.cnt = o.S > 1 ? reinterpret_cast<unsigned*>(base + pl.cnt_off[i]) : nullptr;
        o.part = o.S > 1 ? reinterpret_cast<float*>(base + pl.part_off[i]) : nullptr;
    }
    W4_CUDA_TRY(cudaMemsetAsync(ws, 0, pl.total, stream));
    W4_CUDA_TRY(cudaStreamSynchronize(stream));
    out->args.assign(sizeof(StepArgs), 0);
    StepArgs* a = reinterpret_cast<StepArgs*>(out->args.data());
    a->nops = n;
    a->M = M;
    a->done = reinterpret_cast<unsigned*>(base + pl.done_off);
    a->exit_cnt = reinterpret_cast<unsigned*>(base + pl.exit_off);
    a->status = reinterpret_cast<int*>(base + pl.status_off);
    a->gpc_max = pl.gpc_max;
    a->ring = pl.R | (pl.MP >= 16 ? pl.shares << 16 : 0);
    std::copy(pl.ops.begin(), pl.ops.end(), a->ops);
    out->fn = reinterpret_cast<const void*>(step_fn(MP, act));
    out->status = a->status;
    out->NC = NC;
    out->smem = pl.smem;
    return W4_OK;
}

int step_status(const StepLaunch& s) {
    int v = 0;
    if (!s.status || cudaMemcpy(&v, s.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
    return v;
}

w4_status step_launch(const StepLaunch& s, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)s.NC, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)s.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeCooperative;
    attr.val.cooperative = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    void* params[] = {const_cast<unsigned char*>(s.args.data())};
    cudaError_t e = cudaLaunchKernelExC(&cfg, s.fn, params);
    if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelEx(step)");
    return W4_OK;
}

}  // namespace w4
