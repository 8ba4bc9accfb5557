// Prefill projection y[M, N] = x[M, K] . W^T for M > 16 on the sm_103a
// tensor cores (tcgen05 + TMEM); M <= 16 goes to the decode kernel.
//
// Same arithmetic as the decode kernel and the pages' definition (symmetric
// group-wise INT4, group 128, FP16 scale per group, FP16 activations:
// "Building a Custom LLM Inference Runtime ...", "Technical Specifications and
// Hardware Alignment"): FP16 x FP16 products are exact, each 128-wide group is
// summed in FP32 by the tensor core, and the group's FP32 partial is scaled by
// its FP32 scale and added in FP32 registers.  The scale is never folded into
// an FP16 weight, so the weights reach the tensor core exactly.
//
// A tile is 128 weight rows x BN tokens (192, or 128 where that keeps more SMs
// busy; chosen per call with the K split) over a K range.  The CTAs are
// persistent (one per SM, or per tile if fewer) and walk their tiles in turn,
// one 128-wide group per pipeline step, with warp-specialised roles:
//   warp 0     TMA producer: x tile [BN tokens][128 K] as two 128-byte
//              swizzled boxes (zero fill past M) into a shared-memory stage
//   warp 3     producer of the group's 8 packed weight tiles (one 2-D TMA
//              copy through a tensor map over the packed weight) into the
//              same stage
//   warps 1-2  one thread each issues 8 tcgen05.mma (128xBNx16) per group
//              (warp 1 the even groups, warp 2 the odd ones), A from tensor
//              memory and B (x) from shared memory, into its own TMEM
//              accumulator, then commits
//   warps 4-7  dequant: read the group's packed tiles from the stage, unpack
//              nibbles to exact fp16 q and store them straight into one of
//              two A slots of tensor memory (16-lane x 256-bit stores: the
//              packed tile's lane layout is that store's register layout)
//   warps 8-15 promote: read a group's FP32 partial from TMEM, hand the
//              accumulator back, multiply by the group scale and add to
//              FP32 accumulators in registers (BN/2 per thread: these two
//              warpgroups take registers from the other two); at the end of
//              each tile each warp puts its 32 rows x BN/2 tokens of y (fp16;
//              with K split, its FP32 partial in two halves) into its slice
//              of the x stage of the tile's last group (free once that
//              group's MMAs are done) and one thread issues TMA stores of it;
//              the x producer refills that stage only after the stores have
//              read it (barrier y_done), and the warp goes on to the next
//              tile's groups at once
// Tile width: the MMA instruction is full rate from N = 128 up when issued
// alone, but in this loop, beside the tensor-memory stores of A and the
// reads of every group's FP32 partial, 8 MMAs take about as long at N = 128
// as at N = 192 (~130 SM cycles each), so wide tiles pay.  Two 256-column accumulators
// would fill tensor memory and leave no room for A, and with one accumulator
// the MMAs wait for every group's partial to be read out; 192 tokens leave
// room for two accumulators and two A slots (192 + 192 + 2 x 64 = 512
// columns).
// Every mbarrier wait is bounded; a timeout sets the status word in the
// workspace and the CTA drains and exits instead of hanging.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "tc_ptx.cuh"
#include "w4_device.cuh"
#include "w4_internal.cuh"

namespace w4 {
void default_gemv_config(int M, int64_t N, int64_t K, w4_gemv_config* c);
w4_status launch_gemv(const void* x, const w4_weight* w, void* y, int M, const w4_gemv_config& c,
                      cudaStream_t stream);
w4_status check_gemv_args(const void* x, const w4_weight* w, const void* y, int M);

namespace {

// ---- wide tensor-memory loads and stores (fewer tcgen05 instructions per group) ----
// 32 lanes x 64 columns of 32-bit words in one instruction: thread i receives
// lane (base + i), columns col .. col + 63 (two 32-column loads' registers,
// one after the other).
__device__ __forceinline__ void tmem_ld_32x32_x64(uint32_t taddr, uint32_t (&v)[64]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31]), "=r"(v[32]), "=r"(v[33]), "=r"(v[34]), "=r"(v[35]), "=r"(v[36]), "=r"(v[37]), "=r"(v[38]), "=r"(v[39]), "=r"(v[40]), "=r"(v[41]), "=r"(v[42]), "=r"(v[43]), "=r"(v[44]), "=r"(v[45]), "=r"(v[46]), "=r"(v[47]), "=r"(v[48]), "=r"(v[49]), "=r"(v[50]), "=r"(v[51]), "=r"(v[52]), "=r"(v[53]), "=r"(v[54]), "=r"(v[55]), "=r"(v[56]), "=r"(v[57]), "=r"(v[58]), "=r"(v[59]), "=r"(v[60]), "=r"(v[61]), "=r"(v[62]), "=r"(v[63])
                 : "r"(taddr)
                 : "memory");
}
// 16 lanes x 256 bits repeated over 8 blocks of 8 columns (64 columns) in
// one instruction: the registers of two 4-block stores, one after the other
// (thread 4r + c: v[4i], v[4i+1] to lane base + r, columns col + 8i + 2c, + 1;
// v[4i+2], v[4i+3] to lane base + r + 8).
__device__ __forceinline__ void tmem_st_16x256_x8(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile("tcgen05.st.sync.aligned.16x256b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
                 : "memory");
}

// ---- TMA stores (the prefill kernel's output) ----------------------------------
// Tiled store of a shared-memory box to global memory (elements outside the
// tensor are not written), tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     (uint64_t)map),
                 "r"(c0), "r"(c1), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                     (uint64_t)map),
                 "r"(c0), "r"(c1), "r"(c2), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// this thread's committed bulk stores have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// ... and are complete (their writes performed)
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// orders this thread's generic-proxy shared-memory writes before later async-proxy (TMA) reads
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

constexpr int kBM = 128;                   // weight rows per CTA (8 bands)
constexpr int kASlots = 2;                 // A slots in tensor memory
constexpr int kWStage = 8 * kTileBytes;    // the group's 8 packed tiles (one per band)
constexpr int kThreads = 512;
constexpr int kTmemCols = 512;
// Per tile width BN (tokens per CTA: 128 or 192): the x stage (BN x 128 fp16;
// at the end of a tile the stage of its last group holds the tile's y, 128
// rows x BN tokens of fp16, the same size), four shared-memory stages (one
// group each), and tensor memory as two BN-column FP32 accumulators followed
// by one 64-column block of fp16 q pairs (128 rows x 128 K) per A slot.
template <int BN>
struct Tile {
    static constexpr int kBStage = BN * 128 * 2;
    static constexpr int kStages = 4;
    static constexpr int kACol0 = 2 * BN;
    static constexpr int kSmemBytes = kStages * (kBStage + kWStage) + 1024 + 256;
    static_assert(8 * 32 * (BN / 2) * 2 == kBStage, "a tile's y fills one x stage");
    static_assert(kACol0 + 64 * kASlots <= kTmemCols, "tensor memory columns");
    static_assert(BN % 64 == 0 && BN <= 256, "MMA N and promote column blocks");
};
// Registers per thread after the split: warpgroups 0-1 (producer, issuer,
// dequant) give up registers to warpgroups 2-3 (promote).  The four shares
// add up to the 128 x 512 the CTA is launched with.
// Registers per thread after the split: warpgroup 0 (producers, MMA issuers:
// one busy thread per warp) 48, warpgroup 1 (dequant) 112, warpgroups 2-3
// (promote) 176, which lets a promote thread hold two 32-column pieces of a
// partial beside its 96 accumulators.  The four shares add up to the 128 x
// 512 the CTA is launched with.
constexpr int kRegsIssue = 48, kRegsDequant = 112, kRegsHigh = 176;
static_assert(kRegsIssue + kRegsDequant + 2 * kRegsHigh == 4 * 128, "register split");
static_assert(kWStage % 128 == 0, "weight stages start 128-byte aligned (TMA destination)");
constexpr size_t kStatusBytes = 256;       // workspace head: status word (+ padding)

struct GemmParams {
    const uint8_t* w;
    uint16_t* y;
    float* part;  // split-K partials [splits][M][N], or null
    int* status;
    int M, N, K, G, bands, splits;
    int tiles_x, tiles_y, tiles;  // token blocks, row blocks, tiles (x fastest, then row block, then split)
    int ystore;                   // 1: y (or the split-K partial) leaves through an x stage and TMA stores
                                  // (omap: y [M][N] fp16, or the partials [splits][M][N] fp32)
};

// Tile t of the call: its first token and band, its K split and group range.
struct TileAt {
    int tok0, band0, split, g_lo, ng;
};
__device__ __forceinline__ TileAt tile_at(const GemmParams& p, int t, int bn) {
    const int x = t % p.tiles_x, r = t / p.tiles_x, yb = r % p.tiles_y, z = r / p.tiles_y;
    TileAt a;
    a.tok0 = x * bn;
    a.band0 = yb * (kBM / 16);
    a.split = z;
    a.g_lo = (int)((long long)p.G * z / p.splits);
    a.ng = (int)((long long)p.G * (z + 1) / p.splits) - a.g_lo;
    return a;
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ CUtensorMap xmap,
                                                              const __grid_constant__ CUtensorMap wmap,
                                                              const __grid_constant__ CUtensorMap omap, GemmParams p) {
    constexpr int kBN = BN, kBStage = Tile<BN>::kBStage, kACol0 = Tile<BN>::kACol0, kStages = Tile<BN>::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sB = smem;
    uint8_t* sW = sB + kStages * kBStage;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sW + kStages * kWStage);
    // barrier slots
    const uint32_t x_full = tc::smem_addr(bars), w_full = x_full + 8 * kStages, empty = w_full + 8 * kStages,
                   a_full = empty + 8 * kStages, a_empty = a_full + 8 * kASlots, d_full = a_empty + 8 * kASlots,
                   d_empty = d_full + 16, y_done = d_empty + 16;
    __shared__ uint32_t tmem_base_sh;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Persistent: CTA c takes tiles c, c + gridDim.x, ...; every role walks the same tiles and
    // groups, and a running group count gi (across tiles) picks stages, A slots, accumulators and
    // their phases, so the pipeline runs on from one tile into the next.

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            tc::mbar_init(x_full + 8 * s, 1);
            tc::mbar_init(w_full + 8 * s, 1);
            tc::mbar_init(empty + 8 * s, 1);
        }
        for (int a = 0; a < kASlots; ++a) {
            tc::mbar_init(a_full + 8 * a, 4);
            tc::mbar_init(a_empty + 8 * a, 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(d_full + 8 * b, 1);
            tc::mbar_init(d_empty + 8 * b, 8);
        }
        tc::mbar_init(y_done, 8);
        tc::mbar_init_fence();
        tc::prefetch_tensormap(&xmap);
        if (p.ystore) tc::prefetch_tensormap(&omap);
    }
    if (warp == 1) tc::tmem_alloc(tc::smem_addr(&tmem_base_sh), kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base_sh;

    // Each role runs under its warpgroup's register limit: the limit is set
    // in the same branch as the role's code.
    if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsIssue));
    if (warp == 0 || warp == 3) {
        // ---- producers: warp 0 the x tile (TMA), warp 3 the group's packed tiles ----
        // (two threads: one thread issuing all ten copies of a group took ~560 ns, near the group's MMA time)
        if (lane == 0) {
            const bool xs = warp == 0;
            const uint32_t full = xs ? x_full : w_full;
            int issued = 0;
            bool ok = true;
            uint32_t ends = 0;  // bit s: the group last loaded into stage s ended its tile
            int ydone = 0;      // tile ends whose y the promote warps have stored out of their stage
            for (int t = blockIdx.x; ok && t < p.tiles; t += gridDim.x) {
                const TileAt tl = tile_at(p, t, kBN);
                for (int it = 0; it < tl.ng; ++it) {
                    const int s = issued % kStages;
                    const uint32_t ph = (issued / kStages) & 1;
                    if (!tc::mbar_wait(empty + 8 * s, ph ^ 1)) {
                        atomicOr(p.status, 1);
                        ok = false;
                        break;
                    }
                    if (xs && p.ystore && ((ends >> s) & 1)) {
                        // the stage held a tile's y: wait until its TMA stores have read it (tile ends are
                        // >= kStages groups apart, so the one barrier's phases come in order)
                        if (!tc::mbar_wait(y_done, ydone & 1)) {
                            atomicOr(p.status, 1);
                            ok = false;
                            break;
                        }
                        ++ydone;
                    }
                    ends = (ends & ~(1u << s)) | ((it == tl.ng - 1 ? 1u : 0u) << s);
                    if (xs) {
                        const uint32_t dst = tc::smem_addr(sB + s * kBStage);
                        tc::mbar_arrive_expect_tx(x_full + 8 * s, kBStage);
                        const int k0 = (tl.g_lo + it) * 128;
                        tc::tma_load_2d(dst, &xmap, k0, tl.tok0, x_full + 8 * s);
                        tc::tma_load_2d(dst + kBStage / 2, &xmap, k0 + 64, tl.tok0, x_full + 8 * s);
                    } else {
                        // the group's packed tiles of the tile's 8 bands in one 2-D copy (rows = bands, 1056
                        // bytes each; rows past the last band are zero-filled and never read)
                        tc::mbar_arrive_expect_tx(w_full + 8 * s, (uint32_t)kWStage);
                        tc::tma_load_2d(tc::smem_addr(sW + s * kWStage), &wmap, (tl.g_lo + it) * (kTileBytes / 8),
                                        tl.band0, w_full + 8 * s);
                    }
                    ++issued;
                }
            }
            // drain: the last loads of every stage have landed before the CTA exits
            for (int it = issued - 1; it >= 0 && it >= issued - kStages; --it)
                if (!tc::mbar_wait(full + 8 * (it % kStages), (it / kStages) & 1)) atomicOr(p.status, 2);
        }
    } else if (warp == 1 || warp == 2) {
        // ---- MMA issuers: warp 1 the even groups (accumulator 0, A slot 0), warp 2 the odd ones ----
        // One thread issuing every group left the tensor pipe idle between groups (the 8 MMAs are
        // accepted only as fast as they run, and the next group's waits and commits came after
        // them: 717 ns per group for 457 ns of MMAs); with two, one waits while the other issues.
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_f16_f32(kBM, kBN);
            int done = 0, ngrp = 0;  // groups of this CTA's tiles so far
            for (int t = blockIdx.x; t < p.tiles; t += gridDim.x) ngrp += tile_at(p, t, kBN).ng;
            for (int it = warp - 1; it < ngrp; it += 2) {
                const int s = it % kStages, a = it % kASlots, b = it & 1;
                const uint32_t ph = (it / kStages) & 1, aph = (it / kASlots) & 1;
                // accumulator b was read out (two groups back) by the promote warps
                if (!tc::mbar_wait(x_full + 8 * s, ph) || !tc::mbar_wait(a_full + 8 * a, aph) ||
                    !tc::mbar_wait(d_empty + 8 * b, ((it >> 1) & 1) ^ 1)) {
                    atomicOr(p.status, 4);
                    break;
                }
                tc::fence_after_sync();
                const uint32_t a0 = tmem + kACol0 + 64 * a, b0 = tc::smem_addr(sB + s * kBStage);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t off = (j >> 2) * (kBStage / 2) + (j & 3) * 32;
                    tc::mma_f16_ta(tmem + b * kBN, a0 + 8 * j, tc::sw128_kmajor_desc(b0 + off), idesc, j > 0);
                }
                tc::mma_commit(empty + 8 * s);
                tc::mma_commit(a_empty + 8 * a);
                tc::mma_commit(d_full + 8 * b);
                done = it + 1;
            }
            // drain: every issued MMA has completed before TMEM is released
            if (done > 0 && !tc::mbar_wait(d_full + 8 * ((done - 1) & 1), ((done - 1) >> 1) & 1))
                atomicOr(p.status, 8);
        }
    }
    } else if (warp < 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsDequant));
    {
        // ---- dequant: 2 bands per warp, TMEM lanes 32*dw .. 32*dw + 31 -------
        const int dw = warp - 4;
        int gi = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < p.tiles; t += gridDim.x) {
          const int band0 = tile_at(p, t, kBN).band0, ng = tile_at(p, t, kBN).ng;
          for (int it = 0; it < ng; ++it, ++gi) {
            const int s = gi % kStages, a = gi % kASlots;
            const uint32_t ph = (gi / kStages) & 1, aph = (gi / kASlots) & 1;
            // the packed tiles have landed: unpack them into registers, and only then wait for the A
            // slot (the MMAs that read it kASlots groups back have completed), so that refilling the
            // slot takes only the stores (the issuers had waited ~320 ns per group for the A slot;
            // layer at 512 tokens 264.8 -> 258.2 us)
            if (!tc::mbar_wait(w_full + 8 * s, ph)) {
                atomicOr(p.status, 16);
                ok = false;
                break;
            }
            uint32_t q16[2][32];  // per band: k 0..63 (registers 0..15) then k 64..127
#pragma unroll
            for (int bi = 0; bi < 2; ++bi) {
                uint4 lo, hi;
                if (band0 + 2 * dw + bi < p.bands) {
                    const uint32_t t = tc::smem_addr(sW + s * kWStage + (2 * dw + bi) * kTileBytes);
                    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                                 : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w)
                                 : "r"(t + 16 * lane));
                    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                                 : "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
                                 : "r"(t + 512 + 16 * lane));
                } else {
                    lo = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);  // q = 0
                    hi = lo;
                }
                // K step j -> columns 8j .. 8j+7: lane (r, c) holds rows r and
                // r + 8, k pairs 2c and 2c + 1 of the step; two stores of four
                // steps (k 0..63 from lo, 64..127 from hi)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint4 wv = h ? hi : lo;
                    const uint32_t wd[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t q4[4];
                        unpack_word(wd[j], q4);
                        q16[bi][16 * h + 4 * j + 0] = q4[0];
                        q16[bi][16 * h + 4 * j + 1] = q4[2];
                        q16[bi][16 * h + 4 * j + 2] = q4[1];
                        q16[bi][16 * h + 4 * j + 3] = q4[3];
                    }
                }
            }
            if (!tc::mbar_wait(a_empty + 8 * a, aph ^ 1)) {
                atomicOr(p.status, 16);
                ok = false;
                break;
            }
            tc::fence_after_sync();
#pragma unroll
            for (int bi = 0; bi < 2; ++bi) {
                const uint32_t taddr = tmem + ((uint32_t)(32 * dw + 16 * bi) << 16) + kACol0 + 64 * a;
                tmem_st_16x256_x8(taddr, q16[bi]);
            }
            tc::tmem_wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(a_full + 8 * a);
          }
        }
    }
    } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
    {
        // ---- promote + epilogue -------------------------------------------------
        const int quarter = warp & 3, half = (warp - 8) >> 2;
        const int row = 32 * quarter + lane;  // TMEM lane = weight row within the tile
        const int rr = row & 15;
        constexpr int kCols = kBN / 2;  // tokens of this thread: the warp's half of the tile
        int gi = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < p.tiles; t += gridDim.x) {
            const TileAt tl = tile_at(p, t, kBN);
            const int bandg = tl.band0 + (row >> 4);
            const bool row_ok = bandg < p.bands;
            const uint8_t* sc =
                p.w + (size_t)bandg * p.G * kTileBytes + kScaleOffset + 4 * (rr & 7) + 2 * (rr >> 3);
            float acc[kCols];
#pragma unroll
            for (int i = 0; i < kCols; ++i) acc[i] = 0.f;
            auto scale_of = [&](int it) -> float {
                if (!row_ok) return 0.f;
                const unsigned short h =
                    __ldg(reinterpret_cast<const unsigned short*>(sc + (size_t)(tl.g_lo + it) * kTileBytes));
                return __half2float(__ushort_as_half(h));
            };
            // scales two groups ahead of the accumulator they multiply
            float s_cur = tl.ng > 0 ? scale_of(0) : 0.f;
            float s_nxt = tl.ng > 1 ? scale_of(1) : 0.f;
            for (int it = 0; it < tl.ng; ++it, ++gi) {
                const int b = gi & 1;
                const float s_far = (it + 2 < tl.ng) ? scale_of(it + 2) : 0.f;
                if (!tc::mbar_wait(d_full + 8 * b, (gi >> 1) & 1)) {
                    atomicOr(p.status, 32);
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t taddr = tmem + ((uint32_t)(32 * quarter) << 16) + b * kBN + kCols * half;
                // a 64-column piece per tensor-memory wait (one at a time, three waits per group at 192
                // tokens held the accumulator ~100 ns longer), in one load instruction: every group's
                // tensor-memory loads and stores share the tensor pipe with its MMAs
                static_assert(kCols == 64 || kCols == 96, "promote pieces");
                uint32_t v[64];
                tmem_ld_32x32_x64(taddr, v);
                tc::tmem_wait_ld();
                if (kCols == 64) {
                    // the whole partial is in registers: hand the accumulator back
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(d_empty + 8 * b);
                }
#pragma unroll
                for (int i = 0; i < 64; ++i) acc[i] = fmaf(s_cur, __uint_as_float(v[i]), acc[i]);
                if (kCols == 96) {
                    uint32_t w3[32];
                    tc::tmem_ld_32x32(taddr + 64, w3);
                    tc::tmem_wait_ld();
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(d_empty + 8 * b);
#pragma unroll
                    for (int i = 0; i < 32; ++i) acc[64 + i] = fmaf(s_cur, __uint_as_float(w3[i]), acc[64 + i]);
                }
                s_cur = s_nxt;
                s_nxt = s_far;
            }
            const int n = tl.band0 * 16 + row;
            if (ok && p.ystore) {
                // y (or the split's FP32 partial) through the x stage of the tile's last group (its
                // MMAs are done): this warp's 32 rows x kCols tokens into its slice, TMA stores, and
                // once they have read it the x producer may refill the stage (a thread's kCols
                // separate global stores had held the promote warps 2-4 us per tile, the next tile's
                // MMAs waiting for the accumulators meanwhile).  The slice's shared address is
                // recomputed from the array here: keeping the stages' base pointer live through the
                // group loop spilled a register.
                const uint32_t slice = ((tc::smem_addr(smem_raw) + 1023u) & ~1023u) +
                                       (uint32_t)(((gi - 1) % kStages) * kBStage + (warp - 8) * (32 * kCols * 2));
                const int n0 = tl.band0 * 16 + 32 * quarter, t0 = tl.tok0 + kCols * half;
                if (p.part == nullptr) {
                    // fp16 y: [token][32 rows], one store of 32 rows x kCols tokens
#pragma unroll
                    for (int i = 0; i < kCols; ++i)
                        asm volatile("st.shared.u16 [%0], %1;" ::"r"(slice + 2 * lane + 64 * i),
                                     "h"(__half_as_ushort(__float2half_rn(acc[i])))
                                     : "memory");
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && n0 < p.N && t0 < p.M) {
                        tma_store_2d(&omap, slice, n0, t0);
                        bulk_commit_group();
                    }
                } else {
                    // FP32 partial: the slice holds half the warp's tokens, so two rounds of
                    // [token][32 rows] and a store each (the partials are [split][M][N]: tokens
                    // past M are clipped, not written into the next split's rows)
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        if (r == 1) {
                            if (lane == 0) bulk_wait_read_all();
                            __syncwarp();
                        }
#pragma unroll
                        for (int i = 0; i < kCols / 2; ++i)
                            asm volatile("st.shared.f32 [%0], %1;" ::"r"(slice + 4 * lane + 128 * i),
                                         "f"(acc[r * (kCols / 2) + i])
                                         : "memory");
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0 && n0 < p.N && t0 + r * (kCols / 2) < p.M) {
                            tma_store_3d(&omap, slice, n0, t0 + r * (kCols / 2), tl.split);
                            bulk_commit_group();
                        }
                    }
                }
                if (lane == 0) {
                    bulk_wait_read_all();
                    tc::mbar_arrive(y_done);
                }
            } else if (ok && row_ok && n < p.N) {
                const int t0 = tl.tok0 + kCols * half;
                if (p.part == nullptr) {
#pragma unroll
                    for (int i = 0; i < kCols; ++i)
                        if (t0 + i < p.M) p.y[(size_t)(t0 + i) * p.N + n] = __half_as_ushort(__float2half_rn(acc[i]));
                } else {
                    float* dst = p.part + (size_t)tl.split * p.M * p.N;
#pragma unroll
                    for (int i = 0; i < kCols; ++i)
                        if (t0 + i < p.M) dst[(size_t)(t0 + i) * p.N + n] = acc[i];
                }
            }
        }
        if (lane == 0) bulk_wait_all();  // the y stores are done before the slices go away
    }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// Fixed-order sum of the split-K partials: y = fp16(sum_s part[s]), four
// outputs per thread and step (16-byte loads of every split, one 8-byte
// store) when count is a multiple of 4, else one at a time.
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ part, int splits, size_t count,
                                                            uint16_t* __restrict__ y) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    if (count % 4 == 0) {
        const size_t n4 = count / 4;
        const float4* p4 = reinterpret_cast<const float4*>(part);
        for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += stride) {
            float4 s = __ldcg(p4 + i);
            for (int k = 1; k < splits; ++k) {
                const float4 v = __ldcg(p4 + (size_t)k * n4 + i);
                s.x += v.x;
                s.y += v.y;
                s.z += v.z;
                s.w += v.w;
            }
            const uint32_t lo = (uint32_t)__half_as_ushort(__float2half_rn(s.x)) |
                                ((uint32_t)__half_as_ushort(__float2half_rn(s.y)) << 16);
            const uint32_t hi = (uint32_t)__half_as_ushort(__float2half_rn(s.z)) |
                                ((uint32_t)__half_as_ushort(__float2half_rn(s.w)) << 16);
            reinterpret_cast<uint2*>(y)[i] = make_uint2(lo, hi);
        }
        return;
    }
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < count; i += stride) {
        float s = part[i];
        for (int k = 1; k < splits; ++k) s += part[(size_t)k * count + i];
        y[i] = __half_as_ushort(__float2half_rn(s));
    }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// Tile width and K splits of one call, from a cost in units of one group's
// work on one SM at the 192-token width (~0.9 us measured): waves of CTAs
// (the device's SMs) x groups per CTA x the width's relative group time (a 128-token
// group measured 0.89 of a 192-token one), plus, for s > 1, the FP32
// partials written and read back by the reduce (8 bytes per output and split,
// ~6.2 MB of HBM traffic per unit).  Each split keeps >= 4 groups.  At
// M = 512 this picks 128-token tiles for qkv and o (more CTAs busy) and 192
// for gate_up and down.
struct GemmPlan {
    int bn, splits;
};
GemmPlan gemm_plan(int M, int64_t N, int64_t K) {
    const int G = (int)(K / kGroupK);
    const int sms = device_sm_count();
    GemmPlan best{192, 1};
    double best_t = 1e300;
    for (int bn : {192, 128}) {
        const int64_t tiles = ((N + kBM - 1) / kBM) * ((M + bn - 1) / bn);
        const double rel = bn == 128 ? 0.89 : 1.0;
        for (int s = 1; s <= 16 && (G + s - 1) / s >= 4; ++s) {
            const double waves = (double)((tiles * s + sms - 1) / sms);
            const double t =
                waves * ((G + s - 1) / s) * rel + (s > 1 ? (double)s * M * (double)N * 8.0 / 6.2e6 : 0.0);
            if (t < best_t - 1e-9) {
                best_t = t;
                best = GemmPlan{bn, s};
            }
        }
    }
    return best;
}

size_t gemm_workspace(int M, int64_t N, int64_t K) {
    const int s = gemm_plan(M, N, K).splits;
    return kStatusBytes + (s > 1 ? (size_t)s * M * N * sizeof(float) : 0);
}

// Raise the prefill kernel's dynamic shared-memory limit on the current
// device.  The attribute belongs to the (device, kernel) pair, so it is set
// once per device for each tile width; a failed attempt is not remembered and
// is retried on the next call.
template <int BN>
w4_status allow_tile_smem() {
    static std::mutex mu;
    static bool done[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) {
        set_error("device ordinal %d out of range", dev);
        return W4_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev]) return W4_OK;
    e = cudaFuncSetAttribute(gemm_tc_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, Tile<BN>::kSmemBytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(prefill)");
    done[dev] = true;
    return W4_OK;
}

template <int BN>
w4_status launch_tile(const CUtensorMap& map, const CUtensorMap& wmap, const CUtensorMap& omap, const GemmParams& p,
                      cudaStream_t stream) {
    const w4_status st = allow_tile_smem<BN>();
    if (st != W4_OK) return st;
    GemmParams q = p;
    q.tiles_x = (p.M + BN - 1) / BN;
    q.tiles_y = (p.N + kBM - 1) / kBM;
    q.tiles = q.tiles_x * q.tiles_y * p.splits;
    // persistent: one CTA per SM (or per tile, if fewer), each walking its tiles in turn
    const unsigned ctas = (unsigned)std::min(q.tiles, device_sm_count());
    gemm_tc_kernel<BN><<<ctas, kThreads, Tile<BN>::kSmemBytes, stream>>>(map, wmap, omap, q);
    W4_CUDA_TRY(cudaGetLastError());
    return W4_OK;
}

}  // namespace

w4_status launch_gemm_tc(const void* x, const w4_weight* w, void* y, int M, void* ws, size_t ws_bytes,
                         cudaStream_t stream) {
    const size_t need = gemm_workspace(M, w->N, w->K);
    if (!ws || ws_bytes < need) {
        set_error("workspace of %zu bytes needed (got %zu)", need, ws_bytes);
        return W4_ERR_WORKSPACE;
    }
    if (!aligned16(ws)) {
        set_error("workspace not 16-byte aligned");
        return W4_ERR_ALIGN;
    }
    if (w->N > 0x7FFFFFF0 || w->K > 0x7FFFFFF0 || (int64_t)M * w->N > ((int64_t)1 << 40)) {
        set_error("shape too large");
        return W4_ERR_SHAPE;
    }
    auto encode = tensor_map_encoder();
    if (!encode) {
        set_error("cuTensorMapEncodeTiled is not available from the driver");
        return W4_ERR_UNSUPPORTED;
    }
    const GemmPlan plan = gemm_plan(M, w->N, w->K);
    CUtensorMap map;
    const cuuint64_t gdim[2] = {(cuuint64_t)w->K, (cuuint64_t)M};
    const cuuint64_t gstride[1] = {(cuuint64_t)w->K * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)plan.bn};
    const cuuint32_t estride[2] = {1, 1};
    CUresult cr = encode(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(x), gdim, gstride, box, estride,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed (%d)", (int)cr);
        return W4_ERR_CUDA;
    }
    // the packed weight as rows of bands (G tiles of 1056 bytes each, in 8-byte
    // elements): a box of 8 bands x one tile is a group's tiles for one CTA
    CUtensorMap wmap;
    const int64_t G = num_groups(w->K), bands = num_bands(w->N);
    const cuuint64_t wdim[2] = {(cuuint64_t)(G * (kTileBytes / 8)), (cuuint64_t)bands};
    const cuuint64_t wstride[1] = {(cuuint64_t)(G * kTileBytes)};
    const cuuint32_t wbox[2] = {(cuuint32_t)(kTileBytes / 8), 8};
    cr = encode(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(w->data), wdim, wstride, wbox, estride,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled (weight) failed (%d)", (int)cr);
        return W4_ERR_CUDA;
    }
    // The tiles' output for the TMA stores: y [M][N] fp16 (a box is one promote warp's 32 rows x half a
    // tile's tokens), or with K split the FP32 partials [splits][M][N] (a box is 32 rows x a quarter of
    // the tokens).  Only where every tile has at least 4 groups (one per stage: tile ends then come at
    // least a stage cycle apart) and the tensor can be mapped (row stride a multiple of 16 bytes, base
    // 16-byte aligned); otherwise the promote warps store the output themselves.
    const int64_t Gk = num_groups(w->K);
    CUtensorMap omap = wmap;
    const bool ostore = Gk >= 4 * (int64_t)plan.splits &&
                        (plan.splits == 1 ? w->N % 8 == 0 && aligned16(y) : w->N % 4 == 0);
    if (ostore && plan.splits == 1) {
        const cuuint64_t ydim[2] = {(cuuint64_t)w->N, (cuuint64_t)M};
        const cuuint64_t ystride[1] = {(cuuint64_t)w->N * 2};
        const cuuint32_t ybox[2] = {32, (cuuint32_t)(plan.bn / 2)};
        cr = encode(&omap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, y, ydim, ystride, ybox, estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else if (ostore) {
        const cuuint64_t pdim[3] = {(cuuint64_t)w->N, (cuuint64_t)M, (cuuint64_t)plan.splits};
        const cuuint64_t pstride[2] = {(cuuint64_t)w->N * 4, (cuuint64_t)M * w->N * 4};
        const cuuint32_t pbox[3] = {32, (cuuint32_t)(plan.bn / 4), 1};
        const cuuint32_t pestride[3] = {1, 1, 1};
        cr = encode(&omap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, static_cast<char*>(ws) + kStatusBytes, pdim, pstride,
                    pbox, pestride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (ostore && cr != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled (output) failed (%d)", (int)cr);
        return W4_ERR_CUDA;
    }
    GemmParams p;
    p.ystore = ostore ? 1 : 0;
    p.w = static_cast<const uint8_t*>(w->data);
    p.y = static_cast<uint16_t*>(y);
    p.status = static_cast<int*>(ws);
    p.M = M;
    p.N = (int)w->N;
    p.K = (int)w->K;
    p.G = (int)num_groups(w->K);
    p.bands = (int)num_bands(w->N);
    p.splits = plan.splits;
    p.part = p.splits > 1 ? reinterpret_cast<float*>(static_cast<char*>(ws) + kStatusBytes) : nullptr;

    W4_CUDA_TRY(cudaMemsetAsync(ws, 0, sizeof(int), stream));
    const w4_status st =
        plan.bn == 128 ? launch_tile<128>(map, wmap, omap, p, stream) : launch_tile<192>(map, wmap, omap, p, stream);
    if (st != W4_OK) return st;
    if (p.splits > 1) {
        const size_t count = (size_t)M * p.N;
        size_t blocks = (count % 4 == 0 ? count / 4 + 255 : count + 255) / 256;
        const size_t cap = (size_t)device_sm_count() * 16;  // enough resident blocks to cover every SM
        if (blocks > cap) blocks = cap;
        splitk_reduce_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p.part, p.splits, count, p.y);
        W4_CUDA_TRY(cudaGetLastError());
    }
    return W4_OK;
}

}  // namespace w4

// ---- prefill without a caller workspace -------------------------------------
// Some callers cannot allocate device memory at all (a plugin whose host
// framework owns every device allocation, or code that must not call
// cudaMalloc because it can synchronise the device or fail at a memory cap),
// so they cannot provide the prefill kernel's workspace.  For them the
// workspace lives in this file-scope array: the CUDA module reserves it on
// every device that loads the library, for the life of the process.
namespace w4 {
namespace {

__device__ __align__(256) unsigned char g_static_scratch[W4_STATIC_SCRATCH_BYTES];

// Device address of g_static_scratch on the current device, looked up once per
// device (with that device current).  In host code the array's name is only a
// host-side stand-in, never a device address.
w4_status static_scratch_address(void** out) {
    static std::mutex mu;
    static void* addr[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) {
        set_error("device ordinal %d out of range", dev);
        return W4_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
        addr[dev] = p;
    }
    *out = addr[dev];
    return W4_OK;
}

}  // namespace
}  // namespace w4

using namespace w4;

extern "C" w4_status w4a16_gemm_static_scratch(const void* x, const w4_weight* w, void* y, int M, void* stream) {
    clear_error();
    if (M < 1) {
        set_error("M=%d: need M >= 1", M);
        return W4_ERR_SHAPE;
    }
    w4_status st = check_gemv_args(x, w, y, M < 16 ? M : 16);
    if (st != W4_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (M <= 16) {  // the decode kernel needs no scratch at all
        w4_gemv_config c;
        default_gemv_config(M, w->N, w->K, &c);
        return launch_gemv(x, w, y, M, c, s);
    }
    const size_t need = gemm_workspace(M, w->N, w->K);
    if (need > W4_STATIC_SCRATCH_BYTES) {
        set_error("M=%d N=%lld K=%lld needs %zu bytes of scratch; the static scratch holds %zu "
                  "(use w4a16_gemm with a workspace)",
                  M, (long long)w->N, (long long)w->K, need, (size_t)W4_STATIC_SCRATCH_BYTES);
        return W4_ERR_WORKSPACE;
    }
    void* scratch = nullptr;
    st = static_scratch_address(&scratch);
    if (st != W4_OK) return st;
    return launch_gemm_tc(x, w, y, M, scratch, W4_STATIC_SCRATCH_BYTES, s);
}

extern "C" int w4a16_gemm_static_scratch_status(void) {
    clear_error();
    void* scratch = nullptr;
    if (static_scratch_address(&scratch) != W4_OK) return -1;
    int v = 0;
    const cudaError_t e = cudaMemcpy(&v, scratch, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) {
        cuda_fail(e, "cudaMemcpy(static scratch status)");
        return -1;
    }
    return v;
}

extern "C" size_t w4_workspace_bytes(int M, int64_t N, int64_t K) {
    if (M <= 16 || N < 1 || K < kGroupK || K % kGroupK != 0) return 0;
    return gemm_workspace(M, N, K);
}

extern "C" w4_status w4a16_gemm(const void* x, const w4_weight* w, void* y, int M, void* workspace,
                                size_t workspace_bytes, void* stream) {
    clear_error();
    if (M < 1) {
        set_error("M=%d: need M >= 1", M);
        return W4_ERR_SHAPE;
    }
    w4_status st = check_gemv_args(x, w, y, M < 16 ? M : 16);
    if (st != W4_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (M <= 16) {
        w4_gemv_config c;
        default_gemv_config(M, w->N, w->K, &c);
        return launch_gemv(x, w, y, M, c, s);
    }
    return launch_gemm_tc(x, w, y, M, workspace, workspace_bytes, s);
}
