// Internal helpers of libw4.so: error reporting, packed-layout constants and
// small device primitives shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdarg>
#include <cstdio>
#include <string>

#include "w4.h"

namespace w4 {

// ---- packed layout ------------------------------------------------------
// A tile is 16 rows x 128 K: 1024 bytes of nibbles, then 8 words of paired
// fp16 scales (rows p and p + 8).  Tiles of one 16-row band are contiguous
// along K.
constexpr int kGroupK = 128;
constexpr int kBandRows = 16;
constexpr int kTileNibbleBytes = 1024;
constexpr int kTileBytes = 1056;
constexpr int kScaleOffset = 1024;

inline int64_t num_bands(int64_t N) { return (N + kBandRows - 1) / kBandRows; }
inline int64_t num_groups(int64_t K) { return K / kGroupK; }

// ---- errors --------------------------------------------------------------
void set_error(const char* fmt, ...);
void clear_error();
w4_status cuda_fail(cudaError_t e, const char* what);

#define W4_CUDA_TRY(expr)                                   \
    do {                                                    \
        cudaError_t _e = (expr);                            \
        if (_e != cudaSuccess) return ::w4::cuda_fail(_e, #expr); \
    } while (0)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

w4_status check_weight(const w4_weight* w);

// ---- devices ---------------------------------------------------------------
// Device ordinals the per-device caches of the library cover.
constexpr int kMaxDevices = 64;
// SM count assumed when no device can be queried (a GB300 has 152).
constexpr int kDefaultSms = 152;
// SM count of the current device, looked up once per device; kDefaultSms
// when no device is available (host-only planning).
int device_sm_count();

// ---- device primitives -----------------------------------------------------
// Programmatic dependent launch: wait for the previous grid on the stream to
// finish (and its memory to be visible), and allow the next grid to start.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace w4
