// Device side of the seeded input generators (see synth/__init__.py for the
// definition).  Draws q and fp16 scales for large synthetic weights directly
// in device memory; the host generator yields identical bits for any element.
// No projection arithmetic here: random draws only.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t draw(uint64_t seed, uint64_t i) {
    return mix64(seed + (i + 1ull) * 0x9E3779B97F4A7C15ull);
}

__global__ void q_kernel(uint64_t seed, int64_t first, int64_t n, int8_t* out) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        out[i] = (int8_t)((int)(draw(seed, (uint64_t)(first + i)) >> 60) - 8);
}

__global__ void scale_kernel(uint64_t seed, int64_t first, int64_t n, uint16_t* out) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const double u = (double)(draw(seed, (uint64_t)(first + i)) >> 11) * 0x1p-53;
        const double v = __dadd_rn(0.005, __dmul_rn(0.015, u));  // two roundings, never fused
        out[i] = __half_as_ushort(__double2half(v));
    }
}

int launch_dims(int64_t n) {
    int64_t b = (n + 255) / 256;
    if (b > 65536) b = 65536;
    return b < 1 ? 1 : (int)b;
}

}  // namespace

// q[first .. first+n) of the tensor with this seed, written to out[0 .. n).
extern "C" int synth_q_device(uint64_t seed, int64_t first, int64_t n, int8_t* out, void* stream) {
    if (n <= 0) return 0;
    q_kernel<<<launch_dims(n), 256, 0, (cudaStream_t)stream>>>(seed, first, n, out);
    return (int)cudaGetLastError();
}

// fp16 bit patterns of s[first .. first+n).
extern "C" int synth_scale_device(uint64_t seed, int64_t first, int64_t n, uint16_t* out, void* stream) {
    if (n <= 0) return 0;
    scale_kernel<<<launch_dims(n), 256, 0, (cudaStream_t)stream>>>(seed, first, n, out);
    return (int)cudaGetLastError();
}
