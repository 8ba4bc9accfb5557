// Prefill projection y[M, N] = x[M, K] . W^T for any M >= 1.
//
// M <= 16 goes to the decode kernel.  Larger M is processed as consecutive
// 16-token slices of the decode kernel, each reading the whole weight again.
#include "w4_internal.cuh"

namespace w4 {
void default_gemv_config(int M, int64_t N, int64_t K, w4_gemv_config* c);
w4_status launch_gemv(const void* x, const w4_weight* w, void* y, int M, const w4_gemv_config& c,
                      cudaStream_t stream);
w4_status check_gemv_args(const void* x, const w4_weight* w, const void* y, int M);
}  // namespace w4

using namespace w4;

extern "C" w4_status w4a16_gemm(const void* x, const w4_weight* w, void* y, int M, void* workspace,
                                size_t workspace_bytes, void* stream) {
    (void)workspace;
    (void)workspace_bytes;
    clear_error();
    if (M < 1) {
        set_error("M=%d: need M >= 1", M);
        return W4_ERR_SHAPE;
    }
    const int first = M < 16 ? M : 16;
    w4_status st = check_gemv_args(x, w, y, first);
    if (st != W4_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (int m0 = 0; m0 < M; m0 += 16) {
        const int mc = (M - m0) < 16 ? (M - m0) : 16;
        const char* xs = static_cast<const char*>(x) + (size_t)m0 * w->K * 2;
        char* ys = static_cast<char*>(y) + (size_t)m0 * w->N * 2;
        // slices after the first start at row m0 of x and y: 16-byte aligned
        // whenever K and N are multiples of 8 (always true for K)
        if (!aligned16(ys)) {
            set_error("y row %d is not 16-byte aligned (N=%lld)", m0, (long long)w->N);
            return W4_ERR_ALIGN;
        }
        w4_gemv_config c;
        default_gemv_config(mc, w->N, w->K, &c);
        st = launch_gemv(xs, w, ys, mc, c, s);
        if (st != W4_OK) return st;
    }
    return W4_OK;
}
