// Launch state of the persistent decode-step kernel (step.cu), shared with
// the sequence front end (seq.cu).
#pragma once

#include <cuda_runtime.h>

#include "w4.h"

namespace w4 {

struct StepOp;

struct StepParams {
    const StepOp* ops;
    int nops, M;
    unsigned* done;      // [nops] CTAs finished with each projection
    unsigned* exit_cnt;  // CTAs finished with the step
    int* status;         // set non-zero when a wait gives up
    int gpc_max;         // largest x slice (groups): shared-memory sizing
    int ring;            // ring slots (tiles) per warp
};

using StepFn = void (*)(StepParams);

struct StepLaunch {
    StepFn fn = nullptr;
    StepParams params{};
    int NC = 0, smem = 0;
};

w4_status step_prepare(const w4_weight* w, const void* const* x, void* const* y, int n, int M, void* ws,
                       size_t ws_bytes, cudaStream_t stream, StepLaunch* out);
w4_status step_launch(const StepLaunch& s, cudaStream_t stream);
int step_status(const StepLaunch& s);
size_t step_workspace_bytes(const w4_weight* w, int n, int M);

}  // namespace w4
