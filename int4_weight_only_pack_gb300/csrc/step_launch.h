// Launch state of the persistent decode-step kernel (step.cu), shared with
// the sequence front end (seq.cu).
#pragma once

#include <cuda_runtime.h>

#include <vector>

#include "w4.h"

namespace w4 {

// Projections one persistent launch can carry (its table travels in the
// kernel's parameter space).
constexpr int kMaxStepOps = 448;

struct StepLaunch {
    const void* fn = nullptr;
    std::vector<unsigned char> args;  // the kernel's parameter block
    int* status = nullptr;            // device status word
    int NC = 0, smem = 0;
};

// act: 0 binary16 activations, 1 bfloat16; op_flags: W4_OP_* per projection (may be NULL).
w4_status step_prepare(const w4_weight* w, const void* const* x, void* const* y, const uint32_t* op_flags, int n,
                       int M, int act, void* ws, size_t ws_bytes, cudaStream_t stream, StepLaunch* out);
w4_status step_launch(const StepLaunch& s, cudaStream_t stream);
int step_status(const StepLaunch& s);
size_t step_workspace_bytes(const w4_weight* w, int n, int M);
// K split per projection of the plan the current device would run.
void step_splits(const w4_weight* w, int n, int M, int act, bool gated, int* splits);

}  // namespace w4
