// Decode-step sequence: the projections of every decoder layer (qkv, o,
// gate_up, down for each of the 28 layers = 112 launches), captured once as a
// CUDA graph and replayed with a single cudaGraphLaunch.
//
// The pages' runtime went from ~119 ms/token with eager per-kernel launches to
// ~17 ms/token once the whole decode step was a captured graph ("Building a
// Custom LLM Inference Runtime ...", "The Impact of CUDA Graphs"; "The
// Architecture of Modern Inference ...", "Eliminating Host Overhead with CUDA
// Graphs").  Here the chain is a straight line, so one static graph suffices
// (the pages' second graph exists only for paged-KV page crossings).  When
// use_pdl is set, consecutive launches carry the programmatic-stream-
// serialization attribute: capture turns them into programmatic edges, and
// each projection starts streaming its weights while its predecessor drains.
#include <vector>

#include "w4_internal.cuh"

namespace w4 {
void default_gemv_config(int M, int64_t N, int64_t K, w4_gemv_config* c);
w4_status launch_gemv(const void* x, const w4_weight* w, void* y, int M, const w4_gemv_config& c,
                      cudaStream_t stream);
w4_status check_gemv_args(const void* x, const w4_weight* w, const void* y, int M);
w4_status prepare_gemv(const w4_weight* w, int M, const w4_gemv_config& c);

// persistent decode-step kernel (step.cu)
struct StepLaunch;
size_t step_workspace_bytes(const w4_weight* w, int n, int M);
}  // namespace w4

#include "step_launch.h"

struct w4_seq {
    int n = 0, M = 0;
    bool persistent = false;
    std::vector<w4_weight> w;
    std::vector<const void*> x;
    std::vector<void*> y;
    std::vector<w4_gemv_config> cfg;
    w4::StepLaunch step;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    // w4_decode_seq_run_host: copy in, the step, copy out as one graph, kept for the
    // buffers it was built for
    cudaGraphExec_t io_exec = nullptr;
    const void* io_xh = nullptr;
    void* io_xd = nullptr;
    void* io_yd = nullptr;
    void* io_yh = nullptr;
    size_t io_xb = 0, io_yb = 0;
};

using namespace w4;

static w4_status enqueue_all(w4_seq* s, cudaStream_t stream) {
    if (s->persistent) return step_launch(s->step, stream);
    for (int i = 0; i < s->n; ++i) {
        w4_status st = launch_gemv(s->x[i], &s->w[i], s->y[i], s->M, s->cfg[i], stream);
        if (st != W4_OK) return st;
    }
    return W4_OK;
}

extern "C" void w4_decode_seq_destroy(w4_seq* seq) {
    if (!seq) return;
    if (seq->io_exec) cudaGraphExecDestroy(seq->io_exec);
    if (seq->exec) cudaGraphExecDestroy(seq->exec);
    if (seq->graph) cudaGraphDestroy(seq->graph);
    delete seq;
}

extern "C" w4_status w4_decode_seq_create(const w4_weight* w, const void* const* x, void* const* y, int n, int M,
                                          int use_pdl, void* stream, w4_seq** out) {
    clear_error();
    if (!w || !x || !y || !out || n < 1) {
        set_error("NULL argument or n < 1");
        return W4_ERR_ARG;
    }
    *out = nullptr;
    w4_seq* s = new w4_seq();
    s->n = n;
    s->M = M;
    for (int i = 0; i < n; ++i) {
        w4_status st = check_gemv_args(x[i], &w[i], y[i], M);
        if (st != W4_OK) {
            delete s;
            return st;
        }
        s->w.push_back(w[i]);
        s->x.push_back(x[i]);
        s->y.push_back(y[i]);
        w4_gemv_config c;
        default_gemv_config(M, w[i].N, w[i].K, &c);
        c.pdl = use_pdl ? 1 : 0;
        s->cfg.push_back(c);
    }
    cudaStream_t user = static_cast<cudaStream_t>(stream);
    // Kernel attributes are set before capture begins (not stream operations).
    w4_status st = W4_OK;
    for (int i = 0; i < n && st == W4_OK; ++i) st = prepare_gemv(&s->w[i], M, s->cfg[i]);
    if (st != W4_OK) {
        w4_decode_seq_destroy(s);
        return st;
    }
    cudaStream_t cap = nullptr;
    cudaError_t e = cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking);
    if (e != cudaSuccess) {
        w4_decode_seq_destroy(s);
        return cuda_fail(e, "cudaStreamCreateWithFlags");
    }
    e = cudaStreamSynchronize(user);
    if (e == cudaSuccess) e = cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal);
    if (e == cudaSuccess) {
        st = enqueue_all(s, cap);
        cudaError_t e2 = cudaStreamEndCapture(cap, &s->graph);
        if (st == W4_OK && e2 != cudaSuccess) st = cuda_fail(e2, "cudaStreamEndCapture");
    } else {
        st = cuda_fail(e, "begin capture");
    }
    if (st == W4_OK) {
        e = cudaGraphInstantiateWithFlags(&s->exec, s->graph, 0);
        if (e != cudaSuccess) st = cuda_fail(e, "cudaGraphInstantiate");
    }
    if (st == W4_OK) {
        e = cudaGraphUpload(s->exec, user);
        if (e == cudaSuccess) e = cudaStreamSynchronize(user);
        if (e != cudaSuccess) st = cuda_fail(e, "cudaGraphUpload");
    }
    cudaStreamDestroy(cap);
    if (st != W4_OK) {
        w4_decode_seq_destroy(s);
        return st;
    }
    *out = s;
    return W4_OK;
}

extern "C" w4_status w4_decode_seq_replay(w4_seq* seq, void* stream) {
    if (!seq || (!seq->exec && !seq->persistent)) {
        set_error("sequence is NULL or not instantiated");
        return W4_ERR_ARG;
    }
    if (!seq->exec) return enqueue_all(seq, static_cast<cudaStream_t>(stream));
    cudaError_t e = cudaGraphLaunch(seq->exec, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaGraphLaunch");
    return W4_OK;
}

extern "C" w4_status w4_decode_seq_eager(w4_seq* seq, void* stream) {
    if (!seq) {
        set_error("sequence is NULL");
        return W4_ERR_ARG;
    }
    return enqueue_all(seq, static_cast<cudaStream_t>(stream));
}

extern "C" w4_status w4_decode_seq_run_host(w4_seq* seq, const void* x_host, void* x_dev, size_t x_bytes,
                                            void* y_dev, void* y_host, size_t y_bytes, void* stream) {
    if (!seq || (!seq->exec && !seq->persistent) || (x_bytes && (!x_host || !x_dev)) ||
        (y_bytes && (!y_host || !y_dev))) {
        set_error("NULL argument");
        return W4_ERR_ARG;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool same = seq->io_exec && seq->io_xh == x_host && seq->io_xd == x_dev && seq->io_xb == x_bytes &&
                      seq->io_yd == y_dev && seq->io_yh == y_host && seq->io_yb == y_bytes;
    if (!same) {
        // one graph of the copy in, the step and the copy out, launched as one unit on every
        // later call with the same buffers (961 -> 957 us per call for the 28-layer step: the
        // rest of the ~55 us beyond the step is the two copies themselves); where it cannot be
        // captured the operations are issued one by one
        if (seq->io_exec) cudaGraphExecDestroy(seq->io_exec);
        seq->io_exec = nullptr;
        cudaStream_t cap = nullptr;
        cudaGraph_t g = nullptr;
        cudaError_t e = cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal);
        if (e == cudaSuccess) {
            if (x_bytes) e = cudaMemcpyAsync(x_dev, x_host, x_bytes, cudaMemcpyHostToDevice, cap);
            w4_status st = e == cudaSuccess ? enqueue_all(seq, cap) : W4_ERR_CUDA;
            if (e == cudaSuccess && st == W4_OK && y_bytes)
                e = cudaMemcpyAsync(y_host, y_dev, y_bytes, cudaMemcpyDeviceToHost, cap);
            const cudaError_t e2 = cudaStreamEndCapture(cap, &g);
            if (e == cudaSuccess && st == W4_OK && e2 == cudaSuccess && g)
                e = cudaGraphInstantiateWithFlags(&seq->io_exec, g, 0);
            else
                e = cudaErrorUnknown;
        }
        if (g) cudaGraphDestroy(g);
        if (cap) cudaStreamDestroy(cap);
        if (e != cudaSuccess) {
            seq->io_exec = nullptr;
            (void)cudaGetLastError();
            clear_error();
        } else {
            seq->io_xh = x_host;
            seq->io_xd = x_dev;
            seq->io_xb = x_bytes;
            seq->io_yd = y_dev;
            seq->io_yh = y_host;
            seq->io_yb = y_bytes;
        }
    }
    if (seq->io_exec) {
        W4_CUDA_TRY(cudaGraphLaunch(seq->io_exec, s));
    } else {
        if (x_bytes) W4_CUDA_TRY(cudaMemcpyAsync(x_dev, x_host, x_bytes, cudaMemcpyHostToDevice, s));
        w4_status st = w4_decode_seq_replay(seq, stream);
        if (st != W4_OK) return st;
        if (y_bytes) W4_CUDA_TRY(cudaMemcpyAsync(y_host, y_dev, y_bytes, cudaMemcpyDeviceToHost, s));
    }
    W4_CUDA_TRY(cudaStreamSynchronize(s));
    return W4_OK;
}

extern "C" int w4_decode_seq_kernels(const w4_seq* seq) { return seq ? (seq->persistent ? 1 : seq->n) : 0; }

extern "C" size_t w4_decode_seq_workspace_bytes(const w4_weight* w, int n, int M) {
    if (!w || n < 1 || M < 1 || M > 16) return 0;
    for (int i = 0; i < n; ++i)
        if (check_weight(&w[i]) != W4_OK) return 0;
    return step_workspace_bytes(w, n, M);
}

extern "C" w4_status w4_decode_seq_splits(const w4_weight* w, int n, int M, int act, const uint32_t* op_flags,
                                          int* splits) {
    clear_error();
    if (!w || !splits || n < 1 || n > kMaxStepOps) {
        set_error("NULL argument or n outside 1..%d", kMaxStepOps);
        return W4_ERR_ARG;
    }
    if (M < 1 || M > 16) {
        set_error("M=%d: the persistent sequence takes 1 <= M <= 16", M);
        return W4_ERR_SHAPE;
    }
    if (act != W4_ACT_F16 && act != W4_ACT_BF16 && act != W4_ACT_I8) {
        set_error("unknown activation type %d", act);
        return W4_ERR_ARG;
    }
    bool gated = false;
    for (int i = 0; i < n; ++i) {
        const w4_status st = check_weight(&w[i]);
        if (st != W4_OK) return st;
        gated = gated || (op_flags && (op_flags[i] & W4_OP_SWIGLU));
    }
    step_splits(w, n, M, act, gated, splits);
    return W4_OK;
}

extern "C" w4_status w4_decode_seq_create_persistent_ex(const w4_weight* w, const void* const* x,
                                                        void* const* y, const uint32_t* op_flags, int n, int M,
                                                        int act, void* workspace, size_t workspace_bytes,
                                                        void* stream, w4_seq** out);

extern "C" w4_status w4_decode_seq_create_persistent(const w4_weight* w, const void* const* x, void* const* y, int n,
                                                     int M, void* workspace, size_t workspace_bytes, void* stream,
                                                     w4_seq** out) {
    return w4_decode_seq_create_persistent_ex(w, x, y, nullptr, n, M, W4_ACT_F16, workspace, workspace_bytes, stream,
                                              out);
}

extern "C" w4_status w4_decode_seq_create_persistent_act(const w4_weight* w, const void* const* x,
                                                         void* const* y, int n, int M, int act, void* workspace,
                                                         size_t workspace_bytes, void* stream, w4_seq** out) {
    return w4_decode_seq_create_persistent_ex(w, x, y, nullptr, n, M, act, workspace, workspace_bytes, stream, out);
}

extern "C" w4_status w4_decode_seq_create_persistent_ex(const w4_weight* w, const void* const* x,
                                                        void* const* y, const uint32_t* op_flags, int n, int M,
                                                        int act, void* workspace, size_t workspace_bytes,
                                                        void* stream, w4_seq** out) {
    clear_error();
    if (!w || !x || !y || !out || n < 1) {
        set_error("NULL argument or n < 1");
        return W4_ERR_ARG;
    }
    *out = nullptr;
    if (act != W4_ACT_F16 && act != W4_ACT_BF16 && act != W4_ACT_I8) {
        set_error("unknown activation type %d", act);
        return W4_ERR_ARG;
    }
    for (int i = 0; i < n; ++i) {
        w4_status st = check_gemv_args(x[i], &w[i], y[i], M);
        if (st != W4_OK) return st;
        const uint32_t f = op_flags ? op_flags[i] : 0u;
        if (f & ~(uint32_t)W4_OP_SWIGLU) {
            set_error("projection %d: unknown flags 0x%x", i, f);
            return W4_ERR_ARG;
        }
        if ((f & W4_OP_SWIGLU) && w[i].N % 16 != 0) {
            set_error("projection %d: a gated weight needs N = 2I rows with I a multiple of 8 (w4_pack_glu)", i);
            return W4_ERR_SHAPE;
        }
    }
    w4_seq* s = new w4_seq();
    s->n = n;
    s->M = M;
    s->persistent = true;
    cudaStream_t user = static_cast<cudaStream_t>(stream);
    w4_status st = step_prepare(w, x, y, op_flags, n, M, act, workspace, workspace_bytes, user, &s->step);
    if (st != W4_OK) {
        delete s;
        return st;
    }
    // capture the single cooperative launch as a one-node graph
    cudaStream_t cap = nullptr;
    cudaError_t e = cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal);
    if (e == cudaSuccess) {
        st = step_launch(s->step, cap);
        cudaError_t e2 = cudaStreamEndCapture(cap, &s->graph);
        if (st == W4_OK && e2 == cudaSuccess) e2 = cudaGraphInstantiateWithFlags(&s->exec, s->graph, 0);
        if (st != W4_OK || e2 != cudaSuccess) {
            // graphs without this launch: replay issues it directly
            if (s->graph) cudaGraphDestroy(s->graph);
            s->graph = nullptr;
            s->exec = nullptr;
            (void)cudaGetLastError();
            clear_error();
        }
    } else {
        (void)cudaGetLastError();
    }
    if (cap) cudaStreamDestroy(cap);
    *out = s;
    return W4_OK;
}

extern "C" int w4_decode_seq_status(const w4_seq* seq) {
    if (!seq) return -1;
    return seq->persistent ? step_status(seq->step) : 0;
}
