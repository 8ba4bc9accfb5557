// Error reporting and version of libw4.so.
#include <mutex>

#include "w4_internal.cuh"

namespace w4 {

static thread_local std::string g_last_error;

void set_error(const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
}

void clear_error() { g_last_error.clear(); }

w4_status cuda_fail(cudaError_t e, const char* what) {
    set_error("%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
    return W4_ERR_CUDA;
}

w4_status check_weight(const w4_weight* w) {
    if (!w || !w->data) {
        set_error("weight descriptor or its data pointer is NULL");
        return W4_ERR_ARG;
    }
    if (w->magic != W4_PACK_MAGIC || w->version != W4_PACK_VERSION) {
        set_error("weight descriptor magic/version %08x/%u, expected %08x/%u", w->magic, w->version,
                  W4_PACK_MAGIC, W4_PACK_VERSION);
        return W4_ERR_ARG;
    }
    if (w->N < 1 || w->K < kGroupK || w->K % kGroupK != 0) {
        set_error("weight shape N=%lld K=%lld: need N >= 1 and K a positive multiple of 128",
                  (long long)w->N, (long long)w->K);
        return W4_ERR_SHAPE;
    }
    if (!aligned16(w->data)) {
        set_error("packed weight pointer is not 16-byte aligned");
        return W4_ERR_ALIGN;
    }
    return W4_OK;
}

int device_sm_count() {
    static std::mutex mu;
    static int cache[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return kDefaultSms;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = kDefaultSms;
        cache[dev] = n;
    }
    return cache[dev];
}

}  // namespace w4

extern "C" const char* w4_strerror(w4_status s) {
    switch (s) {
        case W4_OK: return "ok";
        case W4_ERR_ARG: return "invalid argument";
        case W4_ERR_SHAPE: return "invalid shape";
        case W4_ERR_RANGE: return "quantised value outside [-8, 7]";
        case W4_ERR_ALIGN: return "pointer not 16-byte aligned";
        case W4_ERR_WORKSPACE: return "workspace missing or too small";
        case W4_ERR_CUDA: return "CUDA error";
        case W4_ERR_UNSUPPORTED: return "unsupported configuration";
    }
    return "unknown status";
}

extern "C" const char* w4_last_error(void) { return w4::g_last_error.c_str(); }

extern "C" int w4_version(void) { return 10000; }
