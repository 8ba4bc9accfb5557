// Packed-weight file: one packed weight behind a fixed 256-byte header, laid
// out so that the payload can be mapped and copied to the device in one piece
// with nothing to parse.
//
// The pages' runtime keeps its quantised weights in a memory-mappable file
// whose first 256 bytes are a header that begins with a magic string, and
// refuses to load anything whose magic does not match ("Building a Custom LLM
// Inference Runtime ...", "The .nanoqwen File Format and Safety Protocols";
// "The Architecture of Modern Inference ...", "Data Integrity and
// Serialization: The .nanoqwen Format").  This file holds one weight in this
// library's own packed layout, with its own magic; beyond the magic, every
// header field, the reserved bytes and two checksums are validated before a
// single payload byte is copied.
//
// Header (little-endian):
//   0   char[8]  magic "W4A16PK1"
//   8   u32      version (1)
//   12  u32      header bytes (256)
//   16  i64      N
//   24  i64      K
//   32  u32      group size (128)
//   36  u32      tile bytes (1056)
//   40  u64      payload bytes (= w4_packed_bytes(N, K))
//   48  u64      payload offset (256)
//   56  u64      FNV-1a 64 of the payload, over little-endian 64-bit words
//   64  u64      the same of header bytes 0..63
//   72  ..256    zero
#include <fcntl.h>
#include <sys/mman.h>
#include <sys/stat.h>
#include <unistd.h>

#include <cstdio>
#include <cstring>
#include <vector>

#include "w4_internal.cuh"

namespace {

constexpr char kMagic[8] = {'W', '4', 'A', '1', '6', 'P', 'K', '1'};
constexpr uint32_t kFileVersion = 1;
constexpr uint32_t kHeaderBytes = W4_FILE_HEADER_BYTES;

bool host_little_endian() {
    const uint16_t one = 1;
    uint8_t b;
    std::memcpy(&b, &one, 1);
    return b == 1;
}

// FNV-1a 64 over little-endian 64-bit words (n is a multiple of 8).
uint64_t fnv1a64w(const uint8_t* p, size_t n) {
    uint64_t h = 0xcbf29ce484222325ull;
    for (size_t i = 0; i < n; i += 8) {
        uint64_t v;
        std::memcpy(&v, p + i, 8);
        if (!host_little_endian()) v = __builtin_bswap64(v);
        h ^= v;
        h *= 0x100000001b3ull;
    }
    return h;
}

void put32(uint8_t* p, uint32_t v) {
    for (int i = 0; i < 4; ++i) p[i] = (uint8_t)(v >> (8 * i));
}
void put64(uint8_t* p, uint64_t v) {
    for (int i = 0; i < 8; ++i) p[i] = (uint8_t)(v >> (8 * i));
}
uint32_t get32(const uint8_t* p) {
    uint32_t v = 0;
    for (int i = 0; i < 4; ++i) v |= (uint32_t)p[i] << (8 * i);
    return v;
}
uint64_t get64(const uint8_t* p) {
    uint64_t v = 0;
    for (int i = 0; i < 8; ++i) v |= (uint64_t)p[i] << (8 * i);
    return v;
}

struct Header {
    int64_t N = 0, K = 0;
    uint64_t payload = 0, sum = 0;
};

// Validate a header; on success fill h.  Any mismatch is W4_ERR_ARG.
w4_status parse_header(const uint8_t* b, size_t file_bytes, Header* h) {
    if (file_bytes < kHeaderBytes) {
        w4::set_error("file of %zu bytes is shorter than its %u-byte header", file_bytes, kHeaderBytes);
        return W4_ERR_ARG;
    }
    if (std::memcmp(b, kMagic, 8) != 0) {
        w4::set_error("not a packed-weight file (magic mismatch)");
        return W4_ERR_ARG;
    }
    if (get32(b + 8) != kFileVersion || get32(b + 12) != kHeaderBytes || get32(b + 32) != (uint32_t)w4::kGroupK ||
        get32(b + 36) != (uint32_t)w4::kTileBytes || get64(b + 48) != kHeaderBytes) {
        w4::set_error("unsupported packed-weight file (version %u, header %u, group %u, tile %u, offset %llu)",
                      get32(b + 8), get32(b + 12), get32(b + 32), get32(b + 36), (unsigned long long)get64(b + 48));
        return W4_ERR_ARG;
    }
    if (get64(b + 64) != fnv1a64w(b, 64)) {
        w4::set_error("packed-weight file header checksum mismatch");
        return W4_ERR_ARG;
    }
    for (uint32_t i = 72; i < kHeaderBytes; ++i)
        if (b[i] != 0) {
            w4::set_error("packed-weight file header: reserved byte %u is not zero", i);
            return W4_ERR_ARG;
        }
    h->N = (int64_t)get64(b + 16);
    h->K = (int64_t)get64(b + 24);
    h->payload = get64(b + 40);
    h->sum = get64(b + 56);
    const size_t expect = w4_packed_bytes(h->N, h->K);
    if (expect == 0 || h->payload != expect) {
        w4::set_error("packed-weight file: %lld x %lld needs %zu payload bytes, header says %llu", (long long)h->N,
                      (long long)h->K, expect, (unsigned long long)h->payload);
        return W4_ERR_ARG;
    }
    if (file_bytes != kHeaderBytes + h->payload) {
        w4::set_error("packed-weight file is %zu bytes, expected %llu", file_bytes,
                      (unsigned long long)(kHeaderBytes + h->payload));
        return W4_ERR_ARG;
    }
    return W4_OK;
}

// A read-only mapping of a whole file, unmapped on scope exit.
struct Mapping {
    int fd = -1;
    void* p = MAP_FAILED;
    size_t n = 0;
    ~Mapping() {
        if (p != MAP_FAILED) munmap(p, n);
        if (fd >= 0) close(fd);
    }
    w4_status open_file(const char* path) {
        fd = ::open(path, O_RDONLY);
        struct stat st;
        if (fd < 0 || fstat(fd, &st) != 0) {
            w4::set_error("cannot open %s", path);
            return W4_ERR_ARG;
        }
        n = (size_t)st.st_size;
        if (n == 0) {
            w4::set_error("%s is empty", path);
            return W4_ERR_ARG;
        }
        p = mmap(nullptr, n, PROT_READ, MAP_PRIVATE, fd, 0);
        if (p == MAP_FAILED) {
            w4::set_error("cannot map %s", path);
            return W4_ERR_ARG;
        }
        return W4_OK;
    }
    const uint8_t* bytes() const { return static_cast<const uint8_t*>(p); }
};

}  // namespace

extern "C" w4_status w4_file_write(const char* path, const w4_weight* w, int src_on_device, void* stream) {
    w4::clear_error();
    if (!path || !w) {
        w4::set_error("NULL argument");
        return W4_ERR_ARG;
    }
    w4_status st = w4::check_weight(w);
    if (st != W4_OK) return st;
    const size_t nb = w4_packed_bytes(w->N, w->K);
    std::vector<uint8_t> host;
    const uint8_t* payload = static_cast<const uint8_t*>(w->data);
    if (src_on_device) {
        host.resize(nb);
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        W4_CUDA_TRY(cudaMemcpyAsync(host.data(), w->data, nb, cudaMemcpyDeviceToHost, s));
        W4_CUDA_TRY(cudaStreamSynchronize(s));
        payload = host.data();
    }
    uint8_t h[kHeaderBytes];
    std::memset(h, 0, sizeof h);
    std::memcpy(h, kMagic, 8);
    put32(h + 8, kFileVersion);
    put32(h + 12, kHeaderBytes);
    put64(h + 16, (uint64_t)w->N);
    put64(h + 24, (uint64_t)w->K);
    put32(h + 32, (uint32_t)w4::kGroupK);
    put32(h + 36, (uint32_t)w4::kTileBytes);
    put64(h + 40, nb);
    put64(h + 48, kHeaderBytes);
    put64(h + 56, fnv1a64w(payload, nb));
    put64(h + 64, fnv1a64w(h, 64));
    FILE* f = std::fopen(path, "wb");
    if (!f) {
        w4::set_error("cannot create %s", path);
        return W4_ERR_ARG;
    }
    const bool ok = std::fwrite(h, 1, sizeof h, f) == sizeof h && std::fwrite(payload, 1, nb, f) == nb;
    if (std::fclose(f) != 0 || !ok) {
        w4::set_error("short write to %s", path);
        return W4_ERR_ARG;
    }
    return W4_OK;
}

extern "C" w4_status w4_file_info(const char* path, int64_t* N, int64_t* K, size_t* payload_bytes) {
    w4::clear_error();
    if (!path) {
        w4::set_error("NULL argument");
        return W4_ERR_ARG;
    }
    Mapping m;
    w4_status st = m.open_file(path);
    if (st != W4_OK) return st;
    Header h;
    st = parse_header(m.bytes(), m.n, &h);
    if (st != W4_OK) return st;
    if (N) *N = h.N;
    if (K) *K = h.K;
    if (payload_bytes) *payload_bytes = (size_t)h.payload;
    return W4_OK;
}

extern "C" w4_status w4_file_read(const char* path, void* dst, size_t dst_bytes, int dst_on_device, void* stream,
                                  w4_weight* out) {
    w4::clear_error();
    if (!path || !dst || !out) {
        w4::set_error("NULL argument");
        return W4_ERR_ARG;
    }
    if ((reinterpret_cast<uintptr_t>(dst) & 15) != 0) {
        w4::set_error("destination not 16-byte aligned");
        return W4_ERR_ALIGN;
    }
    Mapping m;
    w4_status st = m.open_file(path);
    if (st != W4_OK) return st;
    Header h;
    st = parse_header(m.bytes(), m.n, &h);
    if (st != W4_OK) return st;
    if (dst_bytes < h.payload) {
        w4::set_error("destination of %zu bytes, the weight needs %llu", dst_bytes, (unsigned long long)h.payload);
        return W4_ERR_WORKSPACE;
    }
    const uint8_t* payload = m.bytes() + kHeaderBytes;
    if (fnv1a64w(payload, (size_t)h.payload) != h.sum) {
        w4::set_error("packed-weight file payload checksum mismatch");
        return W4_ERR_ARG;
    }
    if (dst_on_device) {
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        W4_CUDA_TRY(cudaMemcpyAsync(dst, payload, (size_t)h.payload, cudaMemcpyHostToDevice, s));
        W4_CUDA_TRY(cudaStreamSynchronize(s));  // the mapping goes away on return
    } else {
        std::memcpy(dst, payload, (size_t)h.payload);
    }
    return w4_weight_view(dst, h.N, h.K, out);
}
