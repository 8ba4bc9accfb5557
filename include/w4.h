/*
 * w4.h -- C ABI of libw4.so: symmetric group-wise INT4 weight-only
 * projections (W4A16) for NVIDIA GB300 (sm_103a).
 *
 * The operation ("Building a Custom LLM Inference Runtime for
 * Qwen2.5-Coder-7B on NVIDIA H100 Hopper Architecture", section "Technical
 * Specifications and Hardware Alignment"): weights are signed 4-bit integers
 * q in [-8, 7], symmetric (no zero point), grouped 128 at a time along K,
 * each group of one output row with one FP16 scale s; w[n,k] = q[n,k] *
 * s[n, k/128].  Activations stay FP16 (same page, "The INT8 vs. FP16
 * Activation Trade-off", Path B).  Every projection computes
 *     y[m,n] = fp16( sum_k x[m,k] * w[n,k] )
 * with exact products, FP32 accumulation and one round-to-nearest-even
 * conversion to FP16 at the end.
 *
 * Conventions shared by every entry point
 *  - Ownership: the caller allocates and owns every buffer (packed weights,
 *    x, y, workspace).  The projection entry points and the sequence replay
 *    allocate nothing ("The Architecture of Modern Inference ...", "Data
 *    Integrity and Serialization: The .nanoqwen Format": no heap allocation
 *    during generation).
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *    default stream).  Device work is enqueued on it and the call returns
 *    without waiting, unless the entry point says it is synchronous.
 *  - Errors: arguments are checked before anything is launched; a failed
 *    check launches nothing.  A CUDA launch error maps to W4_ERR_CUDA and
 *    w4_last_error() gives its text (thread-local).
 *  - Alignment: device pointers to packed weights, x and y must be 16-byte
 *    aligned.
 *  - Data types: fp16 values travel as their 16-bit IEEE-754 binary16
 *    patterns (uint16_t); q travels as int8_t, one value per byte.
 */
#ifndef W4_H
#define W4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    W4_OK = 0,
    W4_ERR_ARG = 1,         /* NULL pointer, bad flag, wrong descriptor magic */
    W4_ERR_SHAPE = 2,       /* K % 128 != 0, N < 1, M out of range */
    W4_ERR_RANGE = 3,       /* a q outside [-8, 7] */
    W4_ERR_ALIGN = 4,       /* a pointer not 16-byte aligned */
    W4_ERR_WORKSPACE = 5,   /* workspace missing or too small */
    W4_ERR_CUDA = 6,        /* a CUDA runtime call failed; see w4_last_error() */
    W4_ERR_UNSUPPORTED = 7  /* no kernel for this device / configuration */
} w4_status;

/* Descriptor of a packed weight in device memory (a host-side struct). */
#define W4_PACK_MAGIC 0x4B503457u /* "W4PK" */
#define W4_PACK_VERSION 1u
typedef struct {
    const void* data; /* device pointer to w4_packed_bytes(N, K) bytes */
    int64_t N;        /* output rows */
    int64_t K;        /* reduction length, a multiple of 128 */
    uint32_t magic;   /* W4_PACK_MAGIC */
    uint32_t version; /* W4_PACK_VERSION */
} w4_weight;

const char* w4_strerror(w4_status status);
/* Text of the last failure on the calling thread ("" if none). */
const char* w4_last_error(void);
/* Library version, major * 10000 + minor * 100 + patch. */
int w4_version(void);

/* ------------------------------------------------------------------------
 * Packed layout (the offline repack).  The pages describe a "ValueShuffle"
 * layout in which even and odd nibbles alternate, to suit the byte-permute
 * datapath ("Building a Custom LLM Inference Runtime ...", "The .nanoqwen
 * File Format and Safety Protocols"; "The Architecture of Modern Inference
 * ...", "Data Integrity and Serialization: The .nanoqwen Format"), without the
 * exact permutation.  This library's
 * layout puts each nibble where one warp lane needs it as a tensor-core
 * operand fragment:
 *
 *   - The weight is cut into tiles of 16 rows x 128 K (one scale group per
 *     row).  Tile (band b, group g) starts at byte (b * (K/128) + g) * 1056;
 *     a band's tiles are contiguous along K.  ceil(N/16) bands.
 *   - A tile holds 1024 bytes of nibbles then 32 bytes of scales; every
 *     tile starts on a 32-byte boundary relative to the base.
 *   - Nibbles are offset binary, u = q + 8.  Lane L = 4r + c (r = 0..7,
 *     c = 0..3) and k16-step j = 0..7 own the little-endian 32-bit word at
 *     byte (j < 4 ? 0 : 512) + 16 L + 4 (j mod 4), whose nibble i (bits
 *     4i..4i+3) is, for i = 0..7:
 *        u[r][16j+4c],   u[r+8][16j+4c],   u[r][16j+4c+2], u[r+8][16j+4c+2],
 *        u[r][16j+4c+1], u[r+8][16j+4c+1], u[r][16j+4c+3], u[r+8][16j+4c+3]
 *     (row relative to the band, k relative to the group): a lane holds four
 *     consecutive k of rows r and r + 8.  Masking nibbles {0,4} and {1,5} of
 *     a word (and of the word shifted right by 8) gives four f16x2 registers,
 *     (r, 4c..4c+1), (r+8, 4c..4c+1), (r, 4c+2..4c+3), (r+8, 4c+2..4c+3):
 *     an m16n8k16 A fragment once k inside each 16-block is relabelled
 *     (fragment k 2c, 2c+1, 2c+8, 2c+9 <-> 4c .. 4c+3, the same relabelling
 *     applied to the activations), and, in natural k order, the registers
 *     of one 16-lane x 256-bit tensor-memory store (lanes r and r + 8,
 *     32-bit columns 2c and 2c + 1 of the k16 step).
 *   - Bytes 1024 + 4p .. +3 (p = 0..7) hold the fp16 scales of rows p (low
 *     half) and p + 8 (high half).
 *   - Rows n >= N of the last band are padding: u = 8 (q = 0), scale 0.
 * ---------------------------------------------------------------------- */

/* Bytes of the packed layout for an N x K weight; 0 if N < 1, K < 128 or
 * K % 128 != 0. */
size_t w4_packed_bytes(int64_t N, int64_t K);

/* Fill a descriptor for an already packed device buffer (no device work). */
w4_status w4_weight_view(const void* packed_dev, int64_t N, int64_t K,
                         w4_weight* out);

/* Host-only repack (no GPU needed): q int8 [N, K] row-major, scales fp16
 * [N, K/128] row-major -> dst (dst_bytes >= w4_packed_bytes(N, K)).
 * W4_ERR_RANGE if any q is outside [-8, 7] (nothing is clamped). */
w4_status w4_pack_host(const int8_t* q, const uint16_t* scales, int64_t N,
                       int64_t K, void* dst, size_t dst_bytes);

/* Host-only inverse of w4_pack_host: packed -> q [N, K], scales [N, K/128]. */
w4_status w4_unpack_host(const void* packed, int64_t N, int64_t K, int8_t* q,
                         uint16_t* scales);

/* Offline repack into device memory (the hot path never calls it).
 * src_on_device = 0: q and scales are host arrays, packed on the host and
 * copied in.  src_on_device = 1: they are device arrays, packed by a
 * kernel.  SYNCHRONOUS: returns after the packed bytes are in dst_dev, so
 * that an out-of-range q can be reported (W4_ERR_RANGE; dst_dev contents are
 * then unspecified).  May allocate temporary host or device memory.  On
 * success fills *out (may be NULL). */
w4_status w4_pack(const int8_t* q, const uint16_t* scales, int64_t N, int64_t K,
                  void* dst_dev, size_t dst_bytes, int src_on_device,
                  void* stream, w4_weight* out);

/* Pack a gated MLP weight for W4_OP_SWIGLU (below): q [2I, K] and scales
 * [2I, K/128] hold the stacked [gate (rows 0..I-1); up (rows I..2I-1)]
 * weight.  The packed weight (N = 2I, the size w4_pack gives) puts gate rows
 * 8b..8b+7 and then up rows 8b..8b+7 in 16-row band b, so rows r and r + 8
 * of every band are the gate and up rows of one output.  I must be a
 * positive multiple of 8 (W4_ERR_SHAPE).  Otherwise as w4_pack; w4_unpack
 * returns the interleaved row order. */
w4_status w4_pack_glu(const int8_t* q, const uint16_t* scales, int64_t I, int64_t K,
                      void* dst_dev, size_t dst_bytes, int src_on_device,
                      void* stream, w4_weight* out);

/* Inverse of w4_pack (round trip): q [N, K] int8 and scales [N, K/128]
 * fp16.  dst_on_device selects device (a kernel) or host outputs.
 * Synchronous. */
w4_status w4_unpack(const w4_weight* w, int8_t* q, uint16_t* scales,
                    int dst_on_device, void* stream);

/* ------------------------------------------------------------------------
 * Projections
 * ---------------------------------------------------------------------- */

/* Device workspace bytes a projection of this shape needs (0 = none; pass
 * NULL, 0).  The decode kernel (M <= 16) needs none.  The prefill kernel
 * (M > 16) needs at least 256 bytes: the first 4 hold a status word that the
 * call clears and the kernel sets non-zero if one of its pipeline waits gave
 * up (it then exits instead of hanging; y is not valid); when K is split
 * across CTAs the FP32 partials [splits][M][N] follow at byte 256. */
size_t w4_workspace_bytes(int M, int64_t N, int64_t K);

/* Decode projection, 1 <= M <= 16:  y[M, N] = x[M, K] . W^T.
 * x fp16 [M, K] row-major, y fp16 [M, N] row-major, both device.  Each packed
 * weight byte is read once per call whatever M.  Asynchronous on `stream`;
 * deterministic (same bits run to run).  Launched with programmatic
 * dependent launch enabled: the weight stream starts before the previous
 * kernel on the stream has finished; x is read only after it has. */
w4_status w4a16_gemv(const void* x, const w4_weight* w, void* y, int M,
                     void* workspace, size_t workspace_bytes, void* stream);

/* Launch shape of the decode kernel, for tuning sweeps.  Zero fields take
 * the library's choice.  The kernel is persistent: one CTA per SM (a cluster
 * of `splits` CTAs per K split), each walking blocks of `bands_per_cta`
 * 16-row bands and streaming their tiles through a shared-memory ring that
 * holds `depth` tiles. */
typedef struct {
    int bands_per_cta; /* 16-row bands per work block: 1, 2 or 4 */
    int splits;        /* K splits = CTAs per cluster: 1..8 (at most K/128) */
    int depth;         /* tiles in flight per CTA (ring size): a multiple of 8, 8..96 */
    int pdl;           /* programmatic dependent launch: 1 (default) = dependents may launch once
                          this grid's loads are issued, 2 = at once, 0 = off, -1 = default */
    int ctas_per_sm;   /* persistent CTAs per SM: 1 or 2 */
} w4_gemv_config;

/* w4a16_gemv with an explicit launch shape (W4_ERR_UNSUPPORTED if the shape
 * has no kernel). */
w4_status w4a16_gemv_config(const void* x, const w4_weight* w, void* y, int M,
                            const w4_gemv_config* cfg, void* stream);

/* The launch shape w4a16_gemv picks for (M, N, K). */
w4_status w4a16_gemv_default_config(int M, int64_t N, int64_t K,
                                    w4_gemv_config* out);

/* Prefill projection, any M >= 1 (tuned for M = 512): same contract as
 * w4a16_gemv, plus the workspace of w4_workspace_bytes (W4_ERR_WORKSPACE if
 * it is missing or short).  M <= 16 uses the decode kernel.  M > 16 runs on
 * the tensor cores (tcgen05, accumulators in TMEM): exact fp16 q times fp16 x
 * summed in FP32 per 128-wide group, then scaled and added in FP32.
 * Deterministic.  Not launched with programmatic dependent launch. */
w4_status w4a16_gemm(const void* x, const w4_weight* w, void* y, int M,
                     void* workspace, size_t workspace_bytes, void* stream);

/* Prefill projection for callers that cannot allocate device memory.
 * No passage of the pages corresponds to this entry point: it exists for
 * callers that cannot call cudaMalloc themselves (for example a plugin whose
 * host framework owns every device allocation, or code that must not risk the
 * device synchronisation or the out-of-memory failure an allocation can
 * bring), and so cannot pass w4a16_gemm a workspace.  It runs the same
 * kernels with the same results as w4a16_gemm, taking its workspace from a
 * file-scope device array of W4_STATIC_SCRATCH_BYTES that the library
 * reserves on every GPU that loads it, until the process exits.  It calls no
 * allocator.
 *  - The caller passes x, w and y exactly as for w4a16_gemm.
 *  - Shapes whose workspace (w4_workspace_bytes) exceeds
 *    W4_STATIC_SCRATCH_BYTES are rejected with W4_ERR_WORKSPACE before any
 *    launch; M <= 16 needs no scratch.
 *  - The first call on a device looks up the array's device address (with
 *    that device current); make that first call before any stream capture.
 *  - Every call on a device shares the one array, which keeps the previous
 *    call's contents (the call clears the status word it relies on).  Calls
 *    whose kernels overlap on the GPU (other streams, concurrent graphs) race
 *    on it: serialise them. */
#define W4_STATIC_SCRATCH_BYTES (4u << 20)
w4_status w4a16_gemm_static_scratch(const void* x, const w4_weight* w, void* y, int M, void* stream);

/* Status word of the static scratch on the current device: what the last
 * w4a16_gemm_static_scratch call with M > 16 left there.  0 when every
 * pipeline wait of that call completed; non-zero when one gave up after
 * about a second (that call's y is then not valid), which the caller cannot
 * otherwise see, since the word lives in the library's private array.
 * Synchronous: a plain device-to-host copy of 4 bytes.  Synchronise the
 * call's stream first (a non-blocking stream is not waited for).  -1 if the
 * word cannot be read (w4_last_error() says why).  Allocates nothing. */
int w4a16_gemm_static_scratch_status(void);

/* ------------------------------------------------------------------------
 * Decode step sequence ("Building a Custom LLM Inference Runtime ...",
 * "The Impact of CUDA Graphs": capturing the whole decode step in one CUDA
 * graph took eager launches from ~119 ms to ~17 ms per token).
 * ---------------------------------------------------------------------- */
typedef struct w4_seq w4_seq;

/* Build the projection chain w[0] .. w[n-1] (in that order), projection i
 * reading x[i] and writing y[i], all with the same M (1..16), and capture it
 * once as a CUDA graph.  Consecutive projections are joined by programmatic
 * dependent launch edges when use_pdl != 0.  The pointers are baked into the
 * graph: create a new sequence to change them.  Allocates host-side graph
 * objects and a private capture stream (not on the hot path); synchronous. */
w4_status w4_decode_seq_create(const w4_weight* w, const void* const* x,
                               void* const* y, int n, int M, int use_pdl,
                               void* stream, w4_seq** out);

/* One replay of the captured chain: a single cudaGraphLaunch on `stream`. */
w4_status w4_decode_seq_replay(w4_seq* seq, void* stream);

/* The same launches issued one by one, without the graph (for comparison). */
w4_status w4_decode_seq_eager(w4_seq* seq, void* stream);

/* End to end with host buffers: copy x_bytes from pinned host memory x_host
 * to the device range x_dev, replay, copy y_bytes from y_dev to y_host, and
 * wait for the stream.  x_dev / y_dev are device ranges that hold the
 * sequence's x and y buffers (e.g. one arena each).  Synchronous.  The first
 * call with a given set of the six buffer arguments captures the two copies
 * and the step as one CUDA graph (host-side graph objects allocated then,
 * freed by w4_decode_seq_destroy or the next rebuild) and launches it; later
 * calls with the same arguments launch that graph again.  Where the capture
 * fails the operations are issued one by one, with the same results. */
w4_status w4_decode_seq_run_host(w4_seq* seq, const void* x_host, void* x_dev,
                                 size_t x_bytes, void* y_dev, void* y_host,
                                 size_t y_bytes, void* stream);

/* Device workspace bytes of a persistent sequence over these n weights at M
 * tokens (0 on bad arguments).  Caller-owned, 256-byte aligned. */
size_t w4_decode_seq_workspace_bytes(const w4_weight* w, int n, int M);

/* The same projection chain as w4_decode_seq_create, run by ONE persistent
 * cooperative kernel (one CTA of 16 warps per SM) captured as a one-node
 * graph.  Each warp streams its share of the weights of every projection
 * back to back into its own shared-memory ring, never waiting on the chain,
 * and computes projection i only after every CTA has finished projection
 * i - 1 (completion counters in `workspace`), so the data dependency of a
 * real decode step (x[i] computed from y[i-1]) is honoured.  Same arithmetic
 * as w4a16_gemv; where the two cut K differently the last bits can differ.
 * Every replay gives the same bits.  `workspace` (of
 * w4_decode_seq_workspace_bytes, 256-byte aligned: W4_ERR_WORKSPACE /
 * W4_ERR_ALIGN otherwise) holds the completion counters, the status word and
 * the K-split partials; the projection table travels in the launch's
 * parameters.  The workspace must stay alive and unshared while the sequence
 * exists, and replays of one sequence must not overlap on the GPU.  At most
 * 448 projections; W4_ERR_UNSUPPORTED for a sequence the kernel cannot take.
 * Synchronous (initialises the workspace). */
w4_status w4_decode_seq_create_persistent(const w4_weight* w, const void* const* x,
                                          void* const* y, int n, int M, void* workspace,
                                          size_t workspace_bytes, void* stream, w4_seq** out);

/* Activation types of the persistent sequence. */
#define W4_ACT_F16 0  /* x and y IEEE binary16 (the pages' FP16 activations) */
#define W4_ACT_BF16 1 /* x and y bfloat16; scales stay binary16.  The kernel rescales each
                         group of 128 x of a token by a power of two and rounds it to
                         binary16 (exact for every x within 2^-28 of the group's largest
                         magnitude; |x| below 2^116) and runs the binary16 arithmetic on it */
#define W4_ACT_I8 2   /* the pages' Path A ("3. The INT8 vs. FP16 Activation Trade-off"):
                         x binary16, quantised per token to INT8 inside the kernel
                         (sx = max|x| / 127 and xq = rne(x / sx) in IEEE binary32),
                         exact integer group sums (dp4a), y binary16 =
                         rne(sum_g s * sx * sum_k xq * q) with FP32 scaling */

/* w4_decode_seq_create_persistent with the activation type chosen (act =
 * W4_ACT_F16 is w4_decode_seq_create_persistent; W4_ACT_I8 is described
 * above).  With W4_ACT_BF16, x and y
 * are bfloat16 and y = bf16_rne(sum x * q * s) with FP32 accumulation: the
 * pages' projection ("Building a Custom LLM Inference Runtime ...",
 * "Technical Specifications and Hardware Alignment") with the nibble
 * conversion producing bfloat16 instead of binary16 operands.  Same workspace size as the
 * binary16 sequence.  W4_ERR_ARG for another act. */
w4_status w4_decode_seq_create_persistent_act(const w4_weight* w, const void* const* x,
                                              void* const* y, int n, int M, int act,
                                              void* workspace, size_t workspace_bytes,
                                              void* stream, w4_seq** out);

/* Per-projection options of a persistent sequence. */
#define W4_OP_SWIGLU 1u /* gated MLP: the weight comes from w4_pack_glu (N = 2I rows,
                           gate and up interleaved per band) and y receives
                           h = silu(gate) * up, I columns per token, instead of
                           the 2I projections (SwiGLU, Qwen2.5's MLP activation;
                           the pages do not name it) */

/* The same with options per projection: op_flags[i] (W4_OP_*, or NULL for
 * none).  A W4_OP_SWIGLU projection computes, per token m and row n < I,
 *   y[m, n] = rne(silu(g) * u),  g = sum_k x*q*s over gate row n,
 *   u = the same over up row n,  silu(g) = g / (1 + exp(-g)),
 * from the FP32 sums (no rounding of g and u) with FP32 silu.  W4_ERR_ARG
 * for an unknown flag, W4_ERR_SHAPE for a gated weight with N % 16 != 0. */
w4_status w4_decode_seq_create_persistent_ex(const w4_weight* w, const void* const* x,
                                             void* const* y, const uint32_t* op_flags,
                                             int n, int M, int act, void* workspace,
                                             size_t workspace_bytes, void* stream,
                                             w4_seq** out);

/* The K split of every projection of the persistent sequence these weights
 * would run at M tokens with activation type act and options op_flags (as
 * for w4_decode_seq_create_persistent_ex) on the current device:
 * splits[n] receives S, the number of CTAs that share each band's K range
 * (S > 1: their FP32 partials are added through the workspace).  Planning
 * only: no device work, no allocation; without a device the plan assumes
 * 152 SMs. */
w4_status w4_decode_seq_splits(const w4_weight* w, int n, int M, int act,
                               const uint32_t* op_flags, int* splits);

/* Status word of a persistent sequence (a synchronous device read): 0 when
 * every wait of its replays so far completed, non-zero when one gave up after
 * about a second (the outputs of that replay are then invalid).  0 for graph
 * sequences, -1 on error. */
int w4_decode_seq_status(const w4_seq* seq);

/* Number of kernels one replay launches (1 for a persistent sequence). */
int w4_decode_seq_kernels(const w4_seq* seq);

void w4_decode_seq_destroy(w4_seq* seq);

/* ------------------------------------------------------------------------
 * Packed-weight file.  The pages keep their quantised weights in a
 * memory-mappable file whose first 256 bytes are a header that begins with
 * a magic string, and refuse to load a file whose magic does not match
 * ("Building a Custom LLM Inference Runtime ...", "The .nanoqwen File Format
 * and Safety Protocols"; "The Architecture of Modern Inference ...", "Data
 * Integrity and Serialization: The .nanoqwen Format").  Here a file holds ONE
 * packed weight (the layout above) after a 256-byte little-endian header:
 *   0 magic "W4A16PK1" | 8 u32 version 1 | 12 u32 header bytes 256 |
 *   16 i64 N | 24 i64 K | 32 u32 group 128 | 36 u32 tile bytes 1056 |
 *   40 u64 payload bytes | 48 u64 payload offset 256 |
 *   56 u64 checksum of the payload | 64 u64 checksum of bytes 0..63 |
 *   72..255 zero.  Checksum: FNV-1a 64 taken over little-endian 64-bit
 *   words (h = 0xcbf29ce484222325; per word: h ^= w; h *= 0x100000001b3).
 * Readers check every field, the reserved bytes and both checksums before
 * copying anything (fail fast): any mismatch is W4_ERR_ARG with the reason in
 * w4_last_error().  All three calls are synchronous host calls.
 * ---------------------------------------------------------------------- */
#define W4_FILE_HEADER_BYTES 256

/* Write w to path (created or truncated).  src_on_device: w->data is device
 * memory (copied to the host on `stream` first) or host memory. */
w4_status w4_file_write(const char* path, const w4_weight* w,
                        int src_on_device, void* stream);

/* Validate path's header and return the weight's shape and payload size
 * (any of the outputs may be NULL).  Does not read the payload. */
w4_status w4_file_info(const char* path, int64_t* N, int64_t* K,
                       size_t* payload_bytes);

/* Validate path (header and payload checksum), then copy the payload into
 * the caller's buffer dst (dst_bytes >= payload, 16-byte aligned; device
 * memory when dst_on_device, copied on `stream` and synchronised, else host
 * memory) and describe it in *out.  W4_ERR_WORKSPACE if dst is too small,
 * W4_ERR_ALIGN if misaligned; nothing is written to dst on any error. */
w4_status w4_file_read(const char* path, void* dst, size_t dst_bytes,
                       int dst_on_device, void* stream, w4_weight* out);

#ifdef __cplusplus
}
#endif
#endif /* W4_H */
