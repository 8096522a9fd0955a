/*
 * w12.h — C ABI of the W12 library (libw12.so): lossless ~12-bit BF16 weights
 * decoded bit-exactly inside a memory-bound GEMM on GB300 (sm_103a).
 *
 * What the operation is, from the SpecPilot pages:
 *   "StargazerX0/SpecPilot" (hotrepo.ai), §What it is — W12 is a 12-bit weight
 *     format that decodes bit-exactly inside the GEMM; it speeds up plain BF16
 *     decoding at batch 1-32.
 *   "SpecPilot" (fasttoolhub.com), §Differentiation — a general lossless
 *     12-bit weight format.
 *   "SpecPilot: an agent doubled speculative decoding speed, and the 10.87x
 *     needs context" (ai.jakubjirak.com), §The mechanisms it found — about
 *     12.01-12.02 bits per weight, decoded in the GEMM's registers; 12 instead
 *     of 16 bits cuts the weight traffic of a memory-bound decode by a quarter.
 * The pages define no byte layout; this library defines W12 v1:
 *
 *   tile 128 rows, quarter 32 rows, chunk 32 columns, segment 256 columns.
 *   N is padded to a multiple of 128 and K to a multiple of 32 with +0.0.
 *   blob = 256-byte header | segment headers (32 B per tile x segment)
 *        | packed chunks (6144 B per tile x chunk) | escape bytes; each part
 *          starts on a 256-byte boundary.
 *   segment header: table T[16] (code -> exponent; T[15] = 0 and slots j, j+8
 *     share the exponent's top bit), u32 first-escape offset, u16 escape count
 *     per quarter, u32 mask (bit 8q+j: quarter q has an escape in chunk j).
 *   packed chunk: three 2048-byte slabs of 128 rows x 16 bytes: S bytes of
 *     columns 0-15, S bytes of columns 16-31, 4-bit codes (even column in the
 *     low nibble).  S byte = (mantissa << 1) | sign of the column-xor-1 partner.
 *   code 15 = escape: the exponent is the next byte of the escape list, ordered
 *     by tile, segment, quarter, chunk, row, column.
 *
 * Conventions for every call:
 *   - Returns a w12_status (0 = W12_OK).  Nothing throws across the ABI.  On an
 *     error w12_last_error() (per thread) describes it.
 *   - The caller owns every buffer.  The library allocates no memory of its
 *     own; its only state is one status word per device in static device
 *     memory (see w12_check_status).
 *   - Pointers named *_dev are device pointers; *_host are host pointers.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Device calls are asynchronous on that stream and never synchronise it,
 *     except w12_check_status.
 */
#ifndef W12_H
#define W12_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define W12_FORMAT_VERSION 1

typedef enum w12_status {
    W12_OK = 0,
    W12_ERR_INVALID_ARG = 1,      /* null pointer, M out of range, ...          */
    W12_ERR_SHAPE = 2,            /* N or K < 1, or sizes that overflow          */
    W12_ERR_BUFFER_TOO_SMALL = 3, /* blob or workspace shorter than required     */
    W12_ERR_ALIGNMENT = 4,        /* device pointer not aligned as documented    */
    W12_ERR_CORRUPT_BLOB = 5,     /* header or segment headers inconsistent      */
    W12_ERR_UNSUPPORTED_ARCH = 6, /* current device is not compute capability 10.3 */
    W12_ERR_CUDA = 7,             /* a CUDA runtime call failed                   */
    W12_ERR_TIMEOUT = 8           /* a kernel gave up a bounded wait (device word) */
} w12_status;

/* Geometry and plane offsets of a blob, filled by w12_blob_info. */
typedef struct w12_info {
    int64_t N, K;             /* original shape: W is N x K, y = x . W^T      */
    int64_t N_pad, K_pad;     /* N rounded up to 128, K rounded up to 32       */
    int64_t tiles;            /* N_pad / 128                                   */
    int64_t chunks;           /* K_pad / 32 (per tile)                         */
    int64_t segs;             /* ceil(chunks / 8) (per tile)                   */
    uint64_t off_seghdr, bytes_seghdr;
    uint64_t off_weights, bytes_weights;
    uint64_t off_escapes, bytes_escapes;
    uint64_t n_escapes;
    uint64_t total_bytes;
    double bits_per_weight;   /* 8 * total_bytes / (N * K)                     */
} w12_info;

/* Text of the last error on this thread ("" if none). */
const char *w12_last_error(void);

/* Name of a status code. */
const char *w12_status_string(int status);

/* Format version this library reads and writes (W12_FORMAT_VERSION). */
int w12_format_version(void);

/*
 * Exact blob size for the N x K row-major BF16 matrix w_host (bit patterns).
 * Runs the table and escape count of the encoder.  Errors: INVALID_ARG (null),
 * SHAPE (N or K < 1, size overflow, more than 2^32-1 escapes).
 */
int w12_encoded_size_host(const uint16_t *w_host, int64_t N, int64_t K, size_t *bytes);

/*
 * Encode w_host (N x K, row-major BF16 bit patterns) into blob_host, which must
 * hold at least w12_encoded_size_host bytes (else BUFFER_TOO_SMALL).  The
 * output is canonical: equal inputs give equal bytes.  Uses all host cores.
 * The caller copies the blob to the device (any 256-byte aligned address).
 */
int w12_encode_host(const uint16_t *w_host, int64_t N, int64_t K, void *blob_host,
                    size_t bytes);

/*
 * Read and check the header of a host blob of `bytes` bytes and fill *out.
 * Checks magic, version and every geometry field against N and K (CORRUPT_BLOB
 * on mismatch, BUFFER_TOO_SMALL if the blob is shorter than its total size).
 * Only the first 256 bytes are read: for a blob held on the device, a host
 * copy of its header with `bytes` = the device blob's length is enough.
 */
int w12_blob_info(const void *blob_host, size_t bytes, w12_info *out);

/*
 * Full check of a host blob: the header as above, then every segment header
 * (T[15] = 0, paired slots share the top bit, escape offsets are the running
 * sum of the quarter counts, masks agree with the counts, the counts add up
 * to the header's escape count).  CORRUPT_BLOB on any failure.
 */
int w12_blob_validate(const void *blob_host, size_t bytes);

/*
 * Decode a device-resident blob to BF16: w_out_dev[n * K + k] for n < N, k < K
 * (row-major, N x K).  Bit-exact inverse of the encoder.  `info` comes from
 * w12_blob_info on a host copy of the same blob.  blob_dev must be 256-byte
 * aligned and w_out_dev 2-byte aligned (ALIGNMENT).  Asynchronous on stream.
 */
int w12_decode(const void *blob_dev, const w12_info *info, uint16_t *w_out_dev, void *stream);

/*
 * Workspace bytes w12_gemm needs for this blob and token count M (1..32).
 * The workspace holds the split-K fp32 partials, one arrival counter per
 * tile and, when x is not TMA-aligned, a padded copy of x.
 */
int w12_gemm_workspace_size(const w12_info *info, int M, size_t *bytes);

/*
 * The launch plan w12_gemm uses for this blob and M on the current device:
 * out[0] token rows per CTA (1 or 2 on the CUDA-core path, 16 or 32 on the
 * tensor-core path), out[1] CTAs per 128-row tile along K (split-K; when the
 * CUDA-core path shares one wave of CTAs out as equal contiguous ranges of
 * the tiles' 256-column segments, the most CTAs that can share a tile),
 * out[2] total CTAs, out[3] resident CTAs per SM assumed.
 */
int w12_gemm_launch_info(const w12_info *info, int M, int32_t out[4]);

/*
 * y_dev[m * N + n] = BF16_rne( sum_k x_dev[m * K + k] * W[n][k] ), fp32
 * accumulation, for 1 <= M <= 32, with W held by blob_dev.  The weights are
 * streamed from HBM in packed form and decoded in registers.  One or two
 * tokens: CUDA cores multiply them (fma.rn.f32.bf16, one per weight and
 * token); three or more: tensor cores (tcgen05, weights as the 128-row A
 * operand, tokens as N = 16 or 32).  The sums are reproducible run to run
 * (fixed split-K order); w12_gemm_launch_info reports the plan.
 * x_dev: M x K row-major BF16; y_dev: M x N row-major BF16, 2-byte
 * aligned.  blob_dev must be 256-byte aligned.  workspace: at least
 * w12_gemm_workspace_size bytes, 256-byte aligned, ZERO-FILLED BEFORE ITS
 * FIRST USE; every successful call leaves the counters zero again (after a
 * TIMEOUT, zero it again).  Calls sharing one workspace must be ordered on
 * the GPU (same stream, or synchronised).  Asynchronous on stream; errors found
 * on the device are reported by w12_check_status.
 */
int w12_gemm(const uint16_t *x_dev, const void *blob_dev, const w12_info *info,
             uint16_t *y_dev, int M, void *workspace, size_t ws_bytes, void *stream);

/*
 * Grouped product: y_devs[i] = x_dev . W_i^T for up to W12_MAX_GROUP matrices
 * that share x (and so K) — the q/k/v projections of a decoder layer, or its
 * gate/up projections — in one launch, planned as one matrix of all their
 * 128-row tiles (no passage of the pages has a counterpart; it removes the
 * per-launch fixed cost that dominates small matrices such as k and v).  Each
 * output meets the same bound as w12_gemm's and is bit-identical to it when
 * both split K the same way (fixed split-K with the same split count).  blobs_dev[i] 256-byte aligned, y_devs[i] M x N_i BF16;
 * infos[i] from w12_blob_info; all K equal (SHAPE otherwise).  Workspace:
 * w12_gemm_group_workspace_size bytes, same rules as w12_gemm.
 */
#define W12_MAX_GROUP 4

int w12_gemm_group_workspace_size(int count, const w12_info *infos, int M, size_t *bytes);

/*
 * The plan of a grouped launch (count = 1: of a single w12_gemm): out[0..3]
 * as w12_gemm_launch_info, out[4] which kernel runs it (W12_KERNEL_*).
 */
#define W12_KERNEL_GEMV 0     /* CUDA cores, two CTAs per SM                 */
#define W12_KERNEL_GEMV_SM 1  /* CUDA cores, one CTA per SM                  */
#define W12_KERNEL_TC 2       /* tcgen05, several CTAs per SM, fixed split-K */
#define W12_KERNEL_TC_SM 3    /* tcgen05, one CTA per SM, stream-K ranges    */

int w12_gemm_group_launch_info(int count, const w12_info *infos, int M, int32_t out[5]);

int w12_gemm_group(const uint16_t *x_dev, int count, const void *const *blobs_dev, const w12_info *infos,
                   uint16_t *const *y_devs, int M, void *workspace, size_t ws_bytes, void *stream);

/*
 * LM-head product with a fused exact argmax ("SpecPilot: an agent doubled
 * speculative decoding speed, and the 10.87x needs context" (ai.jakubjirak.com),
 * §The mechanisms it found, lists a certified exact-argmax LM head; the page
 * does not say how it is certified).  Reading taken: for each token m,
 * idx_dev[m] = the row n that maximizes logit[m][n] = sum_k x[m][k] * W[n][k]
 * as w12_gemm accumulates it (fp32, the same order), compared in fp32 before
 * any rounding to BF16, ties to the smallest n; val_dev[m] = that fp32 logit.
 * -0 compares equal to +0 and a NaN logit ranks as -infinity (val is then
 * -inf).  y_dev may be NULL; otherwise it receives the BF16 logits exactly as
 * w12_gemm would.  x_dev, blob_dev, info and M as w12_gemm; idx_dev int32[M],
 * val_dev float[M], 4-byte aligned; N must fit in int32 (SHAPE).  workspace:
 * w12_gemm_argmax_workspace_size bytes, 256-byte aligned, zero-filled before
 * its first use (the call clears its own argmax keys).  Asynchronous on
 * stream: a memset, the GEMM kernel with the argmax epilogue (each CTA folds
 * its rows' best candidate into one 64-bit key per token with an atomic max)
 * and a one-warp finalize kernel.
 */
int w12_gemm_argmax_workspace_size(const w12_info *info, int M, size_t *bytes);

int w12_gemm_argmax(const uint16_t *x_dev, const void *blob_dev, const w12_info *info, int M,
                    uint16_t *y_dev, int32_t *idx_dev, float *val_dev, void *workspace,
                    size_t ws_bytes, void *stream);

/*
 * Size of the fixed scratch array behind w12_gemm_noalloc (16 MiB).
 */
#define W12_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * The same product as w12_gemm, for callers that cannot allocate device
 * memory.  No passage of the SpecPilot pages has a counterpart; this entry
 * point exists for integration.  Callers that cannot call cudaMalloc include
 * serving engines whose allocator has reserved all free HBM up front (for
 * weights and KV cache) and would fail or fragment on a new allocation,
 * plug-ins that must not allocate behind their host framework's memory
 * accounting, and latency-critical paths where cudaMalloc's implicit device
 * synchronisation is not acceptable.
 *
 * The split-K partials, arrival counters and padded x copy live in one array
 * of W12_NOALLOC_SCRATCH_BYTES in static device memory inside the library;
 * every device that loads the library keeps that array until the process
 * exits.  The call allocates nothing (no cudaMalloc, cudaFree or allocating
 * library routine): it clears the counters with cudaMemsetAsync on `stream`
 * and launches the GEMM.  The first call on each device looks up the array's
 * device address (with that device current); make that first call before any
 * stream capture.  A problem whose scratch need (w12_gemm_workspace_size)
 * exceeds W12_NOALLOC_SCRATCH_BYTES is rejected with W12_ERR_BUFFER_TOO_SMALL
 * before anything is launched.  All calls share the one array, which keeps
 * the last call's contents: calls that overlap on the GPU (different streams
 * without ordering, or several host threads) race and give wrong results;
 * order them on one stream.  Arguments and errors otherwise as w12_gemm.
 */
int w12_gemm_noalloc(const uint16_t *x_dev, const void *blob_dev, const w12_info *info,
                     uint16_t *y_dev, int M, void *stream);

/*
 * Device encoder: the same canonical bytes as w12_encode_host, computed on the
 * GPU from weights already in device memory (for example a whole model
 * checkpoint loaded to HBM, encoded without a round trip through the host).
 * It produces the format the pages call lossless and bit-exact ("SpecPilot"
 * (fasttoolhub.com) §Differentiation; "StargazerX0/SpecPilot" §What it is);
 * the pages do not say where the encoding runs.
 *
 * w12_encode_workspace_size: scratch bytes both calls below need for N x K
 *   (one 32-byte plan record and one 8-byte offset per 128 x 256 segment, plus
 *   256).  SHAPE as for w12_encoded_size_host.
 * w12_encoded_size_device: runs the encoder's table and escape-count passes on
 *   `stream` over w_dev (N x K row-major BF16 bit patterns, 2-byte aligned;
 *   16-byte aligned with K % 8 == 0 reads faster), then SYNCHRONISES `stream`
 *   and stores the exact blob size (equal to w12_encoded_size_host's) in
 *   *bytes.  SHAPE if the matrix has more than 2^32-1 escapes.
 * w12_encode_device: writes the whole blob into blob_dev (256-byte aligned,
 *   `bytes` long), asynchronously on `stream`; it repeats the table pass, so
 *   it needs no state from the size call.  A buffer shorter than the packed
 *   planes is refused on the host (BUFFER_TOO_SMALL); a buffer too short for
 *   the escape bytes is found on the device: nothing is written past `bytes`,
 *   the header is not written and w12_check_status returns BUFFER_TOO_SMALL
 *   (SHAPE for more than 2^32-1 escapes).  workspace: 256-byte aligned, at
 *   least w12_encode_workspace_size bytes, no initial contents; calls sharing
 *   one workspace must be ordered on the GPU.
 */
int w12_encode_workspace_size(int64_t N, int64_t K, size_t *bytes);

int w12_encoded_size_device(const uint16_t *w_dev, int64_t N, int64_t K, void *workspace,
                            size_t ws_bytes, size_t *bytes, void *stream);

int w12_encode_device(const uint16_t *w_dev, int64_t N, int64_t K, void *blob_dev, size_t bytes,
                      void *workspace, size_t ws_bytes, void *stream);

/*
 * ---------------------------------------------------------------- Q8 copy
 * An 8-bit copy of a weight matrix for the first level of a two-level
 * verification ("SpecPilot: an agent doubled speculative decoding speed, and
 * the 10.87x needs context" (ai.jakubjirak.com), §The mechanisms it found,
 * names a two-level verification with an 8-bit or INT6/INT8 weight copy; it
 * gives no scheme).  Reading taken: symmetric INT8 per output row, lossy by
 * design (it only drafts; W12 stays the exact weights):
 *   a[n] = max_k |W[n][k]|, s[n] = a[n] / 127 in fp32, q[n][k] = rint(W[n][k]
 *   / s[n]) in fp32 (nearest, ties to even) clamped to [-127, 127]; a zero row
 *   has s = 0, q = 0; a row with Inf or NaN is rejected (INVALID_ARG).
 * Q8 v1 blob: 256-byte header | scales fp32[N_pad] (pad rows 0) | q plane,
 * each part 256-byte aligned.  q plane: per 128-row tile, per 32-column chunk
 * (chunks in column order), two 2048-byte slabs of 128 rows x 16 int8
 * (columns 0-15, then 16-31); padding is 0.  Header (little-endian): 0x00
 * "Q8W1", 0x04 u32 1, 0x08 u32 256, 0x0C u32 0, 0x10 i64 N, 0x18 K, 0x20 N_pad,
 * 0x28 K_pad, 0x30 tiles, 0x38 chunks, 0x40/0x48 u64 scales offset/size,
 * 0x50/0x58 q offset/size, 0x60 total; the rest 0.
 */
typedef struct w12_q8_info {
    int64_t N, K, N_pad, K_pad, tiles, chunks, segs;
    uint64_t off_scales, bytes_scales, off_q, bytes_q, total_bytes;
} w12_q8_info;

/* Blob size for an N x K matrix (SHAPE on bad sizes). */
int w12_q8_encoded_size(int64_t N, int64_t K, size_t *bytes);

/* Quantize w_host (N x K BF16 bit patterns) into blob_host (>= the size);
 * canonical bytes; all host cores. */
int w12_q8_encode_host(const uint16_t *w_host, int64_t N, int64_t K, void *blob_host, size_t bytes);

/* Check the header of a Q8 blob (a host copy of its first 256 bytes is
 * enough) and fill *out.  CORRUPT_BLOB / BUFFER_TOO_SMALL as w12_blob_info. */
int w12_q8_blob_info(const void *blob_host, size_t bytes, w12_q8_info *out);

/* Workspace bytes w12_q8_gemm needs (1 <= M <= 32). */
int w12_q8_gemm_workspace_size(const w12_q8_info *info, int M, size_t *bytes);

/*
 * y_dev[m * N + n] = BF16_rne( s[n] * sum_k x_dev[m * K + k] * q[n][k] ), fp32
 * accumulation and scale multiply, 1 <= M <= 32, on the same tcgen05 kernel as
 * w12_gemm (the copy is converted to BF16 exactly in registers: |q| <= 127).
 * Arguments, alignment, workspace rules and errors as w12_gemm.
 */
int w12_q8_gemm(const uint16_t *x_dev, const void *blob_dev, const w12_q8_info *info,
                uint16_t *y_dev, int M, void *workspace, size_t ws_bytes, void *stream);

/*
 * Q8 copies of up to W12_MAX_GROUP matrices that multiply the same x (the
 * q/k/v or gate/up projections) in one launch, as w12_gemm_group does for
 * W12 blobs: y_devs[i] = the w12_q8_gemm product of x with blob i, with
 * blob i's own row scales.  blobs_dev[i] 256-byte aligned, y_devs[i] M x N_i
 * BF16; infos[i] from w12_q8_blob_info; all K equal (SHAPE otherwise).
 * Workspace: w12_q8_gemm_group_workspace_size bytes; launch_info fills
 * out[0..4] as w12_gemm_group_launch_info.  Errors as w12_gemm_group.
 */
int w12_q8_gemm_group_workspace_size(int count, const w12_q8_info *infos, int M, size_t *bytes);

int w12_q8_gemm_group_launch_info(int count, const w12_q8_info *infos, int M, int32_t out[5]);

int w12_q8_gemm_group(const uint16_t *x_dev, int count, const void *const *blobs_dev, const w12_q8_info *infos,
                      uint16_t *const *y_devs, int M, void *workspace, size_t ws_bytes, void *stream);

/*
 * Measurement helper with no counterpart on the pages: reads `bytes` (a
 * multiple of 16) of device memory at buf_dev (16-byte aligned) once, with
 * 16-byte streaming loads spread over every SM, and writes the 4-byte word at
 * sink_dev only if the XOR of everything read equals `never` (pick a value
 * the data cannot fold to, and the kernel writes nothing).  Timed over a
 * buffer larger than L2, it gives the HBM read ceiling for the GEMM kernels,
 * which read ~1.5 B per weight and write almost nothing.  Asynchronous on
 * `stream`; INVALID_ARG / ALIGNMENT on bad pointers or sizes.
 */
int w12_read_stream(const void *buf_dev, size_t bytes, void *sink_dev, uint32_t never, void *stream);

/*
 * Synchronise `stream`, then read and clear the current device's status word,
 * which kernels set when a bounded wait gives up (TIMEOUT) or the device
 * encoder finds its output buffer too short (BUFFER_TOO_SMALL) or too many
 * escapes (SHAPE).  Returns that status, CUDA on a CUDA error, else OK.
 */
int w12_check_status(void *stream);

/*
 * Launch options, process-wide (every device and thread sees the same
 * values).  The library reads no environment variables: a plan changes only
 * through these calls.  No passage of the pages has a counterpart; they exist
 * for tuning and for tests that must reach every kernel variant.  Setting an
 * option while another thread launches is safe but that launch may see the
 * old or the new value.  Names (default; accepted values):
 *   gemv_max_m      (2; 0..2)   largest M on the CUDA-core path; 0 sends
 *                               every M to the tensor cores
 *   token_tile      (0; 0, 16, 32) tensor-core token tile, 0 = the planner's
 *   a_operand_smem  (0; 0..1)   1: tensor-core A operand from shared memory
 *   gemv_sm         (-1; -1..1) CUDA-core kernel: -1 planner, 0 two CTAs per
 *                               SM, 1 one CTA per SM
 *   stream_k        (1; 0..1)   0: fixed split-K on the CUDA-core path
 *   splits          (0; 0..2^20) n > 0: fixed split-K with n splits where the
 *                               kernel's per-CTA limits allow it
 *   pdl             (1; 0..1)   programmatic dependent launch on GEMMs
 *   timeout_ms      (4000; 1..600000) bounded waits give up after this
 *   tc_sm           (1; 0..1)   tensor-core path: 1 one CTA per SM walking
 *                               stream-K ranges (A operand in TMEM), 0 several
 *                               CTAs per SM with fixed split-K
 * INVALID_ARG for an unknown name or a value out of range (nothing changes).
 */
int w12_set_option(const char *name, int64_t value);

int w12_get_option(const char *name, int64_t *value);

/*
 * Diagnostic: launch one kernel on `stream` that waits on a barrier nothing
 * ever completes, giving up after timeout_us microseconds and recording the
 * timeout in the status word — the same bounded-wait path the GEMM uses, with
 * no fault.  A following w12_check_status(stream) returns W12_ERR_TIMEOUT.
 * (No passage of the pages covers this; it tests the library's failure path.)
 */
int w12_selftest_timeout(uint32_t timeout_us, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* W12_H */
