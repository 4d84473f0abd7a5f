/*
 * affqmm.h -- C ABI of libaffqmm, the GB300 (sm_103a) group-affine quantized
 * linear projection.
 *
 * The operation (MLX affine tables, as used by the TensorFold pages):
 *
 *     W[n,k] = bf16( s[n, k/g] * q[n,k] + b[n, k/g] )      one rounding
 *     y[m,n] = bf16( sum_k x[m,k] * W[n,k] )                fp32 accumulation
 *
 *   - q are integer codes of `bits` bits (2, 3, 4, 5, 6 or 8) with one bf16
 *     scale s and one bf16 bias b per group of g = 32, 64 or 128 consecutive
 *     k of a row: "cuda gemma4: images on the 12B" page, the embed_rows
 *     commit (MLX's affine tables at those widths and group sizes), and the
 *     widths commit of the same page (AffineN tiles).
 *   - each weight is rounded once, bf16(fma(s, q, b)), and the products are
 *     accumulated over the whole depth: "Gemma 4 12B on the native Metal
 *     engine" page, the commit where the prompt tiles dequantize each weight
 *     the way mlx-lm's quantized matmul does.
 *   - M = 1..16 activation rows (decode lanes) run a memory-bound kernel;
 *     M >= 17 runs the tcgen05 tensor-core kernel in chunks of up to 128 rows
 *     (prompt chunks: the same page's commit that runs a window's 128 rows on
 *     one read of the weights).
 *
 * Conventions for every entry point:
 *   - Device pointers are CUDA device (or managed) memory of the current
 *     device; host pointers are named as such.  All work is enqueued on
 *     `stream` (a cudaStream_t; NULL means the legacy default stream) and is
 *     asynchronous: the call returns once the launches are queued.
 *   - The caller allocates and owns every buffer; the library never
 *     allocates device memory and keeps no state between calls.  The
 *     exceptions: affqmm_run_noalloc works in a fixed scratch array that the
 *     library's module places in device memory (see there), and the test
 *     hook affqmm_test_fault_wait sets a process-wide switch.
 *   - Every argument is validated on the host before anything is launched.
 *     A rejected call returns a nonzero affqmm_status, which names the reason
 *     (affqmm_strerror), and launches nothing -- refusals by name, as the
 *     pages' engines refuse what they do not serve ("Gemma 4 12B on the
 *     native Metal engine" page, the serving commit that refuses unsupported
 *     options by name).  Nothing is thrown or aborted across the ABI.
 *   - bf16 values travel as uint16_t bit patterns.
 */
#ifndef AFFQMM_H
#define AFFQMM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define AFFQMM_API __attribute__((visibility("default")))
#else
#define AFFQMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    AFFQMM_OK = 0,
    AFFQMM_E_NULL = 1,      /* a required pointer is NULL */
    AFFQMM_E_BITS = 2,      /* bits not in {2,3,4,5,6,8} */
    AFFQMM_E_GROUP = 3,     /* group not in {32,64,128} */
    AFFQMM_E_SHAPE = 4,     /* N < 0, K < 0, K % group != 0, or sizes that overflow */
    AFFQMM_E_ALIGN = 5,     /* a pointer violates its stated alignment */
    AFFQMM_E_M = 6,         /* M < 0 or M > AFFQMM_MAX_M */
    AFFQMM_E_WORKSPACE = 7, /* workspace NULL or smaller than affqmm_workspace_bytes */
    AFFQMM_E_TIMEOUT = 8,   /* a bounded device wait gave up (see affqmm_workspace_status) */
    AFFQMM_E_CUDA = 9,      /* a CUDA runtime call or launch failed */
    AFFQMM_E_ARG = 10,      /* other bad argument: count, mismatched stacked weights */
    AFFQMM_E_DEVICE = 11,   /* the current device is not an sm_103 GPU */
    AFFQMM_E_SCRATCH = 12   /* affqmm_run_noalloc: the call needs more than its built-in scratch */
} affqmm_status;

/* Largest M one call accepts (larger batches: split them). */
#define AFFQMM_MAX_M (1 << 20)
/* Most projections one affqmm_run_stacked call takes. */
#define AFFQMM_MAX_STACK 8
/* Leading workspace bytes that must be zero between calls (status + counters). */
#define AFFQMM_WORKSPACE_ZEROED (256 + 65536 * 4)

/* A packed weight: a non-owning view of memory filled by affqmm_pack.
 * `packed` is device memory of affqmm_packed_bytes(bits, group, N, K) bytes,
 * 256-byte aligned.  Its layout is private to this library and may change
 * between versions; only affqmm_pack writes it. */
typedef struct {
    int32_t bits;
    int32_t group;
    int64_t N;
    int64_t K;
    const void* packed;
} affqmm_weight;

/* A static string naming a status code (never NULL). */
AFFQMM_API const char* affqmm_strerror(int status);

/* Library version as major*10000 + minor*100 + patch. */
AFFQMM_API int affqmm_version(void);

/* Bytes of packed storage for an N x K table (host call, no GPU needed).
 * The table is MLX's affine one -- codes of 2, 3, 4, 5, 6 or 8 bits with a
 * bf16 scale and bias per group of 32, 64 or 128 along a row ("cuda gemma4:
 * images on the 12B" page, the embed_rows commit) -- stored in this
 * library's own aligned blocks, as the "Gemma 4 12B on the native Metal
 * engine" page copies each linear's tensors to aligned storage for the
 * projection's word reads (its commit on aligned copies of the MLX tensors).
 * Rows are padded to multiples of 128 and the depth to multiples of 128; the
 * padding holds zero codes with zero scale and bias.  When N and K are
 * multiples of 128 the size is N*K*bits/8 + 4*N*K/group bytes: the codes and
 * one scale and one bias per group, nothing more.
 * Errors: E_NULL (bytes), E_BITS, E_GROUP, E_SHAPE. */
AFFQMM_API int affqmm_packed_bytes(int bits, int group, int64_t N, int64_t K, size_t* bytes);

/* Pack a canonical affine table into the library's layout (the table of the
 * embed_rows commit of the "cuda gemma4: images on the 12B" page: MLX's
 * affine tables at 2/3/4/5/6/8 bits, groups of 32/64/128; copied into
 * aligned blocks as the Metal page's aligned-copies commit does for the
 * projection's u32 word reads).
 *   codes   device, uint8 [N, K] row-major, one code per byte; bits above
 *           `bits` are ignored (a code is taken modulo 2^bits)
 *   scales  device, bf16 [N, K/group] row-major
 *   biases  device, bf16 [N, K/group] row-major
 *   packed  device, affqmm_packed_bytes() bytes, 256-byte aligned, written
 * The same table as MLX's affine quantization stores it (scale and bias per
 * group along a row), unpacked to one code per byte.  The packing kernel
 * makes its writes visible device-wide before it finishes, so a run call
 * enqueued right after it on the same stream reads the new weights (see
 * affqmm_run on weights written by the preceding kernel).
 * Errors: E_NULL, E_BITS, E_GROUP, E_SHAPE, E_ALIGN, E_CUDA. */
AFFQMM_API int affqmm_pack(int bits, int group, int64_t N, int64_t K,
                const uint8_t* codes, const uint16_t* scales, const uint16_t* biases,
                void* packed, void* stream);

/* Bytes of workspace that affqmm_run needs for this weight and M on the
 * current device: a status word, merge counters and the fp32 partial sums of
 * the depth split, which the pages' lane projection also makes ("Gemma 4 12B
 * on the native Metal engine" page, the per-shape K-split commit: o and down
 * split 4 ways, gate/up and the head 8); here the split is cut evenly over
 * the device's SMs and its partials are added in a fixed order.  0 when the
 * call needs none.
 * Errors: E_NULL, E_BITS, E_GROUP, E_SHAPE, E_M, E_DEVICE, E_CUDA. */
AFFQMM_API int affqmm_workspace_bytes(const affqmm_weight* w, int64_t M, size_t* bytes);

/* The same for a stacked call (affqmm_run_stacked) over the `count` weights
 * of the host array `ws`. */
AFFQMM_API int affqmm_workspace_bytes_stacked(int count, const affqmm_weight* ws, int64_t M,
                                   size_t* bytes);

/* y = bf16(x . W^T), fp32 accumulation, the weights dequantized on the fly.
 *   w          host pointer to the weight view (its `packed` is device memory)
 *   x          device, bf16 [M, K] row-major, 16-byte aligned
 *   y          device, bf16 [M, N] row-major, 2-byte aligned; fully written
 *   workspace  device, >= affqmm_workspace_bytes bytes, 256-byte aligned.
 *              Its first AFFQMM_WORKSPACE_ZEROED bytes (a status word and the
 *              merge counters) must be zero before its first use; every call
 *              that returns AFFQMM_OK leaves them zero again, the rest is
 *              scratch.  May be NULL when the required size is 0.  Calls that
 *              share a workspace must not overlap on the GPU.  After a call
 *              reported AFFQMM_E_TIMEOUT, zero that prefix again.
 * M = 0 or N = 0 launches nothing; K = 0 writes zeros.
 * The result is deterministic: the same inputs give the same bits.
 * Ordering: the kernels are launched with programmatic dependent launch.
 * They read x, and write y and the workspace, only after waiting for the
 * kernel ahead of them in the stream, but they start copying the packed
 * weights before that wait.  So the packed weights must be complete when the
 * preceding kernel on `stream` lets its dependents start: affqmm_pack
 * guarantees it; a caller's own kernel that writes packed weights must fence
 * its writes device-wide (__threadfence) before it finishes and must not
 * trigger its dependents early, or the two must be separated by an event
 * wait or a stream synchronization.
 * Errors: E_NULL, E_BITS, E_GROUP, E_SHAPE, E_ALIGN, E_M, E_WORKSPACE,
 *         E_DEVICE, E_CUDA. */
AFFQMM_API int affqmm_run(const affqmm_weight* w, const uint16_t* x, int64_t M, uint16_t* y,
               void* workspace, size_t ws_bytes, void* stream);

/* The exact-codes form of the projection for M <= 16 activation rows -- the
 * pages' lane projection ("Gemma 4 12B on the native Metal engine" page, the
 * reg-variant commit: codes kept exact, group sums of x precomputed):
 *     y[m, n] = bf16( sum_g ( s_g * sum_{k in g} q[n,k] x[m,k]
 *                             + b_g * sum_{k in g} x[m,k] ) ),   fp32 sums
 * The weights are never rounded to bf16, so the result differs from
 * affqmm_run by the rounding of bf16(s * q + b).  Arguments, workspace and
 * errors as affqmm_run, except that M > 16 is refused with E_M.  Same inputs,
 * same bits. */
AFFQMM_API int affqmm_run_exact(const affqmm_weight* w, const uint16_t* x, int64_t M, uint16_t* y, void* workspace,
                                size_t ws_bytes, void* stream);

/* The exact-codes form with the group sums of x supplied by the kernel that
 * produced x ("Gemma 4 12B on the native Metal engine" page: the norm,
 * merge, attention-tail, geglu and dense-tail kernels write the next
 * projection's group sums, so the lane projection runs without computing
 * its own):
 *     y[m, n] = bf16( sum_g ( s_g * sum_{k in g} q[n,k] x[m,k] + b_g * xsums[m, g] ) )
 *   xsums   device, fp32 [M, K/group] row-major, 4-byte aligned: the sums of
 *           each group of x (in whatever fixed order the producer added
 *           them); used as given
 * Arguments, workspace, ordering and errors as affqmm_run_exact (M <= 16),
 * plus E_NULL for a NULL xsums when M > 0 and K > 0, and E_ALIGN. */
AFFQMM_API int affqmm_run_exact_sums(const affqmm_weight* w, const uint16_t* x, const float* xsums, int64_t M,
                                     uint16_t* y, void* workspace, size_t ws_bytes, void* stream);

/* Forms of the decode projection for affqmm_run_geglu. */
#define AFFQMM_FORM_ROUNDED 0     /* bf16(s*q + b) weights, as affqmm_run */
#define AFFQMM_FORM_EXACT 1       /* exact codes, the kernel's own group sums of x, as affqmm_run_exact */
#define AFFQMM_FORM_EXACT_SUMS 2  /* exact codes with the caller's group sums, as affqmm_run_exact_sums */

/* A gate/up stack with GeGLU as its epilogue ("Gemma 4 12B on the native
 * Metal engine" page: geglu fused into the gate/up projection's epilogue,
 * the stack's rows interleaved in 16-row blocks, the fused results equal to
 * the unfused ones; "cuda gemma4" page: mlx_lm's gelu_approx(gate) * up as
 * MLX's bf16 operations).
 *   w      the stack, N = 2F rows interleaved in 16-row blocks: rows
 *          32j .. 32j + 15 are gate rows 16j .. 16j + 15, rows 32j + 16 ..
 *          32j + 31 the up rows of the same hidden units; N % 32 == 0
 *   form   AFFQMM_FORM_ROUNDED, _EXACT or _EXACT_SUMS (xsums as
 *          affqmm_run_exact_sums; ignored otherwise)
 *   h      device, bf16 [M, F] row-major, 2-byte aligned; fully written:
 *              h[m, f] = gelu_approx(gate) * up,
 *          gate and up the bf16 outputs the projection alone would store for
 *          the two rows, and gelu_approx(g) = 0.5 g (1 + tanh(sqrt(2/pi)
 *          (g + 0.044715 g^3))) with every operation rounded to bf16 and the
 *          constants taken as bf16; tanh is the device's tanhf
 * M <= 16; workspace and ordering as affqmm_run.
 * Errors: as affqmm_run, plus E_M for M > 16, E_SHAPE for N % 32 != 0, E_ARG
 * for an unknown form. */
AFFQMM_API int affqmm_run_geglu(const affqmm_weight* w, const uint16_t* x, const float* xsums, int64_t M, int form,
                                uint16_t* h, void* workspace, size_t ws_bytes, void* stream);

/* Several projections of the same x in one launch: a layer's q/k/v or
 * gate/up stack ("Gemma 4 12B on the native Metal engine" page, the commit
 * that packs each layer's q/k/v, o, gate/up and down stacks and the tied
 * head once, so that a layer runs on a handful of packed shapes).
 *   ws      host array of `count` weight views (1 <= count <= AFFQMM_MAX_STACK)
 *           with equal K, bits and group, passed by value in one array (the
 *           views are small structs; an array of them is what the caller
 *           builds once per layer)
 *   ys      host array of `count` device pointers, ys[i] is bf16 [M, ws[i].N]
 * Each ys[i] equals affqmm_run(&ws[i], x, ...) bit for bit.  Workspace and
 * ordering as affqmm_run, sized by affqmm_workspace_bytes_stacked.
 * Errors: as affqmm_run, plus E_ARG for a bad count or mismatched weights. */
AFFQMM_API int affqmm_run_stacked(int count, const affqmm_weight* ws, const uint16_t* x, int64_t M,
                       uint16_t* const* ys, void* workspace, size_t ws_bytes, void* stream);

/* affqmm_run with the activations and outputs in host memory, the whole
 * step of a caller that keeps x and y on the host: x is copied into x_dev,
 * the projection runs, y_dev is copied back into y -- all enqueued on
 * `stream` in that order.  When x and y are page-locked host memory (which
 * the GPU can address), both transfers are small kernels chained to the
 * projection: x is read from host memory while the previous kernel in the
 * stream finishes, and y is written to host memory as soon as the projection
 * has finished.  Otherwise the driver's asynchronous copies move them.
 *   x        host, bf16 [M, K] row-major (page-locked memory keeps the call
 *            asynchronous; pageable memory works and makes it synchronous)
 *   y        host, bf16 [M, N] row-major; complete once the stream reaches
 *            the end of the call
 *   x_dev    device, bf16 [M, K], 16-byte aligned: where x is staged
 *   y_dev    device, bf16 [M, N], 2-byte aligned: where y is computed
 *   w, M, workspace, ws_bytes, stream   as affqmm_run
 * The host buffers must stay valid until the stream has passed the call.
 * y equals affqmm_run on the same inputs bit for bit.  Every argument is
 * checked before anything is enqueued.
 * Errors: as affqmm_run (x_dev, y_dev and the host pointers each NULL-checked). */
AFFQMM_API int affqmm_run_host(const affqmm_weight* w, const uint16_t* x, int64_t M, uint16_t* y, uint16_t* x_dev,
                               uint16_t* y_dev, void* workspace, size_t ws_bytes, void* stream);

/* Test hook: write the dequantized weights W (bf16 [N, K] row-major, device,
 * 2-byte aligned) with the same device arithmetic the run kernels use.
 * Errors: E_NULL, E_BITS, E_GROUP, E_SHAPE, E_ALIGN, E_CUDA. */
AFFQMM_API int affqmm_dequant(const affqmm_weight* w, uint16_t* w_out, void* stream);

/* Scaled embedding rows gathered from a packed table: for t < T,
 *     out[t, k] = bf16( W[ids[t], k] * scale ),  W[n, k] = bf16(s * q + b),
 * each of the two roundings applied to an exact value ("cuda gemma4: images
 * on the 12B" page, the embed_rows commit: Gemma's embedding times
 * bf16(sqrt(hidden))).  The table is any packed weight (a tied head serves).
 *   w          host pointer to the weight view: N rows (vocabulary), K values each
 *   ids        device, int32 [T]
 *   T          rows to gather; 0 launches nothing
 *   has_scale  0: out = W's rows (no second rounding); else multiply by `scale`
 *   scale      bf16 bit pattern
 *   out        device, bf16 [T, K] row-major, 16-byte aligned; fully written
 *   status     device uint32 or NULL: an id outside [0, N) gives a zero row and
 *              sets bit 1 of *status (the caller zeroes it beforehand)
 * Errors: E_NULL, E_BITS, E_GROUP, E_SHAPE, E_ALIGN, E_ARG (T < 0), E_CUDA. */
AFFQMM_API int affqmm_embed_rows(const affqmm_weight* w, const int32_t* ids, int64_t T, int has_scale,
                                 uint16_t scale, uint16_t* out, uint32_t* status, void* stream);

/* The embedding gather from a row-contiguous copy of the table (an
 * extension with no counterpart on the pages; the values are those of
 * affqmm_embed_rows, bit for bit).  The packed blocks keep a row's bytes
 * between those of 31 other rows, so a gather of scattered rows from them
 * fetches several times the bytes it uses; the copy keeps each row's bytes
 * in one contiguous range.  It is made once per table, on the device, by
 * affqmm_pack_rows, and costs about as much memory as the packed table.
 *
 * affqmm_rows_bytes: bytes of the copy of an N x K table (host call):
 *   N * stride, stride = ceil(K/128) * (16*bits + 512/group) bytes rounded
 *   up to 16.  Errors as affqmm_packed_bytes.
 * affqmm_pack_rows: write the copy of the packed weight w into `rows`
 *   (device, affqmm_rows_bytes() bytes, 256-byte aligned).  Like
 *   affqmm_pack, the kernel makes its writes visible device-wide before it
 *   finishes.  Errors: E_NULL, E_BITS, E_GROUP, E_SHAPE, E_ALIGN, E_CUDA.
 * affqmm_embed_rows_copy: affqmm_embed_rows with the rows read from `rows`,
 *   a copy that affqmm_pack_rows made of w (w itself is only read for its
 *   bits, group, N and K; its packed pointer must still be valid).  Same
 *   arguments, results and errors, plus E_NULL / E_ALIGN for `rows`. */
AFFQMM_API int affqmm_rows_bytes(int bits, int group, int64_t N, int64_t K, size_t* bytes);
AFFQMM_API int affqmm_pack_rows(const affqmm_weight* w, void* rows, void* stream);
AFFQMM_API int affqmm_embed_rows_copy(const affqmm_weight* w, const void* rows, const int32_t* ids, int64_t T,
                                      int has_scale, uint16_t scale, uint16_t* out, uint32_t* status,
                                      void* stream);

/* Read the device status word of a workspace that run calls used
 * (synchronizes `stream`).  Returns AFFQMM_OK, or AFFQMM_E_TIMEOUT when a
 * kernel that used this workspace gave up a bounded wait (its outputs are
 * then invalid); in that case the whole AFFQMM_WORKSPACE_ZEROED prefix
 * (status word and merge counters) is zeroed again, so the workspace serves
 * the next call as it is. */
AFFQMM_API int affqmm_workspace_status(void* workspace, void* stream);

/* Test hook for the timeout path (no counterpart on the pages): while
 * `cycles` > 0, every decode launch (M <= 16) that this process makes
 * afterwards first has its consumer warps wait, at most `cycles` SM clock
 * cycles, on a barrier that nothing completes.  The wait runs out; the launch
 * sets its workspace status word (affqmm_workspace_status then returns
 * AFFQMM_E_TIMEOUT), writes no output, waits for the copies it started and
 * exits.  0 restores normal launches.  Not for production use.
 * Errors: E_ARG (cycles < 0). */
AFFQMM_API int affqmm_test_fault_wait(int64_t cycles);

/* Largest M affqmm_run_noalloc takes, and the size of its built-in scratch. */
#define AFFQMM_NOALLOC_MAX_M 16
#define AFFQMM_NOALLOC_SCRATCH_BYTES (8u << 20)

/* affqmm_run for M <= 16 activation rows without any device memory from the
 * caller beyond x and y.  The method's pages have no counterpart to this entry point:
 * it is a convenience of this library.
 *
 * Who needs it: code that runs where it cannot allocate device memory -- a
 * plug-in inside a host engine that owns all of the GPU's memory and hands
 * its plug-ins no allocator, or a latency-critical loop that must not call
 * cudaMalloc/cudaFree (they can synchronize the device) once it has started.
 * Such callers cannot supply the workspace affqmm_run wants, so this call
 * uses a scratch array of AFFQMM_NOALLOC_SCRATCH_BYTES (8 MiB) that the
 * library itself places in device memory; every GPU that loads the library
 * holds it until the process exits.  The call allocates nothing: no
 * cudaMalloc, no cudaFree, no allocating library routine.
 *
 *   w, x, y, stream  as affqmm_run (x 16-byte aligned, y fully written)
 *
 * - The first call on a device finds the scratch's device address (once per
 *   device, with that device current) and sets the kernels' shared-memory
 *   limits; make that first call before any stream capture.
 * - Every call on a device shares the one scratch array, which keeps what the
 *   last call left there.  The call clears the parts that must start at zero
 *   (a status word and the merge counters it uses) on `stream` before its
 *   kernel runs.  Calls that overlap on the GPU (different streams, different
 *   host threads without ordering) race on the scratch and give wrong
 *   results: order them on one stream.
 * - This call cannot report a bounded device wait that gave up (never
 *   expected on a healthy GPU; y is then unspecified).  Callers that need
 *   that report use affqmm_run and affqmm_workspace_status.
 * Same result, bit for bit, as affqmm_run on the same inputs.
 * Errors: as affqmm_run (no E_WORKSPACE), plus E_SCRATCH when M > 16 or when
 * the split of the work on this device would need more than the scratch. */
AFFQMM_API int affqmm_run_noalloc(const affqmm_weight* w, const uint16_t* x, int64_t M, uint16_t* y,
                                  void* stream);

#ifdef __cplusplus
}
#endif
#endif
