/*
 * il.h -- C ABI of the shared-input batched linear for GB300 (sm_103a).
 *
 * One call runs several matmul jobs over one shared fp32 activation:
 *     y_j[t][n_out_j] = x[t][n_in] * W_j^T        (W_j stored [n_out_j][n_in])
 * following the accelerator backend contract of oxinfer 0.0.0, src/gpu.rs:
 * struct `Job` (one matmul of a batch sharing x), `Backend::upload` (prepare
 * device state for one weight) and `Backend::matmul` (all jobs of a batch in
 * one submission).  There is no CPU fallback: an error returns a negative
 * status and launches nothing.
 *
 * Weight storage formats (enum `WeightRef` of the same page; the page names
 * Q8 and Q4 without defining them, this library fixes them as follows):
 *   IL_BF16: u16 bit patterns of bf16, host layout u16 w[n_out][n_in].
 *   IL_Q8  : symmetric int8, one fp32 scale per 32-element block along n_in;
 *            host layout i8 q[n_out][n_in], then f32 d[n_out][n_in/32]
 *            starting at byte n_out*n_in.  w = fp32(d*q).
 *   IL_Q4  : symmetric signed 4-bit (two's complement), two per byte, element
 *            2k in bits 0-3 of byte k and 2k+1 in bits 4-7; one fp32 scale
 *            per 32-block; host layout u8 p[n_out][n_in/2], then
 *            f32 d[n_out][n_in/32] starting at byte n_out*n_in/2.
 *
 * Threading: every entry point is thread-safe.  The library works on the
 * CUDA device that is current on the calling thread.
 */
#ifndef IL_H_
#define IL_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define IL_VERSION 3

/* Storage format of a weight (oxinfer src/gpu.rs, enum WeightRef). */
typedef enum { IL_BF16 = 0, IL_Q8 = 1, IL_Q4 = 2 } il_format;

/* Status codes.  IL_OK is 0; every error is negative.  An entry point that
 * returns an error has launched no work and written no output. */
typedef enum {
  IL_OK = 0,
  IL_ERR_ARG = -1,            /* null pointer, negative size, misaligned or overlapping buffer */
  IL_ERR_SHAPE = -2,          /* n_in / n_out inconsistent with a handle, or not a legal size */
  IL_ERR_FORMAT = -3,         /* unknown storage format */
  IL_ERR_HANDLE = -4,         /* freed, forged or other-device weight handle */
  IL_ERR_OOM = -5,            /* device allocation failed */
  IL_ERR_CUDA = -6,           /* CUDA runtime or launch error */
  IL_ERR_DEVICE_TIMEOUT = -7, /* a device-side wait gave up (see il_check_device_status) */
  IL_ERR_UNSUPPORTED = -8     /* no sm_103a device current, or a size beyond a documented limit */
} il_status;

/* Opaque device weight (the page's `DeviceWeight`).  Owned by the caller,
 * released with il_free_weight. */
typedef struct il_weight il_weight;

/* One job of a batch (the page's `Job`): y[t][n_out] = x[t][n_in] * W^T.
 *   w     : handle from il_upload_weight; its n_in must equal the batch n_in.
 *   n_out : must equal the handle's n_out.
 *   y     : DEVICE pointer (HOST pointer for il_matmul_batch_host), fp32
 *           [t][n_out] row-major, 4-byte aligned; it is overwritten (not
 *           accumulated) and must not overlap x or any other job's y. */
typedef struct {
  const il_weight* w;
  int64_t n_out;
  float* y;
} il_job;

/* Cumulative counters (the page's `Backend::stats`, as numbers). */
typedef struct {
  uint64_t uploads;           /* successful il_upload_weight calls        */
  uint64_t upload_bytes;      /* host bytes uploaded (WeightRef::bytes)   */
  uint64_t batches;           /* successful il_matmul_batch* calls        */
  uint64_t jobs;              /* jobs in those batches                    */
  uint64_t launches;          /* kernels launched by those batches        */
  uint64_t weight_bytes;      /* weight bytes those batches streamed      */
  uint64_t flops;             /* 2 * t * n_in * rows summed over jobs     */
  uint64_t errors;            /* calls that returned an error             */
  uint64_t profiled_batches;  /* IL_PROFILE=1: calls whose device time is in device_ns */
  uint64_t device_ns;         /* IL_PROFILE=1: their summed device time (ns)           */
} il_stats;

/*
 * il_upload_weight -- oxinfer src/gpu.rs, `Backend::upload` ("prepares
 * device-side state for a weight matrix").
 *   format   : il_format.
 *   host_ptr : HOST pointer to the weight in the host layout above; only read
 *              during the call (it is copied, then repacked on the device).
 *              Q8/Q4 scales are read with 4-byte loads from the host copy, so
 *              any alignment is accepted.
 *   n_out    : rows, 1 <= n_out <= 2^31 - 1.
 *   n_in     : columns, 1 <= n_in <= 32768; a multiple of 8 for IL_BF16 and of
 *              32 for IL_Q8 / IL_Q4.
 * Returns a new handle, or NULL on error (il_last_error() says why).
 * Synchronous: when it returns the packed weight is resident in HBM.
 */
il_weight* il_upload_weight(int format, const void* host_ptr, int64_t n_out, int64_t n_in);

/*
 * il_matmul_batch -- oxinfer src/gpu.rs, `Backend::matmul` ("runs a batch of
 * matmuls over one shared input in a single submission").
 *   x      : DEVICE pointer, fp32 [t][n_in] row-major, 16-byte aligned.
 *   t      : tokens, 0 <= t <= 2^20.  t == 0 is a successful no-op.
 *   n_in   : must equal every job's handle n_in.
 *   jobs   : HOST array of n_jobs il_job (read during the call only).
 *   n_jobs : 0 <= n_jobs <= 4096; 0 is a successful no-op.
 *   stream : cudaStream_t to enqueue on (NULL = legacy default stream).
 * All arguments are validated, and every launch of the batch is worked out in
 * full (plans, tensor maps, scratch), before anything is launched; on any such
 * error the call returns a negative il_status with no kernel enqueued and no y
 * written.  Only a launch that the CUDA runtime itself rejects (IL_ERR_CUDA,
 * "launch") can leave the earlier launches of the batch enqueued.  On success
 * the work is enqueued asynchronously on `stream`; x, y and the handles must
 * stay valid until it completes.
 * Kernels: small t runs the grouped decode kernels, each weight byte streamed
 * once: t <= 8 for bf16 weights, t <= 16 for Q8/Q4.  Larger t casts x to bf16
 * once and runs the tensor-core kernel (Q8/Q4 weights dequantised to bf16 in
 * shared memory, bf16(fp32(d*q))).  One launch covers every job of one format,
 * up to 32 jobs on a decode kernel and 8 jobs on the tensor-core kernel; a batch
 * beyond those counts, or with several formats, takes one launch per group.
 * Scratch: the tensor-core path keeps a bf16 copy of x and a split-K workspace
 * per (device, stream), owned by the library.  They grow with the stream-ordered
 * allocator (cudaMallocAsync / cudaFreeAsync on `stream`), so growing never
 * waits for the stream; they cannot grow while `stream` is being captured
 * (IL_ERR_UNSUPPORTED): run one call of the largest size on the stream before
 * capturing it.  il_release_scratch frees them.
 */
int il_matmul_batch(const float* x, int64_t t, int64_t n_in, const il_job* jobs, int n_jobs,
                    void* stream);

/*
 * il_matmul_batch_host -- il_matmul_batch on HOST buffers, the form in which
 * the pages' `Backend::matmul` takes them (oxinfer src/gpu.rs: `x: &[f32]`,
 * and each `Job` holds `y: &mut [f32]`).
 *   x      : HOST pointer, fp32 [t][n_in] row-major (any alignment).
 *   jobs   : as for il_matmul_batch, but every y is a HOST pointer, fp32
 *            [t][n_out] row-major, 4-byte aligned, overwritten.
 *   t, n_in, n_jobs, stream : as for il_matmul_batch.
 * Host memory may be page-locked (cudaHostAlloc, cudaHostRegister, a pinned
 * torch tensor), pageable or managed; a device pointer for x or a y is
 * rejected with IL_ERR_ARG.  Page-locked buffers are used in place: the kernels
 * read x and write y through their mapped device addresses (over NVLink-C2C on
 * GB300), with no copy operation (a page-locked x that is not 16-byte aligned is
 * copied as below).  Other buffers go through a library-owned device buffer:
 * one copy of x in before the launches, and after them one device->host copy
 * per run of y buffers (y buffers that follow one another in host memory, each
 * starting where the previous one ends, come back in one copy).  Everything is
 * enqueued on `stream` and the call returns once it is; y holds the results
 * after `stream` has completed that work (e.g. cudaStreamSynchronize), and x and
 * y must stay valid, x unchanged, until then.  With page-locked memory nothing
 * blocks the calling thread; with pageable memory the copies behave as
 * cudaMemcpyAsync does for it (the copy of y waits for the kernels).
 * Validation and launch preparation happen before anything is enqueued, with
 * the same rule as il_matmul_batch: an error returns a negative il_status with
 * nothing enqueued, except a copy or launch that the CUDA runtime itself
 * rejects (IL_ERR_CUDA) after earlier work of the call was enqueued.  The
 * device buffer of x and y is scratch per (device, stream), grown and freed
 * like the bf16 copy of x (not during stream capture; il_release_scratch).
 */
int il_matmul_batch_host(const float* x, int64_t t, int64_t n_in, const il_job* jobs, int n_jobs,
                         void* stream);

/*
 * il_matmul_batch_noalloc -- the pages have no counterpart of this entry point.
 * Same arguments and checks as il_matmul_batch, the same split over the decode
 * and tensor-core kernels, results equal to il_matmul_batch's within the
 * per-element tolerance (the tensor-core launches here split K only where the
 * two slices of a tile can run as a CTA pair, which needs no workspace), and
 * the same rule that an error enqueues nothing -- but it never allocates
 * device memory: for callers that cannot let a library call cudaMalloc, such
 * as services that give all device memory to their own pool at start-up, or
 * latency-critical threads for which cudaMalloc / cudaFree may block and
 * synchronise the device.
 *   - The bf16 copy of x used by the tensor-core path (t >= 9 with bf16
 *     weights, t >= 17 with Q8/Q4 weights) goes to a fixed 16 MiB device array
 *     inside the library, held by every GPU that loads the library until the
 *     process exits.  A batch needing more, t * round_up(n_in, 256) * 2 bytes
 *     > 16 MiB, is rejected with IL_ERR_UNSUPPORTED (e.g. t = 2048 fits at
 *     n_in = 4096, not at 12288).
 *   - The Q8/Q4 decode kernel's partial sums of tiles whose K it splits over
 *     CTAs go to a fixed 4 MiB device array (with their arrival counters); a
 *     batch whose plan would need more splits K less.
 *   - The first call on a device looks up the arrays' device addresses and
 *     clears the library's status word and counters there, asynchronously on `stream`; make
 *     that first call before any stream capture.
 *   - Every call shares the same arrays: calls that overlap on the GPU (on
 *     different streams, or from different threads) race and may corrupt each
 *     other's results.  Serialise them, e.g. on one stream.
 *   - A device-side wait that gives up records its code in that status word
 *     and ends the kernel early; il_check_device_status reports it.
 */
int il_matmul_batch_noalloc(const float* x, int64_t t, int64_t n_in, const il_job* jobs, int n_jobs,
                            void* stream);

/*
 * il_upload_gate_up -- a fused gate+up weight.  The pages run the gate and up
 * projections as one shared-input batch and pass the two results straight to
 * gelu_mul (oxinfer 0.0.1, src/drafter.rs, `Drafter::step`: `matmul_multi` over
 * gate and up, then `gelu_mul(&mut g, &u)`).  A handle made here computes that
 * pair and the activation in one job:
 *     h[t][n_out] = gelu(x * Wg^T) * (x * Wu^T)        (elementwise)
 * with gelu the tanh form of the Gemma family the pages serve,
 *     gelu(g) = 0.5 * g * (1 + tanh(sqrt(2/pi) * (g + 0.044715 * g^3))).
 * The pages do not print gelu_mul; this is the reading the library takes.
 *   format            : il_format of BOTH weights.
 *   gate_ptr, up_ptr  : HOST pointers, each one weight in the host layout of
 *                       il_upload_weight with the same n_out and n_in; read
 *                       during the call only.
 *   n_out, n_in       : as for il_upload_weight (n_out = width of h).
 * Returns a handle, or NULL on error.  A job of this handle in il_matmul_batch
 * (or il_matmul_batch_noalloc) takes n_out = the width of h and y = h
 * [t][n_out]; it can share a batch with plain jobs.  Inside, the two weights
 * are stored as one matrix of 2*n_out rows, row 2r = gate row r and row 2r+1 =
 * up row r, so every kernel finds a pair in adjacent rows.  il_weight_bytes
 * gives the sum of both weights' bytes; il_weight_info the format, n_out (the
 * width of h) and n_in; il_dequantize_weight writes the interleaved
 * [2*n_out][n_in] matrix.
 */
il_weight* il_upload_gate_up(int format, const void* gate_ptr, const void* up_ptr, int64_t n_out,
                             int64_t n_in);

/*
 * il_centroid_head -- centroid-masked LM head (oxinfer 0.0.1, src/drafter.rs,
 * end of `Drafter::step`): centroid logits cl = centroids * x, the top_k
 * centroids, the exact logits of the tokens of their clusters, and the token
 * of the first maximum.
 *   x          : DEVICE fp32 [h] (one token), 16-byte aligned.
 *   h          : width; must equal both handles' n_in (<= 32768).
 *   centroids  : bf16 handle [n_cent][h], 1 <= n_cent <= 16384 (a plain weight).
 *   embed      : bf16 handle [vocab][h], vocab a multiple of n_cent; cluster c
 *                owns the tokens ordering[c*per .. (c+1)*per), per = vocab / n_cent.
 *   ordering   : DEVICE u32 [vocab].  An entry >= vocab is skipped (never wins)
 *                and flagged in the device status word (see below).
 *   top_k      : >= 1; k = min(top_k, n_cent) clusters are scored.
 *   token_out  : DEVICE u32 [1]: the winning token id.
 *   score_out  : DEVICE fp32 [1] or NULL: its logit.
 *   selected_out : DEVICE u32 [k] or NULL: the selected centroids in rank order.
 *   scores_out : DEVICE fp32 [k*per] or NULL: every scored logit, index i*per + j
 *                for the j-th token of the i-th selected cluster.
 *   stream     : cudaStream_t (NULL = legacy default stream).
 * Order and ties (the page selects with an unstable partition and scans with a
 * strict '>'; this is the reading taken): centroids rank by larger logit, NaN
 * last, ties to the lower index, and are scanned in that order; among equal
 * logits the first in (rank, position) order wins; NaN and -inf never win, and
 * with no winner the token is 0 and the score -inf.  Logits are fp32 sums of
 * bf16 * fp32 products.  Asynchronous; three kernel launches (the centroid
 * logits run as a one-job il_matmul_batch and are counted as a batch).  Calls
 * on one stream are ordered; the library keeps per-stream scratch for it.
 * An out-of-range ordering entry sets the status word, and il_check_device_status
 * then returns IL_ERR_ARG.
 */
int il_centroid_head(const float* x, int64_t h, const il_weight* centroids, const il_weight* embed,
                     const uint32_t* ordering, int64_t top_k, uint32_t* token_out, float* score_out,
                     uint32_t* selected_out, float* scores_out, void* stream);

/* 1 if the handle came from il_upload_gate_up, 0 if from il_upload_weight,
 * -1 for an invalid handle. */
int il_weight_is_gate_up(const il_weight* w);

/* Releases a handle and its device memory (synchronises the device).
 * NULL is ignored; an unknown pointer is ignored and counted as an error. */
void il_free_weight(il_weight* w);

/* Host-layout byte size of the weight, oxinfer src/gpu.rs `WeightRef::bytes`:
 * 2*n_out*n_in (bf16), n_out*n_in*9/8 (Q8), n_out*n_in*5/8 (Q4).  -1 for an
 * invalid handle. */
int64_t il_weight_bytes(const il_weight* w);

/* Format and shape of a handle (for a gate+up handle, n_out is the width of
 * h).  Any out pointer may be NULL. */
int il_weight_info(const il_weight* w, int* format, int64_t* n_out, int64_t* n_in);

/*
 * il_dequantize_weight -- test hook: writes every element of the uploaded
 * weight as fp32 to dev_out [n_out][n_in] (DEVICE pointer, 4-byte aligned),
 * reading the packed device layout with the same element decoders the matmul
 * kernels use.  bf16 widens exactly; Q8/Q4 give fp32(d*q).  Asynchronous on
 * `stream`.  For a gate+up handle dev_out is [2*n_out][n_in], rows interleaved
 * as described at il_upload_gate_up.
 */
int il_dequantize_weight(const il_weight* w, float* dev_out, void* stream);

/* Reads (and clears) the device-side status words that bounded waits in the
 * kernels set when they give up -- the one of il_matmul_batch and
 * il_centroid_head, and the one of il_matmul_batch_noalloc -- on the current
 * device.  Synchronises `stream`.  Returns IL_OK, or IL_ERR_DEVICE_TIMEOUT if a
 * wait timed out since the last call; in that case it also waits for the
 * device and clears the library's split-K workspaces on it, so that later
 * batches start from a clean state.  Returns IL_ERR_ARG if no wait timed out
 * but il_centroid_head met an ordering entry >= vocab. */
int il_check_device_status(void* stream);

/* Frees the scratch the library keeps for `stream` on the current device (the
 * bf16 copy of x, the split-K workspace, the LM-head scratch, the device copies
 * of x and y of il_matmul_batch_host), in stream order:
 * call it before destroying a stream the library has run on.  A later call on
 * the stream allocates afresh.  Returns IL_OK or IL_ERR_CUDA. */
int il_release_scratch(void* stream);

/* Message of the last error on this thread ("" if none). */
const char* il_last_error(void);

/* il_status of the last error on this thread (IL_OK if none); useful after
 * il_upload_weight returned NULL.  Each entry point clears it on entry. */
int il_last_status(void);

/* Copies the cumulative counters into *out (the page's `Backend::stats`, a
 * cumulative timing summary when profiling).  With IL_PROFILE=1 in the
 * environment, il_matmul_batch, il_matmul_batch_host (its launches, not its
 * copies) and il_centroid_head record a CUDA event before and after their
 * launches on their stream (not while the stream is being
 * captured, and not il_matmul_batch_noalloc); il_get_stats then waits for every
 * recorded call to finish and adds its device time to device_ns.  Without
 * IL_PROFILE nothing is recorded and nothing waits.  The entry points also mark
 * their host work with NVTX ranges, which cost nothing unless a tool listens. */
int il_get_stats(il_stats* out);
/* Zeroes the counters (with IL_PROFILE=1, after waiting for the recorded calls). */
void il_reset_stats(void);

/* IL_VERSION of the loaded library. */
int il_version(void);

#ifdef __cplusplus
}
#endif

#endif /* IL_H_ */
