// il_internal.cuh -- declarations shared by the translation units of the
// library: the packed device layout of a weight, the job tables handed to the
// kernels, the element decoders used by both the matmul kernels and the
// dequantise hook, and the launchers.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <cstdlib>
#include <cstring>
#include <memory>
#include <vector>

#include "../../include/il.h"

namespace il {

// ---------------------------------------------------------------------------
// Packed device layout
// ---------------------------------------------------------------------------
// BF16: plain row-major u16 [n_out_pad][n_in_pad], rows padded to a multiple of
//   8 and columns to a multiple of 256 (zeros).  The decode kernel reads 16 bytes
//   (8 consecutive k) per lane; the tensor-core kernel tiles it with TMA
//   (K-major, 128-byte swizzle).
// Q8 / Q4: rows padded to a multiple of 16 (a "pair" of two 8-row groups),
//   columns to a multiple of 256; the weight is a sequence of records, one per
//   (pair, chunk), pair-major: record (p, c) at byte (p * n_chunks + c) * RS.
//   A chunk is kChunkK columns (Q8: 64, Q4: 128), so a group's quants in one
//   chunk are exactly 512 bytes.  A record holds
//     [0, 512)          quants of group 2p   (rows 16p .. 16p+7)
//     [512, 1024)       quants of group 2p+1 (rows 16p+8 .. 16p+15)
//     [1024, 1024+SB)   fp32 scales of group 2p, [8 rows][blocks of the chunk]
//     [1024+SB, RS)     fp32 scales of group 2p+1
//   with SB = 32 * blocks_per_chunk.  In a group's 512 bytes, lane L = 4n + q of
//   a warp owns bytes [16L, 16L+16): the elements of row n that the lane feeds to
//   the MMAs of that chunk (see pack.cu for the order).  Q8 bytes are stored
//   biased, u = q + 128, so that one byte permute makes fp16 1024 + u.
//   Padding decodes to q = 0 with scale 0.
constexpr int kGroupRows = 8;
constexpr int kPairRows = 16;
constexpr int kPadK = 256;
constexpr int kChunkBytes = 512;

__host__ __device__ constexpr int chunk_k(int fmt) { return fmt == IL_BF16 ? 32 : (fmt == IL_Q8 ? 64 : 128); }
__host__ __device__ constexpr int blocks_per_chunk(int fmt) { return fmt == IL_Q8 ? 2 : (fmt == IL_Q4 ? 4 : 0); }
// Scale bytes per (group, chunk): 8 rows x blocks x 4 bytes.
__host__ __device__ constexpr int chunk_scale_bytes(int fmt) { return 32 * blocks_per_chunk(fmt); }
// Bytes of one (pair, chunk) record of a Q8 / Q4 weight: 1152 (Q8), 1280 (Q4).
__host__ __device__ constexpr int record_bytes(int fmt) { return 2 * kChunkBytes + 2 * chunk_scale_bytes(fmt); }
// Row padding of the packed layout.
__host__ __device__ constexpr int pad_rows(int fmt) { return fmt == IL_BF16 ? kGroupRows : kPairRows; }

// A gate+up weight (il_upload_gate_up) is stored as one matrix of n_out = 2*width
// rows, row 2r = gate row r and row 2r+1 = up row r; its jobs write
// h = gelu(gate) * up, `width` columns wide.
struct PackedWeight {
  uint64_t magic;
  int format;
  int device;
  int glu;                     // 1: rows interleaved gate/up, output h = gelu(g) * u
  int64_t n_out, n_in;         // n_out: packed rows (2 * width of h for glu)
  int64_t n_out_pad, n_in_pad;
  int64_t n_groups, n_chunks;  // n_out_pad / 8, n_in_pad / chunk_k
  uint8_t* quants;             // device, packed as above (Q8/Q4: the records, scales inside)
  int64_t host_bytes;          // WeightRef::bytes
  size_t device_bytes;
};
constexpr uint64_t kWeightMagic = 0x696c5f7765696768ull;  // "il_weigh"

// Columns of a job's output: n_out, or n_out / 2 for a gate+up weight.
inline int64_t out_width(const PackedWeight& w) { return w.glu ? w.n_out / 2 : w.n_out; }

// ---------------------------------------------------------------------------
// Decode (t <= 8) job table, passed by value as a kernel parameter
// ---------------------------------------------------------------------------
constexpr int kMaxDecodeJobs = 32;

struct DecodeJob {
  const uint8_t* w;      // packed weight (bf16 rows, or Q8/Q4 records)
  float* y;              // [t][n_out], or h [t][n_out / 2] when glu
  int32_t n_out;         // packed rows
  int32_t group_begin;   // first global 8-row group of this job (even for Q8/Q4)
  int64_t row_stride;    // bf16: n_in_pad (elements); Q8/Q4: n_chunks
  int32_t glu;           // rows interleaved gate/up: store gelu(g) * u
  int32_t pad_;
};

struct DecodeParams {
  const float* x;        // [t][n_in] fp32
  int t;                 // 1..8 tokens handled by this launch
  int x_row_stride;      // elements between token rows of x
  int n_in;
  int n_chunks;          // chunks over n_in_pad
  int chunks_per_slice;  // chunks per cluster rank (K slice)
  int slices;            // cluster size along K
  int total_groups;
  int n_rowblocks;
  int n_jobs;
  int prefetch;          // bf16 decode: weight batches per warp staged in shared memory before the wait
  DecodeJob jobs[kMaxDecodeJobs];
};

// ---------------------------------------------------------------------------
// Element decoders (shared by the decode kernel and the dequantise hook)
// ---------------------------------------------------------------------------
// Programmatic dependent launch: kernels are launched so that the next kernel
// on the stream may start while this one drains.  A kernel waits for the grid
// before it (griddepcontrol.wait) before reading anything that grid may write
// (x) or writing anything it may read (y); work on inputs fixed at upload time
// (the weights) may run before the wait.  Without a preceding grid both are no-ops.
#ifndef IL_NO_PDL
constexpr bool kUsePdl = true;
#else
constexpr bool kUsePdl = false;
#endif
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// fp16 decoders (the Q8/Q4 matmul path multiplies fp16 weights by fp16 x):
// every |q| <= 128 is exact in fp16, and the fp16 with biased exponent 25 is
// 1024 + its 10-bit mantissa, so one byte permute builds 1024 + u from a byte u.
// Q8: word of 4 packed bytes u = q + 128 -> fp16x2 pairs (e0,e1), (e2,e3), each
// exactly q.
__device__ __forceinline__ void q8_word_to_f16x2(uint32_t u, uint32_t& p01, uint32_t& p23) {
  uint32_t a = __byte_perm(u, 0x64646464u, 0x5140);        // [u0, 0x64, u1, 0x64]
  uint32_t b = __byte_perm(u, 0x64646464u, 0x5342);        // [u2, 0x64, u3, 0x64]
  const __half2 bias = __floats2half2_rn(1152.0f, 1152.0f);  // 1024 + 128
  __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
  __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
  p01 = *reinterpret_cast<uint32_t*>(&ha);
  p23 = *reinterpret_cast<uint32_t*>(&hb);
}

// Q4: the four fp16x2 pairs of one packed word, pair i made of the nibbles at
// positions i and i+4 (bits 4i and 16+4i), each exactly q.  Nibbles at the
// bottom of a byte give 1024 + (n^8); those at the top give 1024 + 16*(n^8),
// which a multiply by 1/16 brings back, so only one shift is needed.
__device__ __forceinline__ void q4_word_to_f16x2(uint32_t word, uint32_t (&pr)[4]) {
  const uint32_t hi = word >> 8;
  uint32_t v0, v1, v2, v3;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(v0) : "r"(word), "n"(0x000F000F), "n"(0x64086408));
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(v1) : "r"(word), "n"(0x00F000F0), "n"(0x64806480));
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(v2) : "r"(hi), "n"(0x000F000F), "n"(0x64086408));
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(v3) : "r"(hi), "n"(0x00F000F0), "n"(0x64806480));
  const __half2 b0 = __floats2half2_rn(1032.0f, 1032.0f);      // 1024 + 8
  const __half2 m1 = __floats2half2_rn(0.0625f, 0.0625f);      // 1/16
  const __half2 b1 = __floats2half2_rn(-72.0f, -72.0f);        // -(64 + 8)
  __half2 h0 = __hsub2(*reinterpret_cast<const __half2*>(&v0), b0);
  __half2 h1 = __hfma2(*reinterpret_cast<const __half2*>(&v1), m1, b1);
  __half2 h2 = __hsub2(*reinterpret_cast<const __half2*>(&v2), b0);
  __half2 h3 = __hfma2(*reinterpret_cast<const __half2*>(&v3), m1, b1);
  pr[0] = *reinterpret_cast<uint32_t*>(&h0);
  pr[1] = *reinterpret_cast<uint32_t*>(&h1);
  pr[2] = *reinterpret_cast<uint32_t*>(&h2);
  pr[3] = *reinterpret_cast<uint32_t*>(&h3);
}

__device__ __forceinline__ float f16_lo(uint32_t v) {
  return __half2float(__ushort_as_half((unsigned short)(v & 0xFFFFu)));
}
__device__ __forceinline__ float f16_hi(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v >> 16))); }

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// gelu in the tanh form used by the Gemma family (the model the pages' drafter
// belongs to): 0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))).  Applied to the
// fp32 gate result, then multiplied by the fp32 up result.
// Since 1 + tanh(z) = 2 / (1 + e^(-2z)), gelu(g) = g / (1 + e^(-2z)): one
// exponential and one fast division instead of a tanh.  The exponent is capped
// at 88 (e^88 ~ 1.7e38 is still finite); there the quotient is 0 to fp32, which
// is gelu's limit.
__device__ __forceinline__ float gelu_mul(float g, float u) {
  const float z = 0.7978845608028654f * fmaf(0.044715f * g, g * g, g);
  return __fdividef(g, 1.0f + __expf(fminf(-2.0f * z, 88.0f))) * u;
}

// ---------------------------------------------------------------------------
// Prepared launches
// ---------------------------------------------------------------------------
// A kernel launch worked out in full on the host -- grid, attributes, and the
// argument values copied into storage the record owns.  Every entry point
// prepares all launches of a call (plans, tensor maps, occupancy queries, size
// checks) before it enqueues the first, so a call that fails while preparing
// has enqueued nothing.
struct Launch {
  const void* fn = nullptr;
  dim3 grid, block;
  size_t smem = 0;
  cudaLaunchAttribute attr[3];
  int nattr = 0;
  std::shared_ptr<unsigned char> store;
  void* args[20];
  int nargs = 0;

  // Copies the arguments (each of the kernel's parameter type) into 64-byte
  // aligned storage.  False if the host allocation fails.
  template <class... A>
  bool set_args(const A&... a) {
    constexpr size_t n = sizeof...(A);
    static_assert(n >= 1 && n <= 20, "1 to 20 kernel arguments");
    const size_t sizes[n] = {sizeof(A)...};
    const size_t aligns[n] = {alignof(A)...};
    const void* srcs[n] = {static_cast<const void*>(&a)...};
    size_t offs[n];
    size_t total = 0;
    for (size_t i = 0; i < n; ++i) {
      const size_t al = aligns[i] > 16 ? aligns[i] : 16;
      total = (total + al - 1) / al * al;
      offs[i] = total;
      total += sizes[i];
    }
    unsigned char* mem = static_cast<unsigned char*>(std::aligned_alloc(64, (total + 63) / 64 * 64));
    if (mem == nullptr) return false;
    store.reset(mem, std::free);
    for (size_t i = 0; i < n; ++i) {
      std::memcpy(mem + offs[i], srcs[i], sizes[i]);
      args[i] = mem + offs[i];
    }
    nargs = (int)n;
    return true;
  }
  void allow_early_start() {  // programmatic dependent launch (see grid_dep_wait)
    attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[nattr].val.programmaticStreamSerializationAllowed = 1;
    ++nattr;
  }
  void set_cluster(int c) {
    attr[nattr].id = cudaLaunchAttributeClusterDimension;
    attr[nattr].val.clusterDim.x = c;
    attr[nattr].val.clusterDim.y = 1;
    attr[nattr].val.clusterDim.z = 1;
    ++nattr;
  }
};

// Enqueues the prepared launches in order on `stream`, counting each in
// *launches.  Stops at the first launch the runtime rejects.
cudaError_t run_launches(const std::vector<Launch>& v, cudaStream_t stream, int* launches);

// Upload-time repack and the dequantise hook: single launches, enqueued directly.
cudaError_t launch_pack(const PackedWeight& w, const uint8_t* staging, cudaStream_t stream);
cudaError_t launch_dequant(const PackedWeight& w, float* out, cudaStream_t stream);
// Tokens of one decode launch: bf16 weights 8 (the MMA's 8 columns), Q8/Q4 16 (two
// groups of 8 columns fed by the same decoded weights).
constexpr int kDecodeTokensBf16 = 8;
constexpr int kDecodeTokensQ = 16;

// Decode kernel for one launch of tokens (see above): bf16 weights run the register-streaming kernel
// (gemv.cu), Q8 / Q4 weights the shared-memory ring kernel (qdecode.cu), whose
// bounded waits record a code in `status` when they give up.
cudaError_t prepare_decode(int fmt, const DecodeParams& p, int num_sms, unsigned* status, void* ws,
                           size_t ws_bytes, Launch* out);
cudaError_t prepare_decode_bf16(const DecodeParams& p, int num_sms, Launch* out);
// ws / ws_bytes: split workspace (nullptr: K is never split over CTAs).
cudaError_t prepare_qdecode(int fmt, const DecodeParams& p, int num_sms, unsigned* status, void* ws,
                            size_t ws_bytes, Launch* out);
// Split workspace the Q8/Q4 decode launch of `p` would use given unlimited room
// (0: none).
size_t qdecode_workspace_bytes(int fmt, const DecodeParams& p, int num_sms);
cudaError_t prepare_cast_bf16(const float* x, int64_t t, int64_t n_in, int64_t n_in_pad, __nv_bfloat16* out,
                              int num_sms, Launch* L);

// Token counts from which a batch takes the tensor-core path instead of the
// decode kernels (which stream the weights once per launch of tokens).
constexpr int64_t kGemmMinT = 9;        // bf16 weights
constexpr int64_t kGemmMinTQuant = 17;  // Q8 / Q4 weights

// Split workspace (split-K of the tensor-core kernel, K split over CTAs of the
// Q8/Q4 decode kernel): a fixed block of per-tile arrival counters, then the
// partial results.  The counters read zero before every launch: the last
// arriver of each tile puts its counter back, and a new workspace starts
// zeroed; a launch with more tiles than counters does not split.
constexpr int kSplitCounters = 65536;
constexpr size_t kSplitCounterBytes = (size_t)kSplitCounters * sizeof(unsigned);

struct GemmJob {
  const PackedWeight* w;
  float* y;  // [t][w->n_out], or h [t][w->n_out / 2] when w->glu
};
// Tensor-core path for large t: xb is x cast to bf16, [t][n_in_pad], zero in the
// padding columns.  Every job has format `fmt` (bf16 weights are tiled as they
// are; Q8/Q4 weights are dequantised to bf16 in shared memory inside the kernel).
// ws / ws_bytes: split-K workspace (counters, then fp32 partial tiles); with
// nullptr the kernel never splits K.  gemm_workspace_bytes gives the size the
// launch plan wants (0 when no launch splits K).
// Appends one launch per group of at most kMaxGemmJobs jobs to *out.
cudaError_t prepare_gemm(int fmt, const __nv_bfloat16* xb, int64_t t, int64_t n_in_pad, const GemmJob* jobs,
                         int n_jobs, int num_sms, unsigned* status, void* ws, size_t ws_bytes,
                         std::vector<Launch>* out);
size_t gemm_workspace_bytes(int64_t t, int64_t n_in_pad, const GemmJob* jobs, int n_jobs, int num_sms);

// How a batch splits over the kernels: tensor-core jobs per format (large t)
// and decode jobs per format (indices into the caller's jobs).
struct BatchPlan {
  std::vector<GemmJob> gemm[3];
  std::vector<int> decode[3];
  int64_t n_in_pad = 0;
  size_t xb_bytes = 0;  // the bf16 copy of x the tensor-core jobs read (0: none)
};
// gemm_quant: Q8/Q4 jobs take the tensor-core path from kGemmMinTQuant tokens.
void plan_batch(int64_t t, const il_job* jobs, int n_jobs, const std::vector<const PackedWeight*>& ws,
                bool gemm_quant, BatchPlan* plan);
// Split workspace the plan's launches would use (0: none).
size_t plan_workspace_bytes(const BatchPlan& plan, int64_t t, int64_t n_in, const il_job* jobs,
                            const std::vector<const PackedWeight*>& ws, int num_sms);
// Appends every launch of the batch to *out (nothing is enqueued).  xb: the bf16
// copy of x (plan.xb_bytes); wsp / ws_bytes: split-K workspace or nullptr / 0.
cudaError_t prepare_batch(const BatchPlan& plan, const float* x, int64_t t, int64_t n_in, const il_job* jobs,
                          const std::vector<const PackedWeight*>& ws, __nv_bfloat16* xb, void* wsp,
                          size_t ws_bytes, int num_sms, unsigned* status, std::vector<Launch>* out);

// Argument checks shared by the batch entry points (set the thread's error on failure).
// host_x: x is a host buffer that the call copies (no alignment rule for it).
int check_batch_args(const float* x, int64_t t, int64_t n_in, const il_job* jobs, int n_jobs, bool host_x = false);
int api_check_batch(const float* x, int64_t t, int64_t n_in, const il_job* jobs, int n_jobs, int dev,
                    std::vector<const PackedWeight*>* ws, uint64_t* wbytes, uint64_t* flops, bool host_x = false);
void api_clear_error();
int api_fail(int code, const char* msg);
int api_cuda_fail(cudaError_t e, const char* what);
void api_count_batch(int n_jobs, int launches, uint64_t wbytes, uint64_t flops);
// Device address of il_matmul_batch_noalloc's status word on device `dev`, or
// nullptr before that entry point has set the device up.
unsigned* noalloc_status_word(int dev);
// Its split workspace's arrival counters (nullptr before set-up).
void* noalloc_split_counters(int dev, size_t* bytes);

// Centroid-masked LM head after the centroid logits cl [n_cent] are computed:
// top-k selection (sel [k]), the gathered cluster logits (scores_out [k*per],
// optional) and the first maximum (token_out, score_out optional).  best_key and
// done are zero before the call and zero again after it.
constexpr int kMaxCentroids = 16384;   // the selection sorts them in one CTA's shared memory
constexpr unsigned kStatusBadToken = 0x100;  // status word: an ordering entry >= vocab was skipped
constexpr int kMaxHeadWidth = 32768;   // x is staged in shared memory as fp32
cudaError_t prepare_lmhead(const float* x, int h, const float* cl, int n_cent, int k, const PackedWeight& embed,
                           const uint32_t* ordering, int per, uint32_t* sel, float* scores_out,
                           unsigned long long* best_key, unsigned* done, uint32_t* token_out, float* score_out,
                           unsigned* status, int num_sms, std::vector<Launch>* out);

}  // namespace il
