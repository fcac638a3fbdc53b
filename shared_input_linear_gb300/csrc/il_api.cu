// il_api.cu -- the C ABI (include/il.h): handle registry, validation,
// error reporting, statistics and dispatch to the kernels.
//
// Contract followed (oxinfer 0.0.0, src/gpu.rs): `Backend::upload` prepares
// device state for one weight; `Backend::matmul` runs every job of a batch
// over one shared x in one submission and, when it cannot, computes nothing.
// Here "computes nothing" is: every argument is validated before the first
// launch, and an error returns a negative status with nothing enqueued.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <string>
#include <unordered_set>
#include <utility>
#include <vector>
#include <algorithm>

#include <nvtx3/nvToolsExt.h>

#include "il_internal.cuh"

using namespace il;

namespace {

constexpr int64_t kMaxNIn = 32768;
constexpr int64_t kMaxNOut = 2147483647;
constexpr int64_t kMaxT = 1 << 20;
constexpr int kMaxJobs = 4096;

thread_local std::string t_last_error;
thread_local int t_last_status = IL_OK;

void clear_error() {
  t_last_error.clear();
  t_last_status = IL_OK;
}

struct Stats {
  std::atomic<uint64_t> uploads{0}, upload_bytes{0}, batches{0}, jobs{0}, launches{0},
      weight_bytes{0}, flops{0}, errors{0}, profiled_batches{0}, device_ns{0};
} g_stats;

// ---- optional timing (IL_PROFILE=1): CUDA events around each call's launches
// on its stream; il_get_stats waits for the recorded calls and adds their device
// time.  Calls on a stream that is being captured are not timed.
bool profiling() {
  static const bool on = [] {
    const char* e = getenv("IL_PROFILE");
    return e != nullptr && e[0] == '1';
  }();
  return on;
}

struct TimedCall {
  cudaEvent_t begin, end;
};
std::mutex g_prof_mu;
std::vector<TimedCall> g_prof;  // recorded, not yet added to the counters
constexpr size_t kMaxPendingTimes = 4096;

// Adds the device time of every recorded call (waits for each) and frees its events.
void drain_times() {
  std::vector<TimedCall> v;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    v.swap(g_prof);
  }
  for (const TimedCall& c : v) {
    float ms = 0.f;
    if (cudaEventSynchronize(c.end) == cudaSuccess && cudaEventElapsedTime(&ms, c.begin, c.end) == cudaSuccess) {
      g_stats.profiled_batches.fetch_add(1);
      g_stats.device_ns.fetch_add((uint64_t)((double)ms * 1e6));
    }
    cudaEventDestroy(c.begin);
    cudaEventDestroy(c.end);
  }
}

// run_launches, timed when IL_PROFILE=1 (and the stream is not being captured).
cudaError_t run_timed(const std::vector<Launch>& v, cudaStream_t stream, int* launches) {
  TimedCall c{nullptr, nullptr};
  bool timed = false;
  if (profiling()) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusNone &&
        cudaEventCreate(&c.begin) == cudaSuccess) {
      if (cudaEventCreate(&c.end) == cudaSuccess) {
        timed = cudaEventRecord(c.begin, stream) == cudaSuccess;
      } else {
        cudaEventDestroy(c.begin);
      }
    }
  }
  const cudaError_t e = run_launches(v, stream, launches);
  if (timed) {
    if (e == cudaSuccess && cudaEventRecord(c.end, stream) == cudaSuccess) {
      size_t pending;
      {
        std::lock_guard<std::mutex> lk(g_prof_mu);
        g_prof.push_back(c);
        pending = g_prof.size();
      }
      if (pending > kMaxPendingTimes) drain_times();
    } else {
      cudaEventDestroy(c.begin);
      cudaEventDestroy(c.end);
    }
  }
  return e;
}

// NVTX range over an entry point's host work (no-op unless a tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

std::mutex g_reg_mu;
std::unordered_set<const PackedWeight*> g_registry;

struct DeviceState {
  bool ok = false;
  int num_sms = 0;
  int major = 0, minor = 0;
  unsigned* status = nullptr;  // device word set by bounded waits that gave up
};
std::mutex g_dev_mu;
std::map<int, DeviceState> g_devices;

// Scratch of the tensor-core path, one set per (device, stream): the bf16 copy
// of x and the split-K workspace.  Grown with the stream-ordered allocator, so
// growing never waits for the stream: the old buffer is released in stream
// order, after the work already queued that may still read it.
struct Scratch {
  void* ptr = nullptr;
  size_t bytes = 0;
  void* ws = nullptr;
  size_t ws_bytes = 0;
};

std::mutex g_scratch_mu;
std::map<std::pair<int, cudaStream_t>, Scratch> g_scratch;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  t_last_status = code;
  g_stats.errors.fetch_add(1);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(IL_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Host-side fault injection for the out-of-memory paths: with
// IL_FAULT_ALLOC_FAIL_AFTER=k the (k+1)-th device allocation of the process fails.
std::atomic<long> g_alloc_count{0};
cudaError_t il_malloc(void** p, size_t bytes) {
  const char* env = getenv("IL_FAULT_ALLOC_FAIL_AFTER");
  if (env != nullptr && *env != '\0') {
    const long limit = strtol(env, nullptr, 10);
    if (g_alloc_count.fetch_add(1) >= limit) {
      *p = nullptr;
      return cudaErrorMemoryAllocation;
    }
  }
  return cudaMalloc(p, bytes);
}

// Device of the calling thread, checked to be sm_103.
int current_device(DeviceState** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceState& st = g_devices[dev];
  if (!st.ok) {
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
    st.major = prop.major;
    st.minor = prop.minor;
    st.num_sms = prop.multiProcessorCount;
    if (!(prop.major == 10 && prop.minor == 3))
      return fail(IL_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                  dev, prop.major, prop.minor);
    void* s = nullptr;
    e = il_malloc(&s, 256);
    if (e != cudaSuccess) return fail(IL_ERR_OOM, "allocating the device status word failed");
    e = cudaMemset(s, 0, 256);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset");
    st.status = static_cast<unsigned*>(s);
    st.ok = true;
  }
  *out = &st;
  return dev;
}

bool known_handle(const il_weight* h) {
  const PackedWeight* w = reinterpret_cast<const PackedWeight*>(h);
  std::lock_guard<std::mutex> lk(g_reg_mu);
  return g_registry.count(w) != 0 && w->magic == kWeightMagic;
}

int64_t host_bytes(int format, int64_t n_out, int64_t n_in) {
  if (format == IL_BF16) return 2 * n_out * n_in;
  if (format == IL_Q8) return n_out * n_in + 4 * n_out * (n_in / 32);
  return n_out * (n_in / 2) + 4 * n_out * (n_in / 32);
}

cudaError_t il_malloc_async(void** p, size_t bytes, cudaStream_t stream) {
  const char* env = getenv("IL_FAULT_ALLOC_FAIL_AFTER");
  if (env != nullptr && *env != '\0') {
    const long limit = strtol(env, nullptr, 10);
    if (g_alloc_count.fetch_add(1) >= limit) {
      *p = nullptr;
      return cudaErrorMemoryAllocation;
    }
  }
  return cudaMallocAsync(p, bytes, stream);
}

// Scratch may only grow outside stream capture: an allocation made while a
// stream is captured would belong to the graph, not to the library.
int check_not_capturing(cudaStream_t stream, const char* what) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cs);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  if (cs != cudaStreamCaptureStatusNone)
    return fail(IL_ERR_UNSUPPORTED,
                "%s must grow while the stream is being captured: run one call of this size on the stream "
                "before capturing it",
                what);
  return IL_OK;
}

int get_scratch(int dev, cudaStream_t stream, size_t bytes, void** out) {
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  Scratch& s = g_scratch[{dev, stream}];
  if (s.bytes < bytes) {
    const int rc = check_not_capturing(stream, "the bf16 copy of x");
    if (rc != IL_OK) return rc;
    const size_t want = bytes + bytes / 4;
    void* np = nullptr;
    cudaError_t e = il_malloc_async(&np, want, stream);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(IL_ERR_OOM, "allocating %zu bytes of scratch failed", want);
    }
    if (s.ptr != nullptr) cudaFreeAsync(s.ptr, stream);  // after the queued work that reads it
    s.ptr = np;
    s.bytes = want;
  }
  *out = s.ptr;
  return IL_OK;
}

int get_workspace(int dev, cudaStream_t stream, size_t bytes, void** out, size_t* got) {
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  Scratch& s = g_scratch[{dev, stream}];
  if (s.ws_bytes < bytes) {
    const int rc = check_not_capturing(stream, "the split-K workspace");
    if (rc != IL_OK) return rc;
    void* np = nullptr;
    cudaError_t e = il_malloc_async(&np, bytes, stream);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(IL_ERR_OOM, "allocating %zu bytes of split-K workspace failed", bytes);
    }
    // the per-tile arrival counters at its start must be zero before first use
    e = cudaMemsetAsync(np, 0, bytes, stream);
    if (e != cudaSuccess) {
      cudaFreeAsync(np, stream);
      return cuda_fail(e, "cudaMemsetAsync(workspace)");
    }
    if (s.ws != nullptr) cudaFreeAsync(s.ws, stream);
    s.ws = np;
    s.ws_bytes = bytes;
  }
  *out = s.ws;
  *got = s.ws_bytes;
  return IL_OK;
}

// Scratch of il_centroid_head, one set per (device, stream): centroid logits,
// the selection, and the 64-bit best key + arrival counter (zero between calls).
struct HeadScratch {
  void* ptr = nullptr;
  int64_t n_cent = 0, k = 0;
};
std::map<std::pair<int, cudaStream_t>, HeadScratch> g_head_scratch;

constexpr size_t kHeadStateBytes = 256;  // best key (8 bytes) and counter, at the start

int get_head_scratch(int dev, cudaStream_t stream, int64_t n_cent, int64_t k, uint8_t** out) {
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  HeadScratch& s = g_head_scratch[{dev, stream}];
  if (s.n_cent < n_cent || s.k < k) {
    const int rc = check_not_capturing(stream, "the LM-head scratch");
    if (rc != IL_OK) return rc;
    const int64_t nc = std::max(n_cent, (int64_t)1024), kk = std::max(k, (int64_t)256);
    const size_t bytes = kHeadStateBytes + (size_t)nc * 4 + (size_t)kk * 4;
    void* np = nullptr;
    cudaError_t e = il_malloc_async(&np, bytes, stream);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(IL_ERR_OOM, "allocating %zu bytes of LM-head scratch failed", bytes);
    }
    e = cudaMemsetAsync(np, 0, bytes, stream);
    if (e != cudaSuccess) {
      cudaFreeAsync(np, stream);
      return cuda_fail(e, "cudaMemsetAsync(LM-head scratch)");
    }
    if (s.ptr != nullptr) cudaFreeAsync(s.ptr, stream);
    s.ptr = np;
    s.n_cent = nc;
    s.k = kk;
  }
  *out = static_cast<uint8_t*>(s.ptr);
  return IL_OK;
}

// Device copies of x and y for il_matmul_batch_host, one buffer per (device,
// stream): x at the start, then the y runs.  Grown like the bf16 copy of x.
struct HostStaging {
  void* ptr = nullptr;
  size_t bytes = 0;
};
std::map<std::pair<int, cudaStream_t>, HostStaging> g_host_staging;

int get_host_staging(int dev, cudaStream_t stream, size_t bytes, uint8_t** out) {
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  HostStaging& s = g_host_staging[{dev, stream}];
  if (s.bytes < bytes) {
    const int rc = check_not_capturing(stream, "the device copies of x and y");
    if (rc != IL_OK) return rc;
    const size_t want = bytes + bytes / 4;
    void* np = nullptr;
    cudaError_t e = il_malloc_async(&np, want, stream);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(IL_ERR_OOM, "allocating %zu bytes for the device copies of x and y failed", want);
    }
    if (s.ptr != nullptr) cudaFreeAsync(s.ptr, stream);
    s.ptr = np;
    s.bytes = want;
  }
  *out = static_cast<uint8_t*>(s.ptr);
  return IL_OK;
}

// A buffer of il_matmul_batch_host must be host memory (page-locked or pageable)
// or managed memory; device memory is il_matmul_batch's.  *mapped: the device
// address of page-locked host memory that kernels can access in place (NULL for
// pageable or managed memory).
int host_buffer(const void* ptr, const char* what, int job, void** mapped) {
  *mapped = nullptr;
  cudaPointerAttributes a;
  const cudaError_t e = cudaPointerGetAttributes(&a, ptr);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "il_matmul_batch_host: cudaPointerGetAttributes");
  }
  if (a.type == cudaMemoryTypeDevice) {
    if (job < 0) return fail(IL_ERR_ARG, "il_matmul_batch_host: %s is device memory (use il_matmul_batch)", what);
    return fail(IL_ERR_ARG, "il_matmul_batch_host: job %d %s is device memory (use il_matmul_batch)", job, what);
  }
  if (a.type == cudaMemoryTypeHost) *mapped = a.devicePointer;
  return IL_OK;
}

bool overlaps(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) { return a0 < b1 && b0 < a1; }

// Plan, scratch and every launch of a validated batch on device buffers, all
// worked out before anything is enqueued.
int prepare_device_batch(const char* fn, const float* x, int64_t t, int64_t n_in, const il_job* jobs, int n_jobs,
                         const std::vector<const PackedWeight*>& ws, int dev, DeviceState* ds, cudaStream_t stream,
                         std::vector<Launch>* launches) {
  BatchPlan plan;
  plan_batch(t, jobs, n_jobs, ws, /*gemm_quant=*/true, &plan);
  void* xb = nullptr;
  void* wsp = nullptr;
  size_t ws_bytes = 0;
  if (plan.xb_bytes > 0) {
    const int rc = get_scratch(dev, stream, plan.xb_bytes, &xb);
    if (rc != IL_OK) return rc;
  }
  const size_t want = plan_workspace_bytes(plan, t, n_in, jobs, ws, ds->num_sms);
  if (want > 0) {
    const int rc = get_workspace(dev, stream, want, &wsp, &ws_bytes);
    if (rc != IL_OK) return rc;
  }
  const cudaError_t e = prepare_batch(plan, x, t, n_in, jobs, ws, static_cast<__nv_bfloat16*>(xb), wsp, ws_bytes,
                                      ds->num_sms, ds->status, launches);
  if (e != cudaSuccess) {
    char what[96];
    snprintf(what, sizeof what, "%s: preparing the launches", fn);
    return cuda_fail(e, what);
  }
  return IL_OK;
}

}  // namespace

extern "C" {

int il_version(void) { return IL_VERSION; }

const char* il_last_error(void) { return t_last_error.c_str(); }

int il_last_status(void) { return t_last_status; }

int il_get_stats(il_stats* out) {
  if (out == nullptr) return fail(IL_ERR_ARG, "il_get_stats: out is NULL");
  if (profiling()) drain_times();
  out->uploads = g_stats.uploads.load();
  out->upload_bytes = g_stats.upload_bytes.load();
  out->batches = g_stats.batches.load();
  out->jobs = g_stats.jobs.load();
  out->launches = g_stats.launches.load();
  out->weight_bytes = g_stats.weight_bytes.load();
  out->flops = g_stats.flops.load();
  out->errors = g_stats.errors.load();
  out->profiled_batches = g_stats.profiled_batches.load();
  out->device_ns = g_stats.device_ns.load();
  return IL_OK;
}

void il_reset_stats(void) {
  g_stats.uploads = 0;
  g_stats.upload_bytes = 0;
  g_stats.batches = 0;
  g_stats.jobs = 0;
  g_stats.launches = 0;
  g_stats.weight_bytes = 0;
  g_stats.flops = 0;
  g_stats.errors = 0;
  if (profiling()) drain_times();
  g_stats.profiled_batches = 0;
  g_stats.device_ns = 0;
}

}  // extern "C"

namespace {

// Shared by il_upload_weight (parts = 1) and il_upload_gate_up (parts = 2): the
// parts, host weights of one shape, become one packed matrix whose rows
// interleave them (row parts*r + i is row r of part i).
il_weight* upload_impl(const char* fn, int format, const void* const* host, int parts, int64_t n_out,
                       int64_t n_in) {
  clear_error();
  if (format != IL_BF16 && format != IL_Q8 && format != IL_Q4) {
    fail(IL_ERR_FORMAT, "%s: unknown format %d", fn, format);
    return nullptr;
  }
  for (int i = 0; i < parts; ++i)
    if (host[i] == nullptr) {
      fail(IL_ERR_ARG, "%s: host pointer %d is NULL", fn, i);
      return nullptr;
    }
  if (n_out < 1 || n_out > kMaxNOut / parts || n_in < 1 || n_in > kMaxNIn) {
    fail(IL_ERR_SHAPE, "%s: n_out=%lld n_in=%lld out of range", fn, (long long)n_out, (long long)n_in);
    return nullptr;
  }
  if (format == IL_BF16 && n_in % 8 != 0) {
    fail(IL_ERR_SHAPE, "%s: bf16 needs n_in %% 8 == 0 (got %lld)", fn, (long long)n_in);
    return nullptr;
  }
  if (format != IL_BF16 && n_in % 32 != 0) {
    fail(IL_ERR_SHAPE, "%s: Q8/Q4 need n_in %% 32 == 0 (got %lld)", fn, (long long)n_in);
    return nullptr;
  }
  DeviceState* ds = nullptr;
  const int dev = current_device(&ds);
  if (dev < 0) return nullptr;

  PackedWeight* w = new (std::nothrow) PackedWeight();
  if (w == nullptr) {
    fail(IL_ERR_OOM, "%s: host allocation failed", fn);
    return nullptr;
  }
  const int64_t rows = n_out * parts;
  w->magic = kWeightMagic;
  w->format = format;
  w->device = dev;
  w->glu = parts == 2 ? 1 : 0;
  w->n_out = rows;
  w->n_in = n_in;
  const int64_t pr = pad_rows(format);
  w->n_out_pad = (rows + pr - 1) / pr * pr;
  w->n_in_pad = (n_in + kPadK - 1) / kPadK * kPadK;
  w->n_groups = w->n_out_pad / kGroupRows;
  w->n_chunks = w->n_in_pad / chunk_k(format);
  w->host_bytes = host_bytes(format, rows, n_in);
  w->device_bytes = format == IL_BF16 ? (size_t)w->n_out_pad * w->n_in_pad * 2
                                      : (size_t)(w->n_out_pad / kPairRows) * w->n_chunks * record_bytes(format);

  void* mem = nullptr;
  cudaError_t e = il_malloc(&mem, w->device_bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    const size_t want = w->device_bytes;
    delete w;
    fail(IL_ERR_OOM, "%s: cudaMalloc(%zu) failed", fn, want);
    return nullptr;
  }
  w->quants = static_cast<uint8_t*>(mem);

  void* staging = nullptr;
  e = il_malloc(&staging, (size_t)w->host_bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    cudaFree(mem);
    const long long want = (long long)w->host_bytes;
    delete w;
    fail(IL_ERR_OOM, "%s: staging cudaMalloc(%lld) failed", fn, want);
    return nullptr;
  }
  if (parts == 1) {
    e = cudaMemcpy(staging, host[0], (size_t)w->host_bytes, cudaMemcpyHostToDevice);
  } else {
    // host layout of each part: [n_out rows of qrow bytes][n_out rows of srow bytes];
    // pitched copies put part i's rows at every parts-th row of the staging copy
    const size_t qrow = (size_t)host_bytes(format, 1, n_in) - (format == IL_BF16 ? 0 : 4 * (size_t)(n_in / 32));
    const size_t srow = format == IL_BF16 ? 0 : 4 * (size_t)(n_in / 32);
    uint8_t* st = static_cast<uint8_t*>(staging);
    for (int i = 0; i < parts && e == cudaSuccess; ++i) {
      const uint8_t* src = static_cast<const uint8_t*>(host[i]);
      e = cudaMemcpy2D(st + i * qrow, parts * qrow, src, qrow, qrow, (size_t)n_out, cudaMemcpyHostToDevice);
      if (e == cudaSuccess && srow > 0)
        e = cudaMemcpy2D(st + (size_t)rows * qrow + i * srow, parts * srow, src + (size_t)n_out * qrow, srow, srow,
                         (size_t)n_out, cudaMemcpyHostToDevice);
    }
  }
  if (e == cudaSuccess) e = launch_pack(*w, static_cast<const uint8_t*>(staging), 0);
  if (e == cudaSuccess) e = cudaStreamSynchronize(0);
  cudaFree(staging);
  if (e != cudaSuccess) {
    cudaFree(mem);
    delete w;
    cuda_fail(e, "upload: copy/pack");
    return nullptr;
  }
  {
    std::lock_guard<std::mutex> lk(g_reg_mu);
    g_registry.insert(w);
  }
  g_stats.uploads.fetch_add(1);
  g_stats.upload_bytes.fetch_add((uint64_t)w->host_bytes);
  return reinterpret_cast<il_weight*>(w);
}

}  // namespace

extern "C" {

il_weight* il_upload_weight(int format, const void* host_ptr, int64_t n_out, int64_t n_in) {
  NvtxRange range("il_upload_weight");
  const void* host[1] = {host_ptr};
  return upload_impl("il_upload_weight", format, host, 1, n_out, n_in);
}

il_weight* il_upload_gate_up(int format, const void* gate_ptr, const void* up_ptr, int64_t n_out, int64_t n_in) {
  NvtxRange range("il_upload_gate_up");
  const void* host[2] = {gate_ptr, up_ptr};
  return upload_impl("il_upload_gate_up", format, host, 2, n_out, n_in);
}

int il_weight_is_gate_up(const il_weight* h) {
  if (h == nullptr || !known_handle(h)) return -1;
  return reinterpret_cast<const PackedWeight*>(h)->glu;
}

void il_free_weight(il_weight* h) {
  if (h == nullptr) return;
  PackedWeight* w = reinterpret_cast<PackedWeight*>(h);
  {
    std::lock_guard<std::mutex> lk(g_reg_mu);
    if (g_registry.erase(w) == 0) {
      fail(IL_ERR_HANDLE, "il_free_weight: unknown handle");
      return;
    }
  }
  int prev = -1;
  cudaGetDevice(&prev);
  if (prev != w->device) cudaSetDevice(w->device);
  cudaFree(w->quants);  // synchronises the device
  if (prev >= 0 && prev != w->device) cudaSetDevice(prev);
  w->magic = 0;
  delete w;
}

int64_t il_weight_bytes(const il_weight* h) {
  if (h == nullptr || !known_handle(h)) return -1;
  return reinterpret_cast<const PackedWeight*>(h)->host_bytes;
}

int il_weight_info(const il_weight* h, int* format, int64_t* n_out, int64_t* n_in) {
  if (h == nullptr || !known_handle(h)) return fail(IL_ERR_HANDLE, "il_weight_info: invalid handle");
  const PackedWeight* w = reinterpret_cast<const PackedWeight*>(h);
  if (format) *format = w->format;
  if (n_out) *n_out = out_width(*w);
  if (n_in) *n_in = w->n_in;
  return IL_OK;
}

int il_dequantize_weight(const il_weight* h, float* dev_out, void* stream) {
  clear_error();
  if (h == nullptr || !known_handle(h)) return fail(IL_ERR_HANDLE, "il_dequantize_weight: invalid handle");
  if (dev_out == nullptr) return fail(IL_ERR_ARG, "il_dequantize_weight: dev_out is NULL");
  if (reinterpret_cast<uintptr_t>(dev_out) % 4 != 0)
    return fail(IL_ERR_ARG, "il_dequantize_weight: dev_out is not 4-byte aligned");
  const PackedWeight* w = reinterpret_cast<const PackedWeight*>(h);
  DeviceState* ds = nullptr;
  const int dev = current_device(&ds);
  if (dev < 0) return dev;
  if (dev != w->device) return fail(IL_ERR_HANDLE, "il_dequantize_weight: handle lives on device %d", w->device);
  cudaError_t e = launch_dequant(*w, dev_out, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "il_dequantize_weight: launch");
  return IL_OK;
}

int il_check_device_status(void* stream) {
  DeviceState* ds = nullptr;
  const int dev = current_device(&ds);
  if (dev < 0) return dev;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned word = 0, noalloc_word = 0;
  unsigned* noalloc = noalloc_status_word(dev);
  cudaError_t e = cudaMemcpyAsync(&word, ds->status, sizeof word, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && noalloc != nullptr)
    e = cudaMemcpyAsync(&noalloc_word, noalloc, sizeof noalloc_word, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(ds->status, 0, sizeof word, s);
  if (e == cudaSuccess && noalloc != nullptr) e = cudaMemsetAsync(noalloc, 0, sizeof noalloc_word, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "il_check_device_status");
  word |= noalloc_word;
  if (word == kStatusBadToken) return fail(IL_ERR_ARG, "il_centroid_head met an ordering entry >= vocab");
  if (word != 0) {
    // a kernel that gave up may have left split-K arrival counters behind: clear
    // this device's workspaces, once no stream still uses them, so the next
    // launches start from zero
    e = cudaDeviceSynchronize();
    {
      std::lock_guard<std::mutex> lk(g_scratch_mu);
      for (auto& kv : g_scratch)
        if (kv.first.first == dev && kv.second.ws != nullptr && e == cudaSuccess)
          e = cudaMemset(kv.second.ws, 0, kv.second.ws_bytes);
    }
    size_t nb = 0;
    void* nc = noalloc_split_counters(dev, &nb);
    if (nc != nullptr && e == cudaSuccess) e = cudaMemset(nc, 0, nb);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "il_check_device_status: clearing the split-K workspaces");
    return fail(IL_ERR_DEVICE_TIMEOUT, "a device-side wait gave up (code 0x%x)", word);
  }
  return IL_OK;
}

int il_release_scratch(void* stream_) {
  clear_error();
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  auto it = g_scratch.find({dev, stream});
  if (it != g_scratch.end()) {
    if (it->second.ptr != nullptr) e = cudaFreeAsync(it->second.ptr, stream);
    if (e == cudaSuccess && it->second.ws != nullptr) e = cudaFreeAsync(it->second.ws, stream);
    g_scratch.erase(it);
  }
  auto ih = g_head_scratch.find({dev, stream});
  if (ih != g_head_scratch.end()) {
    if (e == cudaSuccess && ih->second.ptr != nullptr) e = cudaFreeAsync(ih->second.ptr, stream);
    g_head_scratch.erase(ih);
  }
  auto is = g_host_staging.find({dev, stream});
  if (is != g_host_staging.end()) {
    if (e == cudaSuccess && is->second.ptr != nullptr) e = cudaFreeAsync(is->second.ptr, stream);
    g_host_staging.erase(is);
  }
  if (e != cudaSuccess) return cuda_fail(e, "il_release_scratch");
  return IL_OK;
}

int il_matmul_batch(const float* x, int64_t t, int64_t n_in, const il_job* jobs, int n_jobs,
                    void* stream_) {
  NvtxRange range("il_matmul_batch");
  clear_error();
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int rc = check_batch_args(x, t, n_in, jobs, n_jobs);
  if (rc != IL_OK || t == 0 || n_jobs == 0) return rc;
  DeviceState* ds = nullptr;
  const int dev = current_device(&ds);
  if (dev < 0) return dev;
  std::vector<const PackedWeight*> ws;
  uint64_t wbytes = 0, flops = 0;
  rc = api_check_batch(x, t, n_in, jobs, n_jobs, dev, &ws, &wbytes, &flops);
  if (rc != IL_OK) return rc;
  std::vector<Launch> launches;
  rc = prepare_device_batch("il_matmul_batch", x, t, n_in, jobs, n_jobs, ws, dev, ds, stream, &launches);
  if (rc != IL_OK) return rc;
  int n_launched = 0;
  const cudaError_t e = run_timed(launches, stream, &n_launched);
  g_stats.launches.fetch_add((uint64_t)n_launched);
  if (e != cudaSuccess) return cuda_fail(e, "il_matmul_batch: launch");
  g_stats.batches.fetch_add(1);
  g_stats.jobs.fetch_add((uint64_t)n_jobs);
  g_stats.weight_bytes.fetch_add(wbytes);
  g_stats.flops.fetch_add(flops);
  return IL_OK;
}

int il_matmul_batch_host(const float* x, int64_t t, int64_t n_in, const il_job* jobs, int n_jobs,
                         void* stream_) {
  NvtxRange range("il_matmul_batch_host");
  clear_error();
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int rc = check_batch_args(x, t, n_in, jobs, n_jobs, /*host_x=*/true);
  if (rc != IL_OK || t == 0 || n_jobs == 0) return rc;
  DeviceState* ds = nullptr;
  const int dev = current_device(&ds);
  if (dev < 0) return dev;
  std::vector<const PackedWeight*> ws;
  uint64_t wbytes = 0, flops = 0;
  rc = api_check_batch(x, t, n_in, jobs, n_jobs, dev, &ws, &wbytes, &flops, /*host_x=*/true);
  if (rc != IL_OK) return rc;
  // page-locked host memory is read (x, when 16-byte aligned) and written (y) by
  // the kernels in place; the rest goes through a device buffer and copies
  void* x_mapped = nullptr;
  rc = host_buffer(x, "x", -1, &x_mapped);
  if (rc != IL_OK) return rc;
  if (reinterpret_cast<uintptr_t>(x_mapped) % 16 != 0) x_mapped = nullptr;
  std::vector<void*> y_mapped(n_jobs, nullptr);
  for (int j = 0; j < n_jobs && rc == IL_OK; ++j) rc = host_buffer(jobs[j].y, "y", j, &y_mapped[j]);
  if (rc != IL_OK) return rc;

  // ---- device buffer: x (if copied) at offset 0, then the copied y buffers in
  // runs -- a run is a sequence of y buffers each starting where the previous one
  // ends in host memory, kept adjacent on the device too so that one copy brings
  // it back
  struct Run {
    uintptr_t host;
    size_t bytes, dev_off;
  };
  auto round_up = [](size_t v, size_t a) { return (v + a - 1) / a * a; };
  const size_t x_bytes = (size_t)t * (size_t)n_in * sizeof(float);
  std::vector<int> order;
  for (int j = 0; j < n_jobs; ++j)
    if (y_mapped[j] == nullptr) order.push_back(j);
  std::sort(order.begin(), order.end(), [&](int a, int b) {
    return reinterpret_cast<uintptr_t>(jobs[a].y) < reinterpret_cast<uintptr_t>(jobs[b].y);
  });
  std::vector<Run> runs;
  std::vector<size_t> y_off(n_jobs, 0);
  size_t end = x_mapped == nullptr ? round_up(x_bytes, 256) : 0;
  for (int j : order) {
    const uintptr_t y0 = reinterpret_cast<uintptr_t>(jobs[j].y);
    const size_t yb = (size_t)t * (size_t)jobs[j].n_out * sizeof(float);
    if (!runs.empty() && runs.back().host + runs.back().bytes == y0) {
      runs.back().bytes += yb;
    } else {
      runs.push_back(Run{y0, yb, round_up(end, 256)});
    }
    y_off[j] = runs.back().dev_off + (size_t)(y0 - runs.back().host);
    end = runs.back().dev_off + runs.back().bytes;
  }
  uint8_t* staging = nullptr;
  if (end > 0) {
    rc = get_host_staging(dev, stream, end, &staging);
    if (rc != IL_OK) return rc;
  }
  std::vector<il_job> djobs(jobs, jobs + n_jobs);
  for (int j = 0; j < n_jobs; ++j)
    djobs[j].y = y_mapped[j] != nullptr ? static_cast<float*>(y_mapped[j])
                                        : reinterpret_cast<float*>(staging + y_off[j]);
  const float* xd = x_mapped != nullptr ? static_cast<const float*>(x_mapped) : reinterpret_cast<const float*>(staging);
  std::vector<Launch> launches;
  rc = prepare_device_batch("il_matmul_batch_host", xd, t, n_in, djobs.data(), n_jobs, ws, dev, ds, stream,
                            &launches);
  if (rc != IL_OK) return rc;

  // ---- enqueue: x in (if copied), the launches, every run out
  cudaError_t e = cudaSuccess;
  if (x_mapped == nullptr) {
    e = cudaMemcpyAsync(staging, x, x_bytes, cudaMemcpyDefault, stream);
    if (e != cudaSuccess) return cuda_fail(e, "il_matmul_batch_host: copying x to the device");
  }
  int n_launched = 0;
  e = run_timed(launches, stream, &n_launched);
  g_stats.launches.fetch_add((uint64_t)n_launched);
  if (e != cudaSuccess) return cuda_fail(e, "il_matmul_batch_host: launch");
  for (const Run& r : runs) {
    e = cudaMemcpyAsync(reinterpret_cast<void*>(r.host), staging + r.dev_off, r.bytes, cudaMemcpyDefault, stream);
    if (e != cudaSuccess) return cuda_fail(e, "il_matmul_batch_host: copying y to the host");
  }
  g_stats.batches.fetch_add(1);
  g_stats.jobs.fetch_add((uint64_t)n_jobs);
  g_stats.weight_bytes.fetch_add(wbytes);
  g_stats.flops.fetch_add(flops);
  return IL_OK;
}

int il_centroid_head(const float* x, int64_t h, const il_weight* centroids_h, const il_weight* embed_h,
                     const uint32_t* ordering, int64_t top_k, uint32_t* token_out, float* score_out,
                     uint32_t* selected_out, float* scores_out, void* stream_) {
  NvtxRange range("il_centroid_head");
  clear_error();
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (x == nullptr || ordering == nullptr || token_out == nullptr)
    return fail(IL_ERR_ARG, "il_centroid_head: x, ordering and token_out must not be NULL");
  if (reinterpret_cast<uintptr_t>(x) % 16 != 0) return fail(IL_ERR_ARG, "il_centroid_head: x is not 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(ordering) % 4 != 0 || reinterpret_cast<uintptr_t>(token_out) % 4 != 0 ||
      reinterpret_cast<uintptr_t>(score_out) % 4 != 0 || reinterpret_cast<uintptr_t>(selected_out) % 4 != 0 ||
      reinterpret_cast<uintptr_t>(scores_out) % 4 != 0)
    return fail(IL_ERR_ARG, "il_centroid_head: outputs and ordering must be 4-byte aligned");
  if (top_k < 1) return fail(IL_ERR_ARG, "il_centroid_head: top_k=%lld must be >= 1", (long long)top_k);
  DeviceState* ds = nullptr;
  const int dev = current_device(&ds);
  if (dev < 0) return dev;
  const PackedWeight* cw = reinterpret_cast<const PackedWeight*>(centroids_h);
  const PackedWeight* ew = reinterpret_cast<const PackedWeight*>(embed_h);
  if (cw == nullptr || ew == nullptr || !known_handle(centroids_h) || !known_handle(embed_h))
    return fail(IL_ERR_HANDLE, "il_centroid_head: invalid weight handle");
  if (cw->device != dev || ew->device != dev)
    return fail(IL_ERR_HANDLE, "il_centroid_head: a weight lives on another device");
  if (cw->format != IL_BF16 || ew->format != IL_BF16 || cw->glu || ew->glu)
    return fail(IL_ERR_FORMAT, "il_centroid_head: centroids and embed must be plain bf16 weights");
  if (h < 1 || h > kMaxHeadWidth || cw->n_in != h || ew->n_in != h)
    return fail(IL_ERR_SHAPE, "il_centroid_head: h=%lld must equal both weights' n_in", (long long)h);
  const int64_t n_cent = cw->n_out, vocab = ew->n_out;
  if (n_cent > kMaxCentroids)
    return fail(IL_ERR_UNSUPPORTED, "il_centroid_head: %lld centroids, at most %d", (long long)n_cent, kMaxCentroids);
  if (vocab % n_cent != 0)
    return fail(IL_ERR_SHAPE, "il_centroid_head: vocab=%lld is not a multiple of n_cent=%lld", (long long)vocab,
                (long long)n_cent);
  const int64_t k = std::min(top_k, n_cent);
  const int64_t per = vocab / n_cent;
  uint8_t* scratch = nullptr;
  int rc = get_head_scratch(dev, stream, n_cent, k, &scratch);
  if (rc != IL_OK) return rc;
  float* cl = reinterpret_cast<float*>(scratch + kHeadStateBytes);
  uint32_t* sel = selected_out != nullptr ? selected_out : reinterpret_cast<uint32_t*>(cl + std::max(n_cent, (int64_t)1024));
  // 1. centroid logits: a one-job batch on the decode kernel; 2-3. selection,
  // cluster logits and first maximum -- all prepared before any is enqueued
  il_job job{centroids_h, n_cent, cl};
  std::vector<const PackedWeight*> ws{cw};
  BatchPlan plan;
  plan_batch(1, &job, 1, ws, true, &plan);
  std::vector<Launch> launches;
  cudaError_t e = prepare_batch(plan, x, 1, h, &job, ws, nullptr, nullptr, 0, ds->num_sms, ds->status, &launches);
  if (e == cudaSuccess)
    e = prepare_lmhead(x, (int)h, cl, (int)n_cent, (int)k, *ew, ordering, (int)per, sel, scores_out,
                       reinterpret_cast<unsigned long long*>(scratch), reinterpret_cast<unsigned*>(scratch + 8),
                       token_out, score_out, ds->status, ds->num_sms, &launches);
  if (e != cudaSuccess) return cuda_fail(e, "il_centroid_head: preparing the launches");
  int n_launched = 0;
  e = run_timed(launches, stream, &n_launched);
  g_stats.launches.fetch_add((uint64_t)n_launched);
  if (e != cudaSuccess) return cuda_fail(e, "il_centroid_head: launch");
  g_stats.batches.fetch_add(1);
  g_stats.jobs.fetch_add(1);
  g_stats.weight_bytes.fetch_add((uint64_t)cw->host_bytes);
  g_stats.flops.fetch_add(2ull * (uint64_t)h * (uint64_t)n_cent);
  return IL_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Batch planning shared by il_matmul_batch, il_matmul_batch_noalloc and the
// centroid head, and helpers for entry points defined in other translation
// units (they read the handle registry, the error state and the counters kept
// here).
// ---------------------------------------------------------------------------
namespace il {

cudaError_t run_launches(const std::vector<Launch>& v, cudaStream_t stream, int* launches) {
  for (const Launch& L : v) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = L.grid;
    cfg.blockDim = L.block;
    cfg.dynamicSmemBytes = L.smem;
    cfg.stream = stream;
    cfg.attrs = const_cast<cudaLaunchAttribute*>(L.attr);
    cfg.numAttrs = L.nattr;
    cudaError_t e = cudaLaunchKernelExC(&cfg, L.fn, const_cast<void**>(L.args));
    if (launches) ++*launches;
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

void plan_batch(int64_t t, const il_job* jobs, int n_jobs, const std::vector<const PackedWeight*>& ws,
                bool gemm_quant, BatchPlan* plan) {
  *plan = BatchPlan();
  const bool gemm_bf16 = t >= kGemmMinT;
  const bool gemm_q = gemm_quant && t >= kGemmMinTQuant;
  for (int j = 0; j < n_jobs; ++j) {
    const PackedWeight* w = ws[j];
    const bool gemm = w->format == IL_BF16 ? gemm_bf16 : gemm_q;
    if (gemm) {
      plan->gemm[w->format].push_back(GemmJob{w, jobs[j].y});
      plan->n_in_pad = w->n_in_pad;
    } else {
      plan->decode[w->format].push_back(j);
    }
  }
  if (!plan->gemm[0].empty() || !plan->gemm[1].empty() || !plan->gemm[2].empty())
    plan->xb_bytes = (size_t)t * (size_t)plan->n_in_pad * 2;
}

namespace {

// The decode launches of a plan, in launch order: one per format, per
// kMaxDecodeJobs jobs and per 8 tokens (bf16) or 16 tokens (Q8/Q4).
void decode_launch_params(const BatchPlan& plan, const float* x, int64_t t, int64_t n_in, const il_job* jobs,
                          const std::vector<const PackedWeight*>& ws, std::vector<std::pair<int, DecodeParams>>* out) {
  for (int fmt = IL_BF16; fmt <= IL_Q4; ++fmt) {
    const std::vector<int>& idx = plan.decode[fmt];
    for (size_t j0 = 0; j0 < idx.size(); j0 += kMaxDecodeJobs) {
      const size_t j1 = std::min(idx.size(), j0 + (size_t)kMaxDecodeJobs);
      const int64_t tokens = fmt == IL_BF16 ? kDecodeTokensBf16 : kDecodeTokensQ;
      for (int64_t t0 = 0; t0 < t; t0 += tokens) {
        DecodeParams p;
        memset(&p, 0, sizeof p);
        p.x = x != nullptr ? x + t0 * n_in : nullptr;
        p.t = (int)std::min<int64_t>(tokens, t - t0);
        p.x_row_stride = (int)n_in;
        p.n_in = (int)n_in;
        int groups = 0;
        for (size_t j = j0; j < j1; ++j) {
          const PackedWeight* w = ws[idx[j]];
          DecodeJob& dj = p.jobs[p.n_jobs++];
          dj.w = w->quants;
          dj.y = jobs[idx[j]].y + t0 * out_width(*w);
          dj.n_out = (int32_t)w->n_out;
          dj.glu = w->glu;
          dj.group_begin = groups;
          dj.row_stride = fmt == IL_BF16 ? w->n_in_pad : w->n_chunks;
          groups += (int)w->n_groups;
          p.n_chunks = (int)w->n_chunks;
        }
        p.total_groups = groups;
        out->emplace_back(fmt, p);
      }
    }
  }
}

}  // namespace

size_t plan_workspace_bytes(const BatchPlan& plan, int64_t t, int64_t n_in, const il_job* jobs,
                            const std::vector<const PackedWeight*>& ws, int num_sms) {
  size_t need = 0;
  for (int f = 0; f < 3; ++f)
    if (!plan.gemm[f].empty())
      need = std::max(need, gemm_workspace_bytes(t, plan.n_in_pad, plan.gemm[f].data(), (int)plan.gemm[f].size(),
                                                 num_sms));
  if (plan.decode[IL_Q8].empty() && plan.decode[IL_Q4].empty()) return need;  // only Q8/Q4 decode splits
  std::vector<std::pair<int, DecodeParams>> dl;
  decode_launch_params(plan, nullptr, t, n_in, jobs, ws, &dl);
  for (const auto& fp : dl)
    if (fp.first != IL_BF16) need = std::max(need, qdecode_workspace_bytes(fp.first, fp.second, num_sms));
  return need;
}

cudaError_t prepare_batch(const BatchPlan& plan, const float* x, int64_t t, int64_t n_in, const il_job* jobs,
                          const std::vector<const PackedWeight*>& ws, __nv_bfloat16* xb, void* wsp,
                          size_t ws_bytes, int num_sms, unsigned* status, std::vector<Launch>* out) {
  // large t: x cast to bf16 once, then one tensor-core launch per format (and
  // per kMaxGemmJobs jobs)
  if (plan.xb_bytes > 0) {
    if (xb == nullptr) return cudaErrorInvalidValue;
    Launch cast;
    cudaError_t e = prepare_cast_bf16(x, t, n_in, plan.n_in_pad, xb, num_sms, &cast);
    if (e != cudaSuccess) return e;
    out->push_back(cast);
    for (int f = 0; f < 3; ++f)
      if (!plan.gemm[f].empty()) {
        e = prepare_gemm(f, xb, t, plan.n_in_pad, plan.gemm[f].data(), (int)plan.gemm[f].size(), num_sms, status,
                         wsp, ws_bytes, out);
        if (e != cudaSuccess) return e;
      }
  }
  // small t: the decode kernel
  std::vector<std::pair<int, DecodeParams>> dl;
  decode_launch_params(plan, x, t, n_in, jobs, ws, &dl);
  for (const auto& fp : dl) {
    Launch L;
    cudaError_t e = prepare_decode(fp.first, fp.second, num_sms, status, wsp, ws_bytes, &L);
    if (e != cudaSuccess) return e;
    out->push_back(L);
  }
  return cudaSuccess;
}

void api_clear_error() { clear_error(); }

int api_fail(int code, const char* msg) { return fail(code, "%s", msg); }

int api_cuda_fail(cudaError_t e, const char* what) { return cuda_fail(e, what); }

// The checks that need no device: sizes, null pointers, x alignment (device x).
int check_batch_args(const float* x, int64_t t, int64_t n_in, const il_job* jobs, int n_jobs, bool host_x) {
  if (t < 0 || t > kMaxT) return fail(IL_ERR_ARG, "t=%lld out of range", (long long)t);
  if (n_jobs < 0 || n_jobs > kMaxJobs) return fail(IL_ERR_ARG, "n_jobs=%d out of range", n_jobs);
  if (t == 0 || n_jobs == 0) return IL_OK;
  if (x == nullptr) return fail(IL_ERR_ARG, "x is NULL");
  if (jobs == nullptr) return fail(IL_ERR_ARG, "jobs is NULL");
  if (!host_x && reinterpret_cast<uintptr_t>(x) % 16 != 0) return fail(IL_ERR_ARG, "x is not 16-byte aligned");
  if (n_in < 1 || n_in > kMaxNIn) return fail(IL_ERR_SHAPE, "n_in=%lld out of range", (long long)n_in);
  return IL_OK;
}

// Every job's checks on the calling thread's device `dev`; on success fills `ws`
// with the weight of each job.
int api_check_batch(const float* x, int64_t t, int64_t n_in, const il_job* jobs, int n_jobs, int dev,
                    std::vector<const PackedWeight*>* ws, uint64_t* wbytes, uint64_t* flops, bool host_x) {
  ws->clear();
  *wbytes = 0;
  *flops = 0;
  int rc = check_batch_args(x, t, n_in, jobs, n_jobs, host_x);
  if (rc != IL_OK || t == 0 || n_jobs == 0) return rc;
  std::vector<std::pair<uintptr_t, uintptr_t>> ranges;
  ranges.reserve(n_jobs + 1);
  ranges.emplace_back(reinterpret_cast<uintptr_t>(x), reinterpret_cast<uintptr_t>(x) + (uintptr_t)(t * n_in * 4));
  {
    std::lock_guard<std::mutex> lk(g_reg_mu);
    for (int j = 0; j < n_jobs; ++j) {
      const PackedWeight* w = reinterpret_cast<const PackedWeight*>(jobs[j].w);
      if (w == nullptr || g_registry.count(w) == 0 || w->magic != kWeightMagic)
        return fail(IL_ERR_HANDLE, "job %d has an invalid weight handle", j);
      if (w->device != dev)
        return fail(IL_ERR_HANDLE, "job %d weight lives on device %d, current is %d", j, w->device, dev);
      if (w->n_in != n_in) return fail(IL_ERR_SHAPE, "job %d weight n_in=%lld, batch n_in=%lld", j,
                                       (long long)w->n_in, (long long)n_in);
      if (jobs[j].n_out != out_width(*w)) return fail(IL_ERR_SHAPE, "job %d n_out=%lld, weight n_out=%lld", j,
                                                      (long long)jobs[j].n_out, (long long)out_width(*w));
      if (jobs[j].y == nullptr) return fail(IL_ERR_ARG, "job %d y is NULL", j);
      if (reinterpret_cast<uintptr_t>(jobs[j].y) % 4 != 0) return fail(IL_ERR_ARG, "job %d y is not 4-byte aligned", j);
      const uintptr_t y0 = reinterpret_cast<uintptr_t>(jobs[j].y);
      ranges.emplace_back(y0, y0 + (uintptr_t)(t * out_width(*w) * 4));
      ws->push_back(w);
      *wbytes += (uint64_t)w->host_bytes;
      *flops += 2ull * (uint64_t)t * (uint64_t)n_in * (uint64_t)w->n_out;
    }
  }
  std::sort(ranges.begin(), ranges.end());
  for (size_t i = 1; i < ranges.size(); ++i)
    if (overlaps(ranges[i - 1].first, ranges[i - 1].second, ranges[i].first, ranges[i].second))
      return fail(IL_ERR_ARG, "x and the y buffers must not overlap");
  return IL_OK;
}

void api_count_batch(int n_jobs, int launches, uint64_t wbytes, uint64_t flops) {
  g_stats.batches.fetch_add(1);
  g_stats.jobs.fetch_add((uint64_t)n_jobs);
  g_stats.launches.fetch_add((uint64_t)launches);
  g_stats.weight_bytes.fetch_add(wbytes);
  g_stats.flops.fetch_add(flops);
}

}  // namespace il
