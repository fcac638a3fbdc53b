// il_noalloc.cu -- il_matmul_batch_noalloc: the batched linear of
// il_matmul_batch for callers that cannot let the library allocate device
// memory.  Such callers include services that hand all device memory to their
// own pool at start-up (so a cudaMalloc from inside a library would fail or
// break their memory budget), and latency-critical threads that cannot afford
// cudaMalloc / cudaFree, which may block and synchronise the whole device.
//
// The scratch memory the batched linear needs -- the bf16 copy of x that the
// tensor-core path streams, and the split workspace of the Q8/Q4 decode kernel
// when it splits K over CTAs -- lives in file-scope device arrays of fixed
// size, and so does the status word of the kernels' bounded waits.  Every GPU
// that loads the library holds them until the process exits.
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "il_internal.cuh"

namespace {

using namespace il;

// Largest bf16 copy of x the tensor-core path can stage here:
// t * round_up(n_in, 256) * 2 bytes <= 16 MiB (t = 2048 at n_in = 4096).
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

// Split workspace of the Q8/Q4 decode kernel: arrival counters, then per-slice
// partial sums; a launch whose split would need more splits K less.
constexpr size_t kNoAllocWorkspaceBytes = size_t(4) << 20;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
__device__ __align__(256) unsigned char g_noalloc_workspace[kNoAllocWorkspaceBytes];
__device__ __align__(256) unsigned g_noalloc_status[64];

// Device addresses of the arrays, looked up once per device.  In host code the
// array names only stand in for the symbols; the kernels must be given these
// addresses instead.
struct DeviceSlot {
  std::atomic<bool> ready{false};
  int num_sms = 0;
  void* scratch = nullptr;
  void* workspace = nullptr;
  unsigned* status = nullptr;
};
constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceSlot g_slots[kMaxDevices];

// First call on a device: look up the arrays' addresses and clear the status
// word on the caller's stream (ordered before this call's launches; no device
// synchronisation).
int setup_device(int dev, cudaStream_t stream, DeviceSlot** out) {
  if (dev < 0 || dev >= kMaxDevices) return api_fail(IL_ERR_UNSUPPORTED, "il_matmul_batch_noalloc: device id out of range");
  DeviceSlot& s = g_slots[dev];
  if (!s.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!s.ready.load(std::memory_order_relaxed)) {
      cudaDeviceProp prop;
      cudaError_t e = cudaGetDeviceProperties(&prop, dev);
      if (e != cudaSuccess) return api_cuda_fail(e, "il_matmul_batch_noalloc: cudaGetDeviceProperties");
      if (!(prop.major == 10 && prop.minor == 3))
        return api_fail(IL_ERR_UNSUPPORTED, "il_matmul_batch_noalloc: this library is built for sm_103a");
      void* scratch = nullptr;
      void* status = nullptr;
      e = cudaGetSymbolAddress(&scratch, g_noalloc_scratch);
      if (e != cudaSuccess) return api_cuda_fail(e, "il_matmul_batch_noalloc: cudaGetSymbolAddress(scratch)");
      e = cudaGetSymbolAddress(&status, g_noalloc_status);
      if (e != cudaSuccess) return api_cuda_fail(e, "il_matmul_batch_noalloc: cudaGetSymbolAddress(status)");
      void* workspace = nullptr;
      e = cudaGetSymbolAddress(&workspace, g_noalloc_workspace);
      if (e != cudaSuccess) return api_cuda_fail(e, "il_matmul_batch_noalloc: cudaGetSymbolAddress(workspace)");
      // the status word and the workspace's arrival counters must start at zero
      // (the kernels leave the counters at zero); the scratch is fully overwritten
      // by every call
      e = cudaMemsetAsync(status, 0, sizeof(unsigned) * 64, stream);
      if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, kSplitCounterBytes, stream);
      if (e != cudaSuccess) return api_cuda_fail(e, "il_matmul_batch_noalloc: clearing the status word");
      s.scratch = scratch;
      s.workspace = workspace;
      s.status = static_cast<unsigned*>(status);
      s.num_sms = prop.multiProcessorCount;
      s.ready.store(true, std::memory_order_release);
    }
  }
  *out = &s;
  return IL_OK;
}

}  // namespace

namespace il {

unsigned* noalloc_status_word(int dev) {
  if (dev < 0 || dev >= kMaxDevices || !g_slots[dev].ready.load(std::memory_order_acquire)) return nullptr;
  return g_slots[dev].status;
}

void* noalloc_split_counters(int dev, size_t* bytes) {
  if (dev < 0 || dev >= kMaxDevices || !g_slots[dev].ready.load(std::memory_order_acquire)) return nullptr;
  *bytes = kSplitCounterBytes;
  return g_slots[dev].workspace;
}

}  // namespace il

extern "C" int il_matmul_batch_noalloc(const float* x, int64_t t, int64_t n_in, const il_job* jobs, int n_jobs,
                                       void* stream_) {
  api_clear_error();
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return api_cuda_fail(e, "il_matmul_batch_noalloc: cudaGetDevice");
  std::vector<const PackedWeight*> ws;
  uint64_t wbytes = 0, flops = 0;
  int rc = api_check_batch(x, t, n_in, jobs, n_jobs, dev, &ws, &wbytes, &flops);
  if (rc != IL_OK) return rc;
  if (t == 0 || n_jobs == 0) return IL_OK;

  // the same split over the kernels as il_matmul_batch; x's bf16 copy goes to the
  // static scratch and the tensor-core launches split K only as CTA pairs (no workspace)
  BatchPlan plan;
  plan_batch(t, jobs, n_jobs, ws, /*gemm_quant=*/true, &plan);
  if (plan.xb_bytes > kNoAllocScratchBytes)
    return api_fail(IL_ERR_UNSUPPORTED,
                    "il_matmul_batch_noalloc: t * round_up(n_in, 256) * 2 bytes exceeds the 16 MiB static scratch");
  DeviceSlot* slot = nullptr;
  rc = setup_device(dev, stream, &slot);
  if (rc != IL_OK) return rc;
  std::vector<Launch> launches;
  // the tensor-core launches see no workspace (a split runs as CTA pairs or not at all); the
  // decode launches get the static one
  BatchPlan gplan = plan, dplan = plan;
  for (int f = 0; f < 3; ++f) gplan.decode[f].clear();
  for (int f = 0; f < 3; ++f) dplan.gemm[f].clear();
  dplan.xb_bytes = 0;
  e = prepare_batch(gplan, x, t, n_in, jobs, ws, static_cast<__nv_bfloat16*>(slot->scratch), nullptr, 0,
                    slot->num_sms, slot->status, &launches);
  if (e == cudaSuccess)
    e = prepare_batch(dplan, x, t, n_in, jobs, ws, nullptr, slot->workspace, kNoAllocWorkspaceBytes, slot->num_sms,
                      slot->status, &launches);
  if (e != cudaSuccess) return api_cuda_fail(e, "il_matmul_batch_noalloc: preparing the launches");
  int n_launched = 0;
  e = run_launches(launches, stream, &n_launched);
  if (e != cudaSuccess) return api_cuda_fail(e, "il_matmul_batch_noalloc: launch");
  api_count_batch(n_jobs, n_launched, wbytes, flops);
  return IL_OK;
}
