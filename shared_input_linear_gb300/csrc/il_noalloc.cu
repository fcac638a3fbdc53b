// il_noalloc.cu -- il_matmul_batch_noalloc: the batched linear of
// il_matmul_batch for callers that cannot let the library allocate device
// memory.  Such callers include services that hand all device memory to their
// own pool at start-up (so a cudaMalloc from inside a library would fail or
// break their memory budget), and latency-critical threads that cannot afford
// cudaMalloc / cudaFree, which may block and synchronise the whole device.
//
// The one piece of scratch memory the batched linear needs -- the bf16 copy of
// x that the tensor-core path streams -- lives in a file-scope device array of
// fixed size, and so does the status word of the kernel's bounded waits.  Every
// GPU that loads the library holds both until the process exits.
#include <cstring>
#include <mutex>
#include <vector>

#include "il_internal.cuh"

namespace il {
int api_check_batch(const float* x, int64_t t, int64_t n_in, const il_job* jobs, int n_jobs, int dev,
                    std::vector<const PackedWeight*>* ws, uint64_t* wbytes, uint64_t* flops);
void api_clear_error();
int api_fail(int code, const char* msg);
int api_cuda_fail(cudaError_t e, const char* what);
void api_count_batch(int n_jobs, int launches, uint64_t wbytes, uint64_t flops);
}  // namespace il

namespace {

using namespace il;

// Largest bf16 copy of x the tensor-core path can stage here:
// t * round_up(n_in, 128) * 2 bytes <= 16 MiB (t = 2048 at n_in = 4096).
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
__device__ __align__(256) unsigned g_noalloc_status[64];

// Device addresses of the arrays, looked up once per device.  In host code the
// array names only stand in for the symbols; the kernels must be given these
// addresses instead.
struct DeviceSlot {
  bool ready = false;
  int num_sms = 0;
  void* scratch = nullptr;
  unsigned* status = nullptr;
};
constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceSlot g_slots[kMaxDevices];

int setup_device(int dev, DeviceSlot** out) {
  if (dev < 0 || dev >= kMaxDevices) return api_fail(IL_ERR_UNSUPPORTED, "il_matmul_batch_noalloc: device id out of range");
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceSlot& s = g_slots[dev];
  if (!s.ready) {
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
    // the status word must start at zero; the scratch is fully overwritten by every call
    e = cudaMemset(status, 0, sizeof(unsigned) * 64);
    if (e != cudaSuccess) return api_cuda_fail(e, "il_matmul_batch_noalloc: clearing the status word");
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return api_cuda_fail(e, "il_matmul_batch_noalloc: set-up");
    s.scratch = scratch;
    s.status = static_cast<unsigned*>(status);
    s.num_sms = prop.multiProcessorCount;
    s.ready = true;
  }
  *out = &s;
  return IL_OK;
}

}  // namespace

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
  DeviceSlot* slot = nullptr;
  rc = setup_device(dev, &slot);
  if (rc != IL_OK) return rc;

  // tensor-core path (bf16 weights, t > 8): x's bf16 copy goes to the static scratch
  std::vector<GemmJob> gj;
  int64_t n_in_pad = 0;
  if (t > 8) {
    for (int j = 0; j < n_jobs; ++j)
      if (ws[j]->format == IL_BF16) {
        gj.push_back(GemmJob{ws[j], jobs[j].y});
        n_in_pad = ws[j]->n_in_pad;
      }
    if (!gj.empty() && (size_t)t * (size_t)n_in_pad * 2 > kNoAllocScratchBytes)
      return api_fail(IL_ERR_UNSUPPORTED,
                      "il_matmul_batch_noalloc: t * round_up(n_in, 128) * 2 bytes exceeds the 16 MiB static scratch");
  }
  int launches = 0;
  if (!gj.empty()) {
    __nv_bfloat16* xb = static_cast<__nv_bfloat16*>(slot->scratch);
    e = launch_cast_bf16(x, t, n_in, n_in_pad, xb, stream);
    if (e == cudaSuccess) ++launches;
    if (e == cudaSuccess)
      e = launch_gemm(IL_BF16, xb, t, n_in_pad, gj.data(), (int)gj.size(), stream, slot->num_sms, slot->status,
                      &launches, nullptr, 0);
  }
  // decode path (t <= 8, or Q8/Q4 weights): needs no scratch
  for (int fmt = IL_BF16; fmt <= IL_Q4 && e == cudaSuccess; ++fmt) {
    if (!gj.empty() && fmt == IL_BF16) continue;
    std::vector<int> idx;
    for (int j = 0; j < n_jobs; ++j)
      if (ws[j]->format == fmt) idx.push_back(j);
    for (size_t j0 = 0; j0 < idx.size() && e == cudaSuccess; j0 += kMaxDecodeJobs) {
      const size_t j1 = idx.size() < j0 + kMaxDecodeJobs ? idx.size() : j0 + kMaxDecodeJobs;
      for (int64_t t0 = 0; t0 < t && e == cudaSuccess; t0 += 8) {
        DecodeParams p;
        memset(&p, 0, sizeof p);
        p.x = x + t0 * n_in;
        p.t = (int)(t - t0 < 8 ? t - t0 : 8);
        p.x_row_stride = (int)n_in;
        p.n_in = (int)n_in;
        int groups = 0;
        for (size_t j = j0; j < j1; ++j) {
          const PackedWeight* w = ws[idx[j]];
          DecodeJob& dj = p.jobs[p.n_jobs++];
          dj.w = w->quants;
          dj.s = w->scales;
          dj.y = jobs[idx[j]].y + t0 * out_width(*w);
          dj.n_out = (int32_t)w->n_out;
          dj.glu = w->glu;
          dj.group_begin = groups;
          dj.row_stride = fmt == IL_BF16 ? w->n_in_pad : w->n_chunks;
          groups += (int)w->n_groups;
          p.n_chunks = (int)w->n_chunks;
        }
        p.total_groups = groups;
        e = launch_decode(fmt, p, stream, slot->num_sms, &launches);
      }
    }
  }
  if (e != cudaSuccess) return api_cuda_fail(e, "il_matmul_batch_noalloc: launch");
  api_count_batch(n_jobs, launches, wbytes, flops);
  return IL_OK;
}
