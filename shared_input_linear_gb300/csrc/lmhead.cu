// lmhead.cu -- centroid-masked LM head (oxinfer 0.0.1, src/drafter.rs, end of
// `Drafter::step`): the logits of the vocabulary's centroids pick the top-k
// clusters, and only the tokens of those clusters get an exact logit; the
// result is the first maximum.
//
//   1. cl = centroids . x               decode kernel (a one-job batch, t = 1)
//   2. sel = top-k of cl                 topk_kernel: one CTA, bitonic sort of
//                                        rank keys in shared memory
//   3. score[i*per + j] =                cluster_score_kernel: one warp per
//        embed[ordering[sel[i]*per+j]].x gathered row, bf16 x fp32 in fp32
//   4. first maximum                     same kernel: 64-bit keys, atomicMax per
//                                        CTA, the last CTA to finish writes the token
//
// Order and ties (the page selects with an unstable partition and scans with a
// strict '>'): centroids rank by larger logit, NaN last, ties to the lower
// index, and are visited in that order; among equal scores the first in
// (rank, position) order wins; NaN and -inf never win, and with no winner the
// token is 0 and the score -inf.
#include <math.h>

#include <atomic>

#include "il_internal.cuh"

namespace il {
namespace {

constexpr int kTopkThreads = 512;
constexpr int kSelectMax = 4096;  // larger k sorts every key instead of selecting
constexpr int kScoreThreads = 256;
constexpr int kRowVecs = 16;  // rows up to 32 * 16 * 8 = 4096 wide are loaded in one go

// fp32 -> u32 whose unsigned order is the float order (-inf lowest of the numbers).
__device__ __forceinline__ uint32_t orderable(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float from_orderable(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

// Larger key = earlier rank: logit first (NaN as the lowest), then lower index.
// Key 0 is below every centroid (padding of the sort).
__device__ __forceinline__ unsigned long long rank_key(float v, uint32_t i) {
  const uint32_t o = isnan(v) ? 0u : orderable(v);
  return ((unsigned long long)o << 32) | (uint32_t)~i;
}

// Descending bitonic sort of a[0 .. p) in shared memory, p a power of two.
__device__ void bitonic_desc(unsigned long long* a, int p) {
  for (int size = 2; size <= p; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = threadIdx.x; t < (p >> 1); t += blockDim.x) {
        const int lo = 2 * stride * (t / stride) + (t % stride);
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const unsigned long long x = a[lo], y = a[hi];
        if ((x < y) == desc) {
          a[lo] = y;
          a[hi] = x;
        }
      }
      __syncthreads();
    }
  }
}

// One CTA selects the k largest rank keys of the n centroids and writes their
// indices in rank order.  k <= kSelectMax: a radix select over the 64-bit keys
// (8-bit digits from the top; the keys are distinct, so the k-th largest is
// unique) finds the threshold, the k keys at or above it are gathered and only
// they are sorted.  Larger k: the whole key array (padded to p) is sorted.
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float* __restrict__ cl, int n, int p, int k,
                                                            uint32_t* __restrict__ sel) {
  extern __shared__ unsigned long long keys[];
  __shared__ unsigned hist[256];
  __shared__ unsigned s_bin, s_above, s_count, s_gathered;
  grid_dep_wait();  // cl comes from the previous kernel
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (k > kSelectMax) {
    for (int i = threadIdx.x; i < p; i += blockDim.x) keys[i] = i < n ? rank_key(cl[i], (uint32_t)i) : 0ull;
    __syncthreads();
    bitonic_desc(keys, p);
    for (int r = threadIdx.x; r < k; r += blockDim.x) sel[r] = ~(uint32_t)keys[r];
    grid_dep_launch();
    return;
  }
  for (int i = threadIdx.x; i < n; i += blockDim.x) keys[i] = rank_key(cl[i], (uint32_t)i);
  unsigned long long prefix = 0ull, mask = 0ull;
  unsigned remaining = (unsigned)k;  // how many of the keys matching prefix under mask are still to take
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int b = threadIdx.x; b < 256; b += blockDim.x) hist[b] = 0u;
    __syncthreads();
    // most keys share their top bits: lanes with the same bin add once, together
    for (int base = 0; base < n; base += blockDim.x) {
      const int i = base + (int)threadIdx.x;
      const unsigned long long key = i < n ? keys[i] : 0ull;
      const bool is_cand = i < n && (key & mask) == prefix;
      const unsigned bin = is_cand ? ((unsigned)(key >> shift) & 255u) : 256u;
      const unsigned peers = __match_any_sync(0xffffffffu, bin);
      if (is_cand && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], (unsigned)__popc(peers));
    }
    __syncthreads();
    if (warp == 0) {
      // lane L holds bins 8L .. 8L+7; count the candidates in the bins above each
      unsigned c[8], local = 0u;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        c[q] = hist[lane * 8 + q];
        local += c[q];
      }
      unsigned incl = local;  // candidates in this lane's bins and every higher lane's
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned v = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += v;
      }
      unsigned above = incl - local;
#pragma unroll
      for (int q = 7; q >= 0; --q) {
        if (above < remaining && remaining <= above + c[q]) {  // the k-th largest falls in this bin
          s_bin = (unsigned)(lane * 8 + q);
          s_above = above;
          s_count = c[q];
        }
        above += c[q];
      }
    }
    __syncthreads();
    remaining -= s_above;
    prefix |= (unsigned long long)s_bin << shift;
    mask |= 255ull << shift;
    const bool done = s_count == remaining;  // every candidate in the bin is taken
    __syncthreads();                         // s_* are rewritten by the next round
    if (done) break;
  }
  // gather the k keys whose top bits (under mask) are at least prefix
  unsigned long long* cand = keys + n;
  int pk = 1;
  while (pk < k) pk <<= 1;
  if (threadIdx.x == 0) s_gathered = 0u;
  for (int i = threadIdx.x; i < pk; i += blockDim.x) cand[i] = 0ull;
  __syncthreads();
  for (int base = 0; base < n; base += blockDim.x) {
    const int i = base + (int)threadIdx.x;
    const unsigned long long key = i < n ? keys[i] : 0ull;
    const bool win = i < n && (key & mask) >= prefix;
    const unsigned ballot = __ballot_sync(0xffffffffu, win);
    unsigned at = 0u;
    if (lane == 0 && ballot != 0u) at = atomicAdd(&s_gathered, (unsigned)__popc(ballot));
    at = __shfl_sync(0xffffffffu, at, 0);
    if (win) cand[at + __popc(ballot & ((1u << lane) - 1u))] = key;
  }
  __syncthreads();
  bitonic_desc(cand, pk);
  for (int r = threadIdx.x; r < k; r += blockDim.x) sel[r] = ~(uint32_t)cand[r];
  grid_dep_launch();
}

// Warp per gathered row; x staged once per CTA.  Each CTA folds its best key into
// *best_key; the last CTA to finish turns it into the token and resets the state.
__global__ void __launch_bounds__(kScoreThreads) cluster_score_kernel(
    const float* __restrict__ x, int h, const uint16_t* __restrict__ embed, int64_t row_pitch,
    const uint32_t* __restrict__ ordering, int64_t vocab, const uint32_t* __restrict__ sel, int k, int per,
    float* __restrict__ scores_out, unsigned long long* best_key, unsigned* done, uint32_t* __restrict__ token_out,
    float* __restrict__ score_out, unsigned* status) {
  extern __shared__ float4 xs4[];
  __shared__ unsigned long long warp_best[kScoreThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  grid_dep_wait();  // sel comes from the previous kernel
  const float4* x4 = reinterpret_cast<const float4*>(x);
  for (int i = threadIdx.x; i < h / 4; i += blockDim.x) xs4[i] = x4[i];
  __syncthreads();

  const int rows = k * per;
  unsigned long long best = 0ull;
  for (int row = blockIdx.x * (kScoreThreads / 32) + warp; row < rows; row += gridDim.x * (kScoreThreads / 32)) {
    const int i = row / per, j = row - (row / per) * per;
    const uint32_t tok = ordering[(int64_t)sel[i] * per + j];
    const bool valid = (int64_t)tok < vocab;
    float acc = 0.f;
    if (valid) {
      const uint4* w = reinterpret_cast<const uint4*>(embed + (int64_t)tok * row_pitch);
      const int nv = h / 8;  // 16-byte vectors in the row
      auto dot8 = [&](const uint4& v, int e) {
        const float4 a = xs4[2 * e], b = xs4[2 * e + 1];
        acc = fmaf(bf16_lo(v.x), a.x, acc);
        acc = fmaf(bf16_hi(v.x), a.y, acc);
        acc = fmaf(bf16_lo(v.y), a.z, acc);
        acc = fmaf(bf16_hi(v.y), a.w, acc);
        acc = fmaf(bf16_lo(v.z), b.x, acc);
        acc = fmaf(bf16_hi(v.z), b.y, acc);
        acc = fmaf(bf16_lo(v.w), b.z, acc);
        acc = fmaf(bf16_hi(v.w), b.w, acc);
      };
      if (nv <= 32 * kRowVecs) {
        // the whole row in flight at once: every lane issues all its loads first
        uint4 v[kRowVecs];
#pragma unroll
        for (int m = 0; m < kRowVecs; ++m)
          if (lane + 32 * m < nv) v[m] = __ldg(w + lane + 32 * m);
#pragma unroll
        for (int m = 0; m < kRowVecs; ++m)
          if (lane + 32 * m < nv) dot8(v[m], lane + 32 * m);
      } else {
#pragma unroll 4
        for (int e = lane; e < nv; e += 32) dot8(__ldg(w + e), e);
      }
    } else if (lane == 0) {
      atomicOr(status, kStatusBadToken);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
      if (scores_out != nullptr) scores_out[row] = valid ? acc : __int_as_float(0x7fc00000);
      if (valid && acc > -INFINITY) {  // false for NaN
        const unsigned long long key = ((unsigned long long)orderable(acc) << 32) | (uint32_t)~(uint32_t)row;
        best = key > best ? key : best;
      }
    }
  }
  if (lane == 0) warp_best[warp] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long b = 0ull;
    for (int w = 0; w < kScoreThreads / 32; ++w) b = warp_best[w] > b ? warp_best[w] : b;
    if (b != 0ull) atomicMax(best_key, b);
    __threadfence();
    const unsigned prev = atomicAdd(done, 1u);
    if (prev == gridDim.x - 1) {
      // every other CTA has folded its key in (they fenced before counting)
      __threadfence();
      const unsigned long long key = atomicAdd(best_key, 0ull);
      if (key == 0ull) {
        *token_out = 0u;
        if (score_out != nullptr) *score_out = -INFINITY;
      } else {
        const int row = (int)~(uint32_t)key;
        const int i = row / per, j = row - (row / per) * per;
        *token_out = ordering[(int64_t)sel[i] * per + j];
        if (score_out != nullptr) *score_out = from_orderable((uint32_t)(key >> 32));
      }
      *best_key = 0ull;  // ready for the next call on this stream
      *done = 0u;
    }
  }
  grid_dep_launch();
}

}  // namespace

// Shared memory of topk_kernel: the sorted key array (padded to a power of two)
// for k > kSelectMax, else the keys and the gathered winners (padded).
size_t topk_smem(int n_cent, int k) {
  int p = 1;
  while (p < n_cent) p <<= 1;
  int pk = 1;
  while (pk < k) pk <<= 1;
  return k > kSelectMax ? (size_t)p * sizeof(unsigned long long)
                        : ((size_t)n_cent + (size_t)pk) * sizeof(unsigned long long);
}

cudaError_t prepare_lmhead(const float* x, int h, const float* cl, int n_cent, int k, const PackedWeight& embed,
                           const uint32_t* ordering, int per, uint32_t* sel, float* scores_out,
                           unsigned long long* best_key, unsigned* done, uint32_t* token_out, float* score_out,
                           unsigned* status, int num_sms, std::vector<Launch>* out) {
  int p = 1;
  while (p < n_cent) p <<= 1;
  static std::atomic<unsigned long long> attr_set{0};  // one bit per device (setting it twice is harmless)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !(attr_set.load() & (1ull << dev))) {
    // the largest need: kMaxCentroids keys plus kSelectMax winners
    cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)topk_smem(kMaxCentroids, kSelectMax));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(cluster_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)(kMaxHeadWidth * sizeof(float)));
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set.fetch_or(1ull << dev);
  }
  Launch a;
  a.fn = reinterpret_cast<const void*>(topk_kernel);
  a.grid = dim3(1);
  a.block = dim3(kTopkThreads);
  a.smem = topk_smem(n_cent, k);
  if (kUsePdl) a.allow_early_start();
  if (!a.set_args(cl, n_cent, p, k, sel)) return cudaErrorMemoryAllocation;

  const int rows = k * per;
  const int warps_per_cta = kScoreThreads / 32;
  int grid = (rows + warps_per_cta - 1) / warps_per_cta;
  if (grid > 4 * num_sms) grid = 4 * num_sms;
  Launch b;
  b.fn = reinterpret_cast<const void*>(cluster_score_kernel);
  b.grid = dim3(grid);
  b.block = dim3(kScoreThreads);
  b.smem = (size_t)h * sizeof(float);
  if (kUsePdl) b.allow_early_start();
  if (!b.set_args(x, h, reinterpret_cast<const uint16_t*>(embed.quants), (int64_t)embed.n_in_pad, ordering,
                  (int64_t)embed.n_out, (const uint32_t*)sel, k, per, scores_out, best_key, done, token_out,
                  score_out, status))
    return cudaErrorMemoryAllocation;
  out->push_back(a);
  out->push_back(b);
  return cudaSuccess;
}

}  // namespace il
