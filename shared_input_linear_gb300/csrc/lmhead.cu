// lmhead.cu -- centroid-masked LM head (oxinfer 0.0.1, src/drafter.rs, end of
// `Drafter::step`): the logits of the vocabulary's centroids pick the top-k
// clusters, and only the tokens of those clusters get an exact logit; the
// result is the first maximum.
//
//   1. cl = centroids . x               decode kernel (a one-job batch, t = 1)
//   2. sel = top-k of cl                 k <= 32: inside the scoring kernel, every
//                                        CTA for itself (select_score_kernel);
//                                        larger k: topk_kernel, one CTA, radix
//                                        select of rank keys in shared memory
//   3. score[i*per + j] =                one warp per gathered row, bf16 x fp32
//        embed[ordering[sel[i]*per+j]].x in fp32 (cluster_score_kernel after
//                                        topk_kernel)
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
constexpr int kFusedK = 32;   // k up to this: selection inside the scoring kernel
constexpr int kFusedThreads = 512;
constexpr int kKeyRegs = 8;  // centroid keys per thread held in registers by the selection

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

// x [h] -> shared memory as fp32 (h is a multiple of 8: bf16 weights are
// uploaded only so, and h is their row length).
__device__ __forceinline__ void stage_x(const float* __restrict__ x, int h, float4* xs4) {
  const float4* x4 = reinterpret_cast<const float4*>(x);
  for (int i = threadIdx.x; i < h / 4; i += blockDim.x) xs4[i] = x4[i];
}

// The exact logits of the k selected clusters' tokens, a warp per gathered row
// (xs4: x staged in shared memory), and the first maximum.  Each CTA folds its
// best key into *best_key; the last CTA to finish turns it into the token and
// resets the state.  sel may be global or shared memory.
template <int NW>
__device__ __forceinline__ void score_rows(const float4* xs4, int h, const uint16_t* __restrict__ embed,
                                           int64_t row_pitch, const uint32_t* __restrict__ ordering, int64_t vocab,
                                           const uint32_t* sel, int k, int per, float* __restrict__ scores_out,
                                           unsigned long long* best_key, unsigned* done,
                                           uint32_t* __restrict__ token_out, float* __restrict__ score_out,
                                           unsigned* status, unsigned long long* warp_best) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rows = k * per;
  unsigned long long best = 0ull;
  for (int row = blockIdx.x * NW + warp; row < rows; row += gridDim.x * NW) {
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
    for (int w = 0; w < NW; ++w) b = warp_best[w] > b ? warp_best[w] : b;
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
}

// Scoring after topk_kernel (k > kFusedK): x staged once per CTA.
__global__ void __launch_bounds__(kScoreThreads) cluster_score_kernel(
    const float* __restrict__ x, int h, const uint16_t* __restrict__ embed, int64_t row_pitch,
    const uint32_t* __restrict__ ordering, int64_t vocab, const uint32_t* __restrict__ sel, int k, int per,
    float* __restrict__ scores_out, unsigned long long* best_key, unsigned* done, uint32_t* __restrict__ token_out,
    float* __restrict__ score_out, unsigned* status) {
  extern __shared__ float4 xs4[];
  __shared__ unsigned long long warp_best[kScoreThreads / 32];
  grid_dep_wait();  // sel comes from the previous kernel
  stage_x(x, h, xs4);
  __syncthreads();
  score_rows<kScoreThreads / 32>(xs4, h, embed, row_pitch, ordering, vocab, sel, k, per, scores_out, best_key, done,
                                 token_out, score_out, status, warp_best);
  grid_dep_launch();
}

// ---- selection of at most 32 centroids inside the scoring kernel

__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
  return a > b ? a : b;
}
__device__ __forceinline__ unsigned long long umin64(unsigned long long a, unsigned long long b) {
  return a < b ? a : b;
}

// One key per lane, sorted descending over the lanes (lane 0 the largest): a
// bitonic network whose blocks alternate direction until the last pass.
__device__ __forceinline__ unsigned long long warp_sort_desc(unsigned long long key, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, key, stride);
      const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0);
      key = keep_max ? umax64(key, o) : umin64(key, o);
    }
  return key;
}

// A bitonic sequence over the lanes, sorted descending.
__device__ __forceinline__ unsigned long long warp_merge_desc(unsigned long long key, int lane) {
#pragma unroll
  for (int stride = 16; stride > 0; stride >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xffffffffu, key, stride);
    key = (lane & stride) == 0 ? umax64(key, o) : umin64(key, o);
  }
  return key;
}

// The 32 largest of two descending lists a and b (one key per lane): the lane-wise
// maximum of a and reversed b is bitonic and holds them.
__device__ __forceinline__ unsigned long long warp_top_of_two(unsigned long long a, unsigned long long b, int lane) {
  return warp_merge_desc(umax64(a, __shfl_sync(0xffffffffu, b, 31 - lane)), lane);
}

// k <= kFusedK: every CTA selects the top k centroids itself (16 KB of logits from
// L2) and scores its share of their rows -- one launch instead of two.
//
// Selection, exact for any input: (1) each lane's largest key over its share of
// the n keys; each warp's two largest lane maxima; T = the least of those 32
// values.  They come from 32 distinct lanes, each holding a key >= T, so at least
// 32 keys are >= T and the top 32 are among them.  (2) Keys >= T are gathered in
// shared memory, (3) sorted 32 at a time with a warp bitonic network into a
// running top 32 per warp, (4) the warps' lists are merged pairwise.
__global__ void __launch_bounds__(kFusedThreads, 1) select_score_kernel(
    const float* __restrict__ x, int h, const float* __restrict__ cl, int n, const uint16_t* __restrict__ embed,
    int64_t row_pitch, const uint32_t* __restrict__ ordering, int64_t vocab, uint32_t* __restrict__ sel_out, int k,
    int per, float* __restrict__ scores_out, unsigned long long* best_key, unsigned* done,
    uint32_t* __restrict__ token_out, float* __restrict__ score_out, unsigned* status) {
  constexpr int NW = kFusedThreads / 32;
  extern __shared__ float4 xs4[];  // x [h] | candidates [n]
  __shared__ unsigned long long lists[NW][32];
  __shared__ unsigned long long pair_min[NW];
  __shared__ unsigned long long warp_best[NW];
  __shared__ uint32_t sel[kFusedK];
  __shared__ unsigned n_cand;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long* cand = reinterpret_cast<unsigned long long*>(xs4 + h / 4);

  // x is this call's input, written before the previous kernel of the call began
  stage_x(x, h, xs4);
  if (threadIdx.x == 0) n_cand = 0u;
  grid_dep_wait();  // cl comes from the previous kernel

  // (1) threshold.  The first kKeyRegs * 512 keys stay in registers for the gather
  // (all their loads in flight at once); keys past them are read again from L2.
  unsigned long long kr[kKeyRegs];
#pragma unroll
  for (int u = 0; u < kKeyRegs; ++u) {
    const int i = (int)threadIdx.x + u * kFusedThreads;
    const float v = i < n ? __ldcg(cl + i) : 0.f;
    kr[u] = i < n ? rank_key(v, (uint32_t)i) : 0ull;
  }
  unsigned long long lmax = 0ull;
#pragma unroll
  for (int u = 0; u < kKeyRegs; ++u) lmax = umax64(lmax, kr[u]);
  for (int i = (int)threadIdx.x + kKeyRegs * kFusedThreads; i < n; i += kFusedThreads)
    lmax = umax64(lmax, rank_key(__ldcg(cl + i), (uint32_t)i));
  unsigned long long m1 = lmax, m2 = 0ull;  // the warp's two largest lane maxima
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long b1 = __shfl_xor_sync(0xffffffffu, m1, o), b2 = __shfl_xor_sync(0xffffffffu, m2, o);
    m2 = umax64(umin64(m1, b1), umax64(m2, b2));
    m1 = umax64(m1, b1);
  }
  if (lane == 0) pair_min[warp] = m2;
  __syncthreads();
  unsigned long long thr = pair_min[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) thr = umin64(thr, pair_min[w]);
  // (2) gather the keys >= T (0 pads past n and is never >= T: T is a real key or 0,
  // and real keys are not 0 -- see rank_key)
  auto gather = [&](unsigned long long key, bool real) {
    const bool take = real && key >= thr;
    const unsigned ballot = __ballot_sync(0xffffffffu, take);
    unsigned at = 0u;
    if (lane == 0 && ballot != 0u) at = atomicAdd(&n_cand, (unsigned)__popc(ballot));
    at = __shfl_sync(0xffffffffu, at, 0);
    if (take) cand[at + __popc(ballot & ((1u << lane) - 1u))] = key;
  };
#pragma unroll
  for (int u = 0; u < kKeyRegs; ++u)
    if (u * kFusedThreads < n) gather(kr[u], (int)threadIdx.x + u * kFusedThreads < n);
  for (int base = kKeyRegs * kFusedThreads; base < n; base += kFusedThreads) {
    const int i = base + (int)threadIdx.x;
    gather(i < n ? rank_key(__ldcg(cl + i), (uint32_t)i) : 0ull, i < n);
  }
  __syncthreads();
  // (3) running top 32 per warp over chunks of 32 candidates
  const int nc = (int)n_cand;
  const int chunks = (nc + 31) / 32;
  const int nl = chunks < NW ? chunks : NW;  // lists that hold candidates
  if (warp < nl) {
    unsigned long long top = 0ull;
    for (int c = warp; c < chunks; c += NW) {
      const int e = c * 32 + lane;
      const unsigned long long s = warp_sort_desc(e < nc ? cand[e] : 0ull, lane);
      top = c == warp ? s : warp_top_of_two(top, s, lane);
    }
    lists[warp][lane] = top;
  }
  __syncthreads();
  // (4) pairwise merge of the lists: list w takes list w + s
  int span = 1;
  while (span < nl) span <<= 1;
  for (int s = span >> 1; s >= 1; s >>= 1) {
    if (warp < s && warp + s < nl) {
      const unsigned long long m = warp_top_of_two(lists[warp][lane], lists[warp + s][lane], lane);
      __syncwarp();
      lists[warp][lane] = m;
    }
    __syncthreads();
  }
  if (threadIdx.x < k) {
    const uint32_t c = ~(uint32_t)lists[0][threadIdx.x];
    sel[threadIdx.x] = c;
    if (blockIdx.x == 0 && sel_out != nullptr) sel_out[threadIdx.x] = c;
  }
  __syncthreads();
  // the next kernel may start; it waits for this one before reading its results
  grid_dep_launch();
  score_rows<NW>(xs4, h, embed, row_pitch, ordering, vocab, sel, k, per, scores_out, best_key, done, token_out,
                 score_out, status, warp_best);
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

// Dynamic shared memory of select_score_kernel: x, then the candidate keys (at
// most every centroid).
size_t fused_smem(int h, int n_cent) {
  return (size_t)h * sizeof(float) + (size_t)n_cent * sizeof(unsigned long long);
}
constexpr size_t kFusedSmemMax = 200 * 1024;

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
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(select_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kFusedSmemMax);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set.fetch_or(1ull << dev);
  }
  const int rows = k * per;
  if (k <= kFusedK && fused_smem(h, n_cent) <= kFusedSmemMax) {
    // one launch: every CTA selects, then scores its share of the rows
    int grid = (rows + kFusedThreads / 32 - 1) / (kFusedThreads / 32);
    if (grid > num_sms) grid = num_sms;
    Launch f;
    f.fn = reinterpret_cast<const void*>(select_score_kernel);
    f.grid = dim3(grid);
    f.block = dim3(kFusedThreads);
    f.smem = fused_smem(h, n_cent);
    if (kUsePdl) f.allow_early_start();
    if (!f.set_args(x, h, cl, n_cent, reinterpret_cast<const uint16_t*>(embed.quants), (int64_t)embed.n_in_pad,
                    ordering, (int64_t)embed.n_out, sel, k, per, scores_out, best_key, done, token_out, score_out,
                    status))
      return cudaErrorMemoryAllocation;
    out->push_back(f);
    return cudaSuccess;
  }
  Launch a;
  a.fn = reinterpret_cast<const void*>(topk_kernel);
  a.grid = dim3(1);
  a.block = dim3(kTopkThreads);
  a.smem = topk_smem(n_cent, k);
  if (kUsePdl) a.allow_early_start();
  if (!a.set_args(cl, n_cent, p, k, sel)) return cudaErrorMemoryAllocation;

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
