// pack.cu -- upload-time repacking of a weight into its device layout
// (oxinfer src/gpu.rs, `Backend::upload`: prepare device state for one weight),
// and the dequantise hook that reads the packed layout back element by element.
//
// Q8 chunk (8 rows x 64 columns, 512 bytes): lane L = 4n + q owns 16 bytes.
//   Byte 4i + j of the lane (i = 0..3 is the MMA slot, j = 0..3) holds column
//   16i + 4q + j of row n.  Slots 0,1 cover the chunk's first 32-block, 2,3 the
//   second, so every MMA stays inside one scale block.
// Q4 chunk (8 rows x 128 columns, 512 bytes): lane L owns four 32-bit words;
//   word w covers the 32-block w of the chunk (MMA slots 2w and 2w+1).  Nibble
//   position p (bits 4p..4p+3) of the word holds column 32w + 16*sub + 4q + j of
//   row n with sub = (p >> 1) & 1 and j = ((p & 1) << 1) | (p >> 2).  Taking the
//   nibbles at bits s and s+16 (s = 0, 4, 8, 12) then yields the bf16x2 operand
//   pairs (j = 0,1) and (j = 2,3) of slot 2w, then of slot 2w+1.
// Scales (Q8: 16 bytes, Q4: 32 bytes per (group, chunk, q)): the fp32 scales of
//   rows 2q and 2q+1 of the group for each 32-block of the chunk, row-major
//   (row 2q first).
#include "il_internal.cuh"

namespace il {
namespace {

__global__ void pack_bf16_kernel(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst,
                                 int64_t n_out, int64_t n_in, int64_t n_out_pad,
                                 int64_t n_in_pad) {
  const int64_t vec_per_row = n_in_pad / 8;
  const int64_t total = n_out_pad * vec_per_row;
  for (int64_t v = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; v < total;
       v += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = v / vec_per_row;
    const int64_t k = (v % vec_per_row) * 8;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (r < n_out && k < n_in) val = *reinterpret_cast<const uint4*>(src + r * n_in + k);
    *reinterpret_cast<uint4*>(dst + r * n_in_pad + k) = val;
  }
}

__global__ void pack_q8_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                               float* __restrict__ dst_s, int64_t n_out, int64_t n_in,
                               int64_t n_groups, int64_t n_chunks) {
  const float* src_s = reinterpret_cast<const float*>(src + n_out * n_in);
  const int64_t n_blocks = n_in / 32;
  const int64_t words = n_groups * n_chunks * 32 * 4;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < words;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int i = e & 3;
    const int lane = (e >> 2) & 31;
    const int64_t gc = e >> 7;  // group * n_chunks + chunk
    const int64_t g = gc / n_chunks, c = gc % n_chunks;
    const int n = lane >> 2, q = lane & 3;
    const int64_t row = g * 8 + n;
    const int64_t k = c * 64 + 16 * i + 4 * q;
    uint32_t val = 0;
    if (row < n_out && k < n_in) val = *reinterpret_cast<const uint32_t*>(src + row * n_in + k);
    reinterpret_cast<uint32_t*>(dst)[e] = val;
    // scales: 4 floats per (group, chunk, q); the i == 0 word of lanes n == 0 writes them
    if (n == 0 && i == 0) {
      float* out = dst_s + (gc * 4 + q) * 4;
      for (int s = 0; s < 4; ++s) {
        const int64_t srow = g * 8 + 2 * q + (s >> 1);
        const int64_t blk = c * 2 + (s & 1);
        out[s] = (srow < n_out && blk < n_blocks) ? src_s[srow * n_blocks + blk] : 0.0f;
      }
    }
  }
}

__global__ void pack_q4_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                               float* __restrict__ dst_s, int64_t n_out, int64_t n_in,
                               int64_t n_groups, int64_t n_chunks) {
  const float* src_s = reinterpret_cast<const float*>(src + n_out * (n_in / 2));
  const int64_t n_blocks = n_in / 32;
  const int64_t words = n_groups * n_chunks * 32 * 4;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < words;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int w = e & 3;
    const int lane = (e >> 2) & 31;
    const int64_t gc = e >> 7;
    const int64_t g = gc / n_chunks, c = gc % n_chunks;
    const int n = lane >> 2, q = lane & 3;
    const int64_t row = g * 8 + n;
    uint32_t val = 0;
    if (row < n_out) {
      for (int p = 0; p < 8; ++p) {
        const int sub = (p >> 1) & 1;
        const int j = ((p & 1) << 1) | (p >> 2);
        const int64_t k = c * 128 + 32 * w + 16 * sub + 4 * q + j;
        if (k < n_in) {
          const uint8_t byte = src[row * (n_in / 2) + k / 2];
          const uint32_t nib = (k & 1) ? (byte >> 4) : (byte & 0xF);
          val |= nib << (4 * p);
        }
      }
    }
    reinterpret_cast<uint32_t*>(dst)[e] = val;
    if (n == 0 && w == 0) {
      float* out = dst_s + (gc * 4 + q) * 8;
      for (int s = 0; s < 8; ++s) {
        const int64_t srow = g * 8 + 2 * q + (s >> 2);
        const int64_t blk = c * 4 + (s & 3);
        out[s] = (srow < n_out && blk < n_blocks) ? src_s[srow * n_blocks + blk] : 0.0f;
      }
    }
  }
}

// Element (r, k) of a packed weight as fp32: bf16 widened exactly, Q8/Q4 as
// fp32(d*q) -- the element decoders of the matmul kernels, then one multiply.
__device__ __forceinline__ float packed_element(int fmt, const uint8_t* __restrict__ wq,
                                                const float* __restrict__ ws, int64_t n_in_pad,
                                                int64_t n_chunks, int64_t r, int64_t k) {
  const int64_t g = r >> 3;
  const int n = (int)(r & 7);
  if (fmt == IL_BF16) {
    const uint16_t b = reinterpret_cast<const uint16_t*>(wq)[r * n_in_pad + k];
    return __uint_as_float((uint32_t)b << 16);
  }
  if (fmt == IL_Q8) {
    const int64_t c = k / 64;
    const int kk = (int)(k % 64);
    const int i = kk / 16, q = (kk % 16) / 4, j = kk % 4;
    const int lane = 4 * n + q;
    const uint32_t word = reinterpret_cast<const uint32_t*>(wq)[((g * n_chunks + c) * 32 + lane) * 4 + i];
    uint32_t p01, p23;
    q8_word_to_f16x2(word, p01, p23);
    const uint32_t pr = (j < 2) ? p01 : p23;
    const float qv = (j & 1) ? f16_hi(pr) : f16_lo(pr);
    const int qs = n >> 1, blk = kk / 32;
    const float d = ws[((g * n_chunks + c) * 4 + qs) * 4 + (n & 1) * 2 + blk];
    return __fmul_rn(d, qv);
  }
  const int64_t c = k / 128;
  const int kk = (int)(k % 128);
  const int w = kk / 32, sub = (kk % 32) / 16, q = (kk % 16) / 4, j = kk % 4;
  const int lane = 4 * n + q;
  const uint32_t word = reinterpret_cast<const uint32_t*>(wq)[((g * n_chunks + c) * 32 + lane) * 4 + w];
  const int p = sub * 2 + (j >> 1) + (j & 1) * 4;
  uint32_t prs[4];
  q4_word_to_f16x2(word, prs);
  const uint32_t pr = prs[p & 3];
  const float qv = (p >> 2) ? f16_hi(pr) : f16_lo(pr);
  const int qs = n >> 1;
  const float d = ws[((g * n_chunks + c) * 4 + qs) * 8 + (n & 1) * 4 + w];
  return __fmul_rn(d, qv);
}

// One thread per element of [n_out][n_in]; reads the packed layout back.
__global__ void dequant_kernel(int fmt, const uint8_t* __restrict__ wq, const float* __restrict__ ws,
                               int64_t n_out, int64_t n_in, int64_t n_in_pad, int64_t n_chunks,
                               float* __restrict__ out) {
  const int64_t total = n_out * n_in;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = e / n_in, k = e % n_in;
    out[e] = packed_element(fmt, wq, ws, n_in_pad, n_chunks, r, k);
  }
}

int grid_for(int64_t work) {
  int64_t g = (work + 255) / 256;
  if (g > 65536) g = 65536;
  if (g < 1) g = 1;
  return (int)g;
}

}  // namespace

cudaError_t launch_pack(const PackedWeight& w, const uint8_t* staging, cudaStream_t stream) {
  if (w.format == IL_BF16) {
    const int64_t work = w.n_out_pad * (w.n_in_pad / 8);
    pack_bf16_kernel<<<grid_for(work), 256, 0, stream>>>(
        reinterpret_cast<const uint16_t*>(staging), reinterpret_cast<uint16_t*>(w.quants), w.n_out,
        w.n_in, w.n_out_pad, w.n_in_pad);
  } else {
    const int64_t work = w.n_groups * w.n_chunks * 128;
    if (w.format == IL_Q8)
      pack_q8_kernel<<<grid_for(work), 256, 0, stream>>>(staging, w.quants, w.scales, w.n_out,
                                                         w.n_in, w.n_groups, w.n_chunks);
    else
      pack_q4_kernel<<<grid_for(work), 256, 0, stream>>>(staging, w.quants, w.scales, w.n_out,
                                                         w.n_in, w.n_groups, w.n_chunks);
  }
  return cudaGetLastError();
}

cudaError_t launch_dequant(const PackedWeight& w, float* out, cudaStream_t stream) {
  dequant_kernel<<<grid_for(w.n_out * w.n_in), 256, 0, stream>>>(
      w.format, w.quants, w.scales, w.n_out, w.n_in, w.n_in_pad, w.n_chunks, out);
  return cudaGetLastError();
}

}  // namespace il
