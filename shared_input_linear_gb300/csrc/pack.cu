// pack.cu -- upload-time repacking of a weight into its device layout
// (oxinfer src/gpu.rs, `Backend::upload`: prepare device state for one weight),
// and the dequantise hook that reads the packed layout back element by element.
//
// Q8 / Q4 weights become pair-major records (il_internal.cuh): record (p, c)
// holds the quants of groups 2p and 2p+1 for chunk c, then their scales.
// Q8 group chunk (8 rows x 64 columns, 512 bytes): lane L = 4n + q owns 16 bytes.
//   Byte 4i + j of the lane (i = 0..3 is the MMA slot, j = 0..3) holds column
//   16i + 4q + j of row n, stored biased (q + 128).  Slots 0,1 cover the chunk's
//   first 32-block, 2,3 the second, so every MMA stays inside one scale block.
// Q4 group chunk (8 rows x 128 columns, 512 bytes): lane L owns four 32-bit words;
//   word w covers the 32-block w of the chunk (MMA slots 2w and 2w+1).  Nibble
//   position p (bits 4p..4p+3) of the word holds column 32w + 16*sub + 4q + j of
//   row n with sub = (p >> 1) & 1 and j = ((p & 1) << 1) | (p >> 2).  Taking the
//   nibbles at bits s and s+16 (s = 0, 4, 8, 12) then yields the fp16x2 operand
//   pairs (j = 0,1) and (j = 2,3) of slot 2w, then of slot 2w+1.
// Scales of a group in a record: fp32 [8 rows][blocks of the chunk], row-major.
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

// One thread per 32-bit word of a record's quants (256 words a record), then one
// per scale: the quants of row 16p + 8h + n (h = group in the pair) and the
// scales of its blocks.
__global__ void pack_q8_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int64_t n_out,
                               int64_t n_in, int64_t n_pairs, int64_t n_chunks) {
  constexpr int RS = record_bytes(IL_Q8), SB = chunk_scale_bytes(IL_Q8), BL = blocks_per_chunk(IL_Q8);
  const float* src_s = reinterpret_cast<const float*>(src + n_out * n_in);
  const int64_t n_blocks = n_in / 32;
  const int64_t records = n_pairs * n_chunks;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < records * 256;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int i = e & 3;
    const int lane = (e >> 2) & 31;
    const int h = (e >> 7) & 1;
    const int64_t rec = e >> 8;  // pair * n_chunks + chunk
    const int64_t pr = rec / n_chunks, c = rec % n_chunks;
    const int n = lane >> 2, q = lane & 3;
    const int64_t row = pr * 16 + h * 8 + n;
    const int64_t k = c * 64 + 16 * i + 4 * q;
    uint32_t val = 0x80808080u;  // q = 0
    if (row < n_out && k < n_in) val = *reinterpret_cast<const uint32_t*>(src + row * n_in + k) ^ 0x80808080u;
    *reinterpret_cast<uint32_t*>(dst + rec * RS + h * 512 + lane * 16 + i * 4) = val;
  }
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < records * 16 * BL;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int b = (int)(e % BL);
    const int r16 = (int)((e / BL) & 15);  // row in the pair
    const int64_t rec = e / (16 * BL);
    const int64_t pr = rec / n_chunks, c = rec % n_chunks;
    const int64_t row = pr * 16 + r16, blk = c * BL + b;
    const float v = (row < n_out && blk < n_blocks) ? src_s[row * n_blocks + blk] : 0.0f;
    *reinterpret_cast<float*>(dst + rec * RS + 1024 + (r16 >> 3) * SB + ((r16 & 7) * BL + b) * 4) = v;
  }
}

__global__ void pack_q4_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int64_t n_out,
                               int64_t n_in, int64_t n_pairs, int64_t n_chunks) {
  constexpr int RS = record_bytes(IL_Q4), SB = chunk_scale_bytes(IL_Q4), BL = blocks_per_chunk(IL_Q4);
  const float* src_s = reinterpret_cast<const float*>(src + n_out * (n_in / 2));
  const int64_t n_blocks = n_in / 32;
  const int64_t records = n_pairs * n_chunks;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < records * 256;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int w = e & 3;
    const int lane = (e >> 2) & 31;
    const int h = (e >> 7) & 1;
    const int64_t rec = e >> 8;
    const int64_t pr = rec / n_chunks, c = rec % n_chunks;
    const int n = lane >> 2, q = lane & 3;
    const int64_t row = pr * 16 + h * 8 + n;
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
    *reinterpret_cast<uint32_t*>(dst + rec * RS + h * 512 + lane * 16 + w * 4) = val;
  }
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < records * 16 * BL;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int b = (int)(e % BL);
    const int r16 = (int)((e / BL) & 15);
    const int64_t rec = e / (16 * BL);
    const int64_t pr = rec / n_chunks, c = rec % n_chunks;
    const int64_t row = pr * 16 + r16, blk = c * BL + b;
    const float v = (row < n_out && blk < n_blocks) ? src_s[row * n_blocks + blk] : 0.0f;
    *reinterpret_cast<float*>(dst + rec * RS + 1024 + (r16 >> 3) * SB + ((r16 & 7) * BL + b) * 4) = v;
  }
}

// Element (r, k) of a packed weight as fp32: bf16 widened exactly, Q8/Q4 as
// fp32(d*q) -- the element decoders of the matmul kernels, then one multiply.
__device__ __forceinline__ float packed_element(int fmt, const uint8_t* __restrict__ wq, int64_t n_in_pad,
                                                int64_t n_chunks, int64_t r, int64_t k) {
  if (fmt == IL_BF16) {
    const uint16_t b = reinterpret_cast<const uint16_t*>(wq)[r * n_in_pad + k];
    return __uint_as_float((uint32_t)b << 16);
  }
  const int64_t pr = r >> 4;
  const int h = (int)((r >> 3) & 1), n = (int)(r & 7);
  if (fmt == IL_Q8) {
    const int64_t c = k / 64;
    const int kk = (int)(k % 64);
    const int i = kk / 16, q = (kk % 16) / 4, j = kk % 4;
    const uint8_t* rec = wq + (pr * n_chunks + c) * record_bytes(IL_Q8);
    const uint32_t word = *reinterpret_cast<const uint32_t*>(rec + h * 512 + (4 * n + q) * 16 + i * 4);
    uint32_t p01, p23;
    q8_word_to_f16x2(word, p01, p23);
    const uint32_t pr2 = (j < 2) ? p01 : p23;
    const float qv = (j & 1) ? f16_hi(pr2) : f16_lo(pr2);
    const float d = reinterpret_cast<const float*>(rec + 1024 + h * chunk_scale_bytes(IL_Q8))[n * 2 + kk / 32];
    return __fmul_rn(d, qv);
  }
  const int64_t c = k / 128;
  const int kk = (int)(k % 128);
  const int w = kk / 32, sub = (kk % 32) / 16, q = (kk % 16) / 4, j = kk % 4;
  const uint8_t* rec = wq + (pr * n_chunks + c) * record_bytes(IL_Q4);
  const uint32_t word = *reinterpret_cast<const uint32_t*>(rec + h * 512 + (4 * n + q) * 16 + w * 4);
  const int p = sub * 2 + (j >> 1) + (j & 1) * 4;
  uint32_t prs[4];
  q4_word_to_f16x2(word, prs);
  const uint32_t pr2 = prs[p & 3];
  const float qv = (p >> 2) ? f16_hi(pr2) : f16_lo(pr2);
  const float d = reinterpret_cast<const float*>(rec + 1024 + h * chunk_scale_bytes(IL_Q4))[n * 4 + w];
  return __fmul_rn(d, qv);
}

// One thread per element of [n_out][n_in]; reads the packed layout back.
__global__ void dequant_kernel(int fmt, const uint8_t* __restrict__ wq, int64_t n_out, int64_t n_in,
                               int64_t n_in_pad, int64_t n_chunks, float* __restrict__ out) {
  const int64_t total = n_out * n_in;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = e / n_in, k = e % n_in;
    out[e] = packed_element(fmt, wq, n_in_pad, n_chunks, r, k);
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
    const int64_t n_pairs = w.n_groups / 2;
    const int64_t work = n_pairs * w.n_chunks * 256;
    if (w.format == IL_Q8)
      pack_q8_kernel<<<grid_for(work), 256, 0, stream>>>(staging, w.quants, w.n_out, w.n_in, n_pairs, w.n_chunks);
    else
      pack_q4_kernel<<<grid_for(work), 256, 0, stream>>>(staging, w.quants, w.n_out, w.n_in, n_pairs, w.n_chunks);
  }
  return cudaGetLastError();
}

cudaError_t launch_dequant(const PackedWeight& w, float* out, cudaStream_t stream) {
  dequant_kernel<<<grid_for(w.n_out * w.n_in), 256, 0, stream>>>(w.format, w.quants, w.n_out, w.n_in,
                                                                  w.n_in_pad, w.n_chunks, out);
  return cudaGetLastError();
}

}  // namespace il
