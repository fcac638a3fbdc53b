// gemm.cu -- tensor-core path for large token counts: x cast once to bf16,
// then one persistent tcgen05 GEMM launch over every job of the batch.
//
// For each job j (oxinfer src/gpu.rs, struct `Job` / `Backend::matmul`):
//     y_j[t][o] = sum_k x_bf16[t][k] * W_j[o][k]      (fp32 accumulate)
//
// Tile: BM = 128 weight rows (MMA M) x BN tokens (MMA N) x BK = 64 columns per
// pipeline stage.  Both operands are K-major in HBM (W is [n_out][n_in], x is
// [t][n_in]) and arrive by TMA with the 128-byte swizzle that the tcgen05
// shared-memory descriptors read directly.  The accumulator lives in tensor
// memory (TMEM): 128 lanes = weight rows, BN columns = tokens, double
// buffered so the epilogue of one tile overlaps the MMAs of the next.  With
// TMEM lane = output column o, a warp's 32 lanes write 32 consecutive floats
// of y[t][.], so the epilogue stores are coalesced without a transpose.
//
// Warp roles (6 warps): 0 = TMA producer, 1 = TMEM allocator + MMA issuer,
// 2..5 = epilogue (warp w reads TMEM lanes 32*(w%4) .. +31).
//
// Q8 / Q4 weights (a mixed-input GEMM, 22 warps): the producer brings the packed
// quants and scales of 16 row groups (128 rows) x one chunk by TMA into a ring of
// raw stages; warps 6..21 turn them into the bf16 A tile of a pipeline stage,
// bf16(fp32(d*q)) with round to nearest even, written in the 128-byte swizzle
// the MMA reads.  The weight crosses HBM once, in its packed form.
// Tiles are taken round-robin by persistent CTAs; when the tiles cannot fill the
// SMs, each is split over K in two.  Where every unit gets its own CTA, the two
// slices of a tile run as the two CTAs of a cluster: each finishes half of the
// tile's tokens, taking the other slice's partial sums for that half from its
// peer through distributed shared memory.  Otherwise the slice that arrives last
// adds both partial tiles from a global workspace in slice order.
// Every mbarrier wait is bounded; a wait that gives up records an error code
// in the device status word, raises a CTA-wide abort flag and lets every role
// leave its loop; TMEM is always released before exit.
#include <cooperative_groups.h>
#include <cuda.h>

#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>

#include "il_internal.cuh"
#include "il_ptx.cuh"

namespace il {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;            // bf16 columns per stage: one 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kThreadsGemm = 192;  // 6 warps (bf16 weights)
constexpr int kXfWarps = 16;       // Q8/Q4: warps that dequantise raw stages into A tiles
constexpr int kThreadsQ = kThreadsGemm + 32 * kXfWarps;
constexpr int kRawStages = 3;
constexpr uint32_t kRawQuantBytes = 16 * 512;   // one chunk of 16 row groups
constexpr uint32_t kRawStageBytes = kRawQuantBytes + 16 * 8 * 4 * 4;  // + scales (Q4: 4 blocks a chunk)

__host__ __device__ constexpr int gemm_threads(int fmt) { return fmt == IL_BF16 ? kThreadsGemm : kThreadsQ; }
// fp32 scales per (row group, chunk): 8 rows x the chunk's 32-blocks
__host__ __device__ constexpr int scales_per_chunk(int fmt) { return 8 * blocks_per_chunk(fmt); }

constexpr int kMaxGemmJobs = 8;

struct GemmParams {  // CUtensorMap members give it their 64-byte (or larger) alignment
  CUtensorMap wmap[kMaxGemmJobs];  // bf16: W tiles; Q8/Q4: packed quants, 4D over the records (see make_quant_map)
  CUtensorMap smap[kMaxGemmJobs];  // Q8/Q4: packed scales, 4D over the records
  CUtensorMap xmap;
  float* y[kMaxGemmJobs];
  int n_out[kMaxGemmJobs];
  int tile_begin[kMaxGemmJobs + 1];  // prefix over jobs of m_tiles * n_tiles
  int n_jobs;
  int t;
  int n_tiles_n;
  int num_kb;
  int total_tiles;
  int splits;          // K slices per tile (split-K); units = total_tiles * splits
  int kb_per_split;
  float* ws;           // split-K partial tiles [tile][split][BN][BM] (splits > 1)
  unsigned* counters;  // split-K arrivals per tile, zero before the launch
  int stall_producer;  // failure-detection test: the producer never loads, so the MMA wait runs out
  unsigned* status;
  unsigned glu_mask;   // bit j: job j's rows interleave gate/up; y[j] is h = gelu(g) * u, n_out/2 wide
  int pair;            // split-K in two, one unit per CTA, the two slices of a tile the two CTAs of a
                       // cluster: partial sums exchanged through distributed shared memory (no ws)
};
static_assert(alignof(GemmParams) >= 64, "tensor maps must stay 64-byte aligned in the kernel parameters");
static_assert(sizeof(GemmParams) <= 4096, "kernel parameters must fit the classic 4 KB limit");

// ---- PTX wrappers (tcgen05) ---------------------------------------------------
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row swizzle atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFFu);        // start address
  d |= (uint64_t)1 << 16;                         // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;               // stride byte offset: next 8-row atom
  d |= (uint64_t)1 << 46;                         // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;                         // swizzle: 128 bytes
  return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "setp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void locate_tile(const GemmParams& p, int tile, int& job, int& mt, int& nt) {
  int j = p.n_jobs - 1;
  while (j > 0 && p.tile_begin[j] > tile) --j;
  const int local = tile - p.tile_begin[j];
  job = j;
  mt = local / p.n_tiles_n;
  nt = local - mt * p.n_tiles_n;
}

// Work unit -> (tile, K block range).
__device__ __forceinline__ void unit_range(const GemmParams& p, int unit, int& tile, int& split, int& kb0, int& kb1) {
  tile = unit / p.splits;
  split = unit - tile * p.splits;
  kb0 = split * p.kb_per_split;
  kb1 = min(p.num_kb, kb0 + p.kb_per_split);
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Status codes of the bounded waits (or-ed into the device status word).
constexpr unsigned kStProducer = 0x1;
constexpr unsigned kStMma = 0x2;
constexpr unsigned kStEpilogue = 0x4;
constexpr unsigned kStTransform = 0x8;

// Two fp32 values as one 64-bit register pair, and the packed fp32 operations
// of sm_100-class cores on them (one instruction for both lanes).
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2unpack(uint64_t r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t f2mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// bf16x2 (round to nearest even) of a pair.
__device__ __forceinline__ uint32_t f2bf16x2(uint64_t v) {
  float lo, hi;
  f2unpack(v, lo, hi);
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Dequantise one 16-byte unit of an A tile (row r, columns 8u .. 8u+7 of the
// k-block) from a raw stage: 8 consecutive columns of one row sit in two
// neighbouring lanes' words of the packed chunk (4 columns each) and share one
// 32-block scale.  half: which 64 columns of a Q4 chunk (128 columns) this k-block
// is.  Each value is bf16(fp32(d * q)): q exact in fp32, one rounded multiply,
// one round to bf16.  Q8: a byte permute puts the stored byte u = q + 128 under
// the exponent of 2^23 (the float 2^23 + u) and one packed subtract leaves q;
// Q4: the nibbles decode to exact fp16 and widen.
template <int FMT>
__device__ __forceinline__ uint4 dequant_unit(const uint32_t* __restrict__ qw, const float* __restrict__ sc, int r,
                                              int u, int half) {
  const int gl = r >> 3, n = r & 7;
  const int q0 = (u & 1) * 2;
  uint64_t qp[4];  // four pairs of q as fp32
  float d;
  if (FMT == IL_Q8) {
    const int base = gl * 128 + (4 * n + q0) * 4 + (u >> 1);
    const uint64_t bias = f2pack(8388736.0f, 8388736.0f);  // 2^23 + 128
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // lanes q0 and q0 + 1
      const uint32_t w = qw[base + 4 * h];
      qp[2 * h] = f2sub(f2pack(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540)),
                               __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7541))), bias);
      qp[2 * h + 1] = f2sub(f2pack(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7542)),
                                   __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7543))), bias);
    }
    d = sc[gl * 16 + n * 2 + (u >> 2)];
  } else {
    const int w = 2 * half + (u >> 2), sub = (u >> 1) & 1;
    const int base = gl * 128 + (4 * n + q0) * 4 + w;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t prs[4];
      q4_word_to_f16x2(qw[base + 4 * h], prs);
      const uint32_t p01 = sub ? prs[2] : prs[0], p23 = sub ? prs[3] : prs[1];  // no local-memory indexing
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&p01));
      const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&p23));
      qp[2 * h] = f2pack(a.x, a.y);
      qp[2 * h + 1] = f2pack(b.x, b.y);
    }
    d = sc[gl * 32 + n * 4 + w];
  }
  const uint64_t dd = f2pack(d, d);
  return make_uint4(f2bf16x2(f2mul(dd, qp[0])), f2bf16x2(f2mul(dd, qp[1])), f2bf16x2(f2mul(dd, qp[2])),
                    f2bf16x2(f2mul(dd, qp[3])));
}

// Gate/up epilogue of 32 token columns held by a lane pair: lanes 2i (gate row) and
// 2i+1 (up row) of output column i each finish 16 of the tokens, trading the other
// half with the partner (the even lane keeps r[0..15], the odd lane r[16..31]; tok0 is
// the lane's first token).  All 16 activations are computed before any store, so
// their latency chains overlap.  h: this column of the output (stride h_ld per
// token); store: the column lies inside the weight.
__device__ __forceinline__ void glu_store16(const uint32_t (&r)[32], bool odd, bool store, int tok0, int t,
                                            float* h, int h_ld) {
  float v[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float keep = __uint_as_float(odd ? r[j + 16] : r[j]);
    const float got = __shfl_xor_sync(0xffffffffu, __uint_as_float(odd ? r[j] : r[j + 16]), 1);
    v[j] = gelu_mul(odd ? got : keep, odd ? keep : got);
  }
  if (!store) return;
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if (tok0 + j < t) h[(int64_t)(tok0 + j) * h_ld] = v[j];
}

template <int BN, int FMT>
__global__ void __launch_bounds__(gemm_threads(FMT), 1) gemm_kernel(const __grid_constant__ GemmParams p) {
  constexpr bool kQ = FMT != IL_BF16;
  // tokens per round of the split-K fixup: 32 where registers allow (bf16: 6 warps)
  constexpr int kFix = kQ ? 16 : 32;
  constexpr uint32_t kABytes = kBM * kBK * 2;
  constexpr uint32_t kBBytes = BN * kBK * 2;
  constexpr uint32_t kStageBytes = kABytes + kBBytes;
  constexpr uint32_t kTmemCols = 2 * BN;  // two accumulators
  // Q4: one raw stage (a 128-column chunk) feeds two k-blocks
  constexpr int kKbPerRaw = FMT == IL_Q4 ? 2 : 1;
  constexpr uint32_t kRawTx = kRawQuantBytes + 16u * scales_per_chunk(FMT) * 4u;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tiles = smem;
  uint8_t* raw = smem + kStages * kStageBytes;  // Q8/Q4 only
  uint64_t* bars = reinterpret_cast<uint64_t*>(raw + (kQ ? kRawStages * kRawStageBytes : 0));
  uint64_t* full = bars;                // [kStages]
  uint64_t* empty = bars + kStages;     // [kStages]
  uint64_t* tfull = bars + 2 * kStages; // [2]
  uint64_t* tempty = tfull + 2;         // [2]
  uint64_t* raw_full = tempty + 2;      // [kRawStages]
  uint64_t* raw_empty = raw_full + kRawStages;  // [kRawStages]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(raw_empty + kRawStages);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      // Q8/Q4: the x tile's bytes plus one arrival per dequantising warp
      mbar_init(smem_u32(&full[s]), kQ ? 1 + kXfWarps : 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), 4);
    }
    for (int r = 0; r < kRawStages; ++r) {
      mbar_init(smem_u32(&raw_full[r]), 1);
      mbar_init(smem_u32(&raw_empty[r]), kXfWarps);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // set-up above overlaps the previous kernel; x (bf16 copy) and y need it finished
  grid_dep_wait();
  // split-K pair: the tile whose accumulator (buffer 0) this CTA's epilogue holds
  bool pair_ready = false;
  int pair_job = 0, pair_mt = 0, pair_nt = 0;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && !p.stall_producer) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.xmap)) : "memory");
      int stage = 0, rstage = 0;
      uint32_t phase = 0, rphase = 0;
      const int units = p.total_tiles * p.splits;
      bool ok = true;
      for (int unit = blockIdx.x; ok && unit < units && !*abort_flag; unit += gridDim.x) {
        int tile, split, kb0, kb1, job, mt, nt;
        unit_range(p, unit, tile, split, kb0, kb1);
        locate_tile(p, tile, job, mt, nt);
        const CUtensorMap* wm = &p.wmap[job];
        for (int kb = kb0; kb < kb1; ++kb) {
          if (kQ && kb % kKbPerRaw == 0) {
            // packed quants + scales of row groups 16*mt .. +15, chunk kb / kKbPerRaw
            if (!mbar_wait(smem_u32(&raw_empty[rstage]), rphase ^ 1, abort_flag, p.status, kStProducer)) {
              ok = false;
              break;
            }
            const uint32_t rb = smem_u32(&raw_full[rstage]);
            mbar_expect_tx(rb, kRawTx);
            const uint32_t r_dst = smem_u32(raw + rstage * kRawStageBytes);
            const int c = kb / kKbPerRaw;
            // 8 row pairs (16 groups) of chunk c: [pair][group][words] = 16 groups x 512 bytes
            tma_load_4d(r_dst, wm, 0, 0, c, mt * 8, rb);
            tma_load_4d(r_dst + kRawQuantBytes, &p.smap[job], 0, 0, c, mt * 8, rb);
            if (++rstage == kRawStages) {
              rstage = 0;
              rphase ^= 1;
            }
          }
          if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1, abort_flag, p.status, kStProducer)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&full[stage]);
          const uint32_t a_dst = smem_u32(tiles + stage * kStageBytes);
          if (kQ) {
            mbar_expect_tx(fb, kBBytes);
          } else {
            mbar_expect_tx(fb, kStageBytes);
            tma_load_2d(a_dst, wm, kb * kBK, mt * kBM, fb);
          }
          tma_load_2d(a_dst + kABytes, &p.xmap, kb * kBK, nt * BN, fb);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (kQ && warp >= 6) {
    // ------------------------------------------------------------ dequantise raw -> A tiles
    const int xt = threadIdx.x - 6 * 32;  // 0 .. 32 * kXfWarps - 1
    int stage = 0, rstage = 0;
    uint32_t phase = 0, rphase = 0;
    const int units = p.total_tiles * p.splits;
    bool ok = true;
    for (int unit = blockIdx.x; ok && unit < units && !*abort_flag; unit += gridDim.x) {
      int tile, split, kb0, kb1;
      unit_range(p, unit, tile, split, kb0, kb1);
      for (int kb = kb0; kb < kb1; ++kb) {
        if (kb % kKbPerRaw == 0 &&
            !mbar_wait(smem_u32(&raw_full[rstage]), rphase, abort_flag, p.status, kStTransform)) {
          ok = false;
          break;
        }
        if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1, abort_flag, p.status, kStTransform)) {
          ok = false;
          break;
        }
        const uint8_t* rs = raw + rstage * kRawStageBytes;
        const uint32_t* qw = reinterpret_cast<const uint32_t*>(rs);
        const float* sc = reinterpret_cast<const float*>(rs + kRawQuantBytes);
        uint8_t* a_tile = tiles + stage * kStageBytes;
        const int half = kb % kKbPerRaw;
#pragma unroll
        for (int it = 0; it < (kBM * 8) / (32 * kXfWarps); ++it) {
          // a warp covers 4 rows x 8 units: 512 contiguous bytes of the tile
          const int idx = it * (32 * kXfWarps) + xt;
          const int r = idx >> 3, u = idx & 7;
          const uint4 v = dequant_unit<FMT>(qw, sc, r, u, half);
          *reinterpret_cast<uint4*>(a_tile + r * 128 + ((u ^ (r & 7)) << 4)) = v;
        }
        // make the generic-proxy stores visible to the tensor core, then report
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&full[stage]));
          if (half == kKbPerRaw - 1) mbar_arrive(smem_u32(&raw_empty[rstage]));
        }
        if (half == kKbPerRaw - 1 && ++rstage == kRawStages) {
          rstage = 0;
          rphase ^= 1;
        }
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kBM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      const int units = p.total_tiles * p.splits;
      for (int unit = blockIdx.x; unit < units && !*abort_flag; unit += gridDim.x, ++it) {
        int tile, split, kb0, kb1;
        unit_range(p, unit, tile, split, kb0, kb1);
        const int acc = it & 1;
        const uint32_t aphase = (it >> 1) & 1;
        if (!mbar_wait(smem_u32(&tempty[acc]), aphase ^ 1, abort_flag, p.status, kStMma)) break;
        tc_fence_after();
        const uint32_t tmem_d = tmem_base + acc * BN;
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(smem_u32(&full[stage]), phase, abort_flag, p.status, kStMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(tiles + stage * kStageBytes);
          const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            // advance 16 columns = 32 bytes inside the 128-byte swizzle row
            tc_mma(tmem_d, smem_desc_sw128(a_addr + 32 * k), smem_desc_sw128(b_addr + 32 * k), idesc,
                   (kb > kb0 || k > 0) ? 1u : 0u);
          }
          tc_commit(smem_u32(&empty[stage]));  // frees the stage when these MMAs finish
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(smem_u32(&tfull[acc]));  // accumulator ready for the epilogue
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    volatile int* last_flag = abort_flag + 1;
    const int units = p.total_tiles * p.splits;
    int it = 0;
    for (int unit = blockIdx.x; unit < units; unit += gridDim.x, ++it) {
      int tile, split, kb0, kb1;
      unit_range(p, unit, tile, split, kb0, kb1);
      const int acc = it & 1;
      const uint32_t aphase = (it >> 1) & 1;
      if (!mbar_wait(smem_u32(&tfull[acc]), aphase, abort_flag, p.status, kStEpilogue)) break;
      tc_fence_after();
      int job, mt, nt;
      locate_tile(p, tile, job, mt, nt);
      if (p.pair) {  // the CTA's only unit: finished below, with the peer
        pair_ready = true;
        pair_job = job;
        pair_mt = mt;
        pair_nt = nt;
        break;
      }
      const int n_out = p.n_out[job];
      float* y = p.y[job];
      const bool glu = (p.glu_mask >> job) & 1u;  // uniform over the CTA
      const int lrow = quarter * 32 + lane;
      const int row = mt * kBM + lrow;
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
      float* part = p.splits > 1 ? p.ws + ((size_t)tile * p.splits + split) * (BN * kBM) : nullptr;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(taddr + c0, r);
        if (part != nullptr) {
          // partial tile stored [token][row]: each store of the warp is 128 contiguous bytes
#pragma unroll
          for (int j = 0; j < 32; ++j) part[(c0 + j) * kBM + lrow] = __uint_as_float(r[j]);
        } else if (glu) {
          // lanes 2i (gate) and 2i+1 (up) hold output column row / 2 for 32 tokens and
          // split them: the even lane finishes tokens 0..15, the odd lane 16..31, each
          // trading the other half with its partner.  n_out is even, so a pair is
          // either wholly inside or wholly outside the weight.
          const bool odd = lane & 1;
          glu_store16(r, odd, row < n_out, nt * BN + c0 + (odd ? 16 : 0), p.t, y + (row >> 1), n_out >> 1);
        } else {
          const int tok0 = nt * BN + c0;
          if (row < n_out) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int tok = tok0 + j;
              if (tok < p.t) y[(int64_t)tok * n_out + row] = __uint_as_float(r[j]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));  // accumulator free for the MMA warp
      if (part != nullptr) {
        // split-K: the last K slice to arrive sums every slice's partial, in slice order
        __threadfence();
        epi_bar();
        if (warp == 2 && lane == 0) {
          const unsigned old = atomicAdd(p.counters + tile, 1u);
          const int last = old == (unsigned)(p.splits - 1);
          if (last) {
            p.counters[tile] = 0u;
            __threadfence();
          }
          *last_flag = last;
        }
        epi_bar();
        // *last_flag is the same for the whole CTA, so the warps stay converged for
        // the gate/up exchange below
        if (*last_flag && (glu || row < n_out)) {
          const float* base = p.ws + (size_t)tile * p.splits * (BN * kBM) + lrow;
          const int ntok = min(BN, p.t - nt * BN);
#pragma unroll 1
          for (int c0 = 0; c0 < ntok; c0 += kFix) {
            // kFix tokens at a time, both slices' loads issued before any add (the plan
            // splits at most in two), summed in slice order (a partial tile holds every
            // token column, so reads past ntok stay inside it)
            float v[kFix], w1[kFix];
            const float* src0 = base + (size_t)c0 * kBM;
            const float* src1 = base + ((size_t)BN + c0) * kBM;
#pragma unroll
            for (int j = 0; j < kFix; ++j) v[j] = __ldcg(src0 + j * kBM);
            if (p.splits > 1) {
#pragma unroll
              for (int j = 0; j < kFix; ++j) w1[j] = __ldcg(src1 + j * kBM);
#pragma unroll
              for (int j = 0; j < kFix; ++j) v[j] += w1[j];
            }
            if (glu) {
              // as in the direct store: the even lane finishes the first half, the odd the second
              const bool odd = lane & 1;
              float h[kFix / 2];
#pragma unroll
              for (int j = 0; j < kFix / 2; ++j) {  // every activation first: independent chains
                const float keep = odd ? v[j + kFix / 2] : v[j];
                const float got = __shfl_xor_sync(0xffffffffu, odd ? v[j] : v[j + kFix / 2], 1);
                h[j] = gelu_mul(odd ? got : keep, odd ? keep : got);
              }
#pragma unroll
              for (int j = 0; j < kFix / 2; ++j) {
                const int c = c0 + j + (odd ? kFix / 2 : 0);
                if (row < n_out && c < ntok) y[(int64_t)(nt * BN + c) * (n_out >> 1) + (row >> 1)] = h[j];
              }
            } else {
#pragma unroll
              for (int j = 0; j < kFix; ++j)
                if (c0 + j < ntok) y[(int64_t)(nt * BN + c0 + j) * n_out + row] = v[j];
            }
          }
        }
      }
    }
  }

  if (p.pair) {
    // ---- split-K pair.  Every thread of both CTAs takes part in the two cluster
    // barriers (after a wait that gave up too, so the peer never waits for ever).
    // Rank r finishes tokens [r * BN/2, (r + 1) * BN/2) of the tile: it receives the
    // other slice's partial sums of those tokens into its (now idle) pipeline memory,
    // [BN/2 tokens][kBM rows] fp32, and sends its own partial sums of the peer's half.
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    float* xbuf = reinterpret_cast<float*>(tiles);
    const int quarter = warp & 3;
    const int lrow = quarter * 32 + lane;
    const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16);  // accumulator buffer 0
    // (1) both CTAs' MMAs are complete and every load consumed: the pipeline memory is free
    __syncwarp();
    tc_fence_before();
    cluster.sync();
    tc_fence_after();
    // uniform over the warp (the abort flag is read once per lane)
    const bool live = __all_sync(0xffffffffu, warp >= 2 && warp < 6 && pair_ready && !*abort_flag);
    if (live) {
      float* peer = cluster.map_shared_rank(xbuf, rank ^ 1);
      const int c_peer = (rank ^ 1) * (BN / 2);
#pragma unroll 1
      for (int c = 0; c < BN / 2; c += 32) {
        uint32_t r[32];
        tmem_ld32(taddr + c_peer + c, r);
#pragma unroll
        for (int j = 0; j < 32; ++j) peer[(c + j) * kBM + lrow] = __uint_as_float(r[j]);
      }
    }
    // (2) the peer's partial sums of this CTA's half have landed
    __syncwarp();
    tc_fence_before();
    cluster.sync();
    tc_fence_after();
    if (live) {
      const int n_out = p.n_out[pair_job];
      float* y = p.y[pair_job];
      const bool glu = (p.glu_mask >> pair_job) & 1u;
      const int row = pair_mt * kBM + lrow;
      const int c_own = rank * (BN / 2);
#pragma unroll 1
      for (int c = 0; c < BN / 2; c += 32) {
        uint32_t r[32];
        tmem_ld32(taddr + c_own + c, r);
        // slice 0 + slice 1 (two operands: the same sum on either rank)
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) + xbuf[(c + j) * kBM + lrow]);
        const int tok0 = pair_nt * BN + c_own + c;
        if (glu) {
          // as in the direct store: lanes 2i / 2i+1 (gate / up) trade halves of the 32 tokens
          const bool odd = lane & 1;
          glu_store16(r, odd, row < n_out, tok0 + (odd ? 16 : 0), p.t, y + (row >> 1), n_out >> 1);
        } else if (row < n_out) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int tok = tok0 + j;
            if (tok < p.t) y[(int64_t)tok * n_out + row] = __uint_as_float(r[j]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  grid_dep_launch();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                 : "memory");
  }
}

// x fp32 [t][n_in] -> bf16 [t][n_in_pad] (round to nearest even), 0 in the padding.
// One resident wave of CTAs; each thread keeps kCastUnroll vectors of 8 columns in
// flight (all loads issued before the first store).
constexpr int kCastUnroll = 4;
__global__ void __launch_bounds__(256) cast_bf16_kernel(const float* __restrict__ x, int64_t t, int64_t n_in,
                                                        int64_t n_in_pad, __nv_bfloat16* __restrict__ out) {
  const int64_t per_row = n_in_pad / 8;
  const int64_t total = t * per_row;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  grid_dep_wait();
  for (int64_t v0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; v0 < total; v0 += kCastUnroll * stride) {
    float4 a[kCastUnroll], b[kCastUnroll];
#pragma unroll
    for (int u = 0; u < kCastUnroll; ++u) {
      const int64_t v = v0 + u * stride;
      a[u] = b[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (v < total) {
        const int64_t r = v / per_row;
        const int64_t k = (v - r * per_row) * 8;
        if (k < n_in) {  // n_in is a multiple of 8: the 8 columns are all inside or all outside
          a[u] = __ldcs(reinterpret_cast<const float4*>(x + r * n_in + k));
          b[u] = __ldcs(reinterpret_cast<const float4*>(x + r * n_in + k + 4));
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kCastUnroll; ++u) {
      const int64_t v = v0 + u * stride;
      if (v >= total) break;
      const int64_t r = v / per_row;
      const int64_t k = (v - r * per_row) * 8;
      __nv_bfloat162 h0 = __floats2bfloat162_rn(a[u].x, a[u].y), h1 = __floats2bfloat162_rn(a[u].z, a[u].w);
      __nv_bfloat162 h2 = __floats2bfloat162_rn(b[u].x, b[u].y), h3 = __floats2bfloat162_rn(b[u].z, b[u].w);
      uint4 o;
      o.x = *reinterpret_cast<uint32_t*>(&h0);
      o.y = *reinterpret_cast<uint32_t*>(&h1);
      o.z = *reinterpret_cast<uint32_t*>(&h2);
      o.w = *reinterpret_cast<uint32_t*>(&h3);
      *reinterpret_cast<uint4*>(out + r * n_in_pad + k) = o;
    }
  }
  grid_dep_launch();
}

// ---- host: tensor maps through the driver entry point (no libcuda link) -----
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  // looked up once; a function-local static is initialised thread-safely
  static const EncodeTiledFn fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(ptr);
    return static_cast<EncodeTiledFn>(nullptr);
  }();
  return fn;
}

// Host-side fault injection for the failure tests: with
// IL_FAULT_TENSOR_MAP_FAIL_AFTER=k the (k+1)-th tensor-map encoding of the
// process fails (as an encoding the driver rejects would).
std::atomic<long> g_map_count{0};
bool map_fault() {
  const char* env = getenv("IL_FAULT_TENSOR_MAP_FAIL_AFTER");
  if (env == nullptr || *env == '\0') return false;
  return g_map_count.fetch_add(1) >= strtol(env, nullptr, 10);
}

// bf16 [rows][cols] row-major with row pitch `pitch` elements; box = box_cols x box_rows.
bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t pitch, uint32_t box_cols,
              uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || map_fault()) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {pitch * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int grid_cast(int64_t work, int num_sms) {
  // 8 CTAs of 256 threads fill an SM; more than one wave only adds scheduling
  int64_t g = (work + 255) / 256;
  const int64_t wave = 8LL * (num_sms > 0 ? num_sms : 1);
  if (g > wave) g = wave;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t prepare_cast_bf16(const float* x, int64_t t, int64_t n_in, int64_t n_in_pad, __nv_bfloat16* out,
                              int num_sms, Launch* L) {
  *L = Launch();
  L->fn = reinterpret_cast<const void*>(cast_bf16_kernel);
  L->grid = dim3(grid_cast(t * (n_in_pad / 8), num_sms));
  L->block = dim3(256);
  if (kUsePdl) L->allow_early_start();
  if (!L->set_args(x, t, n_in, n_in_pad, out)) return cudaErrorMemoryAllocation;
  return cudaSuccess;
}

namespace {

constexpr int kBN = 256;

// Split-K workspace: a fixed block of per-tile arrival counters, then the partial
// tiles.  The counters must read zero before every launch (the last arriver of
// each tile puts its counter back); at a fixed size they never share bytes with
// the partials of any launch, whatever its tile count, and a grown workspace
// starts zeroed.  Launches with more tiles than counters do not split.
constexpr int kMaxSplitTiles = kSplitCounters;
constexpr size_t kCounterBytes = kSplitCounterBytes;

struct Plan {
  int splits, kb_per_split, total_tiles;
};

// Split-K only when the tiles alone leave SMs idle: estimated time = the larger
// of the tensor work spread over whole waves of units and the weight stream
// (which splitting does not shorten), plus the traffic of writing and summing
// partials.
Plan plan_launch(int64_t t, int64_t n_in_pad, const GemmJob* jobs, int nj, int num_sms, bool allow_split) {
  Plan pl{1, 0, 0};
  const int n_tiles_n = (int)((t + kBN - 1) / kBN);
  const int num_kb = (int)(n_in_pad / kBK);
  int64_t sum_n_out = 0;
  for (int j = 0; j < nj; ++j) {
    pl.total_tiles += (int)((jobs[j].w->n_out + kBM - 1) / kBM) * n_tiles_n;
    sum_n_out += jobs[j].w->n_out;
  }
  pl.kb_per_split = num_kb;
  if (!allow_split || pl.total_tiles > kMaxSplitTiles) return pl;
  const double flops = 2.0 * (double)t * (double)n_in_pad * (double)sum_n_out;
  const int fmt = jobs[0].w->format;
  const double wbytes = (double)sum_n_out * (double)n_in_pad * (fmt == IL_BF16 ? 2.0 : fmt == IL_Q8 ? 1.125 : 0.625);
  // a Q4 chunk spans two k-blocks: slices start on a chunk
  const int align = fmt == IL_Q4 ? 2 : 1;
  double best = 1e30;
  // at most two slices: the partial-tile traffic of more slices costs more than it saves
  for (int s = 1; s <= 2 && s <= num_kb / 4; ++s) {
    const int kbps = ((num_kb + s - 1) / s + align - 1) / align * align;
    const int se = (num_kb + kbps - 1) / kbps;
    const int64_t units = (int64_t)pl.total_tiles * se;
    const int64_t waves = (units + num_sms - 1) / num_sms;
    const double eff = (double)units / ((double)waves * num_sms);
    const double est = std::max(flops / (1.5e15 * eff), wbytes / 6.0e12) +
                       (se > 1 ? 2.0 * se * (double)t * sum_n_out * 4.0 / 5.0e12 : 0.0);
    if (est < best * 0.97 || s == 1) {
      if (s == 1 || est < best * 0.97) {
        best = est;
        pl.splits = se;
        pl.kb_per_split = kbps;
      }
    }
  }
  return pl;
}



}  // namespace

size_t gemm_workspace_bytes(int64_t t, int64_t n_in_pad, const GemmJob* jobs, int n_jobs, int num_sms) {
  size_t need = 0;
  for (int j0 = 0; j0 < n_jobs; j0 += kMaxGemmJobs) {
    const int nj = n_jobs - j0 < kMaxGemmJobs ? n_jobs - j0 : kMaxGemmJobs;
    const Plan pl = plan_launch(t, n_in_pad, jobs + j0, nj, num_sms, true);
    if (pl.splits > 1) {
      const size_t b = kCounterBytes + (size_t)pl.total_tiles * pl.splits * kBN * kBM * sizeof(float);
      if (b > need) need = b;
    }
  }
  return need;
}

namespace {

// Packed Q8/Q4 records (il_internal.cuh) seen as 4D tensors.  Quants: 32-bit
// words, dims {128 words of a group's chunk, 2 groups of a pair, n_chunks,
// n_pairs}; a box of {128, 2, 1, 8} is one chunk of 16 groups (128 rows), laid
// out in shared memory as [group][128 words].  Scales: fp32, dims {8 rows x
// blocks, 2 groups, n_chunks, n_pairs} starting 1024 bytes into the first
// record; box {8 * blocks, 2, 1, 8} gives [group][rows x blocks].
bool make_quant_map(CUtensorMap* m, const PackedWeight& w) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || map_fault()) return false;
  const cuuint64_t rs = (cuuint64_t)record_bytes(w.format);
  const cuuint64_t dims[4] = {128, 2, (cuuint64_t)w.n_chunks, (cuuint64_t)(w.n_groups / 2)};
  const cuuint64_t strides[3] = {512, rs, rs * (cuuint64_t)w.n_chunks};
  const cuuint32_t box[4] = {128, 2, 1, 8};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, w.quants, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_scale_map(CUtensorMap* m, const PackedWeight& w) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || map_fault()) return false;
  const int spc = scales_per_chunk(w.format);
  const cuuint64_t rs = (cuuint64_t)record_bytes(w.format);
  const cuuint64_t dims[4] = {(cuuint64_t)spc, 2, (cuuint64_t)w.n_chunks, (cuuint64_t)(w.n_groups / 2)};
  const cuuint64_t strides[3] = {(cuuint64_t)chunk_scale_bytes(w.format), rs, rs * (cuuint64_t)w.n_chunks};
  const cuuint32_t box[4] = {(cuuint32_t)spc, 2, 1, 8};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, w.quants + 2 * kChunkBytes, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Clusters of two CTAs of gemm_kernel<BN, FMT> that fit on the device at once
// (once per device; 0 if the query fails).
template <int BN, int FMT>
int pair_clusters(int dev, size_t smem) {
  static std::mutex mu;
  static std::map<int, int> cache;
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) return it->second;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeClusterDimension;
  a.val.clusterDim.x = 2;
  a.val.clusterDim.y = 1;
  a.val.clusterDim.z = 1;
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(gemm_threads(FMT));
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = &a;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_kernel<BN, FMT>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cache[dev] = n;
  return n;
}

template <int FMT>
cudaError_t prepare_gemm_fmt(const __nv_bfloat16* xb, int64_t t, int64_t n_in_pad, const GemmJob* jobs, int n_jobs,
                             int num_sms, unsigned* status, void* ws, size_t ws_bytes, std::vector<Launch>* out) {
  constexpr int BN = kBN;
  constexpr size_t smem = (size_t)kStages * (kBM * kBK * 2 + BN * kBK * 2) +
                          (FMT == IL_BF16 ? 0 : (size_t)kRawStages * kRawStageBytes) + 1024 + 256;
  static std::atomic<unsigned long long> attr_set{0};  // one bit per device (setting it twice is harmless)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !(attr_set.load() & (1ull << dev))) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<BN, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set.fetch_or(1ull << dev);
  }
  for (int j0 = 0; j0 < n_jobs; j0 += kMaxGemmJobs) {
    const int nj = n_jobs - j0 < kMaxGemmJobs ? n_jobs - j0 : kMaxGemmJobs;
    // without a workspace a split survives only in the CTA-pair form below
    Plan pl = plan_launch(t, n_in_pad, jobs + j0, nj, num_sms, true);
    const size_t cbytes = kCounterBytes;
    // a split in two whose units all fit at once as CTA pairs needs no workspace.
    // IL_TEST_SPLIT_WORKSPACE=1 (tests only) sends every split through the global
    // workspace, the path taken when the pairs do not fit, so that it stays covered.
    const char* force_ws = getenv("IL_TEST_SPLIT_WORKSPACE");
    const bool pair = !(force_ws != nullptr && force_ws[0] == '1') && pl.splits == 2 &&
                      pl.total_tiles <= pair_clusters<BN, FMT>(dev, smem);
    if (!pair && pl.splits > 1 &&
        cbytes + (size_t)pl.total_tiles * pl.splits * BN * kBM * sizeof(float) > ws_bytes) {
      pl.splits = 1;
      pl.kb_per_split = (int)(n_in_pad / kBK);
    }
    GemmParams p;
    memset(&p, 0, sizeof p);
    p.n_jobs = nj;
    p.t = (int)t;
    p.n_tiles_n = (int)((t + BN - 1) / BN);
    p.num_kb = (int)(n_in_pad / kBK);
    p.splits = pl.splits;
    p.kb_per_split = pl.kb_per_split;
    p.status = status;
    p.pair = pair ? 1 : 0;
    if (pl.splits > 1 && !pair) {
      // counters are zero when the workspace is created and the last arriver of
      // every tile puts its counter back to zero (see kCounterBytes)
      p.counters = static_cast<unsigned*>(ws);
      p.ws = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + cbytes);
    }
    // IL_TEST_STALL_TMA_PRODUCER=1 (failure-detection tests only): the TMA
    // producer issues nothing, the MMA warp's bounded wait gives up after about
    // a second, the kernel records IL_ERR_DEVICE_TIMEOUT's code and exits cleanly.
    const char* stall = getenv("IL_TEST_STALL_TMA_PRODUCER");
    p.stall_producer = (stall != nullptr && stall[0] == '1') ? 1 : 0;
    if (!make_map(&p.xmap, xb, (uint64_t)n_in_pad, (uint64_t)t, (uint64_t)n_in_pad, kBK, BN))
      return cudaErrorInvalidValue;
    int tiles = 0;
    for (int j = 0; j < nj; ++j) {
      const PackedWeight& w = *jobs[j0 + j].w;
      if (w.format != FMT || w.n_in_pad != n_in_pad) return cudaErrorInvalidValue;
      const bool mapped = FMT == IL_BF16
                              ? make_map(&p.wmap[j], w.quants, (uint64_t)w.n_in_pad, (uint64_t)w.n_out_pad,
                                         (uint64_t)w.n_in_pad, kBK, kBM)
                              : make_quant_map(&p.wmap[j], w) && make_scale_map(&p.smap[j], w);
      if (!mapped) return cudaErrorInvalidValue;
      p.y[j] = jobs[j0 + j].y;
      p.n_out[j] = (int)w.n_out;
      if (w.glu) p.glu_mask |= 1u << j;
      p.tile_begin[j] = tiles;
      tiles += (int)((w.n_out + kBM - 1) / kBM) * p.n_tiles_n;
    }
    p.tile_begin[nj] = tiles;
    p.total_tiles = tiles;
    const int units = tiles * p.splits;
    Launch L;
    L.fn = reinterpret_cast<const void*>(gemm_kernel<BN, FMT>);
    // pair: one CTA per unit, a tile's two slices in one cluster (units 2i, 2i + 1)
    L.grid = dim3(pair ? units : (units < num_sms ? units : num_sms));
    L.block = dim3(gemm_threads(FMT));
    L.smem = smem;
    if (pair) L.set_cluster(2);
    if (kUsePdl) L.allow_early_start();
    if (!L.set_args(p)) return cudaErrorMemoryAllocation;
    out->push_back(L);
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t prepare_gemm(int fmt, const __nv_bfloat16* xb, int64_t t, int64_t n_in_pad, const GemmJob* jobs,
                         int n_jobs, int num_sms, unsigned* status, void* ws, size_t ws_bytes,
                         std::vector<Launch>* out) {
  if (fmt == IL_BF16)
    return prepare_gemm_fmt<IL_BF16>(xb, t, n_in_pad, jobs, n_jobs, num_sms, status, ws, ws_bytes, out);
  if (fmt == IL_Q8)
    return prepare_gemm_fmt<IL_Q8>(xb, t, n_in_pad, jobs, n_jobs, num_sms, status, ws, ws_bytes, out);
  if (fmt == IL_Q4)
    return prepare_gemm_fmt<IL_Q4>(xb, t, n_in_pad, jobs, n_jobs, num_sms, status, ws, ws_bytes, out);
  return cudaErrorInvalidValue;
}

}  // namespace il
