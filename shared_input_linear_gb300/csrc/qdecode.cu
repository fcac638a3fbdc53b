// qdecode.cu -- grouped decode kernel for Q8 / Q4 weights at small token counts
// (t <= 8 per launch).
//
// For every job j of a batch over one shared x (oxinfer 0.0.0 src/gpu.rs, struct
// `Job` and `Backend::matmul`):
//     y_j[t][o] = sum_i x[t][i] * fp32(d_j[o][i / 32] * q_j[o][i])
//
// Design (GB300):
//  * Rows of all jobs are cut into tiles of 16 (a pair of 8-row groups); every
//    (tile, chunk) of a packed Q8/Q4 weight is one contiguous record of quants and
//    scales (il_internal.cuh).  Each weight byte crosses HBM once.
//  * The records stream into shared memory by bulk copies (cp.async.bulk,
//    completion counted on an mbarrier).  Every warp owns a ring of stages of up
//    to four consecutive records of one tile (one copy each) and refills a stage
//    as soon as it has consumed it, so the bytes in flight per SM are set by the
//    ring depth, not by registers; the first stages are issued before the launch
//    waits for the previous kernel.
//  * Dot products run on the tensor cores (mma.m16n8k16, fp16 in, fp32
//    accumulate).  The 16 weight rows of a record are the A operand, decoded in
//    registers to exact fp16 integers (one byte permute or LOP3 and one fp16x2
//    subtract per pair); x is the B operand, its tokens the 8 columns: for t <= 4
//    an fp16 high part and the fp16 rounding of the remainder side by side (about
//    22 significant bits), for t <= 8 the fp16 value (11 bits); one MMA per 16
//    columns of K either way.  The fp32 scale of each 32-block multiplies the
//    fp32 partial of that block.
//  * x is staged once per CTA in shared memory, already as B fragments (zeros for
//    tokens >= t), scaled per token by a power of two so that fp16 holds it
//    (undone on the partial sums); the loads, the token maxima and the conversion
//    take one pass over L2 from registers.
//  * Work: the CTAs of a K split of C take the same tiles with different K
//    slices; inside a CTA, warps stand in a grid of wr row tiles x wk parts of
//    the slice (wk = 1: a warp owns whole tiles).  There is no CTA-wide barrier
//    in the stream: the last of the wk warps to finish a tile adds the parts'
//    partial sums in part order (a generation count per partial-sum slot keeps a
//    warp that runs ahead from overwriting a slot before it is summed), and with
//    C > 1 the last CTA to finish a tile adds the C slices' sums from a global
//    workspace in slice order.  Results are deterministic.
//  * Every wait is bounded; a wait that gives up records a code in the device
//    status word, raises a CTA abort flag, and the warps finish without waiting,
//    then drain the copies still in flight.
#include <map>
#include <mutex>
#include <tuple>

#include "il_internal.cuh"
#include "il_ptx.cuh"

namespace il {
namespace {

constexpr int kQWarps = 16;
constexpr int kQThreads = kQWarps * 32;
constexpr int kMaxQStages = 12;
// Records per ring stage (consecutive chunks of one tile, one bulk copy): larger
// copies mean fewer copy operations in flight per SM for the same bytes.
constexpr int kMaxStageRecords = 4;
// Relative cost the planner gives each extra CTA a tile's K is split over (the
// cross-CTA sum through the workspace ends every split tile).
constexpr double kSplitPenalty = 0.03;
// Relative cost per halving of the warps that own a tile (wk doubling).
constexpr double kWarpSplitPenalty = 0.95;
constexpr int kSlotRounds = 2;          // partial-sum slots per warp row: rounds a warp may run ahead
constexpr int kXRegUnits = 6;          // x units per thread staged in one pass from registers
constexpr int kMaxQTokens = 16;        // tokens of one launch (two groups of 8 MMA columns)
constexpr unsigned kStQDecode = 0x10;   // a wait for a record gave up
constexpr unsigned kStQSlot = 0x20;     // a wait for a free partial-sum slot gave up

struct QJob {
  const uint8_t* w;    // records
  float* y;            // [t][n_out], or h [t][n_out / 2] when glu
  int32_t n_out;       // packed rows
  int32_t tile_begin;  // first global 16-row tile of this job
  int32_t glu;
  int32_t pad_;
};

struct QParams {
  const float* x;
  unsigned* status;
  float* ws;           // C > 1: per (tile, slice) sums [tile][C][TT][16]
  unsigned* counters;  // C > 1: arrivals per tile, zero before the launch
  int t;               // tokens of this launch, 1..8
  int x_row_stride;    // elements between token rows of x
  int n_in;
  int n_chunks;        // chunks over n_in_pad
  int slices;          // C: CTAs that split K for one tile
  int cps;             // chunks per slice
  int wr, wk;          // warp grid: wr row tiles at a time x wk parts of the slice (wr * wk = 16)
  int stages;          // ring stages per warp
  int spr;             // records per stage: consecutive chunks of one tile, one bulk copy
  int total_tiles;
  int n_jobs;
  int stall;           // failure-detection test: issue no copies, so the waits run out
  QJob jobs[kMaxDecodeJobs];
};

template <int FMT>
struct QF {
  static constexpr int CK = chunk_k(FMT);            // columns per chunk
  static constexpr int SLOTS = CK / 16;              // 16-column MMA slots per chunk
  static constexpr int BLOCKS = blocks_per_chunk(FMT);
  static constexpr int SB = chunk_scale_bytes(FMT);  // scale bytes of one group in a record
  static constexpr int RS = record_bytes(FMT);
};

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The same with a zero accumulator in: d = a * b (the zero register is shared, so
// no per-call initialisation).
__device__ __forceinline__ void mma_f16_first(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

// Arrival on a per-tile counter in global memory with acquire-release ordering at
// GPU scope: this thread's earlier writes (and those ordered before it by a warp
// barrier) are visible before the increment; the last arriver sees every other
// arriver's writes.  Returns the value before the increment.
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* addr, unsigned v) {
  unsigned old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<const uint32_t*>(&h); }

__device__ __forceinline__ int find_tile_job(const QParams& p, int tile) {
  int j = p.n_jobs - 1;
  while (j > 0 && p.jobs[j].tile_begin > tile) --j;
  return j;
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// x exponent of a token from the bits of its largest |x| (a non-negative float):
// 2^-e brings that value into [2^13, 2^14); e stays in [-126, 114] so both powers
// of two are normal floats.
__device__ __forceinline__ int x_exponent(unsigned max_bits) {
  const float m = __uint_as_float(max_bits);
  return m > 0.f ? max(-126, min(114, ilogbf(m) - 13)) : 0;
}

// One record: 16 rows x CK columns against the x fragments of that chunk (xc:
// this lane's 16 bytes of the chunk's first unit; one unit of 512 bytes per pair
// of slots and token group -- TT = 16 has two groups of 8 token columns, the same
// decoded A fragments feeding one MMA per group).
// acc[grp]: (row g, token col 2q), (row g, col 2q+1), (row g+8, col 2q), (row g+8, col 2q+1).
template <int FMT, int TT>
__device__ __forceinline__ void consume_record(const uint8_t* st, int lane, int g, const uint8_t* xc,
                                               float (&acc)[TT == 16 ? 2 : 1][4]) {
  constexpr int NG = TT == 16 ? 2 : 1;
  using F = QF<FMT>;
  const uint4 q0 = *reinterpret_cast<const uint4*>(st + lane * 16);        // rows 0..7 (group 2p)
  const uint4 q1 = *reinterpret_cast<const uint4*>(st + 512 + lane * 16);  // rows 8..15 (group 2p+1)
  float d0[F::BLOCKS], d1[F::BLOCKS];
  if (FMT == IL_Q8) {
    const float2 a = *reinterpret_cast<const float2*>(st + 1024 + g * 8);
    const float2 b = *reinterpret_cast<const float2*>(st + 1024 + F::SB + g * 8);
    d0[0] = a.x; d0[1 % F::BLOCKS] = a.y;
    d1[0] = b.x; d1[1 % F::BLOCKS] = b.y;
  } else {
    const float4 a = *reinterpret_cast<const float4*>(st + 1024 + g * 16);
    const float4 b = *reinterpret_cast<const float4*>(st + 1024 + F::SB + g * 16);
    d0[0] = a.x; d0[1 % F::BLOCKS] = a.y; d0[2 % F::BLOCKS] = a.z; d0[3 % F::BLOCKS] = a.w;
    d1[0] = b.x; d1[1 % F::BLOCKS] = b.y; d1[2 % F::BLOCKS] = b.z; d1[3 % F::BLOCKS] = b.w;
  }
#pragma unroll
  for (int b = 0; b < F::BLOCKS; ++b) {
    uint32_t A0[4], A1[4];  // slots 2b and 2b+1: {row g k-pair lo, row g+8 lo, row g hi, row g+8 hi}
    if (FMT == IL_Q8) {
      uint32_t p01, p23, r01, r23;
      q8_word_to_f16x2(word_of(q0, 2 * b), p01, p23);
      q8_word_to_f16x2(word_of(q1, 2 * b), r01, r23);
      A0[0] = p01; A0[1] = r01; A0[2] = p23; A0[3] = r23;
      q8_word_to_f16x2(word_of(q0, 2 * b + 1), p01, p23);
      q8_word_to_f16x2(word_of(q1, 2 * b + 1), r01, r23);
      A1[0] = p01; A1[1] = r01; A1[2] = p23; A1[3] = r23;
    } else {
      uint32_t pa[4], pb[4];
      q4_word_to_f16x2(word_of(q0, b), pa);
      q4_word_to_f16x2(word_of(q1, b), pb);
      A0[0] = pa[0]; A0[1] = pb[0]; A0[2] = pa[1]; A0[3] = pb[1];
      A1[0] = pa[2]; A1[1] = pb[2]; A1[2] = pa[3]; A1[3] = pb[3];
    }
#pragma unroll
    for (int grp = 0; grp < NG; ++grp) {
      // B fragments of slots 2b and 2b+1 for this token group: one 16-byte load,
      // one MMA per slot
      const uint4 u = *reinterpret_cast<const uint4*>(xc + (b * NG + grp) * 512);
      float t4[4];
      mma_f16_first(t4, A0, u.x, u.y);
      mma_f16(t4, A1, u.z, u.w);
      acc[grp][0] = fmaf(d0[b], t4[0], acc[grp][0]);
      acc[grp][1] = fmaf(d0[b], t4[1], acc[grp][1]);
      acc[grp][2] = fmaf(d1[b], t4[2], acc[grp][2]);
      acc[grp][3] = fmaf(d1[b], t4[3], acc[grp][3]);
    }
  }
}

// Stores one summed value -- token tk, row `row` of `tile` -- into its job's y.
// Called by every lane of the warp (the gate/up pairing reads the neighbouring
// row's sum from the next lane).
__device__ __forceinline__ void store_item(const QParams& p, const QJob& jb, int tile, float v, int row, int tk) {
  const float up = __shfl_down_sync(0xffffffffu, v, 1);  // row + 1 of the same token
  if (tk >= p.t) return;
  const int r = (tile - jb.tile_begin) * 16 + row;
  if (r >= jb.n_out) return;
  if (jb.glu) {
    // rows 2i and 2i+1 are gate and up of output column i
    if ((row & 1) == 0) jb.y[(size_t)tk * (jb.n_out >> 1) + (r >> 1)] = gelu_mul(v, up);
  } else {
    jb.y[(size_t)tk * jb.n_out + r] = v;
  }
}

template <int FMT, int TT>
__global__ void __launch_bounds__(kQThreads, 1) qdecode_kernel(const __grid_constant__ QParams p) {
  using F = QF<FMT>;
  constexpr int RS = F::RS;
  constexpr int NG = TT == 16 ? 2 : 1;  // token groups of 8 columns
  constexpr int XL = 8 * NG;            // bytes of one lane's B fragments per slot
  constexpr int NI = TT / 2;            // summed items per lane: TT tokens x 16 rows over 32 lanes
  extern __shared__ __align__(128) uint8_t smem[];

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane >> 2;  // A rows g and g+8 of the tile; B column (token slot)
  const int q = lane & 3;

  const int rank = blockIdx.x % p.slices;
  const int stream = blockIdx.x / p.slices;
  const int nstreams = gridDim.x / p.slices;
  const int D = p.stages;
  const int wr_i = warp / p.wk, wk_i = warp - (warp / p.wk) * p.wk;
  // this CTA's K slice and this warp's even share of it (chunk indices from cb)
  const int cb = rank * p.cps;
  const int ns = max(0, min(p.cps, p.n_chunks - cb));
  const int c0 = (wk_i * ns) / p.wk;
  const int cnt = ((wk_i + 1) * ns) / p.wk - c0;
  const int tg_total = (p.total_tiles + p.wr - 1) / p.wr;
  const int rounds = stream < tg_total ? (tg_total - stream + nstreams - 1) / nstreams : 0;

  // shared memory: x fragments | rings | partial sums | slot counts | barriers
  constexpr int XCHUNK = F::SLOTS * 32 * XL;  // bytes of x fragments per chunk
  const size_t xs_bytes = (size_t)p.cps * XCHUNK;
  uint8_t* xs = smem;
  const int SB_ = p.spr * RS;  // bytes per ring stage
  uint8_t* ring = smem + xs_bytes + (size_t)warp * D * SB_;
  float* part = reinterpret_cast<float*>(smem + xs_bytes + (size_t)kQWarps * D * SB_);  // [NB][16 warps][TT][16]
  int* cnt_s = reinterpret_cast<int*>(part + kSlotRounds * kQWarps * TT * 16);           // [NB][16 rows of warps]
  int* gen_s = cnt_s + kSlotRounds * kQWarps;                                            // [NB][16]
  uint64_t* bars = reinterpret_cast<uint64_t*>(gen_s + kSlotRounds * kQWarps) + warp * kMaxQStages;
  unsigned* tok_max = reinterpret_cast<unsigned*>(reinterpret_cast<uint64_t*>(gen_s + kSlotRounds * kQWarps) +
                                                  kQWarps * kMaxQStages);
  float* tok_scale = reinterpret_cast<float*>(tok_max + kMaxQTokens);  // 2^-e(tok): x into fp16 range
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tok_scale + kMaxQTokens);

  if (lane == 0)
    for (int s = 0; s < D; ++s) mbar_init(smem_u32(&bars[s]), 1);
  if (threadIdx.x < kSlotRounds * kQWarps) {
    cnt_s[threadIdx.x] = 0;
    gen_s[threadIdx.x] = 0;
  }
  if (threadIdx.x < kMaxQTokens) tok_max[threadIdx.x] = 0u;
  if (threadIdx.x == 0) *abort_flag = 0;
  if (lane == 0) mbar_init_fence();
  __syncthreads();

  // ---- load cursor (lane 0): this warp's records in consumption order, (round,
  // chunk) with the chunk fastest; a row slot whose tile lies past the last one
  // has no records (only the last rounds can).
  int l_round = 0, l_cc = 0, l_stage = 0, issued = 0;
  const uint8_t* l_src = nullptr;
  const uint64_t policy = policy_evict_first();
  auto tile_records = [&](int round) -> const uint8_t* {
    if (round >= rounds) return nullptr;
    const int tile = (stream + round * nstreams) * p.wr + wr_i;
    if (tile >= p.total_tiles) return nullptr;
    const QJob& jb = p.jobs[find_tile_job(p, tile)];
    return jb.w + ((size_t)(tile - jb.tile_begin) * p.n_chunks + cb + c0) * RS;
  };
  if (lane == 0 && cnt > 0) l_src = tile_records(0);
  auto issue_next = [&]() {
    if (l_src == nullptr) return;
    const int nr = min(p.spr, cnt - l_cc);
    const uint32_t bar = smem_u32(&bars[l_stage]);
    mbar_expect_tx(bar, nr * RS);
    if (!p.stall)
      bulk_g2s_hint(smem_u32(ring + (size_t)l_stage * SB_), l_src + (size_t)l_cc * RS, nr * RS, bar, policy);
    ++issued;
    if (++l_stage == D) l_stage = 0;
    l_cc += nr;
    if (l_cc == cnt) {
      l_cc = 0;
      l_src = tile_records(++l_round);
    }
  };
  // Weights do not depend on the previous kernel: start streaming before waiting for it.
  if (lane == 0)
    for (int s = 0; s < D; ++s) issue_next();
  grid_dep_wait();
  // the next kernel may now be scheduled; it waits for this one before touching x or y
  grid_dep_launch();

  // ---- x of this CTA's slice as B fragments, token by token scaled by 2^-e(tok)
  // so that its largest |x| in the slice lies in [2^13, 2^14).  Per chunk, one
  // unit of 512 bytes per pair of slots, lane L's 16 bytes at 16 L holding its B
  // fragment of both slots: TT = 8, the fp16 of token L/4; TT = 4, the fp16 high
  // part (L/4 < 4) or the fp16 rounding of the remainder (L/4 >= 4) of token
  // (L/4) % 4; TT = 16, two units per pair of slots (tokens 0-7, then 8-15), the
  // fp16 of token 8 * group + L/4.  Lanes of tokens >= t hold zeros.  Thread i
  // always serves lane i % 32 of units of one group, so it sees a single token.
  constexpr int kSlotsPerUnit = 2;
  const int n_el = ns * (F::SLOTS / kSlotsPerUnit) * NG * 32;
  const int my_tk = TT == 16 ? (((threadIdx.x >> 5) & 1) << 3) + (lane >> 2)
                             : (TT == 8 ? (lane >> 2) : ((lane >> 2) & 3));
  const bool my_low = TT == 4 && (lane >> 2) >= 4;
  auto load_unit = [&](int e, float4 (&v)[kSlotsPerUnit]) {
    const int unit = (e >> 5) / NG;  // pair of slots
#pragma unroll
    for (int h = 0; h < kSlotsPerUnit; ++h) {
      const int col = cb * F::CK + 16 * (unit * kSlotsPerUnit + h) + 4 * (lane & 3);
      v[h] = (e < n_el && my_tk < p.t && col < p.n_in)
                 ? __ldg(reinterpret_cast<const float4*>(p.x + (size_t)my_tk * p.x_row_stride + col))
                 : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  auto store_unit = [&](int e, const float4 (&v)[kSlotsPerUnit], float xsc) {
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (my_tk < p.t) {
#pragma unroll
      for (int h = 0; h < kSlotsPerUnit; ++h) {
        const float4 x4 = v[h];
        const __half2 h01 = __floats2half2_rn(x4.x * xsc, x4.y * xsc);
        const __half2 h23 = __floats2half2_rn(x4.z * xsc, x4.w * xsc);
        const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
        const __half2 l01 = __floats2half2_rn(x4.x * xsc - f01.x, x4.y * xsc - f01.y);
        const __half2 l23 = __floats2half2_rn(x4.z * xsc - f23.x, x4.w * xsc - f23.y);
        w[2 * h] = my_low ? h2_bits(l01) : h2_bits(h01);
        w[2 * h + 1] = my_low ? h2_bits(l23) : h2_bits(h23);
      }
    }
    *reinterpret_cast<uint4*>(xs + (size_t)(e >> 5) * 512 + lane * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  };
  // the token's largest |x| over this warp's lanes of that token -> tok_max
  auto fold_max = [&](float m) {
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (TT == 4) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
    if ((lane & 3) == 0 && (TT != 4 || lane < 16) && m > 0.f)
      atomicMax(&tok_max[my_tk], __float_as_uint(m));  // non-negative: bits order as values
  };
  auto amax4 = [](const float4& a) { return fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))); };
  if (n_el <= kXRegUnits * kQThreads) {
    // one pass over global memory: every unit of this thread in registers (all
    // loads in flight at once: x comes from L2 behind the weight stream), the
    // token maxima, then the conversion from registers
    float4 v[kXRegUnits][kSlotsPerUnit];
    float m = 0.f;
#pragma unroll
    for (int u = 0; u < kXRegUnits; ++u) load_unit(threadIdx.x + u * kQThreads, v[u]);
#pragma unroll
    for (int u = 0; u < kXRegUnits; ++u) m = fmaxf(m, fmaxf(amax4(v[u][0]), amax4(v[u][1])));
    fold_max(m);
    __syncthreads();
    if (threadIdx.x < kMaxQTokens) tok_scale[threadIdx.x] = ldexpf(1.0f, -x_exponent(tok_max[threadIdx.x]));
    __syncthreads();
    const float xsc = tok_scale[my_tk];
#pragma unroll
    for (int u = 0; u < kXRegUnits; ++u)
      if (threadIdx.x + u * kQThreads < n_el) store_unit(threadIdx.x + u * kQThreads, v[u], xsc);
  } else {
    // larger slices: the maxima in a first pass, the conversion in a second
    // (loads issued kUnroll units at a time)
    constexpr int kUnroll = 4;
    float m = 0.f;
    for (int e0 = threadIdx.x; e0 < n_el; e0 += kUnroll * kQThreads) {
      float4 v[kUnroll][kSlotsPerUnit];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) load_unit(e0 + u * kQThreads, v[u]);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) m = fmaxf(m, fmaxf(amax4(v[u][0]), amax4(v[u][1])));
    }
    fold_max(m);
    __syncthreads();
    if (threadIdx.x < kMaxQTokens) tok_scale[threadIdx.x] = ldexpf(1.0f, -x_exponent(tok_max[threadIdx.x]));
    __syncthreads();
    const float xsc = tok_scale[my_tk];
    for (int e0 = threadIdx.x; e0 < n_el; e0 += kUnroll * kQThreads) {
      float4 v[kUnroll][kSlotsPerUnit];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) load_unit(e0 + u * kQThreads, v[u]);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (e0 + u * kQThreads < n_el) store_unit(e0 + u * kQThreads, v[u], xsc);
    }
  }
  __syncthreads();
  const uint8_t* xlane = xs + lane * 16;
  // scale back of the partials: this lane's D columns are tokens 2q and 2q+1 of
  // each token group (for t <= 4, lanes q < 2 after folding the low-part columns in)
  const int tq0 = TT == 4 ? 2 * (q & 1) : 2 * q;
  float ys[NG][2];
#pragma unroll
  for (int grp = 0; grp < NG; ++grp) {
    ys[grp][0] = ldexpf(1.0f, x_exponent(tok_max[8 * grp + tq0]));
    ys[grp][1] = ldexpf(1.0f, x_exponent(tok_max[8 * grp + tq0 + 1]));
  }

  int c_stage = 0;
  uint32_t c_phase = 0;
  int consumed = 0;
  bool ok = true;
  auto wait_stage = [&](int st_i, uint32_t ph) {
    return __all_sync(0xffffffffu, mbar_wait_sleep(smem_u32(&bars[st_i]), ph, abort_flag, p.status, kStQDecode));
  };
  for (int r = 0; r < rounds; ++r) {
    const int tile = (stream + r * nstreams) * p.wr + wr_i;
    if (tile >= p.total_tiles) break;  // same for the whole row of warps, and for every later round
    float acc[NG][4];
#pragma unroll
    for (int grp = 0; grp < NG; ++grp) acc[grp][0] = acc[grp][1] = acc[grp][2] = acc[grp][3] = 0.f;
    const uint8_t* xcc = xlane + (size_t)c0 * XCHUNK;
    // one stage at a time: up to spr consecutive chunks of this tile, one wait and
    // one refill for all of them
    for (int cc = 0; cc < cnt && ok; cc += p.spr) {
      const int nr = min(p.spr, cnt - cc);
      ok = wait_stage(c_stage, c_phase);
      if (!ok) break;
      const uint8_t* st = ring + (size_t)c_stage * SB_;
      consume_record<FMT, TT>(st, lane, g, xcc, acc);
#pragma unroll
      for (int i = 1; i < kMaxStageRecords; ++i)
        if (i < nr) consume_record<FMT, TT>(st + i * RS, lane, g, xcc + i * XCHUNK, acc);
      xcc += (size_t)nr * XCHUNK;
      ++consumed;
      // every lane's reads of this stage are done before the copy that refills it
      __syncwarp();
      if (lane == 0) issue_next();
      if (++c_stage == D) {
        c_stage = 0;
        c_phase ^= 1;
      }
    }
    if (TT == 4) {
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[0][k] += __shfl_xor_sync(0xffffffffu, acc[0][k], 2);  // high + low columns
    }
    // ---- this warp's partial -> its slot, once the slot's previous use is summed
    const int sr = r % kSlotRounds;
    const int slot = sr * kQWarps + wr_i;
    if (r >= kSlotRounds) {
      const int want = r / kSlotRounds;
      volatile int* gs = gen_s + slot;
      if (*gs < want) {
        const long long start = clock64();
        while (*gs < want) {
          if (*abort_flag) break;
          if ((unsigned long long)(clock64() - start) > kWaitLimitCycles) {
            *abort_flag = 1;
            atomicOr(p.status, kStQSlot);
            break;
          }
          __nanosleep(64);
        }
      }
      __threadfence_block();
    }
    float* pw = part + (size_t)((sr * kQWarps + warp) * TT) * 16;
    if (TT != 4 || q < 2) {
#pragma unroll
      for (int grp = 0; grp < NG; ++grp) {
        const int tk = 8 * grp + tq0;
        pw[tk * 16 + g] = acc[grp][0] * ys[grp][0];
        pw[(tk + 1) * 16 + g] = acc[grp][1] * ys[grp][1];
        pw[tk * 16 + g + 8] = acc[grp][2] * ys[grp][0];
        pw[(tk + 1) * 16 + g + 8] = acc[grp][3] * ys[grp][1];
      }
    }
    __syncwarp();
    int last = 1;
    if (p.wk > 1) {
      if (lane == 0) {
        __threadfence_block();
        last = atomicAdd(&cnt_s[slot], 1) == p.wk - 1;
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (!last) continue;
      __threadfence_block();
    }
    // ---- the last of the tile's wk parts: sum them in part order, (token, row)
    // items with rows fastest
    const float* pr = part + (size_t)((sr * kQWarps + wr_i * p.wk) * TT) * 16;
    float v[NI];
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int e = lane + 32 * i;
      if (p.wk == 1) {  // the warp's own partial (uniform over the grid)
        v[i] = pr[e];
      } else {
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < kQWarps; ++k)
          if (k < p.wk) s += pr[(size_t)k * TT * 16 + e];
        v[i] = s;
      }
    }
    __syncwarp();
    if (lane == 0) {
      if (p.wk > 1) cnt_s[slot] = 0;
      __threadfence_block();
      atomicAdd(&gen_s[slot], 1);  // the slot may be written again
    }
    if (p.slices > 1) {
      // ---- then over the C slices, through the global workspace: the last CTA to
      // arrive adds them in slice order (one thread fences for the warp, around the
      // warp-wide stores and loads)
      float* wsp = p.ws + ((size_t)tile * p.slices + rank) * TT * 16;
#pragma unroll
      for (int i = 0; i < NI; ++i) __stcg(wsp + lane + 32 * i, v[i]);
      __syncwarp();
      int lastc = 0;
      if (lane == 0) lastc = atom_add_acq_rel_gpu(p.counters + tile, 1u) == (unsigned)(p.slices - 1);
      if (!__shfl_sync(0xffffffffu, lastc, 0)) continue;
      const float* wt = p.ws + (size_t)tile * p.slices * TT * 16;
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        float s = 0.f;
        for (int c = 0; c < p.slices; ++c) s += __ldcg(wt + (size_t)c * TT * 16 + lane + 32 * i);
        v[i] = s;
      }
      if (lane == 0) p.counters[tile] = 0u;  // zero again for the next launch
    }
    const QJob& jb = p.jobs[find_tile_job(p, tile)];
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int e = lane + 32 * i;
      store_item(p, jb, tile, v[i], e & 15, e >> 4);
    }
  }
  // after a wait gave up: let the copies this warp still has in flight land
  // before the CTA's shared memory is released
  if (!ok && lane == 0 && !p.stall) {
    int s = c_stage;
    uint32_t ph = c_phase;
    for (int k = consumed; k < issued; ++k) {
      mbar_wait_for(smem_u32(&bars[s]), ph, kWaitLimitCycles / 8);
      if (++s == D) {
        s = 0;
        ph ^= 1;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// host side: plan + launch
// ---------------------------------------------------------------------------
using QKernelFn = void (*)(QParams);

QKernelFn select_q(int fmt, int TT) {
  if (fmt == IL_Q8)
    return TT == 16 ? qdecode_kernel<IL_Q8, 16> : (TT == 8 ? qdecode_kernel<IL_Q8, 8> : qdecode_kernel<IL_Q8, 4>);
  if (fmt == IL_Q4)
    return TT == 16 ? qdecode_kernel<IL_Q4, 16> : (TT == 8 ? qdecode_kernel<IL_Q4, 8> : qdecode_kernel<IL_Q4, 4>);
  return nullptr;
}

// Token columns of the kernel instance for t tokens: 4 (high and low parts side
// by side), 8, or 16 (two groups of 8).
int q_tt(int t) { return t <= 4 ? 4 : (t <= 8 ? 8 : 16); }

size_t q_x_bytes(int fmt, int t, int cps) {
  return (size_t)cps * (chunk_k(fmt) / 16) * 32 * 8 * (q_tt(t) == 16 ? 2 : 1);
}

// Shared memory besides the x fragments and the rings.
size_t q_fixed_bytes(int TT) {
  return (size_t)kSlotRounds * kQWarps * TT * 16 * sizeof(float) + 2 * (size_t)kSlotRounds * kQWarps * sizeof(int) +
         (size_t)kQWarps * kMaxQStages * 8 + kMaxQTokens * sizeof(unsigned) + kMaxQTokens * sizeof(float) + 16;
}

// Dynamic shared memory a CTA may take, once per device (the kernels' attribute
// is raised to it on first use).
int q_smem_limit(int dev) {
  static std::mutex mu;
  static std::map<int, int> limit;
  std::lock_guard<std::mutex> lk(mu);
  auto it = limit.find(dev);
  if (it != limit.end()) return it->second;
  int optin = 0;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
  for (int fmt = IL_Q8; fmt <= IL_Q4; ++fmt)
    for (int TT = 4; TT <= 16; TT *= 2)
      if (cudaFuncSetAttribute(select_q(fmt, TT), cudaFuncAttributeMaxDynamicSharedMemorySize, optin) != cudaSuccess)
        return 0;
  limit[dev] = optin;
  return optin;
}

struct QPlan {
  int C = 0, cps = 0, wr = 0, wk = 0, stages = 0, spr = 1, streams = 0;
  size_t smem = 0, ws_bytes = 0;
};

// The launch plan: K split over C CTAs, the warp grid (wr row tiles x wk parts),
// the ring depth that fills the shared memory left by the x fragments.  Scored
// by how evenly whole rounds of tile groups fill the SMs (a part-full last round
// idles SMs), by how many warps a round keeps busy, and by the records a warp
// streams per round (each round ends with a partial sum).  ws_room: split
// workspace available (SIZE_MAX: any).
bool plan_q(int fmt, int t, int n_chunks, int total_tiles, int num_sms, int smem_limit, size_t ws_room, QPlan* out) {
  const int TT = q_tt(t);
  const double work = (double)total_tiles * n_chunks;
  double best = -1.0;
  // with tiles for many rounds on every SM, a K split evens nothing out and only
  // adds the cross-CTA sum to every tile: keep C = 1 whenever its x fits
  const bool many_tiles = total_tiles >= 4 * num_sms * kQWarps;
  const bool unsplit_fits = q_x_bytes(fmt, t, n_chunks) + q_fixed_bytes(TT) +
                                2 * (size_t)kQWarps * record_bytes(fmt) <= (size_t)smem_limit;
  for (int c = 1; c <= 8 && c <= n_chunks; ++c) {
    if (c > 1 && many_tiles && unsplit_fits) break;
    const int cps = (n_chunks + c - 1) / c;
    if ((n_chunks + cps - 1) / cps != c) continue;
    size_t ws = 0;
    if (c > 1) {
      if (total_tiles > kSplitCounters) continue;
      ws = kSplitCounterBytes + (size_t)total_tiles * c * TT * 16 * sizeof(float);
      if (ws > ws_room) continue;
    }
    const size_t fixed = q_x_bytes(fmt, t, cps) + q_fixed_bytes(TT);
    if (fixed >= (size_t)smem_limit) continue;
    const int streams = num_sms / c;
    for (int spr = kMaxStageRecords; spr >= 1; spr /= 2) {
      int stages = (int)(((size_t)smem_limit - fixed) / ((size_t)kQWarps * spr * record_bytes(fmt)));
      if (stages > kMaxQStages) stages = kMaxQStages;
      if (stages < 2) continue;
      for (int wk = kQWarps; wk >= 1; wk /= 2) {
        const int wr = kQWarps / wk;
        const int cpw = (cps + wk - 1) / wk;
        const int tg = (total_tiles + wr - 1) / wr;
        const int used = tg < streams ? tg : streams;
        const int rounds = (tg + used - 1) / used;
        const double eff = work / ((double)num_sms * rounds * wr * cps);
        const int busy = (cps < wk ? cps : wk) * wr;  // warps with records in a full round
        // measured: copies of one record stream at about 0.7 of four-record copies
        const int per_copy = cpw < spr ? cpw : spr;
        const double copy = per_copy >= 4 ? 1.0 : (per_copy == 3 ? 0.96 : (per_copy == 2 ? 0.88 : 0.72));
        // measured: warps that split a tile sum partials every round (gate+up Q8 t = 1
        // with wk = 2 instead of 1: 23.5 -> 29.2 us)
        double split_warps = 1.0;
        for (int w = wk; w > 1; w /= 2) split_warps *= kWarpSplitPenalty;
        const double score = eff * (1.0 - kSplitPenalty * (c - 1)) * (busy >= 8 ? 1.0 : busy / 8.0) *
                             cpw / (cpw + 0.5) * copy * split_warps;
        if (score > best) {
          best = score;
          out->C = c;
          out->cps = cps;
          out->wr = wr;
          out->wk = wk;
          out->stages = stages;
          out->spr = spr;
          out->streams = used;
          out->smem = fixed + (size_t)kQWarps * stages * spr * record_bytes(fmt);
          out->ws_bytes = ws;
        }
      }
    }
  }
  return best > 0.0;
}

// plan_q is a pure function of its arguments (t only through its instance TT); a
// call of a shape seen before on this thread reuses the plan.
bool plan_q_memo(int fmt, int t, int n_chunks, int total_tiles, int num_sms, int smem_limit, size_t ws_room,
                 QPlan* out) {
  using Key = std::tuple<int, int, int, int, int, int, size_t>;
  thread_local std::map<Key, std::pair<bool, QPlan>> memo;
  const Key key{fmt, q_tt(t), n_chunks, total_tiles, num_sms, smem_limit, ws_room};
  auto it = memo.find(key);
  if (it == memo.end()) {
    if (memo.size() >= 512) memo.clear();
    QPlan pl;
    const bool ok = plan_q(fmt, t, n_chunks, total_tiles, num_sms, smem_limit, ws_room, &pl);
    it = memo.emplace(key, std::make_pair(ok, pl)).first;
  }
  *out = it->second.second;
  return it->second.first;
}

}  // namespace

size_t qdecode_workspace_bytes(int fmt, const DecodeParams& d, int num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const int limit = q_smem_limit(dev);
  QPlan pl;
  if (limit <= 0 || !plan_q_memo(fmt, d.t, d.n_chunks, d.total_groups / 2, num_sms, limit, SIZE_MAX, &pl)) return 0;
  return pl.ws_bytes;
}

cudaError_t prepare_qdecode(int fmt, const DecodeParams& d, int num_sms, unsigned* status, void* ws, size_t ws_bytes,
                            Launch* out) {
  if (fmt != IL_Q8 && fmt != IL_Q4) return cudaErrorInvalidValue;
  if (d.t < 1 || d.t > kMaxQTokens || d.n_jobs < 1 || d.n_jobs > kMaxDecodeJobs || (d.total_groups & 1)) return cudaErrorInvalidValue;
  const int TT = q_tt(d.t);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int limit = q_smem_limit(dev);
  if (limit <= 0) return cudaErrorInvalidValue;
  QPlan pl;
  if (!plan_q_memo(fmt, d.t, d.n_chunks, d.total_groups / 2, num_sms, limit, ws != nullptr ? ws_bytes : 0, &pl))
    return cudaErrorInvalidValue;

  QParams p;
  memset(&p, 0, sizeof p);
  p.x = d.x;
  p.status = status;
  if (pl.C > 1) {
    p.counters = static_cast<unsigned*>(ws);
    p.ws = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kSplitCounterBytes);
  }
  p.t = d.t;
  p.x_row_stride = d.x_row_stride;
  p.n_in = d.n_in;
  p.n_chunks = d.n_chunks;
  p.slices = pl.C;
  p.cps = pl.cps;
  p.wr = pl.wr;
  p.wk = pl.wk;
  p.stages = pl.stages;
  p.spr = pl.spr;
  p.total_tiles = d.total_groups / 2;
  p.n_jobs = d.n_jobs;
  for (int j = 0; j < d.n_jobs; ++j) {
    if (d.jobs[j].group_begin & 1) return cudaErrorInvalidValue;
    p.jobs[j].w = d.jobs[j].w;
    p.jobs[j].y = d.jobs[j].y;
    p.jobs[j].n_out = d.jobs[j].n_out;
    p.jobs[j].tile_begin = d.jobs[j].group_begin / 2;
    p.jobs[j].glu = d.jobs[j].glu;
  }
  const char* stall = getenv("IL_TEST_STALL_TMA_PRODUCER");
  p.stall = (stall != nullptr && stall[0] == '1') ? 1 : 0;

  Launch& L = *out;
  L = Launch();
  L.fn = reinterpret_cast<const void*>(select_q(fmt, TT));
  L.grid = dim3(pl.streams * pl.C);
  L.block = dim3(kQThreads);
  L.smem = pl.smem;
  // one CTA per SM at most: an early start behind the previous kernel takes
  // SMs as they free up and streams this batch's weights meanwhile
  if (kUsePdl) L.allow_early_start();
  if (!L.set_args(p)) return cudaErrorMemoryAllocation;
  return cudaSuccess;
}

}  // namespace il
