// Grouped W8A8 GEMMs of the prefill path on the 5th-generation tensor cores (tcgen05).
//
// One persistent kernel runs every (expert group, 128-row weight tile, token tile) work item
// of a layer: the gate/up GEMM with a fused SiLU(gate)*up epilogue, or the down GEMM whose
// epilogue adds every row's router-weighted output into the layer output y. This is the
// concatenated-expert computation of the page "Qwen3.6-35B-A3B Linux v1.0.4: ~2.7s fixed
// per-request TTFT ...", section "The fix (concatenated-expert dispatch)": one launch per
// operator and layer instead of one per expert, gate and up concatenated along the weight
// dimension, one GLU region over all experts.
//
// Orientation: the weights are the MMA's M operand (128 rows per tile) and an expert's tokens
// its N operand (N = the tile's row count rounded up to 16, at most the token tile TN <= 192;
// an expert's rows are split into equal tiles), so an expert with 162 tokens costs one
// 176-wide tile. The accumulator holds weight rows in TMEM lanes and tokens in columns. Gate
// and up rows are interleaved in pairs (row 2i = gate channel i, row 2i+1 = up channel i), so
// SiLU(gate)*up is formed by one lane-pair exchange.
//
// Weights: int8 in HBM, A operand in TMEM. TMA brings each 128-row x 128-K int8 weight tile
// into shared memory (128-byte swizzle); converter warps read one row each, widen it exactly
// to fp16 in registers (byte v+128 placed under the fp16 exponent of 1024, then 1152
// subtracted) and store it into TMEM with tcgen05.st, where the MMA reads it as its A operand.
// Shared memory then carries only the int8 tile (written by TMA, read once) and the token
// tile (written by TMA, read by the MMA): the tensor core's shared-memory reads are the token
// operand alone. Tokens (the B operand) are fp16 integer codes written by the permutation step
// / requantisation, TMA-loaded in 64-K boxes with the 128-byte swizzle.
//
// Exact integer products on an fp16 tensor pipe. sm_103a has no int8 tcgen05 MMA, so the
// int8 operands are held as fp16 (every int8 value is an fp16 integer) and multiplied with
// kind::f16 into fp32 TMEM accumulators. fp32 holds every integer below 2^24 exactly, so a
// sum of integer products is exact as long as every partial sum stays below 2^24 in
// magnitude, in whatever order the tensor core adds them. Two ways to guarantee that:
//  - bound: for any subset of terms, |sum a_k b_k| <= sqrt(sum a^2) sqrt(sum b^2)
//    (Cauchy-Schwarz). The producers of the token rows record max_row sum(q^2) and weight
//    packing records max_row sum(q_w^2); when their product is below 2^48 one accumulator over
//    the whole K is exact. This holds for realistic data by a wide margin.
//  - chunks: otherwise a fresh accumulator per 1024-element K chunk bounds every partial
//    sum by 1024 * 127^2 < 2^24; the epilogue rounds each chunk to int32 and adds the chunks
//    in integer arithmetic.
// The kernel picks one of the two for the whole launch at its start (every CTA reads the
// same two words). With one accumulator per tile, TMEM holds two of them (2 x TN columns)
// so the epilogue of one tile overlaps the MMAs of the next.
//
// TMEM (512 columns): accumulator slots in columns [0, 384), two A stages of 64 columns
// (128 rows x 128 K of fp16) in [384, 512).
//
// Warp roles (one CTA per SM; GemmRoles):
//   epilogue warps (8 for gate/up, 12 for down): warp w reads TMEM lanes 32*(w%4).. (weight
//               rows) and every (w/4)-th 16-column chunk (tokens) of its quadrant;
//   two converter groups of four warps: group h widens K half h (64 K) of every stage into
//               the stage's A stage, thread r of a group widening weight row r;
//   one MMA issuer and TMEM owner;
//   one TMA producer of the int8 weight tiles, two of the token tiles (alternate stages).
// Pipeline per 128-K stage: the weight tile lands in a ring of 4 int8 stages (released by the
// converters once read); the token tile (two 64-K boxes) in a ring of 3 stages (released by
// the MMA's commit); the two converter groups widen their K halves of the next stage into
// registers ahead and store them into A stage ks % 2 as soon as the MMAs that last read it
// completed; the MMA thread waits for the A stage and the token stage and issues the stage's
// 8 MMAs and two commits (token stage, A stage) in one asm block. Every mbarrier wait is bounded; a wait that runs out sets the plan's error word and
// the CTA drains its own copies and MMAs, frees TMEM and returns.
//
// The down epilogue adds w * dequant(acc) of every (row, channel) into y[token, channel] with
// 16-byte fp32 reductions (y is zeroed by the permutation step), so the per-row outputs never
// go to HBM and no separate combine pass runs; the order of the additions into y is not fixed.
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kW8Bytes = kBM * kKS;                  // int8 weight tile per stage (16 KB)
constexpr int kXSubBytes = kMaxTokTile * kBK * 2;    // one 64-K token box (<= 24 KB)
constexpr int kXStageBytes = 2 * kXSubBytes;         // token tile per stage (<= 48 KB)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kACols = kKS / 2;                 // one A stage: 128 K of fp16 pairs
constexpr int kAStages = 2;
static_assert(kAccCols + kAStages * kACols == kTmemCols, "TMEM columns");
static_assert(2 * kMaxTokTile <= kAccCols, "two accumulator slots");
static_assert(kXSubBytes % 1024 == 0, "swizzled token boxes stay 1024-byte aligned");

constexpr int kConvWarps = 4;  // one converter group: one thread per weight row
#ifndef MOE_GU_EPI_WARPS
#define MOE_GU_EPI_WARPS 8
#endif
#ifndef MOE_D_EPI_WARPS
#define MOE_D_EPI_WARPS 12
#endif
template <bool GU>
struct GemmRoles {
  static constexpr int kEpiWarps = GU ? MOE_GU_EPI_WARPS : MOE_D_EPI_WARPS;
  static constexpr int kColGroups = kEpiWarps / 4;
  static constexpr int kConvGroups = 2;  // group h widens K half h of every stage
  static constexpr int kConvWarp0 = kEpiWarps;
  static constexpr int kMmaWarp = kEpiWarps + kConvGroups * kConvWarps;
  static constexpr int kWProducerWarp = kMmaWarp + 1;
  static constexpr int kXProducerWarp = kWProducerWarp + 1;  // two warps
  static constexpr int kThreads = (kXProducerWarp + 2) * 32;
  static_assert(kEpiWarps % 4 == 0, "epilogue warps cover the four TMEM lane quadrants");
  static_assert(kConvWarp0 % 4 == 0, "converter warp q%4 writes TMEM lane quadrant q%4");
  static_assert(kThreads <= 1024, "block size");
};

#ifndef MOE_X_STAGES
#define MOE_X_STAGES 3
#endif
#ifndef MOE_L2_HINTS
#define MOE_L2_HINTS 1  // weight tiles evict-first, h32 evict-last (read again by requant)
#endif
#ifndef MOE_W_STAGES
#define MOE_W_STAGES 4
#endif
#ifndef MOE_D_X_STAGES
#define MOE_D_X_STAGES MOE_X_STAGES
#endif
#ifndef MOE_D_W_STAGES
#define MOE_D_W_STAGES 5  // the down GEMM's 4-stage items: one more weight stage in flight
#endif
// Shared-memory layout: token stages, int8 weight stages, barriers (stage counts per GEMM).
template <bool GU>
struct GemmSmem {
  static constexpr int kXStages = GU ? MOE_X_STAGES : MOE_D_X_STAGES;
  static constexpr int kWStages = GU ? MOE_W_STAGES : MOE_D_W_STAGES;
  static constexpr int kOffW8 = kXStages * kXStageBytes;
  static constexpr int kOffBar = kOffW8 + kWStages * kW8Bytes;
  static constexpr int kBarBytes = 256;
  static constexpr int kBytes = kOffBar + kBarBytes + 1024;
  static_assert((2 * kXStages + 2 * kWStages + 2 * kAStages + 5) * 8 + 8 <= kBarBytes, "barriers");
  static_assert(kBytes <= 232448, "shared memory");
  static_assert(kOffW8 % 1024 == 0 && kOffBar % 1024 == 0, "swizzled tiles stay 1024-byte aligned");
  static_assert(kXStages >= 2 && kWStages >= 2, "two token producers");
};

// Whether one fp32 accumulator over the whole K is provably exact for this launch.
__device__ __forceinline__ bool single_accumulator_exact(const GemmArgs& a) {
  const unsigned long long r = (unsigned long long)(unsigned)*a.row_sq_max;
  const unsigned long long w = (unsigned long long)(unsigned)*a.w_sq_max;
  return r * w < (1ull << 48);
}

// 4 int8 (one word) -> 4 fp16, exactly: bytes v+128 placed under the fp16 exponent of 1024,
// then 1152 subtracted. Element 0 lands in the low half of the first word.
__device__ __forceinline__ uint2 widen4(uint32_t w) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t lo = __byte_perm(u, 0x64646464u, 0x4140);
  const uint32_t hi = __byte_perm(u, 0x64646464u, 0x4342);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
  const __half2 a = __hsub2(*reinterpret_cast<const __half2*>(&lo), bias);
  const __half2 b = __hsub2(*reinterpret_cast<const __half2*>(&hi), bias);
  return make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
}

// Converter thread of weight row r, half h of a 128-K stage: 64 int8 weights of the row
// (128-byte-swizzled TMA tile) widened to fp16 pairs in 32 registers, laid out as the 32
// TMEM columns of the thread's lane that the MMA reads (K elements 2c, 2c+1 in column c, the
// even element in the low half).
__device__ __forceinline__ void widen_half_row(const uint8_t* w8_tile, int r, int h,
                                               uint32_t (&o)[32]) {
  const uint8_t* src = w8_tile + r * 128;
  const int sw = r & 7;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 v = *reinterpret_cast<const uint4*>(src + 16 * ((4 * h + c) ^ sw));
    const uint2 e0 = widen4(v.x), e1 = widen4(v.y), e2 = widen4(v.z), e3 = widen4(v.w);
    o[8 * c + 0] = e0.x;
    o[8 * c + 1] = e0.y;
    o[8 * c + 2] = e1.x;
    o[8 * c + 3] = e1.y;
    o[8 * c + 4] = e2.x;
    o[8 * c + 5] = e2.y;
    o[8 * c + 6] = e3.x;
    o[8 * c + 7] = e3.y;
  }
}

// NVFP4 converter thread of weight row r, half h of a 128-K stage (64 K): the row's 32 code
// bytes of the half (chunks 2h and 2h + 1, stored at chunk positions c ^ ((r >> 1) & 3)) and its
// 4 block scales, decoded exactly to fp16 pairs in the same 32-column layout as
// widen_half_row: column c holds K elements 2c, 2c + 1 (code byte c: low nibble = element 2c,
// the low half). e2m1(code) * e4m3(scale) is exact in fp16: at most 5 significant bits,
// magnitude between 2^-10 and 2688 (or zero).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t b) {
  uint32_t d;
  asm("{.reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;}" : "=r"(d) : "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t e4m3_to_f16x2_bcast(uint32_t b) {
  uint32_t d;
  const uint16_t two = (uint16_t)((b & 0xffu) | (b & 0xffu) << 8);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(two));
  return d;
}
__device__ __forceinline__ void widen_half_row_fp4(const uint8_t* tile, int r, int h,
                                                   uint32_t (&o)[32]) {
  const uint8_t* src = tile + r * 64;
  const int sw = (r >> 1) & 3;
  const uint32_t sc = *reinterpret_cast<const uint32_t*>(tile + 8192 + r * 8 + 4 * h);
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const uint4 v = *reinterpret_cast<const uint4*>(src + 16 * ((2 * h + c) ^ sw));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int b = 0; b < 2; ++b) {  // block 2c + b: 8 code bytes = words 2b, 2b + 1
      const uint32_t s2 = e4m3_to_f16x2_bcast(sc >> (8 * (2 * c + b)));
      const __half2 hs = *reinterpret_cast<const __half2*>(&s2);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint32_t f = e2m1x2_to_f16x2(w[2 * b + q / 4] >> (8 * (q % 4)));
        const __half2 p = __hmul2(*reinterpret_cast<const __half2*>(&f), hs);
        o[16 * c + 8 * b + q] = *reinterpret_cast<const uint32_t*>(&p);
      }
    }
  }
}

// 16-column chunks one epilogue warp handles per tile (its column group takes every
// kColGroups-th chunk of at most kMaxTokTile columns).
template <int kColGroups>
__host__ __device__ constexpr int kEpiChunks() {
  return (kMaxTokTile / 16 + kColGroups - 1) / kColGroups;
}

// Per-item values an epilogue lane needs, loaded before the accumulator is ready so that
// their latency overlaps the wait: the output channel's weight scales, and per chunk j the
// row values of column (lane & 15) of the chunk.
template <bool GU>
struct EpiMeta {
  static constexpr int kJ = kEpiChunks<(GU ? MOE_GU_EPI_WARPS : MOE_D_EPI_WARPS) / 4>();
  float s0, s1;       // gate/up: gate and up scale of the channel; down: scale of the channel
  uint64_t pol;       // gate/up: L2 policy of the h32 stores
  float rv[kJ];       // gate/up: the row's activation scale; down: h scale (lanes 0-15) or
                      // routing weight (lanes 16-31) of the row
  int tok[GU ? 1 : kJ];  // down: the row's token
};

// a[j] without dynamic register indexing (j is a compile-time constant in the common path).
template <typename T, int N>
__device__ __forceinline__ T pick(const T (&a)[N], int j) {
  T r = a[0];
#pragma unroll
  for (int i = 1; i < N; ++i)
    if (j == i) r = a[i];
  return r;
}

// An accumulator value as the epilogues consume it: either the fp32 TMEM word, which holds the
// integer exactly (one accumulator over the whole K), or an int32 sum of 1024-K chunks.
// acc_f gives float(acc) as the dequantisation rounds it, acc_i the int32 (for debug taps).
__device__ __forceinline__ float acc_f(float x) { return x; }
__device__ __forceinline__ float acc_f(int x) { return __int2float_rn(x); }
__device__ __forceinline__ int acc_i(float x) { return __float2int_rn(x); }
__device__ __forceinline__ int acc_i(int x) { return x; }

// Drains the accumulator tile chunk by chunk: this warp's 16-column chunks c0 = 16 cg,
// 16 (cg + kColGroups), ..., the next chunk's TMEM load issued before the current one is
// consumed. store(v, c0, j) consumes chunk c0 (this warp's j-th). With one accumulator over
// the whole K, v is the fp32 TMEM words themselves (exact integers: no conversion); with
// several 1024-K chunks, each chunk's partial sums are rounded to int32 and added in integer
// arithmetic (the total may exceed what fp32 holds exactly) and v is the int32 sums.
template <int kColGroups, typename Store>
__device__ __forceinline__ void epilogue_columns(const GemmArgs& a, int nch, uint32_t tbase,
                                                 int cg, int ncols, int TN, Store&& store) {
  if (nch == 1) {
    uint32_t ra[16], rb[16];
    auto emit = [&](const uint32_t (&r)[16], int c, int j) {
      float f[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) f[i] = __uint_as_float(r[i]);
      store(f, c, j);
    };
    constexpr int kStep = 16 * kColGroups;  // this warp's chunks: cg, cg + kColGroups, ...
    int c0 = cg * 16;
    if (c0 >= ncols) return;  // uniform over the warp
    tmem_ld16(tbase + c0, ra);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < kEpiChunks<kColGroups>(); j += 2, c0 += 2 * kStep) {
      const int c1 = c0 + kStep;
      if (c1 < ncols) tmem_ld16(tbase + c1, rb);
      emit(ra, c0, j);
      if (c1 >= ncols) break;
      tmem_ld_wait();
      const int c2 = c1 + kStep;
      if (c2 < ncols) tmem_ld16(tbase + c2, ra);
      emit(rb, c1, j + 1);
      if (c2 >= ncols) break;
      tmem_ld_wait();
    }
    return;
  }
#pragma unroll 1
  for (int c0 = cg * 16, j = 0; c0 < ncols; c0 += 16 * kColGroups, ++j) {
    int v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0;
#pragma unroll 1
    for (int kc = 0; kc < nch; ++kc) {
      uint32_t r[16];
      tmem_ld16(tbase + kc * TN + c0, r);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] += __float2int_rn(__uint_as_float(r[i]));
    }
    store(v, c0, j);
  }
}

// Gate/up epilogue. Lane pair (2i, 2i+1) of quadrant q holds gate and up of channel
// m0/2 + 16q + i for every token column; the even lane finishes columns 0-7 of each 16-column
// chunk and the odd lane columns 8-15. Each column's activation scale is taken by shuffle from
// the lane that loaded it.
__device__ __forceinline__ void load_meta_gate_up(const GemmArgs& a, int4 wi, int cg,
                                                  EpiMeta<true>& m) {
  constexpr int kCG = GemmRoles<true>::kColGroups;
  const int lane = threadIdx.x & 31, q = (threadIdx.x >> 5) & 3;
  const bool shared = wi.x == a.E;
  const int ch = (wi.w >> 1) + q * 16 + (lane >> 1);
  m.s0 = (shared ? a.sh_s_g : a.s_g + (size_t)wi.x * a.I)[ch];
  m.s1 = (shared ? a.sh_s_u : a.s_u + (size_t)wi.x * a.I)[ch];
  m.pol = l2_policy_evict_last();
  const int last = wi.y + wi.z - 1;
#pragma unroll
  for (int j = 0; j < EpiMeta<true>::kJ; ++j)
    m.rv[j] = a.sx[min(wi.y + cg * 16 + j * 16 * kCG + (lane & 15), last)];
}

template <bool FP4>
__device__ __forceinline__ void epilogue_gate_up(const GemmArgs& a, int4 wi, int nch,
                                                 uint32_t tbase, int cg, int TN,
                                                 const EpiMeta<true>& m) {
  const int lane = threadIdx.x & 31, q = (threadIdx.x >> 5) & 3;
  const bool odd = lane & 1;
  const int ch = (wi.w >> 1) + q * 16 + (lane >> 1);
  const int ncols = wi.z;
  epilogue_columns<GemmRoles<true>::kColGroups>(a, nch, tbase, cg, ncols, TN,
                                                [&](const auto& v, int c0, int j) {
    using V = typename std::remove_cv<typename std::remove_reference<decltype(v[0])>::type>::type;
    V recv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) recv[i] = __shfl_xor_sync(0xffffffffu, odd ? v[i] : v[8 + i], 1);
    const float rvj = pick(m.rv, j);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int cc = (odd ? 8 : 0) + i;
      const float sx = __shfl_sync(0xffffffffu, rvj, cc);
      const int col = c0 + cc;
      if (col < ncols) {
        const V g = odd ? recv[i] : v[i];
        const V u = odd ? v[8 + i] : recv[i];
        const int row = wi.y + col;
        const float hv = silu_mul(dequant_f(acc_f(g), sx, m.s0), dequant_f(acc_f(u), sx, m.s1));
        if (MOE_L2_HINTS)
          st_f32_hint(a.h32 + (size_t)row * a.Imax + ch, hv, m.pol);  // read again by requant
        else
          a.h32[(size_t)row * a.Imax + ch] = hv;
        if (FP4 && a.tap_f64) {
          a.tap_f64[(size_t)row * 2 * a.Imax + ch] = (double)acc_f(g);
          a.tap_f64[(size_t)row * 2 * a.Imax + a.Imax + ch] = (double)acc_f(u);
        } else if (!FP4 && a.tap) {
          a.tap[(size_t)row * 2 * a.Imax + ch] = acc_i(g);
          a.tap[(size_t)row * 2 * a.Imax + a.Imax + ch] = acc_i(u);
        }
      }
    }
  });
}

// y[0..3] += v, one 16-byte fp32 reduction (the address is 16-byte aligned).
__device__ __forceinline__ void red_add_v4(float* p, float a0, float a1, float a2, float a3) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a0), "f"(a1),
               "f"(a2), "f"(a3)
               : "memory");
}

// 4 x 4 transpose within each lane quad: on entry lane b (= lane % 4) holds v[i] = M[b][i],
// on exit v[i] = M[i][b]. Two butterfly stages (partners b^1, then b^2), two shuffles each.
template <typename V>
__device__ __forceinline__ void quad_transpose(V (&v)[4], int lane) {
  const bool h1 = (lane & 1) != 0, h2 = (lane & 2) != 0;
#pragma unroll
  for (int p = 0; p < 4; p += 2) {
    const V recv = __shfl_xor_sync(0xffffffffu, h1 ? v[p] : v[p + 1], 1);
    if (h1)
      v[p] = recv;
    else
      v[p + 1] = recv;
  }
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const V recv = __shfl_xor_sync(0xffffffffu, h2 ? v[p] : v[p + 2], 2);
    if (h2)
      v[p] = recv;
    else
      v[p + 2] = recv;
  }
}

// Down epilogue: lane = output channel m0 + 32q + lane holds the accumulators of 16 token
// columns per chunk. A 4 x 4 transpose of the accumulators within each lane quad gives
// every lane four consecutive channels of one column; it dequantises them with that column's
// h scale and routing weight (three shuffles per four columns from the lanes that loaded the
// column metadata) and the four channels' weight scales (taken from the quad once per item),
// and adds them into y with one 16-byte reduction: each warp instruction adds 128 contiguous
// bytes into each of four token rows of y.
__device__ __forceinline__ void load_meta_down(const GemmArgs& a, int4 wi, int cg,
                                               EpiMeta<false>& m) {
  constexpr int kCG = GemmRoles<false>::kColGroups;
  const int lane = threadIdx.x & 31, q = (threadIdx.x >> 5) & 3;
  const bool shared = wi.x == a.E;
  m.s0 = (shared ? a.sh_s_d : a.s_d + (size_t)wi.x * a.H)[wi.w + q * 32 + lane];
  const int last = wi.y + wi.z - 1;
#pragma unroll
  for (int j = 0; j < EpiMeta<false>::kJ; ++j) {
    const int lrow = min(wi.y + cg * 16 + j * 16 * kCG + (lane & 15), last);
    m.rv[j] = lane < 16 ? a.s_h[lrow] : a.row_w[lrow];
    m.tok[j] = a.row_token[lrow];
  }
}

template <bool FP4>
__device__ __forceinline__ void epilogue_down(const GemmArgs& a, int4 wi, int nch, uint32_t tbase,
                                              int cg, int TN, const EpiMeta<false>& m) {
  const int lane = threadIdx.x & 31, q = (threadIdx.x >> 5) & 3;
  const int o = wi.w + q * 32 + lane;
  const int ncols = wi.z;
  const int b = lane & 3;
  float* yq = a.y + (o - b);  // first channel of this lane's quad
  float sw[4];                // weight-row scales of the quad's channels o - b + i
#pragma unroll
  for (int i = 0; i < 4; ++i) sw[i] = __shfl_sync(0xffffffffu, m.s0, (lane & ~3) + i);
  epilogue_columns<GemmRoles<false>::kColGroups>(a, nch, tbase, cg, ncols, TN,
                                                 [&](const auto& v, int c0, int j) {
    using V = typename std::remove_cv<typename std::remove_reference<decltype(v[0])>::type>::type;
    if (FP4 && a.tap_f64) {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (c0 + i < ncols) a.tap_f64[(size_t)(wi.y + c0 + i) * a.H + o] = (double)acc_f(v[i]);
    } else if (!FP4 && a.tap) {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (c0 + i < ncols) a.tap[(size_t)(wi.y + c0 + i) * a.H + o] = acc_i(v[i]);
    }
    const float rvj = pick(m.rv, j);
    const int tokj = pick(m.tok, j);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      V t[4] = {v[4 * jj], v[4 * jj + 1], v[4 * jj + 2], v[4 * jj + 3]};
      quad_transpose(t, lane);  // t[i]: channel (o - b + i), column 4jj + b
      const int col = 4 * jj + b;
      const float shr = __shfl_sync(0xffffffffu, rvj, col);
      const float wr = __shfl_sync(0xffffffffu, rvj, 16 + col);
      const int tok = __shfl_sync(0xffffffffu, tokj, col);
      float d[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) d[i] = __fmul_rn(wr, dequant_f(acc_f(t[i]), shr, sw[i]));
      if (c0 + col < ncols) red_add_v4(yq + (size_t)tok * a.H, d[0], d[1], d[2], d[3]);
    }
  });
}

// DUAL: the launch has a second work list in the chunked accumulation's smaller token tiles
// (int8 weights with K > 2048); without one the list and tile are the parameters' own.
template <bool GU, bool FP4, bool DUAL>
__global__ void __launch_bounds__(GemmRoles<GU>::kThreads, 1)
    grouped_gemm_kernel(const GemmArgs a, const __grid_constant__ XMaps tmX,
                        const __grid_constant__ CUtensorMap tmW,
                        const __grid_constant__ CUtensorMap tmWs) {
  constexpr int kXStages = GemmSmem<GU>::kXStages, kWStages = GemmSmem<GU>::kWStages;
  constexpr int kOffW8 = GemmSmem<GU>::kOffW8, kOffBar = GemmSmem<GU>::kOffBar;
  using R = GemmRoles<GU>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* xfull = reinterpret_cast<uint64_t*>(smem + kOffBar);  // [kXStages]
  uint64_t* xempty = xfull + kXStages;     // [kXStages]
  uint64_t* wfull = xempty + kXStages;     // [kWStages]
  uint64_t* wempty = wfull + kWStages;     // [kWStages]
  uint64_t* afull = wempty + kWStages;     // [kAStages]
  uint64_t* aempty = afull + kAStages;     // [kAStages]
  uint64_t* acc_full = aempty + kAStages;  // [2]
  uint64_t* acc_empty = acc_full + 2;      // [2]
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kXStages; ++s) {
      mbar_init(&xfull[s], 1);
      mbar_init(&xempty[s], 1);
    }
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(&wfull[s], 1);
      mbar_init(&wempty[s], R::kConvGroups * kConvWarps);  // every converter warp reads it
    }
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(&afull[s], R::kConvGroups * kConvWarps);
      mbar_init(&aempty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], R::kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == R::kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (!FP4 && warp == R::kWProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmWs);
  }
  if (warp == R::kXProducerWarp && lane < kXMaps) tma_prefetch_desc(&tmX.m[lane]);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the set-up above touches no global memory; from here on the predecessor's results are read
  pdl_wait();
  pdl_trigger();
  const uint32_t tmem = *tmem_slot;
  // Accumulator layout for this launch: one accumulator over the whole K (two TMEM slots,
  // double-buffered) when the bound proves it exact, else 1024-K chunks (the host sizes the
  // token tile so that the chunks of one tile fit the accumulator columns).
  // NVFP4 weights: one fp32 accumulator over the whole K (the products are not integers,
  // the sum is rounded as the tensor core accumulates it)
  const bool single = FP4 || single_accumulator_exact(a);
  // the work list in the token tiles this accumulator layout fits (every CTA and role
  // takes the same one)
  // (selected from the parameters at each use rather than held in registers: the roles are
  // at their register limits)
  const bool main_list = !DUAL || single;
#define KITEMS (main_list ? a.items : a.items_c)
  const int n_items = main_list ? *a.n_items : *a.n_items_c;
#define KTN (main_list ? a.TN : a.TN_c)
  const int kmax = a.K_r > a.K_s ? a.K_r : a.K_s;
  const int slot_cols = single ? KTN : ((kmax + kChunkK - 1) / kChunkK) * KTN;
  const int nslots = slot_cols <= kAccCols / 2 ? 2 : 1;
  const int kpc = single ? (1 << 30) : kChunkK / kKS;  // stages per accumulator

  if (warp >= R::kWProducerWarp && warp < R::kXProducerWarp + 2) {
    if (lane == 0) {
      // ------- TMA producers: weights (HBM) and tokens (two threads, alternate stages) -------
      // Every producer walks the whole item / stage sequence to keep stage and phase in step.
      const bool wprod = warp == R::kWProducerWarp;
      const int pidx = warp - R::kXProducerWarp;  // token producers only
      const int nst = wprod ? kWStages : kXStages;
      uint64_t* full = wprod ? wfull : xfull;
      uint64_t* empty = wprod ? wempty : xempty;
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_par = 0;  // stages with a load issued, and its phase
      uint32_t ks = 0;                    // running stage index
      const uint64_t pol_first = l2_policy_evict_first();  // weights: read once
      bool ok = true;
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        const int4 wi = KITEMS[item];
        const bool shared = wi.x == a.E;
        const int nks = ((shared ? a.K_s : a.K_r) + kKS - 1) / kKS;
        const int rows = (wi.z + kXStep - 1) / kXStep * kXStep;  // box height
        const uint32_t wbytes = FP4 ? (uint32_t)kFp4TileBytes : (uint32_t)kW8Bytes;
        const uint32_t bytes = wprod ? wbytes : (uint32_t)(2 * rows * kBK * 2);
        // NVFP4: this item's tiles, one block per 128-K stage
        const uint8_t* w4 =
            FP4 ? (shared ? a.w4s
                          : a.w4 + (size_t)wi.x * (a.rows_r / kBM) * nks * kFp4TileBytes) +
                      (size_t)(wi.w / kBM) * nks * kFp4TileBytes
                : nullptr;
        const CUtensorMap* mx = &tmX.m[rows / kXStep - 1];
        for (int kb = 0; kb < nks; ++kb, ++ks) {
          if (wprod || (int)(ks & 1) == pidx) {
            if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, a.err)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[stage], bytes);
            if (wprod && FP4) {
              bulk_load_hint(smem + kOffW8 + stage * kW8Bytes, w4 + (size_t)kb * kFp4TileBytes,
                             kFp4TileBytes, &full[stage], pol_first);
            } else if (wprod) {
              uint8_t* sw = smem + kOffW8 + stage * kW8Bytes;
              if (MOE_L2_HINTS) {
                if (shared)
                  tma_load_2d_hint(sw, &tmWs, &full[stage], kb * kKS, wi.w, pol_first);
                else
                  tma_load_3d_hint(sw, &tmW, &full[stage], kb * kKS, wi.w, wi.x, pol_first);
              } else if (shared)
                tma_load_2d(sw, &tmWs, &full[stage], kb * kKS, wi.w);
              else
                tma_load_3d(sw, &tmW, &full[stage], kb * kKS, wi.w, wi.x);
            } else {
              // the second box of a last stage past K reads zeros (out of bounds)
              uint8_t* sx = smem + stage * kXStageBytes;
              tma_load_2d(sx, mx, &full[stage], kb * kKS, wi.y);
              tma_load_2d(sx + kXSubBytes, mx, &full[stage], kb * kKS + kBK, wi.y);
            }
            armed |= 1u << stage;
            armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          }
          if (++stage == nst) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        // Let every copy this thread issued land before the CTA exits.
        for (int s = 0; s < nst; ++s) {
          if (!(armed >> s & 1)) continue;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(&full[s], (armed_par >> s) & 1) &&
                 globaltimer_ns() - t0 < 100000000ull) {
          }
        }
      }
    }
  } else if (warp >= R::kConvWarp0 && warp < R::kConvWarp0 + R::kConvGroups * kConvWarps) {
    // ---------------- converters: int8 weight rows -> fp16 A operand in TMEM ----------------
    // Both groups work on every stage: group h widens K half h (64 K) of each weight row into
    // the stage's A stage (ks % 2). A group widens the next stage's half into registers as
    // soon as its int8 tile has landed, and only then waits for the A stage to be free (the
    // MMAs that last read it completed, aempty): after that wait just the TMEM store, its
    // completion and the arrival remain on the path from one stage's MMAs to the next's.
    const int cw = warp - R::kConvWarp0;
    const int h = cw / kConvWarps;                // K half of every stage
    const int r = (cw % kConvWarps) * 32 + lane;  // weight row within the tile = TMEM lane
    const uint32_t ta = tmem + ((uint32_t)((cw % kConvWarps) * 32) << 16) +
                        (uint32_t)(kAccCols + 32 * h);
    uint32_t o[32];
    int item = blockIdx.x, kb = 0;
    int nks = item < n_items ? ((KITEMS[item].x == a.E ? a.K_s : a.K_r) + kKS - 1) / kKS : 0;
    uint32_t ks = 0;
    // widen stage k's half into o and release the int8 tile
    auto load = [&](uint32_t k) -> bool {
      const int ws = (int)(k % kWStages);
      if (!__all_sync(0xffffffffu, mbar_wait(&wfull[ws], (k / kWStages) & 1u, abort_flag, a.err)))
        return false;
      if constexpr (FP4)
        widen_half_row_fp4(smem + kOffW8 + ws * kW8Bytes, r, h, o);
      else
        widen_half_row(smem + kOffW8 + ws * kW8Bytes, r, h, o);
      __syncwarp();
      if (lane == 0) mbar_arrive(&wempty[ws]);  // values consumed: the int8 tile may be reused
      return true;
    };
    bool ok = item < n_items && load(0);
    while (ok) {
      const int as = (int)(ks & 1);
      if (!__all_sync(0xffffffffu,
                      mbar_wait(&aempty[as], ((ks >> 1) & 1u) ^ 1u, abort_flag, a.err)))
        break;
      tc_fence_after();  // the MMAs that read this A stage before have completed
      tmem_st32(ta + (uint32_t)(as * kACols), o);
      tmem_st_wait();
      // Converter warp 0 also waits for the stage's token tile, so that afull implies it and
      // the MMA thread has a single barrier to check per stage (the converters run far ahead).
      if (cw == 0 &&
          !__all_sync(0xffffffffu, mbar_wait(&xfull[ks % kXStages], (ks / kXStages) & 1u,
                                             abort_flag, a.err)))
        break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&afull[as]);
      ++ks;
      if (++kb == nks) {
        kb = 0;
        item += gridDim.x;
        if (item >= n_items) break;
        nks = ((KITEMS[item].x == a.E ? a.K_s : a.K_r) + kKS - 1) / kKS;
      }
      ok = load(ks);
    }
  } else if (warp == R::kMmaWarp) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      // The issuing thread is on the tensor pipe's critical path: tcgen05.mma issue blocks
      // once the pipe's queue is full, so every instruction between the last MMA of a stage
      // and the first of the next leaves the pipe idle. Per stage it waits on one barrier,
      // afull (usually already seen by the probe inside the previous stage's issue block),
      // which the converters complete only once the stage's token tile has landed too.
      // Descriptors are a base plus a stage offset (the 14-bit start-address field does not
      // carry).
      const uint64_t dx0 = smem_desc_sw128(smem_u32(smem));
      int xs = 0;
      uint32_t ks = 0, ready = 0;
      bool ok = true;
      int it = 0;
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x, ++it) {
        const int4 wi = KITEMS[item];
        const int nks = ((wi.x == a.E ? a.K_s : a.K_r) + kKS - 1) / kKS;
        const int n_mma = (wi.z + 15) & ~15;
        const uint32_t idesc = idesc_f16_f32(kBM, n_mma);
        const int slot = it % nslots;
        const uint32_t use = (uint32_t)(it / nslots) & 1u;
        if (!mbar_wait(&acc_empty[slot], use ^ 1, abort_flag, a.err)) break;
        tc_fence_after();
        uint32_t dt = tmem + (uint32_t)(slot * slot_cols);
        int kin = 0;  // stage within the current accumulator chunk
        for (int kb = 0; kb < nks; ++kb, ++ks) {
          const int g = (int)(ks & 1);
          // afull also covers the token stage (converter warp 0 waits for it before arriving)
          if (!ready && !mbar_wait(&afull[g], (ks >> 1) & 1u, abort_flag, a.err)) {
            ok = false;
            break;
          }
          const uint32_t kn = ks + 1;
          const uint64_t b0 = dx0 + (uint64_t)((xs * kXStageBytes) >> 4);
          ready = mma_stage_ts(dt, tmem + (uint32_t)(kAccCols + g * kACols), b0,
                               b0 + (uint64_t)(kXSubBytes >> 4), idesc, kin != 0 ? 1u : 0u,
                               smem_u32(&xempty[xs]), smem_u32(&aempty[g]),
                               smem_u32(&afull[kn & 1]), (kn >> 1) & 1u);
          if (++kin == kpc) {
            kin = 0;
            dt += (uint32_t)KTN;
          }
          if (++xs == kXStages) xs = 0;
        }
        if (!ok) break;
        umma_commit(&acc_full[slot]);
      }
      // Every MMA this thread issued has completed once `drain` flips.
      umma_commit(drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < 100000000ull) {
      }
    }
  } else if (warp < R::kEpiWarps) {
    // ---------------- epilogue ----------------
    const int cg = warp / 4;  // column group of this warp within its TMEM lane quadrant
    const uint32_t lane_base = tmem + ((uint32_t)((warp % 4) * 32) << 16);
    int it = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++it) {
      const int4 wi = KITEMS[item];
      const int K = wi.x == a.E ? a.K_s : a.K_r;
      const int nch = single ? 1 : (K + kChunkK - 1) / kChunkK;
      const int slot = it % nslots;
      const uint32_t use = (uint32_t)(it / nslots) & 1u;
      EpiMeta<GU> m;
      if constexpr (GU)
        load_meta_gate_up(a, wi, cg, m);
      else
        load_meta_down(a, wi, cg, m);
      if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[slot], use, abort_flag, a.err))) break;
      tc_fence_after();
      const uint32_t tbase = lane_base + (uint32_t)(slot * slot_cols);
      if constexpr (GU)
        epilogue_gate_up<FP4>(a, wi, nch, tbase, cg, KTN, m);
      else
        epilogue_down<FP4>(a, wi, nch, tbase, cg, KTN, m);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[slot]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == R::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
#undef KITEMS
#undef KTN
}

cudaError_t gemm_set_attributes() {
  const void* ks[] = {(const void*)grouped_gemm_kernel<true, false, false>,
                      (const void*)grouped_gemm_kernel<true, false, true>,
                      (const void*)grouped_gemm_kernel<true, true, false>,
                      (const void*)grouped_gemm_kernel<false, false, false>,
                      (const void*)grouped_gemm_kernel<false, false, true>,
                      (const void*)grouped_gemm_kernel<false, true, false>};
  for (int i = 0; i < 6; ++i) {
    const int bytes = i < 3 ? GemmSmem<true>::kBytes : GemmSmem<false>::kBytes;
    const cudaError_t e =
        cudaFuncSetAttribute(ks[i], cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// CTAs of the GEMM that can run at once (one per SM).
cudaError_t gemm_max_ctas(bool gate_up, int* n) {
  *n = 0;
  int per_sm = 0, dev = 0, sms = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &per_sm,
      gate_up ? (const void*)grouped_gemm_kernel<true, false, false>
              : (const void*)grouped_gemm_kernel<false, false, false>,
      gate_up ? GemmRoles<true>::kThreads : GemmRoles<false>::kThreads,
      gate_up ? GemmSmem<true>::kBytes : GemmSmem<false>::kBytes);
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  *n = per_sm * sms;
  return e;
}

cudaError_t launch_grouped_gemm(bool gate_up, bool fp4, const GemmArgs& a, const XMaps& tmX,
                                const CUtensorMap& tmW, const CUtensorMap& tmWs, int grid,
                                cudaStream_t s) {
  if (grid < 1) return cudaErrorInvalidValue;
  if (fp4 && (!a.w4 || a.rows_r % kBM || a.rows_s % kBM || a.items_c)) return cudaErrorInvalidValue;
  const bool dual = a.items_c != nullptr;
  const dim3 g(grid);
  if (gate_up) {
    const dim3 b(GemmRoles<true>::kThreads);
    constexpr int sm = GemmSmem<true>::kBytes;
    if (fp4) return launch_pdl(grouped_gemm_kernel<true, true, false>, g, b, sm, s, a, tmX, tmW, tmWs);
    return dual ? launch_pdl(grouped_gemm_kernel<true, false, true>, g, b, sm, s, a, tmX, tmW, tmWs)
                : launch_pdl(grouped_gemm_kernel<true, false, false>, g, b, sm, s, a, tmX, tmW, tmWs);
  }
  const dim3 b(GemmRoles<false>::kThreads);
  constexpr int sm = GemmSmem<false>::kBytes;
  if (fp4) return launch_pdl(grouped_gemm_kernel<false, true, false>, g, b, sm, s, a, tmX, tmW, tmWs);
  return dual ? launch_pdl(grouped_gemm_kernel<false, false, true>, g, b, sm, s, a, tmX, tmW, tmWs)
              : launch_pdl(grouped_gemm_kernel<false, false, false>, g, b, sm, s, a, tmX, tmW, tmWs);
}

// One thread per 16-byte piece of a packed tile: code chunk position p of tile row r (four per
// row), or the row's 8 scale bytes (a fifth piece, half used).
__global__ void pack_fp4_tiles_kernel(const uint8_t* __restrict__ c0, const uint8_t* __restrict__ c1,
                                      const uint8_t* __restrict__ s0, const uint8_t* __restrict__ s1,
                                      int n_mats, int rows, int K, uint8_t* __restrict__ out) {
  const int nmat = c1 ? 2 : 1;
  const int trows = nmat * rows;          // tile rows per matrix set
  const int tiles = trows / kBM, stages = (K + kKS - 1) / kKS;
  const size_t total = (size_t)n_mats * tiles * stages * kBM * 5;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const int piece = (int)(i % 5);
    const int r = (int)((i / 5) % kBM);
    const size_t ts = i / 5 / kBM;  // (m * tiles + t) * stages + st
    const int st = (int)(ts % stages);
    const int t = (int)((ts / stages) % tiles);
    const int m = (int)(ts / stages / tiles);
    const int R = t * kBM + r;
    const int mat = nmat == 2 ? R % 2 : 0;
    const int srow = nmat == 2 ? R / 2 : R;
    const uint8_t* cs = mat ? c1 : c0;
    const uint8_t* ss = mat ? s1 : s0;
    uint8_t* tile = out + ts * kFp4TileBytes;
    if (piece < 4) {
      const int c = piece ^ ((r >> 1) & 3);  // the chunk stored at position `piece`
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (st * kKS + c * 32 + 32 <= K)
        v = *reinterpret_cast<const uint4*>(cs + ((size_t)m * rows + srow) * (K / 2) + st * 64 + c * 16);
      *reinterpret_cast<uint4*>(tile + r * 64 + piece * 16) = v;
    } else {
      const uint8_t* sp = ss + ((size_t)m * rows + srow) * (K / 16);
#pragma unroll
      for (int b = 0; b < 8; ++b)
        tile[8192 + r * 8 + b] = st * 8 + b < K / 16 ? sp[st * 8 + b] : (uint8_t)0;
    }
  }
}

cudaError_t launch_pack_fp4_tiles(const uint8_t* codes0, const uint8_t* codes1, const uint8_t* sc0,
                                  const uint8_t* sc1, int n_mats, int rows, int K, uint8_t* out,
                                  cudaStream_t s) {
  if ((codes1 ? 2 : 1) * rows % kBM || K % 64) return cudaErrorInvalidValue;
  pack_fp4_tiles_kernel<<<1024, 256, 0, s>>>(codes0, codes1, sc0, sc1, n_mats, rows, K, out);
  return cudaGetLastError();
}

__global__ void fill_rows_kernel(const float* __restrict__ v, int n_mats, int n, float* __restrict__ out) {
  const size_t total = (size_t)n_mats * n;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x)
    out[i] = v[i / n];
}

cudaError_t launch_fill_rows(const float* v, int n_mats, int n, float* out, cudaStream_t s) {
  fill_rows_kernel<<<256, 256, 0, s>>>(v, n_mats, n, out);
  return cudaGetLastError();
}

// Per-row requantisation of h = SiLU(gate)*up: s = amax/127, q = rne(h/s) (|q| <= 127),
// written as fp16 integers for the down GEMM's token operand, and the running maximum of the
// rows' sums of squared codes (the down GEMM's exactness bound).

// Codes of one row of n values held in registers (lane owns values lane*4 + 128j .. +3).
template <int kRegV>
__device__ __forceinline__ float requant_row_regs(const float4 (&v)[kRegV], int n, int lane,
                                                  __half* __restrict__ q, int& sq) {
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < kRegV; ++j)
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)), fmaxf(fabsf(v[j].z), fabsf(v[j].w))));
  amax = warp_max(amax);
  const float s = __fdiv_rn(amax, 127.0f);
  const float rs = quant_recip(s);
#pragma unroll
  for (int j = 0; j < kRegV; ++j) {
    const int i = lane * 4 + j * 128;
    if (i >= n) break;
    int c[4] = {0, 0, 0, 0};
    if (s > 0.0f) {
      c[0] = quant_code(v[j].x, s, rs);
      c[1] = quant_code(v[j].y, s, rs);
      c[2] = quant_code(v[j].z, s, rs);
      c[3] = quant_code(v[j].w, s, rs);
    }
    sq += c[0] * c[0] + c[1] * c[1] + c[2] * c[2] + c[3] * c[3];
    *reinterpret_cast<__half2*>(q + i) = __halves2half2(__int2half_rn(c[0]), __int2half_rn(c[1]));
    *reinterpret_cast<__half2*>(q + i + 2) = __halves2half2(__int2half_rn(c[2]), __int2half_rn(c[3]));
  }
  return s;
}

// The same for a row too long for the registers: two passes over global memory.
__device__ __forceinline__ float requant_row_loop(const float* __restrict__ h, int n, int lane,
                                                  __half* __restrict__ q, int& sq) {
  float amax = 0.0f;
  for (int i = lane * 4; i < n; i += 128) {
    const float4 v = *reinterpret_cast<const float4*>(h + i);
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
  amax = warp_max(amax);
  const float s = __fdiv_rn(amax, 127.0f);
  const float rs = quant_recip(s);
  for (int i = lane * 4; i < n; i += 128) {
    const float4 v = *reinterpret_cast<const float4*>(h + i);
    int c[4] = {0, 0, 0, 0};
    if (s > 0.0f) {
      c[0] = quant_code(v.x, s, rs);
      c[1] = quant_code(v.y, s, rs);
      c[2] = quant_code(v.z, s, rs);
      c[3] = quant_code(v.w, s, rs);
    }
    sq += c[0] * c[0] + c[1] * c[1] + c[2] * c[2] + c[3] * c[3];
    *reinterpret_cast<__half2*>(q + i) = __halves2half2(__int2half_rn(c[0]), __int2half_rn(c[1]));
    *reinterpret_cast<__half2*>(q + i + 2) = __halves2half2(__int2half_rn(c[2]), __int2half_rn(c[3]));
  }
  return s;
}

// Each warp takes kRequantRows consecutive rows and issues the loads of all of them before
// reducing any; rows of up to 128 * kRegV values stay in registers. Small blocks of one row per
// warp give many short waves, so that no second wave runs nearly alone.
#ifndef MOE_RQ_ROWS
#define MOE_RQ_ROWS 1
#endif
#ifndef MOE_RQ_THREADS
#define MOE_RQ_THREADS 256
#endif
constexpr int kRequantRows = MOE_RQ_ROWS;
constexpr int kRequantThreads = MOE_RQ_THREADS;

template <int kRegV>
__global__ void __launch_bounds__(kRequantThreads) requant_kernel(
    const float* __restrict__ h32, int R, int T_sh, int I, int Is, int Imax,
    __half* __restrict__ hq, float* __restrict__ sh, int* __restrict__ sq_max) {
  pdl_wait();  // the predecessor on the stream (launched with launch_pdl)
  pdl_trigger();
  __shared__ int s_sq[32];
  const int lane = threadIdx.x % 32;
  const int row0 = (blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32) * kRequantRows;
  int sq = 0;
  float4 v[kRequantRows][kRegV];
  int n[kRequantRows];
#pragma unroll
  for (int r = 0; r < kRequantRows; ++r) {
    const int row = row0 + r;
    n[r] = row < R ? (row < T_sh ? Is : I) : 0;
    const bool regs = n[r] <= 128 * kRegV;
    const float* h = h32 + (size_t)row * Imax;
#pragma unroll
    for (int j = 0; j < kRegV; ++j)
      v[r][j] = regs && lane * 4 + j * 128 < n[r]
                    ? *reinterpret_cast<const float4*>(h + lane * 4 + j * 128)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int r = 0; r < kRequantRows; ++r) {
    const int row = row0 + r;
    if (row >= R) break;  // uniform over the warp
    __half* q = hq + (size_t)row * Imax;
    const float s = n[r] <= 128 * kRegV
                        ? requant_row_regs<kRegV>(v[r], n[r], lane, q, sq)
                        : requant_row_loop(h32 + (size_t)row * Imax, n[r], lane, q, sq);
    if (lane == 0) sh[row] = s;
  }
  sq = warp_sum_i(sq);
  if (lane == 0) s_sq[threadIdx.x / 32] = sq;
  __syncthreads();
  // one guarded atomic per block: most blocks do not raise the running maximum
  if (threadIdx.x == 0) {
    int m = 0;
    for (int i = 0; i < (int)(blockDim.x / 32); ++i) m = max(m, s_sq[i]);
    if (m > *(volatile int*)sq_max) atomicMax(sq_max, m);
  }
}

cudaError_t launch_requant(const float* h32, int R, int T_sh, int I, int Is, int Imax,
                           __half* hq, float* sh, int* sq_max, cudaStream_t s) {
  if (R <= 0) return cudaSuccess;
  const int rows_per_blk = (kRequantThreads / 32) * kRequantRows;
  const dim3 grid((R + rows_per_blk - 1) / rows_per_blk), block(kRequantThreads);
  if (Imax <= 512)
    return launch_pdl(requant_kernel<4>, grid, block, 0, s, h32, R, T_sh, I, Is, Imax, hq, sh, sq_max);
  return launch_pdl(requant_kernel<8>, grid, block, 0, s, h32, R, T_sh, I, Is, Imax, hq, sh, sq_max);
}

}  // namespace moe
