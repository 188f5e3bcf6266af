// Batched decode and small batches (T <= 64 rows): experts deduplicated across rows, each
// unique expert's int8 weights streamed from HBM exactly once and applied to every row that
// routed to it, with an int8 dot (dp4a) into exact int32 accumulators. This is the kernel the
// page "[job] Strix Halo: multi-session serving ... #145" names as the C>1 limiter (section
// "Status", items "Batched decode doesn't scale" and "Next": expert dedup across rows plus
// int8 dot). An expert's rows are taken kChunk (8) at a time; with more than 8 rows (the
// batched verify arms of the same page, "Plan") the later passes re-read its weights from L2.
// All four launches use programmatic dependent launch: each kernel's blocks may be scheduled
// while its predecessor drains and wait for it in pdl_wait before touching global memory.
//
//  decode_prep_kernel  block 0: the tokens' routing when logits are given, then the
//                      unique-expert list (with the shared expert as group 0) and the
//                      canonical row order; block 1 + t: token t's int8 quant
//                      (spread over T SMs) and y's row t zeroed.
//  decode_gu_kernel    (16 channels of one unique expert) per block: streams 16 gate and 16
//                      up rows, dp4a against up to 8 of the expert's quantised token rows held
//                      in shared memory per pass; fused SiLU(gate)*up.
//  requant_kernel      (shared with the prefill path) requantises every h row once, two
//                      rows per warp, into fp16 codes and scales.
//  decode_down_kernel  (64 output channels of one unique expert) per block: stages up to 8 of
//                      the expert's h code rows as int8 in shared memory per pass, streams 64
//                      down rows, dp4a, and adds w * d into y.
//  decode_gu_fp4_kernel, decode_down_fp4_kernel
//                      the same two streams for NVFP4 expert weights (see "NVFP4 experts"
//                      below): the codes expanded to int8 in registers, exact int64 sums.
#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace moe {

__device__ __forceinline__ int4 ld_stream(const void* p) {
  int4 v;
  asm("ld.global.nc.L1::no_allocate.v4.s32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ int dot16(int4 a, int4 b, int c) {
  c = __dp4a(a.x, b.x, c);
  c = __dp4a(a.y, b.y, c);
  c = __dp4a(a.z, b.z, c);
  return __dp4a(a.w, b.w, c);
}

// v[i] summed over the warp; afterwards lane L holds the total of index L in v[0].
template <typename V>
__device__ __forceinline__ void transpose_reduce32(V (&v)[32], int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const V send = up ? v[i] : v[i + o];
      const V keep = up ? v[i + o] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
}

constexpr int kPrepThreads = 256;
constexpr int kChunk = 8;  // rows per pass over an expert's weights

// Block 0 builds the routing metadata; block 1 + t quantises token t and zeroes y's row t.
__device__ __forceinline__ void prep_quantise_token(const DecodeArgs& a, int t) {
  __shared__ float s_amax[kPrepThreads / 32];
  const int H = a.H, tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const uint16_t* xr = a.x + (size_t)t * H;
  constexpr int kXv = 4;  // uint4 (8 bf16) per thread: rows up to 256 * 8 * 4 = 8192
  uint4 xv[kXv];
#pragma unroll
  for (int c = 0; c < kXv; ++c) {
    const int e0 = (c * kPrepThreads + tid) * 8;
    xv[c] = e0 < H ? *reinterpret_cast<const uint4*>(xr + e0) : make_uint4(0u, 0u, 0u, 0u);
  }
  float amax = 0.0f;
#pragma unroll
  for (int c = 0; c < kXv; ++c) {
    const uint32_t u[4] = {xv[c].x, xv[c].y, xv[c].z, xv[c].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      amax = fmaxf(amax, fabsf(bf16_bits_to_float((uint16_t)(u[i] & 0xffffu))));
      amax = fmaxf(amax, fabsf(bf16_bits_to_float((uint16_t)(u[i] >> 16))));
    }
  }
  amax = warp_max(amax);
  if (lane == 0) s_amax[warp] = amax;
  __syncthreads();
  amax = s_amax[0];
#pragma unroll
  for (int i = 1; i < kPrepThreads / 32; ++i) amax = fmaxf(amax, s_amax[i]);
  const float s = __fdiv_rn(amax, 127.0f);
  const float rs = quant_recip(s);
#pragma unroll
  for (int c = 0; c < kXv; ++c) {
    const int e0 = (c * kPrepThreads + tid) * 8;
    if (e0 < H) {
      const uint32_t u[4] = {xv[c].x, xv[c].y, xv[c].z, xv[c].w};
      uint2 qv;
      uint8_t* qb = reinterpret_cast<uint8_t*>(&qv);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float lo = bf16_bits_to_float((uint16_t)(u[i] & 0xffffu));
        const float hi = bf16_bits_to_float((uint16_t)(u[i] >> 16));
        qb[2 * i] = (uint8_t)(int8_t)(s > 0.0f ? quant_code(lo, s, rs) : 0);
        qb[2 * i + 1] = (uint8_t)(int8_t)(s > 0.0f ? quant_code(hi, s, rs) : 0);
      }
      *reinterpret_cast<uint2*>(a.qtok + (size_t)t * H + e0) = qv;
    }
  }
  if (tid == 0) a.stok[t] = s;
  float4* y4 = reinterpret_cast<float4*>(a.y + (size_t)t * H);
  for (int i = tid; i < H / 4; i += kPrepThreads) y4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

__global__ void __launch_bounds__(kPrepThreads) decode_prep_kernel(DecodeArgs a) {
  pdl_wait();  // the predecessor on the stream (launched with launch_pdl)
  pdl_trigger();
  if (blockIdx.x > 0) {
    prep_quantise_token(a, blockIdx.x - 1);
    return;
  }
  __shared__ int s_cnt[256];
  __shared__ int s_off[257];
  __shared__ int s_idx[kDecodeMaxRows * 8];
  __shared__ float s_wt[kDecodeMaxRows * 8];
  __shared__ int s_warp[kPrepThreads / 32];
  const int T = a.T, k = a.k, E = a.E;
  const int T_sh = a.has_shared ? T : 0;
  const int tid = threadIdx.x;
  const int warp = tid / 32, lane = tid % 32;
  if (a.logits) {  // the tokens' routing first (warp per token); idx, w = idx_out, w_out
    for (int t = warp; t < T; t += kPrepThreads / 32)
      route_token_warp(a.logits + (size_t)t * E, E, k, a.idx_out + (size_t)t * k,
                       a.w_out + (size_t)t * k, lane, s_idx + t * k, s_wt + t * k);
  } else {
    for (int r = tid; r < T * k; r += blockDim.x) {
      s_idx[r] = a.idx[r];
      s_wt[r] = a.w[r];
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) s_cnt[e] = 0;
  for (int r = tid; r < T * k; r += blockDim.x) {
    int e = s_idx[r];
    if (e < 0 || e >= E) {
      set_error(a.err, kErrDevice);
      e = 0;
    }
    s_idx[r] = e;
  }
  __syncthreads();
  for (int r = tid; r < T * k; r += blockDim.x) {
    atomicAdd(&s_cnt[s_idx[r]], 1);
    const int t = r / k;
    for (int q = t * k; q < r; ++q)
      if (s_idx[q] == s_idx[r]) set_error(a.err, kErrDevice);  // expert repeated in a token
  }
  __syncthreads();
  // row offsets and group positions: block-wide exclusive scans over the experts (E <= 256,
  // one per thread), both counts packed in one word (each is at most T * k <= 512)
  {
    const int e = tid;
    const int c = e < E ? s_cnt[e] : 0;
    const int v = (c << 16) | (c > 0 ? 1 : 0);
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += n;
    }
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int i = 0; i < kPrepThreads / 32; ++i) {
      if (i < warp) before += s_warp[i];
      total += s_warp[i];
    }
    const int ex = before + inc - v;  // exclusive prefix of this expert
    if (e < E) {
      const int off = ex >> 16, gp = ex & 0xffff;
      s_off[e] = off;
      a.offsets[e] = off;
      a.counts[e] = c;
      // a group never has more rows than tokens; more means repeated experts (flagged)
      if (c > 0) a.groups[a.has_shared + gp] = make_int4(e, T_sh + off, min(c, T), 0);
    }
    if (tid == 0) {
      s_off[E] = total >> 16;
      a.offsets[E] = total >> 16;
      *a.n_groups = (total & 0xffff) + a.has_shared;
      if (a.has_shared) a.groups[0] = make_int4(E, 0, T, 0);
    }
  }
  __syncthreads();
  for (int r = tid; r < T * k; r += blockDim.x) {
    const int t = r / k, e = s_idx[r];
    int rank = 0;
    for (int q = 0; q < t * k; ++q) rank += (s_idx[q] == e);
    const int pos = min(s_off[e] + rank, T * k - 1);
    a.perm[pos] = r;
    const int row = T_sh + pos;
    a.row_token[row] = t;
    a.row_w[row] = s_wt[r];
  }
  if (a.has_shared && tid < T) {
    a.row_token[tid] = tid;
    a.row_w[tid] = 1.0f;
  }
}

constexpr int kGuChannelsPerBlock = 16;  // 8 warps x 2 channels
constexpr int kDownRowsPerBlock = 64;    // 8 warps x 8 output rows

__global__ void __launch_bounds__(256, 3) decode_gu_kernel(DecodeArgs a) {
  extern __shared__ __align__(16) int8_t xs[];  // [kChunk][H] token codes of one pass
  pdl_wait();  // the predecessor on the stream (launched with launch_pdl)
  pdl_trigger();
  const int g = blockIdx.y;
  if (g >= *a.n_groups) return;
  const int4 grp = a.groups[g];
  const bool shared = grp.x == a.E;
  const int Ig = shared ? a.Is : a.I;
  const int c0 = blockIdx.x * kGuChannelsPerBlock;
  if (c0 >= Ig) return;
  const int H = a.H, nr = grp.z, row0 = grp.y;
  const int8_t* Wg = shared ? a.sh_gate : a.w_gate + (size_t)grp.x * a.I * H;
  const int8_t* Wu = shared ? a.sh_up : a.w_up + (size_t)grp.x * a.I * H;
  const float* sg = shared ? a.sh_s_gate : a.s_gate + (size_t)grp.x * a.I;
  const float* su = shared ? a.sh_s_up : a.s_up + (size_t)grp.x * a.I;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int c = c0 + 2 * warp;
  const int8_t* rows[4] = {Wg + (size_t)c * H, Wu + (size_t)c * H, Wg + (size_t)(c + 1) * H,
                           Wu + (size_t)(c + 1) * H};
  for (int n0 = 0; n0 < nr; n0 += kChunk) {
    const int nc = min(kChunk, nr - n0);
    if (n0 > 0) __syncthreads();  // the previous pass no longer reads xs
    for (int i = threadIdx.x; i < nc * H / 16; i += blockDim.x) {
      const int n = i / (H / 16), u = i % (H / 16);
      const int tok = a.row_token[row0 + n0 + n];
      reinterpret_cast<int4*>(xs + (size_t)n * H)[u] =
          reinterpret_cast<const int4*>(a.qtok + (size_t)tok * H)[u];
    }
    __syncthreads();
    int acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = 0;
#pragma unroll 4
    for (int u = lane; u < H / 16; u += 32) {
      int4 wv[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) wv[r] = ld_stream(rows[r] + (size_t)u * 16);
#pragma unroll
      for (int n = 0; n < kChunk; ++n) {
        if (n < nc) {
          const int4 xv = *reinterpret_cast<const int4*>(xs + (size_t)n * H + u * 16);
#pragma unroll
          for (int r = 0; r < 4; ++r) acc[r * 8 + n] = dot16(wv[r], xv, acc[r * 8 + n]);
        }
      }
    }
    transpose_reduce32(acc, lane);
    const int mine = acc[0];
    const int other = __shfl_down_sync(0xffffffffu, mine, 8);
    const int r = lane >> 3, n = lane & 7;
    if ((r & 1) == 0 && n < nc) {
      const int ch = c + (r >> 1);
      const int row = row0 + n0 + n;
      const float sx = a.stok[a.row_token[row]];
      a.h32[(size_t)row * a.Imax + ch] =
          silu_mul(dequant(mine, sx, sg[ch]), dequant(other, sx, su[ch]));
      if (a.tap_gu) {
        a.tap_gu[(size_t)row * 2 * a.Imax + ch] = mine;
        a.tap_gu[(size_t)row * 2 * a.Imax + a.Imax + ch] = other;
      }
    }
  }
}

__global__ void __launch_bounds__(256) decode_down_kernel(DecodeArgs a) {
  extern __shared__ __align__(16) int8_t hs[];  // [kChunk][Imax] h codes of one pass
  __shared__ float shs[kChunk];
  pdl_wait();  // the predecessor on the stream (launched with launch_pdl)
  pdl_trigger();
  const int g = blockIdx.y;
  if (g >= *a.n_groups) return;
  const int4 grp = a.groups[g];
  const bool shared = grp.x == a.E;
  const int Ig = shared ? a.Is : a.I;
  const int H = a.H, nr = grp.z, row0 = grp.y, Imax = a.Imax;
  const int o0 = blockIdx.x * kDownRowsPerBlock;
  const int8_t* Wd = shared ? a.sh_down : a.w_down + (size_t)grp.x * H * a.I;
  const float* sd = shared ? a.sh_s_down : a.s_down + (size_t)grp.x * H;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int ob = o0 + warp * 8;
  for (int n0 = 0; n0 < nr; n0 += kChunk) {
    const int nc = min(kChunk, nr - n0);
    if (n0 > 0) __syncthreads();  // the previous pass no longer reads hs and shs
    // up to kChunk of this expert's h code rows (fp16 integers, written by the
    // requantisation pass) -> int8
    for (int i = threadIdx.x; i < nc * (Ig / 8); i += blockDim.x) {
      const int n = i / (Ig / 8), u = i % (Ig / 8);
      const uint4 v = reinterpret_cast<const uint4*>(a.hq + (size_t)(row0 + n0 + n) * Imax)[u];
      const __half2* h2 = reinterpret_cast<const __half2*>(&v);
      uint32_t q[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float2 f0 = __half22float2(h2[2 * j]), f1 = __half22float2(h2[2 * j + 1]);
        q[j] = (uint32_t)(uint8_t)(int8_t)(int)f0.x | (uint32_t)(uint8_t)(int8_t)(int)f0.y << 8 |
               (uint32_t)(uint8_t)(int8_t)(int)f1.x << 16 | (uint32_t)(uint8_t)(int8_t)(int)f1.y << 24;
      }
      *reinterpret_cast<uint2*>(hs + (size_t)n * Imax + u * 8) = make_uint2(q[0], q[1]);
    }
    if ((int)threadIdx.x < nc) shs[threadIdx.x] = a.sh[row0 + n0 + threadIdx.x];
    __syncthreads();
    int acc[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) acc[i] = 0;
#pragma unroll 1
    for (int u = lane; u < Ig / 16; u += 32) {
      int4 wv[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) wv[r] = ld_stream(Wd + (size_t)(ob + r) * Ig + (size_t)u * 16);
#pragma unroll
      for (int n = 0; n < kChunk; ++n) {
        if (n < nc) {
          const int4 xv = *reinterpret_cast<const int4*>(hs + (size_t)n * Imax + u * 16);
#pragma unroll
          for (int r = 0; r < 8; ++r) acc[r * 8 + n] = dot16(wv[r], xv, acc[r * 8 + n]);
        }
      }
    }
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      int v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = acc[half * 32 + i];
      transpose_reduce32(v, lane);
      const int r = half * 4 + (lane >> 3), n = lane & 7;
      if (n < nc) {
        const int o = ob + r;
        const int row = row0 + n0 + n;
        const float d = dequant(v[0], shs[n], sd[o]);
        atomicAdd(a.y + (size_t)a.row_token[row] * H + o, __fmul_rn(a.row_w[row], d));
        if (a.tap_d) a.tap_d[(size_t)row * H + o] = v[0];
      }
    }
  }
}

// ---- NVFP4 experts ---------------------------------------------------------------------
// The same two streaming kernels for weights stored as E2M1 codes (two per byte, element 2j
// in the low nibble) with one E4M3 scale per 16-element block and a matrix scale. The codes
// are expanded in registers to int8 values 2 * e2m1 (integers in [-12, 12]) and dotted with
// the int8 activation (or h) codes by dp4a: a block's sum A is an exact int32
// (|A| <= 16 * 127 * 12). The block scale is an integer S in units of 2^-9 (below 2^18), so
// A * S is the block's exact contribution in units of 2^-10 and a row's sum is an exact int64
// (below 2^42 for 8192 elements). float(acc) is then the round-to-nearest-even of the exact
// sum, as the layer definition takes it.
//
// Shapes of the work (compile-time): a warp takes ROWS weight rows and up to NT token rows
// per pass; each lane step reads BPL consecutive 16-element blocks of every row (8 * BPL
// code bytes and BPL scale bytes per row). The accumulators are int64, two registers each,
// so ROWS * NT is what bounds the registers.
#ifndef MOE_FP4_GU_ROWS
#define MOE_FP4_GU_ROWS 2
#endif
#ifndef MOE_FP4_GU_NT
#define MOE_FP4_GU_NT 8
#endif
#ifndef MOE_FP4_GU_BPL
#define MOE_FP4_GU_BPL 2
#endif
#ifndef MOE_FP4_GU_MINB
#define MOE_FP4_GU_MINB 3
#endif
#ifndef MOE_FP4_DN_ROWS
#define MOE_FP4_DN_ROWS 4
#endif
#ifndef MOE_FP4_DN_NT
#define MOE_FP4_DN_NT 4
#endif
#ifndef MOE_FP4_DN_BPL
#define MOE_FP4_DN_BPL 1
#endif
#ifndef MOE_FP4_DN_MINB
#define MOE_FP4_DN_MINB 3
#endif

__device__ __forceinline__ uint2 ld_stream8(const void* p) {
  uint2 v;
  asm("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ld_stream_u8(const void* p) {
  uint16_t v;
  asm("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ld_stream_u16(const void* p) {
  uint16_t v;
  asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// Four E2M1 codes (the low 16 bits of c, code i in bits 4i..4i+3) -> four int8 values
// 2 * e2m1(code), value i in byte i. Magnitudes come from a byte lookup (prmt) into
// {0, 1, 2, 3, 4, 6, 8, 12} and its negation; the sign bits, replicated over their bytes by
// prmt's sign mode, pick between the two.
__device__ __forceinline__ uint32_t e2m1x4_to_s8(uint32_t c) {
  const uint32_t sel = c & 0x7777u;
  uint32_t pos, neg, sgn;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(pos) : "r"(0x03020100u), "r"(0x0C080604u), "r"(sel));
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(neg) : "r"(0xFDFEFF00u), "r"(0xF4F8FAFCu), "r"(sel));
  // output byte i replicates the top bit of: byte 0 of c << 4 (code 0's sign), byte 0 of c
  // (code 1), byte 1 of c << 4 (code 2), byte 1 of c (code 3)
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(sgn) : "r"(c << 4), "r"(c), "r"(0xD9C8u));
  return (pos & ~sgn) | (neg & sgn);
}

// 16 E2M1 codes (8 bytes) -> 16 int8 values 2 * e2m1, as the int4 dot16 takes.
__device__ __forceinline__ int4 e2m1x16_to_s8(uint32_t lo, uint32_t hi) {
  return make_int4((int)e2m1x4_to_s8(lo), (int)e2m1x4_to_s8(lo >> 16), (int)e2m1x4_to_s8(hi),
                   (int)e2m1x4_to_s8(hi >> 16));
}

// A finite non-negative E4M3 byte (bits 0-7 of b; higher bits ignored) -> its value in units
// of 2^-9: (8 + f) << (e - 1) for a normal value (exponent field e > 0, mantissa f), f for a
// subnormal one.
__device__ __forceinline__ int e4m3_units(uint32_t b) {
  const int e = (int)((b >> 3) & 15u), f = (int)(b & 7u);
  return e ? (8 | f) << (e - 1) : f;
}

// acc + a * b with a 64-bit accumulator, one instruction.
__device__ __forceinline__ long long mad_wide(int a, int b, long long acc) {
  long long d;
  asm("mad.wide.s32 %0, %1, %2, %3;" : "=l"(d) : "r"(a), "r"(b), "l"(acc));
  return d;
}

// float(exact sum) of an accumulator in units of 2^-10 (a power-of-two scaling: exact).
__device__ __forceinline__ float fp4_acc_float(long long acc) {
  return __fmul_rn(__ll2float_rn(acc), 0x1p-10f);
}

// v[i] summed over the warp (N = 8, 16 or 32 values per lane); afterwards lane L holds the
// total of index L % N in v[0].
template <int N, typename V>
__device__ __forceinline__ void transpose_reduce(V (&v)[N], int lane) {
  static_assert(N == 8 || N == 16 || N == 32, "values per lane");
#pragma unroll
  for (int o = N / 2; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const V send = up ? v[i] : v[i + o];
      const V keep = up ? v[i + o] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
#pragma unroll
  for (int o = N; o < 32; o <<= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
}

// Calls f(std::integral_constant<int, n>()) for the runtime count n in [C, NT], so that a loop
// over n tokens is unrolled for exactly n (no predicated iterations for absent tokens).
template <int C, int NT, class F>
__device__ __forceinline__ void with_count(int n, F&& f) {
  if constexpr (C <= NT) {
    if (n == C)
      f(std::integral_constant<int, C>());
    else
      with_count<C + 1, NT>(n, f);
  }
}

// acc[r * NT + n] = exact sum over the K elements of weight row r times token row n (int8
// codes at xs + n * xstride), for n < NC, this lane's share: lane steps u = lane, lane + 32,
// ... each covering BPL blocks. Weight row r is row r / NB of NB interleaved matrices: codes
// at cb[r % NB] + (r / NB) * K / 2, block scales at sb[r % NB] + (r / NB) * K / 16 (gate/up:
// NB = 2, rows gate c, up c, gate c + 1, ...; down: NB = 1, consecutive rows).
template <int ROWS, int NT, int BPL, int NB, int NC>
__device__ __forceinline__ void fp4_dot_rows(const uint8_t* const (&cb)[NB],
                                             const uint8_t* const (&sb)[NB], int K,
                                             const int8_t* xs, int xstride, int lane,
                                             long long (&acc)[ROWS * NT]) {
  static_assert(NC >= 1 && NC <= NT, "token count");
  static_assert(BPL == 1 || BPL == 2, "blocks per lane step");
  const int cstride = K / 2, sstride = K / 16;
#pragma unroll
  for (int i = 0; i < ROWS * NT; ++i) acc[i] = 0;
#pragma unroll 2
  for (int u = lane; u < K / (16 * BPL); u += 32) {
    uint32_t cw[ROWS][2 * BPL];
    uint32_t sw[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      const uint8_t* cp = cb[r % NB] + (r / NB) * cstride;
      const uint8_t* sp = sb[r % NB] + (r / NB) * sstride;
      if constexpr (BPL == 1) {
        const uint2 v = ld_stream8(cp + u * 8);
        cw[r][0] = v.x;
        cw[r][1] = v.y;
        sw[r] = ld_stream_u8(sp + u);
      } else {
        const int4 v = ld_stream(cp + u * 16);
        cw[r][0] = (uint32_t)v.x;
        cw[r][1] = (uint32_t)v.y;
        cw[r][2] = (uint32_t)v.z;
        cw[r][3] = (uint32_t)v.w;
        sw[r] = ld_stream_u16(sp + 2 * u);
      }
    }
#pragma unroll
    for (int b = 0; b < BPL; ++b) {
      int4 wx[ROWS];
      int S[ROWS];
#pragma unroll
      for (int r = 0; r < ROWS; ++r) {
        wx[r] = e2m1x16_to_s8(cw[r][2 * b], cw[r][2 * b + 1]);
        S[r] = e4m3_units(sw[r] >> (8 * b));
      }
#pragma unroll
      for (int n = 0; n < NC; ++n) {
        const int4 xv =
            *reinterpret_cast<const int4*>(xs + (size_t)n * xstride + (u * BPL + b) * 16);
#pragma unroll
        for (int r = 0; r < ROWS; ++r)
          acc[r * NT + n] = mad_wide(dot16(wx[r], xv, 0), S[r], acc[r * NT + n]);
      }
    }
  }
}

constexpr int kFp4GuRows = MOE_FP4_GU_ROWS;  // gate/up rows per warp: channel pairs
constexpr int kFp4GuNt = MOE_FP4_GU_NT;
constexpr int kFp4DnRows = MOE_FP4_DN_ROWS;
constexpr int kFp4DnNt = MOE_FP4_DN_NT;
constexpr int kGuFp4ChannelsPerBlock = 8 * kFp4GuRows / 2;
constexpr int kDownFp4RowsPerBlock = 8 * kFp4DnRows;
static_assert(kFp4GuRows % 2 == 0 && 64 % kGuFp4ChannelsPerBlock == 0, "gate/up channel blocks");
static_assert(128 % kDownFp4RowsPerBlock == 0, "down row blocks");

__global__ void __launch_bounds__(256, MOE_FP4_GU_MINB) decode_gu_fp4_kernel(DecodeArgs a) {
  constexpr int ROWS = kFp4GuRows, NT = kFp4GuNt, N = ROWS * NT;
  extern __shared__ __align__(16) int8_t xs[];  // [NT][H] token codes of one pass
  pdl_wait();  // the predecessor on the stream (launched with launch_pdl)
  pdl_trigger();
  const int g = blockIdx.y;
  if (g >= *a.n_groups) return;
  const int4 grp = a.groups[g];
  const bool shared = grp.x == a.E;
  const int Ig = shared ? a.Is : a.I;
  const int c0 = blockIdx.x * kGuFp4ChannelsPerBlock;
  if (c0 >= Ig) return;
  const int H = a.H, nr = grp.z, row0 = grp.y;
  const size_t cs = H / 2, ss = H / 16;  // code and scale bytes per weight row
  const uint8_t* Wg = shared ? a.f.sh_gate : a.f.w_gate + (size_t)grp.x * a.I * cs;
  const uint8_t* Wu = shared ? a.f.sh_up : a.f.w_up + (size_t)grp.x * a.I * cs;
  const uint8_t* Bg = shared ? a.f.sh_b_gate : a.f.b_gate + (size_t)grp.x * a.I * ss;
  const uint8_t* Bu = shared ? a.f.sh_b_up : a.f.b_up + (size_t)grp.x * a.I * ss;
  // matrix scales: sh_g exists only with a shared expert, so the pointer is chosen first
  const float gg = *(shared ? a.f.sh_g : a.f.g_gate + grp.x);
  const float gu = *(shared ? a.f.sh_g + 1 : a.f.g_up + grp.x);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int c = c0 + warp * (ROWS / 2);
  // rows {gate c, up c, gate c + 1, up c + 1, ...}
  const uint8_t* const cb[2] = {Wg + c * cs, Wu + c * cs};
  const uint8_t* const sb[2] = {Bg + c * ss, Bu + c * ss};
  for (int n0 = 0; n0 < nr; n0 += NT) {
    const int nc = min(NT, nr - n0);
    if (n0 > 0) __syncthreads();  // the previous pass no longer reads xs
    for (int i = threadIdx.x; i < nc * H / 16; i += blockDim.x) {
      const int n = i / (H / 16), u = i % (H / 16);
      const int tok = a.row_token[row0 + n0 + n];
      reinterpret_cast<int4*>(xs + (size_t)n * H)[u] =
          reinterpret_cast<const int4*>(a.qtok + (size_t)tok * H)[u];
    }
    __syncthreads();
    // one specialisation per token count: the dot, the warp reduction and the epilogue
    with_count<1, NT>(nc, [&](auto cnt) {
      long long acc[N];
      fp4_dot_rows<ROWS, NT, MOE_FP4_GU_BPL, 2, decltype(cnt)::value>(cb, sb, H, xs, H, lane, acc);
      transpose_reduce<N>(acc, lane);
      const long long mine = acc[0];
      const long long other = __shfl_down_sync(0xffffffffu, mine, NT);  // the channel's up row
      const int r = lane / NT, n = lane % NT;
      if (lane < N && (r & 1) == 0 && n < nc) {
        const int ch = c + (r >> 1);
        const int row = row0 + n0 + n;
        const float sx = a.stok[a.row_token[row]];
        a.h32[(size_t)row * a.Imax + ch] = silu_mul(dequant_f(fp4_acc_float(mine), sx, gg),
                                                    dequant_f(fp4_acc_float(other), sx, gu));
        if (a.tap_gu_f64) {
          a.tap_gu_f64[(size_t)row * 2 * a.Imax + ch] = (double)mine * 0x1p-10;
          a.tap_gu_f64[(size_t)row * 2 * a.Imax + a.Imax + ch] = (double)other * 0x1p-10;
        }
      }
    });
  }
}

__global__ void __launch_bounds__(256, MOE_FP4_DN_MINB) decode_down_fp4_kernel(DecodeArgs a) {
  constexpr int ROWS = kFp4DnRows, NT = kFp4DnNt, N = ROWS * NT;
  extern __shared__ __align__(16) int8_t hs[];  // [NT][Imax] h codes of one pass
  __shared__ float shs[NT];
  pdl_wait();  // the predecessor on the stream (launched with launch_pdl)
  pdl_trigger();
  const int g = blockIdx.y;
  if (g >= *a.n_groups) return;
  const int4 grp = a.groups[g];
  const bool shared = grp.x == a.E;
  const int Ig = shared ? a.Is : a.I;
  const int H = a.H, nr = grp.z, row0 = grp.y, Imax = a.Imax;
  const int o0 = blockIdx.x * kDownFp4RowsPerBlock;
  const size_t cs = Ig / 2, ss = Ig / 16;
  const uint8_t* Wd = shared ? a.f.sh_down : a.f.w_down + (size_t)grp.x * H * cs;
  const uint8_t* Bd = shared ? a.f.sh_b_down : a.f.b_down + (size_t)grp.x * H * ss;
  const float gd = *(shared ? a.f.sh_g + 2 : a.f.g_down + grp.x);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int ob = o0 + warp * ROWS;
  const uint8_t* const cb[1] = {Wd + (size_t)ob * cs};
  const uint8_t* const sb[1] = {Bd + (size_t)ob * ss};
  for (int n0 = 0; n0 < nr; n0 += NT) {
    const int nc = min(NT, nr - n0);
    if (n0 > 0) __syncthreads();  // the previous pass no longer reads hs and shs
    // up to NT of this expert's h code rows (fp16 integers) -> int8
    for (int i = threadIdx.x; i < nc * (Ig / 8); i += blockDim.x) {
      const int n = i / (Ig / 8), u = i % (Ig / 8);
      const uint4 v = reinterpret_cast<const uint4*>(a.hq + (size_t)(row0 + n0 + n) * Imax)[u];
      const __half2* h2 = reinterpret_cast<const __half2*>(&v);
      uint32_t q[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float2 f0 = __half22float2(h2[2 * j]), f1 = __half22float2(h2[2 * j + 1]);
        q[j] = (uint32_t)(uint8_t)(int8_t)(int)f0.x | (uint32_t)(uint8_t)(int8_t)(int)f0.y << 8 |
               (uint32_t)(uint8_t)(int8_t)(int)f1.x << 16 | (uint32_t)(uint8_t)(int8_t)(int)f1.y << 24;
      }
      *reinterpret_cast<uint2*>(hs + (size_t)n * Imax + u * 8) = make_uint2(q[0], q[1]);
    }
    if ((int)threadIdx.x < nc) shs[threadIdx.x] = a.sh[row0 + n0 + threadIdx.x];
    __syncthreads();
    with_count<1, NT>(nc, [&](auto cnt) {
      long long acc[N];
      fp4_dot_rows<ROWS, NT, MOE_FP4_DN_BPL, 1, decltype(cnt)::value>(cb, sb, Ig, hs, Imax, lane, acc);
      transpose_reduce<N>(acc, lane);
      const int r = lane / NT, n = lane % NT;
      if (lane < N && n < nc) {
        const int o = ob + r;
        const int row = row0 + n0 + n;
        const float d = dequant_f(fp4_acc_float(acc[0]), shs[n], gd);
        atomicAdd(a.y + (size_t)a.row_token[row] * H + o, __fmul_rn(a.row_w[row], d));
        if (a.tap_d_f64) a.tap_d_f64[(size_t)row * H + o] = (double)acc[0] * 0x1p-10;
      }
    });
  }
}

__global__ void check_e4m3_kernel(const uint8_t* __restrict__ b, size_t n, int* err) {
  bool bad = false;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    bad |= b[i] >= 0x7f;  // negative, or the NaN encoding
  if (__syncthreads_or(bad) && threadIdx.x == 0) set_error(err, kErrDevice);
}

cudaError_t launch_check_e4m3(const uint8_t* b, size_t n, int* err, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int blocks = (int)std::min<size_t>((n + 255) / 256, 4096);
  check_e4m3_kernel<<<blocks, 256, 0, s>>>(b, n, err);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s, cudaEvent_t* ev) {
  if (a.T < 1 || a.T > kDecodeMaxRows || a.k > 8 || a.E > 256) return cudaErrorInvalidValue;
  const int R = a.T * a.k + (a.has_shared ? a.T : 0);
  if (ev) cudaEventRecord(ev[0], s);
  cudaError_t e = launch_pdl(decode_prep_kernel, dim3(1 + a.T), dim3(kPrepThreads), 0, s, a);
  if (ev) cudaEventRecord(ev[1], s);
  if (e != cudaSuccess) return e;
  const int gmax = min(a.E, a.T * a.k) + (a.has_shared ? 1 : 0);
  if (a.fp4) {
    const dim3 ggu((a.Imax + kGuFp4ChannelsPerBlock - 1) / kGuFp4ChannelsPerBlock, gmax);
    e = launch_pdl(decode_gu_fp4_kernel, ggu, dim3(256), (size_t)kFp4GuNt * a.H, s, a);
  } else {
    const dim3 ggu((a.Imax + kGuChannelsPerBlock - 1) / kGuChannelsPerBlock, gmax);
    e = launch_pdl(decode_gu_kernel, ggu, dim3(256), (size_t)kChunk * a.H, s, a);
  }
  if (e != cudaSuccess) return e;
  // one requantisation of every h row (warp per row), instead of one per down block
  e = launch_requant(a.h32, R, a.has_shared ? a.T : 0, a.I, a.Is, a.Imax, a.hq, a.sh,
                     a.sq_scratch, s);
  if (e != cudaSuccess) return e;
  if (ev) cudaEventRecord(ev[2], s);
  if (a.fp4)
    e = launch_pdl(decode_down_fp4_kernel, dim3(a.H / kDownFp4RowsPerBlock, gmax), dim3(256),
                   (size_t)kFp4DnNt * a.Imax, s, a);
  else
    e = launch_pdl(decode_down_kernel, dim3(a.H / kDownRowsPerBlock, gmax), dim3(256),
                   (size_t)kChunk * a.Imax, s, a);
  if (ev) cudaEventRecord(ev[3], s);
  return e;
}

bool decode_shape_supported(int H, int Imax) { return H <= kDecodeMaxH && Imax <= kDecodeMaxI; }

// The kernels' dynamic shared-memory limit is a process-wide attribute: it is set once to the
// largest shapes the library accepts (never per plan, so that a plan with smaller shapes
// cannot lower it under a plan with larger ones).
cudaError_t decode_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(decode_gu_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kChunk * kDecodeMaxH);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(decode_gu_fp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kFp4GuNt * kDecodeMaxH);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(decode_down_fp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kFp4DnNt * kDecodeMaxI);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(decode_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kChunk * kDecodeMaxI);
}

}  // namespace moe
