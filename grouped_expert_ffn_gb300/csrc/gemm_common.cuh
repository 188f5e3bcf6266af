// Device code shared by the two grouped-GEMM kernels (one CTA per tile, and the CTA pair of
// the 2-SM MMA): operand widening, exactness test and the two fused epilogues.
#pragma once
#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kW8Bytes = kBM * kBK;       // int8 weight tile per k-block (8 KB)
constexpr int kW16Bytes = kBM * kBK * 2;  // fp16 weight tile per k-block (16 KB)
// Warp roles of the grouped GEMM kernels: epilogue warps (four per TMEM lane quadrant times
// column groups), converter groups of four warps taking turns over k-blocks, one MMA warp,
// two weight-TMA warps, two token-TMA warps. The gate/up GEMM (32 k-blocks per item, light
// epilogue) runs two converter groups and 8 epilogue warps; the down GEMM (8 k-blocks per
// item, an epilogue that writes w * d for every row) two converter groups and 12 epilogue
// warps, so that its epilogue keeps up with its mainloop (the register file caps a block of
// 25 warps at 72 registers a thread).
constexpr int kConvWarps = 4;  // one converter group: one thread per weight row
#ifndef MOE_GU_EPI_WARPS
#define MOE_GU_EPI_WARPS 8
#endif
#ifndef MOE_GU_CONV_GROUPS
#define MOE_GU_CONV_GROUPS 2
#endif
#ifndef MOE_D_EPI_WARPS
#define MOE_D_EPI_WARPS 12
#endif
#ifndef MOE_D_CONV_GROUPS
#define MOE_D_CONV_GROUPS 2
#endif
template <bool GU>
struct GemmRoles {
  static constexpr int kEpiWarps = GU ? MOE_GU_EPI_WARPS : MOE_D_EPI_WARPS;
  static constexpr int kColGroups = kEpiWarps / 4;
  static constexpr int kConvGroups = GU ? MOE_GU_CONV_GROUPS : MOE_D_CONV_GROUPS;
  static constexpr int kConvWarp0 = kEpiWarps;
  static constexpr int kMmaWarp = kEpiWarps + kConvGroups * kConvWarps;
  static constexpr int kWProducerWarp = kMmaWarp + 1;        // two warps
  static constexpr int kXProducerWarp = kWProducerWarp + 2;  // two warps
  static constexpr int kThreads = (kXProducerWarp + 2) * 32;
  static_assert(kEpiWarps % 4 == 0, "epilogue warps cover the four TMEM lane quadrants");
  static_assert(kThreads <= 1024, "block size");
};
constexpr uint32_t kTmemCols = 512;

// Whether one fp32 accumulator over the whole K is provably exact for this launch.
__device__ __forceinline__ bool single_accumulator_exact(const GemmArgs& a) {
  const unsigned long long r = (unsigned long long)(unsigned)*a.row_sq_max;
  const unsigned long long w = (unsigned long long)(unsigned)*a.w_sq_max;
  return r * w < (1ull << 48);
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 4 int8 (one word) -> 4 fp16, exactly: bytes v+128 placed under the fp16 exponent of 1024,
// then 1152 subtracted.
__device__ __forceinline__ uint2 widen4(uint32_t w) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t lo = __byte_perm(u, 0x64646464u, 0x4140);
  const uint32_t hi = __byte_perm(u, 0x64646464u, 0x4342);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
  const __half2 a = __hsub2(*reinterpret_cast<const __half2*>(&lo), bias);
  const __half2 b = __hsub2(*reinterpret_cast<const __half2*>(&hi), bias);
  return make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
}

// Epilogue column loop with one accumulator per tile: TMEM loads of the next 16-column chunk
// are in flight while the current one is dequantised and stored (tcgen05.wait::ld waits for
// all of a thread's outstanding loads, so the two register sets alternate). `store(v, c0)`
// consumes the 16 int32 accumulators of chunk c0 (the fp32 words hold integers). With several
// 1024-K chunks per tile, each chunk's partial sums are rounded to int32 and added in integer
// arithmetic (the total may exceed what fp32 holds exactly).
template <int kColGroups, typename Store>
__device__ __forceinline__ void epilogue_columns(const GemmArgs& a, int nch, uint32_t tbase,
                                                 int cg, int ncols, Store&& store) {
  auto to_int = [](const uint32_t (&r)[16], int (&v)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __float2int_rn(__uint_as_float(r[i]));
  };
  if (nch == 1) {
    uint32_t ra[16], rb[16];
    int v[16];
    constexpr int kStep = 16 * kColGroups;  // this warp's chunks: cg, cg + kColGroups, ...
    int c0 = cg * 16;
    if (c0 >= ncols) return;  // uniform over the warp
    tmem_ld16(tbase + c0, ra);
    tmem_ld_wait();
#pragma unroll 1
    for (; c0 < ncols; c0 += 2 * kStep) {
      const int c1 = c0 + kStep;
      if (c1 < ncols) tmem_ld16(tbase + c1, rb);
      to_int(ra, v);
      store(v, c0);
      if (c1 >= ncols) break;
      tmem_ld_wait();
      const int c2 = c1 + kStep;
      if (c2 < ncols) tmem_ld16(tbase + c2, ra);
      to_int(rb, v);
      store(v, c1);
      if (c2 >= ncols) break;
      tmem_ld_wait();
    }
    return;
  }
#pragma unroll 1
  for (int c0 = cg * 16; c0 < ncols; c0 += 16 * kColGroups) {
    int v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0;
#pragma unroll 1
    for (int kc = 0; kc < nch; ++kc) {
      uint32_t r[16];
      tmem_ld16(tbase + kc * a.TN + c0, r);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] += __float2int_rn(__uint_as_float(r[i]));
    }
    store(v, c0);
  }
}

// Gate/up epilogue. Lane pair (2i, 2i+1) of quadrant q holds gate and up of channel
// m0/2 + 16q + i for every token column; the even lane finishes columns 0-7 of each 16-column
// chunk and the odd lane columns 8-15.
__device__ __forceinline__ void epilogue_gate_up(const GemmArgs& a, int4 wi, int nch,
                                                 uint32_t tbase, int cg) {
  const int lane = threadIdx.x & 31, q = (threadIdx.x >> 5) & 3;
  const bool odd = lane & 1;
  const bool shared = wi.x == a.E;
  const int ch = (wi.w >> 1) + q * 16 + (lane >> 1);
  const float sgc = (shared ? a.sh_s_g : a.s_g + (size_t)wi.x * a.I)[ch];
  const float suc = (shared ? a.sh_s_u : a.s_u + (size_t)wi.x * a.I)[ch];
  const int ncols = wi.z;
  epilogue_columns<GemmRoles<true>::kColGroups>(a, nch, tbase, cg, ncols,
                                                [&](const int (&v)[16], int c0) {
    int recv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) recv[i] = __shfl_xor_sync(0xffffffffu, odd ? v[i] : v[8 + i], 1);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int col = c0 + (odd ? 8 : 0) + i;
      if (col < ncols) {
        const int g = odd ? recv[i] : v[i];
        const int u = odd ? v[8 + i] : recv[i];
        const int row = wi.y + col;
        const float sx = a.sx[row];
        a.h32[(size_t)row * a.Imax + ch] = silu_mul(dequant(g, sx, sgc), dequant(u, sx, suc));
        if (a.tap) {
          a.tap[(size_t)row * 2 * a.Imax + ch] = g;
          a.tap[(size_t)row * 2 * a.Imax + a.Imax + ch] = u;
        }
      }
    }
  });
}

// Down epilogue: lane = output channel m0 + 32q + lane; for each token column the warp stores
// w * dequant(acc) for 32 consecutive channels of that row of yd (one 128-byte store). The
// combine kernel then sums each token's rows in slot order.
__device__ __forceinline__ void epilogue_down(const GemmArgs& a, int4 wi, int nch, uint32_t tbase,
                                              int cg) {
  const int lane = threadIdx.x & 31, q = (threadIdx.x >> 5) & 3;
  const bool shared = wi.x == a.E;
  const int o = wi.w + q * 32 + lane;
  const float sdo = (shared ? a.sh_s_d : a.s_d + (size_t)wi.x * a.H)[o];
  const int ncols = wi.z;
  const int last = wi.y + ncols - 1;
  epilogue_columns<GemmRoles<false>::kColGroups>(a, nch, tbase, cg, ncols,
                                                 [&](const int (&v)[16], int c0) {
    // One load per lane before any store of the chunk (the stores might alias the scales as
    // far as the compiler knows): lanes 0-15 hold the rows' h scales, lanes 16-31 their
    // routing weights; each column takes its two by shuffle.
    const int lrow = min(wi.y + c0 + (lane & 15), last);
    const float lv = lane < 16 ? a.s_h[lrow] : a.row_w[lrow];
    float* dst = a.yd + (size_t)(wi.y + c0) * a.H + o;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float shr = __shfl_sync(0xffffffffu, lv, i);
      const float wr = __shfl_sync(0xffffffffu, lv, 16 + i);
      if (c0 + i < ncols) {
        dst[(size_t)i * a.H] = __fmul_rn(wr, dequant(v[i], shr, sdo));
        if (a.tap) a.tap[(size_t)(wi.y + c0 + i) * a.H + o] = v[i];
      }
    }
  });
}

// Converter thread r: weight row r of one k-block, int8 (64-byte swizzled TMA tile) to fp16
// (128-byte swizzled tile read by the MMA).
__device__ __forceinline__ void widen_row(const uint8_t* w8_tile, uint8_t* w16_tile, int r) {
  const int sw8 = (r >> 1) & 3;  // 64-byte swizzle of the int8 row
  const int sw16 = r & 7;        // 128-byte swizzle of the fp16 row
  const uint8_t* src = w8_tile + r * 64;
  uint8_t* dst = w16_tile + r * 128;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 v = *reinterpret_cast<const uint4*>(src + 16 * (c ^ sw8));
    const uint2 e0 = widen4(v.x), e1 = widen4(v.y), e2 = widen4(v.z), e3 = widen4(v.w);
    *reinterpret_cast<uint4*>(dst + 16 * ((2 * c) ^ sw16)) = make_uint4(e0.x, e0.y, e1.x, e1.y);
    *reinterpret_cast<uint4*>(dst + 16 * ((2 * c + 1) ^ sw16)) = make_uint4(e2.x, e2.y, e3.x, e3.y);
  }
}

// The pair kernel (gemm_pair.cu): items of two adjacent weight tiles, one per CTA of the pair.
cudaError_t pair_set_attributes();
cudaError_t pair_max_clusters(bool gate_up, int* n);
cudaError_t launch_pair_gemm(bool gate_up, const GemmArgs& a, const XMaps& tmX,
                             const CUtensorMap& tmW, const CUtensorMap& tmWs, int grid,
                             cudaStream_t s);

}  // namespace moe
