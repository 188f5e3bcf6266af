// Grouped W8A8 GEMMs of the prefill path on the 5th-generation tensor cores (tcgen05).
//
// One persistent kernel runs every (expert group, 128-row weight tile, token tile) work item
// of a layer: the gate/up GEMM with a fused SiLU(gate)*up epilogue, or the down GEMM with a
// fused router-weighted scatter-combine into y. This is the concatenated-expert computation
// of the page "Qwen3.6-35B-A3B Linux v1.0.4: ~2.7s fixed per-request TTFT ...", section
// "The fix (concatenated-expert dispatch)": one launch per operator and layer instead of one
// per expert, with gate and up concatenated along the weight dimension.
//
// Orientation: the weights are the MMA's M operand (128 rows per tile) and an expert's tokens
// its N operand (N = the expert's row count rounded up to 16, at most the token tile TN <=
// 256), so an expert with 162 tokens costs one 176-wide tile instead of two 128-row tiles.
// The accumulator holds weight rows in TMEM lanes and tokens in columns. Gate and up rows are
// interleaved in pairs (row 2i = gate channel i, row 2i+1 = up channel i), so SiLU(gate)*up
// is formed by one lane-pair exchange.
//
// int8 weights stay int8 in HBM (half the bytes of fp16): TMA brings each 128 x 64 int8 weight
// tile into shared memory (64-byte swizzle), and four converter warps widen it to the fp16
// 128-byte-swizzled tile the MMA reads. The widening is exact: byte v+128 becomes the fp16
// bit pattern 0x6400|(v+128) = 1024 + v + 128, and subtracting 1152 leaves v. Token rows are
// already fp16 integers (written by the permutation step / requantisation) and go straight
// from TMA (64-row boxes, 128-byte swizzle) to the MMA: widening them in shared memory too
// would triple the shared-memory traffic of a k-block (measured slower).
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
// Warp roles (448 threads, one CTA per SM):
//   warps 0-7   epilogue: warp w reads TMEM lanes 32*(w%4).. (weight rows) and every other
//               16-column chunk (tokens) starting at chunk w/4;
//   warps 8-11  converters: thread r widens weight row r of each k-block;
//   warp 12     TMA producer: int8 weight tile and fp16 token tile;
//   warp 13     MMA issuer and TMEM owner.
// Pipeline: 4 load stages (int8 weights + fp16 tokens, released by the MMA's commit) and 2
// fp16 weight buffers (released by the MMA's commit). Every mbarrier wait is bounded; a wait
// that runs out sets the plan's error word and the CTA drains its own copies and MMAs, frees
// TMEM and returns.
//
// The down epilogue writes w * dequant(acc) per (row, channel) to yd; combine_kernel sums each
// token's k routed rows and its shared-expert row in slot order (deterministic, no atomics).
#include "common.cuh"
#include "internal.h"

namespace moe {

#ifndef MOE_LOAD_STAGES
#define MOE_LOAD_STAGES 4
#endif
constexpr int kTokBox = kTokenBox;                   // token rows per TMA box
constexpr int kXBytesMax = kMaxTokTile * kBK * 2;    // fp16 token tile per stage (<= 32 KB)
constexpr int kW8Bytes = kBM * kBK;                  // int8 weight tile per stage (8 KB)
constexpr int kLoadStage = kXBytesMax + kW8Bytes;    // 40 KB
constexpr int kLoadStages = MOE_LOAD_STAGES;
constexpr int kW16Bytes = kBM * kBK * 2;             // fp16 weight tile (16 KB)
constexpr int kConvBufs = 2;
constexpr int kEpiWarps = 8;
constexpr int kConvWarps = 4;
constexpr int kOffConv = kLoadStages * kLoadStage;
constexpr int kOffBar = kOffConv + kConvBufs * kW16Bytes;
constexpr int kBarBytes = 256;
constexpr int kGemmSmem = kOffBar + kBarBytes + 1024;
static_assert((2 * kLoadStages + 2 * kConvBufs + 5) * 8 + 8 <= kBarBytes, "barrier area");
static_assert(kGemmSmem <= 232448, "shared memory");

constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kConvThreads = kConvWarps * 32;        // one thread per weight row
constexpr int kConvWarp0 = kEpiWarps;
constexpr int kProducerWarp = kEpiWarps + kConvWarps;
constexpr int kMmaWarp = kProducerWarp + 1;
constexpr int kGemmThreads = (kMmaWarp + 1) * 32;
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

// Gate/up epilogue. Lane pair (2i, 2i+1) of quadrant q holds gate and up of channel
// m0/2 + 16q + i for every token column; the even lane finishes columns 0-7 of each 16-column
// chunk and the odd lane columns 8-15.
__device__ __forceinline__ void epilogue_gate_up(const GemmArgs& a, int4 wi, int nch,
                                                 uint32_t tbase, int half) {
  const int lane = threadIdx.x & 31, q = (threadIdx.x >> 5) & 3;
  const bool odd = lane & 1;
  const bool shared = wi.x == a.E;
  const int ch = (wi.w >> 1) + q * 16 + (lane >> 1);
  const float sgc = (shared ? a.sh_s_g : a.s_g + (size_t)wi.x * a.I)[ch];
  const float suc = (shared ? a.sh_s_u : a.s_u + (size_t)wi.x * a.I)[ch];
  const int ncols = wi.z;
#pragma unroll 1
  for (int c0 = half * 16; c0 < ncols; c0 += 32) {
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
  }
}

// Down epilogue: lane = output channel m0 + 32q + lane; for each token column the warp stores
// w * dequant(acc) for 32 consecutive channels of that row of yd (one 128-byte store). The
// combine kernel then sums each token's rows in slot order.
__device__ __forceinline__ void epilogue_down(const GemmArgs& a, int4 wi, int nch, uint32_t tbase,
                                              int half) {
  const int lane = threadIdx.x & 31, q = (threadIdx.x >> 5) & 3;
  const bool shared = wi.x == a.E;
  const int o = wi.w + q * 32 + lane;
  const float sdo = (shared ? a.sh_s_d : a.s_d + (size_t)wi.x * a.H)[o];
  const int ncols = wi.z;
#pragma unroll 1
  for (int c0 = half * 16; c0 < ncols; c0 += 32) {
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
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int col = c0 + i;
      if (col < ncols) {
        const int row = wi.y + col;
        a.yd[(size_t)row * a.H + o] = __fmul_rn(a.row_w[row], dequant(v[i], a.s_h[row], sdo));
        if (a.tap) a.tap[(size_t)row * a.H + o] = v[i];
      }
    }
  }
}

template <bool GU>
__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_kernel(const GemmArgs a, const __grid_constant__ CUtensorMap tmX,
                        const __grid_constant__ CUtensorMap tmW,
                        const __grid_constant__ CUtensorMap tmWs) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* empty = full + kLoadStages;
  uint64_t* cfull = empty + kLoadStages;   // [kConvBufs]
  uint64_t* cempty = cfull + kConvBufs;    // [kConvBufs]
  uint64_t* acc_full = cempty + kConvBufs; // [2]
  uint64_t* acc_empty = acc_full + 2;      // [2]
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kLoadStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < kConvBufs; ++s) {
      mbar_init(&cfull[s], kConvThreads);
      mbar_init(&cempty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], kEpiThreads);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmWs);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_items = *a.n_items;
  // Accumulator layout for this launch: one accumulator over the whole K (two TMEM slots,
  // double-buffered) when the bound proves it exact, else 1024-K chunks (the host sizes the
  // token tile so that the chunks of one tile fit the 512 columns).
  const bool single = single_accumulator_exact(a);
  const int kmax = a.K_r > a.K_s ? a.K_r : a.K_s;
  const int slot_cols = single ? a.TN : ((kmax + kChunkK - 1) / kChunkK) * a.TN;
  const int nslots = slot_cols <= (int)kTmemCols / 2 ? 2 : 1;
  const int kpc = single ? (1 << 30) : kChunkK / kBK;  // k-blocks per accumulator

  if (warp == kProducerWarp) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_par = 0;  // stages with a load issued, and its phase
      bool ok = true;
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        const int4 wi = a.items[item];
        const bool shared = wi.x == a.E;
        const int nkb = (shared ? a.K_s : a.K_r) / kBK;
        const int nbox = (wi.z + kTokBox - 1) / kTokBox;
        const uint32_t bytes = kW8Bytes + nbox * kTokBox * kBK * 2;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, a.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], bytes);
          uint8_t* sx = smem + stage * kLoadStage;
          uint8_t* sw = sx + kXBytesMax;
          if (shared)
            tma_load_2d(sw, &tmWs, &full[stage], kb * kBK, wi.w);
          else
            tma_load_3d(sw, &tmW, &full[stage], kb * kBK, wi.w, wi.x);
          for (int b = 0; b < nbox; ++b)
            tma_load_2d(sx + b * kTokBox * kBK * 2, &tmX, &full[stage], kb * kBK, wi.y + b * kTokBox);
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          if (++stage == kLoadStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        // Let every copy this thread issued land before the CTA exits.
        for (int s = 0; s < kLoadStages; ++s) {
          if (!(armed >> s & 1)) continue;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(&full[s], (armed_par >> s) & 1) &&
                 globaltimer_ns() - t0 < 100000000ull) {
          }
        }
      }
    }
  } else if (warp >= kConvWarp0 && warp < kConvWarp0 + kConvWarps) {
    // ---------------- converters: int8 -> fp16 weight rows ----------------
    const int r = threadIdx.x - kConvWarp0 * 32;  // weight row within the tile
    const int sw8 = (r >> 1) & 3;                 // 64-byte swizzle of the int8 row
    const int sw16 = r & 7;                       // 128-byte swizzle of the fp16 row
    int stage = 0, cb = 0;
    uint32_t phase = 0, cphase = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      const int4 wi = a.items[item];
      const int nkb = (wi.x == a.E ? a.K_s : a.K_r) / kBK;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait(&full[stage], phase, abort_flag, a.err) ||
            !mbar_wait(&cempty[cb], cphase ^ 1, abort_flag, a.err)) {
          ok = false;
          break;
        }
        const uint8_t* src = smem + stage * kLoadStage + kXBytesMax + r * 64;
        uint8_t* dst = smem + kOffConv + cb * kW16Bytes + r * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(src + 16 * (c ^ sw8));
          const uint2 e0 = widen4(v.x), e1 = widen4(v.y), e2 = widen4(v.z), e3 = widen4(v.w);
          *reinterpret_cast<uint4*>(dst + 16 * ((2 * c) ^ sw16)) = make_uint4(e0.x, e0.y, e1.x, e1.y);
          *reinterpret_cast<uint4*>(dst + 16 * ((2 * c + 1) ^ sw16)) = make_uint4(e2.x, e2.y, e3.x, e3.y);
        }
        fence_proxy_async_smem();
        mbar_arrive(&cfull[cb]);
        if (++stage == kLoadStages) {
          stage = 0;
          phase ^= 1;
        }
        if (++cb == kConvBufs) {
          cb = 0;
          cphase ^= 1;
        }
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      int stage = 0, cb = 0;
      uint32_t phase = 0, cphase = 0;
      bool ok = true;
      int it = 0;
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x, ++it) {
        const int4 wi = a.items[item];
        const int nkb = (wi.x == a.E ? a.K_s : a.K_r) / kBK;
        const int n_mma = (wi.z + 15) & ~15;
        const uint32_t idesc = idesc_f16_f32(kBM, n_mma);
        const int slot = it % nslots;
        const uint32_t use = (uint32_t)(it / nslots) & 1u;
        if (!mbar_wait(&acc_empty[slot], use ^ 1, abort_flag, a.err)) break;
        tc_fence_after();
        const uint32_t tslot = tmem + (uint32_t)(slot * slot_cols);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, a.err) ||
              !mbar_wait(&cfull[cb], cphase, abort_flag, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dw = smem_desc_sw128(smem_u32(smem + kOffConv + cb * kW16Bytes));
          const uint64_t dx = smem_desc_sw128(smem_u32(smem + stage * kLoadStage));
          const uint32_t dt = tslot + (uint32_t)((kb / kpc) * a.TN);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_f16(dt, dw + 2 * kk, dx + 2 * kk, idesc, (kb % kpc != 0 || kk != 0) ? 1u : 0u);
          umma_commit(&empty[stage]);
          umma_commit(&cempty[cb]);
          if (++stage == kLoadStages) {
            stage = 0;
            phase ^= 1;
          }
          if (++cb == kConvBufs) {
            cb = 0;
            cphase ^= 1;
          }
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
  } else if (warp < kEpiWarps) {
    // ---------------- epilogue (warps 0-7) ----------------
    const int half = warp / 4;
    const uint32_t lane_base = tmem + ((uint32_t)((warp % 4) * 32) << 16);
    int it = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++it) {
      const int4 wi = a.items[item];
      const int K = wi.x == a.E ? a.K_s : a.K_r;
      const int nch = single ? 1 : (K + kChunkK - 1) / kChunkK;
      const int slot = it % nslots;
      const uint32_t use = (uint32_t)(it / nslots) & 1u;
      if (!mbar_wait(&acc_full[slot], use, abort_flag, a.err)) break;
      tc_fence_after();
      const uint32_t tbase = lane_base + (uint32_t)(slot * slot_cols);
      if (GU)
        epilogue_gate_up(a, wi, nch, tbase, half);
      else
        epilogue_down(a, wi, nch, tbase, half);
      tc_fence_before();
      mbar_arrive(&acc_empty[slot]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

cudaError_t gemm_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(grouped_gemm_kernel<false>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
}

cudaError_t launch_grouped_gemm(bool gate_up, const GemmArgs& a, const CUtensorMap& tmX,
                                const CUtensorMap& tmW, const CUtensorMap& tmWs, int grid,
                                cudaStream_t s) {
  if (gate_up)
    grouped_gemm_kernel<true><<<grid, kGemmThreads, kGemmSmem, s>>>(a, tmX, tmW, tmWs);
  else
    grouped_gemm_kernel<false><<<grid, kGemmThreads, kGemmSmem, s>>>(a, tmX, tmW, tmWs);
  return cudaGetLastError();
}

// y[t] = sum over slots j of yd[row(t, j)] + yd[t] (shared expert row), in slot order. Block per
// token, 8 consecutive channels per thread and pass.
__global__ void combine_kernel(const float* __restrict__ yd, const int* __restrict__ slot_row,
                               int T, int k, int H, int has_shared, float* __restrict__ y) {
  const int t = blockIdx.x;
  __shared__ int rows[9];
  if (threadIdx.x < k) rows[threadIdx.x] = slot_row[(size_t)t * k + threadIdx.x];
  if (threadIdx.x == k) rows[k] = has_shared ? t : -1;
  __syncthreads();
  for (int c = threadIdx.x * 4; c < H; c += blockDim.x * 4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j <= k; ++j) {
      const int r = rows[j];
      if (r < 0) continue;
      const float4 v = *reinterpret_cast<const float4*>(yd + (size_t)r * H + c);
      acc.x = __fadd_rn(acc.x, v.x);
      acc.y = __fadd_rn(acc.y, v.y);
      acc.z = __fadd_rn(acc.z, v.z);
      acc.w = __fadd_rn(acc.w, v.w);
    }
    *reinterpret_cast<float4*>(y + (size_t)t * H + c) = acc;
  }
}

cudaError_t launch_combine(const float* yd, const int* slot_row, int T, int k, int H,
                           int has_shared, float* y, cudaStream_t s) {
  combine_kernel<<<T, 256, 0, s>>>(yd, slot_row, T, k, H, has_shared, y);
  return cudaGetLastError();
}

// Per-row requantisation of h = SiLU(gate)*up: s = amax/127, q = rne(h/s) (|q| <= 127),
// written as fp16 integers for the down GEMM's token operand. One warp per row.
__global__ void requant_kernel(const float* __restrict__ h32, int R, int T_sh, int I, int Is,
                               int Imax, __half* __restrict__ hq, float* __restrict__ sh,
                               int* __restrict__ sq_max) {
  constexpr int kRegV = 8;  // float4 per lane held in registers: rows up to 1024 values
  __shared__ int s_sq[32];
  const int row = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  int sq = 0;
  if (row < R) {
    const int n = row < T_sh ? Is : I;
    const float* h = h32 + (size_t)row * Imax;
    __half* q = hq + (size_t)row * Imax;
    if (n <= 128 * kRegV) {
      float4 v[kRegV];
#pragma unroll
      for (int j = 0; j < kRegV; ++j)
        v[j] = lane * 4 + j * 128 < n ? *reinterpret_cast<const float4*>(h + lane * 4 + j * 128)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
      float amax = 0.0f;
#pragma unroll
      for (int j = 0; j < kRegV; ++j)
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)), fmaxf(fabsf(v[j].z), fabsf(v[j].w))));
      amax = warp_max(amax);
      const float s = __fdiv_rn(amax, 127.0f);
#pragma unroll
      for (int j = 0; j < kRegV; ++j) {
        const int i = lane * 4 + j * 128;
        if (i >= n) break;
        int c[4] = {0, 0, 0, 0};
        if (s > 0.0f) {
          c[0] = quant_code(v[j].x, s);
          c[1] = quant_code(v[j].y, s);
          c[2] = quant_code(v[j].z, s);
          c[3] = quant_code(v[j].w, s);
        }
        sq += c[0] * c[0] + c[1] * c[1] + c[2] * c[2] + c[3] * c[3];
        *reinterpret_cast<__half2*>(q + i) = __halves2half2(__int2half_rn(c[0]), __int2half_rn(c[1]));
        *reinterpret_cast<__half2*>(q + i + 2) = __halves2half2(__int2half_rn(c[2]), __int2half_rn(c[3]));
      }
      if (lane == 0) sh[row] = s;
    } else {
      float amax = 0.0f;
      for (int i = lane * 4; i < n; i += 128) {
        const float4 v = *reinterpret_cast<const float4*>(h + i);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
      }
      amax = warp_max(amax);
      const float s = __fdiv_rn(amax, 127.0f);
      for (int i = lane * 4; i < n; i += 128) {
        const float4 v = *reinterpret_cast<const float4*>(h + i);
        int c[4] = {0, 0, 0, 0};
        if (s > 0.0f) {
          c[0] = quant_code(v.x, s);
          c[1] = quant_code(v.y, s);
          c[2] = quant_code(v.z, s);
          c[3] = quant_code(v.w, s);
        }
        sq += c[0] * c[0] + c[1] * c[1] + c[2] * c[2] + c[3] * c[3];
        *reinterpret_cast<__half2*>(q + i) = __halves2half2(__int2half_rn(c[0]), __int2half_rn(c[1]));
        *reinterpret_cast<__half2*>(q + i + 2) = __halves2half2(__int2half_rn(c[2]), __int2half_rn(c[3]));
      }
      if (lane == 0) sh[row] = s;
    }
    sq = warp_sum_i(sq);
  }
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
  const int rows_per_blk = 16;
  requant_kernel<<<(R + rows_per_blk - 1) / rows_per_blk, 32 * rows_per_blk, 0, s>>>(
      h32, R, T_sh, I, Is, Imax, hq, sh, sq_max);
  return cudaGetLastError();
}

}  // namespace moe
