// Grouped W8A8 GEMMs of the prefill path on the 5th-generation tensor cores (tcgen05).
//
// One persistent kernel runs every (expert group, 128-row tile, BN-column tile) work item
// of a layer: the gate/up GEMM with a fused SiLU(gate)*up epilogue, or the down GEMM with a
// fused router-weighted scatter-combine into y. This is the concatenated-expert computation
// of the page "Qwen3.6-35B-A3B Linux v1.0.4: ~2.7s fixed per-request TTFT ...", section
// "The fix (concatenated-expert dispatch)": one launch per operator and layer instead of one
// per expert, with gate and up concatenated along N.
//
// Exact integer products on an fp16 tensor pipe. sm_103a has no int8 tcgen05 MMA, so the
// int8 operands are held as fp16 (every int8 value is an fp16 integer) and multiplied with
// kind::f16 into fp32 TMEM accumulators. fp32 holds every integer below 2^24 exactly, so a
// sum of integer products is exact as long as every partial sum stays below 2^24 in
// magnitude, in whatever order the tensor core adds them. Two ways to guarantee that:
//  - bound: for any subset of terms, |sum a_k b_k| <= sqrt(sum a^2) sqrt(sum b^2)
//    (Cauchy-Schwarz). The producers of the A rows record max_row sum(q^2) and weight packing
//    records max_row sum(q_w^2); when their product is below 2^48 one accumulator over the
//    whole K is exact. This holds for realistic data by a wide margin.
//  - chunks: otherwise a fresh accumulator per 1024-element K chunk bounds every partial
//    sum by 1024 * 127^2 < 2^24; the epilogue rounds each chunk to int32 and adds the chunks
//    in integer arithmetic.
// The kernel picks one of the two for the whole launch at its start (every CTA reads the
// same two words). With one accumulator per tile, TMEM holds two of them (2 x BN columns)
// so the epilogue of one tile overlaps the MMAs of the next.
//
// Warp roles (320 threads, one CTA per SM):
//   warps 0-7  epilogue: warp w reads TMEM lanes 32*(w%4).. (tile rows) and half (w/4) of
//              the tile's columns;
//   warp 8     TMA producer: A (token rows) and B (weight rows) tiles, 128-byte swizzle;
//   warp 9     MMA issuer and TMEM owner.
// Every mbarrier wait is bounded; a wait that runs out sets the plan's error word and the
// CTA drains its own copies and MMAs, frees TMEM and returns.
#include "common.cuh"
#include "internal.h"

namespace moe {

template <int BN>
struct GemmCfg {
  static constexpr int A_BYTES = kBM * kBK * 2;
  static constexpr int B_BYTES = BN * kBK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = (192 * 1024) / STAGE_BYTES;
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + BAR_BYTES + 1024;
  static_assert(STAGES >= 2, "pipeline depth");
  static_assert((2 * STAGES + 5) * 8 + 8 <= BAR_BYTES, "barrier area");
};

constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kProducerWarp = kEpiWarps;
constexpr int kMmaWarp = kEpiWarps + 1;
constexpr int kGemmThreads = (kEpiWarps + 2) * 32;
constexpr uint32_t kTmemCols = 512;

// Whether one fp32 accumulator over the whole K is provably exact for this launch.
__device__ __forceinline__ bool single_accumulator_exact(const GemmArgs& a) {
  const unsigned long long r = (unsigned long long)(unsigned)*a.row_sq_max;
  const unsigned long long w = (unsigned long long)(unsigned)*a.w_sq_max;
  return r * w < (1ull << 48);
}

template <int BN>
__device__ __forceinline__ void epilogue_gate_up(const GemmArgs& a, int4 wi, int nch,
                                                 uint32_t tbase, int half) {
  const int m = (threadIdx.x / 32 % 4) * 32 + threadIdx.x % 32;  // tile row = TMEM lane
  const bool valid = m < wi.z;
  const int row = wi.y + m;
  const bool shared = wi.x == a.E;
  const float* sg = shared ? a.sh_s_g : a.s_g + (size_t)wi.x * a.I;
  const float* su = shared ? a.sh_s_u : a.s_u + (size_t)wi.x * a.I;
  const int cbase = (wi.w / BN) * (BN / 2);
  const float sx = valid ? a.sx[row] : 0.0f;
  constexpr int kCols = BN / 4;  // channels per epilogue half
#pragma unroll 1
  for (int j0 = half * kCols; j0 < (half + 1) * kCols; j0 += 16) {
    int ag[16], au[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) ag[i] = au[i] = 0;
#pragma unroll 1
    for (int c = 0; c < nch; ++c) {
      uint32_t rg[16], ru[16];
      tmem_ld16(tbase + c * BN + j0, rg);
      tmem_ld16(tbase + c * BN + BN / 2 + j0, ru);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        ag[i] += __float2int_rn(__uint_as_float(rg[i]));
        au[i] += __float2int_rn(__uint_as_float(ru[i]));
      }
    }
    if (valid) {
      float hv[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int ch = cbase + j0 + i;
        hv[i] = silu_mul(dequant(ag[i], sx, sg[ch]), dequant(au[i], sx, su[ch]));
      }
      float4* dst = reinterpret_cast<float4*>(a.h32 + (size_t)row * a.Imax + cbase + j0);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        dst[q] = make_float4(hv[4 * q], hv[4 * q + 1], hv[4 * q + 2], hv[4 * q + 3]);
      if (a.tap) {
        int4* tg = reinterpret_cast<int4*>(a.tap + (size_t)row * 2 * a.Imax + cbase + j0);
        int4* tu = reinterpret_cast<int4*>(a.tap + (size_t)row * 2 * a.Imax + a.Imax + cbase + j0);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          tg[q] = make_int4(ag[4 * q], ag[4 * q + 1], ag[4 * q + 2], ag[4 * q + 3]);
          tu[q] = make_int4(au[4 * q], au[4 * q + 1], au[4 * q + 2], au[4 * q + 3]);
        }
      }
    }
  }
}

template <int BN>
__device__ __forceinline__ void epilogue_down(const GemmArgs& a, int4 wi, int nch, uint32_t tbase,
                                              int half) {
  const int m = (threadIdx.x / 32 % 4) * 32 + threadIdx.x % 32;
  const bool valid = m < wi.z;
  const int row = wi.y + m;
  const bool shared = wi.x == a.E;
  const float* sd = shared ? a.sh_s_d : a.s_d + (size_t)wi.x * a.H;
  const float shr = valid ? a.s_h[row] : 0.0f;
  const float wr = valid ? a.row_w[row] : 0.0f;
  const int tok = valid ? a.row_token[row] : 0;
  float* yrow = a.y + (size_t)tok * a.H;
  constexpr int kCols = BN / 2;
#pragma unroll 1
  for (int j0 = half * kCols; j0 < (half + 1) * kCols; j0 += 16) {
    int acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0;
#pragma unroll 1
    for (int c = 0; c < nch; ++c) {
      uint32_t r[16];
      tmem_ld16(tbase + c * BN + j0, r);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[i] += __float2int_rn(__uint_as_float(r[i]));
    }
    if (valid) {
      const int o0 = wi.w + j0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int o = o0 + 4 * q;
        red_add_v4(yrow + o, __fmul_rn(wr, dequant(acc[4 * q + 0], shr, sd[o + 0])),
                   __fmul_rn(wr, dequant(acc[4 * q + 1], shr, sd[o + 1])),
                   __fmul_rn(wr, dequant(acc[4 * q + 2], shr, sd[o + 2])),
                   __fmul_rn(wr, dequant(acc[4 * q + 3], shr, sd[o + 3])));
      }
      if (a.tap) {
        int4* t = reinterpret_cast<int4*>(a.tap + (size_t)row * a.H + o0);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          t[q] = make_int4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
      }
    }
  }
}

template <int BN, bool GU>
__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_kernel(const GemmArgs a, const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmBs) {
  using Cfg = GemmCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::STAGES * Cfg::STAGE_BYTES);
  uint64_t* empty = full + Cfg::STAGES;
  uint64_t* acc_full = empty + Cfg::STAGES;  // [2]
  uint64_t* acc_empty = acc_full + 2;        // [2]
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
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
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmBs);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_items = *a.n_items;
  // Accumulator layout for this launch: one accumulator over the whole K (two TMEM slots,
  // double-buffered) when the bound proves it exact, else 1024-K chunks in one slot.
  const bool single = single_accumulator_exact(a);
  const int kmax = a.K_r > a.K_s ? a.K_r : a.K_s;
  const int slot_cols = single ? BN : ((kmax + kChunkK - 1) / kChunkK) * BN;
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
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, a.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], Cfg::STAGE_BYTES);
          uint8_t* sa = smem + stage * Cfg::STAGE_BYTES;
          uint8_t* sb = sa + Cfg::A_BYTES;
          tma_load_2d(sa, &tmA, &full[stage], kb * kBK, wi.y);
          if (shared)
            tma_load_2d(sb, &tmBs, &full[stage], kb * kBK, wi.w);
          else
            tma_load_3d(sb, &tmB, &full[stage], kb * kBK, wi.w, wi.x);
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          if (++stage == Cfg::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        // Let every copy this thread issued land before the CTA exits.
        for (int s = 0; s < Cfg::STAGES; ++s) {
          if (!(armed >> s & 1)) continue;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(&full[s], (armed_par >> s) & 1) &&
                 globaltimer_ns() - t0 < 100000000ull) {
          }
        }
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t idesc = idesc_f16_f32(kBM, BN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x, ++it) {
        const int4 wi = a.items[item];
        const int nkb = (wi.x == a.E ? a.K_s : a.K_r) / kBK;
        const int slot = it % nslots;
        const uint32_t use = (uint32_t)(it / nslots) & 1u;
        if (!mbar_wait(&acc_empty[slot], use ^ 1, abort_flag, a.err)) break;
        tc_fence_after();
        const uint32_t tslot = tmem + (uint32_t)(slot * slot_cols);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * Cfg::STAGE_BYTES);
          const uint64_t da = smem_desc_sw128(sa);
          const uint64_t db = smem_desc_sw128(sa + Cfg::A_BYTES);
          const uint32_t dt = tslot + (uint32_t)((kb / kpc) * BN);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_f16(dt, da + 2 * kk, db + 2 * kk, idesc, (kb % kpc != 0 || kk != 0) ? 1u : 0u);
          umma_commit(&empty[stage]);
          if (++stage == Cfg::STAGES) {
            stage = 0;
            phase ^= 1;
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
  } else {
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
        epilogue_gate_up<BN>(a, wi, nch, tbase, half);
      else
        epilogue_down<BN>(a, wi, nch, tbase, half);
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

template <int BN, bool GU>
static cudaError_t set_attr() {
  return cudaFuncSetAttribute(grouped_gemm_kernel<BN, GU>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              GemmCfg<BN>::SMEM_BYTES);
}

cudaError_t gemm_set_attributes() {
  cudaError_t e;
  if ((e = set_attr<256, true>()) != cudaSuccess) return e;
  if ((e = set_attr<256, false>()) != cudaSuccess) return e;
  if ((e = set_attr<128, true>()) != cudaSuccess) return e;
  if ((e = set_attr<128, false>()) != cudaSuccess) return e;
  if ((e = set_attr<64, true>()) != cudaSuccess) return e;
  return set_attr<64, false>();
}

template <int BN, bool GU>
static cudaError_t launch_t(const GemmArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmB,
                            const CUtensorMap& tmBs, int grid, cudaStream_t s) {
  grouped_gemm_kernel<BN, GU><<<grid, kGemmThreads, GemmCfg<BN>::SMEM_BYTES, s>>>(a, tmA, tmB, tmBs);
  return cudaGetLastError();
}

cudaError_t launch_grouped_gemm(bool gate_up, int BN, const GemmArgs& a, const CUtensorMap& tmA,
                                const CUtensorMap& tmB, const CUtensorMap& tmBs, int grid,
                                cudaStream_t s) {
  switch (BN) {
    case 256:
      return gate_up ? launch_t<256, true>(a, tmA, tmB, tmBs, grid, s)
                     : launch_t<256, false>(a, tmA, tmB, tmBs, grid, s);
    case 128:
      return gate_up ? launch_t<128, true>(a, tmA, tmB, tmBs, grid, s)
                     : launch_t<128, false>(a, tmA, tmB, tmBs, grid, s);
    case 64:
      return gate_up ? launch_t<64, true>(a, tmA, tmB, tmBs, grid, s)
                     : launch_t<64, false>(a, tmA, tmB, tmBs, grid, s);
    default:
      return cudaErrorInvalidValue;
  }
}

// Per-row requantisation of h = SiLU(gate)*up: s = amax/127, q = rne(h/s) (|q| <= 127),
// written as fp16 integers for the down GEMM's A operand. One warp per row.
__global__ void requant_kernel(const float* __restrict__ h32, int R, int T_sh, int I, int Is,
                               int Imax, __half* __restrict__ hq, float* __restrict__ sh,
                               int* __restrict__ sq_max) {
  __shared__ int s_sq[32];
  const int row = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  int sq = 0;
  if (row < R) {
    const int n = row < T_sh ? Is : I;
    const float* h = h32 + (size_t)row * Imax;
    float amax = 0.0f;
    for (int i = lane * 4; i < n; i += 128) {
      const float4 v = *reinterpret_cast<const float4*>(h + i);
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    amax = warp_max(amax);
    const float s = __fdiv_rn(amax, 127.0f);
    __half* q = hq + (size_t)row * Imax;
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
      *reinterpret_cast<__half2*>(q + i + 2) =
          __halves2half2(__int2half_rn(c[2]), __int2half_rn(c[3]));
    }
    sq = warp_sum_i(sq);
    if (lane == 0) sh[row] = s;
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
