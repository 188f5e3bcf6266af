// Router projection of the stacked prefill on the tensor cores.
//
// logits[T, E] = x[T, H] (bf16) @ W[H, E] (fp32). The fp32 weight splits exactly enough into
// three bf16 parts, W = hi + mid + lo (hi = bf16(W), mid = bf16(W - hi), lo = bf16(W - hi -
// mid); the residual after lo is below 2^-26 |W|). Every bf16 x bf16 product is exact and the
// tensor core accumulates in fp32, so x @ hi, x @ mid and x @ lo each carry the error of an
// fp32 dot product, and their sum (hi + mid) + lo that of the fp32 projection.
//
// Packed weight layout: blocks of kREB experts, each block three parts of kREB rows of H bf16
// ([E / kREB][3][kREB][H]), so one B tile of 3 * kREB rows holds all three parts of kREB
// experts and the reduction runs over H once. One CTA per 128-row x kREB-expert tile (two per
// SM); warp 4 feeds A (x) and B by TMA into a 4-stage ring, warp 5 issues tcgen05.mma
// (kind::f16, bf16 inputs, N = 3 * kREB), warps 0-3 drain TMEM, add the three parts per
// expert and store fp32 rows.
#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kRBN = 3 * kREB;  // MMA N: three parts of kREB experts
constexpr int kRStages = 4;
constexpr int kRA = kBM * kBK * 2;
constexpr int kRB = kRBN * kBK * 2;
constexpr int kRStage = kRA + kRB;
constexpr int kRSmem = kRStages * kRStage + 256 + 1024;
constexpr int kRTmemCols = 64;  // power of two >= kRBN
static_assert(kRBN <= kRTmemCols && kRBN % 16 == 0, "router tile");
static_assert(kRStage % 1024 == 0, "stages stay 1024-byte aligned for 128-byte swizzle");

__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__global__ void __launch_bounds__(192, 2)
    router_tc_kernel(int T, int H, int E, float* __restrict__ out,
                     const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kRStages * kRStage);
  uint64_t* empty = full + kRStages;
  uint64_t* acc_full = empty + kRStages;
  uint64_t* drain = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int m0 = blockIdx.x * kBM, n0 = blockIdx.y * kRBN, e0 = blockIdx.y * kREB;
  const int nkb = H / kBK;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, kRTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();  // the predecessor's results (set-up above touches no global memory)
  pdl_trigger();
  const uint32_t tmem = *tmem_slot;
  if (warp == 4) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_par = 0;
      bool ok = true;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, nullptr)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[stage], kRStage);
        uint8_t* sa = smem + stage * kRStage;
        tma_load_2d(sa, &tmA, &full[stage], kb * kBK, m0);
        tma_load_2d(sa + kRA, &tmB, &full[stage], kb * kBK, n0);
        armed |= 1u << stage;
        armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
        if (++stage == kRStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) {
        for (int s = 0; s < kRStages; ++s) {
          if (!(armed >> s & 1)) continue;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(&full[s], (armed_par >> s) & 1) &&
                 globaltimer_ns() - t0 < 100000000ull) {
          }
        }
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, kRBN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait(&full[stage], phase, abort_flag, nullptr)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + stage * kRStage);
        const uint64_t da = smem_desc_sw128(sa), db = smem_desc_sw128(sa + kRA);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          umma_f16(tmem, da + 2 * kk, db + 2 * kk, idesc, (kb != 0 || kk != 0) ? 1u : 0u);
        umma_commit(&empty[stage]);
        if (++stage == kRStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (ok) umma_commit(acc_full);
      umma_commit(drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < 100000000ull) {
      }
    }
  } else {
    if (mbar_wait(acc_full, 0, abort_flag, nullptr)) {
      tc_fence_after();
      const int row = m0 + threadIdx.x;
      const uint32_t tb = tmem + ((uint32_t)(warp * 32) << 16);
      static_assert(kREB == 16, "one 16-column TMEM load per part");
      uint32_t r[3][16];
#pragma unroll
      for (int p = 0; p < 3; ++p) tmem_ld16(tb + p * kREB, r[p]);
      tmem_ld_wait();
      if (row < T) {
        float4* dst = reinterpret_cast<float4*>(out + (size_t)row * E + e0);
#pragma unroll
        for (int q = 0; q < kREB / 4; ++q) {
          float v[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int c = 4 * q + j;
            v[j] = __fadd_rn(__fadd_rn(__uint_as_float(r[0][c]), __uint_as_float(r[1][c])),
                             __uint_as_float(r[2][c]));
          }
          dst[q] = make_float4(v[0], v[1], v[2], v[3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kRTmemCols);
  }
}

__device__ __forceinline__ uint16_t bf16_rn_bits(float f) {
  const __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<const uint16_t*>(&h);
}

// packed row ((e / kREB) * 3 + p) * kREB + e % kREB, column h = part p of w[h, e]
// (p = 0 hi, 1 mid, 2 lo)
__global__ void router_pack_kernel(const float* __restrict__ w, int H, int E,
                                   uint16_t* __restrict__ packed) {
  const size_t n = (size_t)H * E;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const int h = (int)(i / E), e = (int)(i % E);
    const float v = w[i];
    const uint16_t hi = bf16_rn_bits(v);
    const float r1 = __fsub_rn(v, bf16_bits_to_float(hi));
    const uint16_t mid = bf16_rn_bits(r1);
    const float r2 = __fsub_rn(r1, bf16_bits_to_float(mid));
    const uint16_t lo = bf16_rn_bits(r2);
    const size_t r0 = (size_t)(e / kREB) * 3 * kREB + e % kREB;
    packed[r0 * H + h] = hi;
    packed[(r0 + kREB) * H + h] = mid;
    packed[(r0 + 2 * kREB) * H + h] = lo;
  }
}

cudaError_t launch_router_pack(const float* w, int H, int E, uint16_t* packed, cudaStream_t s) {
  router_pack_kernel<<<512, 256, 0, s>>>(w, H, E, packed);
  return cudaGetLastError();
}

cudaError_t launch_router_tc(int T, int H, int E, float* out, const CUtensorMap& tmA,
                             const CUtensorMap& tmB, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(router_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmem);
  if (e != cudaSuccess) return e;
  const dim3 grid((T + kBM - 1) / kBM, E / kREB);
  return launch_pdl(router_tc_kernel, grid, dim3(192), kRSmem, s, T, H, E, out, tmA, tmB);
}

}  // namespace moe
