// Router projection of the stacked prefill on the tensor cores.
//
// logits[T, E] = x[T, H] (bf16) @ W[H, E] (fp32). The fp32 weight splits exactly enough into
// three bf16 parts, W = hi + mid + lo (hi = bf16(W), mid = bf16(W - hi), lo = bf16(W - hi -
// mid); the residual after lo is below 2^-26 |W|), so the product is one bf16 GEMM with the
// reduction dimension tripled: [x | x | x] @ [hi; mid; lo]. Every bf16 x bf16 product is exact
// and the tensor core accumulates in fp32, so the result has the accuracy of an fp32 dot
// product. One CTA per 128-row x 64-expert tile; warp 4 feeds A (x, re-read for each part)
// and B (packed [E, 3H] bf16) by TMA into an 8-stage ring, warp 5 issues tcgen05.mma
// (kind::f16, bf16 inputs), warps 0-3 drain TMEM and store fp32 rows.
#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kRBN = 64;
constexpr int kRStages = 8;
constexpr int kRA = kBM * kBK * 2;
constexpr int kRB = kRBN * kBK * 2;
constexpr int kRStage = kRA + kRB;
constexpr int kRSmem = kRStages * kRStage + 256 + 1024;

__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__global__ void __launch_bounds__(192, 1)
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
  const int m0 = blockIdx.x * kBM, n0 = blockIdx.y * kRBN;
  const int nkb = 3 * H / kBK;
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
    tmem_alloc(tmem_slot, kRBN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
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
        tma_load_2d(sa, &tmA, &full[stage], (kb * kBK) % H, m0);
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
#pragma unroll
      for (int c = 0; c < kRBN; c += 16) {
        uint32_t r[16];
        tmem_ld16(tb + c, r);
        tmem_ld_wait();
        if (row < T) {
          float4* dst = reinterpret_cast<float4*>(out + (size_t)row * E + n0 + c);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[q] = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                 __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kRBN);
  }
}

__device__ __forceinline__ uint16_t bf16_rn_bits(float f) {
  const __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<const uint16_t*>(&h);
}

// packed[e, p*H + h] = part p of w[h, e] (p = 0 hi, 1 mid, 2 lo)
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
    uint16_t* row = packed + (size_t)e * 3 * H;
    row[h] = hi;
    row[H + h] = mid;
    row[2 * H + h] = lo;
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
  const dim3 grid((T + kBM - 1) / kBM, E / kRBN);
  router_tc_kernel<<<grid, 192, kRSmem, s>>>(T, H, E, out, tmA, tmB);
  return cudaGetLastError();
}

}  // namespace moe
