// Weight packing for the tensor-core path (gate/up rows interleaved in channel pairs, row
// sum-of-squares maxima), and the steps around the layer in a stacked prefill (router
// projection, RMS pre-norm and the bf16 residual update).
#include "common.cuh"
#include "internal.h"

namespace moe {

// max over rows of sum(q^2) of an int8 matrix [rows, cols], into *out (atomicMax). Warp per
// row; cols a multiple of 16.
__global__ void row_sq_max_kernel(const int8_t* __restrict__ w, size_t rows, int cols,
                                  int* __restrict__ out) {
  const size_t nwarps = (size_t)gridDim.x * (blockDim.x / 32);
  const int lane = threadIdx.x % 32;
  for (size_t r = blockIdx.x * (size_t)(blockDim.x / 32) + threadIdx.x / 32; r < rows; r += nwarps) {
    const int4* p = reinterpret_cast<const int4*>(w + r * cols);
    int sq = 0;
    for (int u = lane; u < cols / 16; u += 32) {
      const int4 v = p[u];
      sq = __dp4a(v.x, v.x, sq);
      sq = __dp4a(v.y, v.y, sq);
      sq = __dp4a(v.z, v.z, sq);
      sq = __dp4a(v.w, v.w, sq);
    }
    sq = warp_sum_i(sq);
    if (lane == 0) atomicMax(out, sq);
  }
}

cudaError_t launch_row_sq_max(const int8_t* w, size_t rows, int cols, int* out, cudaStream_t s) {
  row_sq_max_kernel<<<1216, 256, 0, s>>>(w, rows, cols, out);
  return cudaGetLastError();
}

// int8 gate/up rows interleaved in pairs (row 2i = gate channel i, row 2i+1 = up channel i),
// 16 bytes per thread.
__global__ void pack_gu8_kernel(const int8_t* __restrict__ gate, const int8_t* __restrict__ up,
                                int n_mats, int I, int H, int8_t* __restrict__ out) {
  const size_t n16 = (size_t)n_mats * 2 * I * H / 16;
  for (size_t v = blockIdx.x * (size_t)blockDim.x + threadIdx.x; v < n16;
       v += (size_t)gridDim.x * blockDim.x) {
    const size_t el = v * 16;
    const int h = (int)(el % H);
    const size_t prow = el / H;
    const int m = (int)(prow / (2 * I));
    const int p = (int)(prow % (2 * I));
    const int8_t* src = ((p & 1) ? up : gate) + ((size_t)m * I + (p >> 1)) * H + h;
    *reinterpret_cast<int4*>(out + el) = *reinterpret_cast<const int4*>(src);
  }
}

cudaError_t launch_pack_gu8(const int8_t* gate, const int8_t* up, int n_mats, int I, int H,
                            int8_t* out, cudaStream_t s) {
  pack_gu8_kernel<<<1216, 256, 0, s>>>(gate, up, n_mats, I, H, out);
  return cudaGetLastError();
}

// logits[T, E] = float(x[T, H]) @ wr[H, E] in fp32. 64x64 output tile per block, 16-deep K
// slices through shared memory, 4x4 outputs per thread.
__global__ void __launch_bounds__(256) router_logits_kernel(const uint16_t* __restrict__ x,
                                                            const float* __restrict__ wr, int T,
                                                            int H, int E, float* __restrict__ out) {
  pdl_wait();  // the predecessor on the stream (launched with launch_pdl)
  pdl_trigger();
  __shared__ float As[16][64 + 4];
  __shared__ __align__(16) float Bs[16][64];
  const int t0 = blockIdx.y * 64, e0 = blockIdx.x * 64;
  const int tid = threadIdx.x;
  const int ty = tid / 16, tx = tid % 16;
  float acc[4][4] = {};
  const int la_row = tid / 4, la_k = (tid % 4) * 4;   // A: 64 rows x 16 k, 4 per thread
  const int lb_k = tid / 16, lb_c = (tid % 16) * 4;   // B: 16 k x 64 cols, 4 per thread
  for (int k0 = 0; k0 < H; k0 += 16) {
    {
      const int t = t0 + la_row;
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (t < T) {
        const uint2 raw = *reinterpret_cast<const uint2*>(x + (size_t)t * H + k0 + la_k);
        v[0] = bf16_bits_to_float((uint16_t)(raw.x & 0xffffu));
        v[1] = bf16_bits_to_float((uint16_t)(raw.x >> 16));
        v[2] = bf16_bits_to_float((uint16_t)(raw.y & 0xffffu));
        v[3] = bf16_bits_to_float((uint16_t)(raw.y >> 16));
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) As[la_k + i][la_row] = v[i];
    }
    {
      const int c = e0 + lb_c;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c + 3 < E) {
        v = *reinterpret_cast<const float4*>(wr + (size_t)(k0 + lb_k) * E + c);
      } else {
        float* pv = reinterpret_cast<float*>(&v);
        for (int i = 0; i < 4; ++i)
          if (c + i < E) pv[i] = wr[(size_t)(k0 + lb_k) * E + c + i];
      }
      *reinterpret_cast<float4*>(&Bs[lb_k][lb_c]) = v;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = e0 + tx * 4 + j;
      if (c < E) out[(size_t)t * E + c] = acc[i][j];
    }
  }
}

cudaError_t launch_router_logits(const uint16_t* x, const float* wr, int T, int H, int E,
                                 float* out, cudaStream_t s) {
  const dim3 grid((E + 63) / 64, (T + 63) / 64);
  return launch_pdl(router_logits_kernel, grid, dim3(256), 0, s, x, wr, T, H, E, out);
}

__global__ void residual_kernel(uint16_t* __restrict__ x, const float* __restrict__ y, size_t n) {
  pdl_wait();  // the predecessor on the stream (launched with launch_pdl)
  pdl_trigger();
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n / 4;
       i += (size_t)gridDim.x * blockDim.x) {
    const float4 yv = reinterpret_cast<const float4*>(y)[i];
    uint2 xv = reinterpret_cast<uint2*>(x)[i];
    const float f[4] = {bf16_bits_to_float((uint16_t)(xv.x & 0xffffu)) + yv.x,
                        bf16_bits_to_float((uint16_t)(xv.x >> 16)) + yv.y,
                        bf16_bits_to_float((uint16_t)(xv.y & 0xffffu)) + yv.z,
                        bf16_bits_to_float((uint16_t)(xv.y >> 16)) + yv.w};
    uint16_t b[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat16 h = __float2bfloat16_rn(f[j]);
      b[j] = *reinterpret_cast<const uint16_t*>(&h);
    }
    xv.x = (uint32_t)b[0] | ((uint32_t)b[1] << 16);
    xv.y = (uint32_t)b[2] | ((uint32_t)b[3] << 16);
    reinterpret_cast<uint2*>(x)[i] = xv;
  }
}

__device__ __forceinline__ uint16_t f2bf(float f) {
  const __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<const uint16_t*>(&h);
}

// Block per token: optional residual update of x, then the RMS-normalised copy x_in.
__global__ void rmsnorm_residual_kernel(uint16_t* __restrict__ x, const float* __restrict__ y,
                                        uint16_t* __restrict__ x_in, int H) {
  pdl_wait();  // the predecessor on the stream (launched with launch_pdl)
  pdl_trigger();
  const int t = blockIdx.x;
  uint16_t* xr = x + (size_t)t * H;
  __shared__ float red[32];
  float ss = 0.0f;
  for (int c = threadIdx.x * 4; c < H; c += blockDim.x * 4) {
    uint2 xv = *reinterpret_cast<const uint2*>(xr + c);
    float f[4] = {bf16_bits_to_float((uint16_t)(xv.x & 0xffffu)), bf16_bits_to_float((uint16_t)(xv.x >> 16)),
                  bf16_bits_to_float((uint16_t)(xv.y & 0xffffu)), bf16_bits_to_float((uint16_t)(xv.y >> 16))};
    if (y) {
      const float4 yv = *reinterpret_cast<const float4*>(y + (size_t)t * H + c);
      const float yy[4] = {yv.x, yv.y, yv.z, yv.w};
      uint16_t b[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        b[j] = f2bf(f[j] + yy[j]);
        f[j] = bf16_bits_to_float(b[j]);
      }
      xv.x = (uint32_t)b[0] | ((uint32_t)b[1] << 16);
      xv.y = (uint32_t)b[2] | ((uint32_t)b[3] << 16);
      *reinterpret_cast<uint2*>(xr + c) = xv;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) ss = fmaf(f[j], f[j], ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < blockDim.x / 32 ? red[threadIdx.x] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float rms = __fsqrt_rn(__fadd_rn(__fdiv_rn(red[0], (float)H), 1e-6f));
  for (int c = threadIdx.x * 4; c < H; c += blockDim.x * 4) {
    const uint2 xv = *reinterpret_cast<const uint2*>(xr + c);
    const float f[4] = {bf16_bits_to_float((uint16_t)(xv.x & 0xffffu)), bf16_bits_to_float((uint16_t)(xv.x >> 16)),
                        bf16_bits_to_float((uint16_t)(xv.y & 0xffffu)), bf16_bits_to_float((uint16_t)(xv.y >> 16))};
    uint2 o;
    o.x = (uint32_t)f2bf(__fdiv_rn(f[0], rms)) | ((uint32_t)f2bf(__fdiv_rn(f[1], rms)) << 16);
    o.y = (uint32_t)f2bf(__fdiv_rn(f[2], rms)) | ((uint32_t)f2bf(__fdiv_rn(f[3], rms)) << 16);
    *reinterpret_cast<uint2*>(x_in + (size_t)t * H + c) = o;
  }
}

cudaError_t launch_rmsnorm_residual(uint16_t* x, const float* y, uint16_t* x_in, int T, int H,
                                    cudaStream_t s) {
  return launch_pdl(rmsnorm_residual_kernel, dim3(T), dim3(256), 0, s, x, y, x_in, H);
}

cudaError_t launch_residual(uint16_t* x, const float* y, size_t n, cudaStream_t s) {
  return launch_pdl(residual_kernel, dim3(1216), dim3(256), 0, s, x, y, n);
}

// Self-test of the bounded waits: one thread waits, with the kernels' own bounded wait, on
// an mbarrier that nothing ever arrives on. The wait gives up after its time limit and
// records MOE_ERR_TIMEOUT in `err`; nothing is in flight when the kernel returns.
__global__ void selftest_wait_kernel(int* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, err);
}

cudaError_t launch_selftest_wait(int* err, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(err);
  return cudaGetLastError();
}

}  // namespace moe
