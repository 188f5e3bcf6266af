// Routing and the token-by-expert permutation of the prefill path.
//
//  route_kernel      warp per token: top-k of the fp32 logits (ties to the lowest expert id),
//                    softmax over the selected logits.
//  route_hist_scan_kernel
//                    per block of 32 tokens: the tokens' routing (when logits are given), one
//                    64-bit token mask per expert (which of the block's tokens chose it; its
//                    popcount is the block's histogram); the last block to finish runs the
//                    scan: per-expert counts, exclusive prefixes over blocks and over experts,
//                    and each group's base in the grouped-GEMM work lists.
//  scatter_kernel    block per token: per-token int8 quantisation of x, the codes written as
//                    fp16 integers into every row the token occupies (one per routed slot plus
//                    the shared expert's row) with 16-byte stores; row metadata; the token's
//                    row of y zeroed (the down GEMM adds every row's output into it); and the
//                    work items (expert-tile queue) of one group per block.
// Row order: the shared expert's rows [0, T) first (row t = token t), then the routed
// assignments grouped by expert id and, inside an expert, by token. This is the order a
// stable sort of the flattened idx by expert id gives.
#include "common.cuh"
#include "internal.h"

namespace moe {

__global__ void route_kernel(const float* __restrict__ logits, int T, int E, int k,
                             int32_t* __restrict__ idx, float* __restrict__ w, int* err) {
  pdl_wait();  // the predecessor on the stream (launched with launch_pdl)
  pdl_trigger();
  const int t = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (t >= T) return;
  route_token_warp(logits + (size_t)t * E, E, k, idx + (size_t)t * k, w + (size_t)t * k, lane);
}

cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* idx, float* w,
                         int* err, cudaStream_t s) {
  const int warps = 8;
  return launch_pdl(route_kernel, dim3((T + warps - 1) / warps), dim3(32 * warps), 0, s, logits, T,
                    E, k, idx, w, err);
}

// Exclusive scan over up to blockDim.x (<= 1024) values, one per thread; returns the
// exclusive prefix and writes the total to *total. Every thread of the block must call it.
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) s_warp[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int wv = lane < nw ? s_warp[lane] : 0;
    int winc = wv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, winc, o);
      if (lane >= o) winc += n;
    }
    if (lane < nw) s_warp[lane] = winc - wv;
    if (lane == 31) s_warp[32] = winc;
  }
  __syncthreads();
  const int r = s_warp[warp] + inc - v;
  *total = s_warp[32];
  __syncthreads();
  return r;
}

// The last block of route_hist_scan_kernel (1024 threads). Turns bhist into exclusive
// per-expert prefixes over blocks,
// writes counts/offsets and the two work lists (gate/up and down): per group, every
// (128-row weight tile, token tile) pair, ordered by group, then weight tile, then token tile,
// so consecutive items of a large group reuse one weight tile from L2. A group of cnt rows is
// split into ceil(cnt / TN) token tiles of equal size (within one row), so no tile is a thin
// remainder.
__device__ __forceinline__ void scan_block(const PrepArgs& a, int nblk) {
  __shared__ int s_cnt[257];
  __shared__ int s_base[4][258];
  __shared__ int s_warp[33];
  const int E = a.E;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, nwarps = blockDim.x / 32;
  // exclusive prefix over blocks of each expert's histogram (row e of [E][nblk]), warp per
  // expert; a warp takes its experts kSE at a time with all their loads issued together
  // (128 blocks per pass), so the load latency is paid once per pass, not once per expert
  constexpr int kSE = 4;
  for (int e0 = warp; e0 < E; e0 += nwarps * kSE) {
    int carry[kSE];
#pragma unroll
    for (int x = 0; x < kSE; ++x) carry[x] = 0;
    for (int b0 = 0; b0 < nblk; b0 += 128) {
      int v[kSE][4];
#pragma unroll
      for (int x = 0; x < kSE; ++x) {
        const int e = e0 + x * nwarps;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int b = b0 + i * 32 + lane;
          v[x][i] = e < E && b < nblk ? __ldcg(a.bhist + (size_t)e * nblk + b) : 0;
        }
      }
#pragma unroll
      for (int x = 0; x < kSE; ++x) {
        const int e = e0 + x * nwarps;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          int incl = v[x][i];
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
          }
          const int b = b0 + i * 32 + lane;
          if (e < E && b < nblk) a.bhist[(size_t)e * nblk + b] = carry[x] + incl - v[x][i];
          carry[x] += __shfl_sync(0xffffffffu, incl, 31);
        }
      }
    }
#pragma unroll
    for (int x = 0; x < kSE; ++x) {
      const int e = e0 + x * nwarps;
      if (lane == 0 && e < E) {
        s_cnt[e] = carry[x];
        a.counts[e] = carry[x];
      }
    }
  }
  __syncthreads();
  // row offsets of the experts, and item bases of the groups (group g: shared when
  // g < has_shared, else expert g - has_shared)
  const int ng = E + (a.has_shared ? 1 : 0);
  int total;
  const int ecnt = (int)threadIdx.x < E ? s_cnt[threadIdx.x] : 0;
  const int eoff = block_exclusive_scan(ecnt, s_warp, &total);
  if ((int)threadIdx.x < E) {
    a.offsets[threadIdx.x] = eoff;
  }
  if (threadIdx.x == 0) a.offsets[E] = total;
  // item counts of every group in each work list (l = 0 gate/up, 1 down, 2 and 3 the same
  // in the chunked accumulation's token tiles), their exclusive prefixes = the groups' bases
  const int g = threadIdx.x;
#pragma unroll
  for (int l = 0; l < 4; ++l) {  // unrolled: the parameter arrays are indexed by constants
    if (!a.items[l]) continue;  // uniform over the block
    int n = 0;
    if (g < ng) {
      const bool sh = a.has_shared && g == 0;
      const int cnt = sh ? a.T : s_cnt[g - a.has_shared];
      const int nwt = l % 2 == 0 ? 2 * (sh ? a.Is : a.I) / kBM : a.H / kBM;
      n = nwt * ((cnt + a.tn[l] - 1) / a.tn[l]);
    }
    const int base = block_exclusive_scan(n, s_warp, &total);
    if (g < ng) s_base[l][g] = base;
    if (threadIdx.x == 0) {
      s_base[l][ng] = total;
      a.n_items[l] = total;
    }
  }
  __syncthreads();
  // the item bases of the groups; the scatter kernel writes the items from them
#pragma unroll
  for (int l = 0; l < 4; ++l) {
    if (!a.items[l]) continue;
    for (int i = threadIdx.x; i <= ng; i += blockDim.x) a.gbase[l * (kMaxGroups + 1) + i] = s_base[l][i];
  }
}

// (t * cnt) / tt for 0 <= t <= tt, in 32-bit arithmetic when the product fits.
__device__ __forceinline__ int tile_bound(int t, int cnt, int tt) {
  return cnt <= 46340 ? (t * cnt) / tt : (int)(((long long)t * cnt) / tt);
}

// The work items of group g (shared when g < has_shared, else expert g - has_shared) in every
// list that is built, all threads of the block: per (128-row weight tile, token tile) pair,
// ordered by weight tile, then token tile, so consecutive items of a large group reuse one
// weight tile from L2. A group of cnt rows is split into ceil(cnt / TN) token tiles of equal
// size (within one row), so no tile is a thin remainder.
__device__ __forceinline__ void write_group_items(const PrepArgs& a, int g) {
  const bool sh = a.has_shared && g == 0;
  const int gid = sh ? a.E : g - a.has_shared;
  const int cnt = sh ? a.T : a.counts[gid];
  if (cnt == 0) return;
  const int row0 = sh ? 0 : (a.has_shared ? a.T : 0) + a.offsets[gid];
#pragma unroll 1
  for (int list = 0; list < 4; ++list) {
    int4* const base = list == 0 ? a.items[0] : list == 1 ? a.items[1] : list == 2 ? a.items[2] : a.items[3];
    if (!base) continue;
    const int tn = list == 0 ? a.tn[0] : list == 1 ? a.tn[1] : list == 2 ? a.tn[2] : a.tn[3];
    const int nwt = list % 2 == 0 ? 2 * (sh ? a.Is : a.I) / kBM : a.H / kBM;
    int4* items = base + a.gbase[list * (kMaxGroups + 1) + g];
    const int tt = (cnt + tn - 1) / tn;
    for (int i = threadIdx.x; i < nwt * tt; i += blockDim.x) {
      const int wt = i / tt, t = i - wt * tt;
      const int r0 = tile_bound(t, cnt, tt), r1 = tile_bound(t + 1, cnt, tt);
      items[i] = make_int4(gid, row0 + r0, r1 - r0, wt * kBM);
    }
  }
}

// Block of kTokPerBlk tokens, 1024 threads: the tokens' routing when logits are given (warp per
// token), the block's per-expert token masks and their popcounts (the block's histogram),
// then a per-layer counter; the last block to count in runs scan_block over every block's
// histogram (no block waits for another) and resets the counter for the next call.
__global__ void __launch_bounds__(1024) route_hist_scan_kernel(PrepArgs a, int nblk) {
  pdl_wait();  // the predecessor on the stream (launched with launch_pdl)
  pdl_trigger();
  __shared__ unsigned long long s_mask[256];
  __shared__ int s_idx[kTokPerBlk * 8];  // this block's routing (when computed here)
  __shared__ int s_last;
  const int T = a.T, k = a.k, E = a.E;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, nwarps = blockDim.x / 32;
  if (blockIdx.x == 0 && threadIdx.x < 2) a.sq_max[threadIdx.x] = 0;  // maxima of this forward
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_mask[e] = 0ull;
  const int t0 = blockIdx.x * kTokPerBlk;
  const int nt = min(kTokPerBlk, T - t0);
  if (a.logits) {
    for (int tt = warp; tt < nt; tt += nwarps) {
      const size_t t = (size_t)(t0 + tt);
      route_token_warp(a.logits + t * E, E, k, a.idx_out + t * k, a.w_out + t * k, lane,
                       s_idx + tt * k);
    }
  }
  __syncthreads();  // this block's routing and the cleared masks are visible to the block
  for (int r = threadIdx.x; r < nt * k; r += blockDim.x) {
    const int e = a.logits ? s_idx[r] : a.idx[(size_t)t0 * k + r];
    if (e < 0 || e >= E) {
      set_error(a.err, kErrDevice);
      continue;
    }
    const unsigned long long bit = 1ull << (r / k);
    const unsigned long long old = atomicOr(&s_mask[e], bit);
    if (old & bit) set_error(a.err, kErrDevice);  // an expert repeated within a token
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    a.bmask[(size_t)blockIdx.x * E + e] = s_mask[e];
    a.bhist[(size_t)e * nblk + blockIdx.x] = __popcll(s_mask[e]);  // [E][nblk]
  }
  __threadfence();  // this thread's histogram stores visible device-wide before the count
  __syncthreads();
  if (threadIdx.x == 0) {
    s_last = atomicAdd(a.scan_ctr, 1) == nblk - 1;
    if (s_last) *a.scan_ctr = 0;  // every block has counted: ready for the next call
  }
  __syncthreads();
  if (!s_last) return;  // uniform over the block
  __threadfence();
  scan_block(a, nblk);
}

// Block per token: quantise x[t] once, write its codes (fp16 integers) to each of its rows.
// Block b also writes the work items of groups b, b + T, ... (the grouped GEMMs read them).
__global__ void __launch_bounds__(256, 6) scatter_kernel(PrepArgs a) {
  pdl_wait();  // the predecessor on the stream (launched with launch_pdl)
  pdl_trigger();
  const int ng = a.E + (a.has_shared ? 1 : 0);
  for (int g = blockIdx.x; g < ng; g += gridDim.x) write_group_items(a, g);
  const int t = blockIdx.x;
  const int H = a.H, k = a.k, E = a.E;
  const int T_sh = a.has_shared ? a.T : 0;
  __shared__ int s_rows[9];
  __shared__ float s_red[32];
  __shared__ int s_sq[32];
  if (threadIdx.x < k) {
    const int j = threadIdx.x;
    int e = a.idx[(size_t)t * k + j];
    if (e < 0 || e >= E) e = 0;  // flagged by hist_kernel; keep the index in range
    const int b = t / kTokPerBlk, tl = t % kTokPerBlk;
    const unsigned long long m = a.bmask[(size_t)b * E + e];
    const int rank = __popcll(m & ((1ull << tl) - 1ull));
    const int nblk = (a.T + kTokPerBlk - 1) / kTokPerBlk;
    int pos = a.offsets[e] + a.bhist[(size_t)e * nblk + b] + rank;
    if (pos < 0 || pos >= a.T * k) {
      set_error(a.err, kErrDevice);
      pos = 0;
    }
    a.perm[pos] = t * k + j;
    const int row = T_sh + pos;
    s_rows[j] = row;
    a.row_token[row] = t;
    a.row_w[row] = a.w[(size_t)t * k + j];
  } else if (threadIdx.x == k && a.has_shared) {
    s_rows[k] = t;
    a.row_token[t] = t;
    a.row_w[t] = 1.0f;
  }
  float4* y4 = reinterpret_cast<float4*>(a.y + (size_t)t * H);
  for (int c = threadIdx.x; c < H / 4; c += blockDim.x) y4[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  // amax over the row (8 bf16 per thread per pass)
  const uint16_t* xr = a.x + (size_t)t * H;
  float amax = 0.0f;
  for (int c = threadIdx.x * 8; c < H; c += blockDim.x * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + c);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      amax = fmaxf(amax, fabsf(bf16_bits_to_float((uint16_t)(u[i] & 0xffffu))));
      amax = fmaxf(amax, fabsf(bf16_bits_to_float((uint16_t)(u[i] >> 16))));
    }
  }
  amax = warp_max(amax);
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x / 32] = amax;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < blockDim.x / 32 ? s_red[threadIdx.x] : 0.0f;
    v = warp_max(v);
    if (threadIdx.x == 0) s_red[0] = v;
  }
  __syncthreads();
  const float s = __fdiv_rn(s_red[0], 127.0f);
  const float rs = quant_recip(s);
  const int nrows = k + (a.has_shared ? 1 : 0);
  if (threadIdx.x < nrows) a.sx[s_rows[threadIdx.x]] = s;
  if (threadIdx.x == 0 && a.stok) a.stok[t] = s;
  int sq = 0;  // sum of squared codes of this token (exactness bound of the gate/up GEMM)
  for (int c = threadIdx.x * 8; c < H; c += blockDim.x * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + c);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
    int q[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float lo = bf16_bits_to_float((uint16_t)(u[i] & 0xffffu));
      const float hi = bf16_bits_to_float((uint16_t)(u[i] >> 16));
      q[2 * i] = s > 0.0f ? quant_code(lo, s, rs) : 0;
      q[2 * i + 1] = s > 0.0f ? quant_code(hi, s, rs) : 0;
      sq += q[2 * i] * q[2 * i] + q[2 * i + 1] * q[2 * i + 1];
    }
    uint4 hv;
    uint32_t* hw = reinterpret_cast<uint32_t*>(&hv);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 h2 = __halves2half2(__int2half_rn(q[2 * i]), __int2half_rn(q[2 * i + 1]));
      hw[i] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    for (int r = 0; r < nrows; ++r)
      *reinterpret_cast<uint4*>(a.xq + (size_t)s_rows[r] * H + c) = hv;
    if (a.qtok) {
      uint2 qv;
      uint8_t* qb = reinterpret_cast<uint8_t*>(&qv);
#pragma unroll
      for (int i = 0; i < 8; ++i) qb[i] = (uint8_t)(int8_t)q[i];
      *reinterpret_cast<uint2*>(a.qtok + (size_t)t * H + c) = qv;
    }
  }
  sq = warp_sum_i(sq);
  if ((threadIdx.x & 31) == 0) s_sq[threadIdx.x / 32] = sq;
  __syncthreads();
  if (threadIdx.x < 32) {
    int v = threadIdx.x < blockDim.x / 32 ? s_sq[threadIdx.x] : 0;
    v = warp_sum_i(v);
    if (threadIdx.x == 0 && v > *(volatile int*)a.sq_max) atomicMax(a.sq_max, v);
  }
}

cudaError_t launch_prefill_prep(const PrepArgs& a, cudaStream_t s) {
  const int nblk = (a.T + kTokPerBlk - 1) / kTokPerBlk;
  cudaError_t e = launch_pdl(route_hist_scan_kernel, dim3(nblk), dim3(1024), 0, s, a, nblk);
  if (e != cudaSuccess) return e;
  return launch_pdl(scatter_kernel, dim3(a.T), dim3(256), 0, s, a);
}

}  // namespace moe
