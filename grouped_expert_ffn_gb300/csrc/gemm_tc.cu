// Grouped W8A8 GEMMs of the prefill path on the 5th-generation tensor cores (tcgen05).
//
// One persistent kernel runs every (expert group, 128-row weight tile, token tile) work item
// of a layer: the gate/up GEMM with a fused SiLU(gate)*up epilogue, or the down GEMM whose
// epilogue writes every row's router-weighted output (combine_kernel then sums each token's
// rows). This is the concatenated-expert computation
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
// from TMA (one box per stage, 128-byte swizzle) to the MMA: widening them in shared memory
// too would triple the shared-memory traffic of a k-block (measured slower).
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
// The 2-SM form of the same items (one MMA of M = 256 over two CTAs, each holding half of the
// token tile) is in gemm_pair.cu; a plan selects it per GEMM.
//
// Warp roles (one CTA per SM; GemmRoles in gemm_common.cuh): gate/up 672 threads, down 800.
//   epilogue warps (8 for gate/up, 12 for down): warp w reads TMEM lanes 32*(w%4).. (weight
//               rows) and every (w/4)-th 16-column chunk (tokens) of its quadrant;
//   converter groups of four warps (2 for each GEMM) taking turns over k-blocks: thread r of
//               a group widens weight row r;
//   one MMA issuer and TMEM owner;
//   two TMA producers of the int8 weight tiles (alternate stages);
//   two TMA producers of the fp16 token tiles (alternate stages).
// Pipeline: the weights stream from HBM through a ring of small int8 stages (4 x 8 KB,
// released by the converters as soon as they have widened a stage); the token tiles, mostly
// L2 hits, through a ring of large stages (4 x 32 KB), one TMA load per stage (box heights
// 16..256 rows); one fp16 weight buffer per token stage, released together with it by the
// MMA's commit. A converter group widens its k-block as soon as the int8 tile and the fp16
// buffer are free and waits for the token tile only afterwards, so the token load overlaps
// the conversion. A TMA-issuing thread completes only a few loads per microsecond, so each ring
// has two issuing threads and each token tile is one load rather than several 64-row ones.
// Barrier arrivals are one per warp (after __syncwarp) and the MMA thread commits once per
// k-block: every arrival and commit sits on the critical path of a k-block.
// Every mbarrier wait is bounded; a wait
// that runs out sets the plan's error word and the CTA drains its own copies and MMAs, frees
// TMEM and returns.
//
// The down epilogue writes w * dequant(acc) per (row, channel) to yd; combine_kernel sums each
// token's k routed rows and its shared-expert row in slot order (deterministic, no atomics).
#include "gemm_common.cuh"

namespace moe {

#ifndef MOE_W_STAGES
#define MOE_W_STAGES 4
#endif
#ifndef MOE_X_STAGES
#define MOE_X_STAGES 4  // token stages of the gate/up GEMM
#endif
#ifndef MOE_D_X_STAGES
#define MOE_D_X_STAGES 4  // token stages of the down GEMM
#endif
constexpr int kXBytesMax = kMaxTokTile * kBK * 2;    // fp16 token tile per stage (<= 32 KB)

// Shared-memory layout of one GEMM instance: token stages, int8 weight stages, fp16 weight
// buffers (buffer s goes with token stage s), barriers.
template <bool GU>
struct GemmSmem {
  static constexpr int kXStages = GU ? MOE_X_STAGES : MOE_D_X_STAGES;
  static constexpr int kWStages = MOE_W_STAGES;
  static constexpr int kConvBufs = kXStages;
  static constexpr int kOffW8 = kXStages * kXBytesMax;
  static constexpr int kOffConv = kOffW8 + kWStages * kW8Bytes;
  static constexpr int kOffBar = kOffConv + kConvBufs * kW16Bytes;
  static constexpr int kBarBytes = 512;
  static constexpr int kBytes = kOffBar + kBarBytes + 1024;
  static_assert((2 * kXStages + 2 * kWStages + kConvBufs + 5) * 8 + 8 <= kBarBytes, "barriers");
  static_assert(kBytes <= 232448, "shared memory");
  static_assert(kOffW8 % 1024 == 0 && kOffConv % 1024 == 0,
                "swizzled tiles stay 1024-byte aligned");
  // Two producers per ring: stage s belongs to producer s % 2 (any stage count >= 2 works).
  static_assert(kXStages >= 2 && kWStages >= 2, "two producers per ring");
};



template <bool GU>
__global__ void __launch_bounds__(GemmRoles<GU>::kThreads, 1)
    grouped_gemm_kernel(const GemmArgs a, const __grid_constant__ XMaps tmX,
                        const __grid_constant__ CUtensorMap tmW,
                        const __grid_constant__ CUtensorMap tmWs) {
  constexpr int kXStages = GemmSmem<GU>::kXStages, kWStages = GemmSmem<GU>::kWStages;
  constexpr int kConvBufs = GemmSmem<GU>::kConvBufs;
  constexpr int kOffW8 = GemmSmem<GU>::kOffW8, kOffConv = GemmSmem<GU>::kOffConv;
  constexpr int kOffBar = GemmSmem<GU>::kOffBar;
  using R = GemmRoles<GU>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* xfull = reinterpret_cast<uint64_t*>(smem + kOffBar);  // [kXStages]
  uint64_t* xempty = xfull + kXStages;     // [kXStages]
  uint64_t* wfull = xempty + kXStages;     // [kWStages]
  uint64_t* wempty = wfull + kWStages;     // [kWStages]
  uint64_t* cfull = wempty + kWStages;     // [kConvBufs]
  uint64_t* acc_full = cfull + kConvBufs;  // [2]
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
      mbar_init(&wempty[s], kConvWarps);
    }
    for (int s = 0; s < kConvBufs; ++s) mbar_init(&cfull[s], kConvWarps);
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
  if (warp == R::kWProducerWarp && lane == 0) {
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
  const int n_items = *a.n_items;
  // Accumulator layout for this launch: one accumulator over the whole K (two TMEM slots,
  // double-buffered) when the bound proves it exact, else 1024-K chunks (the host sizes the
  // token tile so that the chunks of one tile fit the 512 columns).
  const bool single = single_accumulator_exact(a);
  const int kmax = a.K_r > a.K_s ? a.K_r : a.K_s;
  const int slot_cols = single ? a.TN : ((kmax + kChunkK - 1) / kChunkK) * a.TN;
  const int nslots = slot_cols <= (int)kTmemCols / 2 ? 2 : 1;
  const int kpc = single ? (1 << 30) : kChunkK / kBK;  // k-blocks per accumulator

  if (warp >= R::kWProducerWarp && warp < R::kXProducerWarp + 2) {
    if (lane == 0) {
      // ------- TMA producers: weights (HBM) and tokens, two threads per ring -------
      // Producer pidx of a ring owns the ring's stages with index % 2 == pidx; both walk the
      // whole item / k-block sequence to keep stage and phase in step.
      const bool wprod = warp < R::kXProducerWarp;
      const int pidx = warp - (wprod ? R::kWProducerWarp : R::kXProducerWarp);
      const int nst = wprod ? kWStages : kXStages;
      uint64_t* full = wprod ? wfull : xfull;
      uint64_t* empty = wprod ? wempty : xempty;
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_par = 0;  // stages with a load issued, and its phase
      bool ok = true;
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        const int4 wi = a.items[item];
        const bool shared = wi.x == a.E;
        const int nkb = (shared ? a.K_s : a.K_r) / kBK;
        const int rows = (wi.z + kXStep1 - 1) / kXStep1 * kXStep1;  // box height
        const uint32_t bytes = wprod ? (uint32_t)kW8Bytes : (uint32_t)(rows * kBK * 2);
        const CUtensorMap* mx = &tmX.m[rows / kXStep1 - 1];
        for (int kb = 0; kb < nkb; ++kb) {
          if ((stage & 1) == pidx) {
            if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, a.err)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[stage], bytes);
            if (wprod) {
              uint8_t* sw = smem + kOffW8 + stage * kW8Bytes;
              if (shared)
                tma_load_2d(sw, &tmWs, &full[stage], kb * kBK, wi.w);
              else
                tma_load_3d(sw, &tmW, &full[stage], kb * kBK, wi.w, wi.x);
            } else {
              tma_load_2d(smem + stage * kXBytesMax, mx, &full[stage], kb * kBK, wi.y);
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
    // ---------------- converters: int8 -> fp16 weight rows ----------------
    // Group g converts the k-blocks whose running index is g modulo R::kConvGroups, so the
    // latency of one group's fence and arrivals overlaps the other groups' work. The fp16
    // buffer of token stage cb is free once the MMAs of its previous use completed (the token
    // stage's empty barrier).
    const int cw = warp - R::kConvWarp0;
    const int group = cw / kConvWarps;
    const int r = (cw % kConvWarps) * 32 + lane;  // weight row within the tile
    int stage = 0, cb = 0, gk = 0;
    uint32_t phase = 0, cphase = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      const int4 wi = a.items[item];
      const int nkb = (wi.x == a.E ? a.K_s : a.K_r) / kBK;
      for (int kb = 0; kb < nkb; ++kb, ++gk) {
        if (gk % R::kConvGroups != group) {
          if (++stage == kWStages) {
            stage = 0;
            phase ^= 1;
          }
          if (++cb == kConvBufs) {
            cb = 0;
            cphase ^= 1;
          }
          continue;
        }
        // warp-uniform outcome: the per-warp arrivals below need every lane
        const bool got = mbar_wait(&wfull[stage], phase, abort_flag, a.err) &&
                         mbar_wait(&xempty[cb], cphase ^ 1, abort_flag, a.err);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        widen_row(smem + kOffW8 + stage * kW8Bytes, smem + kOffConv + cb * kW16Bytes, r);
        fence_proxy_async_smem();  // this thread's fp16 stores, before the MMA reads them
        __syncwarp();
        if (lane == 0) mbar_arrive(&wempty[stage]);
        // The token stage cb is waited for after the conversion (which overlaps its load), so
        // that cfull alone tells the MMA thread that both operands are in shared memory.
        if (!__all_sync(0xffffffffu, lane != 0 || mbar_wait(&xfull[cb], cphase, abort_flag, a.err))) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive(&cfull[cb]);
        if (++stage == kWStages) {
          stage = 0;
          phase ^= 1;
        }
        if (++cb == kConvBufs) {
          cb = 0;
          cphase ^= 1;
        }
      }
    }
  } else if (warp == R::kMmaWarp) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      // The issuing thread is on the tensor pipe's critical path: tcgen05.mma issue blocks
      // once the pipe's queue is full, so every instruction between the last MMA of a k-block
      // and the first of the next leaves the pipe idle. Per k-block it therefore waits on one
      // barrier only (cfull: converted weights and token stage), and usually not even that:
      // mma_kblock_commit_probe probes the next k-block's barrier while the current MMAs
      // issue. Descriptors are a base plus a stage offset (the 14-bit start-address field
      // does not carry).
      const uint64_t dw0 = smem_desc_sw128(smem_u32(smem + kOffConv));
      const uint64_t dx0 = smem_desc_sw128(smem_u32(smem));
      int stage = 0;
      uint32_t phase = 0, ready = 0;
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
        uint32_t dt = tmem + (uint32_t)(slot * slot_cols);
        int kin = 0;  // k-block within the current accumulator chunk
        for (int kb = 0; kb < nkb; ++kb) {
          if (!ready && !mbar_wait(&cfull[stage], phase, abort_flag, a.err)) {
            ok = false;
            break;
          }
          const int ns = stage + 1 == kXStages ? 0 : stage + 1;
          const uint32_t nph = ns == 0 ? phase ^ 1u : phase;
          // one commit frees the token stage and the fp16 weight buffer that goes with it
          ready = mma_kblock_commit_probe<false>(
              dt, dw0 + (uint64_t)((stage * kW16Bytes) >> 4),
              dx0 + (uint64_t)((stage * kXBytesMax) >> 4), idesc, kin != 0 ? 1u : 0u,
              smem_u32(&xempty[stage]), smem_u32(&cfull[ns]), nph);
          if (++kin == kpc) {
            kin = 0;
            dt += (uint32_t)a.TN;
          }
          stage = ns;
          phase = nph;
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
      const int4 wi = a.items[item];
      const int K = wi.x == a.E ? a.K_s : a.K_r;
      const int nch = single ? 1 : (K + kChunkK - 1) / kChunkK;
      const int slot = it % nslots;
      const uint32_t use = (uint32_t)(it / nslots) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[slot], use, abort_flag, a.err))) break;
      tc_fence_after();
      const uint32_t tbase = lane_base + (uint32_t)(slot * slot_cols);
      if (GU)
        epilogue_gate_up(a, wi, nch, tbase, cg);
      else
        epilogue_down(a, wi, nch, tbase, cg);
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
}

cudaError_t gemm_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, GemmSmem<true>::kBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(grouped_gemm_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, GemmSmem<false>::kBytes);
  if (e == cudaSuccess) e = pair_set_attributes();
  return e;
}

// Work items that can run at once: CTAs for cs = 1, CTA pairs for cs = 2.
cudaError_t gemm_max_clusters(bool gate_up, int cs, int* n) {
  *n = 0;
  if (cs == 2) return pair_max_clusters(gate_up, n);
  if (cs != 1) return cudaErrorInvalidValue;
  int per_sm = 0, dev = 0, sms = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &per_sm, gate_up ? (const void*)grouped_gemm_kernel<true> : (const void*)grouped_gemm_kernel<false>,
      gate_up ? GemmRoles<true>::kThreads : GemmRoles<false>::kThreads,
      gate_up ? GemmSmem<true>::kBytes : GemmSmem<false>::kBytes);
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  *n = per_sm * sms;
  return e;
}

// grid: a multiple of cs (whole clusters).
cudaError_t launch_grouped_gemm(bool gate_up, int cs, const GemmArgs& a, const XMaps& tmX,
                                const CUtensorMap& tmW, const CUtensorMap& tmWs, int grid,
                                cudaStream_t s) {
  if (grid < cs || grid % cs) return cudaErrorInvalidValue;
  if (cs == 2) return launch_pair_gemm(gate_up, a, tmX, tmW, tmWs, grid, s);
  if (cs != 1) return cudaErrorInvalidValue;
  if (gate_up)
    return launch_pdl(grouped_gemm_kernel<true>, dim3(grid), dim3(GemmRoles<true>::kThreads),
                      GemmSmem<true>::kBytes, s, a, tmX, tmW, tmWs);
  return launch_pdl(grouped_gemm_kernel<false>, dim3(grid), dim3(GemmRoles<false>::kThreads),
                    GemmSmem<false>::kBytes, s, a, tmX, tmW, tmWs);
}

// y[t] = sum over slots j of yd[row(t, j)] + yd[t] (shared expert row), in slot order. Block per
// token, 8 consecutive channels per thread and pass.
__global__ void combine_kernel(const float* __restrict__ yd, const int* __restrict__ slot_row,
                               int T, int k, int H, int has_shared, float* __restrict__ y) {
  pdl_wait();  // the predecessor on the stream (launched with launch_pdl)
  pdl_trigger();
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
  return launch_pdl(combine_kernel, dim3(T), dim3(256), 0, s, yd, slot_row, T, k, H, has_shared, y);
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

// Each warp takes kRows consecutive rows and issues the loads of all of them before reducing
// any (more bytes in flight per warp); rows of up to 128 * kRegV values stay in registers.
constexpr int kRequantRows = 2;
constexpr int kRequantThreads = 512;

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
