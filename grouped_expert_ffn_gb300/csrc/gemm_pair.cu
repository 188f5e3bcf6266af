// Grouped W8A8 GEMMs on the 2-SM MMA (tcgen05 cta_group::2).
//
// The same work as grouped_gemm_kernel (gemm_tc.cu: concatenated-expert dispatch, weights as
// the M operand, exact integer products on the fp16 tensor pipe, the same two fused
// epilogues), computed by a cluster of two CTAs on neighbouring SMs: a work item is two
// adjacent 128-row weight tiles of one token tile, and one MMA of M = 256 rows covers both.
// Each CTA holds its own 128 weight rows and HALF of the token tile (N/2 rows), so an SM
// receives half the token bytes per tensor-core operation that the one-CTA kernel needs. The
// token operand is what limits the one-CTA kernel: every token stage has to come back from L2
// within the few k-blocks that the shared-memory ring covers.
//
// Roles, per CTA (GemmRoles in gemm_common.cuh; gate/up 672 threads, down 800):
//   epilogue warps of this CTA's 128 weight rows (its own TMEM lanes);
//   converter groups of this CTA's int8 weight tiles to fp16 (alternate k-blocks);
//   rank 0 only: the MMA issuer for the pair (both CTAs allocate TMEM);
//   two TMA producers of this CTA's int8 weight tiles (alternate stages);
//   two TMA producers of this CTA's half token tiles (alternate stages).
// Synchronisation across the pair:
//   - rank 0's MMA thread waits for its own token stage and for the fp16 weight buffer of
//     both CTAs: cfull on rank 0 completes on the arrivals of rank 0's converter warps and on
//     16 signal bytes per converter warp of rank 1, copied asynchronously into rank 0's shared
//     memory once that warp's rows and rank 1's token stage are ready;
//   - rank 0's commits arrive on both CTAs' barriers (multicast): the stage (token half and
//     fp16 weight buffer) is free again, or the accumulator is ready for the epilogue;
//   - acc_empty on rank 0 counts the epilogue warps of both CTAs.
// Every wait is bounded (cluster-scope acquire); the CTAs leave through a cluster barrier, so
// neither exits while the other may still arrive on its barriers or use its shared memory.
#include "gemm_common.cuh"

namespace moe {

constexpr int kPXStages = 6;                          // half token tiles
constexpr int kPXBytes = (kMaxTokTile / 2) * kBK * 2;  // 16 KB: at most 128 token rows
constexpr int kPWStages = 4;                          // int8 weight tiles (from HBM)
constexpr int kPConv = kPXStages;                     // fp16 weight buffer s goes with stage s
constexpr int kPOffW8 = kPXStages * kPXBytes;
constexpr int kPOffConv = kPOffW8 + kPWStages * kW8Bytes;
constexpr int kPOffBar = kPOffConv + kPConv * kW16Bytes;
constexpr int kPBarBytes = 512;
constexpr int kPairSmem = kPOffBar + kPBarBytes + 1024;
static_assert(kPairSmem <= 232448, "shared memory");
static_assert((2 * kPXStages + 2 * kPWStages + kPConv + 5) * 8 + 64 + 16 * 4 <= kPBarBytes,
              "barriers and signal slots");
static_assert(kPXStages % 2 == 0 && kPWStages % 2 == 0, "two producers per ring");
static_assert(kPXBytes % 1024 == 0 && kPOffW8 % 1024 == 0 && kPOffConv % 1024 == 0,
              "swizzled tiles stay 1024-byte aligned");
constexpr uint16_t kPairMask = 0x3;
#ifndef MOE_PAIR_TMEM_COLS
#define MOE_PAIR_TMEM_COLS 512
#endif
constexpr uint32_t kPairTmemCols = MOE_PAIR_TMEM_COLS;  // allocated in each CTA of the pair

template <bool GU>
__global__ void __launch_bounds__(GemmRoles<GU>::kThreads, 1)
    pair_gemm_kernel(const GemmArgs a, const __grid_constant__ XMaps tmX,
                     const __grid_constant__ CUtensorMap tmW,
                     const __grid_constant__ CUtensorMap tmWs) {
  using R = GemmRoles<GU>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* xfull = reinterpret_cast<uint64_t*>(smem + kPOffBar);  // [kPXStages]
  uint64_t* xempty = xfull + kPXStages;    // [kPXStages]
  uint64_t* wfull = xempty + kPXStages;    // [kPWStages]
  uint64_t* wempty = wfull + kPWStages;    // [kPWStages]
  uint64_t* cfull = wempty + kPWStages;    // [kPConv]  (rank 0's is used)
  uint64_t* acc_full = cfull + kPConv;     // [2]
  uint64_t* acc_empty = acc_full + 2;      // [2]      (rank 0's is used)
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // 16-byte signal slots: rank 1's converter warps copy 16 bytes each into rank 0's
  uint8_t* sig = reinterpret_cast<uint8_t*>(drain) + 64;  // [kConvWarps][16]

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int rank = (int)cluster_ctarank();  // 0 issues the MMAs
  const bool leader = rank == 0;
  const int pair = blockIdx.x / 2, n_pairs = gridDim.x / 2;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPXStages; ++s) {
      mbar_init(&xfull[s], 1);
      mbar_init(&xempty[s], 1);
    }
    for (int s = 0; s < kPWStages; ++s) {
      mbar_init(&wfull[s], 1);
      mbar_init(&wempty[s], kConvWarps);
    }
    for (int s = 0; s < kPConv; ++s)
      mbar_init(&cfull[s], kConvWarps);  // rank 0's converter warps (+ rank 1's bytes)
    for (int s = 0; s < 2; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 2 * R::kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == R::kMmaWarp) {
    tmem_alloc_pair(tmem_slot, kPairTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == R::kWProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmWs);
  }
  if (warp == R::kXProducerWarp && lane < kXMaps) tma_prefetch_desc(&tmX.m[lane]);
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers and TMEM exist before either uses the other's
  tc_fence_after();
  pdl_wait();  // the predecessor's results
  pdl_trigger();
  const uint32_t tmem = *tmem_slot;
  const bool single = single_accumulator_exact(a);
  const int kmax = a.K_r > a.K_s ? a.K_r : a.K_s;
  const int slot_cols = single ? a.TN : ((kmax + kChunkK - 1) / kChunkK) * a.TN;
  const int nslots = slot_cols <= (int)kPairTmemCols / 2 ? 2 : 1;
  const int kpc = single ? (1 << 30) : kChunkK / kBK;
  // an accumulator layout that does not fit the allocation is refused, not run
  const bool fits = slot_cols <= (int)kPairTmemCols;
  if (!fits && threadIdx.x == 0 && leader) set_error(a.err, kErrDevice);
  const int n_items = fits ? *a.n_items : 0;

  if (warp >= R::kWProducerWarp && warp < R::kXProducerWarp + 2) {
    if (lane == 0) {
      // ------- TMA producers, two threads per ring, each CTA its own operands -------
      const bool wprod = warp < R::kXProducerWarp;
      const int pidx = warp - (wprod ? R::kWProducerWarp : R::kXProducerWarp);
      const int nst = wprod ? kPWStages : kPXStages;
      uint64_t* full = wprod ? wfull : xfull;
      uint64_t* empty = wprod ? wempty : xempty;
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_par = 0;
      bool ok = true;
      for (int item = pair; ok && item < n_items; item += n_pairs) {
        int4 wi = a.items[item];
        wi.w += rank * kBM;
        const bool shared = wi.x == a.E;
        const int nkb = (shared ? a.K_s : a.K_r) / kBK;
        const int half = ((wi.z + 15) & ~15) / 2;  // token rows held by each CTA
        const uint32_t bytes = wprod ? (uint32_t)kW8Bytes : (uint32_t)(half * kBK * 2);
        const CUtensorMap* mx = &tmX.m[half / kXStep2 - 1];
        const int row0 = wi.y + rank * half;
        for (int kb = 0; kb < nkb; ++kb) {
          if ((stage & 1) == pidx) {
            // the token stage is freed by rank 0's commit: cluster-scope acquire
            const bool got = wprod ? mbar_wait(&empty[stage], phase ^ 1, abort_flag, a.err)
                                   : mbar_wait_cl(&empty[stage], phase ^ 1, abort_flag, a.err);
            if (!got) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[stage], bytes);
            if (wprod) {
              uint8_t* sw = smem + kPOffW8 + stage * kW8Bytes;
              if (shared)
                tma_load_2d(sw, &tmWs, &full[stage], kb * kBK, wi.w);
              else
                tma_load_3d(sw, &tmW, &full[stage], kb * kBK, wi.w, wi.x);
            } else {
              tma_load_2d(smem + stage * kPXBytes, mx, &full[stage], kb * kBK, row0);
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
    // ---------------- converters ----------------
    // Group g converts the k-blocks whose running index is g modulo R::kConvGroups. On rank 0
    // the group's warps arrive on cfull (warp 0 also expects the 64 signal bytes of rank 1);
    // on rank 1 each warp, once its rows and rank 1's token stage are ready, copies 16 bytes
    // into rank 0's signal slot with completion on rank 0's cfull. The copy is asynchronous,
    // so no thread waits for a cluster-scope release.
    const int cw = warp - R::kConvWarp0;
    const int group = cw / kConvWarps, gw = cw % kConvWarps;
    const int r = gw * 32 + lane;
    const uint32_t cfull_leader = mapa_shared(smem_u32(cfull), 0);
    const uint32_t sig_leader = mapa_shared(smem_u32(sig + 16 * gw), 0);
    int ws = 0, cb = 0, gk = 0;  // cb: token stage = fp16 buffer
    uint32_t wph = 0, cph = 0;
    bool ok = true;
    for (int item = pair; ok && item < n_items; item += n_pairs) {
      const int4 wi = a.items[item];
      const int nkb = (wi.x == a.E ? a.K_s : a.K_r) / kBK;
      for (int kb = 0; kb < nkb; ++kb, ++gk) {
        if (gk % R::kConvGroups == group) {
          // the buffer's previous MMAs are done (rank 0's commit)
          const bool got = mbar_wait(&wfull[ws], wph, abort_flag, a.err) &&
                           mbar_wait_cl(&xempty[cb], cph ^ 1, abort_flag, a.err);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          widen_row(smem + kPOffW8 + ws * kW8Bytes, smem + kPOffConv + cb * kW16Bytes, r);
          // this thread's fp16 stores (to its own CTA's shared memory) before any tensor-core
          // read of them, whichever CTA of the pair issues the MMA
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&wempty[ws]);
          // this CTA's token stage has landed (its load overlapped the conversion): the
          // arrival / signal below then certifies both operands of this CTA
          if (!__all_sync(0xffffffffu, lane != 0 || mbar_wait(&xfull[cb], cph, abort_flag, a.err))) {
            ok = false;
            break;
          }
          if (lane == 0) {
            if (leader) {
              if (gw == 0)
                mbar_arrive_expect_tx(&cfull[cb], 16 * kConvWarps);
              else
                mbar_arrive(&cfull[cb]);
            } else {
              bulk_copy_to_peer(sig_leader, sig + 16 * gw, 16, cfull_leader + 8u * (uint32_t)cb);
            }
          }
        }
        if (++ws == kPWStages) {
          ws = 0;
          wph ^= 1;
        }
        if (++cb == kPConv) {
          cb = 0;
          cph ^= 1;
        }
      }
    }
  } else if (warp == R::kMmaWarp) {
    if (leader && lane == 0) {
      // ---------------- MMA issuer of the pair ----------------
      // Same lean loop as the one-CTA kernel: one barrier per k-block (cfull: both CTAs'
      // converted weights and token halves), probed for the next k-block while the current
      // MMAs issue; one multicast commit frees the stage (tokens and fp16 buffer) in both CTAs.
      const uint64_t dw0 = smem_desc_sw128(smem_u32(smem + kPOffConv));
      const uint64_t dx0 = smem_desc_sw128(smem_u32(smem));
      int xs = 0;
      uint32_t xph = 0, ready = 0;
      bool ok = true;
      int it = 0;
      for (int item = pair; ok && item < n_items; item += n_pairs, ++it) {
        const int4 wi = a.items[item];
        const int nkb = (wi.x == a.E ? a.K_s : a.K_r) / kBK;
        const int n_mma = (wi.z + 15) & ~15;
        const uint32_t idesc = idesc_f16_f32(2 * kBM, n_mma);
        const int slot = it % nslots;
        const uint32_t use = (uint32_t)(it / nslots) & 1u;
        if (!mbar_wait_cl(&acc_empty[slot], use ^ 1, abort_flag, a.err)) break;
        tc_fence_after();
        uint32_t dt = tmem + (uint32_t)(slot * slot_cols);
        int kin = 0;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!ready && !mbar_wait_cl(&cfull[xs], xph, abort_flag, a.err)) {
            ok = false;
            break;
          }
          const int ns = xs + 1 == kPXStages ? 0 : xs + 1;
          const uint32_t nph = ns == 0 ? xph ^ 1u : xph;
          ready = mma_kblock_commit_probe<true>(
              dt, dw0 + (uint64_t)((xs * kW16Bytes) >> 4), dx0 + (uint64_t)((xs * kPXBytes) >> 4),
              idesc, kin != 0 ? 1u : 0u, smem_u32(&xempty[xs]), smem_u32(&cfull[ns]), nph);
          if (++kin == kpc) {
            kin = 0;
            dt += (uint32_t)a.TN;
          }
          xs = ns;
          xph = nph;
        }
        if (!ok) break;
        umma_commit_pair(&acc_full[slot], kPairMask);
      }
      umma_commit_pair(drain, 0x1);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < 100000000ull) {
      }
    }
  } else if (warp < R::kEpiWarps) {
    // ---------------- epilogue of this CTA's weight rows ----------------
    const int cg = warp / 4;  // column group of this warp within its TMEM lane quadrant
    const uint32_t lane_base = tmem + ((uint32_t)((warp % 4) * 32) << 16);
    const uint32_t acc_empty_leader = mapa_shared(smem_u32(acc_empty), 0);
    int it = 0;
    for (int item = pair; item < n_items; item += n_pairs, ++it) {
      int4 wi = a.items[item];
      wi.w += rank * kBM;
      const int K = wi.x == a.E ? a.K_s : a.K_r;
      const int nch = single ? 1 : (K + kChunkK - 1) / kChunkK;
      const int slot = it % nslots;
      const uint32_t use = (uint32_t)(it / nslots) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait_cl(&acc_full[slot], use, abort_flag, a.err))) break;
      tc_fence_after();
      const uint32_t tbase = lane_base + (uint32_t)(slot * slot_cols);
      if (GU)
        epilogue_gate_up(a, wi, nch, tbase, cg);
      else
        epilogue_down(a, wi, nch, tbase, cg);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(&acc_empty[slot]);
        else
          mbar_arrive_remote(acc_empty_leader + 8u * (uint32_t)slot);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == R::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kPairTmemCols);
  }
}

static cudaLaunchConfig_t pair_config(cudaLaunchAttribute* attr, int grid, int threads,
                                      cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = kPairSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

cudaError_t pair_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(pair_gemm_kernel<true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(pair_gemm_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmem);
  return e;
}

cudaError_t pair_max_clusters(bool gate_up, int* n) {
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg =
      pair_config(attr, 2, gate_up ? GemmRoles<true>::kThreads : GemmRoles<false>::kThreads,
                  nullptr);
  return gate_up ? cudaOccupancyMaxActiveClusters(n, pair_gemm_kernel<true>, &cfg)
                 : cudaOccupancyMaxActiveClusters(n, pair_gemm_kernel<false>, &cfg);
}

cudaError_t launch_pair_gemm(bool gate_up, const GemmArgs& a, const XMaps& tmX,
                             const CUtensorMap& tmW, const CUtensorMap& tmWs, int grid,
                             cudaStream_t s) {
  cudaLaunchAttribute attr[2];
  if (gate_up) {
    const cudaLaunchConfig_t cfg = pair_config(attr, grid, GemmRoles<true>::kThreads, s);
    return cudaLaunchKernelEx(&cfg, pair_gemm_kernel<true>, a, tmX, tmW, tmWs);
  }
  const cudaLaunchConfig_t cfg = pair_config(attr, grid, GemmRoles<false>::kThreads, s);
  return cudaLaunchKernelEx(&cfg, pair_gemm_kernel<false>, a, tmX, tmW, tmWs);
}

}  // namespace moe
