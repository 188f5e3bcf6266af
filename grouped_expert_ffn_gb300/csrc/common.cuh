// Device-side helpers shared by the library's kernels: inline PTX for mbarriers, TMA bulk
// tensor copies and the 5th-generation tensor core (tcgen05 / TMEM), bounded waits and the
// plan's sticky error word.
#pragma once
#include <utility>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace moe {

// ---- sticky device error word -----------------------------------------------------------
// Codes match moe_status. The first failing thread wins; later ones leave it unchanged.
enum : int { kErrTimeout = 6, kErrDevice = 7 };

__device__ __forceinline__ void set_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// A wait that takes longer than this is a bug (a tile takes microseconds).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete. Gives up after kWaitLimitNs or as soon as
// *abort is set by another role of the CTA; on give-up sets *abort and the error word and
// returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      set_error(err, kErrTimeout);
      return false;
    }
  }
}

// Non-blocking probe of phase `parity` of `bar`.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// ---- programmatic dependent launch ------------------------------------------------------
// Kernels of the layer chain are launched with launch_pdl: a kernel's blocks may be scheduled
// while its predecessor on the stream drains, and wait for it (its completion and memory) in
// pdl_wait before touching global memory. pdl_trigger lets the successor be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... Params, typename... Args>
static cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- TMA ----------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// L2 cache policies (createpolicy): data read once (evict first) and data re-read soon by
// another kernel (evict last).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* m, uint64_t* bar,
                                                 int c0, int c1, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const CUtensorMap* m, uint64_t* bar,
                                                 int c0, int c1, int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}
// Untiled bulk copy global -> shared: addresses 16-byte aligned, bytes a multiple of 16;
// completes as transaction bytes on bar.
__device__ __forceinline__ void bulk_load_hint(void* dst, const void* src, uint32_t bytes,
                                               uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void st_f32_hint(float* p, float v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(policy) : "memory");
}

// ---- tcgen05 / TMEM -----------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, fp16 inputs, fp32 accumulate (kind::f16).
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every tcgen05 op issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns written from 32 registers per thread (thread i of
// the warp writes lane base + i). Asynchronous: tmem_st_wait waits for the thread's stores.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0],"
      " {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16,"
      " %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
      "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
      "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// One pipeline stage of the grouped GEMM (128 K): eight MMAs of K = 16 with the A operand
// (weights, fp16) in TMEM, a_tmem + 8 columns per MMA, and B (tokens) in shared memory, two
// 64-K sub-tiles b0 and b1 (descriptors advance 32 bytes per MMA); one commit to `commit_x`
// (the token stage is free once these MMAs completed) and one to `commit_a` (the TMEM A stage
// is free); and a non-blocking probe of phase `next_parity` of `next_bar` (the barrier of the
// next stage), all in one block, so that the probe's shared-memory round trip overlaps the
// MMA issue. The block opens with tcgen05.fence::after_thread_sync: the A stage was written
// by other threads (tcgen05.st) and observed complete through an mbarrier. `accumulate`
// applies to the first MMA. Returns whether the next stage is ready.
__device__ __forceinline__ uint32_t mma_stage_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b0,
                                                 uint64_t b1, uint32_t idesc, uint32_t accumulate,
                                                 uint32_t commit_x, uint32_t commit_a,
                                                 uint32_t next_bar, uint32_t next_parity) {
  uint32_t ready;
  asm volatile(
      "{\n\t.reg .pred pa, pt, pn;\n\t"
      "tcgen05.fence::after_thread_sync;\n\t"
      "setp.ne.b32 pa, %5, 0;\n\t"
      "setp.eq.b32 pt, 1, 1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], [%2], %3, %4, pa;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], [%10], %11, %4, pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], [%12], %13, %4, pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], [%14], %15, %4, pt;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 pn, [%8], %9;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], [%16], %17, %4, pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], [%18], %19, %4, pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], [%20], %21, %4, pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], [%22], %23, %4, pt;\n\t"
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%6];\n\t"
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%7];\n\t"
      "selp.u32 %0, 1, 0, pn;\n\t}\n"
      : "=r"(ready)
      : "r"(d_tmem), "r"(a_tmem), "l"(b0), "r"(idesc), "r"(accumulate), "r"(commit_x),
        "r"(commit_a), "r"(next_bar), "r"(next_parity), "r"(a_tmem + 8), "l"(b0 + 2),
        "r"(a_tmem + 16), "l"(b0 + 4), "r"(a_tmem + 24), "l"(b0 + 6), "r"(a_tmem + 32), "l"(b1),
        "r"(a_tmem + 40), "l"(b1 + 2), "r"(a_tmem + 48), "l"(b1 + 4), "r"(a_tmem + 56),
        "l"(b1 + 6)
      : "memory");
  return ready;
}

// 32 lanes x 16 consecutive 32-bit columns; thread i of the warp gets lane (base lane + i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32"
      " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major tile stored in the 128-byte swizzled layout
// that a TMA load with CU_TENSOR_MAP_SWIZZLE_128B writes: rows of 128 bytes, groups of 8
// rows 1024 bytes apart (stride byte offset), tile base 1024-byte aligned.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);        // start address
  d |= (uint64_t)(16 >> 4) << 16;                // leading byte offset (unused for SW128 K-major)
  d |= (uint64_t)(1024 >> 4) << 32;              // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                        // descriptor version (tcgen05)
  d |= (uint64_t)2 << 61;                        // layout: 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: A and B fp16, D fp32, both K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4)                      // D format: f32
         | (0u << 7) | (0u << 10)       // A, B format: f16
         | (0u << 15) | (0u << 16)      // A, B K-major
         | ((uint32_t)(N >> 3) << 17)   // N / 8
         | ((uint32_t)(M >> 4) << 24);  // M / 16
}

// ---- small numeric helpers ------------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Reciprocal of a row scale for quant_code, computed once per row. NaN (every element takes
// the exact division) when s is so small that 1/s could overflow.
__device__ __forceinline__ float quant_recip(float s) {
  return s >= 0x1p-100f ? __frcp_rn(s) : __int_as_float(0x7fffffff);
}

// Symmetric int8 code of v with scale s (s > 0, r = quant_recip(s)): round-half-even of the
// correctly rounded fp32 quotient v / s, clamped to +-127.
// Fast path: y = v * r differs from the exact quotient q by less than 3|q|u (u = 2^-24) and the
// fp32 quotient differs from q by at most |q|u. Every caller derives s = amax / 127 from the
// row's amax, so |q| < 128 and the two stay within 2^-15 of each other. When y lies farther than 2^-11
// from every half-integer, no rounding boundary separates y from the fp32 quotient and rne(y)
// is the exact answer; otherwise (about one element in a thousand) the quotient is taken by an
// IEEE division.
__device__ __forceinline__ int quant_code(float v, float s, float r) {
  const float y = __fmul_rn(v, r);
  const float n = rintf(y);
  int q;
  if (fabsf(__fsub_rn(y, n)) < 0.4995f)
    q = (int)n;
  else
    q = __float2int_rn(__fdiv_rn(v, s));
  return max(-127, min(127, q));
}

// SiLU(g) * u in fp32 with an IEEE division: the expert's gated activation.
__device__ __forceinline__ float silu_mul(float g, float u) {
  return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
}

// Dequantise an int32 accumulator: (float(acc) * s_row) * s_col, each step rounded.
__device__ __forceinline__ float dequant(int acc, float s_row, float s_col) {
  return __fmul_rn(__fmul_rn(__int2float_rn(acc), s_row), s_col);
}
// The same from accf = float(acc) (round to nearest even), e.g. an fp32 accumulator that
// holds the integer exactly.
__device__ __forceinline__ float dequant_f(float accf, float s_row, float s_col) {
  return __fmul_rn(__fmul_rn(accf, s_row), s_col);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---- top-k softmax routing of one token, one warp ---------------------------------------
// The k (<= 8) largest of the E (<= 256) fp32 logits l[0..E) (ties to the lowest expert id;
// slots ordered by logit descending, then id ascending) and their softmax weights
// exp(l_j - l_max) / sum_i exp(l_i - l_max), the sum taken in slot order. Lane j < k writes
// slot j of idx[0..k) and w[0..k). Every lane of the warp must call it.
// Routing keeps E / 32 logits per lane in registers: 4 slots for E <= 128, 8 for E <= 256.

template <int kMaxEPerLane>
__device__ __forceinline__ void route_token_warp_n(const float* __restrict__ l, int E, int k,
                                                 int32_t* __restrict__ idx, float* __restrict__ w,
                                                 int lane, int* s_idx = nullptr,
                                                 float* s_w = nullptr) {
  float v[kMaxEPerLane];
  bool taken[kMaxEPerLane];
#pragma unroll
  for (int i = 0; i < kMaxEPerLane; ++i) {
    const int e = i * 32 + lane;
    v[i] = e < E ? l[e] : 0.0f;
    taken[i] = e >= E;
  }
  float sel_v[8];
  int sel_e[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < k) {
      // lane-local best among untaken: highest value, then lowest id
      float bv = 0.0f;
      int be = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < kMaxEPerLane; ++i) {
        const int e = i * 32 + lane;
        if (!taken[i] && (be == 0x7fffffff || v[i] > bv)) {
          bv = v[i];
          be = e;
        }
      }
      // warp argmax on (value desc, id asc); lanes with nothing left carry id = INT_MAX
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        const bool better = (oe != 0x7fffffff) &&
                            (be == 0x7fffffff || ov > bv || (ov == bv && oe < be));
        if (better) {
          bv = ov;
          be = oe;
        }
      }
      sel_v[j] = bv;
      sel_e[j] = be;
      if ((be & 31) == lane) {
#pragma unroll
        for (int i = 0; i < kMaxEPerLane; ++i)
          if (i == (be >> 5)) taken[i] = true;
      }
    } else {
      sel_v[j] = 0.0f;
      sel_e[j] = 0;
    }
  }
  // softmax over the selected logits: lane j < k handles slot j
  const float m = sel_v[0];
  float ex = 0.0f;
  int my_e = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (lane == j && j < k) {
      ex = expf(sel_v[j] - m);
      my_e = sel_e[j];
    }
  float z = 0.0f;
  // sum in slot order (j = 0..k-1), identical for every lane
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float ej = __shfl_sync(0xffffffffu, ex, j);
    if (j < k) z += ej;
  }
  if (lane < k) {
    const float wl = ex / z;
    idx[lane] = my_e;
    w[lane] = wl;
    if (s_idx) s_idx[lane] = my_e;  // a shared-memory copy for the calling block
    if (s_w) s_w[lane] = wl;
  }
}

// E <= 128 keeps 4 logits per lane (the top-k loop scans 4 register slots per round), larger
// E (<= 256) 8.
__device__ __forceinline__ void route_token_warp(const float* __restrict__ l, int E, int k,
                                                 int32_t* __restrict__ idx, float* __restrict__ w,
                                                 int lane, int* s_idx = nullptr,
                                                 float* s_w = nullptr) {
  if (E <= 128)
    route_token_warp_n<4>(l, E, k, idx, w, lane, s_idx, s_w);
  else
    route_token_warp_n<8>(l, E, k, idx, w, lane, s_idx, s_w);
}

}  // namespace moe
