// The C ABI (include/moe.h): argument checks, plan workspace, weight packing, TMA tensor
// maps, and the per-call launch sequence of the decode and prefill paths.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "internal.h"

using namespace moe;

struct moe_plan_s {
  int E = 0, k = 0, H = 0, I = 0, Is = 0, max_tokens = 0, Imax = 0, has_shared = 0;
  int device = 0, num_sms = 0;
  // token tiles of the two GEMMs with the exact chunked accumulation (fit TMEM with its 1024-K
  // chunks); with one accumulator over the whole K both take kMaxTokTile rows
  int tn_gu = 0, tn_d = 0;
  int grid_gu = 0, grid_d = 0;
  size_t R_max = 0;
  int max_items[4] = {0, 0, 0, 0};  // work lists: gate/up, down, and both in the chunked tiles
  // workspace (device)
  __half* xq = nullptr;  // [R, H] activation codes (fp16 integers) in row order
  float* sx = nullptr;
  int* row_token = nullptr;
  float* row_w = nullptr;
  float* h32 = nullptr;
  __half* hq = nullptr;  // [R, Imax] codes of SiLU(gate)*up (fp16 integers)
  float* sh = nullptr;
  int* counts = nullptr;
  int* offsets = nullptr;
  int* perm = nullptr;
  unsigned long long* bmask = nullptr;
  int* bhist = nullptr;
  int4* items[4] = {nullptr, nullptr, nullptr, nullptr};  // lists 2, 3 only when tn < kMaxTokTile
  int* n_items = nullptr;
  int8_t* qtok = nullptr;
  float* stok = nullptr;
  int4* groups = nullptr;
  int* n_groups = nullptr;
  int* sq_max = nullptr;  // [2] per-forward maxima of row sum(q^2): gate/up rows, down rows
  int* scan_ctr = nullptr;  // blocks of the routing/histogram kernel counted in (zero between calls)
  int* gbase = nullptr;     // [2][kMaxGroups + 1] work-item bases of the groups
  int* err = nullptr;
  // taps
  int debug = 0;
  int32_t* tap_gu = nullptr;
  int32_t* tap_d = nullptr;
  int last_T = 0;
  int decode_rows = kDecodeDefaultRows;  // T <= decode_rows runs the streaming decode kernels
  // per-stage timing
  int profile = 0;
  struct ProfRec {
    int path;
    cudaEvent_t ev[5];
  };
  std::vector<ProfRec> prof_pending;
  std::vector<cudaEvent_t> ev_pool;
  // token rows of the two GEMMs (N operand), one map per box height (16-row steps)
  XMaps tmX_gu, tmX_d;
  std::vector<void*> allocs;
};

struct moe_packed_s {
  moe_plan_s* plan = nullptr;
  int fp4 = 0;     // NVFP4 weights (f) instead of int8 (w)
  Fp4Weights f;
  // NVFP4 tensor-core tiles (gate/up interleaved; down) and the matrix scales as per-row scales
  uint8_t* gu4 = nullptr;
  uint8_t* gu4s = nullptr;
  uint8_t* d4 = nullptr;
  uint8_t* d4s = nullptr;
  float* rs4 = nullptr;  // [E*I gate | E*I up | E*H down | Is gate | Is up | H down]
  moe_weights w;
  int8_t* gu8 = nullptr;    // [E, 2I, H] gate/up rows interleaved in pairs
  int8_t* shgu8 = nullptr;  // [2Is, H]
  int* w_sq = nullptr;  // [2] max over weight rows of sum(q^2): gate/up rows, down rows
  CUtensorMap tmW_gu, tmWs_gu, tmW_d, tmWs_d;  // weights (M operand): routed, shared
};

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-byte tensor of `rank` dims (innermost first), box {64, box_rows[, 1]}, 128-byte swizzle.
bool encode_2byte(CUtensorMap* m, CUtensorMapDataType dt, const void* base, int rank,
                  const uint64_t* dims, const uint64_t* strides_bytes, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[3], st[2];
  cuuint32_t box[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) d[i] = dims[i];
  for (int i = 0; i < rank - 1; ++i) st[i] = strides_bytes[i];
  box[0] = kBK;
  box[1] = box_rows;
  box[2] = 1;
  CUresult r = fn(m, dt, rank, const_cast<void*>(base), d, st, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// int8 weight tiles: box {128 bytes (one 128-K stage), box_rows[, 1]}, 128-byte swizzle.
bool encode_u8(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
               const uint64_t* strides_bytes, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[3], st[2];
  cuuint32_t box[3] = {(cuuint32_t)kKS, box_rows, 1}, es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) d[i] = dims[i];
  for (int i = 0; i < rank - 1; ++i) st[i] = strides_bytes[i];
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<void*>(base), d, st, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_f16(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                const uint64_t* strides_bytes, uint32_t box_rows) {
  return encode_2byte(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, base, rank, dims, strides_bytes, box_rows);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <class T>
moe_status dalloc(moe_plan_s* p, T** out, size_t count) {
  void* ptr = nullptr;
  if (count == 0) count = 1;
  if (cudaMalloc(&ptr, count * sizeof(T)) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_OOM;
  }
  p->allocs.push_back(ptr);
  *out = static_cast<T*>(ptr);
  return MOE_OK;
}

void free_plan(moe_plan_s* p) {
  for (auto& r : p->prof_pending)
    for (cudaEvent_t e : r.ev) p->ev_pool.push_back(e);
  for (cudaEvent_t e : p->ev_pool) cudaEventDestroy(e);
  for (void* a : p->allocs) cudaFree(a);
  if (p->tap_gu) cudaFree(p->tap_gu);
  if (p->tap_d) cudaFree(p->tap_d);
  delete p;
}

// Token tile of a GEMM with reduction length K: kMaxTokTile rows, or fewer when the exact
// 1024-K chunks of one tile would not fit the accumulator columns (chunks x tile <= kAccCols),
// a multiple of 16.
int token_tile(int K) {
  const int nch = (K + kChunkK - 1) / kChunkK;
  int tn = (kAccCols / nch) & ~15;
  return tn > kMaxTokTile ? kMaxTokTile : tn;
}

moe_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  if (e == cudaErrorMemoryAllocation) return MOE_ERR_OOM;
  return MOE_ERR_CUDA;
}

// Five timing events for one forward, from the plan's pool (NULL when profiling is off).
cudaEvent_t* prof_events(moe_plan_s* p, int path) {
  if (!p->profile) return nullptr;
  moe_plan_s::ProfRec r;
  r.path = path;
  for (int i = 0; i < 5; ++i) {
    if (p->ev_pool.empty()) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
      p->ev_pool.push_back(e);
    }
    r.ev[i] = p->ev_pool.back();
    p->ev_pool.pop_back();
  }
  p->prof_pending.push_back(r);
  return p->prof_pending.back().ev;
}

size_t tap_bytes(const moe_plan_s* p, int which, int T) {
  const size_t R = (size_t)T * p->k + (p->has_shared ? T : 0);
  switch (which) {
    case MOE_TAP_COUNTS: return (size_t)p->E * 4;
    case MOE_TAP_OFFSETS: return (size_t)(p->E + 1) * 4;
    case MOE_TAP_PERM: return (size_t)T * p->k * 4;
    case MOE_TAP_QX: return (size_t)T * p->H;
    case MOE_TAP_SX: return (size_t)T * 4;
    case MOE_TAP_ACC_GU: return R * 2 * p->Imax * 4;
    case MOE_TAP_HQ: return R * p->Imax;
    case MOE_TAP_SH: return R * 4;
    case MOE_TAP_ACC_D: return R * p->H * 4;
    case MOE_TAP_ACC_GU_F64: return R * 2 * p->Imax * 8;
    case MOE_TAP_ACC_D_F64: return R * p->H * 8;
    default: return 0;
  }
}

}  // namespace

namespace {
// Grid of each GEMM: as many CTAs as fit at once (one per SM).
cudaError_t size_gemm_grids(moe_plan_s* p) {
  for (int gu = 0; gu < 2; ++gu) {
    int n = 0;
    const cudaError_t e = gemm_max_ctas(gu != 0, &n);
    if (e != cudaSuccess) return e;
    (gu ? p->grid_gu : p->grid_d) = n < 1 ? p->num_sms : n;
  }
  return cudaSuccess;
}
}  // namespace

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_OOM: return "out of device memory";
    case MOE_ERR_CAPACITY: return "more tokens than the plan's max_tokens";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_DEVICE: return "device-side range check failed";
    case MOE_ERR_NO_DEVICE: return "no sm_103 CUDA device";
    default: return "unknown status";
  }
}

moe_status moe_plan(int E, int top_k, int H, int I, int I_shared, int max_tokens,
                    moe_plan_t* out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (E < 1 || top_k < 1 || top_k > E || H < 1 || I < 1 || I_shared < 0 || max_tokens < 1)
    return MOE_ERR_INVALID_ARG;
  if (E > 256 || top_k > 8 || H % 128 || I % 64 || I_shared % 64 || H > 8192 || I > 4096 ||
      I_shared > 4096 || max_tokens > (1 << 20))
    return MOE_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_NO_DEVICE;
  }
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess || prop.major != 10 || prop.minor != 3) {
    cudaGetLastError();
    return MOE_ERR_NO_DEVICE;
  }
  moe_plan_s* p = new (std::nothrow) moe_plan_s();
  if (!p) return MOE_ERR_OOM;
  p->E = E;
  p->k = top_k;
  p->H = H;
  p->I = I;
  p->Is = I_shared;
  p->has_shared = I_shared > 0;
  p->Imax = std::max(I, I_shared);
  p->max_tokens = max_tokens;
  p->device = dev;
  p->num_sms = prop.multiProcessorCount;
  p->tn_gu = token_tile(H);
  p->tn_d = token_tile(p->Imax);
  const size_t T = max_tokens;
  p->R_max = T * top_k + (p->has_shared ? T : 0);
  const size_t nblk = (T + kTokPerBlk - 1) / kTokPerBlk;
  // sum over groups of ceil(rows / tile) <= (routed rows + (tile-1) E) / tile + shared tiles
  auto tiles = [&](int tn) {
    return (T * top_k + (size_t)(tn - 1) * E) / tn + (p->has_shared ? (T + tn - 1) / tn : 0) + 1;
  };
  p->max_items[0] = (int)(tiles(kMaxTokTile) * (2 * p->Imax / kBM));
  p->max_items[1] = (int)(tiles(kMaxTokTile) * (H / kBM));
  if (p->tn_gu < kMaxTokTile) p->max_items[2] = (int)(tiles(p->tn_gu) * (2 * p->Imax / kBM));
  if (p->tn_d < kMaxTokTile) p->max_items[3] = (int)(tiles(p->tn_d) * (H / kBM));
  moe_status st = MOE_OK;
#define ALLOC(ptr, n)                                  \
  if ((st = dalloc(p, &p->ptr, (n))) != MOE_OK) {      \
    free_plan(p);                                      \
    return st;                                         \
  }
  ALLOC(xq, p->R_max * H);
  ALLOC(sx, p->R_max);
  ALLOC(row_token, p->R_max);
  ALLOC(row_w, p->R_max);
  ALLOC(h32, p->R_max * p->Imax);
  ALLOC(hq, p->R_max * p->Imax);
  ALLOC(sh, p->R_max);
  ALLOC(counts, (size_t)E);
  ALLOC(offsets, (size_t)E + 1);
  ALLOC(perm, T * top_k);
  ALLOC(bmask, nblk * E);
  ALLOC(bhist, nblk * E);
  for (int l = 0; l < 4; ++l)
    if (p->max_items[l] > 0) ALLOC(items[l], (size_t)p->max_items[l]);
  ALLOC(n_items, 4);
  ALLOC(qtok, T * H);
  ALLOC(stok, T);
  ALLOC(groups, (size_t)E + 1);
  ALLOC(n_groups, 1);
  ALLOC(sq_max, 2);
  ALLOC(err, 1);
  ALLOC(scan_ctr, 1);
  ALLOC(gbase, 4 * (kMaxGroups + 1));
#undef ALLOC
  if (cudaMemset(p->err, 0, sizeof(int)) != cudaSuccess ||
      cudaMemset(p->scan_ctr, 0, sizeof(int)) != cudaSuccess ||
      cudaMemset(p->hq, 0, p->R_max * p->Imax * sizeof(__half)) != cudaSuccess) {
    free_plan(p);
    return MOE_ERR_CUDA;
  }
  // Token-row operands of the two GEMMs (fp16 rows in the plan's row order).
  {
    const uint64_t dims[2] = {(uint64_t)H, (uint64_t)p->R_max};
    const uint64_t st2[1] = {(uint64_t)H * 2};
    const uint64_t dims_d[2] = {(uint64_t)p->Imax, (uint64_t)p->R_max};
    const uint64_t st_d[1] = {(uint64_t)p->Imax * 2};
    for (int j = 0; j < kXMaps; ++j) {
      const uint32_t r1 = (uint32_t)(kXStep * (j + 1));
      if (!encode_f16(&p->tmX_gu.m[j], p->xq, 2, dims, st2, r1) ||
          !encode_f16(&p->tmX_d.m[j], p->hq, 2, dims_d, st_d, r1)) {
        free_plan(p);
        return MOE_ERR_CUDA;
      }
    }
  }
  cudaError_t e = gemm_set_attributes();
  if (e == cudaSuccess) e = decode_set_attributes();
  if (e == cudaSuccess) e = size_gemm_grids(p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    free_plan(p);
    return MOE_ERR_CUDA;
  }
  *out = p;
  return MOE_OK;
}

moe_status moe_plan_set_decode_rows(moe_plan_t p, int rows) {
  if (!p || rows < 0 || rows > kDecodeMaxRows) return MOE_ERR_INVALID_ARG;
  p->decode_rows = rows;
  return MOE_OK;
}

moe_status moe_plan_destroy(moe_plan_t plan) {
  if (!plan) return MOE_ERR_INVALID_ARG;
  free_plan(plan);
  return MOE_OK;
}

moe_status moe_pack_weights(moe_plan_t p, const moe_weights* w, void* stream, moe_packed_t* out) {
  if (!p || !w || !out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  const void* need[] = {w->w_gate, w->w_up, w->w_down, w->s_gate, w->s_up, w->s_down};
  for (const void* q : need)
    if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  if (p->has_shared) {
    const void* nsh[] = {w->sh_gate, w->sh_up, w->sh_down, w->sh_s_gate, w->sh_s_up, w->sh_s_down};
    for (const void* q : nsh)
      if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  moe_packed_s* pk = new (std::nothrow) moe_packed_s();
  if (!pk) return MOE_ERR_OOM;
  pk->plan = p;
  pk->w = *w;
  const size_t E = p->E, H = p->H, I = p->I, Is = p->Is;
  auto fail = [&](moe_status st) {
    if (pk->gu8) cudaFree(pk->gu8);
    if (pk->shgu8) cudaFree(pk->shgu8);
    if (pk->w_sq) cudaFree(pk->w_sq);
    cudaGetLastError();
    delete pk;
    return st;
  };
  if (cudaMalloc(&pk->gu8, E * 2 * I * H) != cudaSuccess) return fail(MOE_ERR_OOM);
  if (cudaMalloc(&pk->w_sq, 2 * sizeof(int)) != cudaSuccess) return fail(MOE_ERR_OOM);
  if (p->has_shared && cudaMalloc(&pk->shgu8, 2 * Is * H) != cudaSuccess) return fail(MOE_ERR_OOM);
  cudaError_t e = launch_pack_gu8(w->w_gate, w->w_up, (int)E, (int)I, (int)H, pk->gu8, s);
  if (e == cudaSuccess && p->has_shared)
    e = launch_pack_gu8(w->sh_gate, w->sh_up, 1, (int)Is, (int)H, pk->shgu8, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(pk->w_sq, 0, 2 * sizeof(int), s);
  if (e == cudaSuccess) e = launch_row_sq_max(w->w_gate, E * I, (int)H, pk->w_sq, s);
  if (e == cudaSuccess) e = launch_row_sq_max(w->w_up, E * I, (int)H, pk->w_sq, s);
  if (e == cudaSuccess) e = launch_row_sq_max(w->w_down, E * H, (int)I, pk->w_sq + 1, s);
  if (e == cudaSuccess && p->has_shared) {
    e = launch_row_sq_max(w->sh_gate, Is, (int)H, pk->w_sq, s);
    if (e == cudaSuccess) e = launch_row_sq_max(w->sh_up, Is, (int)H, pk->w_sq, s);
    if (e == cudaSuccess) e = launch_row_sq_max(w->sh_down, H, (int)Is, pk->w_sq + 1, s);
  }
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA);
  bool ok = true;
  {
    // weights (the MMA's M operand): int8, 128 rows x 64 bytes per tile
    const uint64_t dims[3] = {H, 2 * I, E};
    const uint64_t st[2] = {H, 2 * I * H};
    ok = ok && encode_u8(&pk->tmW_gu, pk->gu8, 3, dims, st, kBM);
    const uint64_t dd[3] = {I, H, E};
    const uint64_t sd[2] = {I, H * I};
    ok = ok && encode_u8(&pk->tmW_d, w->w_down, 3, dd, sd, kBM);
    if (p->has_shared) {
      const uint64_t ds[2] = {H, 2 * Is};
      const uint64_t ss[1] = {H};
      ok = ok && encode_u8(&pk->tmWs_gu, pk->shgu8, 2, ds, ss, kBM);
      const uint64_t dsd[2] = {Is, H};
      const uint64_t ssd[1] = {Is};
      ok = ok && encode_u8(&pk->tmWs_d, w->sh_down, 2, dsd, ssd, kBM);
    } else {
      pk->tmWs_gu = pk->tmW_gu;  // never read: no shared group exists
      pk->tmWs_d = pk->tmW_d;
    }
  }
  if (!ok) return fail(MOE_ERR_CUDA);
  *out = pk;
  return MOE_OK;
}

moe_status moe_pack_weights_nvfp4(moe_plan_t p, const moe_weights_nvfp4* w, void* stream,
                                  moe_packed_t* out) {
  if (!p || !w || !out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  const void* need[] = {w->w_gate, w->w_up, w->w_down, w->b_gate, w->b_up,
                        w->b_down, w->g_gate, w->g_up, w->g_down};
  for (const void* q : need)
    if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  if (p->has_shared) {
    const void* nsh[] = {w->sh_gate, w->sh_up, w->sh_down, w->sh_b_gate, w->sh_b_up, w->sh_b_down, w->sh_g};
    for (const void* q : nsh)
      if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  }
  if (p->H % 16 || p->I % 16 || p->Is % 16) return MOE_ERR_UNSUPPORTED;
  moe_packed_s* pk = new (std::nothrow) moe_packed_s();
  if (!pk) return MOE_ERR_OOM;
  pk->plan = p;
  pk->fp4 = 1;
  std::memset(&pk->w, 0, sizeof(pk->w));
  Fp4Weights& f = pk->f;
  f.w_gate = w->w_gate;
  f.w_up = w->w_up;
  f.w_down = w->w_down;
  f.b_gate = w->b_gate;
  f.b_up = w->b_up;
  f.b_down = w->b_down;
  f.g_gate = w->g_gate;
  f.g_up = w->g_up;
  f.g_down = w->g_down;
  if (p->has_shared) {
    f.sh_gate = w->sh_gate;
    f.sh_up = w->sh_up;
    f.sh_down = w->sh_down;
    f.sh_b_gate = w->sh_b_gate;
    f.sh_b_up = w->sh_b_up;
    f.sh_b_down = w->sh_b_down;
    f.sh_g = w->sh_g;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t E = p->E, H = p->H, I = p->I, Is = p->Is;
  auto fail = [&](moe_status st) {
    moe_packed_destroy(pk);
    cudaGetLastError();
    return st;
  };
  // tensor-core tiles: one kFp4TileBytes block per (128-row tile, 128-K stage)
  const size_t stH = (H + kKS - 1) / kKS, stI = (I + kKS - 1) / kKS, stIs = (Is + kKS - 1) / kKS;
  const size_t n_rs = 2 * E * I + E * H + (p->has_shared ? 2 * Is + H : 0);
  if (cudaMalloc(&pk->gu4, E * (2 * I / kBM) * stH * kFp4TileBytes) != cudaSuccess ||
      cudaMalloc(&pk->d4, E * (H / kBM) * stI * kFp4TileBytes) != cudaSuccess ||
      cudaMalloc(&pk->rs4, n_rs * sizeof(float)) != cudaSuccess)
    return fail(MOE_ERR_OOM);
  if (p->has_shared && (cudaMalloc(&pk->gu4s, (2 * Is / kBM) * stH * kFp4TileBytes) != cudaSuccess ||
                        cudaMalloc(&pk->d4s, (H / kBM) * stIs * kFp4TileBytes) != cudaSuccess))
    return fail(MOE_ERR_OOM);
  float* rs = pk->rs4;
  cudaError_t e = launch_pack_fp4_tiles(f.w_gate, f.w_up, f.b_gate, f.b_up, (int)E, (int)I, (int)H,
                                        pk->gu4, s);
  if (e == cudaSuccess)
    e = launch_pack_fp4_tiles(f.w_down, nullptr, f.b_down, nullptr, (int)E, (int)H, (int)I, pk->d4, s);
  if (e == cudaSuccess) e = launch_fill_rows(f.g_gate, (int)E, (int)I, rs, s);
  if (e == cudaSuccess) e = launch_fill_rows(f.g_up, (int)E, (int)I, rs + E * I, s);
  if (e == cudaSuccess) e = launch_fill_rows(f.g_down, (int)E, (int)H, rs + 2 * E * I, s);
  if (e == cudaSuccess && p->has_shared) {
    float* rsh = rs + 2 * E * I + E * H;
    e = launch_pack_fp4_tiles(f.sh_gate, f.sh_up, f.sh_b_gate, f.sh_b_up, 1, (int)Is, (int)H, pk->gu4s, s);
    if (e == cudaSuccess)
      e = launch_pack_fp4_tiles(f.sh_down, nullptr, f.sh_b_down, nullptr, 1, (int)H, (int)Is, pk->d4s, s);
    if (e == cudaSuccess) e = launch_fill_rows(f.sh_g, 1, (int)Is, rsh, s);
    if (e == cudaSuccess) e = launch_fill_rows(f.sh_g + 1, 1, (int)Is, rsh + Is, s);
    if (e == cudaSuccess) e = launch_fill_rows(f.sh_g + 2, 1, (int)H, rsh + 2 * Is, s);
  }
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA);
  e = launch_check_e4m3(f.b_gate, E * I * (H / 16), p->err, s);
  if (e == cudaSuccess) e = launch_check_e4m3(f.b_up, E * I * (H / 16), p->err, s);
  if (e == cudaSuccess) e = launch_check_e4m3(f.b_down, E * H * (I / 16), p->err, s);
  if (e == cudaSuccess && p->has_shared) {
    e = launch_check_e4m3(f.sh_b_gate, Is * (H / 16), p->err, s);
    if (e == cudaSuccess) e = launch_check_e4m3(f.sh_b_up, Is * (H / 16), p->err, s);
    if (e == cudaSuccess) e = launch_check_e4m3(f.sh_b_down, H * (Is / 16), p->err, s);
  }
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA);
  *out = pk;
  return MOE_OK;
}

moe_status moe_packed_destroy(moe_packed_t pk) {
  if (!pk) return MOE_ERR_INVALID_ARG;
  for (void* q : {(void*)pk->gu4, (void*)pk->gu4s, (void*)pk->d4, (void*)pk->d4s, (void*)pk->rs4})
    if (q) cudaFree(q);
  if (pk->gu8) cudaFree(pk->gu8);
  if (pk->shgu8) cudaFree(pk->shgu8);
  if (pk->w_sq) cudaFree(pk->w_sq);
  delete pk;
  return MOE_OK;
}

moe_status moe_route(moe_plan_t p, const float* logits, int T, int32_t* idx, float* w,
                     void* stream) {
  if (!p || !logits || !idx || !w) return MOE_ERR_INVALID_ARG;
  if (!aligned16(logits) || !aligned16(idx) || !aligned16(w)) return MOE_ERR_INVALID_ARG;
  if (T < 1) return MOE_ERR_INVALID_ARG;
  if (T > p->max_tokens) return MOE_ERR_CAPACITY;
  return cuda_status(launch_route(logits, T, p->E, p->k, idx, w, p->err,
                                  static_cast<cudaStream_t>(stream)));
}

// moe_forward, and moe_route_forward when logits is not null (then idx, w are the outputs
// the routing writes, read back by the later kernels).
static moe_status forward_impl(moe_plan_t p, moe_packed_t pk, const uint16_t* x, int T,
                        const float* logits, const int32_t* idx, const float* w, float* y,
                        void* stream) {
  if (!p || !pk || !x || !idx || !w || !y || pk->plan != p) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(idx) || !aligned16(w) || !aligned16(y))
    return MOE_ERR_INVALID_ARG;
  if (T < 1) return MOE_ERR_INVALID_ARG;
  if (T > p->max_tokens) return MOE_ERR_CAPACITY;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int T_sh = p->has_shared ? T : 0;
  const int R = T * p->k + T_sh;
  cudaError_t e;
  const bool stream_path = decode_shape_supported(p->H, p->Imax) && T <= p->decode_rows;
  p->last_T = T;
  if (stream_path) {
    DecodeArgs a;
    a.idx = idx;
    a.w = w;
    a.logits = logits;
    a.idx_out = const_cast<int32_t*>(idx);
    a.w_out = const_cast<float*>(w);
    a.x = x;
    a.T = T;
    a.k = p->k;
    a.E = p->E;
    a.H = p->H;
    a.I = p->I;
    a.Is = p->Is;
    a.Imax = p->Imax;
    a.has_shared = p->has_shared;
    a.num_sms = p->num_sms;
    a.w_gate = pk->w.w_gate;
    a.w_up = pk->w.w_up;
    a.w_down = pk->w.w_down;
    a.s_gate = pk->w.s_gate;
    a.s_up = pk->w.s_up;
    a.s_down = pk->w.s_down;
    a.sh_gate = pk->w.sh_gate;
    a.sh_up = pk->w.sh_up;
    a.sh_down = pk->w.sh_down;
    a.sh_s_gate = pk->w.sh_s_gate;
    a.sh_s_up = pk->w.sh_s_up;
    a.sh_s_down = pk->w.sh_s_down;
    a.counts = p->counts;
    a.offsets = p->offsets;
    a.perm = p->perm;
    a.groups = p->groups;
    a.n_groups = p->n_groups;
    a.row_token = p->row_token;
    a.row_w = p->row_w;
    a.qtok = p->qtok;
    a.stok = p->stok;
    a.h32 = p->h32;
    a.hq = p->hq;
    a.sh = p->sh;
    a.sq_scratch = p->sq_max + 1;
    a.y = y;
    a.tap_gu = p->debug ? p->tap_gu : nullptr;
    a.tap_d = p->debug ? p->tap_d : nullptr;
    a.err = p->err;
    if (pk->fp4) {
      a.fp4 = 1;
      a.f = pk->f;
      a.tap_gu = nullptr;
      a.tap_d = nullptr;
      a.tap_gu_f64 = p->debug ? reinterpret_cast<double*>(p->tap_gu) : nullptr;
      a.tap_d_f64 = p->debug ? reinterpret_cast<double*>(p->tap_d) : nullptr;
    }
    e = launch_decode(a, s, prof_events(p, 1));
    return cuda_status(e);
  }
  // work lists: in full token tiles for one accumulator over the whole K; for int8 weights
  // also in the plan's smaller tiles when the exact chunked accumulation needs them (the
  // GEMMs pick one at launch from the exactness bound); NVFP4 weights always take one
  // accumulator
  const bool fp4 = pk->fp4 != 0;
  PrepArgs pa;
  pa.idx = idx;
  pa.w = w;
  pa.logits = logits;
  pa.idx_out = const_cast<int32_t*>(idx);
  pa.w_out = const_cast<float*>(w);
  pa.scan_ctr = p->scan_ctr;
  pa.x = x;
  pa.T = T;
  pa.k = p->k;
  pa.E = p->E;
  pa.H = p->H;
  pa.I = p->I;
  pa.Is = p->Is;
  pa.has_shared = p->has_shared;
  pa.tn[0] = pa.tn[1] = kMaxTokTile;
  pa.tn[2] = p->tn_gu;
  pa.tn[3] = p->tn_d;
  for (int l = 0; l < 4; ++l) pa.items[l] = (l >= 2 && fp4) ? nullptr : p->items[l];
  pa.bmask = p->bmask;
  pa.bhist = p->bhist;
  pa.gbase = p->gbase;
  pa.counts = p->counts;
  pa.offsets = p->offsets;
  pa.perm = p->perm;
  pa.n_items = p->n_items;
  pa.xq = p->xq;
  pa.sx = p->sx;
  pa.row_token = p->row_token;
  pa.row_w = p->row_w;
  pa.y = y;
  pa.qtok = p->debug ? p->qtok : nullptr;
  pa.stok = p->debug ? p->stok : nullptr;
  pa.sq_max = p->sq_max;
  pa.err = p->err;
  cudaEvent_t* ev = prof_events(p, 0);
  if (ev) cudaEventRecord(ev[0], s);
  if ((e = launch_prefill_prep(pa, s)) != cudaSuccess) return cuda_status(e);
  if (ev) cudaEventRecord(ev[1], s);

  GemmArgs g;
  std::memset(&g, 0, sizeof(g));
  g.E = p->E;
  g.I = p->I;
  g.Is = p->Is;
  g.Imax = p->Imax;
  g.H = p->H;
  g.sx = p->sx;
  g.s_g = pk->w.s_gate;
  g.s_u = pk->w.s_up;
  g.sh_s_g = pk->w.sh_s_gate;
  g.sh_s_u = pk->w.sh_s_up;
  g.h32 = p->h32;
  g.s_h = p->sh;
  g.s_d = pk->w.s_down;
  g.sh_s_d = pk->w.sh_s_down;
  g.row_token = p->row_token;
  g.row_w = p->row_w;
  g.y = y;
  g.err = p->err;
  if (fp4) {  // matrix scales as per-row scales; taps fp64
    const size_t E = p->E, I = p->I, H = p->H, Is = p->Is;
    const float* rsh = pk->rs4 + 2 * E * I + E * H;
    g.s_g = pk->rs4;
    g.s_u = pk->rs4 + E * I;
    g.s_d = pk->rs4 + 2 * E * I;
    g.sh_s_g = p->has_shared ? rsh : nullptr;
    g.sh_s_u = p->has_shared ? rsh + Is : nullptr;
    g.sh_s_d = p->has_shared ? rsh + 2 * Is : nullptr;
  }
  // gate/up: K = H for every group
  g.items = p->items[0];
  g.n_items = p->n_items;
  g.items_c = pa.items[2];
  g.n_items_c = p->n_items + 2;
  g.TN_c = p->tn_gu;
  g.K_r = p->H;
  g.K_s = p->H;
  g.TN = kMaxTokTile;
  g.tap = p->debug && !fp4 ? p->tap_gu : nullptr;
  g.tap_f64 = p->debug && fp4 ? reinterpret_cast<double*>(p->tap_gu) : nullptr;
  g.row_sq_max = p->sq_max;
  g.w_sq_max = pk->w_sq;
  g.w4 = pk->gu4;
  g.w4s = pk->gu4s;
  g.rows_r = 2 * p->I;
  g.rows_s = 2 * p->Is;
  if ((e = launch_grouped_gemm(true, fp4, g, p->tmX_gu, pk->tmW_gu, pk->tmWs_gu, p->grid_gu, s)) !=
      cudaSuccess)
    return cuda_status(e);
  if (ev) cudaEventRecord(ev[2], s);
  if ((e = launch_requant(p->h32, R, T_sh, p->I, p->Is, p->Imax, p->hq, p->sh, p->sq_max + 1, s)) !=
      cudaSuccess)
    return cuda_status(e);
  if (ev) cudaEventRecord(ev[3], s);
  // down: K = I (routed) or I_shared (shared)
  g.items = p->items[1];
  g.n_items = p->n_items + 1;
  g.items_c = pa.items[3];
  g.n_items_c = p->n_items + 3;
  g.TN_c = p->tn_d;
  g.K_r = p->I;
  g.K_s = p->has_shared ? p->Is : p->I;
  g.TN = kMaxTokTile;
  g.tap = p->debug && !fp4 ? p->tap_d : nullptr;
  g.tap_f64 = p->debug && fp4 ? reinterpret_cast<double*>(p->tap_d) : nullptr;
  g.row_sq_max = p->sq_max + 1;
  g.w_sq_max = fp4 ? nullptr : pk->w_sq + 1;
  g.w4 = pk->d4;
  g.w4s = pk->d4s;
  g.rows_r = p->H;
  g.rows_s = p->H;
  e = launch_grouped_gemm(false, fp4, g, p->tmX_d, pk->tmW_d, pk->tmWs_d, p->grid_d, s);
  if (ev) cudaEventRecord(ev[4], s);
  return cuda_status(e);
}

moe_status moe_forward(moe_plan_t p, moe_packed_t pk, const uint16_t* x, int T,
                       const int32_t* idx, const float* w, float* y, void* stream) {
  return forward_impl(p, pk, x, T, nullptr, idx, w, y, stream);
}

moe_status moe_route_forward(moe_plan_t p, moe_packed_t pk, const uint16_t* x, int T,
                             const float* logits, int32_t* idx, float* w, float* y,
                             void* stream) {
  if (!logits || !aligned16(logits)) return MOE_ERR_INVALID_ARG;
  return forward_impl(p, pk, x, T, logits, idx, w, y, stream);
}

moe_status moe_profile_enable(moe_plan_t p, int on) {
  if (!p) return MOE_ERR_INVALID_ARG;
  p->profile = on ? 1 : 0;
  return MOE_OK;
}

moe_status moe_profile_read(moe_plan_t p, int path, float* ms_out, int* calls) {
  if (!p || !ms_out || !calls || (path != 0 && path != 1)) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < 4; ++i) ms_out[i] = 0.0f;
  *calls = 0;
  std::vector<moe_plan_s::ProfRec> keep;
  moe_status st = MOE_OK;
  for (auto& r : p->prof_pending) {
    if (r.path != path) {
      keep.push_back(r);
      continue;
    }
    const int nst = path == 0 ? 4 : 3;
    if (cudaEventSynchronize(r.ev[nst]) != cudaSuccess) st = MOE_ERR_CUDA;
    for (int i = 0; i < nst && st == MOE_OK; ++i) {
      float ms = 0.0f;
      if (cudaEventElapsedTime(&ms, r.ev[i], r.ev[i + 1]) != cudaSuccess) st = MOE_ERR_CUDA;
      ms_out[i] += ms;
    }
    *calls += 1;
    for (cudaEvent_t e : r.ev) p->ev_pool.push_back(e);
  }
  p->prof_pending.swap(keep);
  return st;
}

moe_status moe_get_error(moe_plan_t p) {
  if (!p) return MOE_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, p->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  return static_cast<moe_status>(v);
}

moe_status moe_clear_error(moe_plan_t p) {
  if (!p) return MOE_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemset(p->scan_ctr, 0, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  return cudaMemset(p->err, 0, sizeof(int)) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_selftest_wait_timeout(moe_plan_t p, void* stream) {
  if (!p) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_selftest_wait(p->err, static_cast<cudaStream_t>(stream)));
}

moe_status moe_debug_enable(moe_plan_t p, int on) {
  if (!p) return MOE_ERR_INVALID_ARG;
  if (on && !p->tap_gu) {
    // 8 bytes per accumulator: int32 taps use the first half, fp64 (NVFP4) taps all of it
    if (cudaMalloc(&p->tap_gu, p->R_max * 2 * p->Imax * sizeof(double)) != cudaSuccess ||
        cudaMalloc(&p->tap_d, p->R_max * p->H * sizeof(double)) != cudaSuccess) {
      cudaGetLastError();
      if (p->tap_gu) cudaFree(p->tap_gu);
      p->tap_gu = nullptr;
      return MOE_ERR_OOM;
    }
  }
  p->debug = on ? 1 : 0;
  return MOE_OK;
}

size_t moe_debug_tap_bytes(moe_plan_t p, int which) {
  if (!p) return 0;
  return tap_bytes(p, which, p->last_T);
}

moe_status moe_debug_tap(moe_plan_t p, int which, void* dst, size_t bytes) {
  if (!p || !dst || p->last_T < 1) return MOE_ERR_INVALID_ARG;
  const size_t need = tap_bytes(p, which, p->last_T);
  if (need == 0 || bytes != need) return MOE_ERR_INVALID_ARG;
  if ((which == MOE_TAP_ACC_GU || which == MOE_TAP_ACC_D || which == MOE_TAP_ACC_GU_F64 ||
       which == MOE_TAP_ACC_D_F64) && !p->tap_gu)
    return MOE_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  const void* src = nullptr;
  switch (which) {
    case MOE_TAP_COUNTS: src = p->counts; break;
    case MOE_TAP_OFFSETS: src = p->offsets; break;
    case MOE_TAP_PERM: src = p->perm; break;
    case MOE_TAP_QX: src = p->qtok; break;
    case MOE_TAP_SX: src = p->stok; break;
    case MOE_TAP_ACC_GU: src = p->tap_gu; break;
    case MOE_TAP_SH: src = p->sh; break;
    case MOE_TAP_ACC_D: src = p->tap_d; break;
    case MOE_TAP_ACC_GU_F64: src = p->tap_gu; break;
    case MOE_TAP_ACC_D_F64: src = p->tap_d; break;
    case MOE_TAP_HQ: {
      const size_t n = need;
      std::vector<__half> tmp(n);
      if (cudaMemcpy(tmp.data(), p->hq, n * sizeof(__half), cudaMemcpyDeviceToHost) != cudaSuccess)
        return MOE_ERR_CUDA;
      int8_t* d = static_cast<int8_t*>(dst);
      for (size_t i = 0; i < n; ++i) d[i] = static_cast<int8_t>(__half2float(tmp[i]));
      return MOE_OK;
    }
    default: return MOE_ERR_INVALID_ARG;
  }
  return cudaMemcpy(dst, src, need, cudaMemcpyDeviceToHost) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_router_logits(const uint16_t* x, const float* w_router, int T, int H, int E,
                             float* logits, void* stream) {
  if (!x || !w_router || !logits || T < 1 || H < 16 || E < 1 || H % 16) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(logits)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_router_logits(x, w_router, T, H, E, logits,
                                          static_cast<cudaStream_t>(stream)));
}

moe_status moe_router_pack(const float* w_router, int H, int E, uint16_t* packed, void* stream) {
  if (!w_router || !packed || H < 64 || E < kREB || H % 64 || E % kREB) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w_router) || !aligned16(packed)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_router_pack(w_router, H, E, packed, static_cast<cudaStream_t>(stream)));
}

moe_status moe_router_logits_packed(const uint16_t* x, const uint16_t* packed, int T, int H, int E,
                                    float* logits, void* stream) {
  if (!x || !packed || !logits || T < 1 || H < 64 || E < kREB || H % 64 || E % kREB)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(packed) || !aligned16(logits)) return MOE_ERR_INVALID_ARG;
  CUtensorMap ta, tb;
  const uint64_t da[2] = {(uint64_t)H, (uint64_t)T};
  const uint64_t sa[1] = {(uint64_t)H * 2};
  const uint64_t db[2] = {(uint64_t)H, (uint64_t)3 * E};
  const uint64_t sb[1] = {(uint64_t)H * 2};
  if (!encode_2byte(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, 2, da, sa, kBM) ||
      !encode_2byte(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, packed, 2, db, sb, 3 * kREB))
    return MOE_ERR_CUDA;
  return cuda_status(launch_router_tc(T, H, E, logits, ta, tb, static_cast<cudaStream_t>(stream)));
}

moe_status moe_rmsnorm_residual(uint16_t* x, const float* y, uint16_t* x_in, int T, int H,
                                void* stream) {
  if (!x || !x_in || T < 1 || H < 4 || H % 4) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(x_in) || (y && !aligned16(y))) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_rmsnorm_residual(x, y, x_in, T, H, static_cast<cudaStream_t>(stream)));
}

moe_status moe_residual_add(uint16_t* x, const float* y, int T, int H, void* stream) {
  if (!x || !y || T < 1 || H < 4 || H % 4) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_residual(x, y, (size_t)T * H, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
