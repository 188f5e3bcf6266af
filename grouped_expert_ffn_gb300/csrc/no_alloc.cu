// Allocation-free batched decode: the decode kernels of decode.cu driven with their scratch
// memory carved out of one file-scope device array instead of a plan's workspace.
//
// Who needs it: callers that must not allocate device memory on the call path. Examples are
// a plugin running inside another runtime that owns every device allocation and forbids its
// guests from calling cudaMalloc, and latency-critical serving loops where cudaMalloc/cudaFree
// would implicitly synchronise the device and stall other streams. moe_plan allocates a
// workspace, so those callers cannot use it on the call path.
//
// The scratch array lives in this library's device image: every GPU that loads the library
// holds kScratchBytes of it until the process exits, whether or not this entry point is used.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr size_t kScratchBytes = 2u << 20;  // 2 MiB
constexpr int kStaticMaxRows = 8;           // largest T this entry point takes
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

namespace {

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

// Device address of the scratch array for the current device, looked up once per device.
// In host code `g_decode_scratch` names a host-side stand-in, not device memory, so the
// address must come from cudaGetSymbolAddress with that device current.
cudaError_t scratch_for_current_device(void** out, int* num_sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_num_sms[dev] = n;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  *num_sms = g_num_sms[dev];
  return cudaSuccess;
}

size_t carve(size_t& off, size_t bytes) {
  const size_t at = off;
  off = (off + bytes + 255) & ~size_t(255);
  return at;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_forward_decode_static(int E, int top_k, int H, int I, int I_shared,
                                                const moe_weights* wt, const uint16_t* x, int T,
                                                const int32_t* idx, const float* w, float* y,
                                                int32_t* status, void* stream) {
  if (!wt || !x || !idx || !w || !y) return MOE_ERR_INVALID_ARG;
  if (E < 1 || top_k < 1 || top_k > E || H < 1 || I < 1 || I_shared < 0) return MOE_ERR_INVALID_ARG;
  if (T < 1 || T > kStaticMaxRows) return MOE_ERR_CAPACITY;
  if (E > 256 || top_k > 8 || H % 128 || I % 64 || I_shared % 64 ||
      !decode_shape_supported(H, I > I_shared ? I : I_shared))
    return MOE_ERR_UNSUPPORTED;
  const void* need[] = {x, idx, w, y, wt->w_gate, wt->w_up, wt->w_down, wt->s_gate, wt->s_up,
                        wt->s_down};
  for (const void* p : need)
    if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  const int has_shared = I_shared > 0;
  if (has_shared) {
    const void* nsh[] = {wt->sh_gate, wt->sh_up, wt->sh_down, wt->sh_s_gate, wt->sh_s_up,
                         wt->sh_s_down};
    for (const void* p : nsh)
      if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  }
  if (status && (reinterpret_cast<uintptr_t>(status) & 3u)) return MOE_ERR_INVALID_ARG;

  // Scratch layout for this call; rejected when it would not fit the static array.
  const int Imax = I > I_shared ? I : I_shared;
  const size_t R = (size_t)T * top_k + (has_shared ? T : 0);
  size_t off = 0;
  const size_t o_err = carve(off, sizeof(int));
  const size_t o_counts = carve(off, sizeof(int) * E);
  const size_t o_offsets = carve(off, sizeof(int) * (E + 1));
  const size_t o_perm = carve(off, sizeof(int) * T * top_k);
  const size_t o_groups = carve(off, sizeof(int4) * (E + 1));
  const size_t o_ngroups = carve(off, sizeof(int));
  const size_t o_rtok = carve(off, sizeof(int) * R);
  const size_t o_rw = carve(off, sizeof(float) * R);
  const size_t o_q = carve(off, (size_t)T * H);
  const size_t o_s = carve(off, sizeof(float) * T);
  const size_t o_h = carve(off, sizeof(float) * R * Imax);
  const size_t o_hq = carve(off, sizeof(__half) * R * Imax);
  const size_t o_sh = carve(off, sizeof(float) * R);
  const size_t o_sq = carve(off, sizeof(int));
  if (off > kScratchBytes) return MOE_ERR_CAPACITY;

  unsigned char* base = nullptr;
  int num_sms = 0;
  cudaError_t e = scratch_for_current_device(reinterpret_cast<void**>(&base), &num_sms);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver ? MOE_ERR_NO_DEVICE
                                                                       : MOE_ERR_CUDA;
  }
  // The decode kernels take up to 8 rows x H (gate/up) and 8 rows x Imax (down) bytes of
  // dynamic shared memory; their limit is set to this library's largest shapes.
  if ((e = decode_set_attributes()) != cudaSuccess) return MOE_ERR_CUDA;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* err = reinterpret_cast<int*>(base + o_err);
  // Only the error word must start at zero; every other scratch buffer is written before it
  // is read within the call (previous calls' contents are left in place).
  if (cudaMemsetAsync(err, 0, sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;

  DecodeArgs a;
  a.idx = idx;
  a.w = w;
  a.x = x;
  a.T = T;
  a.k = top_k;
  a.E = E;
  a.H = H;
  a.I = I;
  a.Is = I_shared;
  a.Imax = Imax;
  a.has_shared = has_shared;
  a.num_sms = num_sms;
  a.w_gate = wt->w_gate;
  a.w_up = wt->w_up;
  a.w_down = wt->w_down;
  a.s_gate = wt->s_gate;
  a.s_up = wt->s_up;
  a.s_down = wt->s_down;
  a.sh_gate = wt->sh_gate;
  a.sh_up = wt->sh_up;
  a.sh_down = wt->sh_down;
  a.sh_s_gate = wt->sh_s_gate;
  a.sh_s_up = wt->sh_s_up;
  a.sh_s_down = wt->sh_s_down;
  a.counts = reinterpret_cast<int*>(base + o_counts);
  a.offsets = reinterpret_cast<int*>(base + o_offsets);
  a.perm = reinterpret_cast<int*>(base + o_perm);
  a.groups = reinterpret_cast<int4*>(base + o_groups);
  a.n_groups = reinterpret_cast<int*>(base + o_ngroups);
  a.row_token = reinterpret_cast<int*>(base + o_rtok);
  a.row_w = reinterpret_cast<float*>(base + o_rw);
  a.qtok = reinterpret_cast<int8_t*>(base + o_q);
  a.stok = reinterpret_cast<float*>(base + o_s);
  a.h32 = reinterpret_cast<float*>(base + o_h);
  a.hq = reinterpret_cast<__half*>(base + o_hq);
  a.sh = reinterpret_cast<float*>(base + o_sh);
  a.sq_scratch = reinterpret_cast<int*>(base + o_sq);
  a.y = y;
  a.tap_gu = nullptr;
  a.tap_d = nullptr;
  a.err = err;
  if ((e = launch_decode(a, s, nullptr)) != cudaSuccess) return MOE_ERR_CUDA;
  if (status &&
      cudaMemcpyAsync(status, err, sizeof(int), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
