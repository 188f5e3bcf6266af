// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kBM = 128;        // tensor-core tile rows (weight rows: the MMA's M)
#ifndef MOE_MAX_TOK_TILE
#define MOE_MAX_TOK_TILE 192
#endif
constexpr int kMaxTokTile = MOE_MAX_TOK_TILE;  // token rows per tile (the MMA's N), at most
static_assert(kMaxTokTile % 16 == 0 && kMaxTokTile <= 192, "token tile");
// Token-tile TMA boxes: one tensor map per box height (multiples of kXStep rows up to the
// token tile) over the same token-row operand, so that each 64-K half of a token stage is one
// TMA load.
constexpr int kXStep = 16;
constexpr int kXMaps = kMaxTokTile / kXStep;
struct XMaps {
  CUtensorMap m[kXMaps];
};
constexpr int kBK = 64;         // K elements per token TMA box (128 bytes of fp16)
constexpr int kKS = 128;        // K elements per pipeline stage (two token boxes, 8 MMAs)
constexpr int kChunkK = 1024;   // K elements summed in one fp32 TMEM accumulator
// TMEM columns of the GEMMs: two accumulator slots of up to kMaxTokTile columns each, then
// the A-operand stages (one 128-row x 128-K fp16 weight tile = 64 columns each).
constexpr int kAccCols = 384;
constexpr int kTokPerBlk = 32;  // tokens per routing/histogram block (a 64-bit mask per expert holds them)
// Largest T the deduplicated weight-streaming kernels take, and the default dispatch
// threshold of a plan (T <= threshold runs them, larger T the grouped GEMMs). Measured on
// GB300 for the 35B-A3B-shaped layer (H=2048, E=128, k=8, I=512, Zipf 1.1 routing, routing
// inside the forward, weights streamed from HBM): streaming 67.7 us against grouped 73.6 us
// per layer at T=24, 78.4 against 74.2 at T=32.
constexpr int kDecodeMaxRows = 64;
constexpr int kDecodeDefaultRows = 24;
constexpr int kDecodeMaxH = 8192;  // largest H and intermediate size the decode kernels take
constexpr int kDecodeMaxI = 4096;
constexpr int kREB = 16;  // experts per router tensor-core tile (packed router weight block)

// One unit of grouped-GEMM work: token rows [row0, row0 + rows) of group `group` (expert id,
// or E for the shared expert) against weight rows [m0, m0 + 128).
// Stored as int4 {group, row0, rows, m0}.

struct GemmArgs {
  const int4* items;
  const int* n_items;
  int E;
  int TN;                // token tile (items have rows <= TN)
  // The same work in token tiles of TN_c rows, for a launch whose exactness bound fails and
  // takes 1024-K accumulator chunks (which fit TMEM only with the smaller tile); NULL when
  // TN_c == TN.
  const int4* items_c = nullptr;
  const int* n_items_c = nullptr;
  int TN_c = 0;
  int K_r, K_s;          // reduction length of routed / shared groups
  int I, Is, Imax, H;
  // gate/up epilogue
  const float* sx;       // per row activation scale
  const float* s_g;      // [E, I]
  const float* s_u;      // [E, I]
  const float* sh_s_g;   // [Is]
  const float* sh_s_u;   // [Is]
  float* h32;            // [R, Imax]
  // down epilogue
  const float* s_h;      // per row
  const float* s_d;      // [E, H]
  const float* sh_s_d;   // [H]
  const int* row_token;  // per row
  const float* row_w;    // per row
  float* y;              // [T, H] layer output: every row adds w * d into its token's row
  // exactness bound of one fp32 accumulator over the whole K (see gemm_tc.cu)
  const int* row_sq_max;  // max over A rows of sum(q^2), written by the row producer
  const int* w_sq_max;    // max over weight rows of sum(q_w^2), written at packing
  // taps (NULL = off)
  int32_t* tap;
  int* err;
  // NVFP4 weights (the fp4 kernels): tiles packed by launch_pack_fp4_tiles, one
  // kFp4TileBytes block per (128-row tile, 128-K stage); rows_r / rows_s = weight rows of a
  // routed / the shared group. Accumulator taps are then fp64.
  const uint8_t* w4 = nullptr;
  const uint8_t* w4s = nullptr;
  int rows_r = 0, rows_s = 0;
  double* tap_f64 = nullptr;
};

// One (128-row, 128-K) NVFP4 weight tile as the tensor-core kernels read it: 8192 code bytes
// (row r's 64 bytes at r * 64, its 16-byte chunk c at chunk position c ^ ((r >> 1) & 3)), then
// 1024 block-scale bytes (row r's 8 at 8192 + r * 8).
constexpr int kFp4TileBytes = 9216;

cudaError_t launch_grouped_gemm(bool gate_up, bool fp4, const GemmArgs& a, const XMaps& tmX,
                                const CUtensorMap& tmW, const CUtensorMap& tmWs, int grid,
                                cudaStream_t s);
// Repacks NVFP4 weight rows (codes [n_mats, rows, K/2], scales [n_mats, rows, K/16]; with
// codes1 / sc1 given, two matrices interleaved row by row: tile row 2i = row i of matrix 0,
// 2i + 1 = row i of matrix 1) into tiles [n_mats][tiles][ceil(K/128)][kFp4TileBytes], K past
// the matrix zero.
cudaError_t launch_pack_fp4_tiles(const uint8_t* codes0, const uint8_t* codes1, const uint8_t* sc0,
                                  const uint8_t* sc1, int n_mats, int rows, int K, uint8_t* out,
                                  cudaStream_t s);
// out[m * n + i] = v[m] (m < n_mats, i < n): a matrix scale as per-row scales.
cudaError_t launch_fill_rows(const float* v, int n_mats, int n, float* out, cudaStream_t s);
cudaError_t gemm_set_attributes();
cudaError_t gemm_max_ctas(bool gate_up, int* n);

cudaError_t launch_requant(const float* h32, int R, int T_sh, int I, int Is, int Imax,
                           __half* hq, float* sh, int* sq_max, cudaStream_t s);

// routing / permutation
cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* idx, float* w,
                         int* err, cudaStream_t s);

struct PrepArgs {
  const int32_t* idx;
  const float* w;
  const float* logits = nullptr;  // [T, E]: route here into idx_out / w_out (idx, w = those)
  int32_t* idx_out = nullptr;
  float* w_out = nullptr;
  int* scan_ctr = nullptr;        // one zero-initialised counter, left at zero
  const uint16_t* x;
  int T, k, E, H, I, Is, has_shared;
  unsigned long long* bmask;  // [nblk, E]
  int* bhist;                 // [nblk, E]
  int* counts;                // [E]
  int* offsets;               // [E + 1]
  int* perm;                  // [T*k]
  // work lists: 0 gate/up, 1 down (token tiles tn[0], tn[1]); 2, 3 the same in the smaller
  // tiles of the exact chunked accumulation (items[l] NULL: list not built)
  int tn[4];
  int4* items[4];
  int* n_items;               // [4]
  __half* xq;                 // [R, H] activation codes as fp16 integers, row order
  float* sx;                  // [R]
  int* row_token;             // [R]
  float* row_w;               // [R]
  float* y;                   // [T, H] layer output, zeroed here (the down GEMM adds into it)
  int8_t* qtok;               // [T, H] or NULL
  float* stok;                // [T]   or NULL
  int* sq_max;                // [2] row sum(q^2) maxima (gate/up rows, down rows), reset here
  int* err;
  int* gbase = nullptr;       // [4][kMaxGroups + 1] item bases per group and list
};
constexpr int kMaxGroups = 257;  // routed experts (<= 256) + the shared expert
cudaError_t launch_prefill_prep(const PrepArgs& a, cudaStream_t s);

// One layer's NVFP4 expert weights (the caller's arrays; see moe_weights_nvfp4).
struct Fp4Weights {
  const uint8_t* w_gate = nullptr;   // [E, I, H/2] E2M1 codes, element 2j in the low nibble
  const uint8_t* w_up = nullptr;
  const uint8_t* w_down = nullptr;   // [E, H, I/2]
  const uint8_t* b_gate = nullptr;   // [E, I, H/16] E4M3 block scales
  const uint8_t* b_up = nullptr;
  const uint8_t* b_down = nullptr;   // [E, H, I/16]
  const float* g_gate = nullptr;     // [E] matrix scales
  const float* g_up = nullptr;
  const float* g_down = nullptr;
  const uint8_t* sh_gate = nullptr;  // [Is, H/2]
  const uint8_t* sh_up = nullptr;
  const uint8_t* sh_down = nullptr;  // [H, Is/2]
  const uint8_t* sh_b_gate = nullptr;
  const uint8_t* sh_b_up = nullptr;
  const uint8_t* sh_b_down = nullptr;
  const float* sh_g = nullptr;       // [3] gate, up, down
};

struct DecodeArgs {
  const int32_t* idx;
  const float* w;
  const float* logits = nullptr;  // [T, E]: route in the prep kernel into idx_out / w_out
  int32_t* idx_out = nullptr;
  float* w_out = nullptr;
  const uint16_t* x;
  int T, k, E, H, I, Is, Imax, has_shared, num_sms;
  const int8_t* w_gate;
  const int8_t* w_up;
  const int8_t* w_down;
  const float* s_gate;
  const float* s_up;
  const float* s_down;
  const int8_t* sh_gate;
  const int8_t* sh_up;
  const int8_t* sh_down;
  const float* sh_s_gate;
  const float* sh_s_up;
  const float* sh_s_down;
  int* counts;
  int* offsets;
  int* perm;
  int4* groups;      // [E + 1] {group, row0, nrows, 0}
  int* n_groups;
  int* row_token;
  float* row_w;
  int8_t* qtok;      // [T, H]
  float* stok;       // [T]
  float* h32;        // [R, Imax]
  __half* hq;        // [R, Imax] requantised h codes (fp16 integers)
  float* sh;         // [R]       their scales
  int* sq_scratch;   // one word the requantisation pass writes its sum(q^2) maximum to
  float* y;
  int32_t* tap_gu;   // NULL = off
  int32_t* tap_d;
  int* err;
  // NVFP4 experts (fp4 != 0): the weights above are unused, these are read instead, and the
  // accumulator taps are fp64 (exact sums of q * e2m1 * e4m3)
  int fp4 = 0;
  Fp4Weights f;
  double* tap_gu_f64 = nullptr;
  double* tap_d_f64 = nullptr;
};
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s, cudaEvent_t* ev);
cudaError_t decode_set_attributes();
bool decode_shape_supported(int H, int Imax);  // shapes the streaming kernels take

// Sets *err to MOE_ERR_DEVICE when one of the n bytes is not a finite non-negative E4M3 value.
cudaError_t launch_check_e4m3(const uint8_t* b, size_t n, int* err, cudaStream_t s);

// weight packing and the stacked-prefill helpers
cudaError_t launch_pack_gu8(const int8_t* gate, const int8_t* up, int n_mats, int I, int H,
                            int8_t* out, cudaStream_t s);
cudaError_t launch_row_sq_max(const int8_t* w, size_t rows, int cols, int* out, cudaStream_t s);
cudaError_t launch_router_logits(const uint16_t* x, const float* wr, int T, int H, int E,
                                 float* out, cudaStream_t s);
cudaError_t launch_residual(uint16_t* x, const float* y, size_t n, cudaStream_t s);
cudaError_t launch_selftest_wait(int* err, cudaStream_t s);
cudaError_t launch_router_pack(const float* w, int H, int E, uint16_t* packed, cudaStream_t s);
cudaError_t launch_router_tc(int T, int H, int E, float* out, const CUtensorMap& tmA,
                             const CUtensorMap& tmB, cudaStream_t s);
cudaError_t launch_rmsnorm_residual(uint16_t* x, const float* y, uint16_t* x_in, int T, int H,
                                    cudaStream_t s);

}  // namespace moe
