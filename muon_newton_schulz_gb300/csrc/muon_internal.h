// Internal structures shared by the host planner and the kernels.
// Everything a launch needs travels in its (large, __grid_constant__) kernel
// parameter block, so a step issues no host-to-device copies.
#pragma once

#include <cstdint>
#include <string>
#include <cuda.h>
#include <cuda_bf16.h>

struct muon_handle_s;

namespace muon {

constexpr int kMaxGroups = 16;     // shape groups per Newton-Schulz launch
constexpr int kMaxEltMats = 64;    // matrices per elementwise launch
constexpr int kEltTile = 64;       // elementwise kernels work on 64 x 64 tiles
constexpr int kSimtTile = 64;      // fp32 validation kernels: 64 x 64 output tiles

// Status bits written by kernels into the workspace status word.
constexpr uint32_t kStatusTimeoutProducer = 1u << 0;
constexpr uint32_t kStatusTimeoutMma = 1u << 1;
constexpr uint32_t kStatusTimeoutEpilogue = 1u << 2;
constexpr uint32_t kStatusTimeoutDrain = 1u << 3;

// Weight-update target of one matrix, written into the workspace by the
// momentum kernel and read by the last GEMM, which applies the update in its
// epilogue.  wmap is a 2-D tensor map of W whose box covers one epilogue
// chunk: kGemmChunk columns x 32 rows (wide) or 32 columns x kGemmChunk rows
// (tall, where W is X transposed).
struct ApplyDesc {
  void* W;
  float* O_out;
  int64_t ldw, ldo;
  float lr_eff;
  int32_t w_bf16;
  int32_t tall;
  int32_t rows, cols;
  int32_t pad[3];
};

struct ApplyEntry {   // 128-byte aligned through CUtensorMap
  CUtensorMap wmap;
  ApplyDesc d;
};

// One matrix as the momentum / norm / cast and apply kernels see it.
struct EltMat {
  const float* G;
  float* M;
  void* W;
  float* O_out;
  // X0 written by K1 (wide orientation): fp32 (validation mode) or the bf16
  // pair hi = bf16(x), lo = bf16(x - hi) (tensor-core mode); the other null
  float* xm0;
  __nv_bfloat16* xhi0;
  __nv_bfloat16* xlo0;
  // X after the last iteration, read by the apply kernel, in the same form
  const float* xm_final;
  const __nv_bfloat16* xhi_final;
  const __nv_bfloat16* xlo_final;
  int64_t ldg, ldm, ldw, ldo, ldx;
  int64_t tile_begin;      // first 64x64 tile of this matrix in the launch-wide numbering
  int64_t partial_begin;   // first partial-sum slot of this matrix
  int32_t rows, cols;
  int32_t tiles_c;         // 64-wide tiles along cols
  int32_t ntiles;          // tiles of this matrix
  int32_t tall;            // rows > cols: X is M^T
  int32_t w_bf16;
  int32_t mat;             // global matrix index (scale[])
  float lr_eff;            // lr * scale_coeff * sqrt(max(rows, cols))
  CUtensorMap wmap;        // W tensor map published for the last GEMM (bf16 mode)
};

struct EltParams {
  EltMat mats[kMaxEltMats];
  int32_t nmats;
  int32_t nesterov;
  int32_t dampening;       // 1: the gradient enters the momentum as (1 - beta) * G
  int32_t apply_scale;     // apply: multiply O by scale[] (zero iterations)
  float beta;
  float eps;
  int64_t total_tiles;
  double* partials;        // one sum of squares per 64x64 tile
  float* scale;            // per matrix 1 / (||X0||_F + eps)
  uint32_t* status;        // kernel status word: cleared by the first momentum CTA of a step
  ApplyEntry* apply;       // per matrix, filled by the momentum kernel (or null)
};

// One group of same-shape matrices (wide orientation m x n) in one
// Newton-Schulz phase launch.
struct PhaseGroup {
  int32_t m, n;            // wide dims
  int32_t count;           // matrices in the group
  int32_t first;           // global index of its first matrix (scale[])
  int32_t K;               // contraction length
  int32_t ni, nj;          // output tile grid per matrix
  int32_t tiles_per_mat;
  int32_t tile_begin;      // first tile of this group in the launch
  int32_t buf_in;          // ping-pong coordinate of the X operand (tensor maps)
  int32_t buf_out;         // ping-pong coordinate of the GEMM output (tensor maps)
  // operands, for kernels that read them directly (fp32 validation path)
  const void* opP; int64_t ld_p; int64_t p_stride;   // Gram operand / GEMM left operand
  const void* opX; int64_t ld_x; int64_t x_stride;   // GEMM right operand
  // epilogue
  const void* prev; int64_t ld_prev; int64_t prev_stride;  // Gram 2: A; GEMM (validation mode): fp32 X
  void* out; int64_t ld_out; int64_t out_stride;           // Gram: A or B; GEMM (validation mode): fp32 X'
  __nv_bfloat16* out_b; int64_t ld_outb; int64_t outb_stride;  // unused (null)
  // fp32 per-row diagonal terms (tensor-core path; null elsewhere), stride per matrix
  const float* diag_in; float* diag_out; int64_t diag_stride;
};

struct PhaseParams {
  CUtensorMap map_a[kMaxGroups];   // tensor-core path: left operand (and Gram right operand)
  CUtensorMap map_b[kMaxGroups];   // tensor-core path: GEMM right operand (MN-major X)
  CUtensorMap map_c[kMaxGroups];   // epilogue: Gram output (bf16, 32x32 box) / GEMM X hi in+out (32 rows x chunk)
  CUtensorMap map_d[kMaxGroups];   // epilogue: Gram 2 previous A (32x32 box) / GEMM X lo in+out (32 rows x chunk)
  PhaseGroup g[kMaxGroups];
  int32_t ngroups;
  int32_t total_tiles;
  const float* scale;      // per-matrix s folded into this phase, or null
  float coef_acc;          // Gram: multiplies the product (1 or c)
  float coef_prev;         // Gram 2: b (times A); GEMM: a (times X)
  int32_t diag_exact;      // Gram 2: 1 = keep B's diagonal out of the bf16 matrix (fp32 only)
  uint32_t* status;        // kernel status word (bounded waits)
  const ApplyEntry* apply; // last GEMM: apply W -= lr_eff * X' instead of storing X' (or null)
  int32_t withhold_loads;  // test hook: the producer issues no loads, so the waits run out
  int32_t x_lo_in;         // GEMM: the input X has its lo half (else X = hi)
  int32_t x_lo_out;        // GEMM: store the lo half of X' (else X' = hi only)
};

// Handle accessors for the allocation-free entry point (defined in muon_api.cpp).
int handle_device(::muon_handle_s* h);
void set_handle_error(::muon_handle_s* h, const std::string& msg);
// Device address of muon_step_noalloc's fixed array on `device` (defined in
// muon_noalloc.cu); returns a cudaError_t as int.
int static_workspace(int device, void** out);

// Launch wrappers (defined in the .cu files).  Each returns the launch's
// cudaError_t as int.  pdl: launch as a programmatic dependent of the
// previous kernel on the stream (every launch of a step but the first).
int launch_momentum_norm(const EltParams& p, void* stream, bool pdl);
int launch_norm_finalize(const EltParams& p, void* stream, bool pdl);
int launch_apply(const EltParams& p, void* stream, bool pdl);
int launch_gram_f32(const PhaseParams& p, void* stream, bool pdl);
int launch_gemm_f32(const PhaseParams& p, void* stream, bool pdl);
int launch_gram_tc(const PhaseParams& p, int grid, void* stream, bool pdl);
int launch_gemm_tc(const PhaseParams& p, int grid, void* stream, bool pdl);
int launch_gram_tc_pair(const PhaseParams& p, int sm_count, void* stream, bool pdl);
int launch_gemm_tc_pair(const PhaseParams& p, int sm_count, void* stream, bool pdl);

// Programmatic dependent launch between the kernels of a step, unless built
// with -DMUON_USE_PDL=0.
#ifndef MUON_USE_PDL
#define MUON_USE_PDL 1
#endif
constexpr bool kUsePdl = MUON_USE_PDL != 0;
int tc_smem_bytes();

// Tensor-core tile shape (used by the planner to count tiles): a CTA covers
// kTcM rows; a CTA pair (cta_group::2) covers 2 * kTcM rows.
constexpr int kTcM = 128;
constexpr int kTcN = 256;
constexpr int kTcK = 64;

// Columns per GEMM epilogue chunk (16 or 32): the X tiles it moves are
// 32 rows x chunk bf16, i.e. 32- or 64-byte rows.
#ifndef MUON_GEMM_CHUNK
#define MUON_GEMM_CHUNK 32
#endif
constexpr int kGemmChunk = MUON_GEMM_CHUNK;
static_assert(kGemmChunk == 16 || kGemmChunk == 32, "GEMM epilogue chunk of 16 or 32 columns");

// Stored Newton-Schulz iterates, counted from the last, that keep only the
// bf16 hi half of X (tensor-core mode).
#ifndef MUON_X_LO_TAIL
#define MUON_X_LO_TAIL 1
#endif

// The Newton-Schulz phases run on CTA pairs (256 x 256 tiles) unless built
// with -DMUON_USE_PAIR=0 (single CTAs, 128 x 256 tiles).
#ifndef MUON_USE_PAIR
#define MUON_USE_PAIR 1
#endif
constexpr bool kUsePair = MUON_USE_PAIR != 0;

}  // namespace muon
