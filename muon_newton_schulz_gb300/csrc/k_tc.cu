// Tensor-core Newton-Schulz phases for sm_103a: tcgen05 UMMA with TMEM
// accumulators fed by TMA, in one persistent, warp-specialised kernel that is
// instantiated twice:
//
//   Gram (kGram = true):  C = alpha * P P^T (+ coef_prev * prev)
//       P is X (m x n, K = n) for A = X X^T, or A (m x m, K = m) for A A^T.
//       Only 128 x 256 output tiles that reach the upper triangle are
//       computed ("compute only the upper triangle of X X^T",
//       jsqmd.com/news/1098463, section 4.2); each element (r, c), r <= c,
//       is written to (r, c) and (c, r), so the result is exactly symmetric.
//   GEMM (kGram = false): X' = s * (a X + Bm X), Bm = b A + c A^2 (m x m).
//       The left operand is K-major (rows of Bm), the right one MN-major
//       (rows of X), so no transposed copy of X is ever made.
//
// One CTA per SM walks a flattened list of (group, matrix, tile) entries with
// a static stride (tile t -> CTA t mod grid): deterministic, and one launch
// covers the whole ragged batch.  Warp 0 issues TMA loads into a 4-stage
// shared-memory ring, warp 1 issues the MMAs (128 x 256 x 16 per instruction)
// into one of two TMEM accumulators (2 x 256 columns), and warps 2-5 drain the
// other accumulator through the fused epilogue, so the epilogue of tile t
// overlaps the MMAs of tile t + 1.
//
// Every wait is bounded (one second): on a time-out the kernel records the
// role in the status word, lets its copies and MMAs in flight finish, frees
// its TMEM and returns.
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "muon_internal.h"
#include "ptx_sm100.cuh"

namespace muon {

namespace {

constexpr int TM = kTcM;                    // 128 rows per tile (UMMA M)
constexpr int TN = kTcN;                    // 256 columns per tile (UMMA N)
constexpr int TK = kTcK;                    // 64 bf16 = 128 bytes = one swizzle row
constexpr int UK = 16;                      // K per UMMA instruction
constexpr int STAGES = 4;
constexpr int A_BYTES = TM * TK * 2;        // 16 KiB
constexpr int B_BYTES = TN * TK * 2;        // 32 KiB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 2 * TN;           // two fp32 accumulators
constexpr int kThreads = 192;               // 6 warps
constexpr int kEpiThreads = 128;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + 256;
constexpr uint64_t kWaitLimitNs = 1000000000ull;

struct Tile { int g, mat, bi, bj; };

__device__ __forceinline__ Tile decode_tile(const PhaseParams& p, int t, bool gram) {
  int g = 0;
  while (g + 1 < p.ngroups && t >= p.g[g + 1].tile_begin) ++g;
  const PhaseGroup& G = p.g[g];
  const int local = t - G.tile_begin;
  Tile tl;
  tl.g = g;
  tl.mat = local / G.tiles_per_mat;
  int r = local - tl.mat * G.tiles_per_mat;
  if (gram) {
    // column block bj (256 wide) needs row blocks bi (128 high) with
    // 128*bi < 256*(bj+1), i.e. bi <= 2*bj + 1
    int bj = 0;
    while (true) {
      const int cnt = min(2 * bj + 2, G.ni);
      if (r < cnt) break;
      r -= cnt;
      ++bj;
    }
    tl.bi = r;
    tl.bj = bj;
  } else {
    tl.bj = r / G.ni;
    tl.bi = r - tl.bj * G.ni;
  }
  return tl;
}

__device__ __forceinline__ bool wait_drain(uint64_t* bar, uint32_t parity) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

template <bool kGram>
__device__ __forceinline__ void run_producer(const PhaseParams& p, uint8_t* smem, uint64_t* full, uint64_t* empty,
                                             volatile int* abort) {
  int stage = 0;
  uint32_t phase = 0;
  uint32_t outstanding = 0, fill_parity = 0;
  bool ok = true;
  for (int t = blockIdx.x; ok && t < p.total_tiles; t += gridDim.x) {
    const Tile tl = decode_tile(p, t, kGram);
    const PhaseGroup& G = p.g[tl.g];
    const int nk = (G.K + TK - 1) / TK;
    const CUtensorMap* ma = &p.map_a[tl.g];
    const CUtensorMap* mb = &p.map_b[tl.g];
    for (int kb = 0; kb < nk; ++kb) {
      if (!ptx::mbar_wait_bounded(&empty[stage], phase ^ 1u, abort, p.status, kStatusTimeoutProducer,
                                  kWaitLimitNs)) {
        ok = false;
        break;
      }
      outstanding &= ~(1u << stage);
      uint8_t* sa = smem + stage * STAGE_BYTES;
      uint8_t* sb = sa + A_BYTES;
      ptx::mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
      const int k0 = kb * TK;
      if (kGram) {
        ptx::tma_load_4d(sa, ma, k0, tl.bi * TM, tl.mat, G.buf_in, &full[stage]);
        ptx::tma_load_4d(sb, ma, k0, tl.bj * TN, tl.mat, G.buf_in, &full[stage]);
        ptx::tma_load_4d(sb + A_BYTES, ma, k0, tl.bj * TN + TM, tl.mat, G.buf_in, &full[stage]);
      } else {
        ptx::tma_load_4d(sa, ma, k0, tl.bi * TM, tl.mat, 0, &full[stage]);
#pragma unroll
        for (int q = 0; q < TN / 64; ++q)
          ptx::tma_load_4d(sb + q * (64 * TK * 2), mb, tl.bj * TN + 64 * q, k0, tl.mat, G.buf_in, &full[stage]);
      }
      outstanding |= 1u << stage;
      fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
      if (++stage == STAGES) { stage = 0; phase ^= 1u; }
    }
  }
  if (!ok) {
    // let every copy this thread issued land before the CTA can exit
    for (int s = 0; s < STAGES; ++s)
      if ((outstanding >> s) & 1u)
        if (!wait_drain(&full[s], (fill_parity >> s) & 1u) && p.status) atomicOr(p.status, kStatusTimeoutDrain);
  }
}

template <bool kGram>
__device__ __forceinline__ void run_mma(const PhaseParams& p, uint8_t* smem, uint64_t* full, uint64_t* empty,
                                        uint64_t* tfull, uint64_t* tempty, uint64_t* drain, uint32_t tmem_base,
                                        volatile int* abort) {
  constexpr uint32_t idesc = ptx::idesc_bf16_f32(TM, TN, !kGram);
  int stage = 0;
  uint32_t phase = 0;
  int acc = 0;
  uint32_t acc_phase = 0;
  bool ok = true, issued = false;
  for (int t = blockIdx.x; ok && t < p.total_tiles; t += gridDim.x) {
    const Tile tl = decode_tile(p, t, kGram);
    const int nk = (p.g[tl.g].K + TK - 1) / TK;
    if (!ptx::mbar_wait_bounded(&tempty[acc], acc_phase ^ 1u, abort, p.status, kStatusTimeoutMma, kWaitLimitNs)) {
      ok = false;
      break;
    }
    ptx::tc_fence_after();
    const uint32_t d = tmem_base + (uint32_t)(acc * TN);
    for (int kb = 0; kb < nk; ++kb) {
      if (!ptx::mbar_wait_bounded(&full[stage], phase, abort, p.status, kStatusTimeoutMma, kWaitLimitNs)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t sa = ptx::smem_u32(smem + stage * STAGE_BYTES);
      const uint32_t sb = sa + A_BYTES;
#pragma unroll
      for (int kk = 0; kk < TK / UK; ++kk) {
        // K-major, 128B swizzle: rows 128 B apart, 8-row groups 1024 B apart;
        // the K offset inside the swizzle row is a plain start-address offset.
        const uint64_t ad = ptx::smem_desc(sa + kk * UK * 2, 16, 1024);
        uint64_t bd;
        if (kGram) {
          bd = ptx::smem_desc(sb + kk * UK * 2, 16, 1024);
        } else {
          // MN-major, 128B swizzle: 64-element MN blocks 8 KiB apart (LBO),
          // 8-row K groups 1024 B apart (SBO); UK rows of K = 2 KiB.
          bd = ptx::smem_desc(sb + kk * UK * 128, 64 * TK * 2, 1024);
        }
        ptx::umma_f16(d, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
      }
      ptx::umma_commit(&empty[stage]);
      issued = true;
      if (++stage == STAGES) { stage = 0; phase ^= 1u; }
    }
    if (!ok) break;
    ptx::umma_commit(&tfull[acc]);
    acc ^= 1;
    if (acc == 0) acc_phase ^= 1u;
  }
  if (!ok && issued) {
    ptx::umma_commit(drain);
    if (!wait_drain(drain, 0) && p.status) atomicOr(p.status, kStatusTimeoutDrain);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Gram epilogue for one 32-column chunk of one row.
//   Gram 1 (no prev):  A = alpha * acc, alpha = s^2 in the first iteration.
//   Gram 2 (prev = A): B = b * A + c * A^2 with A = A~ + R, where A~ is the
//     stored bf16 A and R the fp32 residual of its diagonal (diag_in), so
//     A^2 = acc + A~ o (R_r + R_c) + R^2 on the diagonal, acc = A~ A~.
// The diagonal goes to diag_out: its bf16 rounding residual, or with
// diag_exact the value itself (the bf16 matrix then holds 0 there).
__device__ __forceinline__ void gram_chunk(const PhaseParams& p, const PhaseGroup& G, const Tile& tl, int row,
                                           int c0, const uint32_t (&v)[32]) {
  const int m = G.m;
  if (row >= m) return;
  const bool full_chunk = c0 + 32 <= m;
  float f[32];
  if (G.prev) {
    const __nv_bfloat16* pr =
        reinterpret_cast<const __nv_bfloat16*>(G.prev) + (int64_t)tl.mat * G.prev_stride + (int64_t)row * G.ld_prev + c0;
    const float* rin = G.diag_in ? G.diag_in + (int64_t)tl.mat * G.diag_stride : nullptr;
    float pa[32], rc[32];
    if (full_chunk) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 u = *reinterpret_cast<const uint4*>(pr + 8 * i);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&w[h]);
          pa[8 * i + 2 * h] = __low2float(b2);
          pa[8 * i + 2 * h + 1] = __high2float(b2);
        }
      }
      if (rin) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 q = *reinterpret_cast<const float4*>(rin + c0 + 4 * i);
          rc[4 * i] = q.x; rc[4 * i + 1] = q.y; rc[4 * i + 2] = q.z; rc[4 * i + 3] = q.w;
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        pa[j] = c0 + j < m ? __bfloat162float(pr[j]) : 0.f;
        rc[j] = (rin && c0 + j < m) ? rin[c0 + j] : 0.f;
      }
    }
    if (!rin) {
#pragma unroll
      for (int j = 0; j < 32; ++j) rc[j] = 0.f;
    }
    const float rr = rin ? rin[row] : 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      float acc = fmaf(pa[j], rr + rc[j], __uint_as_float(v[j]));
      float aex = pa[j];
      if (c0 + j == row) {
        acc = fmaf(rr, rr, acc);
        aex += rr;
      }
      f[j] = fmaf(p.coef_prev, aex, p.coef_acc * acc);
    }
  } else {
    float alpha = p.coef_acc;
    if (p.scale) {
      const float s = p.scale[G.first + tl.mat];
      alpha *= s * s;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) f[j] = alpha * __uint_as_float(v[j]);
  }
  if (G.diag_out && row >= c0 && row < c0 + 32) {
    float* dout = G.diag_out + (int64_t)tl.mat * G.diag_stride;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (c0 + j == row) {
        const float d = f[j];
        if (p.diag_exact) {
          dout[row] = d;
          f[j] = 0.f;
        } else {
          dout[row] = d - __bfloat162float(__float2bfloat16_rn(d));
        }
      }
    }
  }
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(G.out) + (int64_t)tl.mat * G.out_stride;
  const int64_t ld = G.ld_out;
  __nv_bfloat16* o = out + (int64_t)row * ld + c0;
  if (row <= c0 && full_chunk) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint4 u;
      u.x = pack_bf16x2(f[8 * i + 0], f[8 * i + 1]);
      u.y = pack_bf16x2(f[8 * i + 2], f[8 * i + 3]);
      u.z = pack_bf16x2(f[8 * i + 4], f[8 * i + 5]);
      u.w = pack_bf16x2(f[8 * i + 6], f[8 * i + 7]);
      *reinterpret_cast<uint4*>(o + 8 * i) = u;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (c0 + j < m && row <= c0 + j) o[j] = __float2bfloat16_rn(f[j]);
  }
  // mirror the strict upper part: lanes hold consecutive rows, so each
  // column's 32 values form one contiguous 64-byte run of row (c0 + j)
#pragma unroll
  for (int j = 0; j < 32; ++j)
    if (c0 + j < m && row < c0 + j) out[(int64_t)(c0 + j) * ld + row] = __float2bfloat16_rn(f[j]);
}

__device__ __forceinline__ void gemm_chunk(const PhaseParams& p, const PhaseGroup& G, const Tile& tl, int row,
                                           int c0, const uint32_t (&v)[32]) {
  const int m = G.m, n = G.n;
  if (row >= m) return;
  const float s = p.scale ? p.scale[G.first + tl.mat] : 1.f;
  // a plus this row's fp32 diagonal term of B (residual or exact diagonal)
  const float a = p.coef_prev + (G.diag_in ? G.diag_in[(int64_t)tl.mat * G.diag_stride + row] : 0.f);
  const float* xin = reinterpret_cast<const float*>(G.prev) + (int64_t)tl.mat * G.prev_stride +
                     (int64_t)row * G.ld_prev + c0;
  float* xo = reinterpret_cast<float*>(G.out) + (int64_t)tl.mat * G.out_stride + (int64_t)row * G.ld_out + c0;
  __nv_bfloat16* xb = G.out_b ? G.out_b + (int64_t)tl.mat * G.outb_stride + (int64_t)row * G.ld_outb + c0 : nullptr;
  float f[32];
  if (c0 + 32 <= n) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 x = *reinterpret_cast<const float4*>(xin + 4 * i);
      f[4 * i + 0] = s * fmaf(a, x.x, __uint_as_float(v[4 * i + 0]));
      f[4 * i + 1] = s * fmaf(a, x.y, __uint_as_float(v[4 * i + 1]));
      f[4 * i + 2] = s * fmaf(a, x.z, __uint_as_float(v[4 * i + 2]));
      f[4 * i + 3] = s * fmaf(a, x.w, __uint_as_float(v[4 * i + 3]));
      *reinterpret_cast<float4*>(xo + 4 * i) = make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
    }
    if (xb) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint4 u;
        u.x = pack_bf16x2(f[8 * i + 0], f[8 * i + 1]);
        u.y = pack_bf16x2(f[8 * i + 2], f[8 * i + 3]);
        u.z = pack_bf16x2(f[8 * i + 4], f[8 * i + 5]);
        u.w = pack_bf16x2(f[8 * i + 6], f[8 * i + 7]);
        *reinterpret_cast<uint4*>(xb + 8 * i) = u;
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (c0 + j < n) {
        const float val = s * fmaf(a, xin[j], __uint_as_float(v[j]));
        xo[j] = val;
        if (xb) xb[j] = __float2bfloat16_rn(val);
      }
    }
  }
}

template <bool kGram>
__device__ __forceinline__ void run_epilogue(const PhaseParams& p, uint64_t* tfull, uint64_t* tempty,
                                             uint32_t tmem_base, int quarter, int lane, volatile int* abort) {
  int acc = 0;
  uint32_t acc_phase = 0;
  for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
    const Tile tl = decode_tile(p, t, kGram);
    const PhaseGroup& G = p.g[tl.g];
    if (!ptx::mbar_wait_bounded(&tfull[acc], acc_phase, abort, p.status, kStatusTimeoutEpilogue, kWaitLimitNs))
      break;
    ptx::tc_fence_after();
    const int row0 = tl.bi * TM + quarter * 32;   // first row of this warp
    const int row = row0 + lane;
    const int limit = kGram ? G.m : G.n;
    const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * TN);
#pragma unroll 1
    for (int ch = 0; ch < TN / 32; ++ch) {
      const int c0 = tl.bj * TN + ch * 32;
      if (c0 >= limit) break;                       // uniform across the CTA
      if (kGram && c0 + 31 < row0) continue;        // chunk wholly below the diagonal for this warp
      uint32_t v[32];
      ptx::tmem_ld_32x32b_x32(tbase + (uint32_t)(ch * 32), v);
      ptx::tmem_ld_wait();
      if (kGram) gram_chunk(p, G, tl, row, c0, v);
      else gemm_chunk(p, G, tl, row, c0, v);
    }
    ptx::tc_fence_before();
    ptx::mbar_arrive(&tempty[acc]);
    acc ^= 1;
    if (acc == 0) acc_phase ^= 1u;
  }
}

template <bool kGram>
__global__ void __launch_bounds__(kThreads, 1) k_ns_tc(const __grid_constant__ PhaseParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], kEpiThreads);
    }
    ptx::mbar_init(drain, 1);
    *abort = 0;
    ptx::fence_mbar_init();
    for (int g = 0; g < p.ngroups; ++g) {
      ptx::prefetch_tmap(&p.map_a[g]);
      if (!kGram) ptx::prefetch_tmap(&p.map_b[g]);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) run_producer<kGram>(p, smem, full, empty, abort);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) run_mma<kGram>(p, smem, full, empty, tfull, tempty, drain, tmem_base, abort);
    __syncwarp();
  } else {
    run_epilogue<kGram>(p, tfull, tempty, tmem_base, warp & 3, lane, abort);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <bool kGram>
int launch_tc(const PhaseParams& p, int grid, void* stream) {
  if (p.total_tiles == 0) return 0;
  cudaError_t e = cudaFuncSetAttribute(k_ns_tc<kGram>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return (int)e;
  if (grid > p.total_tiles) grid = p.total_tiles;
  k_ns_tc<kGram><<<grid, kThreads, SMEM_BYTES, (cudaStream_t)stream>>>(p);
  return (int)cudaGetLastError();
}

}  // namespace

int tc_smem_bytes() { return SMEM_BYTES; }
int launch_gram_tc(const PhaseParams& p, int grid, void* stream) { return launch_tc<true>(p, grid, stream); }
int launch_gemm_tc(const PhaseParams& p, int grid, void* stream) { return launch_tc<false>(p, grid, stream); }

}  // namespace muon
