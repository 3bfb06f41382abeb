// fp32 validation path of the Newton-Schulz phases on the CUDA cores.
//
// Same phase structure and epilogues as the tensor-core path, fp32 operands
// and fp32 FMA accumulation throughout, so that it can be held to a much
// tighter tolerance against the fp64 oracle.  64 x 64 output tiles, 256
// threads, 4 x 4 outputs per thread, K staged through shared memory in
// chunks of 16.  Gram tiles: only tiles with bi <= bj are computed and each
// element is written to (r, c) and mirrored to (c, r).
#include <cuda_runtime.h>

#include "muon_internal.h"
#include "launch_util.cuh"

namespace muon {

namespace {

constexpr int T = kSimtTile;   // 64
constexpr int KC = 16;
constexpr int kThreads = 256;

struct Tile { int g, mat, bi, bj; };

__device__ __forceinline__ Tile decode(const PhaseParams& p, int t, bool gram) {
  int g = 0;
  while (g + 1 < p.ngroups && t >= p.g[g + 1].tile_begin) ++g;
  const PhaseGroup& G = p.g[g];
  const int local = t - G.tile_begin;
  Tile tl;
  tl.g = g;
  tl.mat = local / G.tiles_per_mat;
  int r = local - tl.mat * G.tiles_per_mat;
  if (gram) {  // column block bj holds bj+1 upper tiles
    int bj = 0;
    while (r >= bj + 1) { r -= bj + 1; ++bj; }
    tl.bi = r;
    tl.bj = bj;
  } else {
    tl.bj = r / G.ni;
    tl.bi = r - tl.bj * G.ni;
  }
  return tl;
}

// out = alpha * P P^T (+ coef_prev * prev), alpha = coef_acc * s^2.
__global__ void __launch_bounds__(kThreads) k_gram_f32(const __grid_constant__ PhaseParams p) {
  __shared__ float As[KC][T + 4];
  __shared__ float Bs[KC][T + 4];
  grid_dependency_wait();
  allow_dependent_launch();
  const Tile tl = decode(p, blockIdx.x, true);
  const PhaseGroup& G = p.g[tl.g];
  const float* P = reinterpret_cast<const float*>(G.opP) + (int64_t)tl.mat * G.p_stride;
  const int m = G.m, K = G.K;
  const int64_t ld = G.ld_p;
  const int i0 = tl.bi * T, j0 = tl.bj * T;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};

  for (int k0 = 0; k0 < K; k0 += KC) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int idx = threadIdx.x + kThreads * e;
      const int row = idx >> 4, kk = idx & 15;
      const int gk = k0 + kk;
      As[kk][row] = (i0 + row < m && gk < K) ? P[(int64_t)(i0 + row) * ld + gk] : 0.f;
      Bs[kk][row] = (j0 + row < m && gk < K) ? P[(int64_t)(j0 + row) * ld + gk] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < KC; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) { a[u] = As[kk][ty * 4 + u]; b[u] = Bs[kk][tx * 4 + u]; }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(a[u], b[v], acc[u][v]);
    }
    __syncthreads();
  }

  float alpha = p.coef_acc;
  if (p.scale) { const float s = p.scale[G.first + tl.mat]; alpha *= s * s; }
  const float* prev = G.prev ? reinterpret_cast<const float*>(G.prev) + (int64_t)tl.mat * G.prev_stride : nullptr;
  float* out = reinterpret_cast<float*>(G.out) + (int64_t)tl.mat * G.out_stride;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int r = i0 + ty * 4 + u;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int c = j0 + tx * 4 + v;
      if (r < m && c < m && r <= c) {
        float val = alpha * acc[u][v];
        if (prev) val = fmaf(p.coef_prev, prev[(int64_t)r * G.ld_prev + c], val);
        out[(int64_t)r * G.ld_out + c] = val;
        if (r < c) out[(int64_t)c * G.ld_out + r] = val;
      }
    }
  }
}

// out = s * (coef_prev * prev + Bm X), Bm = opP (m x m), X = opX (m x n).
__global__ void __launch_bounds__(kThreads) k_gemm_f32(const __grid_constant__ PhaseParams p) {
  __shared__ float As[KC][T + 4];
  __shared__ float Bs[KC][T + 4];
  grid_dependency_wait();
  allow_dependent_launch();
  const Tile tl = decode(p, blockIdx.x, false);
  const PhaseGroup& G = p.g[tl.g];
  const float* Bm = reinterpret_cast<const float*>(G.opP) + (int64_t)tl.mat * G.p_stride;
  const float* X = reinterpret_cast<const float*>(G.opX) + (int64_t)tl.mat * G.x_stride;
  const int m = G.m, n = G.n, K = G.K;
  const int i0 = tl.bi * T, j0 = tl.bj * T;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};

  for (int k0 = 0; k0 < K; k0 += KC) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int idx = threadIdx.x + kThreads * e;
      {
        const int row = idx >> 4, kk = idx & 15;
        const int gk = k0 + kk;
        As[kk][row] = (i0 + row < m && gk < K) ? Bm[(int64_t)(i0 + row) * G.ld_p + gk] : 0.f;
      }
      {
        const int kk = idx >> 6, col = idx & 63;
        const int gk = k0 + kk;
        Bs[kk][col] = (gk < K && j0 + col < n) ? X[(int64_t)gk * G.ld_x + j0 + col] : 0.f;
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < KC; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) { a[u] = As[kk][ty * 4 + u]; b[u] = Bs[kk][tx * 4 + u]; }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(a[u], b[v], acc[u][v]);
    }
    __syncthreads();
  }

  const float s = p.scale ? p.scale[G.first + tl.mat] : 1.f;
  const float* xin = reinterpret_cast<const float*>(G.prev) + (int64_t)tl.mat * G.prev_stride;
  float* xout = reinterpret_cast<float*>(G.out) + (int64_t)tl.mat * G.out_stride;
  __nv_bfloat16* xb = G.out_b ? G.out_b + (int64_t)tl.mat * G.outb_stride : nullptr;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int r = i0 + ty * 4 + u;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int c = j0 + tx * 4 + v;
      if (r < m && c < n) {
        const float val = s * fmaf(p.coef_prev, xin[(int64_t)r * G.ld_prev + c], acc[u][v]);
        xout[(int64_t)r * G.ld_out + c] = val;
        if (xb) xb[(int64_t)r * G.ld_outb + c] = __float2bfloat16_rn(val);
      }
    }
  }
}

}  // namespace

int launch_gram_f32(const PhaseParams& p, void* stream, bool pdl) {
  if (p.total_tiles == 0) return 0;
  return launch_kernel(k_gram_f32, dim3((unsigned)p.total_tiles), dim3(kThreads), 0, stream, pdl, p);
}

int launch_gemm_f32(const PhaseParams& p, void* stream, bool pdl) {
  if (p.total_tiles == 0) return 0;
  return launch_kernel(k_gemm_f32, dim3((unsigned)p.total_tiles), dim3(kThreads), 0, stream, pdl, p);
}

}  // namespace muon
