// HBM-bound kernels of the step: momentum + sum of squares + orientation and
// cast (K1), the per-matrix norm finish, and the scaled weight update (K5).
//
// All three work on 64 x 64 tiles of the caller's rows x cols matrices, one
// 256-thread CTA per tile.  Each thread moves 4 float4 groups (16-byte,
// coalesced along a row).  Tall matrices are transposed through a padded
// shared-memory tile so that both the read of M and the write of X stay
// coalesced.
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "muon_internal.h"
#include "launch_util.cuh"

namespace muon {

namespace {

constexpr int kT = kEltTile;       // 64
constexpr int kThreads = 256;

__device__ __forceinline__ int find_mat(const EltParams& p, int64_t tile) {
  int lo = 0, hi = p.nmats - 1;
  while (lo < hi) {  // last matrix whose tile_begin <= tile
    int mid = (lo + hi + 1) >> 1;
    if (p.mats[mid].tile_begin <= tile) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ int64_t block_tile() {
  return (int64_t)blockIdx.y * gridDim.x + blockIdx.x;
}

__device__ __forceinline__ double block_sum(double v, double* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  double s = 0.0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kThreads / 32; ++i) s += red[i];  // fixed order
  }
  return s;
}

// X storage: fp32 (validation mode) or a bf16 pair hi = bf16(x),
// lo = bf16(x - hi) (tensor-core mode; hi is also the MMA operand).  x - hi
// is exact in fp32 and hi + lo carries about 17 significant bits.
__device__ __forceinline__ void store_x4(const EltMat& e, int64_t off, const float (&v)[4], int nvalid) {
  if (e.xm0) {
    if (nvalid == 4) {
      *reinterpret_cast<float4*>(e.xm0 + off) = make_float4(v[0], v[1], v[2], v[3]);
    } else {
      for (int q = 0; q < nvalid; ++q) e.xm0[off + q] = v[q];
    }
    return;
  }
  __nv_bfloat16 h[4], l[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    h[q] = __float2bfloat16_rn(v[q]);
    l[q] = __float2bfloat16_rn(v[q] - __bfloat162float(h[q]));
  }
  if (nvalid == 4) {
    *reinterpret_cast<uint2*>(e.xhi0 + off) = *reinterpret_cast<const uint2*>(h);
    *reinterpret_cast<uint2*>(e.xlo0 + off) = *reinterpret_cast<const uint2*>(l);
  } else {
    for (int q = 0; q < nvalid; ++q) {
      e.xhi0[off + q] = h[q];
      e.xlo0[off + q] = l[q];
    }
  }
}

__device__ __forceinline__ void load_x4(const EltMat& e, int64_t off, float (&v)[4], int nvalid) {
  if (e.xm_final) {
    if (nvalid == 4) {
      const float4 t = *reinterpret_cast<const float4*>(e.xm_final + off);
      v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    } else {
      for (int q = 0; q < nvalid; ++q) v[q] = e.xm_final[off + q];
    }
    return;
  }
  if (nvalid == 4) {
    const uint2 hu = *reinterpret_cast<const uint2*>(e.xhi_final + off);
    const uint2 lu = *reinterpret_cast<const uint2*>(e.xlo_final + off);
    const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&hu);
    const __nv_bfloat16* l = reinterpret_cast<const __nv_bfloat16*>(&lu);
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = __bfloat162float(h[q]) + __bfloat162float(l[q]);
  } else {
    for (int q = 0; q < nvalid; ++q)
      v[q] = __bfloat162float(e.xhi_final[off + q]) + __bfloat162float(e.xlo_final[off + q]);
  }
}

// ---------------------------------------------------------------- K1
// M <- beta*M + G (fp32 fma, in place); X0 = M (or G + beta*M with Nesterov).
// With dampening the gradient term is (1 - beta)*G, formed exactly as p + e
// (p = fl(d*G), e = fma(d, G, -p), d = 1 - beta exact in fp32), so that
// M = fma(beta, M, p) + e stays within one rounding of beta*M + (1 - beta)*G.
// written in wide orientation (fp32, or as the bf16 hi/lo pair); one fp64
// sum of squares of X0 per tile.  The normalisation 1/(||X0||+eps) is not
// applied here: it is folded into the first iteration's epilogues.
__global__ void __launch_bounds__(kThreads) k_momentum_norm(const __grid_constant__ EltParams p) {
  __shared__ float tile[kT][kT + 1];
  __shared__ double red[kThreads / 32];
  grid_dependency_wait();
  allow_dependent_launch();
  const int64_t bt = block_tile();
  if (bt >= p.total_tiles) return;
  if (bt == 0 && threadIdx.x == 0 && p.status) *p.status = 0u;
  const EltMat& e = p.mats[find_mat(p, bt)];
  const int64_t lt = bt - e.tile_begin;
  if (lt == 0 && p.apply && threadIdx.x < 8) {
    // publish this matrix's weight-update target for the last GEMM: the W
    // tensor map (128 B, eight 16-byte pieces) and its descriptor
    ApplyEntry* ae = p.apply + e.mat;
    reinterpret_cast<uint4*>(&ae->wmap)[threadIdx.x] = reinterpret_cast<const uint4*>(&e.wmap)[threadIdx.x];
    if (threadIdx.x == 0) {
      ApplyDesc a = {};
      a.W = e.W;
      a.O_out = e.O_out;
      a.ldw = e.ldw;
      a.ldo = e.ldo;
      a.lr_eff = e.lr_eff;
      a.w_bf16 = e.w_bf16;
      a.tall = e.tall;
      a.rows = e.rows;
      a.cols = e.cols;
      ae->d = a;
    }
  }
  const int r0 = (int)(lt / e.tiles_c) * kT;
  const int c0 = (int)(lt % e.tiles_c) * kT;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const float beta = p.beta;
  const float damp = 1.f - beta;   // exact for beta in [0.5, 2] (Sterbenz)
  float ss = 0.f;
  double ssd = 0.0;

#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int r = r0 + ty + 16 * k;
    const int c = c0 + tx * 4;
    float g[4] = {0.f, 0.f, 0.f, 0.f}, mm[4] = {0.f, 0.f, 0.f, 0.f}, x[4] = {0.f, 0.f, 0.f, 0.f};
    const bool row_ok = r < e.rows;
    const bool vec = row_ok && (c + 3 < e.cols);
    if (vec) {
      const float4 gv = *reinterpret_cast<const float4*>(e.G + (int64_t)r * e.ldg + c);
      const float4 mv = *reinterpret_cast<const float4*>(e.M + (int64_t)r * e.ldm + c);
      g[0] = gv.x; g[1] = gv.y; g[2] = gv.z; g[3] = gv.w;
      mm[0] = mv.x; mm[1] = mv.y; mm[2] = mv.z; mm[3] = mv.w;
    } else if (row_ok) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (c + q < e.cols) {
          g[q] = e.G[(int64_t)r * e.ldg + c + q];
          mm[q] = e.M[(int64_t)r * e.ldm + c + q];
        }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (p.dampening) {
        const float gp = damp * g[q];
        const float ge = fmaf(damp, g[q], -gp);
        mm[q] = fmaf(beta, mm[q], gp) + ge;
        x[q] = p.nesterov ? fmaf(beta, mm[q], gp) + ge : mm[q];
      } else {
        mm[q] = fmaf(beta, mm[q], g[q]);
        x[q] = p.nesterov ? fmaf(beta, mm[q], g[q]) : mm[q];
      }
      ss = fmaf(x[q], x[q], ss);
    }
    if (vec) {
      *reinterpret_cast<float4*>(e.M + (int64_t)r * e.ldm + c) = make_float4(mm[0], mm[1], mm[2], mm[3]);
    } else if (row_ok) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (c + q < e.cols) e.M[(int64_t)r * e.ldm + c + q] = mm[q];
    }
    if (!e.tall) {
      if (row_ok) store_x4(e, (int64_t)r * e.ldx + c, x, vec ? 4 : max(0, min(4, e.cols - c)));
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) tile[ty + 16 * k][tx * 4 + q] = x[q];
    }
    if ((k & 1) == 1) { ssd += (double)ss; ss = 0.f; }
  }

  if (e.tall) {
    __syncthreads();
    // X row = caller column, X column = caller row
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int xr = c0 + ty + 16 * k;   // < cols
      const int xc = r0 + tx * 4;        // < rows
      if (xr >= e.cols) continue;
      float v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) v[q] = tile[tx * 4 + q][ty + 16 * k];
      store_x4(e, (int64_t)xr * e.ldx + xc, v, max(0, min(4, e.rows - xc)));
    }
  }

  const double s = block_sum(ssd, red);
  if (threadIdx.x == 0) p.partials[e.partial_begin + lt] = s;
}

// One CTA per matrix: fixed-order sum of its tile partials, then
// scale = 1 / (sqrt(sum) + eps).
__global__ void __launch_bounds__(kThreads) k_norm_finalize(const __grid_constant__ EltParams p) {
  __shared__ double red[kThreads / 32];
  grid_dependency_wait();
  allow_dependent_launch();
  const EltMat& e = p.mats[blockIdx.x];
  double s = 0.0;
  for (int64_t i = threadIdx.x; i < e.ntiles; i += kThreads) s += p.partials[e.partial_begin + i];
  s = block_sum(s, red);
  if (threadIdx.x == 0) p.scale[e.mat] = (float)(1.0 / (sqrt(s) + (double)p.eps));
}

// ---------------------------------------------------------------- K5
// W <- W - lr_eff * O, O = X_final (wide) oriented back to rows x cols.
__global__ void __launch_bounds__(kThreads) k_apply(const __grid_constant__ EltParams p) {
  __shared__ float tile[kT][kT + 1];
  grid_dependency_wait();
  allow_dependent_launch();
  const int64_t bt = block_tile();
  if (bt >= p.total_tiles) return;
  const EltMat& e = p.mats[find_mat(p, bt)];
  const int64_t lt = bt - e.tile_begin;
  const int r0 = (int)(lt / e.tiles_c) * kT;
  const int c0 = (int)(lt % e.tiles_c) * kT;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const float os = p.apply_scale ? p.scale[e.mat] : 1.f;
  const float lr = e.lr_eff;

  if (e.tall) {
    // stage X rows c0.. (caller columns), X columns r0.. (caller rows)
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int xr = c0 + ty + 16 * k;
      const int xc = r0 + tx * 4;
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (xr < e.cols) load_x4(e, (int64_t)xr * e.ldx + xc, v, max(0, min(4, e.rows - xc)));
#pragma unroll
      for (int q = 0; q < 4; ++q) tile[tx * 4 + q][ty + 16 * k] = v[q];
    }
    __syncthreads();
  }

#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int r = r0 + ty + 16 * k;
    const int c = c0 + tx * 4;
    if (r >= e.rows) continue;
    float o[4] = {0.f, 0.f, 0.f, 0.f};
    const bool vec = c + 3 < e.cols;
    if (e.tall) {
#pragma unroll
      for (int q = 0; q < 4; ++q) o[q] = tile[ty + 16 * k][tx * 4 + q];
    } else {
      load_x4(e, (int64_t)r * e.ldx + c, o, vec ? 4 : max(0, min(4, e.cols - c)));
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) o[q] *= os;

    if (e.w_bf16) {
      __nv_bfloat16* W = reinterpret_cast<__nv_bfloat16*>(e.W) + (int64_t)r * e.ldw + c;
      if (vec) {
        uint2 pk = *reinterpret_cast<const uint2*>(W);
        __nv_bfloat162 lo = *reinterpret_cast<__nv_bfloat162*>(&pk.x);
        __nv_bfloat162 hi = *reinterpret_cast<__nv_bfloat162*>(&pk.y);
        const float w0 = fmaf(-lr, o[0], __low2float(lo));
        const float w1 = fmaf(-lr, o[1], __high2float(lo));
        const float w2 = fmaf(-lr, o[2], __low2float(hi));
        const float w3 = fmaf(-lr, o[3], __high2float(hi));
        lo = __floats2bfloat162_rn(w0, w1);
        hi = __floats2bfloat162_rn(w2, w3);
        pk.x = *reinterpret_cast<uint32_t*>(&lo);
        pk.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(W) = pk;
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (c + q < e.cols) W[q] = __float2bfloat16_rn(fmaf(-lr, o[q], __bfloat162float(W[q])));
      }
    } else {
      float* W = reinterpret_cast<float*>(e.W) + (int64_t)r * e.ldw + c;
      if (vec) {
        float4 w = *reinterpret_cast<const float4*>(W);
        w.x = fmaf(-lr, o[0], w.x);
        w.y = fmaf(-lr, o[1], w.y);
        w.z = fmaf(-lr, o[2], w.z);
        w.w = fmaf(-lr, o[3], w.w);
        *reinterpret_cast<float4*>(W) = w;
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (c + q < e.cols) W[q] = fmaf(-lr, o[q], W[q]);
      }
    }
    if (e.O_out) {
      float* Op = e.O_out + (int64_t)r * e.ldo + c;
      if (vec) {
        *reinterpret_cast<float4*>(Op) = make_float4(o[0], o[1], o[2], o[3]);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (c + q < e.cols) Op[q] = o[q];
      }
    }
  }
}

dim3 tile_grid(int64_t tiles) {
  const int64_t x = tiles < 65536 ? tiles : 65536;
  const int64_t y = (tiles + x - 1) / x;
  return dim3((unsigned)x, (unsigned)y, 1);
}

}  // namespace

int launch_momentum_norm(const EltParams& p, void* stream, bool pdl) {
  if (p.total_tiles == 0) return 0;
  return launch_kernel(k_momentum_norm, tile_grid(p.total_tiles), dim3(kThreads), 0, stream, pdl, p);
}

int launch_norm_finalize(const EltParams& p, void* stream, bool pdl) {
  if (p.nmats == 0) return 0;
  return launch_kernel(k_norm_finalize, dim3((unsigned)p.nmats), dim3(kThreads), 0, stream, pdl, p);
}

int launch_apply(const EltParams& p, void* stream, bool pdl) {
  if (p.total_tiles == 0) return 0;
  return launch_kernel(k_apply, tile_grid(p.total_tiles), dim3(kThreads), 0, stream, pdl, p);
}

}  // namespace muon
