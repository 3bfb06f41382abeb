// Tensor-core Newton-Schulz phases for sm_103a: tcgen05 UMMA with TMEM
// accumulators fed by TMA, in one persistent, warp-specialised kernel that is
// instantiated for two products:
//
//   Gram (kGram = true):  C = alpha * P P^T (+ coef_prev * prev)
//       P is X (m x n, K = n) for A = X X^T, or A (m x m, K = m) for A A^T.
//       Only output tiles that reach the upper triangle are computed
//       ("compute only the upper triangle of X X^T", jsqmd.com/news/1098463,
//       section 4.2); each element (r, c), r <= c, is written to (r, c) and
//       (c, r), so the result is exactly symmetric.
//   GEMM (kGram = false): X' = s * ((a + d) X + Bm X), Bm = b A + c A^2 (m x m)
//       and d its fp32 per-row diagonal term.  X is stored as a bf16 pair
//       (hi, lo); hi is the right operand, read MN-major (rows of X), so no
//       transposed copy of X is ever made.
//
// and for two tile shapes:
//
//   kPair = false: one CTA per SM computes 128 x 256 tiles with
//       tcgen05.mma.cta_group::1 (M = 128, N = 256).
//   kPair = true: a cluster of two CTAs on two SMs computes 256 x 256 tiles
//       with tcgen05.mma.cta_group::2 (M = 256, N = 256): each CTA loads 128
//       rows of the left operand and 128 columns of the right one, so a stage
//       is 32 KiB instead of 48 and six (Gram) or five (GEMM, whose epilogue
//       staging is larger) stages fit; the even CTA issues the MMAs, and the
//       odd CTA's copies complete on the even CTA's barriers.
//
// Tiles of all matrices of a launch form one flattened list walked with a
// static stride (deterministic; one launch per phase covers the whole ragged
// batch).  Warp 0 issues TMA loads into a shared-memory ring, warp 1 issues
// the MMAs into one of two TMEM accumulators (2 x 256 columns), and the
// epilogue warps drain the other accumulator through swizzled shared-memory
// staging with TMA loads and stores, so the epilogue of tile t overlaps the
// MMAs of tile t + 1.
//
// In the last iteration the GEMM applies the weight update instead of storing
// X': each matrix's W arrives by TMA with its X tile (tensor maps the momentum
// kernel publishes in the workspace) and leaves updated the same way.
//
// Every launch waits for its predecessor on the stream (griddepcontrol) after
// its set-up, so it can be launched as a programmatic dependent.
//
// Every wait is bounded (one second): on a time-out the kernel records the
// role in the status word, lets its copies and MMAs in flight finish, frees
// its TMEM and returns.
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <atomic>
#include <cstdio>

#include "muon_internal.h"
#include "ptx_sm100.cuh"
#include "launch_util.cuh"

// Pipeline shape of the single-CTA instantiations (ring stages, epilogue
// warps, output staging buffers of the GEMM epilogue).  Defaults are the
// measured best.
#ifndef MUON_GRAM_STAGES
#define MUON_GRAM_STAGES 4
#endif
#ifndef MUON_GRAM_EPI_WARPS
#define MUON_GRAM_EPI_WARPS 4
#endif
#ifndef MUON_GEMM_STAGES
#define MUON_GEMM_STAGES (MUON_GEMM_CHUNK == 32 ? 3 : 4)
#endif
#ifndef MUON_GEMM_EPI_WARPS
#define MUON_GEMM_EPI_WARPS 4
#endif
#ifndef MUON_GEMM_OUT_BUFS
#define MUON_GEMM_OUT_BUFS 2
#endif
// ... and of the CTA-pair instantiations
#ifndef MUON_PAIR_GRAM_STAGES
#define MUON_PAIR_GRAM_STAGES 6
#endif
#ifndef MUON_PAIR_GEMM_STAGES
#define MUON_PAIR_GEMM_STAGES (MUON_GEMM_CHUNK == 32 ? 5 : 6)
#endif
#ifndef MUON_PAIR_GRAM_EPI_WARPS
#define MUON_PAIR_GRAM_EPI_WARPS 4
#endif
#ifndef MUON_PAIR_GEMM_EPI_WARPS
#define MUON_PAIR_GEMM_EPI_WARPS 4
#endif
#ifndef MUON_PAIR_GEMM_OUT_BUFS
#define MUON_PAIR_GEMM_OUT_BUFS 2
#endif

namespace muon {

namespace {

constexpr int TC = kTcM;                    // 128 rows per CTA (UMMA M per CTA)
constexpr int TN = kTcN;                    // 256 columns per tile (UMMA N)
constexpr int TK = kTcK;                    // 64 bf16 = 128 bytes = one swizzle row
constexpr int UK = 16;                      // K per UMMA instruction
constexpr int A_BYTES = TC * TK * 2;        // 16 KiB: 128 rows of the left operand
constexpr int TMEM_COLS = 2 * TN;           // two fp32 accumulators
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr int kSmemLimit = 232448;          // 227 KiB per CTA

template <bool kGram, bool kPair>
struct Cfg {
  static constexpr int kStages = kPair ? (kGram ? MUON_PAIR_GRAM_STAGES : MUON_PAIR_GEMM_STAGES)
                                       : (kGram ? MUON_GRAM_STAGES : MUON_GEMM_STAGES);
  static constexpr int kEpiWarps = kPair ? (kGram ? MUON_PAIR_GRAM_EPI_WARPS : MUON_PAIR_GEMM_EPI_WARPS)
                                         : (kGram ? MUON_GRAM_EPI_WARPS : MUON_GEMM_EPI_WARPS);
  static constexpr int kOutBufs = kGram ? 2 : (kPair ? MUON_PAIR_GEMM_OUT_BUFS : MUON_GEMM_OUT_BUFS);
  static constexpr int kSlices = kEpiWarps / 4;   // epilogue warps per TMEM lane quarter
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr int kTileM = kPair ? 2 * TC : TC;        // rows of an output tile
  static constexpr int kBCols = kPair ? TN / 2 : TN;        // right-operand rows/columns per CTA
  static constexpr int kBBytes = kBCols * TK * 2;
  static constexpr int kStageBytes = A_BYTES + kBBytes;
  // Gram: row-major and transposed 32x32 bf16 output blocks, double-buffered
  // (Gram 1), or single-buffered beside two prefetched blocks of the previous
  // A (Gram 2): 8 KiB.
  // GEMM: two input and two output buffers of (hi, lo) X boxes, 32 rows x
  // kGemmChunk bf16 each (8 or 16 KiB).
  static constexpr int kEpiWarpBytes = kGram ? 8192 : 8 * 32 * kGemmChunk * 2;
  static constexpr int kBarBytes = 512;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kEpiWarps * kEpiWarpBytes + kBarBytes;
  static_assert(kEpiWarps % 4 == 0, "epilogue warps come in groups of four (one per TMEM lane quarter)");
  static_assert(kOutBufs == 1 || kOutBufs == 2, "one or two output staging buffers");
  static_assert(kSmemBytes <= kSmemLimit, "shared memory over the per-CTA limit");
};

struct Tile { int g, mat, bi, bj; };

// Optional wait-time counters (build with -DMUON_TC_PROFILE): cycles summed
// over CTAs into 64-bit slots after the status word, read from the workspace.
//   [1] MMA waiting for a full stage   [2] MMA waiting for a free accumulator
//   [3] TMA waiting for an empty stage [4] epilogue waiting for an accumulator
//   [5] CTA lifetime; slots 6-10 the same for the GEMM, 11-15 for the Gram
//   launches that combine with the previous A (Gram 2)
#ifdef MUON_TC_PROFILE
#define TC_PROF_T0(v) const long long v = clock64()
#define TC_PROF_ADD(slot, v)                                                                          \
  atomicAdd(reinterpret_cast<unsigned long long*>(p.status) + (slot) + (kGram ? (p.g[0].prev ? 10 : 0) : 5), \
            (unsigned long long)(clock64() - (v)))
#else
#define TC_PROF_T0(v)
#define TC_PROF_ADD(slot, v)
#endif

// Optional per-tile trace (build with -DMUON_TC_TRACE): clock64 stamps of the
// leader CTA of each pair (or each CTA), per launch kind (0 Gram X X^T,
// 1 Gram with the previous A, 2 GEMM, 3 GEMM that applies the update; the
// last launch of a kind wins):
//   [0] MMA issuer: accumulator granted     [1] MMA issuer: last MMA of the tile issued
//   [2] epilogue warp 0: accumulator full   [3] epilogue warp 0: tile done
// g_tc_life: %globaltimer (ns) at [0] kernel entry, [1] after the grid
// dependency wait (set-up done, the previous kernel complete), [2] CTA end;
// [3..5] clock64 at the same points.
// g_tc_epi: cycles the tracing epilogue warp (lane 0 of warp quarter 0 of the
// leader) spends in [0] X-prefetch waits, [1] waits for its previous TMA
// store to release the staging buffer, [2] TMEM load waits (GEMM).
// g_tc_mma: cycles the MMA issuer waits for a full stage: [0] on the tile's
// first k-block, [1] on its first four, [2] on all.
// Read with muon_tc_trace_read.
#ifdef MUON_TC_TRACE
constexpr int kTraceCtas = 160, kTraceTiles = 96;
__device__ long long g_tc_trace[4][kTraceCtas][kTraceTiles][4];
__device__ long long g_tc_life[4][kTraceCtas][6];
__device__ long long g_tc_epi[4][kTraceCtas][4];
__device__ long long g_tc_mma[4][kTraceCtas][4];
#define TC_KIND (kGram ? (p.g[0].prev ? 1 : 0) : (p.apply ? 3 : 2))
#define TC_TRACE(k, slot)                                                                          \
  do {                                                                                             \
    if (blockIdx.x < kTraceCtas && (k) < kTraceTiles) g_tc_trace[TC_KIND][blockIdx.x][(k)][(slot)] = clock64(); \
  } while (0)
#define TC_LIFE(slot)                                                              \
  do {                                                                             \
    if (blockIdx.x < kTraceCtas) {                                                 \
      g_tc_life[TC_KIND][blockIdx.x][(slot)] = (long long)ptx::globaltimer();      \
      g_tc_life[TC_KIND][blockIdx.x][(slot) + 3] = clock64();                      \
    }                                                                              \
  } while (0)
#define TC_EPI_T0(v) const long long v = clock64()
#define TC_EPI_ADD(ec, kind, slot, v)                                                               \
  do {                                                                                              \
    if ((ec).quarter == 0 && (ec).slice == 0 && (ec).lane == 0 && (blockIdx.x & 1) == 0 &&          \
        blockIdx.x < kTraceCtas)                                                                    \
      g_tc_epi[(kind)][blockIdx.x][(slot)] += clock64() - (v);                                      \
  } while (0)
#define TC_MMA_ADD(kb, v)                 \
  do {                                    \
    const long long d_ = clock64() - (v); \
    if ((kb) == 0) tc_mw[0] += d_;        \
    if ((kb) < 4) tc_mw[1] += d_;         \
    tc_mw[2] += d_;                       \
  } while (0)
#else
#define TC_TRACE(k, slot)
#define TC_LIFE(slot)
#define TC_EPI_T0(v)
#define TC_EPI_ADD(ec, kind, slot, v)
#define TC_MMA_ADD(kb, v)
#endif

// Flattened tile t -> (group, matrix, row block, column block).  Gram tiles
// are the upper ones: for 128 x 256 tiles, column block bj (256 wide) needs
// row blocks bi < 2 bj + 2 (rows start before the block's last column); for
// 256 x 256 tiles, bi <= bj.
template <bool kPair>
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
    int bj = 0;
    while (true) {
      const int cnt = kPair ? bj + 1 : min(2 * bj + 2, G.ni);
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

// A CTA pair's Gram tile on the diagonal (bi == bj): CTA r's left operand
// (rows 256 bi + 128 r) and its half of the right operand (rows
// 256 bj + 128 r) are the same rows of the same matrix.
template <bool kGram, bool kPair>
__device__ __forceinline__ bool gram_diag_tile(const Tile& tl) {
  return kGram && kPair && tl.bi == tl.bj;
}

__device__ __forceinline__ bool wait_drain(uint64_t* bar, uint32_t parity) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

template <bool kPair>
__device__ __forceinline__ bool wait_role(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t* status,
                                          uint32_t code) {
  if (kPair) return ptx::mbar_wait_bounded_cluster(bar, parity, abort, status, code, kWaitLimitNs);
  return ptx::mbar_wait_bounded(bar, parity, abort, status, code, kWaitLimitNs);
}

struct PairInfo {
  int rank;      // 0 or 1 within the pair (0 when single-CTA)
  int unit;      // this CTA's (or pair's) index in the persistent grid
  int nunits;    // number of CTAs (or pairs)
};

template <bool kGram, bool kPair>
__device__ __forceinline__ void run_producer(const PhaseParams& p, const PairInfo& pi, uint8_t* smem,
                                             uint64_t* full, uint64_t* empty, volatile int* abort) {
  using C = Cfg<kGram, kPair>;
  constexpr int S = C::kStages;
  int stage = 0;
  uint32_t phase = 0;
  uint32_t outstanding = 0, fill_parity = 0;
  bool ok = true;
  for (int t = pi.unit; ok && t < p.total_tiles; t += pi.nunits) {
    const Tile tl = decode_tile<kPair>(p, t, kGram);
    const PhaseGroup& G = p.g[tl.g];
    const int nk = (G.K + TK - 1) / TK;
    const CUtensorMap* ma = &p.map_a[tl.g];
    const CUtensorMap* mb = &p.map_b[tl.g];
    const int arow = tl.bi * C::kTileM + TC * pi.rank;     // this CTA's left-operand rows
    const int bcol = tl.bj * TN + C::kBCols * pi.rank;     // this CTA's right-operand rows/columns
    // a pair's Gram tile on the diagonal: each CTA's right-operand half is
    // its left operand (the same rows), loaded once
    const bool same = gram_diag_tile<kGram, kPair>(tl);
    const uint32_t stage_bytes = same ? (uint32_t)A_BYTES : (uint32_t)C::kStageBytes;
    for (int kb = 0; kb < nk; ++kb) {
      TC_PROF_T0(t_e);
      if (!wait_role<false>(&empty[stage], phase ^ 1u, abort, p.status, kStatusTimeoutProducer)) {
        ok = false;
        break;
      }
      TC_PROF_ADD(3, t_e);
      outstanding &= ~(1u << stage);
      uint8_t* sa = smem + stage * C::kStageBytes;
      uint8_t* sb = sa + A_BYTES;
      const int k0 = kb * TK;
      if (p.withhold_loads) {
        // failure-path test: nothing arrives on the stage barriers, so the
        // MMA's bounded wait runs out and the kernel reports a time-out
      } else if (!kPair || pi.rank == 0) {
        // the even CTA's barrier counts the bytes of both CTAs of a pair
        ptx::mbar_arrive_expect_tx(&full[stage], (kPair ? 2u : 1u) * stage_bytes);
        if (kGram) {
          ptx::tma_load_4d(sa, ma, k0, arow, tl.mat, G.buf_in, &full[stage]);
          if (!same) {
#pragma unroll
            for (int q = 0; q < C::kBCols / TC; ++q)
              ptx::tma_load_4d(sb + q * A_BYTES, ma, k0, bcol + TC * q, tl.mat, G.buf_in, &full[stage]);
          }
        } else {
          ptx::tma_load_4d(sa, ma, k0, arow, tl.mat, 0, &full[stage]);
#pragma unroll
          for (int q = 0; q < C::kBCols / 64; ++q)
            ptx::tma_load_4d(sb + q * (64 * TK * 2), mb, bcol + 64 * q, k0, tl.mat, G.buf_in, &full[stage]);
        }
      } else {
        // odd CTA: its copies land in its own shared memory and complete on
        // the even CTA's barrier of the same stage
        const uint32_t bar = ptx::mapa(ptx::smem_u32(&full[stage]), 0);
        if (kGram) {
          ptx::tma_load_4d_pair(sa, ma, k0, arow, tl.mat, G.buf_in, bar);
          if (!same) ptx::tma_load_4d_pair(sb, ma, k0, bcol, tl.mat, G.buf_in, bar);
        } else {
          ptx::tma_load_4d_pair(sa, ma, k0, arow, tl.mat, 0, bar);
#pragma unroll
          for (int q = 0; q < C::kBCols / 64; ++q)
            ptx::tma_load_4d_pair(sb + q * (64 * TK * 2), mb, bcol + 64 * q, k0, tl.mat, G.buf_in, bar);
        }
      }
      if (!p.withhold_loads) outstanding |= 1u << stage;
      fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
      if (++stage == S) { stage = 0; phase ^= 1u; }
    }
  }
  if (!ok && (!kPair || pi.rank == 0)) {
    // let every copy issued (by this CTA, and by the odd CTA of a pair,
    // whose copies complete on these barriers) land before the CTAs exit
    for (int s = 0; s < S; ++s)
      if ((outstanding >> s) & 1u)
        if (!wait_drain(&full[s], (fill_parity >> s) & 1u) && p.status) atomicOr(p.status, kStatusTimeoutDrain);
  }
}

template <bool kGram, bool kPair>
__device__ __forceinline__ void run_mma(const PhaseParams& p, const PairInfo& pi, uint8_t* smem, uint64_t* full,
                                        uint64_t* empty, uint64_t* tfull, uint64_t* tempty, uint64_t* drain,
                                        uint32_t tmem_base, volatile int* abort) {
  using C = Cfg<kGram, kPair>;
  constexpr int S = C::kStages;
  constexpr uint32_t idesc = ptx::idesc_bf16_f32(C::kTileM, TN, !kGram);
  int stage = 0;
  uint32_t phase = 0;
  int acc = 0;
  uint32_t acc_phase = 0;
  bool ok = true, issued = false;
#ifdef MUON_TC_TRACE
  long long tc_mw[3] = {0, 0, 0};
#endif
  int lt = 0;   // local tile count (trace)
  (void)lt;
  for (int t = pi.unit; ok && t < p.total_tiles; t += pi.nunits, ++lt) {
    const Tile tl = decode_tile<kPair>(p, t, kGram);
    const int nk = (p.g[tl.g].K + TK - 1) / TK;
    const bool same = gram_diag_tile<kGram, kPair>(tl);   // right operand = the left one
    TC_PROF_T0(t_a);
    if (!wait_role<kPair>(&tempty[acc], acc_phase ^ 1u, abort, p.status, kStatusTimeoutMma)) {
      ok = false;
      break;
    }
    TC_PROF_ADD(2, t_a);
    TC_TRACE(lt, 0);
    ptx::tc_fence_after();
    const uint32_t d = tmem_base + (uint32_t)(acc * TN);
    for (int kb = 0; kb < nk; ++kb) {
      TC_PROF_T0(t_f);
      TC_EPI_T0(t_fw);
      if (!wait_role<false>(&full[stage], phase, abort, p.status, kStatusTimeoutMma)) {
        ok = false;
        break;
      }
      TC_PROF_ADD(1, t_f);
      TC_MMA_ADD(kb, t_fw);
      ptx::tc_fence_after();
      const uint32_t sa = ptx::smem_u32(smem + stage * C::kStageBytes);
      const uint32_t sb = sa + A_BYTES;
#pragma unroll
      for (int kk = 0; kk < TK / UK; ++kk) {
        // K-major, 128B swizzle: rows 128 B apart, 8-row groups 1024 B apart;
        // the K offset inside the swizzle row is a plain start-address offset.
        const uint64_t ad = ptx::smem_desc(sa + kk * UK * 2, 16, 1024);
        uint64_t bd;
        if (kGram) {
          bd = ptx::smem_desc((same ? sa : sb) + kk * UK * 2, 16, 1024);
        } else {
          // MN-major, 128B swizzle: 64-element MN blocks 8 KiB apart (LBO),
          // 8-row K groups 1024 B apart (SBO); UK rows of K = 2 KiB.
          bd = ptx::smem_desc(sb + kk * UK * 128, 64 * TK * 2, 1024);
        }
        if (kPair) ptx::umma_f16_pair(d, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
        else ptx::umma_f16(d, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
      }
      if (kPair) ptx::umma_commit_pair_mc(&empty[stage], 0x3);   // frees the stage in both CTAs
      else ptx::umma_commit(&empty[stage]);
      issued = true;
      if (++stage == S) { stage = 0; phase ^= 1u; }
    }
    if (!ok) break;
    if (kPair) ptx::umma_commit_pair_mc(&tfull[acc], 0x3);
    else ptx::umma_commit(&tfull[acc]);
    TC_TRACE(lt, 1);
    acc ^= 1;
    if (acc == 0) acc_phase ^= 1u;
  }
#ifdef MUON_TC_TRACE
  if (blockIdx.x < kTraceCtas)
    for (int q = 0; q < 3; ++q) g_tc_mma[TC_KIND][blockIdx.x][q] = tc_mw[q];
#endif
  if (!ok && issued) {
    if (kPair) ptx::umma_commit_pair_mc(drain, 0x1);
    else ptx::umma_commit(drain);
    if (!wait_drain(drain, 0) && p.status) atomicOr(p.status, kStatusTimeoutDrain);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

struct EpiCtx {
  uint8_t* buf;        // this warp's staging (1024-B aligned sub-buffers)
  uint64_t* xfull;     // this warp's two X-prefetch barriers (GEMM)
  uint32_t xphase;     // parity bits of xfull[0..1]
  int obuf;            // next output staging buffer
  int quarter;         // TMEM lane quarter (warp index mod 4)
  int slice;           // which of the column slices this warp drains
  int nslices;
  int out_bufs;        // GEMM output staging buffers (1 or 2)
  int lane;
  bool skip_w;         // last GEMM: an earlier launch of the step timed out, leave W as it is
};

// ---------------------------------------------------------------- Gram epilogue

__device__ __forceinline__ void unpack_bf16x8(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&w[h]);
    f[2 * h] = __low2float(b2);
    f[2 * h + 1] = __high2float(b2);
  }
}


// fp32 diagonal residuals of the previous A that one warp needs for a Gram-2
// tile, loaded once per tile before the accumulator wait: lane l holds
// R[col0 + 8 l .. col0 + 8 l + 7] (zero past m), and rr = R[row].
struct GramDiag {
  float rcv[8];
  float rr;
};

__device__ __forceinline__ void gram_diag_load(const PhaseGroup& G, const Tile& tl, int lane, int row, int col0,
                                               GramDiag& gd) {
#pragma unroll
  for (int q = 0; q < 8; ++q) gd.rcv[q] = 0.f;
  gd.rr = 0.f;
  if (!G.prev || !G.diag_in) return;
  const float* rin = G.diag_in + (int64_t)tl.mat * G.diag_stride;
  const int c = col0 + 8 * lane;
  if (c + 8 <= G.m) {
    const float4 q0 = *reinterpret_cast<const float4*>(rin + c);
    const float4 q1 = *reinterpret_cast<const float4*>(rin + c + 4);
    gd.rcv[0] = q0.x; gd.rcv[1] = q0.y; gd.rcv[2] = q0.z; gd.rcv[3] = q0.w;
    gd.rcv[4] = q1.x; gd.rcv[5] = q1.y; gd.rcv[6] = q1.z; gd.rcv[7] = q1.w;
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (c + q < G.m) gd.rcv[q] = rin[c + q];
  }
  if (row < G.m) gd.rr = rin[row];
}

// Gram values of one 32-column chunk for one row (fp32, before rounding).
//   Gram 1 (no prev):  A = alpha * acc, alpha = s^2 in the first iteration.
//   Gram 2 (prev = A): B = b * A + c * A^2 with A = A~ + R, A~ the stored bf16
//     A (pa: this row's 32 values, from the prefetched block) and R the fp32
//     residual of its diagonal (gd):
//     A^2 = acc + A~ o (R_r + R_c) + R_r^2 on the diagonal, acc = A~ A~.
// All lanes of the warp call this (the column residuals move by shuffles).
__device__ __forceinline__ void gram_values(const PhaseParams& p, const PhaseGroup& G, const Tile& tl, int row,
                                            int c0, int col0, const uint32_t (&v)[32], const float (&pa)[32],
                                            const GramDiag& gd, float (&f)[32]) {
  if (G.prev) {
    const int src = (c0 - col0) >> 3;   // lane holding R[c0 .. c0 + 7]
    const float rr = gd.rr;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float rc = __shfl_sync(0xffffffffu, gd.rcv[j & 7], src + (j >> 3));
      float acc = fmaf(pa[j], rr + rc, __uint_as_float(v[j]));
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
}

// The diagonal value of a diagonal 32 x 32 block (or its bf16 residual) goes
// to diag_out; with diag_exact the block keeps a zero in its place.
__device__ __forceinline__ void gram_diag_out(const PhaseParams& p, const PhaseGroup& G, const Tile& tl, int row,
                                              int c0, float (&f)[32]) {
  if (!G.diag_out || row >= G.m) return;
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

// Store one 32 x 32 block of a Gram tile on or above the diagonal with TMA
// (rows and columns past m are clipped by the tensor map).  Staging per warp
// (8 KiB): Gram 1 double-buffers a (block, transpose) pair at 0 / 2048 and
// 4096 / 6144; Gram 2 has one pair at 0 / 2048 and its prefetched blocks of
// the previous A at 4096 and 6144.
//   Above the diagonal: the block and its transpose, two stores.
//   On the diagonal (c0 == r0): each row is written whole, then its part below
//   the diagonal is overwritten with the mirror of the part above, so the
//   stored block is exactly symmetric; one store.
__device__ __forceinline__ void gram_store_block(const PhaseParams& p, const Tile& tl, EpiCtx& ec, int r0, int c0,
                                                 const float (&f)[32], bool single, bool diag) {
  const int o = single ? 0 : ec.obuf;
  uint8_t* ro = ec.buf + o * 4096;
  uint8_t* tr = diag ? ro : ro + 2048;
  const int lane = ec.lane;
  if (lane == 0) {   // the stores that last read this buffer are done with it
    TC_EPI_T0(t_w);
    if (single) ptx::bulk_wait_read_all();
    else ptx::bulk_wait_read_1();
    TC_EPI_ADD(ec, single ? 1 : 0, 1, t_w);
  }
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 u;
    u.x = pack_bf16x2(f[8 * i + 0], f[8 * i + 1]);
    u.y = pack_bf16x2(f[8 * i + 2], f[8 * i + 3]);
    u.z = pack_bf16x2(f[8 * i + 4], f[8 * i + 5]);
    u.w = pack_bf16x2(f[8 * i + 6], f[8 * i + 7]);
    *reinterpret_cast<uint4*>(ro + ptx::sw64_off(lane, i)) = u;
  }
  if (diag) __syncwarp();   // the mirror below overwrites other lanes' rows
  // transposed block: row j (= column c0 + j), column lane (= row r0 + lane);
  // on the diagonal only its part below the diagonal (j > lane)
#pragma unroll
  for (int j = 0; j < 32; ++j)
    if (!diag || j > lane)
      *reinterpret_cast<__nv_bfloat16*>(tr + ptx::sw64_off(j, lane >> 3) + (lane & 7) * 2) = __float2bfloat16_rn(f[j]);
  ptx::fence_async_smem();
  __syncwarp();
  if (lane == 0) {
    const CUtensorMap* mc = &p.map_c[tl.g];
    ptx::tma_store_4d(mc, ro, c0, r0, tl.mat, 0);
    if (!diag) ptx::tma_store_4d(mc, tr, r0, c0, tl.mat, 0);
    ptx::bulk_commit();
  }
  if (!single) ec.obuf ^= 1;
}

// Chunks of a Gram tile this warp handles: ch = first + k * nslices for
// k < count, skipping chunks wholly below the diagonal (c0 < r0; r0 - col0 is
// a multiple of 32) and past the last column.
struct GramChunks { int first, count; };
__device__ __forceinline__ GramChunks gram_chunks(const PhaseGroup& G, const EpiCtx& ec, int r0, int col0) {
  const int lo = r0 > col0 ? (r0 - col0) / 32 : 0;
  const int hi = min(TN / 32, (G.m - col0 + 31) / 32);
  int first = ec.slice;
  if (first < lo) first += (lo - first + ec.nslices - 1) / ec.nslices * ec.nslices;
  const int count = first < hi ? (hi - first + ec.nslices - 1) / ec.nslices : 0;
  return {first, count};
}

// Gram 2: TMA prefetch of the previous A's 32 x 32 block at (c0, r0) into
// buffer b (completes on xfull[b]).
__device__ __forceinline__ void gram_prefetch_prev(const PhaseParams& p, const Tile& tl, EpiCtx& ec, int b, int c0,
                                                   int r0) {
  if (ec.lane == 0) {
    ptx::mbar_arrive_expect_tx(&ec.xfull[b], 2048u);
    ptx::tma_load_4d(ec.buf + 4096 + 2048 * b, &p.map_d[tl.g], c0, r0, tl.mat, 0, &ec.xfull[b]);
  }
}

// One chunk of a Gram tile.  Returns false on a time-out.
__device__ __forceinline__ bool gram_chunk(const PhaseParams& p, const PhaseGroup& G, const Tile& tl, EpiCtx& ec,
                                           const GramChunks& gc, int k, int r0, int col0, const uint32_t (&v)[32],
                                           const GramDiag& gd, volatile int* abort) {
  const int lane = ec.lane;
  const int row = r0 + lane;
  const int c0 = col0 + 32 * (gc.first + k * ec.nslices);
  float pa[32];
  if (G.prev) {
    const int b = k & 1;
    TC_EPI_T0(t_x);
    if (!ptx::mbar_wait_bounded(&ec.xfull[b], (ec.xphase >> b) & 1u, abort, p.status, kStatusTimeoutEpilogue,
                                kWaitLimitNs))
      return false;
    TC_EPI_ADD(ec, G.prev ? 1 : 0, 0, t_x);
    ec.xphase ^= 1u << b;
    const uint8_t* pb = ec.buf + 4096 + 2048 * b;
#pragma unroll
    for (int i = 0; i < 4; ++i) unpack_bf16x8(*reinterpret_cast<const uint4*>(pb + ptx::sw64_off(lane, i)), pa + 8 * i);
    __syncwarp();   // every lane has read buffer b: refill it
    if (k + 2 < gc.count) gram_prefetch_prev(p, tl, ec, b, c0 + 64 * ec.nslices, r0);
  }
  float f[32];
  gram_values(p, G, tl, row, c0, col0, v, pa, gd, f);
  const bool diag = c0 == r0;
  if (diag) gram_diag_out(p, G, tl, row, c0, f);
  gram_store_block(p, tl, ec, r0, c0, f, G.prev != nullptr, diag);
  return true;
}

// The Gram tile's epilogue for this warp; the TMEM load of chunk k + 1 is in
// flight while chunk k is processed.
__device__ __forceinline__ bool gram_tile_epilogue(const PhaseParams& p, const PhaseGroup& G, const Tile& tl,
                                                   EpiCtx& ec, uint32_t tbase, int r0, int col0,
                                                   const GramChunks& gc, const GramDiag& gd, volatile int* abort) {
  if (gc.count <= 0) return true;
  uint32_t va[32], vb[32];
  ptx::tmem_ld_32x32b_x32(tbase + (uint32_t)(32 * gc.first), va);
  {
    TC_EPI_T0(t_m);
    ptx::tmem_ld_wait_regs(va);
    TC_EPI_ADD(ec, G.prev ? 1 : 0, 2, t_m);
  }
#pragma unroll 1
  for (int k = 0; k < gc.count; k += 2) {
    const bool has1 = k + 1 < gc.count;
    if (has1) ptx::tmem_ld_32x32b_x32(tbase + (uint32_t)(32 * (gc.first + (k + 1) * ec.nslices)), vb);
    if (!gram_chunk(p, G, tl, ec, gc, k, r0, col0, va, gd, abort)) {
      if (has1) ptx::tmem_ld_wait_regs(vb);
      return false;
    }
    if (has1) {
      ptx::tmem_ld_wait_regs(vb);
      const bool has2 = k + 2 < gc.count;
      if (has2) ptx::tmem_ld_32x32b_x32(tbase + (uint32_t)(32 * (gc.first + (k + 2) * ec.nslices)), va);
      const bool okb = gram_chunk(p, G, tl, ec, gc, k + 1, r0, col0, vb, gd, abort);
      if (has2) ptx::tmem_ld_wait_regs(va);
      if (!okb) return false;
    }
  }
  return true;
}

// ---------------------------------------------------------------- GEMM epilogue

// X is kept as a bf16 pair hi = bf16(x), lo = bf16(x - hi) (about 17
// significant bits); hi is also the MMA operand of the next iteration.
// A GEMM epilogue chunk covers 32 rows x kGC columns; each of its X boxes
// (hi or lo) is 32 rows x kGC bf16 with the swizzle of that row width.
// Per-warp staging (kXBox = one box): input buffer b holds hi at 2 kXBox b
// and lo at 2 kXBox b + kXBox; output buffer o holds hi' / lo' at
// 4 kXBox + 2 kXBox o (+ kXBox).  In the last iteration output slot b holds
// the W tile loaded with input buffer b (up to 32 x kGC fp32 = 2 kXBox).
constexpr int kGC = kGemmChunk;
constexpr int kXBox = 32 * kGC * 2;
constexpr int kXRowBytes = kGC * 2;

__device__ __forceinline__ uint32_t sw_off(int row, int chunk, int row_bytes) {
  return row_bytes == 32 ? ptx::sw32_off(row, chunk) : row_bytes == 64 ? ptx::sw64_off(row, chunk)
                                                                       : ptx::sw128_off(row, chunk);
}

__device__ __forceinline__ uint8_t* gemm_in(const EpiCtx& ec, int b) { return ec.buf + 2 * kXBox * b; }
__device__ __forceinline__ uint8_t* gemm_out(const EpiCtx& ec, int o) { return ec.buf + 4 * kXBox + 2 * kXBox * o; }

// chunk k of this warp covers columns kGC * (slice + k * nslices) of the tile
__device__ __forceinline__ int gemm_chunk_col(const EpiCtx& ec, int k) { return ec.slice + k * ec.nslices; }

__device__ __forceinline__ void gemm_prefetch(const PhaseParams& p, const PhaseGroup& G, const Tile& tl,
                                              EpiCtx& ec, int b, int c0, int r0) {
  if (ec.lane == 0) {
    const ApplyEntry* ae = p.apply ? &p.apply[G.first + tl.mat] : nullptr;
    const uint32_t wbytes = ae ? (ae->d.w_bf16 ? 32u * kGC * 2u : 32u * kGC * 4u) : 0u;
    ptx::mbar_arrive_expect_tx(&ec.xfull[b], (p.x_lo_in ? 2 : 1) * kXBox + wbytes);
    ptx::tma_load_4d(gemm_in(ec, b), &p.map_c[tl.g], c0, r0, tl.mat, G.buf_in, &ec.xfull[b]);
    if (p.x_lo_in)
      ptx::tma_load_4d(gemm_in(ec, b) + kXBox, &p.map_d[tl.g], c0, r0, tl.mat, G.buf_in, &ec.xfull[b]);
    if (ae) {
      if (ae->d.tall) ptx::tma_load_2d(gemm_out(ec, b), &ae->wmap, r0, c0, &ec.xfull[b]);
      else ptx::tma_load_2d(gemm_out(ec, b), &ae->wmap, c0, r0, &ec.xfull[b]);
    }
  }
}

// W <- W - lr_eff * O on the W tile in slot `ws`, O being this lane's row of
// X' (kGC values).  Wide: 32 rows x kGC columns of W, lane = row.  Tall: W is
// X transposed, so the tile is kGC rows x 32 columns and lane = column.
__device__ __forceinline__ void gemm_apply_slot(const ApplyDesc& d, uint8_t* ws, int lane, const float (&f)[kGC]) {
  const float lr = d.lr_eff;
  if (!d.tall) {
    if (d.w_bf16) {   // rows of kGC bf16
#pragma unroll
      for (int i = 0; i < kGC / 8; ++i) {
        uint4* q = reinterpret_cast<uint4*>(ws + sw_off(lane, i, kGC * 2));
        uint4 u = *q;
        float wv[8];
        unpack_bf16x8(u, wv);
        u.x = pack_bf16x2(fmaf(-lr, f[8 * i + 0], wv[0]), fmaf(-lr, f[8 * i + 1], wv[1]));
        u.y = pack_bf16x2(fmaf(-lr, f[8 * i + 2], wv[2]), fmaf(-lr, f[8 * i + 3], wv[3]));
        u.z = pack_bf16x2(fmaf(-lr, f[8 * i + 4], wv[4]), fmaf(-lr, f[8 * i + 5], wv[5]));
        u.w = pack_bf16x2(fmaf(-lr, f[8 * i + 6], wv[6]), fmaf(-lr, f[8 * i + 7], wv[7]));
        *q = u;
      }
    } else {          // rows of kGC fp32
#pragma unroll
      for (int i = 0; i < kGC / 4; ++i) {
        float4* q = reinterpret_cast<float4*>(ws + sw_off(lane, i, kGC * 4));
        float4 v = *q;
        v.x = fmaf(-lr, f[4 * i + 0], v.x);
        v.y = fmaf(-lr, f[4 * i + 1], v.y);
        v.z = fmaf(-lr, f[4 * i + 2], v.z);
        v.w = fmaf(-lr, f[4 * i + 3], v.w);
        *q = v;
      }
    }
  } else {
    if (d.w_bf16) {   // kGC rows of 32 bf16 (64-byte rows): column `lane` of row j
#pragma unroll
      for (int j = 0; j < kGC; ++j) {
        __nv_bfloat16* q = reinterpret_cast<__nv_bfloat16*>(ws + ptx::sw64_off(j, lane >> 3) + (lane & 7) * 2);
        *q = __float2bfloat16_rn(fmaf(-lr, f[j], __bfloat162float(*q)));
      }
    } else {          // kGC rows of 32 fp32 (128-byte rows)
#pragma unroll
      for (int j = 0; j < kGC; ++j) {
        float* q = reinterpret_cast<float*>(ws + ptx::sw128_off(j, lane >> 2) + (lane & 3) * 4);
        *q = fmaf(-lr, f[j], *q);
      }
    }
  }
}

// Optional fp32 export of O (rows x cols, caller layout) with direct stores.
__device__ __forceinline__ void gemm_export_o(const ApplyDesc& d, int row, int c0, int m, int n,
                                              const float (&f)[kGC]) {
  if (!d.O_out || row >= m) return;
  if (!d.tall) {
    float* o = d.O_out + (int64_t)row * d.ldo + c0;
    if (c0 + kGC <= n) {
#pragma unroll
      for (int i = 0; i < kGC / 4; ++i)
        *reinterpret_cast<float4*>(o + 4 * i) = make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
    } else {
#pragma unroll
      for (int j = 0; j < kGC; ++j)
        if (c0 + j < n) o[j] = f[j];
    }
  } else {
#pragma unroll
    for (int j = 0; j < kGC; ++j)
      if (c0 + j < n) d.O_out[(int64_t)(c0 + j) * d.ldo + row] = f[j];
  }
}

// One chunk: X' = s * ((a + d) * X + acc), written as the bf16 hi/lo pair
// through the staging buffers (or, in the last iteration, applied to W).
// Returns false on a time-out.
__device__ __forceinline__ bool gemm_chunk(const PhaseParams& p, const PhaseGroup& G, const Tile& tl, EpiCtx& ec,
                                           int col0, int k, int cnt, int r0, float s, float ar,
                                           const uint32_t (&v)[kGC], volatile int* abort) {
  const int lane = ec.lane;
  const int b = k & 1;
  const int c0 = col0 + kGC * gemm_chunk_col(ec, k);
  TC_EPI_T0(t_x);
  if (!ptx::mbar_wait_bounded(&ec.xfull[b], (ec.xphase >> b) & 1u, abort, p.status, kStatusTimeoutEpilogue,
                              kWaitLimitNs))
    return false;
  TC_EPI_ADD(ec, p.apply ? 3 : 2, 0, t_x);
  ec.xphase ^= 1u << b;
  const uint8_t* xh = gemm_in(ec, b);
  const uint8_t* xl = xh + kXBox;
  float f[kGC];
  if (p.x_lo_in) {
#pragma unroll
    for (int i = 0; i < kGC / 8; ++i) {
      float hv[8], lv[8];
      unpack_bf16x8(*reinterpret_cast<const uint4*>(xh + sw_off(lane, i, kXRowBytes)), hv);
      unpack_bf16x8(*reinterpret_cast<const uint4*>(xl + sw_off(lane, i, kXRowBytes)), lv);
#pragma unroll
      for (int j = 0; j < 8; ++j) f[8 * i + j] = s * fmaf(ar, hv[j] + lv[j], __uint_as_float(v[8 * i + j]));
    }
  } else {   // X stored as bf16 alone (the last stored iterates)
#pragma unroll
    for (int i = 0; i < kGC / 8; ++i) {
      float hv[8];
      unpack_bf16x8(*reinterpret_cast<const uint4*>(xh + sw_off(lane, i, kXRowBytes)), hv);
#pragma unroll
      for (int j = 0; j < 8; ++j) f[8 * i + j] = s * fmaf(ar, hv[j], __uint_as_float(v[8 * i + j]));
    }
  }
  if (p.apply) {
    // last iteration: update the W tile that came with this X tile and store
    // it; the slot is refilled (chunk k + 2) once the store has read it
    const ApplyEntry* ae = &p.apply[G.first + tl.mat];
    uint8_t* ws = gemm_out(ec, b);
    gemm_apply_slot(ae->d, ws, lane, f);
    gemm_export_o(ae->d, r0 + lane, c0, G.m, G.n, f);
    ptx::fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (r0 < G.m && !ec.skip_w) {
        if (ae->d.tall) ptx::tma_store_2d(&ae->wmap, ws, r0, c0);
        else ptx::tma_store_2d(&ae->wmap, ws, c0, r0);
      }
      ptx::bulk_commit();
      ptx::bulk_wait_read_all();
    }
    __syncwarp();
    if (k + 2 < cnt) gemm_prefetch(p, G, tl, ec, b, c0 + 2 * kGC * ec.nslices, r0);
    return true;
  }
  // the inputs were consumed above; once every lane is past this point the
  // input buffer can be refilled
  if (lane == 0) {
    TC_EPI_T0(t_w);
    if (ec.out_bufs == 2) ptx::bulk_wait_read_1();
    else ptx::bulk_wait_read_all();
    TC_EPI_ADD(ec, p.apply ? 3 : 2, 1, t_w);
  }
  __syncwarp();
  if (k + 2 < cnt) gemm_prefetch(p, G, tl, ec, b, c0 + 2 * kGC * ec.nslices, r0);
  const int o = ec.out_bufs == 2 ? ec.obuf : 0;
  uint8_t* oh = gemm_out(ec, o);
  uint8_t* ol = oh + kXBox;
  const bool lo_out = p.x_lo_out != 0;
#pragma unroll
  for (int i = 0; i < kGC / 8; ++i) {
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float x0 = f[8 * i + 2 * j], x1 = f[8 * i + 2 * j + 1];
      const __nv_bfloat162 h2 = __floats2bfloat162_rn(x0, x1);
      const __nv_bfloat162 l2 = __floats2bfloat162_rn(x0 - __low2float(h2), x1 - __high2float(h2));
      hw[j] = *reinterpret_cast<const uint32_t*>(&h2);
      lw[j] = *reinterpret_cast<const uint32_t*>(&l2);
    }
    *reinterpret_cast<uint4*>(oh + sw_off(lane, i, kXRowBytes)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    if (lo_out)
      *reinterpret_cast<uint4*>(ol + sw_off(lane, i, kXRowBytes)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
  ptx::fence_async_smem();
  __syncwarp();
  if (lane == 0 && r0 < G.m) {  // a box that starts past the last row is not stored
    ptx::tma_store_4d(&p.map_c[tl.g], oh, c0, r0, tl.mat, G.buf_out);
    if (lo_out) ptx::tma_store_4d(&p.map_d[tl.g], ol, c0, r0, tl.mat, G.buf_out);
  }
  if (lane == 0) ptx::bulk_commit();   // one group per chunk (possibly empty)
  ec.obuf ^= 1;
  return true;
}

__device__ __forceinline__ void tmem_ld_chunk(uint32_t taddr, uint32_t (&v)[32]) { ptx::tmem_ld_32x32b_x32(taddr, v); }
__device__ __forceinline__ void tmem_ld_chunk(uint32_t taddr, uint32_t (&v)[16]) { ptx::tmem_ld_32x32b_x16(taddr, v); }

// The GEMM tile's epilogue for this warp; TMEM loads of chunk k + 1 are in
// flight while chunk k is processed.
__device__ __forceinline__ bool gemm_tile_epilogue(const PhaseParams& p, const PhaseGroup& G, const Tile& tl,
                                                   EpiCtx& ec, uint32_t tbase, int r0, int col0, int cnt,
                                                   volatile int* abort) {
  const int row = r0 + ec.lane;
  const float s = p.scale ? p.scale[G.first + tl.mat] : 1.f;
  // a plus this row's fp32 diagonal term of B (residual or exact diagonal)
  const float ar = p.coef_prev + ((G.diag_in && row < G.m) ? G.diag_in[(int64_t)tl.mat * G.diag_stride + row] : 0.f);
  if (cnt <= 0) return true;
  uint32_t va[kGC], vb[kGC];
  tmem_ld_chunk(tbase + (uint32_t)(kGC * gemm_chunk_col(ec, 0)), va);
  ptx::tmem_ld_wait_regs(va);
#pragma unroll 1
  for (int k = 0; k < cnt; k += 2) {
    const bool has1 = k + 1 < cnt;
    if (has1) tmem_ld_chunk(tbase + (uint32_t)(kGC * gemm_chunk_col(ec, k + 1)), vb);
    if (!gemm_chunk(p, G, tl, ec, col0, k, cnt, r0, s, ar, va, abort)) {
      if (has1) ptx::tmem_ld_wait_regs(vb);
      return false;
    }
    if (has1) {
      ptx::tmem_ld_wait_regs(vb);
      const bool has2 = k + 2 < cnt;
      if (has2) tmem_ld_chunk(tbase + (uint32_t)(kGC * gemm_chunk_col(ec, k + 2)), va);
      const bool okb = gemm_chunk(p, G, tl, ec, col0, k + 1, cnt, r0, s, ar, vb, abort);
      if (has2) ptx::tmem_ld_wait_regs(va);
      if (!okb) return false;
    }
  }
  return true;
}

template <bool kGram, bool kPair>
__device__ __forceinline__ void run_epilogue(const PhaseParams& p, const PairInfo& pi, uint64_t* tfull,
                                             uint64_t* tempty, uint32_t tmem_base, EpiCtx& ec, volatile int* abort) {
  using C = Cfg<kGram, kPair>;
  int acc = 0;
  uint32_t acc_phase = 0;
  bool ok = true;
  int lt = 0;   // local tile count (trace)
  (void)lt;
  const bool tracer = ec.quarter == 0 && ec.slice == 0 && ec.lane == 0 && pi.rank == 0;
  (void)tracer;
  for (int t = pi.unit; ok && t < p.total_tiles; t += pi.nunits, ++lt) {
    const Tile tl = decode_tile<kPair>(p, t, kGram);
    const PhaseGroup& G = p.g[tl.g];
    const int r0 = tl.bi * C::kTileM + TC * pi.rank + ec.quarter * 32;   // first row of this warp
    const int col0 = tl.bj * TN;
    int cnt = 0;
    GramChunks gc{0, 0};
    GramDiag gd;
    if (kGram) {
      gc = gram_chunks(G, ec, r0, col0);
      gram_diag_load(G, tl, ec.lane, r0 + ec.lane, col0, gd);
      if (G.prev) {
        cnt = gc.count;
        for (int k = 0; k < 2 && k < cnt; ++k) gram_prefetch_prev(p, tl, ec, k, col0 + 32 * (gc.first + k * ec.nslices), r0);
      }
    } else {
      const int nch = min(TN / kGC, (G.n - col0 + kGC - 1) / kGC);
      cnt = nch > ec.slice ? (nch - ec.slice + ec.nslices - 1) / ec.nslices : 0;
      // the W tensor map was written to global memory by the momentum kernel
      if (p.apply && ec.lane == 0) ptx::fence_tensormap_acquire(&p.apply[G.first + tl.mat].wmap);
      for (int k = 0; k < 2 && k < cnt; ++k) gemm_prefetch(p, G, tl, ec, k, col0 + kGC * gemm_chunk_col(ec, k), r0);
    }
    TC_PROF_T0(t_t);
    if (!wait_role<false>(&tfull[acc], acc_phase, abort, p.status, kStatusTimeoutEpilogue)) ok = false;
#ifdef MUON_TC_PROFILE
    if (ec.lane == 0) TC_PROF_ADD(4, t_t);
#endif
    if (tracer) TC_TRACE(lt, 2);
    if (ok) {
      ptx::tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(ec.quarter * 32) << 16) + (uint32_t)(acc * TN);
      if (kGram) ok = gram_tile_epilogue(p, G, tl, ec, tbase, r0, col0, gc, gd, abort);
      else ok = gemm_tile_epilogue(p, G, tl, ec, tbase, r0, col0, cnt, abort);
    }
    if (!ok) {
      // let this warp's prefetches in flight (X, or the previous A) land
      // before the CTA can exit
      for (int b = 0; b < 2; ++b)
        if (b < cnt) wait_drain(&ec.xfull[b], (ec.xphase >> b) & 1u);
      break;
    }
    if (tracer) TC_TRACE(lt, 3);
    ptx::tc_fence_before();
    if (kPair) {
      // one arrival per warp, on the even CTA's barrier
      __syncwarp();
      if (ec.lane == 0) ptx::mbar_arrive_cluster(ptx::mapa(ptx::smem_u32(&tempty[acc]), 0));
    } else {
      ptx::mbar_arrive(&tempty[acc]);
    }
    acc ^= 1;
    if (acc == 0) acc_phase ^= 1u;
  }
  if (ec.lane == 0) ptx::bulk_wait_all();
  __syncwarp();
}

template <bool kGram, bool kPair>
__device__ __forceinline__ void ns_tc_body(const PhaseParams& p) {
  using C = Cfg<kGram, kPair>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  uint8_t* epi = smem + C::kStages * C::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi + C::kEpiWarps * C::kEpiWarpBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::kStages;
  uint64_t* tfull = bars + 2 * C::kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* xfull = drain + 1;                 // 2 per epilogue warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xfull + 2 * C::kEpiWarps);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  PairInfo pi;
  if (kPair) {
    pi.rank = (int)ptx::cluster_ctarank();
    pi.unit = blockIdx.x >> 1;
    pi.nunits = gridDim.x >> 1;
  } else {
    pi.rank = 0;
    pi.unit = blockIdx.x;
    pi.nunits = gridDim.x;
  }
  TC_PROF_T0(t_cta);
  if (threadIdx.x == 0) TC_LIFE(0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], kPair ? 2 * C::kEpiWarps : 32 * C::kEpiWarps);
    }
    ptx::mbar_init(drain, 1);
    for (int i = 0; i < 2 * C::kEpiWarps; ++i) ptx::mbar_init(&xfull[i], 1);
    *abort = 0;
    ptx::fence_mbar_init();
    for (int g = 0; g < p.ngroups; ++g) {
      ptx::prefetch_tmap(&p.map_a[g]);
      ptx::prefetch_tmap(&p.map_c[g]);
      if (!kGram) ptx::prefetch_tmap(&p.map_b[g]);
      if (!kGram || p.g[g].prev) ptx::prefetch_tmap(&p.map_d[g]);
    }
  }
  if (warp == 1) {
    if (kPair) {
      ptx::tmem_alloc_pair(tmem_slot, TMEM_COLS);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(tmem_slot, TMEM_COLS);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  if (kPair) ptx::cluster_sync();   // both CTAs' barriers exist before any remote arrival
  else __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // set-up done: from here on this CTA reads and writes what earlier kernels
  // of the step produced
  grid_dependency_wait();
  if (threadIdx.x == 0) allow_dependent_launch();
  if (threadIdx.x == 0) TC_LIFE(1);

  if (warp == 0) {
    if (lane == 0) run_producer<kGram, kPair>(p, pi, smem, full, empty, abort);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && (!kPair || pi.rank == 0))
      run_mma<kGram, kPair>(p, pi, smem, full, empty, tfull, tempty, drain, tmem_base, abort);
    __syncwarp();
  } else {
    const int e = warp - 2;
    EpiCtx ec;
    ec.buf = epi + e * C::kEpiWarpBytes;
    ec.xfull = xfull + 2 * e;
    ec.xphase = 0;
    ec.obuf = 0;
    ec.quarter = warp & 3;   // TMEM lanes 32*(warp % 4) .. +31 are this warp's
    ec.slice = e / 4;
    ec.nslices = C::kSlices;
    ec.out_bufs = C::kOutBufs;
    ec.lane = lane;
    // the earlier kernels of the step have completed (grid dependency wait
    // above): a time-out among them leaves its bit in the status word
    ec.skip_w = !kGram && p.apply && p.status && *reinterpret_cast<volatile uint32_t*>(p.status) != 0u;
    run_epilogue<kGram, kPair>(p, pi, tfull, tempty, tmem_base, ec, abort);
  }

  ptx::tc_fence_before();
  if (kPair) ptx::cluster_sync();   // no CTA leaves while its pair may still touch its memory
  else __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    if (kPair) ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else ptx::tmem_dealloc(tmem_base, TMEM_COLS);
  }
#ifdef MUON_TC_PROFILE
  if (threadIdx.x == 0) TC_PROF_ADD(5, t_cta);
#endif
  if (threadIdx.x == 0) TC_LIFE(2);
}

template <bool kGram>
__global__ void __launch_bounds__(Cfg<kGram, false>::kThreads, 1) k_ns_tc(const __grid_constant__ PhaseParams p) {
  ns_tc_body<kGram, false>(p);
}

template <bool kGram>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Cfg<kGram, true>::kThreads, 1)
    k_ns_tc_pair(const __grid_constant__ PhaseParams p) {
  ns_tc_body<kGram, true>(p);
}

// Per device and kernel: the shared-memory opt-in is set, and the number of
// co-resident clusters found, on the first launch only (neither changes).
constexpr int kMaxDevices = 64;

template <typename K>
struct LaunchSetup {
  std::atomic<int> clusters[kMaxDevices];   // 0: not yet set up
};

// Sets the dynamic shared-memory size of `kernel` on the current device once;
// with `cluster` > 0 also returns how many clusters of that size fit at once.
template <typename K>
int setup_kernel(K kernel, LaunchSetup<K>& st, int smem, int threads, int sm_count, int cluster, int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  if (dev >= 0 && dev < kMaxDevices) {
    const int v = st.clusters[dev].load(std::memory_order_acquire);
    if (v > 0) {
      *out = v;
      return 0;
    }
  }
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return (int)e;
  int n = 1;
  if (cluster > 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)sm_count, 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
    if (e != cudaSuccess) return (int)e;
    if (n <= 0) return (int)cudaErrorLaunchOutOfResources;
  }
  if (dev >= 0 && dev < kMaxDevices) st.clusters[dev].store(n, std::memory_order_release);
  *out = n;
  return 0;
}

template <bool kGram>
int launch_tc(const PhaseParams& p, int grid, void* stream, bool pdl) {
  using C = Cfg<kGram, false>;
  if (p.total_tiles == 0) return 0;
  static LaunchSetup<decltype(&k_ns_tc<kGram>)> setup;
  int unused = 0;
  const int e = setup_kernel(&k_ns_tc<kGram>, setup, C::kSmemBytes, C::kThreads, grid, 0, &unused);
  if (e != 0) return e;
  if (grid > p.total_tiles) grid = p.total_tiles;
  return launch_kernel(k_ns_tc<kGram>, dim3((unsigned)grid), dim3(C::kThreads), C::kSmemBytes, stream, pdl, p);
}

// Pairs: as many co-resident clusters of two as the device holds, capped by
// the number of tiles.
template <bool kGram>
int launch_tc_pair(const PhaseParams& p, int sm_count, void* stream, bool pdl) {
  using C = Cfg<kGram, true>;
  if (p.total_tiles == 0) return 0;
  static LaunchSetup<decltype(&k_ns_tc_pair<kGram>)> setup;
  int clusters = 0;
  const int e = setup_kernel(&k_ns_tc_pair<kGram>, setup, C::kSmemBytes, C::kThreads, sm_count, 2, &clusters);
  if (e != 0) return e;
  if (clusters > sm_count / 2) clusters = sm_count / 2;
  if (clusters > p.total_tiles) clusters = p.total_tiles;
#ifdef MUON_TC_PROFILE
  fprintf(stderr, "k_ns_tc_pair<%d>: %d clusters of 2 for %d tiles (%d SMs)\n", (int)kGram, clusters, p.total_tiles,
          sm_count);
#endif
  return launch_kernel(k_ns_tc_pair<kGram>, dim3((unsigned)(2 * clusters)), dim3(C::kThreads), C::kSmemBytes, stream,
                       pdl, p);
}

}  // namespace

int tc_smem_bytes() { return Cfg<true, false>::kSmemBytes; }
int launch_gram_tc(const PhaseParams& p, int grid, void* stream, bool pdl) {
  return launch_tc<true>(p, grid, stream, pdl);
}
int launch_gemm_tc(const PhaseParams& p, int grid, void* stream, bool pdl) {
  return launch_tc<false>(p, grid, stream, pdl);
}
int launch_gram_tc_pair(const PhaseParams& p, int sm_count, void* stream, bool pdl) {
  return launch_tc_pair<true>(p, sm_count, stream, pdl);
}
int launch_gemm_tc_pair(const PhaseParams& p, int sm_count, void* stream, bool pdl) {
  return launch_tc_pair<false>(p, sm_count, stream, pdl);
}

}  // namespace muon

#ifdef MUON_TC_TRACE
// Trace reader of -DMUON_TC_TRACE builds: copies g_tc_trace, g_tc_life,
// g_tc_epi and g_tc_mma, in that order, into dst (bytes >= their sizes) and
// clears them.
extern "C" int muon_tc_trace_read(void* dst, size_t bytes) {
  struct Part { const void* sym; size_t size; };
  const Part parts[4] = {{&muon::g_tc_trace, sizeof(muon::g_tc_trace)},
                         {&muon::g_tc_life, sizeof(muon::g_tc_life)},
                         {&muon::g_tc_epi, sizeof(muon::g_tc_epi)},
                         {&muon::g_tc_mma, sizeof(muon::g_tc_mma)}};
  size_t total = 0;
  for (const Part& q : parts) total += q.size;
  if (bytes < total) return -1;
  size_t off = 0;
  for (const Part& q : parts) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, q.sym) != cudaSuccess) return -2;
    if (cudaMemcpy(static_cast<char*>(dst) + off, addr, q.size, cudaMemcpyDeviceToHost) != cudaSuccess) return -3;
    if (cudaMemset(addr, 0, q.size) != cudaSuccess) return -4;
    off += q.size;
  }
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -5;
}
#endif
