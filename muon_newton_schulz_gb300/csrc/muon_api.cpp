// C ABI of the batched Muon step: validation, batch planning (shape groups,
// workspace layout, tile lists, TMA tensor maps) and the stream-ordered
// launch sequence.  See include/muon.h for the contract.
#include "muon.h"

#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <array>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <map>
#include <memory>
#include <new>
#include <string>
#include <utility>
#include <vector>

#include "muon_internal.h"

using muon::EltMat;
using muon::EltParams;
using muon::PhaseGroup;
using muon::PhaseParams;

namespace {

constexpr int64_t kMaxMinDim = 32768;        // m = min(rows, cols)
constexpr int64_t kMaxMaxDim = 1ll << 24;    // n = max(rows, cols)
constexpr int kMaxIters = 64;
constexpr int kMaxProfiledSteps = 1024;

struct StepEvents {
  std::vector<cudaEvent_t> ev;
  int iters = 0;
  int apply_launches = 0;
};

// One entry of a step's launch sequence: a kernel with its parameter block
// (an index into StepPlan::elt or StepPlan::phase), or a profiling mark.
struct LaunchRec {
  enum Kind : uint8_t { kMomentum, kFinalize, kGram, kGemm, kApply, kMark } kind;
  uint32_t index;
  bool pdl;
};

// Everything muon_step launches for one batch: validated once, then reused
// while the caller passes the same descriptors (byte for byte) and workspace.
struct StepPlan {
  std::vector<muon_matrix_desc> key;
  const void* ws = nullptr;
  size_t need = 0;
  std::vector<muon::EltParams> elt;
  std::vector<muon::PhaseParams> phase;
  std::vector<LaunchRec> seq;
  int iters = 0;
  int apply_launches = 0;
  int kernels = 0;                  // kernel launches in seq
  int uses = 0;                     // steps run from this plan
  cudaGraphExec_t exec = nullptr;   // the launch sequence as a graph, from the second use on
  bool graph_tried = false;
  ~StepPlan() {
    if (exec) cudaGraphExecDestroy(exec);
  }
};

constexpr size_t kPlanCacheEntries = 32;

}  // namespace

struct muon_handle_s {
  muon_config cfg{};
  int device = -1;
  int sm_count = 0;
  std::string err;
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  int64_t launches = 0;
  bool profiling = false;
  std::vector<StepEvents> recorded;
  std::vector<cudaEvent_t> pool;
  // failure-path test hook, read once at muon_create: the first Gram launch of
  // every step issues no loads, so its bounded waits run out
  bool withhold_loads = false;
  // most recently used step plans first
  std::vector<std::unique_ptr<StepPlan>> plans;
  int64_t plan_builds = 0;
  // stream on which plans are captured into graphs, created on first use
  cudaStream_t capture_stream = nullptr;
  int64_t graph_launches = 0;
  // muon_step_host: copy-in, step and copy-out streams and their events,
  // created on first use
  cudaStream_t host_streams[3] = {nullptr, nullptr, nullptr};
  std::vector<cudaEvent_t> host_events;
  // the workspace of the last muon_step_host call: a status word at the start
  // of each of its slots
  const void* host_ws = nullptr;
  size_t host_slot_bytes = 0;
  int host_slots = 0;
};

namespace {

struct MatPlan {
  int desc;          // index into the caller's descriptor array
  int64_t rows, cols, m, n;
  bool tall;
  int group, in_group;
  int global;        // group.first + in_group
  int64_t elt_tiles, tiles_c;
  int64_t partial_begin;
};

struct GroupPlan {
  int64_t m, n, ldx, lda;
  int count = 0, first = 0;
  std::vector<int> mats;  // indices into Plan::mats
  size_t off_xm = 0, off_xb = 0, off_a = 0, off_b = 0;
  size_t off_da = 0, off_db = 0;  // fp32 diagonal terms of A and B (tensor-core path)
};

struct Plan {
  std::vector<MatPlan> mats;
  std::vector<GroupPlan> groups;
  size_t off_status = 0, off_scale = 0, off_partials = 0, off_apply = 0, bytes = 0;
  int64_t total_partials = 0;
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool finite_f(float x) { return std::isfinite(x); }

muon_status fail(muon_handle h, muon_status s, const std::string& why) {
  if (h) h->err = why;
  return s;
}

muon_status check_config(const muon_config& c, std::string& why) {
  if (!finite_f(c.beta) || !finite_f(c.a) || !finite_f(c.b) || !finite_f(c.c) || !finite_f(c.eps) ||
      !finite_f(c.scale_coeff)) {
    why = "config: beta, a, b, c, eps and scale_coeff must be finite";
    return MUON_ERR_INVALID_ARG;
  }
  if (c.eps < 0.f) { why = "config: eps must be >= 0"; return MUON_ERR_INVALID_ARG; }
  if (c.ns_iters < 0 || c.ns_iters > kMaxIters) { why = "config: ns_iters must be in [0, 64]"; return MUON_ERR_INVALID_ARG; }
  if (c.nesterov != 0 && c.nesterov != 1) { why = "config: nesterov must be 0 or 1"; return MUON_ERR_INVALID_ARG; }
  if (c.dampening != 0 && c.dampening != 1) { why = "config: dampening must be 0 or 1"; return MUON_ERR_INVALID_ARG; }
  if (c.mode != MUON_MODE_BF16 && c.mode != MUON_MODE_FP32_VALIDATE) { why = "config: unknown mode"; return MUON_ERR_UNSUPPORTED; }
  return MUON_OK;
}

struct Range { uintptr_t lo, hi; int desc; const char* what; };

// Checks every descriptor; on success `ranges` holds the byte range of each
// caller buffer (sorted by address, none overlapping).
muon_status validate(const muon_matrix_desc* d, int n, std::string& why, std::vector<Range>& ranges) {
  ranges.clear();
  if (n < 0) { why = "n must be >= 0"; return MUON_ERR_INVALID_ARG; }
  if (n > 0 && !d) { why = "descs is NULL"; return MUON_ERR_INVALID_ARG; }
  for (int i = 0; i < n; ++i) {
    const muon_matrix_desc& x = d[i];
    const std::string at = "desc " + std::to_string(i) + ": ";
    if (x.rows < 0 || x.cols < 0) { why = at + "rows and cols must be >= 0"; return MUON_ERR_INVALID_ARG; }
    if (x.rows == 0 || x.cols == 0) continue;  // empty matrix: skipped
    const int64_t m = std::min(x.rows, x.cols), nn = std::max(x.rows, x.cols);
    if (m > kMaxMinDim || nn > kMaxMaxDim) {
      why = at + "min(rows, cols) must be <= 32768 and max(rows, cols) <= 16777216";
      return MUON_ERR_INVALID_ARG;
    }
    if (x.w_dtype != MUON_F32 && x.w_dtype != MUON_BF16) { why = at + "w_dtype must be MUON_F32 or MUON_BF16"; return MUON_ERR_INVALID_ARG; }
    if (!x.W || !x.G || !x.M) { why = at + "W, G and M must be non-NULL"; return MUON_ERR_INVALID_ARG; }
    const int64_t wes = x.w_dtype == MUON_BF16 ? 2 : 4;
    struct B { const void* p; int64_t ld; int64_t es; const char* name; };
    const B bufs[4] = {{x.W, x.ldw, wes, "W"}, {x.G, x.ldg, 4, "G"}, {x.M, x.ldm, 4, "M"}, {x.O_out, x.ldo, 4, "O_out"}};
    for (const B& b : bufs) {
      if (!b.p) continue;
      if (reinterpret_cast<uintptr_t>(b.p) % 16 != 0) { why = at + b.name + " must be 16-byte aligned"; return MUON_ERR_INVALID_ARG; }
      if (b.ld < x.cols) { why = at + "ld of " + b.name + " must be >= cols"; return MUON_ERR_INVALID_ARG; }
      if ((b.ld * b.es) % 16 != 0) { why = at + "ld of " + b.name + " times its element size must be a multiple of 16 bytes"; return MUON_ERR_INVALID_ARG; }
      const uintptr_t lo = reinterpret_cast<uintptr_t>(b.p);
      const uintptr_t hi = lo + (uintptr_t)(((x.rows - 1) * b.ld + x.cols) * b.es);
      ranges.push_back({lo, hi, i, b.name});
    }
    if (!std::isfinite(x.lr)) { why = at + "lr must be finite"; return MUON_ERR_INVALID_ARG; }
  }
  std::sort(ranges.begin(), ranges.end(), [](const Range& a, const Range& b) { return a.lo < b.lo; });
  for (size_t i = 1; i < ranges.size(); ++i) {
    if (ranges[i].lo < ranges[i - 1].hi) {
      why = "buffers overlap: desc " + std::to_string(ranges[i - 1].desc) + " " + ranges[i - 1].what + " and desc " +
            std::to_string(ranges[i].desc) + " " + ranges[i].what;
      return MUON_ERR_INVALID_ARG;
    }
  }
  return MUON_OK;
}

Plan build_plan(const muon_config& cfg, const muon_matrix_desc* d, int n) {
  Plan P;
  std::map<std::pair<int64_t, int64_t>, int> by_shape;
  for (int i = 0; i < n; ++i) {
    if (d[i].rows == 0 || d[i].cols == 0) continue;
    MatPlan mp{};
    mp.desc = i;
    mp.rows = d[i].rows;
    mp.cols = d[i].cols;
    mp.tall = mp.rows > mp.cols;
    mp.m = std::min(mp.rows, mp.cols);
    mp.n = std::max(mp.rows, mp.cols);
    mp.tiles_c = cdiv(mp.cols, muon::kEltTile);
    mp.elt_tiles = cdiv(mp.rows, muon::kEltTile) * mp.tiles_c;
    auto key = std::make_pair(mp.m, mp.n);
    auto it = by_shape.find(key);
    if (it == by_shape.end()) {
      GroupPlan g;
      g.m = mp.m;
      g.n = mp.n;
      g.ldx = (int64_t)align_up((size_t)mp.n, 64);
      g.lda = (int64_t)align_up((size_t)mp.m, 64);
      P.groups.push_back(g);
      it = by_shape.emplace(key, (int)P.groups.size() - 1).first;
    }
    mp.group = it->second;
    P.groups[mp.group].mats.push_back((int)P.mats.size());
    P.mats.push_back(mp);
  }
  // largest per-tile work first (static schedules then end with short tiles)
  std::vector<int> order(P.groups.size());
  for (size_t i = 0; i < order.size(); ++i) order[i] = (int)i;
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
    const GroupPlan &x = P.groups[a], &y = P.groups[b];
    if (x.n != y.n) return x.n > y.n;
    return x.m > y.m;
  });
  std::vector<GroupPlan> sorted;
  for (int gi : order) sorted.push_back(P.groups[gi]);
  P.groups.swap(sorted);
  int first = 0;
  for (size_t g = 0; g < P.groups.size(); ++g) {
    GroupPlan& G = P.groups[g];
    G.first = first;
    G.count = (int)G.mats.size();
    for (int k = 0; k < G.count; ++k) {
      MatPlan& mp = P.mats[G.mats[k]];
      mp.group = (int)g;
      mp.in_group = k;
      mp.global = first + k;
    }
    first += G.count;
  }
  int64_t partials = 0;
  for (MatPlan& mp : P.mats) {
    mp.partial_begin = partials;
    partials += mp.elt_tiles;
  }
  P.total_partials = partials;

  const bool bf16 = cfg.mode == MUON_MODE_BF16;
  const size_t es = bf16 ? 2 : 4;
  size_t off = 0;
  P.off_status = off;
  off += 256;
  P.off_scale = off;
  off = align_up(off + P.mats.size() * sizeof(float), 256);
  P.off_partials = off;
  off = align_up(off + (size_t)partials * sizeof(double), 256);
  P.off_apply = off;
  off = align_up(off + P.mats.size() * sizeof(muon::ApplyEntry), 1024);
  for (GroupPlan& G : P.groups) {
    const size_t xel = (size_t)G.count * G.m * G.ldx;
    const size_t ael = (size_t)G.count * G.m * G.lda;
    // X ping-pong: fp32 (validation mode), or bf16 hi at off_xm and bf16 lo
    // at off_xb (tensor-core mode)
    G.off_xm = off;
    off = align_up(off + 2 * xel * (bf16 ? 2 : 4), 1024);
    if (bf16) {
      G.off_xb = off;
      off = align_up(off + 2 * xel * 2, 1024);
    }
    G.off_a = off;
    off = align_up(off + ael * es, 1024);
    G.off_b = off;
    off = align_up(off + ael * es, 1024);
    if (bf16) {
      G.off_da = off;
      off = align_up(off + (size_t)G.count * G.lda * sizeof(float), 1024);
      G.off_db = off;
      off = align_up(off + (size_t)G.count * G.lda * sizeof(float), 1024);
    }
  }
  P.bytes = off;
  return P;
}

bool encode_map(muon_handle h, CUtensorMap* map, void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t d3,
                uint64_t ld_bytes, uint64_t mat_bytes, uint64_t buf_bytes, uint32_t box0, uint32_t box1,
                CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  cuuint64_t dims[4] = {d0, d1, d2, d3};
  cuuint64_t strides[3] = {ld_bytes, mat_bytes, buf_bytes};
  cuuint32_t box[4] = {box0, box1, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = h->encode(map, dtype, 4, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    h->err = "cuTensorMapEncodeTiled failed with CUresult " + std::to_string((int)r);
    return false;
  }
  return true;
}

// 2-D map of a caller's weight matrix whose box is one GEMM epilogue chunk:
// kGemmChunk columns x 32 rows (wide), 32 columns x kGemmChunk rows (tall: W
// is X^T), with the swizzle matching the box row (32 B..128 B).
bool encode_w_map(muon_handle h, CUtensorMap* map, const muon_matrix_desc& d, bool tall) {
  const bool bf = d.w_dtype == MUON_BF16;
  const uint64_t es = bf ? 2 : 4;
  cuuint64_t dims[2] = {(cuuint64_t)d.cols, (cuuint64_t)d.rows};
  cuuint64_t strides[1] = {(cuuint64_t)(d.ldw * es)};
  const cuuint32_t chunk = (cuuint32_t)muon::kGemmChunk;
  cuuint32_t box[2] = {tall ? 32u : chunk, tall ? chunk : 32u};
  cuuint32_t estr[2] = {1, 1};
  const uint64_t row_bytes = box[0] * es;
  const CUtensorMapSwizzle swz = row_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                 : row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                   : CU_TENSOR_MAP_SWIZZLE_128B;
  CUresult r = h->encode(map, bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, d.W, dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    h->err = "cuTensorMapEncodeTiled (W) failed with CUresult " + std::to_string((int)r);
    return false;
  }
  return true;
}

// Tile counts of one group for the kernel that will run the phase.
void set_tiles(PhaseGroup& pg, bool gram, bool tc) {
  if (tc && muon::kUsePair) {
    // CTA pairs: 256 x 256 tiles; Gram keeps the tiles with bi <= bj
    pg.ni = (int32_t)cdiv(pg.m, 2 * muon::kTcM);
    if (gram) {
      pg.nj = pg.ni;
      pg.tiles_per_mat = pg.ni * (pg.ni + 1) / 2;
    } else {
      pg.nj = (int32_t)cdiv(pg.n, muon::kTcN);
      pg.tiles_per_mat = pg.ni * pg.nj;
    }
  } else if (tc) {
    pg.ni = (int32_t)cdiv(pg.m, muon::kTcM);
    if (gram) {
      pg.nj = (int32_t)cdiv(pg.m, muon::kTcN);
      int t = 0;
      for (int bj = 0; bj < pg.nj; ++bj) t += std::min(2 * bj + 2, pg.ni);
      pg.tiles_per_mat = t;
    } else {
      pg.nj = (int32_t)cdiv(pg.n, muon::kTcN);
      pg.tiles_per_mat = pg.ni * pg.nj;
    }
  } else {
    pg.ni = (int32_t)cdiv(pg.m, muon::kSimtTile);
    if (gram) {
      pg.nj = pg.ni;
      pg.tiles_per_mat = pg.ni * (pg.ni + 1) / 2;
    } else {
      pg.nj = (int32_t)cdiv(pg.n, muon::kSimtTile);
      pg.tiles_per_mat = pg.ni * pg.nj;
    }
  }
}

struct DeviceGuard {
  int old = -1;
  bool changed = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&old) == cudaSuccess && old != dev) changed = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (changed) cudaSetDevice(old);
  }
};

cudaEvent_t take_event(muon_handle h) {
  if (!h->pool.empty()) {
    cudaEvent_t e = h->pool.back();
    h->pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Cached plan for exactly these descriptors and this workspace, moved to the
// front of the cache, or null.
StepPlan* find_plan(muon_handle h, const muon_matrix_desc* descs, int n, const void* ws) {
  if (n <= 0 || !descs) return nullptr;
  for (size_t i = 0; i < h->plans.size(); ++i) {
    const StepPlan& p = *h->plans[i];
    if (p.ws != ws || p.key.size() != (size_t)n) continue;
    if (std::memcmp(p.key.data(), descs, sizeof(muon_matrix_desc) * (size_t)n) != 0) continue;
    if (i > 0) std::rotate(h->plans.begin(), h->plans.begin() + i, h->plans.begin() + i + 1);
    return h->plans.front().get();
  }
  return nullptr;
}

// Builds every parameter block of one step (elementwise launches, the
// Newton-Schulz phase launches with their tensor maps) and the launch order.
muon_status make_plan(muon_handle h, const Plan& P, const muon_matrix_desc* descs, int n, void* ws, StepPlan& out) {
  const muon_config& cfg = h->cfg;
  const bool bf16 = cfg.mode == MUON_MODE_BF16;
  const int iters = cfg.ns_iters;
  out.key.assign(descs, descs + n);
  out.ws = ws;
  out.need = P.bytes;
  out.iters = iters;
  uint8_t* base = static_cast<uint8_t*>(ws);
  uint32_t* status = reinterpret_cast<uint32_t*>(base + P.off_status);
  float* scale = reinterpret_cast<float*>(base + P.off_scale);
  double* partials = reinterpret_cast<double*>(base + P.off_partials);
  // tensor-core mode applies the weight update in the last GEMM's epilogue,
  // reading each matrix's W from a table the momentum kernel fills
  const bool fused_apply = bf16 && iters > 0;
  const bool withhold = bf16 && h->withhold_loads;
  muon::ApplyEntry* apply_table = reinterpret_cast<muon::ApplyEntry*>(base + P.off_apply);

  // X of matrix k of a group, ping-pong buffer `buf`: fp32 in validation
  // mode; the bf16 pair (hi, lo) in tensor-core mode
  auto xm_ptr = [&](const GroupPlan& G, int buf, int k) -> float* {
    return reinterpret_cast<float*>(base + G.off_xm) + ((size_t)buf * G.count + k) * (size_t)G.m * G.ldx;
  };
  auto xhi_ptr = [&](const GroupPlan& G, int buf, int k) -> __nv_bfloat16* {
    return reinterpret_cast<__nv_bfloat16*>(base + G.off_xm) + ((size_t)buf * G.count + k) * (size_t)G.m * G.ldx;
  };
  auto xlo_ptr = [&](const GroupPlan& G, int buf, int k) -> __nv_bfloat16* {
    return reinterpret_cast<__nv_bfloat16*>(base + G.off_xb) + ((size_t)buf * G.count + k) * (size_t)G.m * G.ldx;
  };

  // ---- elementwise parameter blocks (momentum/norm and apply), chunked
  auto fill_elt = [&](EltParams& ep, size_t b, size_t e, int final_buf) {
    std::memset(&ep, 0, sizeof(ep));
    ep.nmats = (int32_t)(e - b);
    ep.nesterov = cfg.nesterov;
    ep.dampening = cfg.dampening;
    ep.apply_scale = iters == 0 ? 1 : 0;
    ep.beta = cfg.beta;
    ep.eps = cfg.eps;
    ep.partials = partials;
    ep.scale = scale;
    ep.status = b == 0 ? status : nullptr;
    ep.apply = fused_apply ? apply_table : nullptr;
    int64_t tiles = 0;
    for (size_t i = b; i < e; ++i) {
      const MatPlan& mp = P.mats[i];
      const GroupPlan& G = P.groups[mp.group];
      const muon_matrix_desc& d = descs[mp.desc];
      EltMat& x = ep.mats[i - b];
      x.G = d.G;
      x.M = d.M;
      x.W = d.W;
      x.O_out = d.O_out;
      if (bf16) {
        x.xhi0 = xhi_ptr(G, 0, mp.in_group);
        x.xlo0 = xlo_ptr(G, 0, mp.in_group);
        x.xhi_final = xhi_ptr(G, final_buf, mp.in_group);
        x.xlo_final = xlo_ptr(G, final_buf, mp.in_group);
      } else {
        x.xm0 = xm_ptr(G, 0, mp.in_group);
        x.xm_final = xm_ptr(G, final_buf, mp.in_group);
      }
      x.ldg = d.ldg;
      x.ldm = d.ldm;
      x.ldw = d.ldw;
      x.ldo = d.ldo;
      x.ldx = G.ldx;
      x.tile_begin = tiles;
      x.partial_begin = mp.partial_begin;
      x.rows = (int32_t)mp.rows;
      x.cols = (int32_t)mp.cols;
      x.tiles_c = (int32_t)mp.tiles_c;
      x.ntiles = (int32_t)mp.elt_tiles;
      x.tall = mp.tall ? 1 : 0;
      x.w_bf16 = d.w_dtype == MUON_BF16 ? 1 : 0;
      x.mat = mp.global;
      x.lr_eff = (float)((double)d.lr * (double)cfg.scale_coeff * std::sqrt((double)mp.n));
      if (fused_apply && !encode_w_map(h, &x.wmap, d, mp.tall)) return false;
      tiles += mp.elt_tiles;
    }
    ep.total_tiles = tiles;
    return true;
  };

  const int final_buf = iters % 2;
  // every launch after the step's first is a programmatic dependent of the
  // kernel before it (the kernels wait for their predecessor themselves)
  bool pdl = false;
  auto push = [&](LaunchRec::Kind k, uint32_t idx) {
    out.seq.push_back({k, idx, pdl});
    if (k != LaunchRec::kMark) {
      pdl = muon::kUsePdl;
      out.kernels += 1;
    }
  };
  push(LaunchRec::kMark, 0);
  for (size_t b = 0; b < P.mats.size(); b += muon::kMaxEltMats) {
    const size_t e = std::min(P.mats.size(), b + (size_t)muon::kMaxEltMats);
    out.elt.emplace_back();
    if (!fill_elt(out.elt.back(), b, e, final_buf)) return MUON_ERR_CUDA;
    const uint32_t idx = (uint32_t)(out.elt.size() - 1);
    push(LaunchRec::kMomentum, idx);
    push(LaunchRec::kFinalize, idx);
  }
  push(LaunchRec::kMark, 0);

  // ---- Newton-Schulz iterations
  // tensor-core mode stores X_t as the bf16 pair (hi, lo) for t < lo_iters and
  // as bf16 alone for the last MUON_X_LO_TAIL stored iterates, whose rounding
  // the remaining iterations amplify least (X0, written by the momentum
  // kernel, always has both halves)
  const int lo_iters = std::max(1, iters - MUON_X_LO_TAIL);
  for (int it = 0; it < iters; ++it) {
    const int cur = it % 2, nxt = 1 - cur;
    for (int phase = 0; phase < 3; ++phase) {
      const bool gram = phase < 2;
      for (size_t gb = 0; gb < P.groups.size(); gb += muon::kMaxGroups) {
        const size_t ge = std::min(P.groups.size(), gb + (size_t)muon::kMaxGroups);
        out.phase.emplace_back();
        PhaseParams* pp = &out.phase.back();
        std::memset(pp, 0, sizeof(*pp));
        pp->ngroups = (int32_t)(ge - gb);
        pp->status = status;
        pp->apply = (fused_apply && phase == 2 && it + 1 == iters) ? apply_table : nullptr;
        // failure-path test hook: the step's first Gram launch withholds its
        // loads so its bounded waits expire
        pp->withhold_loads = (withhold && it == 0 && phase == 0 && gb == 0) ? 1 : 0;
        pp->x_lo_in = (phase == 2 && it < lo_iters) ? 1 : 0;
        pp->x_lo_out = (phase == 2 && it + 1 < lo_iters) ? 1 : 0;
        pp->scale = (it == 0 && phase != 1) ? scale : nullptr;
        pp->coef_acc = phase == 1 ? cfg.c : 1.f;
        pp->coef_prev = phase == 1 ? cfg.b : (phase == 2 ? cfg.a : 0.f);
        int tiles = 0;
        for (size_t gi = gb; gi < ge; ++gi) {
          const GroupPlan& G = P.groups[gi];
          PhaseGroup& pg = pp->g[gi - gb];
          pg.m = (int32_t)G.m;
          pg.n = (int32_t)G.n;
          pg.count = G.count;
          pg.first = G.first;
          pg.K = (int32_t)(phase == 0 ? G.n : G.m);
          set_tiles(pg, gram, bf16);
          pg.tile_begin = tiles;
          tiles += pg.tiles_per_mat * G.count;
          pg.buf_in = phase == 1 ? 0 : cur;
          pg.buf_out = nxt;
          const size_t es = bf16 ? 2 : 4;
          uint8_t* Abuf = base + G.off_a;
          uint8_t* Bbuf = base + G.off_b;
          const int64_t a_stride = G.m * G.lda;
          const int64_t x_stride = G.m * G.ldx;
          if (bf16) {
            // fp32 diagonal terms: the bf16 rounding residual of A's diagonal
            // (Gram 1 -> Gram 2), and B's diagonal residual, or in the last
            // two iterations B's exact diagonal (Gram 2 -> GEMM)
            float* dA = reinterpret_cast<float*>(base + G.off_da);
            float* dB = reinterpret_cast<float*>(base + G.off_db);
            pg.diag_stride = G.lda;
            pg.diag_in = phase == 0 ? nullptr : (phase == 1 ? dA : dB);
            pg.diag_out = phase == 0 ? dA : (phase == 1 ? dB : nullptr);
            pp->diag_exact = (phase == 1 && it + 2 >= iters) ? 1 : 0;
          }
          if (phase == 0) {          // A = s^2 X X^T
            pg.opP = bf16 ? (const void*)xhi_ptr(G, cur, 0) : (const void*)xm_ptr(G, cur, 0);
            pg.ld_p = G.ldx;
            pg.p_stride = x_stride;
            pg.prev = nullptr;
            pg.out = Abuf;
            pg.ld_out = G.lda;
            pg.out_stride = a_stride;
          } else if (phase == 1) {   // B = b A + c A A^T
            pg.opP = Abuf;
            pg.ld_p = G.lda;
            pg.p_stride = a_stride;
            pg.prev = Abuf;
            pg.ld_prev = G.lda;
            pg.prev_stride = a_stride;
            pg.out = Bbuf;
            pg.ld_out = G.lda;
            pg.out_stride = a_stride;
          } else {                   // X' = s (a X + B X)
            pg.opP = Bbuf;
            pg.ld_p = G.lda;
            pg.p_stride = a_stride;
            pg.opX = bf16 ? (const void*)xhi_ptr(G, cur, 0) : (const void*)xm_ptr(G, cur, 0);
            pg.ld_x = G.ldx;
            pg.x_stride = x_stride;
            // validation mode reads and writes fp32 X directly; the tensor-core
            // kernel moves the (hi, lo) pair through the tensor maps below
            pg.prev = bf16 ? nullptr : xm_ptr(G, cur, 0);
            pg.ld_prev = G.ldx;
            pg.prev_stride = x_stride;
            pg.out = bf16 ? nullptr : xm_ptr(G, nxt, 0);
            pg.ld_out = G.ldx;
            pg.out_stride = x_stride;
          }
          if (bf16) {
            const uint64_t cnt = (uint64_t)G.count;
            const uint64_t xrow = (uint64_t)G.ldx * es, xmat = (uint64_t)x_stride * es;
            const uint64_t arow = (uint64_t)G.lda * es, amat = (uint64_t)a_stride * es;
            bool ok = true;
            CUtensorMap* ma = &pp->map_a[gi - gb];
            CUtensorMap* mb = &pp->map_b[gi - gb];
            CUtensorMap* mc = &pp->map_c[gi - gb];
            CUtensorMap* md = &pp->map_d[gi - gb];
            if (phase == 0) {
              ok = encode_map(h, ma, xhi_ptr(G, 0, 0), G.n, G.m, cnt, 2, xrow, xmat, xmat * cnt, 64, 128) &&
                   encode_map(h, mc, Abuf, G.m, G.m, cnt, 1, arow, amat, amat * cnt, 32, 32,
                              CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, CU_TENSOR_MAP_SWIZZLE_64B);
            } else if (phase == 1) {
              // map_d: 32 x 32 blocks of A itself, prefetched by the epilogue
              ok = encode_map(h, ma, Abuf, G.m, G.m, cnt, 1, arow, amat, amat * cnt, 64, 128) &&
                   encode_map(h, mc, Bbuf, G.m, G.m, cnt, 1, arow, amat, amat * cnt, 32, 32,
                              CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, CU_TENSOR_MAP_SWIZZLE_64B) &&
                   encode_map(h, md, Abuf, G.m, G.m, cnt, 1, arow, amat, amat * cnt, 32, 32,
                              CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, CU_TENSOR_MAP_SWIZZLE_64B);
            } else {
              // epilogue boxes: 32 rows x kGemmChunk bf16 (32- or 64-byte rows)
              const uint32_t gc = (uint32_t)muon::kGemmChunk;
              const CUtensorMapSwizzle eswz = gc == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
              ok = encode_map(h, ma, Bbuf, G.m, G.m, cnt, 1, arow, amat, amat * cnt, 64, 128) &&
                   encode_map(h, mb, xhi_ptr(G, 0, 0), G.n, G.m, cnt, 2, xrow, xmat, xmat * cnt, 64, 64) &&
                   encode_map(h, mc, xhi_ptr(G, 0, 0), G.n, G.m, cnt, 2, xrow, xmat, xmat * cnt, gc, 32,
                              CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, eswz) &&
                   encode_map(h, md, xlo_ptr(G, 0, 0), G.n, G.m, cnt, 2, xrow, xmat, xmat * cnt, gc, 32,
                              CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, eswz);
            }
            if (!ok) return MUON_ERR_CUDA;
          }
        }
        pp->total_tiles = tiles;
        push(gram ? LaunchRec::kGram : LaunchRec::kGemm, (uint32_t)(out.phase.size() - 1));
      }
      push(LaunchRec::kMark, 0);
    }
  }

  // ---- apply (a separate kernel unless the last GEMM did it)
  if (!fused_apply) {
    for (size_t b = 0; b < P.mats.size(); b += muon::kMaxEltMats) {
      const size_t e = std::min(P.mats.size(), b + (size_t)muon::kMaxEltMats);
      out.elt.emplace_back();
      if (!fill_elt(out.elt.back(), b, e, final_buf)) return MUON_ERR_CUDA;
      push(LaunchRec::kApply, (uint32_t)(out.elt.size() - 1));
      out.apply_launches += 1;
    }
  }
  push(LaunchRec::kMark, 0);
  return MUON_OK;
}

// Launches a plan's kernels in order on `stream` (profiling events at its
// marks when enabled).
muon_status issue_plan(muon_handle h, const StepPlan& plan, void* stream) {
  DeviceGuard guard(h->device);
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const bool record = h->profiling && (int)h->recorded.size() < kMaxProfiledSteps;
  StepEvents se;
  muon_status st = MUON_OK;
  for (const LaunchRec& r : plan.seq) {
    int rc = 0;
    const char* what = "";
    switch (r.kind) {
      case LaunchRec::kMark:
        if (record) {
          cudaEvent_t e = take_event(h);
          if (e) {
            cudaEventRecord(e, cs);
            se.ev.push_back(e);
          }
        }
        continue;
      case LaunchRec::kMomentum:
        nvtxRangePushA("muon.momentum_norm");
        rc = muon::launch_momentum_norm(plan.elt[r.index], stream, r.pdl);
        nvtxRangePop();
        what = "momentum/norm kernel";
        break;
      case LaunchRec::kFinalize:
        nvtxRangePushA("muon.norm_finalize");
        rc = muon::launch_norm_finalize(plan.elt[r.index], stream, r.pdl);
        nvtxRangePop();
        what = "norm finalize kernel";
        break;
      case LaunchRec::kApply:
        nvtxRangePushA("muon.apply");
        rc = muon::launch_apply(plan.elt[r.index], stream, r.pdl);
        nvtxRangePop();
        what = "apply kernel";
        break;
      case LaunchRec::kGram:
      case LaunchRec::kGemm: {
        const bool gram = r.kind == LaunchRec::kGram;
        const PhaseParams& pp = plan.phase[r.index];
        // one range per launch: the phase's name as the bench's profile uses it
        nvtxRangePushA(!gram ? "muon.gemm_update" : (pp.ngroups > 0 && pp.g[0].prev ? "muon.gram_aa_combine" : "muon.gram_xxt"));
        if (h->cfg.mode == MUON_MODE_BF16 && muon::kUsePair)
          rc = gram ? muon::launch_gram_tc_pair(pp, h->sm_count, stream, r.pdl)
                    : muon::launch_gemm_tc_pair(pp, h->sm_count, stream, r.pdl);
        else if (h->cfg.mode == MUON_MODE_BF16)
          rc = gram ? muon::launch_gram_tc(pp, h->sm_count, stream, r.pdl)
                    : muon::launch_gemm_tc(pp, h->sm_count, stream, r.pdl);
        else
          rc = gram ? muon::launch_gram_f32(pp, stream, r.pdl) : muon::launch_gemm_f32(pp, stream, r.pdl);
        nvtxRangePop();
        what = gram ? "Gram kernel" : "GEMM kernel";
        break;
      }
    }
    if (rc != 0) {
      st = fail(h, MUON_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString((cudaError_t)rc));
      break;
    }
    h->launches += 1;
  }
  if (!se.ev.empty()) {
    se.iters = plan.iters;
    se.apply_launches = plan.apply_launches;
    if (st == MUON_OK && (int)se.ev.size() == 3 + 3 * plan.iters) h->recorded.push_back(std::move(se));
    else for (cudaEvent_t e : se.ev) h->pool.push_back(e);
  }
  return st;
}

// Captures a plan's launches into a graph on the handle's capture stream
// (on failure the plan keeps running eagerly).
void build_graph(muon_handle h, StepPlan& plan) {
  plan.graph_tried = true;
  if (!h->capture_stream && cudaStreamCreateWithFlags(&h->capture_stream, cudaStreamNonBlocking) != cudaSuccess) {
    cudaGetLastError();
    return;
  }
  if (cudaStreamBeginCapture(h->capture_stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaGetLastError();
    return;
  }
  const int64_t launches = h->launches;
  const std::string err = h->err;
  const muon_status st = issue_plan(h, plan, h->capture_stream);
  h->launches = launches;   // captured, not run
  h->err = err;
  cudaGraph_t g = nullptr;
  cudaError_t e = cudaStreamEndCapture(h->capture_stream, &g);
  if (st != MUON_OK || e != cudaSuccess || !g) {
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();
    return;
  }
  cudaGraphExec_t ex = nullptr;
  e = cudaGraphInstantiate(&ex, g, 0);
  cudaGraphDestroy(g);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return;
  }
  plan.exec = ex;
}

// Runs one step from a plan: its first use launches the kernels one by one
// (which also does the kernels' one-time set-up), later uses replay the plan
// as a CUDA graph, unless profiling is on (events go between the launches) or
// the caller's stream is being captured (the launches then join the caller's
// graph).
muon_status run_plan(muon_handle h, StepPlan& plan, void* stream) {
  const int use = plan.uses++;
  if (use > 0 && !h->profiling) {
    DeviceGuard guard(h->device);
    cudaStreamCaptureStatus cst = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(reinterpret_cast<cudaStream_t>(stream), &cst) != cudaSuccess) {
      cudaGetLastError();
      cst = cudaStreamCaptureStatusActive;
    }
    if (cst == cudaStreamCaptureStatusNone) {
      if (!plan.exec && !plan.graph_tried) build_graph(h, plan);
      if (plan.exec) {
        nvtxRangePushA("muon.step_graph_replay");
        const cudaError_t e = cudaGraphLaunch(plan.exec, reinterpret_cast<cudaStream_t>(stream));
        nvtxRangePop();
        if (e != cudaSuccess) return fail(h, MUON_ERR_CUDA, std::string("cudaGraphLaunch: ") + cudaGetErrorString(e));
        h->launches += plan.kernels;
        h->graph_launches += 1;
        return MUON_OK;
      }
    }
  }
  return issue_plan(h, plan, stream);
}

// ---- steps on host-resident buffers// ---- steps on host-resident buffers

constexpr uint32_t kHostBits = MUON_HOST_W | MUON_HOST_G | MUON_HOST_M | MUON_HOST_O;

// Where one chunk of matrices is staged inside a slot of the device workspace.
struct HostChunk {
  std::vector<int> mats;                    // caller descriptor indices
  std::vector<std::array<size_t, 4>> off;   // per matrix: staged W, G, M, O_out (or SIZE_MAX)
  std::vector<std::array<int64_t, 4>> ld;   // their leading dimensions (elements)
  size_t ws_off = 0, ws_bytes = 0;          // the chunk's muon_step workspace in the slot
};

struct HostLayout {
  std::vector<HostChunk> chunks;
  size_t slot_bytes = 0;
};

// Elements per staged row: cols rounded up to 16 bytes.
int64_t staged_ld(int64_t cols, int64_t es) { return (int64_t)align_up((size_t)(cols * es), 16) / es; }

// Chunks of consecutive non-empty matrices and the slot layout: every slot
// starts with the step workspace (so its status word is at the slot's first
// byte), followed by the staged host-resident buffers of its chunk.
void host_layout(const muon_config& cfg, const muon_matrix_desc* d, int n, const muon_host_pipeline& pl,
                 HostLayout& L) {
  std::vector<int> mats;
  for (int i = 0; i < n; ++i)
    if (d[i].rows > 0 && d[i].cols > 0) mats.push_back(i);
  size_t ws_max = 0;
  for (size_t b = 0; b < mats.size(); b += (size_t)pl.chunk_matrices) {
    HostChunk c;
    const size_t e = std::min(mats.size(), b + (size_t)pl.chunk_matrices);
    std::vector<muon_matrix_desc> shapes;
    for (size_t k = b; k < e; ++k) {
      c.mats.push_back(mats[k]);
      shapes.push_back(d[mats[k]]);
    }
    c.ws_off = 0;
    c.ws_bytes = build_plan(cfg, shapes.data(), (int)shapes.size()).bytes;
    ws_max = std::max(ws_max, c.ws_bytes);
    L.chunks.push_back(std::move(c));
  }
  const size_t stage0 = align_up(ws_max, 1024);
  L.slot_bytes = stage0;
  for (HostChunk& c : L.chunks) {
    size_t off = stage0;
    for (int idx : c.mats) {
      const muon_matrix_desc& x = d[idx];
      std::array<size_t, 4> o;
      std::array<int64_t, 4> ld;
      const int64_t wes = x.w_dtype == MUON_BF16 ? 2 : 4;
      const int64_t es[4] = {wes, 4, 4, 4};
      const uint32_t bit[4] = {MUON_HOST_W, MUON_HOST_G, MUON_HOST_M, MUON_HOST_O};
      const bool present[4] = {true, true, true, x.O_out != nullptr};
      for (int q = 0; q < 4; ++q) {
        o[q] = SIZE_MAX;
        ld[q] = 0;
        if (!present[q] || !(pl.host_buffers & bit[q])) continue;
        ld[q] = staged_ld(x.cols, es[q]);
        o[q] = off;
        off = align_up(off + (size_t)(x.rows * ld[q] * es[q]), 256);
      }
      c.off.push_back(o);
      c.ld.push_back(ld);
    }
    L.slot_bytes = std::max(L.slot_bytes, align_up(off, 1024));
  }
}

muon_status check_pipeline(const muon_host_pipeline* pl, std::string& why) {
  if (!pl) { why = "pipeline is NULL"; return MUON_ERR_INVALID_ARG; }
  if ((uint32_t)pl->host_buffers & ~kHostBits) { why = "host_buffers has unknown bits"; return MUON_ERR_INVALID_ARG; }
  if (pl->chunk_matrices < 1) { why = "chunk_matrices must be >= 1"; return MUON_ERR_INVALID_ARG; }
  if (pl->slots < 2 || pl->slots > 64) { why = "slots must be in [2, 64]"; return MUON_ERR_INVALID_ARG; }
  if (pl->reserved != 0) { why = "reserved must be 0"; return MUON_ERR_INVALID_ARG; }
  return MUON_OK;
}

}  // namespace

extern "C" {

void muon_config_default(muon_config* c) {
  if (!c) return;
  c->beta = 0.95f;
  c->a = 3.4445f;
  c->b = -4.7750f;
  c->c = 2.0315f;
  c->eps = 1e-7f;
  c->scale_coeff = 0.2f;
  c->ns_iters = 5;
  c->nesterov = 0;
  c->dampening = 0;
  c->mode = MUON_MODE_BF16;
}

const char* muon_status_string(muon_status s) {
  switch (s) {
    case MUON_OK: return "MUON_OK";
    case MUON_ERR_INVALID_ARG: return "MUON_ERR_INVALID_ARG";
    case MUON_ERR_UNSUPPORTED: return "MUON_ERR_UNSUPPORTED";
    case MUON_ERR_WORKSPACE: return "MUON_ERR_WORKSPACE";
    case MUON_ERR_CUDA: return "MUON_ERR_CUDA";
    case MUON_ERR_TIMEOUT: return "MUON_ERR_TIMEOUT";
  }
  return "MUON_ERR_UNKNOWN";
}

muon_status muon_create(const muon_config* cfg, int device, muon_handle* out) {
  if (!out) return MUON_ERR_INVALID_ARG;
  *out = nullptr;
  muon_config c;
  if (cfg) c = *cfg; else muon_config_default(&c);
  std::string why;
  muon_status st = check_config(c, why);
  if (st != MUON_OK) return st;
  if (device < -1) return MUON_ERR_INVALID_ARG;
  muon_handle h = new (std::nothrow) muon_handle_s();
  if (!h) return MUON_ERR_CUDA;
  h->cfg = c;
  if (device >= 0) {
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || device >= count) {
      cudaGetLastError();
      delete h;
      return MUON_ERR_UNSUPPORTED;
    }
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    // kernels are built for sm_103a, whose tcgen05 features are not forward compatible
    if (major != 10 || minor != 3) {
      delete h;
      return MUON_ERR_UNSUPPORTED;
    }
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
      cudaGetLastError();
      delete h;
      return MUON_ERR_CUDA;
    }
    h->encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    h->device = device;
    h->sm_count = sms;
    const char* hook = std::getenv("MUON_GB300_TEST_WITHHOLD_LOADS");
    h->withhold_loads = hook && hook[0] == '1';
  }
  *out = h;
  return MUON_OK;
}

muon_status muon_destroy(muon_handle h) {
  if (!h) return MUON_ERR_INVALID_ARG;
  if (h->device >= 0) {
    DeviceGuard g(h->device);
    for (auto& s : h->recorded)
      for (cudaEvent_t e : s.ev) cudaEventDestroy(e);
    for (cudaEvent_t e : h->pool) cudaEventDestroy(e);
    for (cudaEvent_t e : h->host_events) cudaEventDestroy(e);
    for (cudaStream_t st : h->host_streams)
      if (st) cudaStreamDestroy(st);
    h->plans.clear();   // their graphs, with this device current
    if (h->capture_stream) cudaStreamDestroy(h->capture_stream);
  }
  delete h;
  return MUON_OK;
}

const char* muon_last_error_message(muon_handle h) { return h ? h->err.c_str() : ""; }

int64_t muon_launch_count(muon_handle h) { return h ? h->launches : 0; }

muon_status muon_workspace_size(muon_handle h, const muon_matrix_desc* descs, int n, size_t* bytes) {
  if (!h || !bytes) return MUON_ERR_INVALID_ARG;
  h->err.clear();
  std::string why;
  std::vector<Range> ranges;
  muon_status st = validate(descs, n, why, ranges);
  if (st != MUON_OK) return fail(h, st, why);
  Plan P = build_plan(h->cfg, descs, n);
  *bytes = P.mats.empty() ? 0 : P.bytes;
  return MUON_OK;
}

muon_status muon_set_profiling(muon_handle h, int enable) {
  if (!h) return MUON_ERR_INVALID_ARG;
  if (h->device < 0) return fail(h, MUON_ERR_UNSUPPORTED, "host-only handle");
  h->profiling = enable != 0;
  return MUON_OK;
}

muon_status muon_read_profile(muon_handle h, muon_phase_stats* out) {
  if (!h || !out) return MUON_ERR_INVALID_ARG;
  std::memset(out, 0, sizeof(*out));
  if (h->device < 0) return fail(h, MUON_ERR_UNSUPPORTED, "host-only handle");
  DeviceGuard guard(h->device);
  muon_status st = MUON_OK;
  for (StepEvents& s : h->recorded) {
    const std::vector<cudaEvent_t>& e = s.ev;
    if (cudaEventSynchronize(e.back()) != cudaSuccess) {
      st = fail(h, MUON_ERR_CUDA, std::string("cudaEventSynchronize: ") + cudaGetErrorString(cudaGetLastError()));
      break;
    }
    float t = 0.f;
    // e[0] start, e[1] after momentum+norm, then 3 per iteration, then after apply
    cudaEventElapsedTime(&t, e[0], e[1]);
    out->ms[0] += t;
    out->launches[0] += 2;
    for (int it = 0; it < s.iters; ++it) {
      for (int k = 0; k < 3; ++k) {
        cudaEventElapsedTime(&t, e[1 + 3 * it + k], e[2 + 3 * it + k]);
        out->ms[1 + k] += t;
        out->launches[1 + k] += 1;
      }
    }
    cudaEventElapsedTime(&t, e[e.size() - 2], e[e.size() - 1]);
    out->ms[4] += t;
    out->launches[4] += s.apply_launches;
    out->steps += 1;
  }
  for (StepEvents& s : h->recorded)
    for (cudaEvent_t e : s.ev) h->pool.push_back(e);
  h->recorded.clear();
  return st;
}

muon_status muon_check_status(muon_handle h, void* ws, void* stream) {
  if (!h) return MUON_ERR_INVALID_ARG;
  if (h->device < 0) return fail(h, MUON_ERR_UNSUPPORTED, "host-only handle");
  if (!ws) {
    // the fixed array that muon_step_noalloc uses on this handle's device
    const cudaError_t e = (cudaError_t)muon::static_workspace(h->device, &ws);
    if (e != cudaSuccess)
      return fail(h, MUON_ERR_CUDA, std::string("muon_check_status: fixed workspace: ") + cudaGetErrorString(e));
  }
  DeviceGuard guard(h->device);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // a muon_step_host workspace holds one status word per staging slot
  const int words = ws == h->host_ws ? h->host_slots : 1;
  const size_t stride = ws == h->host_ws ? h->host_slot_bytes : 0;
  uint32_t word = 0;
  cudaError_t e = cudaSuccess;
  for (int k = 0; k < words && e == cudaSuccess; ++k) {
    uint8_t* at = static_cast<uint8_t*>(ws) + (size_t)k * stride;
    uint32_t w = 0;
    e = cudaMemcpyAsync(&w, at, sizeof(w), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemsetAsync(at, 0, sizeof(w), s);
    word |= w;
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(h, MUON_ERR_CUDA, std::string("muon_check_status: ") + cudaGetErrorString(e));
  if (word != 0) return fail(h, MUON_ERR_TIMEOUT, "a kernel gave up a bounded wait, status bits " + std::to_string(word));
  return MUON_OK;
}

muon_status muon_step(muon_handle h, const muon_matrix_desc* descs, int n, void* ws, size_t ws_bytes, void* stream) {
  if (!h) return MUON_ERR_INVALID_ARG;
  h->err.clear();
  // a batch seen before (same descriptor bytes, same workspace) reuses its
  // validated plan, parameter blocks and tensor maps
  StepPlan* plan = find_plan(h, descs, n, ws);
  if (plan) {
    if (ws_bytes < plan->need)
      return fail(h, MUON_ERR_WORKSPACE, "workspace too small: need " + std::to_string(plan->need) + " bytes");
    return run_plan(h, *plan, stream);
  }
  std::string why;
  std::vector<Range> ranges;
  muon_status st = validate(descs, n, why, ranges);
  if (st != MUON_OK) return fail(h, st, why);
  Plan P = build_plan(h->cfg, descs, n);
  if (P.mats.empty()) return MUON_OK;  // nothing to launch
  if (!ws) return fail(h, MUON_ERR_WORKSPACE, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(ws) % 256 != 0) return fail(h, MUON_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (ws_bytes < P.bytes)
    return fail(h, MUON_ERR_WORKSPACE, "workspace too small: need " + std::to_string(P.bytes) + " bytes");
  {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(ws), hi = lo + P.bytes;
    for (const Range& r : ranges)
      if (r.lo < hi && lo < r.hi)
        return fail(h, MUON_ERR_INVALID_ARG,
                    std::string("workspace overlaps desc ") + std::to_string(r.desc) + " " + r.what);
  }
  if (h->device < 0) return fail(h, MUON_ERR_UNSUPPORTED, "host-only handle: create it with a device to run steps");
  std::unique_ptr<StepPlan> fresh(new (std::nothrow) StepPlan);
  if (!fresh) return fail(h, MUON_ERR_CUDA, "host allocation failed");
  if ((st = make_plan(h, P, descs, n, ws, *fresh)) != MUON_OK) return st;
  h->plan_builds += 1;
  if (h->plans.size() >= kPlanCacheEntries) h->plans.pop_back();
  h->plans.insert(h->plans.begin(), std::move(fresh));
  return run_plan(h, *h->plans.front(), stream);
}

int64_t muon_plan_builds(muon_handle h) { return h ? h->plan_builds : 0; }

int64_t muon_graph_launches(muon_handle h) { return h ? h->graph_launches : 0; }

muon_status muon_host_workspace_size(muon_handle h, const muon_matrix_desc* descs, int n,
                                     const muon_host_pipeline* pl, size_t* bytes) {
  if (!h || !bytes) return MUON_ERR_INVALID_ARG;
  h->err.clear();
  std::string why;
  muon_status st = check_pipeline(pl, why);
  if (st != MUON_OK) return fail(h, st, why);
  std::vector<Range> ranges;
  if ((st = validate(descs, n, why, ranges)) != MUON_OK) return fail(h, st, why);
  HostLayout L;
  host_layout(h->cfg, descs, n, *pl, L);
  *bytes = L.chunks.empty() ? 0 : L.slot_bytes * (size_t)std::min<size_t>((size_t)pl->slots, L.chunks.size());
  return MUON_OK;
}

muon_status muon_step_host(muon_handle h, const muon_matrix_desc* descs, int n, const muon_host_pipeline* pl,
                           void* ws, size_t ws_bytes, void* stream) {
  if (!h) return MUON_ERR_INVALID_ARG;
  h->err.clear();
  std::string why;
  muon_status st = check_pipeline(pl, why);
  if (st != MUON_OK) return fail(h, st, why);
  std::vector<Range> ranges;
  if ((st = validate(descs, n, why, ranges)) != MUON_OK) return fail(h, st, why);
  HostLayout L;
  host_layout(h->cfg, descs, n, *pl, L);
  if (L.chunks.empty()) return MUON_OK;
  // no more slots than chunks
  const int S = (int)std::min<size_t>((size_t)pl->slots, L.chunks.size());
  const size_t need = L.slot_bytes * (size_t)S;
  if (!ws) return fail(h, MUON_ERR_WORKSPACE, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(ws) % 256 != 0) return fail(h, MUON_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (ws_bytes < need) return fail(h, MUON_ERR_WORKSPACE, "workspace too small: need " + std::to_string(need) + " bytes");
  {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(ws), hi = lo + need;
    for (const Range& r : ranges)
      if (r.lo < hi && lo < r.hi)
        return fail(h, MUON_ERR_INVALID_ARG,
                    std::string("workspace overlaps desc ") + std::to_string(r.desc) + " " + r.what);
  }
  if (h->device < 0) return fail(h, MUON_ERR_UNSUPPORTED, "host-only handle: create it with a device to run steps");
  DeviceGuard guard(h->device);
  cudaError_t e = cudaSuccess;
  for (cudaStream_t& hs : h->host_streams)
    if (!hs && (e = cudaStreamCreateWithFlags(&hs, cudaStreamNonBlocking)) != cudaSuccess)
      return fail(h, MUON_ERR_CUDA, std::string("cudaStreamCreate: ") + cudaGetErrorString(e));
  // events: start, done, then per slot: loaded, stepped, free
  const size_t nev = 2 + 3 * (size_t)S;
  while (h->host_events.size() < nev) {
    cudaEvent_t ev = nullptr;
    if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess)
      return fail(h, MUON_ERR_CUDA, std::string("cudaEventCreate: ") + cudaGetErrorString(e));
    h->host_events.push_back(ev);
  }
  cudaStream_t s_in = h->host_streams[0], s_run = h->host_streams[1], s_out = h->host_streams[2];
  cudaEvent_t ev_start = h->host_events[0], ev_done = h->host_events[1];
  auto loaded = [&](int k) { return h->host_events[2 + k]; };
  auto stepped = [&](int k) { return h->host_events[2 + S + k]; };
  auto freed = [&](int k) { return h->host_events[2 + 2 * S + k]; };
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  auto ck = [&](cudaError_t r, const char* what) -> bool {
    if (r == cudaSuccess) return true;
    e = r;
    h->err = std::string("muon_step_host: ") + what + ": " + cudaGetErrorString(r);
    return false;
  };
  if (!ck(cudaEventRecord(ev_start, cs), "cudaEventRecord")) return MUON_ERR_CUDA;
  for (cudaStream_t q : {s_in, s_run, s_out})
    if (!ck(cudaStreamWaitEvent(q, ev_start, 0), "cudaStreamWaitEvent")) return MUON_ERR_CUDA;
  uint8_t* base = static_cast<uint8_t*>(ws);
  std::vector<muon_matrix_desc> dd;
  for (size_t c = 0; c < L.chunks.size(); ++c) {
    const HostChunk& C = L.chunks[c];
    const int slot = (int)(c % (size_t)S);
    uint8_t* sb = base + (size_t)slot * L.slot_bytes;
    if (c >= (size_t)S && !ck(cudaStreamWaitEvent(s_in, freed(slot), 0), "cudaStreamWaitEvent")) return MUON_ERR_CUDA;
    dd.clear();
    for (size_t k = 0; k < C.mats.size(); ++k) {
      const muon_matrix_desc& x = descs[C.mats[k]];
      muon_matrix_desc y = x;
      const int64_t wes = x.w_dtype == MUON_BF16 ? 2 : 4;
      const size_t rowb[4] = {(size_t)(x.cols * wes), (size_t)x.cols * 4, (size_t)x.cols * 4, (size_t)x.cols * 4};
      const void* src[4] = {x.W, x.G, x.M, x.O_out};
      const int64_t sld[4] = {x.ldw, x.ldg, x.ldm, x.ldo};
      const int64_t es[4] = {wes, 4, 4, 4};
      void* dst[4] = {nullptr, nullptr, nullptr, nullptr};
      for (int q = 0; q < 4; ++q) {
        if (C.off[k][q] == SIZE_MAX) continue;
        dst[q] = sb + C.off[k][q];
        // inputs: W, G, M (O_out is written only)
        if (q < 3 && !ck(cudaMemcpy2DAsync(dst[q], (size_t)(C.ld[k][q] * es[q]), src[q], (size_t)(sld[q] * es[q]),
                                           rowb[q], (size_t)x.rows, cudaMemcpyHostToDevice, s_in),
                         "cudaMemcpy2DAsync (in)"))
          return MUON_ERR_CUDA;
      }
      if (dst[0]) { y.W = dst[0]; y.ldw = C.ld[k][0]; }
      if (dst[1]) { y.G = static_cast<const float*>(dst[1]); y.ldg = C.ld[k][1]; }
      if (dst[2]) { y.M = static_cast<float*>(dst[2]); y.ldm = C.ld[k][2]; }
      if (dst[3]) { y.O_out = static_cast<float*>(dst[3]); y.ldo = C.ld[k][3]; }
      dd.push_back(y);
    }
    if (!ck(cudaEventRecord(loaded(slot), s_in), "cudaEventRecord") ||
        !ck(cudaStreamWaitEvent(s_run, loaded(slot), 0), "cudaStreamWaitEvent"))
      return MUON_ERR_CUDA;
    if ((st = muon_step(h, dd.data(), (int)dd.size(), sb + C.ws_off, C.ws_bytes, s_run)) != MUON_OK) return st;
    if (!ck(cudaEventRecord(stepped(slot), s_run), "cudaEventRecord") ||
        !ck(cudaStreamWaitEvent(s_out, stepped(slot), 0), "cudaStreamWaitEvent"))
      return MUON_ERR_CUDA;
    for (size_t k = 0; k < C.mats.size(); ++k) {
      const muon_matrix_desc& x = descs[C.mats[k]];
      const int64_t wes = x.w_dtype == MUON_BF16 ? 2 : 4;
      // outputs: W, M, O_out
      const int qs[3] = {0, 2, 3};
      void* hdst[4] = {x.W, nullptr, x.M, x.O_out};
      const int64_t hld[4] = {x.ldw, 0, x.ldm, x.ldo};
      const int64_t es[4] = {wes, 4, 4, 4};
      for (int q : qs) {
        if (C.off[k][q] == SIZE_MAX) continue;
        if (!ck(cudaMemcpy2DAsync(hdst[q], (size_t)(hld[q] * es[q]), sb + C.off[k][q], (size_t)(C.ld[k][q] * es[q]),
                                  (size_t)(x.cols * es[q]), (size_t)x.rows, cudaMemcpyDeviceToHost, s_out),
                "cudaMemcpy2DAsync (out)"))
          return MUON_ERR_CUDA;
      }
    }
    if (!ck(cudaEventRecord(freed(slot), s_out), "cudaEventRecord")) return MUON_ERR_CUDA;
  }
  if (!ck(cudaEventRecord(ev_done, s_out), "cudaEventRecord") || !ck(cudaStreamWaitEvent(cs, ev_done, 0), "cudaStreamWaitEvent"))
    return MUON_ERR_CUDA;
  h->host_ws = ws;
  h->host_slot_bytes = L.slot_bytes;
  h->host_slots = S;
  return MUON_OK;
}

}  // extern "C"

namespace muon {

int handle_device(::muon_handle_s* h) { return h ? h->device : -1; }

void set_handle_error(::muon_handle_s* h, const std::string& msg) {
  if (h) h->err = msg;
}

}  // namespace muon
