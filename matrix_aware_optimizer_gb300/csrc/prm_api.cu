// C ABI and host engine of libprm: argument checks, the planner (launch
// groups by shape, NS5 groups by wide orientation, MuonBP block views,
// workspace layout) and the launch sequence of one step on the caller's
// stream. Method: "Scaling Muon for Diffusion Transformers" (PaperDaily
// walkthrough, section "Periodic Row-wise Muon", Fig. 3 update rule) and
// "MuonBP: Faster Muon via Block-Periodic Orthogonalization" (abstract).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <new>
#include <string>
#include <tuple>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "internal.h"
#include "prm.h"

namespace prm {
namespace {

// NVTX range over the host-side enqueue of one kernel family (or one step),
// named as the timer's families are, so that profilers can select launches
// by range (e.g. ncu --nvtx --nvtx-include "prm_step/ns_combine/"). A no-op
// unless a tool is attached.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

const char* const kFamilyNames[PRM_FAMILY_COUNT] = {"rownorm_wide", "rownorm_tall", "ns_prep",
                                                    "ns_gram",      "ns_poly",      "ns_combine",
                                                    "ns_sym",       "ns_small"};

constexpr float NS_EPS = 1e-7f;  // added to ||M||_F before NS5 pre-normalisation
constexpr float DEFAULT_COEFFS[3] = {3.4445f, -4.7750f, 2.0315f};
constexpr int NS_STEPS = 5;

thread_local std::string g_create_error;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int64_t round8(int64_t x) { return (x + 7) / 8 * 8; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Views of one exact shape and orientation, launched together.
struct LaunchSet {
  int64_t rows = 0, cols = 0;
  bool bf16 = false;
  bool vec_ok = true;
  std::vector<View> views;
  View* d_views = nullptr;
  // tall RowNorm: the one-launch form (aligned views within its size limits)
  // or three launches; scratch offsets relative to the workspace base
  bool fused = false;
  bool ring = false;  // the one-launch form with the TMA ring (needs tall_ring_ok)
  CUtensorMap* d_maps = nullptr;  // ring: per view the tensor maps of M, G and W (device)
  size_t off_partials = 0, off_inv = 0, off_flags = 0;
};

// Maps of one Gram-route Y buffer: per matrix Q and T side by side (r rows,
// pitch 2 ldr fp16 elements, T starting at column ldr).
struct YMaps {
  NsMaps q, t;
};

// Same wide-orientation shape r x c: one batch for the GRAM and COMBINE
// GEMMs. Direct route: its r x r Gram / polynomial matrices live in the
// r-class arrays. Gram route (c >= 2 r): its own C and P arrays and two Y
// buffers.
struct NsGroup {
  int64_t r = 0, c = 0, ldc = 0, ldr = 0;
  int count = 0;
  int rclass = -1;        // direct route: index of its r-class
  bool gram = false;      // Gram route
  bool small = false;     // r < NS_SMALL_R: fp32 rounds on CUDA cores (ns_small.cu), no tensor maps
  int64_t base_slot = 0;  // first slot of this group inside its r-class arrays
  int64_t slots = 0;      // Frobenius partial slots per matrix
  std::vector<LaunchSet> sets;
  size_t off_x0 = 0, off_x1 = 0, off_scale = 0, off_partials = 0;
  size_t off_c = 0, off_p = 0, off_ya = 0, off_yb = 0;  // Gram route
  size_t off_sx = 0, off_spart = 0, off_sp = 0;          // small: X, Gram partials, P (fp32)
  // tensor maps for the bound workspace
  const void* maps_base = nullptr;
  NsMaps mx0{}, mx1{};
  SymMaps mb{};  // direct: this group's slice of the r-class B array (P; COMBINE operand)
  SymMaps ma{};  // direct: this group's slice of the r-class A array (P when POLY is skipped, c = 0)
  SymMaps mc{}, mp{};  // Gram route: C and P
  YMaps ya{}, yb{};    // Gram route
  View* d_slot_views = nullptr;  // device: the group's views by slot (the last COMBINE applies D through them)
};

// All matrices with the same short side r: their A = X X^T and
// B = b A + c A A sit in one batch, so POLY runs as one launch for the class.
struct NsRClass {
  int64_t r = 0, ldr = 0;
  int count = 0;
  size_t off_a = 0, off_b = 0;
  const void* maps_base = nullptr;
  SymMaps ma{};  // the r-class A array (GRAM output C, POLY operand)
  SymMaps mb{};  // the r-class B array (POLY output P)
};

// Every group's buffers are live at once: the five NS5 rounds of all groups
// run in lockstep (GRAM per group, POLY per r-class, COMBINE per group).
struct NsPlan {
  std::vector<NsGroup> groups;
  std::vector<NsRClass> rclasses;
  size_t bytes = 0;
};

struct RowNormPlan {
  std::vector<LaunchSet> wide, tall;
  size_t bytes = 0;
};

void free_sets(std::vector<LaunchSet>& sets) {
  for (auto& s : sets) {
    if (s.d_views) cudaFree(s.d_views);
    if (s.d_maps) cudaFree(s.d_maps);
    s.d_views = nullptr;
    s.d_maps = nullptr;
  }
}

// Tensor maps of a ring-form tall launch set: per view M (fp32), G (fp32 or
// bf16) and W (fp32), boxes of the ring kernel's stage shape, copied to
// device memory (the kernel reads them from there).
cudaError_t upload_ring_maps(LaunchSet& s) {
  std::vector<CUtensorMap> maps(3 * s.views.size());
  const uint32_t bc = static_cast<uint32_t>(tall_ring_box_cols()), br = static_cast<uint32_t>(tall_ring_box_rows());
  for (size_t i = 0; i < s.views.size(); ++i) {
    const View& v = s.views[i];
    if (encode_rows_2d(&maps[3 * i + 0], v.M, false, v.rows, v.cols, v.ld, bc, br) != 0 ||
        encode_rows_2d(&maps[3 * i + 1], v.G, s.bf16, v.rows, v.cols, v.ld, bc, br) != 0 ||
        encode_rows_2d(&maps[3 * i + 2], v.W, false, v.rows, v.cols, v.ld, bc, br) != 0)
      return cudaErrorInvalidValue;
  }
  const size_t bytes = maps.size() * sizeof(CUtensorMap);
  cudaError_t e = cudaMalloc(reinterpret_cast<void**>(&s.d_maps), bytes);
  if (e != cudaSuccess) return e;
  return cudaMemcpy(s.d_maps, maps.data(), bytes, cudaMemcpyHostToDevice);
}

void free_plan(NsPlan& p) {
  for (auto& g : p.groups) {
    free_sets(g.sets);
    if (g.d_slot_views) cudaFree(g.d_slot_views);
    g.d_slot_views = nullptr;
  }
  p.groups.clear();
  p.bytes = 0;
}

cudaError_t upload_sets(std::vector<LaunchSet>& sets) {
  for (auto& s : sets) {
    if (s.views.empty()) continue;
    const size_t b = s.views.size() * sizeof(View);
    cudaError_t e = cudaMalloc(reinterpret_cast<void**>(&s.d_views), b);
    if (e != cudaSuccess) return e;
    if ((e = cudaMemcpy(s.d_views, s.views.data(), b, cudaMemcpyHostToDevice)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Uploads a group's launch tables: the per-shape sets (prep kernels) and the
// slot-indexed view table through which the last COMBINE round applies D.
cudaError_t upload_group(NsGroup& g) {
  cudaError_t e = upload_sets(g.sets);
  if (e != cudaSuccess) return e;
  std::vector<View> by_slot(static_cast<size_t>(g.count));
  for (const auto& st : g.sets)
    for (const View& v : st.views) by_slot[static_cast<size_t>(v.slot)] = v;
  const size_t bytes = by_slot.size() * sizeof(View);
  if ((e = cudaMalloc(reinterpret_cast<void**>(&g.d_slot_views), bytes)) != cudaSuccess) return e;
  return cudaMemcpy(g.d_slot_views, by_slot.data(), bytes, cudaMemcpyHostToDevice);
}

bool view_vec_ok(const View& v) {
  const bool base = (v.cols % 4 == 0) && (v.ld % 4 == 0);
  const bool ptrs = (v.W == nullptr || aligned16(v.W)) && aligned16(v.M) && (v.out == nullptr || aligned16(v.out));
  const bool g = v.G == nullptr || (v.grad_bf16 ? (reinterpret_cast<uintptr_t>(v.G) & 7u) == 0 : aligned16(v.G));
  return base && ptrs && g;
}

// Share of a symmetric r x r output's dense products that the GEMM kernels
// execute: the upper-triangle 256 x 256 super-blocks, nb (nb + 1) / 2 of nb^2
// (36 / 64 at r = 2048).
double sym_share(int64_t r) {
  const double nb = static_cast<double>((r + 255) / 256);
  return (nb + 1.0) / (2.0 * nb);
}

// Whether the Gram route (see run_ns) pays for an r x c group: its executed
// work for the five default rounds (legs of three and two) against the
// direct rounds', in units of r^3 with rho = c / r and f the executed share
// of a symmetric product (upper 256 x 256 super-blocks of nb x nb):
//   Gram   4 rho f + 4 rho + 28 f     direct  10 rho f + 10 f + 10 rho
// It is taken when at least 10 % cheaper: from c = 1.37 r at r = 2048 (for
// square matrices it would cost 4 % more), from c = 1.9 r at r <= 256.
bool gram_route_pays(int64_t r, int64_t c) {
  const double nb = static_cast<double>((r + 255) / 256);
  const double f = (nb + 1.0) / (2.0 * nb), rho = static_cast<double>(c) / static_cast<double>(r);
  const double gram = 4.0 * rho * f + 4.0 * rho + 28.0 * f;
  const double direct = 10.0 * rho * f + 10.0 * f + 10.0 * rho;
  return gram <= 0.9 * direct;
}

// Groups views for the NS5 branch and lays out the shared group workspace.
// `form` PRM_NS_FORM_AUTO puts the groups for which gram_route_pays on the
// Gram route.
void build_ns_plan(const std::vector<View>& views, NsPlan& plan, int form) {
  std::map<std::pair<int64_t, int64_t>, size_t> index;
  for (const View& v0 : views) {
    const bool tall = v0.rows > v0.cols;
    const int64_t r = tall ? v0.cols : v0.rows, c = tall ? v0.rows : v0.cols;
    auto key = std::make_pair(r, c);
    auto it = index.find(key);
    if (it == index.end()) {
      NsGroup g;
      g.r = r;
      g.c = c;
      g.ldc = round8(c);
      g.ldr = round8(r);
      plan.groups.push_back(std::move(g));
      it = index.emplace(key, plan.groups.size() - 1).first;
    }
    NsGroup& g = plan.groups[it->second];
    View v = v0;
    v.slot = g.count++;
    LaunchSet* set = nullptr;
    for (auto& s : g.sets)
      if (s.rows == v.rows && s.cols == v.cols && s.bf16 == (v.grad_bf16 != 0)) set = &s;
    if (set == nullptr) {
      g.sets.emplace_back();
      set = &g.sets.back();
      set->rows = v.rows;
      set->cols = v.cols;
      set->bf16 = v.grad_bf16 != 0;
    }
    set->vec_ok = set->vec_ok && view_vec_ok(v);
    set->views.push_back(v);
  }
  size_t off = 0;
  std::map<int64_t, int> rindex;
  for (auto& g : plan.groups) {
    if (g.r < NS_SMALL_R) {
      // short side below 64: fp32 rounds on CUDA cores, own buffers only
      g.small = true;
      const int64_t tiles = ns_small_tiles(g.c), chunks = ns_small_chunks(g.c);
      g.off_sx = off;
      off += align_up(static_cast<size_t>(g.count) * tiles * g.r * NS_SMALL_TC * 4, 256);
      g.off_spart = off;
      off += align_up(static_cast<size_t>(g.count) * chunks * (g.r * (g.r + 1) / 2) * 4, 256);
      g.off_sp = off;
      off += align_up(static_cast<size_t>(g.count) * g.r * g.r * 4, 256);
      continue;
    }
    g.slots = prep_slots(g.sets.front().rows, g.sets.front().cols);
    for (auto& s : g.sets) g.slots = std::max(g.slots, prep_slots(s.rows, s.cols));
    const size_t xb = align_up(static_cast<size_t>(g.count) * g.r * g.ldc * 2, 256);
    g.off_x0 = off;
    off += xb;
    g.off_x1 = off;
    off += xb;
    g.off_scale = off;
    off += align_up(static_cast<size_t>(g.count) * 4, 256);
    g.off_partials = off;
    off += align_up(static_cast<size_t>(g.count) * g.slots * 4, 256);
    g.gram = form == PRM_NS_FORM_AUTO && gram_route_pays(g.r, g.c);
    if (g.gram) {
      const size_t cb = align_up(static_cast<size_t>(g.count) * g.r * g.ldr * 2, 256);
      const size_t yb = align_up(static_cast<size_t>(g.count) * g.r * 2 * g.ldr * 2, 256);
      g.off_c = off;
      off += cb;
      g.off_p = off;
      off += cb;
      g.off_ya = off;
      off += yb;
      g.off_yb = off;
      off += yb;
      continue;
    }
    auto it = rindex.find(g.r);
    if (it == rindex.end()) {
      NsRClass rc;
      rc.r = g.r;
      rc.ldr = g.ldr;
      plan.rclasses.push_back(rc);
      it = rindex.emplace(g.r, static_cast<int>(plan.rclasses.size()) - 1).first;
    }
    g.rclass = it->second;
    g.base_slot = plan.rclasses[g.rclass].count;
    plan.rclasses[g.rclass].count += g.count;
  }
  for (auto& rc : plan.rclasses) {
    const size_t ab = align_up(static_cast<size_t>(rc.count) * rc.r * rc.ldr * 2, 256);
    rc.off_a = off;
    off += ab;
    rc.off_b = off;
    off += ab;
  }
  plan.bytes = off;
}

// Automatic workspace policy (limit 0): a plan whose buffers would exceed
// AUTO_SPLIT_ABOVE runs as sequential sub-plans of at most AUTO_SUBPLAN_BYTES.
// Measured on the 15B-shaped set (75 GB as one plan): 3 / 10 / 40 GB
// sub-plans run the K = 3 cycle 10 / 8.5 / 4 % faster than one plan, the SM
// clock under the power cap rising as the per-launch working set shrinks;
// on the 1.3B-shaped set (6 GB) splitting gains nothing, so plans below the
// threshold stay whole (all groups in lockstep, POLY once per r-class).
constexpr size_t AUTO_SPLIT_ABOVE = size_t(16) << 30;
constexpr size_t AUTO_SUBPLAN_BYTES = size_t(4) << 30;

// Splits the views into sequential sub-plans whose workspace fits `limit`
// bytes (SIZE_MAX: one plan for everything; 0: the automatic policy above).
// Views are taken in (r, c) order so that same-shape matrices stay together;
// a sub-plan holds at least one view.
void build_ns_subplans(const std::vector<View>& views, size_t limit, int form, std::vector<NsPlan>& out) {
  out.clear();
  if (views.empty()) return;
  if (limit == 0 || limit == SIZE_MAX) {
    out.emplace_back();
    build_ns_plan(views, out.back(), form);
    if (limit == SIZE_MAX || out.back().bytes <= AUTO_SPLIT_ABOVE) return;
    out.clear();
    limit = AUTO_SUBPLAN_BYTES;
  }
  std::vector<View> sorted = views;
  std::stable_sort(sorted.begin(), sorted.end(), [](const View& x, const View& y) {
    const int64_t rx = std::min(x.rows, x.cols), cx = std::max(x.rows, x.cols);
    const int64_t ry = std::min(y.rows, y.cols), cy = std::max(y.rows, y.cols);
    return rx != ry ? rx < ry : cx < cy;
  });
  std::vector<View> cur;
  for (const View& v : sorted) {
    cur.push_back(v);
    NsPlan trial;
    build_ns_plan(cur, trial, form);
    if (trial.bytes > limit && cur.size() > 1) {
      cur.pop_back();
      out.emplace_back();
      build_ns_plan(cur, out.back(), form);
      cur.assign(1, v);
    }
  }
  out.emplace_back();
  build_ns_plan(cur, out.back(), form);
}

size_t plans_bytes(const std::vector<NsPlan>& plans) {
  size_t b = 0;
  for (const auto& p : plans) b = std::max(b, p.bytes);
  return b;
}

}  // namespace
}  // namespace prm

using namespace prm;

// Event-pair records of kernel families (prm_profile).
struct Profiler {
  struct Rec {
    int family;
    size_t ev;       // index of the start event; stop is ev + 1
    int kernels;
    double work;
  };
  bool on = false;
  std::vector<cudaEvent_t> pool;
  std::vector<Rec> recs;
  size_t used = 0;

  cudaEvent_t next() {
    if (used == pool.size()) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
      pool.push_back(e);
    }
    return pool[used++];
  }
  // Returns the start-event index, or SIZE_MAX when not recording.
  size_t begin(cudaStream_t st) {
    if (!on) return SIZE_MAX;
    const size_t i = used;
    cudaEvent_t a = next(), b = next();
    if (a == nullptr || b == nullptr) return SIZE_MAX;
    cudaEventRecord(a, st);
    return i;
  }
  void end(size_t i, int family, int kernels, double work, cudaStream_t st) {
    if (i == SIZE_MAX) return;
    cudaEventRecord(pool[i + 1], st);
    recs.push_back(Rec{family, i, kernels, work});
  }
  void reset() {
    recs.clear();
    used = 0;
  }
  ~Profiler() {
    for (auto e : pool) cudaEventDestroy(e);
  }
};

struct prm_ctx {
  Profiler prof;
  int device = 0;
  int num_sms = 0;
  std::string err;
  int* d_err = nullptr;  // device error word of the bounded waits
  int count = 0;
  int blocks = 0;
  RowNormPlan rn;
  std::vector<NsPlan> ns_full, ns_blocks;  // sequential sub-plans (one unless a workspace cap splits them)
  size_t ws_limit = 0;                     // prm_set_workspace_limit; 0 = automatic, SIZE_MAX = no cap
  int ns_form = PRM_NS_FORM_AUTO;          // prm_set_ns_form
  struct {
    int stripe = -1;                       // prm_debug_withhold_tall_norms: for the next RowNorm step only
    uint64_t wait_ns = 0;
  } withhold;
  std::vector<View> full;                  // registered matrices, in registration order
  struct {
    bool valid = false;
    int64_t t = 0;
    int K = 1, mode = PRM_MODE_PRMUON;
    float eps = 0.f;
    float coeffs[3] = {0.f, 0.f, 0.f};
  } last;                                  // the most recent prm_step (prm_debug_last_direction)
  bool registered = false;
  void* ws = nullptr;
  size_t ws_bytes = 0;
};

namespace {

int fail(prm_ctx* c, int code, const std::string& msg) {
  if (c)
    c->err = msg;
  else
    g_create_error = msg;
  return code;
}

int cuda_fail(prm_ctx* c, cudaError_t e, const char* what) {
  return fail(c, PRM_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

// Makes the context's device current for the duration of a call.
struct DeviceGuard {
  int prev = -1;
  bool changed = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) {
      changed = cudaSetDevice(dev) == cudaSuccess;
    }
  }
  ~DeviceGuard() {
    if (changed) cudaSetDevice(prev);
  }
};

void clear_registration(prm_ctx* c) {
  free_sets(c->rn.wide);
  free_sets(c->rn.tall);
  c->rn.wide.clear();
  c->rn.tall.clear();
  c->rn.bytes = 0;
  for (auto& p : c->ns_full) free_plan(p);
  for (auto& p : c->ns_blocks) free_plan(p);
  c->ns_full.clear();
  c->ns_blocks.clear();
  c->full.clear();
  c->last.valid = false;
  c->count = 0;
  c->blocks = 0;
  c->registered = false;
}

// MuonBP blocks of one matrix: P contiguous pieces along the long side, the
// last one taking the remainder ("MuonBP: Faster Muon via Block-Periodic
// Orthogonalization", abstract: each device orthogonalises its own block).
void make_blocks(const View& v, int P, std::vector<View>& out) {
  const bool wide = v.rows <= v.cols;
  const int64_t L = wide ? v.cols : v.rows;
  const int64_t base = L / P;
  for (int k = 0; k < P; ++k) {
    const int64_t lo = k * base, hi = (k == P - 1) ? L : lo + base;
    const int64_t off = wide ? lo : lo * v.ld;
    View b = v;
    b.W = v.W + off;
    b.M = v.M + off;
    b.G = v.grad_bf16 ? static_cast<const void*>(static_cast<const uint16_t*>(v.G) + off)
                      : static_cast<const void*>(static_cast<const float*>(v.G) + off);
    if (wide)
      b.cols = hi - lo;
    else
      b.rows = hi - lo;
    out.push_back(b);
  }
}

void add_to_sets(std::vector<LaunchSet>& sets, const View& v) {
  for (auto& s : sets) {
    if (s.rows == v.rows && s.cols == v.cols && s.bf16 == (v.grad_bf16 != 0)) {
      s.vec_ok = s.vec_ok && view_vec_ok(v);
      s.views.push_back(v);
      return;
    }
  }
  LaunchSet s;
  s.rows = v.rows;
  s.cols = v.cols;
  s.bf16 = v.grad_bf16 != 0;
  s.vec_ok = view_vec_ok(v);
  s.views.push_back(v);
  sets.push_back(std::move(s));
}

int bind_maps(prm_ctx* c, NsPlan& plan, void* base) {
  char* b = static_cast<char*>(base);
  for (auto& rc : plan.rclasses) {
    if (rc.maps_base == base) continue;
    int e = encode_sym_maps(&rc.ma, b + rc.off_a, rc.count, rc.r, rc.ldr);
    if (e == 0) e = encode_sym_maps(&rc.mb, b + rc.off_b, rc.count, rc.r, rc.ldr);
    if (e != 0) return fail(c, PRM_ERR_CUDA, "cuTensorMapEncodeTiled failed (code " + std::to_string(e) + ")");
    rc.maps_base = base;
  }
  for (auto& g : plan.groups) {
    if (g.small || g.maps_base == base) continue;
    int e = encode_x_maps(&g.mx0, b + g.off_x0, g.count, g.r, g.c, g.ldc);
    if (e == 0) e = encode_x_maps(&g.mx1, b + g.off_x1, g.count, g.r, g.c, g.ldc);
    if (g.gram) {
      if (e == 0) e = encode_sym_maps(&g.mc, b + g.off_c, g.count, g.r, g.ldr);
      if (e == 0) e = encode_sym_maps(&g.mp, b + g.off_p, g.count, g.r, g.ldr);
      for (auto yy : {std::make_pair(&g.ya, g.off_ya), std::make_pair(&g.yb, g.off_yb)}) {
        char* y = b + yy.second;
        const int64_t ld = 2 * g.ldr;
        if (e == 0) e = encode_x_maps(&yy.first->q, y, g.count, g.r, g.r, ld);
        if (e == 0) e = encode_x_maps(&yy.first->t, y + g.ldr * 2, g.count, g.r, g.r, ld);
      }
    } else {
      const NsRClass& rc = plan.rclasses[g.rclass];
      const size_t slice = static_cast<size_t>(g.base_slot) * g.r * g.ldr * 2;
      if (e == 0) e = encode_sym_maps(&g.mb, b + rc.off_b + slice, g.count, g.r, g.ldr);
      if (e == 0) e = encode_sym_maps(&g.ma, b + rc.off_a + slice, g.count, g.r, g.ldr);
    }
    if (e != 0) return fail(c, PRM_ERR_CUDA, "cuTensorMapEncodeTiled failed (code " + std::to_string(e) + ")");
    g.maps_base = base;
  }
  return PRM_OK;
}

// NS5 of one group with a short side below NS_SMALL_R, all in fp32 on CUDA
// cores (ns_small.cu): momentum and Gram partials, then per round P from the
// partials and X' = P X over column chunks; the last round applies the update.
int run_ns_small(prm_ctx* c, NsGroup& g, char* b, bool update_momentum, float beta, float decay, float eta,
                 const float coeffs[3], int steps, cudaStream_t stream) {
  NsSmallArgs a;
  a.r = static_cast<int>(g.r);
  a.c = g.c;
  a.tiles = ns_small_tiles(g.c);
  a.chunks = ns_small_chunks(g.c);
  a.X = reinterpret_cast<float*>(b + g.off_sx);
  a.partials = reinterpret_cast<float*>(b + g.off_spart);
  a.P = reinterpret_cast<float*>(b + g.off_sp);
  const double r = static_cast<double>(g.r), cw = static_cast<double>(g.c);
  // executed flops per matrix: Gram pairs r (r + 1) c per round, P X 2 r^2 c, P 2 r^3
  const double flops = g.count * steps * (r * (r + 1) * cw + 2 * r * r * cw + 2 * r * r * r);
  NvtxRange nr(kFamilyNames[PRM_FAMILY_NS_SMALL]);
  const size_t ev = c->prof.begin(stream);
  cudaError_t e;
  for (auto& s : g.sets) {
    e = launch_ns_small_prep(a, s.d_views, static_cast<int>(s.views.size()), s.rows > s.cols, s.bf16,
                             update_momentum, beta, stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "small NS5 prep launch");
  }
  for (int it = 0; it < steps; ++it) {
    if ((e = launch_ns_small_poly(a, g.count, it == 0, coeffs, NS_EPS, stream)) != cudaSuccess)
      return cuda_fail(c, e, "small NS5 polynomial launch");
    for (auto& s : g.sets) {
      e = launch_ns_small_combine(a, s.d_views, static_cast<int>(s.views.size()), s.rows > s.cols, it == 0,
                                  it == steps - 1, decay, eta, stream);
      if (e != cudaSuccess) return cuda_fail(c, e, "small NS5 combine launch");
    }
  }
  c->prof.end(ev, PRM_FAMILY_NS_SMALL, static_cast<int>(g.sets.size()) * (steps + 1) + steps, flops, stream);
  return PRM_OK;
}

// One NS5 refresh over every group of `plan`: prep (momentum + pack + norm
// partials), scale, five GRAM / POLY / COMBINE rounds, apply. Groups with a
// short side below NS_SMALL_R run on their own path (run_ns_small) first.
int run_ns(prm_ctx* c, NsPlan& plan, void* base, bool update_momentum, float beta, float decay, float eta,
           const float coeffs[3], int steps, cudaStream_t stream) {
  char* b = static_cast<char*>(base);
  int rc = bind_maps(c, plan, base);
  if (rc != PRM_OK) return rc;
  cudaError_t e;
  for (auto& g : plan.groups) {
    if (!g.small) continue;
    rc = run_ns_small(c, g, b, update_momentum, beta, decay, eta, coeffs, steps, stream);
    if (rc != PRM_OK) return rc;
  }
  // 1. momentum update, bf16 pack (transposed for tall views), Frobenius norms
  for (auto& g : plan.groups) {
    if (g.small) continue;
    float* scale = reinterpret_cast<float*>(b + g.off_scale);
    float* partials = reinterpret_cast<float*>(b + g.off_partials);
    uint16_t* x0 = reinterpret_cast<uint16_t*>(b + g.off_x0);
    double prep_bytes = 0;
    for (auto& s : g.sets)
      prep_bytes += static_cast<double>(s.views.size()) * s.rows * s.cols *
                    (update_momentum ? (s.bf16 ? 12.0 : 14.0) : 6.0);
    NvtxRange nr(kFamilyNames[PRM_FAMILY_NS_PREP]);
    const size_t ev = c->prof.begin(stream);
    // Views of one group may fill different numbers of partial slots (wide:
    // one per row; tall: one per 64x64 tile): unused slots must read as zero.
    if ((e = cudaMemsetAsync(partials, 0, static_cast<size_t>(g.count) * g.slots * sizeof(float), stream)) !=
        cudaSuccess)
      return cuda_fail(c, e, "partials reset");
    for (auto& s : g.sets) {
      e = launch_prep(s.d_views, static_cast<int>(s.views.size()), s.rows, s.cols, s.vec_ok, s.bf16,
                      update_momentum, beta, x0, g.ldc, g.r * g.ldc, partials, g.slots, stream);
      if (e != cudaSuccess) return cuda_fail(c, e, "prep launch");
    }
    if ((e = launch_norm_finish(partials, g.slots, scale, g.count, NS_EPS, stream)) != cudaSuccess)
      return cuda_fail(c, e, "norm launch");
    c->prof.end(ev, PRM_FAMILY_NS_PREP, static_cast<int>(g.sets.size()) + 1, prep_bytes, stream);
  }
  // P = a I + b A + c A A as a completed square (see ns5_gemm.cu): GRAM
  // writes C = sqrt|c| A + sgn(c) b / (2 sqrt|c|) I, POLY P = sgn(c) C C +
  // (a - b^2 / (4c)) I; for c = 0 GRAM writes P = b A + a I and POLY is skipped.
  const double ca = coeffs[0], cb = coeffs[1], cc = coeffs[2];
  const bool square = cc != 0.0;
  const double root = square ? std::sqrt(std::fabs(cc)) : 0.0, sg = cc > 0.0 ? 1.0 : -1.0;
  const float gram_gain = static_cast<float>(square ? root : cb);
  const float gram_diag = static_cast<float>(square ? sg * cb / (2.0 * root) : ca);
  const float poly_gain = static_cast<float>(sg);
  const float poly_diag = static_cast<float>(square ? ca - cb * cb / (4.0 * cc) : 0.0);
  GemmEpilogue epi;
  epi.decay = decay;
  epi.eta = eta;
  epi.err = c->d_err;
  epi.num_sms = c->num_sms;
  auto launches_for = [](size_t segments) {
    return static_cast<int>((segments + GEMM_MAX_SEGMENTS - 1) / GEMM_MAX_SEGMENTS);
  };
  int nlaunch = 0;
  auto run = [&](GemmKind kind, const std::vector<GemmSegSpec>& specs, int family, double flops,
                 const char* what) -> int {
    if (specs.empty()) return PRM_OK;
    // Alternate launches visit each segment's matrices last to first, so
    // that a launch starts on the matrices whose inputs the previous launch
    // wrote last and L2 may still hold (about 0.5 % off the GEMM launches).
    epi.reverse = (nlaunch++ & 1) != 0;
    NvtxRange nr(kFamilyNames[family]);
    const size_t ev = c->prof.begin(stream);
    const cudaError_t err = launch_gemm(kind, specs.data(), static_cast<int>(specs.size()), epi, stream);
    if (err != cudaSuccess) return cuda_fail(c, err, what);
    c->prof.end(ev, family, launches_for(specs.size()), flops, stream);
    return PRM_OK;
  };
  // Gram route: the rounds run in legs of at most three. A leg starts from an
  // explicit X_s (X_0, or the previous leg's result) and iterates r x r
  // matrices only: with A_0 = X_s X_s^T and Q_j = P_j ... P_1 (so that
  // X_j = Q_j X_s and A_j = Q_{j-1} A_0 Q_{j-1}^T), round j computes
  //   C_j = sqrt|c| T_{j-1} Q_{j-1}^T / S + sgn(c) b / (2 sqrt|c|) I
  //         (T = S Q A_0; round 1: C_1 from X_s X_s^T directly),
  //   P_j = sgn(c) C_j C_j + (a - b^2 / (4c)) I,
  //   Q_j = P_j Q_{j-1},  T_j = P_j T_{j-1}   (Q_0 = I, T_0 = S A_0),
  // and the leg ends with X_e = Q_L X_s. Every P, Q and T is a polynomial in
  // A_0, so all of them are symmetric and commute: P Q = P Q^T, and the
  // updates run on the symmetric-output kernel (upper super-blocks, the rest
  // mirrored), like C. Round 1's GRAM also writes S A_0 (its second output)
  // and its POLY writes P_1 = Q_1 in place; the last round forms Q_L alone,
  // in bf16 for the product with X_s. Per matrix a leg of L > 1 rounds costs
  // 2 r^2 c (GRAM) + 2 r^2 c (X_e) + (8L - 6) r^3 dense-equivalent flops on
  // the symmetric kernel (about half of it computed), against L (4 r^2 c +
  // 2 r^3) for the direct rounds.
  std::vector<int> leg_first, leg_len;  // per round: first round and length of its leg
  for (int r0 = 0; r0 < steps; r0 += 3)
    for (int k = r0; k < std::min(steps, r0 + 3); ++k) {
      leg_first.push_back(r0);
      leg_len.push_back(std::min(3, steps - r0));
    }
  auto gram_scale = [](int64_t r) {  // S: a power of two near r, so S A_0 and T stay well inside fp16
    double S = 1.0;
    while (S * 2.0 <= static_cast<double>(r) && S < 8192.0) S *= 2.0;
    return S;
  };
  // 2. the rounds. Each stage is one launch over every group: GRAM, POLY
  // (every direct r-class and Gram group), the Gram route's symmetric
  // updates, and COMBINE (direct rounds and the Gram legs' ends).
  for (int it = 0; it < steps; ++it) {
    const bool last = it == steps - 1;
    const int leg = leg_first[it] / 3, j = it - leg_first[it] + 1, L = leg_len[it];
    std::vector<GemmSegSpec> gram, poly, sym, comb;
    double f_gram = 0, f_poly = 0, f_sym = 0, f_comb = 0;
    for (const NsGroup& g : plan.groups) {
      if (g.small) continue;
      const double n = g.count, r = static_cast<double>(g.r), cw = static_cast<double>(g.c);
      // flops each launch executes: symmetric r x r outputs (GRAM, POLY, the
      // Gram route's updates) compute only their upper super-blocks
      const double sh = sym_share(g.r);
      const double r3 = 2 * n * r * r * r * sh, r2c = 2 * n * r * r * cw;
      const float* scale0 = reinterpret_cast<const float*>(b + g.off_scale);
      if (g.gram && square) {
        const NsMaps& xs = (leg & 1) ? g.mx1 : g.mx0;
        const NsMaps& xe = (leg & 1) ? g.mx0 : g.mx1;
        const float* sc = leg == 0 ? scale0 : nullptr;
        const YMaps& yprev = ((j - 1) & 1) ? g.yb : g.ya;  // holds Q_{j-1}, T_{j-1} for j >= 2
        const YMaps& ycur = (j & 1) ? g.yb : g.ya;
        const double S = gram_scale(g.r);
        GemmSegSpec gs, ps{&g.mc.rows128, &g.mc.rows128, &g.mp.store, nullptr, g.count, g.r, g.r, 0};
        ps.in_fp16 = ps.out_fp16 = true;
        ps.gain = poly_gain;
        ps.diag = poly_diag;
        if (j == 1) {
          gs = GemmSegSpec{&xs.x_rows128, &xs.x_rows128, &g.mc.store, sc, g.count, g.r, g.c, 0};
          if (L > 1) {
            gs.out2 = &g.ya.t.store;
            gs.gain2 = static_cast<float>(S);
            ps.out = &g.yb.q.store;  // P_1 = Q_1
            GemmSegSpec ts{&g.yb.q.x_rows128, &g.ya.t.x_rows128, &g.yb.t.store, nullptr, g.count, g.r, g.r, 0};
            ts.in_fp16 = ts.out_fp16 = true;
            sym.push_back(ts);
            f_sym += r3;
          } else {
            ps.out_fp16 = false;  // P in bf16, the type of X_s
            GemmSegSpec cs{&g.mp.rows128, &xs.x_k64, &xe.store, sc, g.count, g.r, g.c, 0};
            if (last) cs.views = g.d_slot_views;
            comb.push_back(cs);
            f_comb += r2c;
          }
          gs.gain = gram_gain;
          f_gram += r2c * sh;
        } else {
          gs = GemmSegSpec{&yprev.t.x_rows128, &yprev.q.x_rows128, &g.mc.store, nullptr, g.count, g.r, g.r, 0};
          gs.in_fp16 = true;
          gs.gain = static_cast<float>(root / S);
          f_gram += r3;
          GemmSegSpec qs{&g.mp.rows128, &yprev.q.x_rows128, &ycur.q.store, nullptr, g.count, g.r, g.r, 0};
          qs.in_fp16 = true;
          qs.out_fp16 = j < L;  // Q_L in bf16, the type of X_s
          sym.push_back(qs);
          f_sym += r3;
          if (j < L) {
            GemmSegSpec ts{&g.mp.rows128, &yprev.t.x_rows128, &ycur.t.store, nullptr, g.count, g.r, g.r, 0};
            ts.in_fp16 = ts.out_fp16 = true;
            sym.push_back(ts);
            f_sym += r3;
          } else {
            GemmSegSpec es{&ycur.q.x_rows128, &xs.x_k64, &xe.store, sc, g.count, g.r, g.c, 0};
            if (last) es.views = g.d_slot_views;
            comb.push_back(es);
            f_comb += r2c;
          }
        }
        gs.out_fp16 = true;
        gs.diag = gram_diag;
        gram.push_back(gs);
        poly.push_back(ps);
        f_poly += r3;
        continue;
      }
      // direct rounds: X_it in x0 on even rounds, x1 on odd ones
      const bool odd = (it & 1) != 0;
      const NsMaps& cur = odd ? g.mx1 : g.mx0;
      const NsMaps& nxt = odd ? g.mx0 : g.mx1;
      const float* sc = it == 0 ? scale0 : nullptr;
      const CUtensorMap* c_out = g.gram ? &g.mc.store : &plan.rclasses[g.rclass].ma.store;
      GemmSegSpec gs{&cur.x_rows128, &cur.x_rows128, c_out, sc, g.count, g.r, g.c,
                     g.gram ? 0 : static_cast<int>(g.base_slot)};
      gs.out_fp16 = square;  // C (fp16) for POLY; P (bf16) for COMBINE when c = 0
      gs.gain = gram_gain;
      gs.diag = gram_diag;
      gram.push_back(gs);
      f_gram += r2c * sh;
      const SymMaps& pm = g.gram ? g.mc : (square ? g.mb : g.ma);
      GemmSegSpec cs{&pm.rows128, &cur.x_k64, &nxt.store, sc, g.count, g.r, g.c, 0};
      if (last) cs.views = g.d_slot_views;
      comb.push_back(cs);
      f_comb += r2c;
    }
    if (square)
      for (const NsRClass& rcl : plan.rclasses) {
        GemmSegSpec ps{&rcl.ma.rows128, &rcl.ma.rows128, &rcl.mb.store, nullptr, rcl.count, rcl.r, rcl.r, 0};
        ps.in_fp16 = true;
        ps.gain = poly_gain;
        ps.diag = poly_diag;
        poly.push_back(ps);
        f_poly += 2.0 * rcl.count * double(rcl.r) * rcl.r * rcl.r * sym_share(rcl.r);
      }
    // 3. the last round applies D = X_steps instead of storing it:
    // W <- W (1 - lr wd) - eta s D, transposed back for tall views
    int rc2;
    if ((rc2 = run(GEMM_GRAM, gram, PRM_FAMILY_NS_GRAM, f_gram, "gram launch")) != PRM_OK) return rc2;
    if (square && (rc2 = run(GEMM_POLY, poly, PRM_FAMILY_NS_POLY, f_poly, "poly launch")) != PRM_OK) return rc2;
    if ((rc2 = run(GEMM_GRAM, sym, PRM_FAMILY_NS_SYM, f_sym, "symmetric update launch")) != PRM_OK) return rc2;
    if ((rc2 = run(GEMM_COMBINE, comb, PRM_FAMILY_NS_COMBINE, f_comb, "combine launch")) != PRM_OK) return rc2;
  }
  return PRM_OK;
}

int run_rownorm(prm_ctx* c, void* base, StepScalars sc, cudaStream_t stream) {
  char* b = static_cast<char*>(base);
  cudaError_t e;
  for (auto& s : c->rn.wide) {
    const double bytes = static_cast<double>(s.views.size()) * s.rows * s.cols * (s.bf16 ? 18.0 : 20.0);
    NvtxRange nr(kFamilyNames[PRM_FAMILY_ROWNORM_WIDE]);
    const size_t ev = c->prof.begin(stream);
    e = launch_rownorm_wide(s.d_views, static_cast<int>(s.views.size()), s.rows, s.cols, s.vec_ok, s.bf16, sc,
                            stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "rownorm wide launch");
    c->prof.end(ev, PRM_FAMILY_ROWNORM_WIDE, 1, bytes, stream);
  }
  for (auto& s : c->rn.tall) {
    const double bytes = static_cast<double>(s.views.size()) * s.rows * s.cols * (s.bf16 ? 18.0 : 20.0);
    NvtxRange nr(kFamilyNames[PRM_FAMILY_ROWNORM_TALL]);
    const size_t ev = c->prof.begin(stream);
    float* partials = reinterpret_cast<float*>(b + s.off_partials);
    float* inv = reinterpret_cast<float*>(b + s.off_inv);
    const int n = static_cast<int>(s.views.size());
    if (s.fused)
      e = launch_rownorm_tall_fused(s.d_views, n, s.rows, s.cols, s.bf16, sc, partials, inv, b + s.off_flags,
                                    c->d_err, c->num_sms, stream, s.ring ? s.d_maps : nullptr, c->withhold.stripe,
                                    c->withhold.wait_ns);
    else
      e = launch_rownorm_tall(s.d_views, n, s.rows, s.cols, s.vec_ok, s.bf16, sc, partials, inv, stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "rownorm tall launch");
    c->prof.end(ev, PRM_FAMILY_ROWNORM_TALL, s.fused ? 1 : 3, bytes, stream);
  }
  c->withhold.stripe = -1;  // the test aid covers one step
  c->withhold.wait_ns = 0;
  return PRM_OK;
}

bool finite(float x) { return std::isfinite(x); }

// Per-device state of the standalone entry points (no context).
struct DeviceState {
  int num_sms = 0;
  int* d_err = nullptr;
  bool ready = false;
};
std::mutex g_dev_mutex;
DeviceState g_dev[64];

int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PRM_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceState& d = g_dev[dev];
  if (!d.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return PRM_ERR_CUDA;
    if (prop.major != 10) return PRM_ERR_UNSUPPORTED;
    d.num_sms = prop.multiProcessorCount;
    if (gemm_setup_attributes() != cudaSuccess || rownorm_setup_attributes() != cudaSuccess) return PRM_ERR_CUDA;
    if (cudaMalloc(reinterpret_cast<void**>(&d.d_err), sizeof(int)) != cudaSuccess) return PRM_ERR_CUDA;
    if (cudaMemset(d.d_err, 0, sizeof(int)) != cudaSuccess) return PRM_ERR_CUDA;
    d.ready = true;
  }
  *out = &d;
  return PRM_OK;
}

}  // namespace

extern "C" {

int prm_create(prm_ctx** out, int cuda_device) {
  if (out == nullptr) return fail(nullptr, PRM_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  int ndev = 0;
  cudaError_t e = cudaGetDeviceCount(&ndev);
  if (e != cudaSuccess) return fail(nullptr, PRM_ERR_CUDA, std::string("cudaGetDeviceCount: ") + cudaGetErrorString(e));
  if (cuda_device < 0 || cuda_device >= ndev) return fail(nullptr, PRM_ERR_INVALID_ARG, "no such CUDA device");
  cudaDeviceProp prop;
  if ((e = cudaGetDeviceProperties(&prop, cuda_device)) != cudaSuccess)
    return fail(nullptr, PRM_ERR_CUDA, std::string("cudaGetDeviceProperties: ") + cudaGetErrorString(e));
  if (prop.major != 10)
    return fail(nullptr, PRM_ERR_UNSUPPORTED,
                "device compute capability " + std::to_string(prop.major) + "." + std::to_string(prop.minor) +
                    " is not in the sm_100 family this library is built for");
  prm_ctx* c = new (std::nothrow) prm_ctx();
  if (c == nullptr) return fail(nullptr, PRM_ERR_OOM, "out of host memory");
  c->device = cuda_device;
  c->num_sms = prop.multiProcessorCount;
  DeviceGuard guard(cuda_device);
  if ((e = gemm_setup_attributes()) != cudaSuccess || (e = rownorm_setup_attributes()) != cudaSuccess) {
    delete c;
    return fail(nullptr, PRM_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
  }
  if ((e = cudaMalloc(reinterpret_cast<void**>(&c->d_err), sizeof(int))) != cudaSuccess ||
      (e = cudaMemset(c->d_err, 0, sizeof(int))) != cudaSuccess) {
    if (c->d_err) cudaFree(c->d_err);
    delete c;
    return fail(nullptr, PRM_ERR_CUDA, std::string("error word: ") + cudaGetErrorString(e));
  }
  *out = c;
  return PRM_OK;
}

int prm_destroy(prm_ctx* c) {
  if (c == nullptr) return PRM_OK;
  DeviceGuard guard(c->device);
  clear_registration(c);
  if (c->d_err) cudaFree(c->d_err);
  delete c;
  return PRM_OK;
}

int prm_register_matrices(prm_ctx* c, const prm_matrix_desc* d, int count, int muonbp_blocks) {
  if (c == nullptr) return fail(nullptr, PRM_ERR_INVALID_ARG, "ctx is NULL");
  if (count < 0 || (count > 0 && d == nullptr)) return fail(c, PRM_ERR_INVALID_ARG, "bad descriptor array");
  if (count > 65535 / std::max(1, muonbp_blocks))
    return fail(c, PRM_ERR_UNSUPPORTED, "too many matrices for one registration (limit 65535 views)");
  if (muonbp_blocks < 0) return fail(c, PRM_ERR_INVALID_ARG, "muonbp_blocks must be >= 0");
  DeviceGuard guard(c->device);
  clear_registration(c);
  c->ws = nullptr;
  c->ws_bytes = 0;
  std::vector<View> full;
  full.reserve(count);
  for (int i = 0; i < count; ++i) {
    const prm_matrix_desc& m = d[i];
    if (m.param == nullptr || m.momentum == nullptr || m.grad == nullptr)
      return fail(c, PRM_ERR_INVALID_ARG, "matrix " + std::to_string(i) + ": NULL pointer");
    if (m.grad_dtype != PRM_FP32 && m.grad_dtype != PRM_BF16)
      return fail(c, PRM_ERR_INVALID_ARG, "matrix " + std::to_string(i) + ": unknown grad_dtype");
    if (m.reserved != 0 || m.reserved2 != 0.f)
      return fail(c, PRM_ERR_INVALID_ARG, "matrix " + std::to_string(i) + ": reserved fields must be 0");
    if (m.rows < 1 || m.cols < 1 || m.rows > (int64_t(1) << 31) - 1 || m.cols > (int64_t(1) << 31) - 1)
      return fail(c, PRM_ERR_SHAPE, "matrix " + std::to_string(i) + ": rows and cols must be in [1, 2^31)");
    // Launch-grid limits: views of one shape share grid.y / grid.z (<= 65535),
    // tall row blocks of 256 rows and 64 x 64 transpose tiles use grid.y.
    if (std::min(m.rows, m.cols) > int64_t(65535) * 64 || (m.rows > m.cols && m.rows > int64_t(65535) * 64))
      return fail(c, PRM_ERR_UNSUPPORTED, "matrix " + std::to_string(i) + ": shape beyond the kernels' grid limits");
    if (!aligned16(m.param) || !aligned16(m.momentum) || !aligned16(m.grad))
      return fail(c, PRM_ERR_ALIGNMENT, "matrix " + std::to_string(i) + ": pointers must be 16-byte aligned");
    if (!std::isfinite(m.shape_scale))
      return fail(c, PRM_ERR_INVALID_ARG, "matrix " + std::to_string(i) + ": shape_scale not finite");
    View v{};
    v.W = m.param;
    v.M = m.momentum;
    v.G = m.grad;
    v.rows = m.rows;
    v.cols = m.cols;
    v.ld = m.cols;
    v.grad_bf16 = m.grad_dtype == PRM_BF16;
    v.shape_scale = m.shape_scale > 0.f
                        ? m.shape_scale
                        : static_cast<float>(std::sqrt(std::max(1.0, double(m.rows) / double(m.cols))));
    full.push_back(v);
  }
  // MuonBP blocks: P contiguous pieces along the long side, last takes the remainder.
  std::vector<View> blocks;
  if (muonbp_blocks > 0) {
    for (int i = 0; i < count; ++i) {
      const View& v = full[i];
      if ((v.rows <= v.cols ? v.cols : v.rows) < muonbp_blocks)
        return fail(c, PRM_ERR_SHAPE, "matrix " + std::to_string(i) + ": long side shorter than muonbp_blocks");
      make_blocks(v, muonbp_blocks, blocks);
    }
  }
  // RowNorm launch sets (whole matrices), tall scratch laid out back to back.
  for (const View& v : full) add_to_sets(v.rows <= v.cols ? c->rn.wide : c->rn.tall, v);
  size_t off = 0;
  for (auto& s : c->rn.tall) {
    s.fused = s.vec_ok && tall_fused_fits(static_cast<int>(s.views.size()), s.rows, s.cols);
    s.ring = s.fused && tall_ring_ok(s.cols, s.bf16);
    if (s.fused) {
      const TallFusedScratch t = tall_fused_scratch(static_cast<int>(s.views.size()), s.rows, s.cols);
      s.off_partials = off;
      off += align_up(t.partials_bytes, 256);
      s.off_inv = off;
      off += align_up(t.inv_bytes, 256);
      s.off_flags = off;
      off += align_up(t.flag_bytes, 256);
      continue;
    }
    s.off_partials = off;
    off += align_up(s.views.size() * tall_row_blocks(s.rows) * s.cols * 4, 256);
    s.off_inv = off;
    off += align_up(s.views.size() * s.cols * 4, 256);
  }
  c->rn.bytes = off;
  build_ns_subplans(full, c->ws_limit, c->ns_form, c->ns_full);
  if (muonbp_blocks > 0) build_ns_subplans(blocks, c->ws_limit, c->ns_form, c->ns_blocks);
  cudaError_t e = upload_sets(c->rn.wide);
  if (e == cudaSuccess) e = upload_sets(c->rn.tall);
  for (auto& s : c->rn.tall) {
    if (e != cudaSuccess || !s.ring) continue;
    // a view the tensor maps cannot describe keeps the register form
    if (upload_ring_maps(s) != cudaSuccess) {
      if (s.d_maps) cudaFree(s.d_maps);
      s.d_maps = nullptr;
      s.ring = false;
      cudaGetLastError();
    }
  }
  for (auto* plans : {&c->ns_full, &c->ns_blocks})
    for (auto& p : *plans)
      for (auto& g : p.groups)
        if (e == cudaSuccess) e = upload_group(g);
  if (e != cudaSuccess) {
    clear_registration(c);
    return cuda_fail(c, e, "uploading launch tables");
  }
  c->full = std::move(full);
  c->count = count;
  c->blocks = muonbp_blocks;
  c->registered = true;
  return PRM_OK;
}

int prm_set_workspace_limit(prm_ctx* c, size_t max_bytes) {
  if (c == nullptr) return fail(nullptr, PRM_ERR_INVALID_ARG, "ctx is NULL");
  c->ws_limit = max_bytes;
  return PRM_OK;
}

int prm_set_ns_form(prm_ctx* c, int form) {
  if (c == nullptr) return fail(nullptr, PRM_ERR_INVALID_ARG, "ctx is NULL");
  if (form != PRM_NS_FORM_AUTO && form != PRM_NS_FORM_DIRECT) return fail(c, PRM_ERR_INVALID_ARG, "unknown NS5 form");
  c->ns_form = form;
  return PRM_OK;
}

int prm_debug_withhold_tall_norms(prm_ctx* c, int stripe, double wait_limit_s) {
  if (c == nullptr) return fail(nullptr, PRM_ERR_INVALID_ARG, "ctx is NULL");
  if (stripe < 0 || !(wait_limit_s > 0.0) || wait_limit_s > 2.0)
    return fail(c, PRM_ERR_INVALID_ARG, "stripe must be >= 0 and wait_limit_s in (0, 2]");
  c->withhold.stripe = stripe;
  c->withhold.wait_ns = static_cast<uint64_t>(wait_limit_s * 1e9);
  return PRM_OK;
}

int prm_workspace_bytes(const prm_ctx* c, size_t* bytes) {
  if (c == nullptr || bytes == nullptr) return PRM_ERR_INVALID_ARG;
  *bytes = c->registered ? std::max({c->rn.bytes, plans_bytes(c->ns_full), plans_bytes(c->ns_blocks)}) : 0;
  return PRM_OK;
}

int prm_set_workspace(prm_ctx* c, void* dev_ptr, size_t bytes) {
  if (c == nullptr) return fail(nullptr, PRM_ERR_INVALID_ARG, "ctx is NULL");
  size_t need = 0;
  prm_workspace_bytes(c, &need);
  if (need > 0 && dev_ptr == nullptr) return fail(c, PRM_ERR_INVALID_ARG, "workspace pointer is NULL");
  if ((reinterpret_cast<uintptr_t>(dev_ptr) & 255u) != 0)
    return fail(c, PRM_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  if (bytes < need)
    return fail(c, PRM_ERR_WORKSPACE, "workspace of " + std::to_string(bytes) + " bytes is smaller than the " +
                                          std::to_string(need) + " required");
  c->ws = dev_ptr;
  c->ws_bytes = bytes;
  return PRM_OK;
}

int prm_ns_route(int64_t m, int64_t n, int form) {
  if (m < 1 || n < 1 || (form != PRM_NS_FORM_AUTO && form != PRM_NS_FORM_DIRECT)) return -PRM_ERR_INVALID_ARG;
  if (std::min(m, n) < NS_SMALL_R) return 2;
  return (form == PRM_NS_FORM_AUTO && gram_route_pays(std::min(m, n), std::max(m, n))) ? 1 : 0;
}

int prm_branch(int64_t t, int K, int mode) {
  if (t < 0 || K < 1 || (mode != PRM_MODE_PRMUON && mode != PRM_MODE_MUONBP)) return -PRM_ERR_INVALID_ARG;
  return (t % K == 0) ? 1 : 0;
}

int prm_step(prm_ctx* c, int64_t t, int K, float gamma, float lr, float wd, float beta, float eps,
             const float* ns_coeffs, int mode, void* stream) {
  if (c == nullptr) return fail(nullptr, PRM_ERR_INVALID_ARG, "ctx is NULL");
  if (t < 0) return fail(c, PRM_ERR_INVALID_ARG, "t must be >= 0");
  if (K < 1) return fail(c, PRM_ERR_INVALID_ARG, "K must be >= 1");
  if (mode != PRM_MODE_PRMUON && mode != PRM_MODE_MUONBP) return fail(c, PRM_ERR_INVALID_ARG, "unknown mode");
  if (!(beta >= 0.f && beta < 1.f)) return fail(c, PRM_ERR_INVALID_ARG, "beta must be in [0, 1)");
  if (!(eps > 0.f) || !finite(eps)) return fail(c, PRM_ERR_INVALID_ARG, "eps must be > 0");
  if (!finite(lr) || !finite(wd) || !finite(gamma)) return fail(c, PRM_ERR_INVALID_ARG, "lr, wd, gamma must be finite");
  float coeffs[3] = {DEFAULT_COEFFS[0], DEFAULT_COEFFS[1], DEFAULT_COEFFS[2]};
  if (ns_coeffs != nullptr) {
    for (int i = 0; i < 3; ++i) {
      if (!finite(ns_coeffs[i])) return fail(c, PRM_ERR_INVALID_ARG, "ns_coeffs must be finite");
      coeffs[i] = ns_coeffs[i];
    }
  }
  if (!c->registered) return fail(c, PRM_ERR_NOT_REGISTERED, "no matrices registered");
  if (mode == PRM_MODE_MUONBP && c->blocks == 0)
    return fail(c, PRM_ERR_NOT_REGISTERED, "MuonBP step needs a registration with muonbp_blocks > 0");
  size_t need = 0;
  prm_workspace_bytes(c, &need);
  if (need > 0 && (c->ws == nullptr || c->ws_bytes < need))
    return fail(c, PRM_ERR_WORKSPACE, "workspace not set or too small");
  if (c->count == 0) return PRM_OK;
  DeviceGuard guard(c->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool refresh = (t % K) == 0;
  NvtxRange nr("prm_step");
  StepScalars sc;
  sc.beta = beta;
  sc.decay = 1.f - lr * wd;
  sc.eta = refresh ? lr : lr * gamma;
  sc.eps = eps;
  c->last.valid = false;
  if (mode == PRM_MODE_PRMUON && !refresh) {
    const int rc = run_rownorm(c, c->ws, sc, st);
    if (rc != PRM_OK) return rc;
  } else {
    std::vector<NsPlan>& plans = (mode == PRM_MODE_MUONBP && !refresh) ? c->ns_blocks : c->ns_full;
    for (auto& plan : plans) {
      const int rc = run_ns(c, plan, c->ws, true, beta, sc.decay, sc.eta, coeffs, NS_STEPS, st);
      if (rc != PRM_OK) return rc;
    }
  }
  c->last.valid = true;
  c->last.t = t;
  c->last.K = K;
  c->last.mode = mode;
  c->last.eps = eps;
  for (int i = 0; i < 3; ++i) c->last.coeffs[i] = coeffs[i];
  return PRM_OK;
}

// The launch set of the RowNorm step that holds this tall view (its choice
// of the one-launch kernel and of the ring form), or nullptr.
static const LaunchSet* tall_set_of(const prm_ctx* c, const View& v) {
  for (const auto& s : c->rn.tall)
    if (s.rows == v.rows && s.cols == v.cols && s.bf16 == (v.grad_bf16 != 0)) return &s;
  return nullptr;
}

// Recomputes the direction D of the last step for one matrix from its
// momentum (which, after the step, is the M_t the direction was taken from)
// with the step's own kernels, on scratch buffers: the NS5 branch runs the
// prep / GEMM / apply launches with the apply writing D instead of updating W;
// the RowNorm branch runs the RowNorm kernels on a copy of M with beta = 1,
// G = 0, W = 0, decay = 1 and eta * s = -1, so that the "update" leaves
// W = M / max(||v||, eps) = D.
int prm_debug_last_direction(prm_ctx* c, int idx, float* host_out) {
  if (c == nullptr) return fail(nullptr, PRM_ERR_INVALID_ARG, "ctx is NULL");
  if (!c->registered) return fail(c, PRM_ERR_NOT_REGISTERED, "no matrices registered");
  if (idx < 0 || idx >= c->count) return fail(c, PRM_ERR_INVALID_ARG, "matrix index out of range");
  if (host_out == nullptr) return fail(c, PRM_ERR_INVALID_ARG, "host_out is NULL");
  if (!c->last.valid) return fail(c, PRM_ERR_INVALID_ARG, "no step has been taken since registration");
  DeviceGuard guard(c->device);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(c, e, "device synchronize");
  const View& v = c->full[idx];
  const size_t n = static_cast<size_t>(v.rows) * v.cols;
  const bool refresh = c->last.t % c->last.K == 0;
  const cudaStream_t st = nullptr;
  std::vector<void*> scratch;  // freed on every return path
  auto dev_alloc = [&](size_t bytes) -> void* {
    void* p = nullptr;
    if (cudaMalloc(&p, bytes < 256 ? 256 : bytes) != cudaSuccess) return nullptr;
    scratch.push_back(p);
    return p;
  };
  auto finish = [&](int rc) {
    for (void* p : scratch) cudaFree(p);
    return rc;
  };
  float* d_out = static_cast<float*>(dev_alloc(n * sizeof(float)));
  if (d_out == nullptr) return finish(fail(c, PRM_ERR_OOM, "no device memory for the direction"));
  if (c->last.mode == PRM_MODE_PRMUON && !refresh) {
    float* d_m = static_cast<float*>(dev_alloc(n * sizeof(float)));
    float* d_g = static_cast<float*>(dev_alloc(n * sizeof(float)));
    if (d_m == nullptr || d_g == nullptr) return finish(fail(c, PRM_ERR_OOM, "no device memory for scratch"));
    if ((e = cudaMemcpy(d_m, v.M, n * sizeof(float), cudaMemcpyDeviceToDevice)) != cudaSuccess ||
        (e = cudaMemset(d_g, 0, n * sizeof(float))) != cudaSuccess ||
        (e = cudaMemset(d_out, 0, n * sizeof(float))) != cudaSuccess)
      return finish(cuda_fail(c, e, "scratch set-up"));
    View dv = v;
    dv.W = d_out;
    dv.M = d_m;
    dv.G = d_g;
    dv.grad_bf16 = 0;
    dv.shape_scale = 1.f;
    std::vector<LaunchSet> sets;
    add_to_sets(sets, dv);
    if ((e = upload_sets(sets)) != cudaSuccess) {
      free_sets(sets);
      return finish(cuda_fail(c, e, "uploading the launch table"));
    }
    StepScalars sc;
    sc.beta = 1.f;
    sc.decay = 1.f;
    sc.eta = -1.f;
    sc.eps = c->last.eps;
    const LaunchSet& s = sets.front();
    if (v.rows <= v.cols) {
      e = launch_rownorm_wide(s.d_views, 1, v.rows, v.cols, s.vec_ok, false, sc, st);
    } else if (tall_set_of(c, v) != nullptr && tall_set_of(c, v)->fused && tall_fused_fits(1, v.rows, v.cols)) {
      // the step's own one-launch kernel, so that D matches what it applied
      const TallFusedScratch t = tall_fused_scratch(1, v.rows, v.cols);
      float* d_part = static_cast<float*>(dev_alloc(t.partials_bytes));
      float* d_inv = static_cast<float*>(dev_alloc(t.inv_bytes));
      void* d_flags = dev_alloc(t.flag_bytes);
      if (d_part == nullptr || d_inv == nullptr || d_flags == nullptr) {
        free_sets(sets);
        return finish(fail(c, PRM_ERR_OOM, "no device memory for scratch"));
      }
      // the same form as the step (the fp32 zero G here qualifies for the
      // ring whenever the step's gradients did)
      LaunchSet& ls = sets.front();
      const bool ring = tall_set_of(c, v)->ring;
      if (ring && (e = upload_ring_maps(ls)) != cudaSuccess) {
        free_sets(sets);
        return finish(cuda_fail(c, e, "ring tensor maps"));
      }
      e = launch_rownorm_tall_fused(ls.d_views, 1, v.rows, v.cols, false, sc, d_part, d_inv, d_flags, c->d_err,
                                    c->num_sms, st, ring ? ls.d_maps : nullptr);
    } else {
      const size_t pb = static_cast<size_t>(tall_row_blocks(v.rows)) * v.cols * sizeof(float);
      float* d_part = static_cast<float*>(dev_alloc(pb));
      float* d_inv = static_cast<float*>(dev_alloc(static_cast<size_t>(v.cols) * sizeof(float)));
      if (d_part == nullptr || d_inv == nullptr) {
        free_sets(sets);
        return finish(fail(c, PRM_ERR_OOM, "no device memory for scratch"));
      }
      e = launch_rownorm_tall(s.d_views, 1, v.rows, v.cols, s.vec_ok, false, sc, d_part, d_inv, st);
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    free_sets(sets);
    if (e != cudaSuccess) return finish(cuda_fail(c, e, "rownorm direction"));
  } else {
    // NS5 of the whole matrix (refresh / full step) or of each MuonBP block.
    std::vector<View> parts;
    if (refresh)
      parts.push_back(v);
    else
      make_blocks(v, c->blocks, parts);
    for (View& p : parts) {
      p.out = d_out + (p.M - v.M);  // same offset and pitch as the block inside M
      p.W = nullptr;
    }
    NsPlan plan;
    build_ns_plan(parts, plan, c->ns_form);
    for (auto& g : plan.groups) {
      if ((e = upload_group(g)) != cudaSuccess) {
        free_plan(plan);
        return finish(cuda_fail(c, e, "uploading launch tables"));
      }
    }
    void* ws = dev_alloc(plan.bytes);
    if (ws == nullptr) {
      free_plan(plan);
      return finish(fail(c, PRM_ERR_OOM, "no device memory for the NS5 workspace"));
    }
    prm_ctx tmp;
    tmp.num_sms = c->num_sms;
    tmp.d_err = c->d_err;
    int rc = run_ns(&tmp, plan, ws, false, 0.f, 1.f, 1.f, c->last.coeffs, NS_STEPS, st);
    e = cudaStreamSynchronize(st);
    free_plan(plan);
    tmp.d_err = nullptr;
    if (rc != PRM_OK) return finish(fail(c, rc, tmp.err));
    if (e != cudaSuccess) return finish(cuda_fail(c, e, "NS5 direction"));
  }
  if ((e = cudaMemcpy(host_out, d_out, n * sizeof(float), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return finish(cuda_fail(c, e, "copying the direction to the host"));
  return finish(PRM_OK);
}

int prm_sync_status(prm_ctx* c, void* stream) {
  if (c == nullptr) return fail(nullptr, PRM_ERR_INVALID_ARG, "ctx is NULL");
  DeviceGuard guard(c->device);
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(c, e, "stream synchronize");
  int word = 0;
  if ((e = cudaMemcpy(&word, c->d_err, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(c, e, "reading error word");
  if (word != 0) {
    cudaMemset(c->d_err, 0, sizeof(int));
    return fail(c, PRM_ERR_TIMEOUT, "a device-side wait gave up (error word " + std::to_string(word) + ")");
  }
  return PRM_OK;
}

int prm_profile(prm_ctx* c, int enable) {
  if (c == nullptr) return fail(nullptr, PRM_ERR_INVALID_ARG, "ctx is NULL");
  DeviceGuard guard(c->device);
  if (enable) c->prof.reset();
  c->prof.on = enable != 0;
  return PRM_OK;
}

int prm_profile_read(prm_ctx* c, int family, double* total_ms, int64_t* records, int64_t* kernels,
                     double* work) {
  if (c == nullptr) return fail(nullptr, PRM_ERR_INVALID_ARG, "ctx is NULL");
  if (family < -1 || family >= PRM_FAMILY_COUNT) return fail(c, PRM_ERR_INVALID_ARG, "unknown family");
  DeviceGuard guard(c->device);
  double ms = 0, w = 0;
  int64_t n = 0, k = 0;
  for (const auto& r : c->prof.recs) {
    if (family != -1 && r.family != family) continue;
    cudaError_t e = cudaEventSynchronize(c->prof.pool[r.ev + 1]);
    if (e != cudaSuccess) return cuda_fail(c, e, "event synchronize");
    float dt = 0.f;
    if ((e = cudaEventElapsedTime(&dt, c->prof.pool[r.ev], c->prof.pool[r.ev + 1])) != cudaSuccess)
      return cuda_fail(c, e, "event elapsed time");
    ms += dt;
    w += r.work;
    ++n;
    k += r.kernels;
  }
  if (total_ms) *total_ms = ms;
  if (records) *records = n;
  if (kernels) *kernels = k;
  if (work) *work = w;
  return PRM_OK;
}

const char* prm_last_error(const prm_ctx* c) {
  if (c == nullptr) return g_create_error.c_str();
  return c->err.c_str();
}

// ---------------------------------------------------------------- standalone
int prm_ns_gram(const uint16_t* X, uint16_t* C, const float* scale, float gain, float diag, int out_dtype,
                int batch, int64_t r, int64_t c, int64_t ldc, int64_t ldr, void* stream) {
  if (X == nullptr || C == nullptr || batch < 0 || r < 1 || c < r || ldc < c || ldr < r) return PRM_ERR_INVALID_ARG;
  if (!finite(gain) || !finite(diag) || (out_dtype != PRM_BF16 && out_dtype != PRM_FP16)) return PRM_ERR_INVALID_ARG;
  if (ldc % 8 || ldr % 8 || !aligned16(X) || !aligned16(C)) return PRM_ERR_ALIGNMENT;
  if (batch == 0) return PRM_OK;
  DeviceState* ds;
  int rc = device_state(&ds);
  if (rc != PRM_OK) return rc;
  NsMaps mx;
  SymMaps mc;
  if (encode_x_maps(&mx, X, batch, r, c, ldc) != 0 || encode_sym_maps(&mc, C, batch, r, ldr) != 0)
    return PRM_ERR_CUDA;
  GemmSegSpec seg{&mx.x_rows128, &mx.x_rows128, &mc.store, scale, batch, r, c, 0};
  seg.out_fp16 = out_dtype == PRM_FP16;
  seg.gain = gain;
  seg.diag = diag;
  GemmEpilogue epi;
  epi.err = ds->d_err;
  epi.num_sms = ds->num_sms;
  return launch_gemm(GEMM_GRAM, &seg, 1, epi, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PRM_OK
                                                                                              : PRM_ERR_CUDA;
}

int prm_ns_poly(const uint16_t* C, uint16_t* P, float gain, float diag, int in_dtype, int batch, int64_t r,
                int64_t ldr, void* stream) {
  if (C == nullptr || P == nullptr || batch < 0 || r < 1 || ldr < r) return PRM_ERR_INVALID_ARG;
  if (C == P || !finite(gain) || !finite(diag) || (in_dtype != PRM_BF16 && in_dtype != PRM_FP16))
    return PRM_ERR_INVALID_ARG;
  if (ldr % 8 || !aligned16(C) || !aligned16(P)) return PRM_ERR_ALIGNMENT;
  if (batch == 0) return PRM_OK;
  DeviceState* ds;
  int rc = device_state(&ds);
  if (rc != PRM_OK) return rc;
  SymMaps mc, mp;
  if (encode_sym_maps(&mc, C, batch, r, ldr) != 0 || encode_sym_maps(&mp, P, batch, r, ldr) != 0)
    return PRM_ERR_CUDA;
  GemmSegSpec seg{&mc.rows128, &mc.rows128, &mp.store, nullptr, batch, r, r, 0};
  seg.in_fp16 = in_dtype == PRM_FP16;
  seg.gain = gain;
  seg.diag = diag;
  GemmEpilogue epi;
  epi.err = ds->d_err;
  epi.num_sms = ds->num_sms;
  return launch_gemm(GEMM_POLY, &seg, 1, epi, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PRM_OK
                                                                                              : PRM_ERR_CUDA;
}

int prm_ns_combine(const uint16_t* X, const uint16_t* B, uint16_t* Xout, const float* scale, int batch, int64_t r,
                   int64_t c, int64_t ldc, int64_t ldr, void* stream) {
  if (X == nullptr || B == nullptr || Xout == nullptr || batch < 0 || r < 1 || c < r || ldc < c || ldr < r)
    return PRM_ERR_INVALID_ARG;
  if (X == Xout) return PRM_ERR_INVALID_ARG;
  if (ldc % 8 || ldr % 8 || !aligned16(X) || !aligned16(B) || !aligned16(Xout)) return PRM_ERR_ALIGNMENT;
  if (batch == 0) return PRM_OK;
  DeviceState* ds;
  int rc = device_state(&ds);
  if (rc != PRM_OK) return rc;
  NsMaps mx, mo;
  SymMaps mb;
  if (encode_x_maps(&mx, X, batch, r, c, ldc) != 0 || encode_sym_maps(&mb, B, batch, r, ldr) != 0 ||
      encode_x_maps(&mo, Xout, batch, r, c, ldc) != 0)
    return PRM_ERR_CUDA;
  GemmSegSpec seg{&mb.rows128, &mx.x_k64, &mo.store, scale, batch, r, c, 0};
  GemmEpilogue epi;
  epi.err = ds->d_err;
  epi.num_sms = ds->num_sms;
  return launch_gemm(GEMM_COMBINE, &seg, 1, epi, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PRM_OK
                                                                                                 : PRM_ERR_CUDA;
}

static void standalone_group(int batch, int64_t m, int64_t n, NsPlan& plan) {
  std::vector<View> views(batch);
  for (int i = 0; i < batch; ++i) {
    views[i] = View{};
    views[i].rows = m;
    views[i].cols = n;
    views[i].ld = n;
  }
  build_ns_plan(views, plan, PRM_NS_FORM_AUTO);
}

int prm_newton_schulz_workspace(int batch, int64_t m, int64_t n, size_t* bytes) {
  if (bytes == nullptr || batch < 0 || m < 1 || n < 1) return PRM_ERR_INVALID_ARG;
  if (batch == 0) {
    *bytes = 0;
    return PRM_OK;
  }
  NsPlan plan;
  standalone_group(batch, m, n, plan);
  *bytes = plan.bytes;
  return PRM_OK;
}

int prm_newton_schulz(const float* in, float* out, int batch, int64_t m, int64_t n, const float* ns_coeffs,
                      int steps, void* workspace, size_t ws_bytes, void* stream) {
  if (in == nullptr || out == nullptr || batch < 0 || m < 1 || n < 1 || steps < 1) return PRM_ERR_INVALID_ARG;
  if (!aligned16(in) || !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return PRM_ERR_ALIGNMENT;
  if (batch == 0) return PRM_OK;
  float coeffs[3] = {DEFAULT_COEFFS[0], DEFAULT_COEFFS[1], DEFAULT_COEFFS[2]};
  if (ns_coeffs)
    for (int i = 0; i < 3; ++i) {
      if (!finite(ns_coeffs[i])) return PRM_ERR_INVALID_ARG;
      coeffs[i] = ns_coeffs[i];
    }
  DeviceState* ds;
  int rc = device_state(&ds);
  if (rc != PRM_OK) return rc;
  NsPlan plan;
  std::vector<View> views(batch);
  for (int i = 0; i < batch; ++i) {
    View v{};
    v.M = const_cast<float*>(in) + static_cast<int64_t>(i) * m * n;
    v.out = out + static_cast<int64_t>(i) * m * n;
    v.rows = m;
    v.cols = n;
    v.ld = n;
    v.shape_scale = 1.f;
    views[i] = v;
  }
  build_ns_plan(views, plan, PRM_NS_FORM_AUTO);
  if (workspace == nullptr || ws_bytes < plan.bytes) return PRM_ERR_WORKSPACE;
  if (upload_group(plan.groups[0]) != cudaSuccess) {
    free_plan(plan);
    return PRM_ERR_CUDA;
  }
  prm_ctx tmp;
  tmp.num_sms = ds->num_sms;
  tmp.d_err = ds->d_err;
  rc = run_ns(&tmp, plan, workspace, false, 0.f, 1.f, 1.f, coeffs, steps, static_cast<cudaStream_t>(stream));
  // The launch tables must outlive the kernels that read them.
  cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  free_plan(plan);
  tmp.d_err = nullptr;
  return rc;
}

}  // extern "C"
