// The three tensor-core GEMMs of one Newton-Schulz round, as persistent
// tcgen05/TMEM kernels for sm_103a ("Scaling Muon for Diffusion
// Transformers", PaperDaily walkthrough, section "Periodic Row-wise Muon":
// NS5 is five rounds of matrix products and scalings):
//
//   GRAM    : C  = gain * s^2 * X X^T + diag * I   (r x r, symmetric; upper
//                                         super-blocks computed, lower ones mirrored)
//   POLY    : P  = gain * C C + diag * I          (C symmetric, so C C = C C^T;
//                                         same triangle scheme)
//   COMBINE : X' = s * P X                         (r x c; scaling in the epilogue)
//
// One round X' = a X + (b A + c A A) X, A = X X^T, is evaluated as P X with
// P = a I + b A + c A A written as a completed square: for c != 0, with
// C = sqrt|c| A + sgn(c) b / (2 sqrt|c|) I, P = sgn(c) C C + (a - b^2 / (4c)) I
// (C is a polynomial in A, so it commutes with A and the identity is exact).
// GRAM therefore writes C (gain sqrt|c|, diag sgn(c) b / (2 sqrt|c|)) and
// POLY squares it (gain sgn(c), diag a - b^2 / (4c)): no epilogue re-reads an
// operand from memory. C is stored in fp16, not bf16: its diagonal carries
// the shift b / (2 sqrt|c|) (-1.68 for the default quintic), next to which
// bf16's 8-bit significand would drop most of sqrt|c| A_ii, while fp16's
// 11 bits keep it (in emulation the fp16 form is as accurate as evaluating
// a X + B X with bf16 A, the bf16 one about 30 % less accurate). For c = 0,
// GRAM writes P = b A + a I directly (bf16) and POLY is skipped.
//
// Each launch covers every matrix of a same-shape batch: the tile queue runs
// over (matrix, tile) pairs, so small r x r products still fill the GPU. A
// launch can visit each segment's matrices last to first (the engine
// alternates, so that a launch starts where its predecessor's outputs are
// still in L2); the results do not depend on the order.
//
// CTA pairs. The kernel runs in 2-CTA clusters, one CTA per SM; a pair owns a
// 256 x 256 output tile and computes it with tcgen05.mma.cta_group::2
// (M = 256, N = 256, K = 16): the even CTA issues the MMAs, each CTA holds
// 128 rows of A and 128 rows (N) of B in its own shared memory, and each
// CTA's TMEM receives its 128 output rows. Per SM this halves the operand
// bytes read from shared memory and L2 for a given number of FLOPs, and it
// leaves room for a 6-stage TMA ring.
//
// CTA layout (320 threads, one CTA per SM):
//   warp 0     : TMA producer (one lane): per stage a 128x64 A tile and a
//                128-row (N) slice of B, 128-byte swizzle; completion counted
//                on the even CTA's barrier
//   warp 1     : TMEM allocation for the pair (512 columns: two 128x256 fp32
//                accumulators); in the even CTA one lane issues the MMAs
//   warps 2..9 : epilogue -- tcgen05.ld of this CTA's 128 accumulator rows
//                (one TMEM lane = one output row per thread; warp w reads
//                lane quarter w % 4, warps 2-5 the tile's left 128 columns,
//                warps 6-9 the right ones), fused scaling and diagonal
//                shift, 16-bit results staged per 32 x 32 box in shared
//                memory and written by TMA stores (plus the transposed box
//                for the mirrored half of symmetric outputs)
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "internal.h"
#include "ptx.cuh"

namespace prm {
namespace {

constexpr int PAIR_M = 256;  // output rows per CTA pair (UMMA M)
constexpr int BM = 128;      // output rows per CTA
constexpr int BN = 256;      // output cols per tile (UMMA N); also the super-block edge of symmetric outputs
constexpr int BN_HALF = 128; // B rows (N) held by each CTA
constexpr int BK = 64;       // reduction slice per pipeline stage (64 bf16 = one 128-byte swizzle row)
constexpr int UK = 16;       // reduction length of one tcgen05.mma kind::f16
constexpr int STAGES = 6;
constexpr uint32_t A_TILE_BYTES = BM * BK * 2;       // 16 KB
constexpr uint32_t B_TILE_BYTES = BN_HALF * BK * 2;  // 16 KB
constexpr uint32_t STAGE_BYTES = A_TILE_BYTES + B_TILE_BYTES;
constexpr uint32_t PAIR_STAGE_BYTES = 2 * STAGE_BYTES;  // what the even CTA's full barrier expects
constexpr uint32_t MN_CHUNK_BYTES = 64 * BK * 2;        // one 64-column MN-major box of the B operand
constexpr int NUM_THREADS = 320;
constexpr int EPI_WARPS = 8;     // two per TMEM lane quarter, each taking half of a tile's columns
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr size_t BARRIER_BYTES = 256;
// Epilogue staging: per epilogue warp two 32 x 32 16-bit boxes (64-byte rows;
// one for the tile's own chunk, one for its mirror) from which TMA stores
// write the output. The boxes follow the
// output maps' 64-byte swizzle: the 16-byte chunk c of box row rho sits at
// chunk c ^ ((rho >> 1) & 3) (address bits [5:4] ^= bits [8:7] of a
// 512-byte aligned box), which also keeps the row-per-lane writes free of
// bank conflicts.
constexpr int STAGE_ROW_BYTES = 64;
constexpr uint32_t EPI_BUF_BYTES = 32 * STAGE_ROW_BYTES;
constexpr uint32_t EPI_WARP_BYTES = 2 * EPI_BUF_BYTES;
constexpr size_t EPI_SMEM_BYTES = EPI_WARPS * EPI_WARP_BYTES;
constexpr size_t SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_SMEM_BYTES + BARRIER_BYTES;
static_assert(SMEM_BYTES <= 232448, "dynamic shared memory above the 227 KB per-block limit");
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // 2 s per individual wait

// One same-shape batch of a launch: an NS5 group (GRAM, COMBINE) or an
// r-class (POLY). A launch runs the tiles of up to MAX_SEGS segments from one
// queue, so the tail of one batch overlaps the next instead of idling SMs
// between launches.
constexpr int MAX_SEGS = GEMM_MAX_SEGMENTS;  // 6: keeps the parameter block within 4 KB (a segment is 640 bytes)
constexpr int SEG_IN_FP16 = 1;   // operands are fp16 (else bf16)
constexpr int SEG_OUT_FP16 = 2;  // output packed as fp16 (else bf16)
constexpr int SEG_DUAL = 4;      // GRAM / POLY: also write gain2 * scale^2 * acc through mapOut2
struct Segment {
  CUtensorMap mapA;     // A operand, 128-row K-major boxes
  CUtensorMap mapB;     // B operand: K-major rows (GRAM, POLY), 64 x 64 MN-major boxes (COMBINE)
  CUtensorMap mapOut;   // output, 32 x 32 store boxes
  CUtensorMap mapOut2;  // second output of a SEG_DUAL segment (no diagonal shift)
  const float* scale;   // per-matrix s (GRAM applies s^2, COMBINE s), or nullptr
  int64_t tile_begin;   // first tile of this segment in the launch's queue
  int M;                // output rows (r)
  int N;                // output cols (r for GRAM/POLY, c for COMBINE)
  int K;                // reduction length (c for GRAM, r otherwise)
  int tiles_m;          // COMBINE: ceil(M / 256)
  int nb;               // GRAM/POLY: ceil(M / 256) super-blocks per side
  int tiles_per_mat;
  int out_z0;           // first matrix of the output map this segment writes
  int flags;            // SEG_*
  float gain, diag;     // GRAM / POLY: out = gain * (scale^2) * acc + diag * [i == j]
  float gain2;          // SEG_DUAL: gain of the second output
  const View* views;    // COMBINE: apply D to these views (by batch slot) instead of storing it
  int batch;            // matrices of this segment
  int reverse;          // visit the matrices last to first
};

struct GemmParams {
  Segment seg[MAX_SEGS];
  int nseg;
  int64_t total_tiles;
  float decay, eta;     // apply: W <- W * decay - eta * shape_scale * D
  int* err;
  uint64_t timeout_ns;
};
static_assert(sizeof(GemmParams) <= 4096, "kernel parameters above the 4 KB classic limit");

struct TileCoord {
  int mat;
  int m0;  // first output row of the pair's 256-row tile
  int n0;
  bool mirror;
};

// Segment holding queue tile `tile` (segments are stored in queue order).
__device__ __forceinline__ int seg_of(const GemmParams& p, int64_t tile) {
  int s = 0;
  while (s + 1 < p.nseg && tile >= p.seg[s + 1].tile_begin) ++s;
  return s;
}

// Tile `tile` of segment `p` (counted from the segment's first tile):
// (matrix, 256-row block, 256-column block).
template <int KIND>
__device__ __forceinline__ TileCoord tile_coord(const Segment& p, int64_t tile) {
  TileCoord t;
  t.mat = static_cast<int>(tile / p.tiles_per_mat);
  const int local = static_cast<int>(tile - static_cast<int64_t>(t.mat) * p.tiles_per_mat);
  if (p.reverse) t.mat = p.batch - 1 - t.mat;
  if (KIND == GEMM_COMBINE) {
    // m fastest: consecutive tiles share the same 256-column stripe of X.
    const int tm = local % p.tiles_m;
    const int tn = local / p.tiles_m;
    t.m0 = tm * PAIR_M;
    t.n0 = tn * BN;
    t.mirror = false;
  } else {
    // Upper-triangle super-block pairs (I <= J), row by row.
    int rem = local;
    int I = 0, rowlen = p.nb;
    while (rem >= rowlen) {
      rem -= rowlen;
      ++I;
      --rowlen;
    }
    const int J = I + rem;
    t.m0 = I * PAIR_M;
    t.n0 = J * BN;
    t.mirror = J > I;
  }
  return t;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

constexpr int EPI_CHUNKS = BN / 32;  // 32-column chunks per output row of a tile

__device__ __forceinline__ uint32_t stage_off(int row, int chunk) {
  return static_cast<uint32_t>(row * STAGE_ROW_BYTES + ((chunk ^ ((row >> 1) & 3)) << 4));
}

// ---- last round: D = X5 applied to W in the COMBINE epilogue -------------
// (the parameter update of the refresh, W <- W (1 - lr wd) - eta s D, with D
// the bf16 X5 as the separate update pass would read it). Each 32 x 32 chunk
// of X5 is staged in W's orientation (tall views transposed while staging),
// so both orientations update W the same way: 8 W rows x 128 contiguous bytes
// per instruction, each lane two float4 of one row. W is read and written
// with streaming (evict-first) hints, so that its 8 bytes per parameter do
// not push the operand tiles other pairs still re-read out of L2 (about 1 %
// off the update launches). A warp loads the W values
// of its first two chunks while the accumulator is computed, and those of
// chunk q + 2 right after using chunk q's, so each load has a whole chunk of
// work to hide behind.

struct ApplyTarget {
  float* dst;    // W, or the D output of a view without W (orthogonaliser only)
  int64_t ld;
  float step;    // eta * shape_scale
  bool tall;
  bool upd;      // dst is W (update) rather than D's output
  bool vec;      // 16-byte aligned rows
};

__device__ __forceinline__ ApplyTarget apply_target(const GemmParams& p, const View* views, int mat) {
  const View* v = views + mat;
  ApplyTarget t;
  float* W = v->W;
  t.upd = W != nullptr;
  t.dst = t.upd ? W : v->out;
  t.ld = v->ld;
  t.step = p.eta * v->shape_scale;
  t.tall = v->rows > v->cols;
  t.vec = (t.ld % 4 == 0) && ((reinterpret_cast<uintptr_t>(t.dst) & 15u) == 0);
  return t;
}

__device__ __forceinline__ float bf16_half(uint32_t word, int hi) {
  return __uint_as_float(hi ? (word & 0xFFFF0000u) : (word << 16));
}

// The chunk of X rows i0.., X columns j0.. in W's orientation: first row,
// first column and extents of W (wide: the same; tall: transposed).
struct ApplyBox {
  int r0, c0, R, C;
};

__device__ __forceinline__ ApplyBox apply_box(const ApplyTarget& t, int M, int N, int i0, int j0) {
  return t.tall ? ApplyBox{j0, i0, N, M} : ApplyBox{i0, j0, M, N};
}

// W values of the chunk, value 8 * it + e at W row b.r0 + 8 it + lane / 4,
// column b.c0 + 8 (lane % 4) + e. Out-of-range values are 0 and never stored.
__device__ __forceinline__ void apply_load(const ApplyTarget& t, const ApplyBox& b, int lane, float (&wv)[32]) {
  if (!t.upd) return;
  const int j = b.c0 + 8 * (lane & 3);
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int i = b.r0 + 8 * it + (lane >> 2);
    const float* row = t.dst + static_cast<int64_t>(i) * t.ld + j;
    if (i < b.R && t.vec && j + 8 <= b.C) {
      const float4 a = __ldcs(reinterpret_cast<const float4*>(row));  // read once: evict first
      const float4 c = __ldcs(reinterpret_cast<const float4*>(row + 4));
      wv[8 * it + 0] = a.x;
      wv[8 * it + 1] = a.y;
      wv[8 * it + 2] = a.z;
      wv[8 * it + 3] = a.w;
      wv[8 * it + 4] = c.x;
      wv[8 * it + 5] = c.y;
      wv[8 * it + 6] = c.z;
      wv[8 * it + 7] = c.w;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) wv[8 * it + e] = (i < b.R && j + e < b.C) ? row[e] : 0.f;
    }
  }
}

// W <- W decay - step D (or D itself for a view without W) over the chunk,
// D from the staged box (row = W row - b.r0, column = W column - b.c0).
__device__ __forceinline__ void apply_store(const GemmParams& p, const ApplyTarget& t, const ApplyBox& b, int lane,
                                            const float (&wv)[32], const uint8_t* box) {
  const int c4 = lane & 3;
  const int j = b.c0 + 8 * c4;
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int rho = 8 * it + (lane >> 2);
    const int i = b.r0 + rho;
    if (i >= b.R) continue;
    const uint4 u = *reinterpret_cast<const uint4*>(box + stage_off(rho, c4));
    const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
    float o[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float d = bf16_half(uw[e >> 1], e & 1);
      o[e] = t.upd ? fmaf(wv[8 * it + e], p.decay, -t.step * d) : d;
    }
    float* row = t.dst + static_cast<int64_t>(i) * t.ld + j;
    if (t.vec && j + 8 <= b.C) {
      __stcs(reinterpret_cast<float4*>(row), make_float4(o[0], o[1], o[2], o[3]));  // written once
      __stcs(reinterpret_cast<float4*>(row + 4), make_float4(o[4], o[5], o[6], o[7]));
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (j + e < b.C) row[e] = o[e];
    }
  }
}

// Stages one lane's 32 packed values (row `lane` of the box) and, for a
// mirrored tile, the transposed box, then issues their TMA stores. The
// warp's boxes are rewritten only after its previous stores have read them.
__device__ __forceinline__ void stage_and_store(const CUtensorMap* tm, uint8_t* stage, int lane, const uint32_t (&w)[16],
                                                bool mirror, bool rows_in, int i0, int j0, int z) {
  uint8_t* bd = stage;
  uint8_t* bm = stage + EPI_BUF_BYTES;
  if (lane == 0) bulk_wait_group_read<0>();
  __syncwarp();
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(bd + stage_off(lane, c)) = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
  if (mirror) {
    // Lower super-block (J, I): out[j][i] for this chunk's 32 columns j and
    // the warp's 32 rows i, staged transposed (box row = j).
#pragma unroll
    for (int k = 0; k < 32; ++k)
      *reinterpret_cast<uint16_t*>(bm + stage_off(k, lane >> 3) + (lane & 7) * 2) =
          static_cast<uint16_t>(w[k >> 1] >> ((k & 1) * 16));
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    if (rows_in) {
      tma_store_3d(tm, bd, j0, i0, z);
      if (mirror) tma_store_3d(tm, bm, i0, j0, z);
    }
    bulk_commit_group();
  }
}

// One tile's epilogue for this warp's 32 accumulator rows and its half of
// the columns (chunks qbase .. qbase + 3).
template <int KIND>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, const Segment& sg, const TileCoord& tc, int i,
                                              uint32_t t_row, uint8_t* stage, int lane, int qbase,
                                              const ApplyTarget& at, float (&weven)[32], float (&wodd)[32]) {
  const int i0 = i - lane;  // first output row of this warp
  float s = 1.f;
  if (KIND == GEMM_GRAM && sg.scale != nullptr) {
    const float q = sg.scale[tc.mat];
    s = q * q;
  }
  if (KIND == GEMM_COMBINE && sg.scale != nullptr) s = sg.scale[tc.mat];
  const float s2 = s * sg.gain2;  // SEG_DUAL
  if (KIND != GEMM_COMBINE) s *= sg.gain;
  const int z = sg.out_z0 + tc.mat;
  const bool rows_in = i0 < sg.M;  // warp-uniform
  const bool out16 = (sg.flags & SEG_OUT_FP16) != 0;
  const bool dual = KIND != GEMM_COMBINE && (sg.flags & SEG_DUAL) != 0;
  const bool apply = KIND == GEMM_COMBINE && sg.views != nullptr;
  const bool mirror = KIND != GEMM_COMBINE && tc.mirror;

#pragma unroll
  for (int qq = 0; qq < EPI_CHUNKS / 2; ++qq) {
    const int q = qbase + qq;
    const int j0 = tc.n0 + q * 32;
    if (j0 < sg.N) {  // uniform over the warp: depends on the tile only
      float v[32];
      tmem_load_32cols(t_row + static_cast<uint32_t>(q * 32), v);
      uint32_t w2[16];
      if (dual) {
#pragma unroll
        for (int h = 0; h < 16; ++h) w2[h] = pack_f16x2(v[2 * h] * s2, v[2 * h + 1] * s2);
      }
#pragma unroll
      for (int k = 0; k < 32; ++k) v[k] *= s;
      if (KIND != GEMM_COMBINE && j0 == i0) {  // the warp's 32 diagonal elements (warp-uniform)
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (k == lane) v[k] += sg.diag;
      }
      uint32_t w[16];
#pragma unroll
      for (int h = 0; h < 16; ++h)
        w[h] = out16 ? pack_f16x2(v[2 * h], v[2 * h + 1]) : pack_bf16x2(v[2 * h], v[2 * h + 1]);
      if (apply) {
        // D = X' from the staged box; this chunk's W values sit in the array
        // of its parity (loaded two chunks earlier, or before the
        // accumulator wait for the first two); once they are used, the array
        // takes the values two chunks ahead
        uint8_t* bd = stage;
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
        if (!at.tall) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            *reinterpret_cast<uint4*>(bd + stage_off(lane, c)) =
                make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
        } else {
          // W's orientation: box row k = X column j0 + k, this lane's X row
          // i0 + lane in box column `lane`
#pragma unroll
          for (int k = 0; k < 32; ++k)
            *reinterpret_cast<uint16_t*>(bd + stage_off(k, lane >> 3) + (lane & 7) * 2) =
                static_cast<uint16_t>(w[k >> 1] >> ((k & 1) * 16));
        }
        float(&wcur)[32] = (qq & 1) ? wodd : weven;
        __syncwarp();
        if (rows_in) apply_store(p, at, apply_box(at, sg.M, sg.N, i0, j0), lane, wcur, bd);
        if (qq + 2 < EPI_CHUNKS / 2) apply_load(at, apply_box(at, sg.M, sg.N, i0, j0 + 64), lane, wcur);
        __syncwarp();
        continue;
      }
      stage_and_store(&sg.mapOut, stage, lane, w, mirror, rows_in, i0, j0, z);
      if (dual) stage_and_store(&sg.mapOut2, stage, lane, w2, mirror, rows_in, i0, j0, z);
    }
  }
}

template <int KIND>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    ns_gemm_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_TILE_BYTES;
  uint8_t* sEpi = smem + STAGES * STAGE_BYTES;  // 1024-byte aligned
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(sEpi + EPI_SMEM_BYTES);
  uint64_t* empty_bar = full_bar + STAGES;
  uint64_t* tfull_bar = empty_bar + STAGES;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* drain_bar = tempty_bar + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs; 1: its peer
  const int64_t pair_id = blockIdx.x >> 1;
  const int64_t num_pairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);   // used in the even CTA: its producer's arrive + both CTAs' bytes
      mbar_init(&empty_bar[s], 1);  // one multicast commit per use
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], 2 * EPI_WARPS);  // even CTA: one arrival per epilogue warp of both CTAs
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_holder, TMEM_COLS);
    tmem_relinquish_pair();
  }
  // Both CTAs' barriers must exist before either signals the other.
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    if (lane == 0) {
      for (int q = 0; q < p.nseg; ++q) {
        tma_prefetch_desc(&p.seg[q].mapA);
        tma_prefetch_desc(&p.seg[q].mapB);
      }
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;
      bool ok = true;
      for (int64_t tile = pair_id; ok && tile < p.total_tiles; tile += num_pairs) {
        const Segment& sg = p.seg[seg_of(p, tile)];
        const TileCoord tc = tile_coord<KIND>(sg, tile - sg.tile_begin);
        const int num_kb = (sg.K + BK - 1) / BK;
        const int m_cta = tc.m0 + static_cast<int>(rank) * BM;
        const int n_cta = tc.n0 + static_cast<int>(rank) * BN_HALF;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_bounded(&empty_bar[stage], phase ^ 1u, abort_flag, p.err, p.timeout_ns)) {
            ok = false;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(&full_bar[stage], PAIR_STAGE_BYTES);
          const uint32_t bar = mapa_shared(smem_u32(&full_bar[stage]), 0);
          uint8_t* a_dst = sA + stage * A_TILE_BYTES;
          uint8_t* b_dst = sB + stage * B_TILE_BYTES;
          tma_load_3d_pair(a_dst, &sg.mapA, bar, kb * BK, m_cta, tc.mat);
          if (KIND == GEMM_COMBINE) {
#pragma unroll
            for (int q = 0; q < BN_HALF / 64; ++q)
              tma_load_3d_pair(b_dst + q * MN_CHUNK_BYTES, &sg.mapB, bar, n_cta + q * 64, kb * BK, tc.mat);
          } else {
            tma_load_3d_pair(b_dst, &sg.mapB, bar, kb * BK, n_cta, tc.mat);
          }
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && issued) {
        // Let every load already in flight land before the CTA exits. The
        // even CTA can watch its full barriers; the odd CTA's loads complete
        // on the peer's barrier, so it waits a fixed, ample time instead.
        if (rank == 0) {
          for (int s = 0; s < STAGES; ++s)
            if (issued & (1u << s)) wait_drain(&full_bar[s], (issued_parity >> s) & 1u, 50000000ull);
        } else {
          spin_for_ns(2000000ull);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      const uint32_t idesc_bf16 = idesc_f16kind_f32(PAIR_M, BN, false, KIND == GEMM_COMBINE, false);
      const uint32_t idesc_fp16 = idesc_f16kind_f32(PAIR_M, BN, false, KIND == GEMM_COMBINE, true);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, issued_any = false;
      for (int64_t tile = pair_id; ok && tile < p.total_tiles; tile += num_pairs) {
        const Segment& sg = p.seg[seg_of(p, tile)];
        const int num_kb = (sg.K + BK - 1) / BK;
        const uint32_t idesc = (sg.flags & SEG_IN_FP16) ? idesc_fp16 : idesc_bf16;
        if (!wait_bounded(&tempty_bar[acc], acc_phase ^ 1u, abort_flag, p.err, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_bounded(&full_bar[stage], phase, abort_flag, p.err, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a_addr = smem_u32(sA + stage * A_TILE_BYTES);
          const uint32_t b_addr = smem_u32(sB + stage * B_TILE_BYTES);
#pragma unroll
          for (int k = 0; k < BK / UK; ++k) {
            const uint64_t ad = smem_desc_sw128(a_addr + k * UK * 2, 16, 1024);
            const uint64_t bd = (KIND == GEMM_COMBINE)
                                    ? smem_desc_sw128(b_addr + k * UK * 128, MN_CHUNK_BYTES, 1024)
                                    : smem_desc_sw128(b_addr + k * UK * 2, 16, 1024);
            umma_bf16_pair(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
          }
          issued_any = true;
          umma_commit_pair_multicast(&empty_bar[stage], 0x3);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair_multicast(&tfull_bar[acc], 0x3);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok && issued_any) {
        // Let every MMA already issued finish before TMEM is released.
        umma_commit_pair_multicast(drain_bar, 0x1);
        wait_drain(drain_bar, 0, 50000000ull);
      }
    }
  } else {
    const int quarter = warp & 3;  // TMEM lanes [32 * quarter, 32 * quarter + 32) belong to this warp
    const int ew = warp - 2;                         // epilogue warp 0..7
    const int qbase = (ew >> 2) * (EPI_CHUNKS / 2);  // first 32-column chunk of this warp's half
    uint8_t* stage = sEpi + ew * EPI_WARP_BYTES;
    if (lane == 0)
      for (int q = 0; q < p.nseg; ++q) {
        tma_prefetch_desc(&p.seg[q].mapOut);
        if (p.seg[q].flags & SEG_DUAL) tma_prefetch_desc(&p.seg[q].mapOut2);
      }
    const uint32_t tempty_even = mapa_shared(smem_u32(&tempty_bar[0]), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int64_t tile = pair_id; tile < p.total_tiles; tile += num_pairs) {
      const Segment& sg = p.seg[seg_of(p, tile)];
      const TileCoord tc = tile_coord<KIND>(sg, tile - sg.tile_begin);
      const int i = tc.m0 + static_cast<int>(rank) * BM + quarter * 32 + lane;
      ApplyTarget at{};
      float weven[32], wodd[32];
      if (KIND == GEMM_COMBINE && sg.views != nullptr) {
        // the first two chunks' W values load while the accumulator is computed
        at = apply_target(p, sg.views, tc.mat);
        apply_load(at, apply_box(at, sg.M, sg.N, i - lane, tc.n0 + qbase * 32), lane, weven);
        apply_load(at, apply_box(at, sg.M, sg.N, i - lane, tc.n0 + qbase * 32 + 32), lane, wodd);
      }
      const bool got = wait_bounded(&tfull_bar[acc], acc_phase, abort_flag, p.err, p.timeout_ns);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after_sync();
      const uint32_t t_row = tmem_base + static_cast<uint32_t>(acc * BN) + (static_cast<uint32_t>(quarter * 32) << 16);
      epilogue_tile<KIND>(p, sg, tc, i, t_row, stage, lane, qbase, at, weven, wodd);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(tempty_even + static_cast<uint32_t>(acc * sizeof(uint64_t)));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // the staging boxes must stay valid until every issued store has run
    if (lane == 0) bulk_wait_group_all();
  }
  __syncwarp();
  // No CTA may leave (or free TMEM) while its peer can still touch its
  // barriers, shared memory or accumulators.
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 3-D bf16 tensor map over `batch` row-major matrices of rows x cols with row
// pitch ld (elements); box = box_inner x box_rows x 1. Loads use the 128-byte
// swizzle (out-of-range elements read as zero); the epilogue's 32 x 32 store
// boxes the 64-byte one (out-of-range elements are not written).
int encode_3d(CUtensorMap* map, const void* base, int batch, int64_t rows, int64_t cols, int64_t ld,
              uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return -1;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(batch)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * 2), static_cast<cuuint64_t>(rows * ld * 2)};
  cuuint32_t box[3] = {box_inner, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : static_cast<int>(r);
}

// How many CTA pairs of this kernel fit on the device at once (clusters
// must sit inside one GPC, so this can be below half the SM count).
template <int KIND>
int max_resident_pairs(int num_sms) {
  static std::atomic<int> cached[64];  // zero-initialised (static storage); races only repeat the query
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  const int known = cached[dev].load(std::memory_order_relaxed);
  if (known > 0) return known;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(num_sms & ~1));
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, ns_gemm_kernel<KIND>, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();  // clear the query's error state
    n = num_sms / 2;
  }
  cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

template <int KIND>
cudaError_t launch_kind(const GemmParams& p, int num_sms, cudaStream_t stream) {
  if (p.total_tiles == 0) return cudaSuccess;
  const int64_t pairs = std::min<int64_t>(p.total_tiles, max_resident_pairs<KIND>(num_sms));
  ns_gemm_kernel<KIND><<<static_cast<unsigned>(2 * pairs), NUM_THREADS, SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

// 2-D map over a row-major rows x cols matrix of fp32 or bf16 elements with
// row pitch ld (elements), box = box_cols x box_rows, no swizzle;
// out-of-range elements of a box read as zero.
int encode_rows_2d(CUtensorMap* map, const void* base, bool bf16_elems, int64_t rows, int64_t cols, int64_t ld,
                   uint32_t box_cols, uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return -1;
  const cuuint64_t esize = bf16_elems ? 2 : 4;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * esize};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, bf16_elems ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : static_cast<int>(r);
}

size_t gemm_smem_bytes() { return SMEM_BYTES; }

cudaError_t gemm_setup_attributes() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(ns_gemm_kernel<GEMM_GRAM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(SMEM_BYTES))) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(ns_gemm_kernel<GEMM_POLY>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(SMEM_BYTES))) != cudaSuccess)
    return e;
  return cudaFuncSetAttribute(ns_gemm_kernel<GEMM_COMBINE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(SMEM_BYTES));
}

int encode_x_maps(NsMaps* maps, const void* X, int batch, int64_t r, int64_t c, int64_t ldc) {
  int e;
  if ((e = encode_3d(&maps->x_rows128, X, batch, r, c, ldc, BK, BM)) != 0) return e;
  if ((e = encode_3d(&maps->x_k64, X, batch, r, c, ldc, 64, BK)) != 0) return e;
  return encode_3d(&maps->store, X, batch, r, c, ldc, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}

int encode_sym_maps(SymMaps* maps, const void* A, int batch, int64_t r, int64_t ldr) {
  int e;
  if ((e = encode_3d(&maps->rows128, A, batch, r, r, ldr, BK, BM)) != 0) return e;
  return encode_3d(&maps->store, A, batch, r, r, ldr, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}

cudaError_t launch_gemm(GemmKind kind, const GemmSegSpec* specs, int count, const GemmEpilogue& epi,
                        cudaStream_t stream) {
  // Longest tiles (largest K) first, so that the queue's last wave holds the
  // shortest ones.
  std::vector<int> order;
  for (int i = 0; i < count; ++i)
    if (specs[i].batch > 0) order.push_back(i);
  auto reduction = [&](const GemmSegSpec& g) { return kind == GEMM_GRAM ? g.c : g.r; };
  std::stable_sort(order.begin(), order.end(),
                   [&](int x, int y) { return reduction(specs[x]) > reduction(specs[y]); });
  for (size_t first = 0; first < order.size(); first += MAX_SEGS) {
    GemmParams p{};
    p.decay = epi.decay;
    p.eta = epi.eta;
    p.err = epi.err;
    p.timeout_ns = WAIT_LIMIT_NS;
    int64_t tiles = 0;
    for (size_t k = first; k < order.size() && p.nseg < MAX_SEGS; ++k) {
      const GemmSegSpec& g = specs[order[k]];
      Segment& sg = p.seg[p.nseg++];
      sg.mapA = *g.a;
      sg.mapB = *g.b;
      sg.mapOut = *g.out;
      if (g.out2 != nullptr) sg.mapOut2 = *g.out2;
      sg.scale = g.scale;
      sg.views = kind == GEMM_COMBINE ? g.views : nullptr;
      sg.flags = (g.in_fp16 ? SEG_IN_FP16 : 0) | (g.out_fp16 ? SEG_OUT_FP16 : 0) |
                 (kind != GEMM_COMBINE && g.out2 != nullptr ? SEG_DUAL : 0);
      sg.gain = g.gain;
      sg.diag = g.diag;
      sg.gain2 = g.gain2;
      sg.tile_begin = tiles;
      sg.out_z0 = g.out_z0;
      sg.batch = g.batch;
      sg.reverse = epi.reverse ? 1 : 0;
      if (kind == GEMM_COMBINE) {
        sg.M = static_cast<int>(g.r);
        sg.N = static_cast<int>(g.c);
        sg.K = static_cast<int>(g.r);
        sg.tiles_m = static_cast<int>((g.r + PAIR_M - 1) / PAIR_M);
        sg.nb = 0;
        sg.tiles_per_mat = sg.tiles_m * static_cast<int>((g.c + BN - 1) / BN);
      } else {
        sg.M = static_cast<int>(g.r);
        sg.N = static_cast<int>(g.r);
        sg.K = static_cast<int>(kind == GEMM_GRAM ? g.c : g.r);
        sg.tiles_m = 0;
        sg.nb = static_cast<int>((g.r + BN - 1) / BN);
        sg.tiles_per_mat = sg.nb * (sg.nb + 1) / 2;  // upper-triangle 256 x 256 super-blocks
      }
      tiles += static_cast<int64_t>(sg.tiles_per_mat) * g.batch;
    }
    p.total_tiles = tiles;
    cudaError_t e = kind == GEMM_GRAM   ? launch_kind<GEMM_GRAM>(p, epi.num_sms, stream)
                    : kind == GEMM_POLY ? launch_kind<GEMM_POLY>(p, epi.num_sms, stream)
                                        : launch_kind<GEMM_COMBINE>(p, epi.num_sms, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace prm
