// RowNorm step of Periodic Row-wise Muon (non-refresh steps), memory bound.
//
// "Scaling Muon for Diffusion Transformers", PaperDaily walkthrough, section
// "Periodic Row-wise Muon", Fig. 3 / Fig. 4: on steps with t % K != 0 the
// direction is gamma * R_eps(M_t), where R_eps divides each short-side vector
// by max(||v||_2, eps). Section "Distributed co-design", Fig. 8: for a tall
// matrix (m > n) the statistics are per-column sums of squares.
//
// Per element the step is
//   M <- beta * M + G ;  D = M / max(||v||, eps) ;  W <- W * (1 - lr wd) - eta s D
// with eta = lr * gamma. Algorithmic traffic: G read (2 B bf16), M read and
// written (8 B), W read and written (8 B) = 18 B per parameter.
//
// Wide matrices: one CTA per row, the updated momentum row kept in registers
// between the sum of squares and the update, so every byte moves once.
// Tall matrices: columns span the whole matrix, so the update has to wait for
// a pass over all rows: (1) momentum update + per-row-block column partial
// sums, (2) per-column inverse norms, (3) update reading M again. One launch
// pipelines the three over column stripes so that (3) reads M back from L2
// (16-byte aligned views with cols % 4 == 0); otherwise three launches.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace prm {
namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int THREADS>
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < THREADS / 32 ? red[lane] : 0.f;
    v = warp_sum(v);
    if (lane == 0) red[32] = v;
  }
  __syncthreads();
  return red[32];
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

template <bool BF16>
__device__ __forceinline__ float4 load_grad4(const void* G, int64_t off) {
  if (BF16) {
    const uint2 u = __ldcs(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(G) + off));
    return make_float4(bf16_bits_to_float(u.x & 0xFFFFu), bf16_bits_to_float(u.x >> 16),
                       bf16_bits_to_float(u.y & 0xFFFFu), bf16_bits_to_float(u.y >> 16));
  } else {
    return __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(G) + off));
  }
}

template <bool BF16>
__device__ __forceinline__ float load_grad1(const void* G, int64_t off) {
  if (BF16) return bf16_bits_to_float(static_cast<const uint16_t*>(G)[off]);
  return static_cast<const float*>(G)[off];
}

// ------------------------------------------------------------ wide rows
// Bulk prefetch of `bytes` (multiple of 16, 16-byte aligned) into L2.

// One CTA per row; each thread keeps NV float4 (or 4*NV floats) of the
// updated momentum in registers across the block reduction. Short rows also
// hold W in registers (its loads overlap the momentum pass); long rows
// (PREFETCH_W) instead have the W row pulled into L2 by one bulk prefetch at
// the start and read after the reduction, which keeps registers -- and so
// rows in flight per SM -- at the level short rows get.
template <int THREADS, int NV, bool BF16, bool VEC, bool PREFETCH_W = false>
__global__ void __launch_bounds__(THREADS) rownorm_wide_kernel(const View* __restrict__ views, int64_t cols,
                                                               StepScalars s) {
  __shared__ float red[33];
  const View v = views[blockIdx.y];
  const int64_t row = blockIdx.x;
  float* Mr = v.M + row * v.ld;
  float* Wr = v.W + row * v.ld;
  const int64_t goff = row * v.ld;
  float ss = 0.f;
  if constexpr (VEC) {
    float4 m[NV], w[PREFETCH_W ? 1 : NV];
    if constexpr (PREFETCH_W) {
      if (threadIdx.x == 0) prefetch_l2_bulk(Wr, static_cast<uint32_t>(cols * 4));
    }
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int64_t c = (static_cast<int64_t>(k) * THREADS + threadIdx.x) * 4;
      if (c < cols) {
        const float4 g = load_grad4<BF16>(v.G, goff + c);
        float4 mm = __ldcs(reinterpret_cast<const float4*>(Mr + c));
        mm.x = fmaf(s.beta, mm.x, g.x);
        mm.y = fmaf(s.beta, mm.y, g.y);
        mm.z = fmaf(s.beta, mm.z, g.z);
        mm.w = fmaf(s.beta, mm.w, g.w);
        __stcs(reinterpret_cast<float4*>(Mr + c), mm);
        ss = fmaf(mm.x, mm.x, ss);
        ss = fmaf(mm.y, mm.y, ss);
        ss = fmaf(mm.z, mm.z, ss);
        ss = fmaf(mm.w, mm.w, ss);
        m[k] = mm;
        if constexpr (!PREFETCH_W) w[k] = __ldcs(reinterpret_cast<const float4*>(Wr + c));
      }
    }
    const float total = block_sum<THREADS>(ss, red);
    const float coef = s.eta * v.shape_scale / fmaxf(sqrtf(total), s.eps);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int64_t c = (static_cast<int64_t>(k) * THREADS + threadIdx.x) * 4;
      if (c < cols) {
        float4 ww;
        if constexpr (PREFETCH_W)
          ww = __ldcs(reinterpret_cast<const float4*>(Wr + c));
        else
          ww = w[PREFETCH_W ? 0 : k];
        ww.x = fmaf(ww.x, s.decay, -coef * m[k].x);
        ww.y = fmaf(ww.y, s.decay, -coef * m[k].y);
        ww.z = fmaf(ww.z, s.decay, -coef * m[k].z);
        ww.w = fmaf(ww.w, s.decay, -coef * m[k].w);
        __stcs(reinterpret_cast<float4*>(Wr + c), ww);
      }
    }
  } else {
    constexpr int NE = 4 * NV;
    float m[NE], w[NE];
#pragma unroll
    for (int k = 0; k < NE; ++k) {
      const int64_t c = static_cast<int64_t>(k) * THREADS + threadIdx.x;
      if (c < cols) {
        const float mm = fmaf(s.beta, Mr[c], load_grad1<BF16>(v.G, goff + c));
        Mr[c] = mm;
        ss = fmaf(mm, mm, ss);
        m[k] = mm;
        w[k] = Wr[c];
      }
    }
    const float total = block_sum<THREADS>(ss, red);
    const float coef = s.eta * v.shape_scale / fmaxf(sqrtf(total), s.eps);
#pragma unroll
    for (int k = 0; k < NE; ++k) {
      const int64_t c = static_cast<int64_t>(k) * THREADS + threadIdx.x;
      if (c < cols) Wr[c] = fmaf(w[k], s.decay, -coef * m[k]);
    }
  }
}

// Rows too long for registers: two sweeps over the row (the second re-reads
// the freshly written momentum, mostly from L2).
template <bool BF16>
__global__ void __launch_bounds__(512) rownorm_wide_long_kernel(const View* __restrict__ views, int64_t cols,
                                                                StepScalars s) {
  __shared__ float red[33];
  const View v = views[blockIdx.y];
  const int64_t row = blockIdx.x;
  float* Mr = v.M + row * v.ld;
  float* Wr = v.W + row * v.ld;
  const int64_t goff = row * v.ld;
  float ss = 0.f;
  for (int64_t c = threadIdx.x; c < cols; c += 512) {
    const float mm = fmaf(s.beta, Mr[c], load_grad1<BF16>(v.G, goff + c));
    Mr[c] = mm;
    ss = fmaf(mm, mm, ss);
  }
  const float total = block_sum<512>(ss, red);
  const float coef = s.eta * v.shape_scale / fmaxf(sqrtf(total), s.eps);
  for (int64_t c = threadIdx.x; c < cols; c += 512) Wr[c] = fmaf(Wr[c], s.decay, -coef * Mr[c]);
}

// ------------------------------------------------------------ tall columns
constexpr int TALL_TX = 32;   // threads along a row
constexpr int TALL_TY = 8;    // thread rows
constexpr int TALL_RB = 256;  // rows per row block

// Phase 1: M <- beta M + G over a (TALL_RB rows) x (32 * VW columns) block,
// column partial sums of M^2 written to partials[view][row_block][col].
template <bool BF16, bool VEC>
__global__ void __launch_bounds__(TALL_TX* TALL_TY) tall_phase1_kernel(const View* __restrict__ views,
                                                                       int64_t rows, int64_t cols, float beta,
                                                                       float* __restrict__ partials,
                                                                       int64_t row_blocks) {
  constexpr int VW = VEC ? 4 : 1;
  __shared__ float red[TALL_TY][TALL_TX * VW + 1];
  const View v = views[blockIdx.z];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int64_t c = static_cast<int64_t>(blockIdx.x) * (TALL_TX * VW) + tx * VW;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * TALL_RB;
  const int64_t r1 = (r0 + TALL_RB < rows) ? r0 + TALL_RB : rows;
  float acc[VW];
#pragma unroll
  for (int k = 0; k < VW; ++k) acc[k] = 0.f;
  if (c < cols) {
    for (int64_t r = r0 + ty; r < r1; r += TALL_TY) {
      float* Mp = v.M + r * v.ld + c;
      if constexpr (VEC) {
        const float4 g = load_grad4<BF16>(v.G, r * v.ld + c);
        float4 mm = *reinterpret_cast<const float4*>(Mp);
        mm.x = fmaf(beta, mm.x, g.x);
        mm.y = fmaf(beta, mm.y, g.y);
        mm.z = fmaf(beta, mm.z, g.z);
        mm.w = fmaf(beta, mm.w, g.w);
        *reinterpret_cast<float4*>(Mp) = mm;
        acc[0] = fmaf(mm.x, mm.x, acc[0]);
        acc[1] = fmaf(mm.y, mm.y, acc[1]);
        acc[2] = fmaf(mm.z, mm.z, acc[2]);
        acc[3] = fmaf(mm.w, mm.w, acc[3]);
      } else {
        const float mm = fmaf(beta, *Mp, load_grad1<BF16>(v.G, r * v.ld + c));
        *Mp = mm;
        acc[0] = fmaf(mm, mm, acc[0]);
      }
    }
  }
#pragma unroll
  for (int k = 0; k < VW; ++k) red[ty][tx * VW + k] = acc[k];
  __syncthreads();
  // Column sums over the TALL_TY thread rows, in a fixed order.
  for (int col = ty * TALL_TX + tx; col < TALL_TX * VW; col += TALL_TX * TALL_TY) {
    float sum = 0.f;
#pragma unroll
    for (int y = 0; y < TALL_TY; ++y) sum += red[y][col];
    const int64_t cc = static_cast<int64_t>(blockIdx.x) * (TALL_TX * VW) + col;
    if (cc < cols) partials[(static_cast<int64_t>(blockIdx.z) * row_blocks + blockIdx.y) * cols + cc] = sum;
  }
}

// Phase 2: inv[view][col] = 1 / max(sqrt(sum over row blocks), eps).
__global__ void __launch_bounds__(256) tall_inv_kernel(const float* __restrict__ partials, int64_t row_blocks,
                                                       int64_t cols, float eps, float* __restrict__ inv) {
  const int64_t c = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
  if (c >= cols) return;
  const float* p = partials + static_cast<int64_t>(blockIdx.y) * row_blocks * cols + c;
  float sum = 0.f;
  for (int64_t b = 0; b < row_blocks; ++b) sum += p[b * cols];
  inv[static_cast<int64_t>(blockIdx.y) * cols + c] = 1.f / fmaxf(sqrtf(sum), eps);
}

// Phase 3: W <- W * decay - eta * s * M * inv[col].
template <bool VEC>
__global__ void __launch_bounds__(TALL_TX* TALL_TY) tall_update_kernel(const View* __restrict__ views,
                                                                       int64_t rows, int64_t cols,
                                                                       const float* __restrict__ inv,
                                                                       float decay, float eta) {
  constexpr int VW = VEC ? 4 : 1;
  const View v = views[blockIdx.z];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int64_t c = static_cast<int64_t>(blockIdx.x) * (TALL_TX * VW) + tx * VW;
  if (c >= cols) return;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * TALL_RB;
  const int64_t r1 = (r0 + TALL_RB < rows) ? r0 + TALL_RB : rows;
  const float* iv = inv + static_cast<int64_t>(blockIdx.z) * cols + c;
  const float step = eta * v.shape_scale;
  if constexpr (VEC) {
    const float4 q = *reinterpret_cast<const float4*>(iv);
    const float4 k = make_float4(step * q.x, step * q.y, step * q.z, step * q.w);
    for (int64_t r = r0 + ty; r < r1; r += TALL_TY) {
      const float4 mm = *reinterpret_cast<const float4*>(v.M + r * v.ld + c);
      float4* Wp = reinterpret_cast<float4*>(v.W + r * v.ld + c);
      float4 ww = *Wp;
      ww.x = fmaf(ww.x, decay, -k.x * mm.x);
      ww.y = fmaf(ww.y, decay, -k.y * mm.y);
      ww.z = fmaf(ww.z, decay, -k.z * mm.z);
      ww.w = fmaf(ww.w, decay, -k.w * mm.w);
      *Wp = ww;
    }
  } else {
    const float k = step * iv[0];
    for (int64_t r = r0 + ty; r < r1; r += TALL_TY) {
      float* Wp = v.W + r * v.ld + c;
      *Wp = fmaf(*Wp, decay, -k * v.M[r * v.ld + c]);
    }
  }
}

// ------------------------------------------------- tall columns, fused
// The same step in one launch, moving 18 B per parameter. Work splits into
// stripes of FT_COLS columns of one view and tiles of FT_TILE_ROWS rows of a
// stripe. Phase-1 tiles (momentum update + column partial sums of M^2) and
// phase-3 tiles (the update) are claimed by persistent CTAs from one queue
// in the order
//   P1(0) .. P1(D-1), P1(D) P3(0), P1(D+1) P3(1), .., P1(S-1) P3(S-1-D),
//   P3(S-D) .. P3(S-1)          (Pk(s): the tiles of stripe s)
// so a stripe's momentum is read back by its update D stripes after it was
// written, from L2 rather than HBM: D just covers the resident CTAs' window
// on the queue (1.3B-shaped set: 10 - 11 stripes of 4 MB), and the momentum is
// stored with an evict-last L2 policy while G and W stream through
// evict-first. The phase-1 tile that completes a stripe (the last one to
// count itself on the stripe's counter) sums the stripe's partials in a
// fixed order and publishes its inverse column norms; phase-3 tiles wait for
// that flag. A phase-3 tile waits only for tiles claimed before it, by CTAs
// that wait for nothing, so the queue always drains; the wait is bounded
// anyway. Measured on 24 x 8192 x 2048 (bf16 G): 1.24 ms per step against
// 1.43 ms for the three-launch form, DRAM traffic 7.26 GB (algorithmic
// 7.25) against 8.76.
constexpr int FT_THREADS = 512;
constexpr int FT_COLS = 128;                 // columns per stripe
constexpr int FT_CX = FT_COLS / 4;           // threads along a row, a float4 each
constexpr int FT_TY = FT_THREADS / FT_CX;    // thread rows
constexpr int FT_RPT = 4;                    // rows per thread in a register tile
constexpr int FT_ROWS = FT_TY * FT_RPT;      // rows per register tile
constexpr int FT_SUB = 4;                    // register tiles per queue tile
constexpr int FT_TILE_ROWS = FT_ROWS * FT_SUB;
constexpr int FT_RED = FT_THREADS / FT_COLS;  // threads per column in a stripe's final reduction
static_assert(FT_THREADS % FT_CX == 0 && FT_COLS <= FT_THREADS && FT_THREADS % FT_COLS == 0,
              "stripe width and block shape");
constexpr int FT_CTAS_PER_SM = 2;  // 64 registers per thread: two 512-thread CTAs per SM
constexpr int FT_LAG_MUL = 1;      // D = FT_LAG_MUL * ceil(resident CTAs / tiles per stripe) + 1
// The ring form runs two CTAs per SM with three stages each, and a lag of
// exactly one window of them, D = ceil(resident CTAs / tiles per stripe): a
// longer lag lets fewer update tiles wait for their stripe's norms but keeps
// more momentum live in L2 than it holds (24 tall 8192 x 2048 matrices:
// 1.117 against 1.120 ms with one stripe more, and each further stripe
// slower again; 8 of 20480 x 5120: 2.486 against 2.525 ms with one more and
// 2.580 with two more).
constexpr int RG_LAG_MUL = 1;
constexpr int RG_LAG_ADD = 0;  // the register form adds one stripe
constexpr int RG_CTAS_PER_SM = 2;
constexpr uint64_t FT_WAIT_LIMIT_NS = 2000000000ull;

struct FusedTall {
  const View* views;
  int64_t rows, cols;
  int spv;           // stripes per view
  int S;             // stripes
  int R;             // tiles per stripe
  int D;             // lag of a stripe's update behind its phase 1, in stripes (1 <= D <= S)
  int total;         // tiles in the queue: 2 S R
  float beta, decay, eta, eps;
  float* partials;   // [S][R][FT_COLS]
  float* inv;        // [S][FT_COLS]
  unsigned long long* claim;  // queue position
  int* counters;     // [S] phase-1 tiles done
  int* ready;        // [S] inverse norms published
  int* err;
  int withhold;      // test aid: stripe whose norms are not published (-1: none)
  uint64_t wait_ns;  // limit of one update tile's wait
  const CUtensorMap* maps;  // ring form: per view the maps of M, G and W
};

// Queue position -> (phase 3?, stripe, row block); the queue holds fewer
// than 2^31 tiles (checked by the launcher), so 32-bit arithmetic suffices.
__device__ __forceinline__ void ft_decode(const FusedTall& a, int i, bool& p3, int& s, int& rb) {
  const int R = a.R;
  const int a_end = a.D * R;
  const int b_end = a_end + 2 * R * (a.S - a.D);
  if (i < a_end) {
    p3 = false;
    s = i / R;
    rb = i - s * R;
  } else if (i < b_end) {
    const int j = i - a_end, k = j / (2 * R), w = j - k * 2 * R;
    p3 = w >= R;
    s = p3 ? k : a.D + k;
    rb = p3 ? w - R : w;
  } else {
    const int j = i - b_end, q = j / R;
    p3 = true;
    s = a.S - a.D + q;
    rb = j - q * R;
  }
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int atom_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// L2 eviction-priority policies: the updated momentum is stored "evict last"
// so that the streams of G and W do not push it out of L2 before the
// stripe's update reads it back, and read back (and first read) "evict
// first".
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ float4 ld_cg_hint(const float* ptr, uint64_t policy) {
  float4 v;
  asm volatile("ld.global.cg.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(ptr), "l"(policy));
  return v;
}

__device__ __forceinline__ void st_hint(float* ptr, float4 v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(ptr), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w), "l"(policy)
               : "memory");
}

// Both phases run one code path: load M and a second operand (G in phase 1,
// W in phase 3), write one result (M, or W); only the column sums and the
// wait differ. Sharing the path keeps the register count of one phase.
template <bool BF16>
__global__ void __launch_bounds__(FT_THREADS, FT_CTAS_PER_SM) tall_fused_kernel(const FusedTall a) {
  __shared__ float red[FT_TY][FT_COLS];
  __shared__ int tile_sh;
  __shared__ int flag_sh;
  const int tx = threadIdx.x % FT_CX, ty = threadIdx.x / FT_CX;
  const uint64_t pol_first = l2_policy_evict_first(), pol_last = l2_policy_evict_last();
  // Thread 0 claims the next tile while the current one is processed, so the
  // atomic's round trip overlaps the tile's memory traffic. (Still no
  // deadlock: the lowest-numbered unfinished tile is always some CTA's
  // current tile, and everything it waits for is numbered lower.)
  unsigned long long next = 0;
  if (threadIdx.x == 0) next = atomicAdd(a.claim, 1ull);
  for (;;) {
    if (threadIdx.x == 0) {
      tile_sh = static_cast<int>(min(next, 0x7fffffffull));
      if (next < static_cast<unsigned long long>(a.total)) next = atomicAdd(a.claim, 1ull);
    }
    __syncthreads();
    const int tile = tile_sh;
    if (tile >= a.total) break;  // uniform
    bool p3;
    int s, rb;
    ft_decode(a, tile, p3, s, rb);
    const View* v = a.views + s / a.spv;
    const int64_t ld = v->ld;
    const int64_t c = static_cast<int64_t>(s % a.spv) * FT_COLS + tx * 4;
    const int64_t r0 = static_cast<int64_t>(rb) * FT_TILE_ROWS + ty;
    const bool col_in = c < a.cols;  // cols % 4 == 0: a float4 column group is in or out as a whole
    const int step = FT_TY * static_cast<int>(ld);  // the launcher checks FT_TILE_ROWS * ld < 2^31
    float4 k4 = make_float4(0.f, 0.f, 0.f, 0.f);
    bool go = true;
    if (p3) {
      // the stripe's inverse norms must be published before its M is read back
      if (threadIdx.x == 0) {
        bool ok = ld_acquire_gpu(a.ready + s) != 0;
        if (!ok) {
          const uint64_t t0 = global_timer_ns();
          while (!(ok = ld_acquire_gpu(a.ready + s) != 0)) {
            if (global_timer_ns() - t0 > a.wait_ns) {
              atomicExch(a.err, DEV_ERR_TIMEOUT);
              break;
            }
            __nanosleep(200);
          }
        }
        flag_sh = ok;
      }
      __syncthreads();
      go = flag_sh != 0;
      if (go && col_in) {
        const float st = a.eta * v->shape_scale;
        const float4 q = __ldcg(reinterpret_cast<const float4*>(a.inv + static_cast<int64_t>(s) * FT_COLS + tx * 4));
        k4 = make_float4(st * q.x, st * q.y, st * q.z, st * q.w);
      }
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    // FT_SUB register tiles of FT_ROWS rows, one after the other; warps move
    // on independently (no barrier between them)
#pragma unroll 1
    for (int sub = 0; sub < FT_SUB && go && col_in; ++sub) {
      const int64_t rs = r0 + static_cast<int64_t>(sub) * FT_ROWS;
      if (rs >= a.rows) break;
      // rows rs, rs + FT_TY, ... below `rows`: the first nk of FT_RPT
      const int64_t left = (a.rows - rs + FT_TY - 1) / FT_TY;
      const int nk = left < FT_RPT ? static_cast<int>(left) : FT_RPT;
      const int64_t off0 = rs * ld + c;
      float* const mrow = v->M + off0;
      float* const wrow = v->W + off0;
      float4 mm[FT_RPT], bb[FT_RPT];
#pragma unroll
      for (int k = 0; k < FT_RPT; ++k) {
        if (k < nk) {
          mm[k] = ld_cg_hint(mrow + k * step, pol_first);
          bb[k] = p3 ? __ldcs(reinterpret_cast<const float4*>(wrow + k * step))
                     : load_grad4<BF16>(v->G, off0 + k * step);
        }
      }
#pragma unroll
      for (int k = 0; k < FT_RPT; ++k) {
        if (k < nk) {
          const float4 m = mm[k], b = bb[k];
          float4 o;
          if (!p3) {  // M <- beta M + G
            o.x = fmaf(a.beta, m.x, b.x);
            o.y = fmaf(a.beta, m.y, b.y);
            o.z = fmaf(a.beta, m.z, b.z);
            o.w = fmaf(a.beta, m.w, b.w);
            acc.x = fmaf(o.x, o.x, acc.x);
            acc.y = fmaf(o.y, o.y, acc.y);
            acc.z = fmaf(o.z, o.z, acc.z);
            acc.w = fmaf(o.w, o.w, acc.w);
            st_hint(mrow + k * step, o, pol_last);  // kept in L2 for phase 3
          } else {  // W <- W decay - eta s M / norm
            o.x = fmaf(b.x, a.decay, -k4.x * m.x);
            o.y = fmaf(b.y, a.decay, -k4.y * m.y);
            o.z = fmaf(b.z, a.decay, -k4.z * m.z);
            o.w = fmaf(b.w, a.decay, -k4.w * m.w);
            __stcs(reinterpret_cast<float4*>(wrow + k * step), o);
          }
        }
      }
    }
    if (!p3) {
      red[ty][tx * 4 + 0] = acc.x;
      red[ty][tx * 4 + 1] = acc.y;
      red[ty][tx * 4 + 2] = acc.z;
      red[ty][tx * 4 + 3] = acc.w;
      __syncthreads();
      if (threadIdx.x < FT_COLS) {
        float sum = 0.f;
#pragma unroll
        for (int y = 0; y < FT_TY; ++y) sum += red[y][threadIdx.x];
        a.partials[(static_cast<int64_t>(s) * a.R + rb) * FT_COLS + threadIdx.x] = sum;
      }
      // Release: the barrier orders every thread's M and partial stores
      // before thread 0's count, an acquire-release atomic (whose acquire,
      // for the stripe's last tile, takes in the other tiles' partials).
      __syncthreads();
      if (threadIdx.x == 0) flag_sh = atom_add_acq_rel_gpu(a.counters + s, 1) == a.R - 1;
      __syncthreads();
      if (flag_sh) {
        // The stripe's last phase-1 tile: inverse column norms. Every thread
        // sums the partials of one column over every FT_RED-th row block
        // (FT_RED threads per column, loads issued ahead), then one thread
        // per column adds those FT_RED sums: a fixed order, so the result
        // is the same whichever tile comes last. The stripe's updates wait
        // for this, so it must be short.
        const int col = threadIdx.x % FT_COLS, q = threadIdx.x / FT_COLS;
        const float* p = a.partials + (static_cast<int64_t>(s) * a.R + q) * FT_COLS + col;
        float sum = 0.f;
#pragma unroll 8
        for (int b = q; b < a.R; b += FT_RED, p += FT_RED * FT_COLS) sum += __ldcg(p);
        reinterpret_cast<float*>(red)[threadIdx.x] = sum;
        __syncthreads();
        if (threadIdx.x < FT_COLS) {
          float tot = 0.f;
#pragma unroll
          for (int k = 0; k < FT_RED; ++k) tot += reinterpret_cast<float*>(red)[k * FT_COLS + threadIdx.x];
          a.inv[static_cast<int64_t>(s) * FT_COLS + threadIdx.x] = 1.f / fmaxf(sqrtf(tot), a.eps);
        }
        __syncthreads();
        if (threadIdx.x == 0 && s != a.withhold) st_release_gpu(a.ready + s, 1);
      }
    }
    __syncthreads();  // tile_sh, flag_sh and red are rewritten by the next tile
  }
}

// ------------------------------------------ tall columns, fused, TMA ring
// The same queue of phase-1 / phase-3 tiles and the same stripe protocol as
// tall_fused_kernel, with the loads and the stripe bookkeeping moved off the
// compute warps. Two CTAs per SM, each with
//   warp 0     : producer -- claims tiles one at a time, waits for a phase-3
//                tile's stripe norms, and streams each tile into a ring of
//                shared-memory stages with TMA tensor loads (a 128-column x
//                32-row box of M and one of G or W per stage, three stages
//                per CTA: up to ~200 KB of loads in flight per SM from two
//                independent producers). Claiming the next tile ahead was
//                slower: a claimed phase-1 tile then waits behind its CTA's
//                phase-3 wait, and the stripe it belongs to with it;
//   warps 1..8 : consumers -- update M or W from the staged rows and store
//                the results; at the end of a phase-1 tile they leave their
//                column partial sums in one of two shared-memory slots and
//                move on to the next stage at once;
//   warp 9     : publisher -- per finished phase-1 tile: the tile's column
//                partials to global memory, the stripe's counter, and for the
//                stripe's last tile its inverse norms and ready flag.
// Every handoff is an mbarrier with a bounded wait, so a stalled pipeline
// returns instead of hanging. Each stage's metadata carries the destination
// pointer, row pitch and step size, so the consumers read nothing but shared
// memory before their stores. A phase-3 tile's loads of M are issued only
// after its stripe's inverse norms are published (acquire, then a proxy
// fence, so that the tensor loads see the momentum other CTAs stored). The
// maps need 16-byte row pitches: cols % 4 == 0, and cols % 8 == 0 with bf16
// gradients.
constexpr int RG_CONSUMER_WARPS = 8;
constexpr int RG_CONSUMERS = 32 * RG_CONSUMER_WARPS;
constexpr int RG_THREADS = 32 + RG_CONSUMERS + 32;
constexpr int RG_PUBLISHER_WARP = 1 + RG_CONSUMER_WARPS;
constexpr int RG_SR = 32;                              // rows per stage
constexpr int RG_STAGES = 3;
constexpr int RG_ROWS_PER_WARP = RG_SR / RG_CONSUMER_WARPS;  // 4
constexpr uint32_t RG_ROW_BYTES = FT_COLS * 4;         // 512 (fp32 box rows)
constexpr uint32_t RG_GROW_BYTES = FT_COLS * 2;        // 256 (bf16 box rows)
constexpr uint32_t RG_ARR_BYTES = RG_SR * RG_ROW_BYTES;  // 16 KB
constexpr uint32_t RG_STAGE_BYTES = 2 * RG_ARR_BYTES + FT_COLS * 4;  // M, G or W, inverse norms
constexpr int RG_KIND_P1 = 0, RG_KIND_P3 = 1, RG_KIND_DONE = 2;
constexpr int RG_RED_SLOTS = 2;
static_assert(FT_TILE_ROWS % RG_SR == 0, "a tile is a whole number of stages");
static_assert(FT_COLS == 4 * 32, "one float4 column group per consumer lane");

struct RgMeta {
  int kind, s, rb;
  int nrows;     // rows in the stage (the last stage of a ragged tile has fewer)
  int ncols;     // valid columns of the stripe (the ragged last stripe has fewer)
  int last;      // last stage of its tile
  int64_t ld;    // row pitch of the view
  float* dst;    // the stage's first row and column of M (phase 1) or W (phase 3)
  float step;    // phase 3: eta * shape_scale
  int pad;
};
struct RgRedMeta {
  int kind, s, rb, pad;
};
constexpr size_t RG_RED_BYTES = RG_RED_SLOTS * RG_CONSUMER_WARPS * FT_COLS * 4;
constexpr size_t RG_SMEM_BYTES = 128 + RG_STAGES * RG_STAGE_BYTES + RG_STAGES * sizeof(RgMeta) +
                                 (2 * RG_STAGES + 2 * RG_RED_SLOTS) * sizeof(uint64_t) + RG_RED_BYTES +
                                 RG_RED_SLOTS * sizeof(RgRedMeta) + 64;
static_assert(RG_SMEM_BYTES <= 232448, "ring above the 227 KB per-block limit");
static_assert(RG_CTAS_PER_SM * (RG_SMEM_BYTES + 1024) <= 233472, "two ring CTAs per SM");

__device__ __forceinline__ int shfl0(int v) { return __shfl_sync(0xffffffffu, v, 0); }

__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

template <bool BF16>
__global__ void __launch_bounds__(RG_THREADS, RG_CTAS_PER_SM) tall_ring_kernel(const FusedTall a) {
  extern __shared__ uint8_t rg_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(rg_raw) + 127) & ~uintptr_t(127));
  uint8_t* stages = base;
  RgMeta* meta = reinterpret_cast<RgMeta*>(base + RG_STAGES * RG_STAGE_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(meta + RG_STAGES);
  uint64_t* empty = full + RG_STAGES;
  uint64_t* red_full = empty + RG_STAGES;    // a slot's partials written (one arrival per consumer warp)
  uint64_t* red_free = red_full + RG_RED_SLOTS;  // a slot read by the publisher
  float* red = reinterpret_cast<float*>(red_free + RG_RED_SLOTS);  // [slot][warp][FT_COLS]
  RgRedMeta* red_meta = reinterpret_cast<RgRedMeta*>(red + RG_RED_SLOTS * RG_CONSUMER_WARPS * FT_COLS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(red_meta + RG_RED_SLOTS);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int k = 0; k < RG_STAGES; ++k) {
      mbar_init(&full[k], 1);
      mbar_init(&empty[k], RG_CONSUMER_WARPS);
    }
    for (int k = 0; k < RG_RED_SLOTS; ++k) {
      mbar_init(&red_full[k], RG_CONSUMER_WARPS);
      mbar_init(&red_free[k], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ---- producer: claim tiles, wait for phase-3 flags, stream rows in
    const uint64_t pol_first = l2_policy_evict_first();
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, issued_parity = 0;  // stages with copies in flight (for the abort drain)
    bool ok = true;
    // The claim of the next tile is in flight while the current one is
    // issued. (Still no deadlock: the lowest-numbered unfinished tile is the
    // one its CTA is working on -- a CTA's earlier tiles are lower -- and
    // everything it waits for is numbered lower.)
    for (;;) {
      int tile = 0;
      if (lane == 0) tile = static_cast<int>(min(atomicAdd(a.claim, 1ull), 0x7fffffffull));
      tile = shfl0(tile);
      if (tile >= a.total) break;
      bool p3;
      int s, rb;
      ft_decode(a, tile, p3, s, rb);
      const int view = s / a.spv;
      const int64_t c0 = static_cast<int64_t>(s % a.spv) * FT_COLS;
      const int ncols = static_cast<int>(a.cols - c0 < FT_COLS ? a.cols - c0 : FT_COLS);
      const int64_t row0 = static_cast<int64_t>(rb) * FT_TILE_ROWS;
      const int tile_rows = static_cast<int>(a.rows - row0 < FT_TILE_ROWS ? a.rows - row0 : FT_TILE_ROWS);
      float* dst0 = nullptr;
      int64_t ld = 0;
      float step = 0.f;
      if (lane == 0) {
        const View* v = a.views + view;
        ld = v->ld;
        dst0 = (p3 ? v->W : v->M) + c0;
        step = a.eta * v->shape_scale;
      }
      if (p3) {
        int go = 0;
        if (lane == 0) {
          bool got = ld_acquire_gpu(a.ready + s) != 0;
          if (!got) {
            const uint64_t t0 = global_timer_ns();
            while (!(got = ld_acquire_gpu(a.ready + s) != 0)) {
              if (global_timer_ns() - t0 > a.wait_ns) {
                atomicExch(a.err, DEV_ERR_TIMEOUT);
                break;
              }
              __nanosleep(200);
            }
          }
          if (got) fence_proxy_async_global();
          go = got ? 1 : 0;
        }
        if (!shfl0(go)) continue;  // the stripe's norms never came: its W stays as it was
      }
      const int nst = (tile_rows + RG_SR - 1) / RG_SR;
      for (int k = 0; k < nst && ok; ++k) {
        int got = 1;
        if (lane == 0) got = wait_bounded(&empty[stage], phase ^ 1u, abort_flag, a.err, FT_WAIT_LIMIT_NS) ? 1 : 0;
        if (!shfl0(got)) {
          ok = false;
          break;
        }
        const int nrows = min(RG_SR, tile_rows - k * RG_SR);
        const int64_t r0 = row0 + static_cast<int64_t>(k) * RG_SR;
        uint8_t* st = stages + static_cast<size_t>(stage) * RG_STAGE_BYTES;
        if (lane == 0) {
          RgMeta& m = meta[stage];
          m.kind = p3 ? RG_KIND_P3 : RG_KIND_P1;
          m.s = s;
          m.rb = rb;
          m.nrows = nrows;
          m.ncols = ncols;
          m.last = k == nst - 1;
          m.ld = ld;
          m.dst = dst0 + r0 * ld;
          m.step = step;
          // whole boxes land (rows or columns past the matrix read as zero)
          const uint32_t bbytes = p3 || !BF16 ? RG_ARR_BYTES : RG_SR * RG_GROW_BYTES;
          mbar_arrive_expect_tx(&full[stage], RG_ARR_BYTES + bbytes + (p3 ? FT_COLS * 4 : 0));
          const CUtensorMap* mp = a.maps + 3 * view;
          const int x = static_cast<int>(c0), y = static_cast<int>(r0);
          tma_load_2d_hint(st, mp, &full[stage], x, y, pol_first);
          tma_load_2d_hint(st + RG_ARR_BYTES, mp + (p3 ? 2 : 1), &full[stage], x, y, pol_first);
          if (p3)
            bulk_load_hint(st + 2 * RG_ARR_BYTES, a.inv + static_cast<int64_t>(s) * FT_COLS, FT_COLS * 4,
                           &full[stage], pol_first);
        }
        __syncwarp();
        issued |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == RG_STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
    }
    if (ok) {
      // tell the consumers that the queue is empty
      int got = 1;
      if (lane == 0) got = wait_bounded(&empty[stage], phase ^ 1u, abort_flag, a.err, FT_WAIT_LIMIT_NS) ? 1 : 0;
      if (shfl0(got) && lane == 0) {
        meta[stage].kind = RG_KIND_DONE;
        mbar_arrive(&full[stage]);
      }
    } else if (lane == 0) {
      // let every copy in flight land before the CTA's shared memory goes away
      for (int k = 0; k < RG_STAGES; ++k)
        if (issued & (1u << k)) wait_drain(&full[k], (issued_parity >> k) & 1u, 50000000ull);
    }
  } else if (warp < RG_PUBLISHER_WARP) {
    // ---- consumers: warp w takes rows w * 4 .. w * 4 + 3 of every stage
    const int w = warp - 1;
    const uint64_t pol_last = l2_policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    int ends = 0;  // phase-1 tile ends handed to the publisher
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    // Hands the tile end (partials in `acc`, or the end of the queue) to the
    // publisher through slot ends % 2, once the publisher has read that
    // slot's previous contents.
    auto hand_over = [&](int kind, int s, int rb) -> bool {
      const int slot = ends & 1, use = ends >> 1;
      if (use > 0) {
        int got = 1;
        if (lane == 0)
          got = wait_bounded(&red_free[slot], static_cast<uint32_t>(use - 1) & 1u, abort_flag, a.err,
                             FT_WAIT_LIMIT_NS) ? 1 : 0;
        if (!shfl0(got)) return false;
      }
      *reinterpret_cast<float4*>(red + (slot * RG_CONSUMER_WARPS + w) * FT_COLS + lane * 4) = acc;
      if (w == 0 && lane == 0) red_meta[slot] = RgRedMeta{kind, s, rb, 0};
      __syncwarp();
      if (lane == 0) mbar_arrive(&red_full[slot]);
      ++ends;
      return true;
    };
    for (;;) {
      int got = 1;
      if (lane == 0) got = wait_bounded(&full[stage], phase, abort_flag, a.err, FT_WAIT_LIMIT_NS) ? 1 : 0;
      if (!shfl0(got)) break;
      const RgMeta m = meta[stage];
      if (m.kind == RG_KIND_DONE) {
        hand_over(RG_KIND_DONE, 0, 0);
        break;
      }
      const bool p3 = m.kind == RG_KIND_P3;
      const bool col_in = lane * 4 < m.ncols;  // ncols % 4 == 0
      const uint8_t* st = stages + static_cast<size_t>(stage) * RG_STAGE_BYTES;
      float4 k4 = make_float4(0.f, 0.f, 0.f, 0.f);
      if (p3 && col_in) {
        const float4 q = *reinterpret_cast<const float4*>(st + 2 * RG_ARR_BYTES + lane * 16);
        k4 = make_float4(m.step * q.x, m.step * q.y, m.step * q.z, m.step * q.w);
      }
#pragma unroll
      for (int rr = 0; rr < RG_ROWS_PER_WARP; ++rr) {
        const int row = w * RG_ROWS_PER_WARP + rr;
        if (row < m.nrows && col_in) {
          const float4 mm = *reinterpret_cast<const float4*>(st + row * RG_ROW_BYTES + lane * 16);
          float* out = m.dst + row * m.ld + lane * 4;
          float4 o;
          if (!p3) {
            float4 g;
            if (BF16) {
              const uint2 u = *reinterpret_cast<const uint2*>(st + RG_ARR_BYTES + row * RG_GROW_BYTES + lane * 8);
              g = make_float4(bf16_bits_to_float(u.x & 0xFFFFu), bf16_bits_to_float(u.x >> 16),
                              bf16_bits_to_float(u.y & 0xFFFFu), bf16_bits_to_float(u.y >> 16));
            } else {
              g = *reinterpret_cast<const float4*>(st + RG_ARR_BYTES + row * RG_ROW_BYTES + lane * 16);
            }
            o.x = fmaf(a.beta, mm.x, g.x);
            o.y = fmaf(a.beta, mm.y, g.y);
            o.z = fmaf(a.beta, mm.z, g.z);
            o.w = fmaf(a.beta, mm.w, g.w);
            acc.x = fmaf(o.x, o.x, acc.x);
            acc.y = fmaf(o.y, o.y, acc.y);
            acc.z = fmaf(o.z, o.z, acc.z);
            acc.w = fmaf(o.w, o.w, acc.w);
            st_hint(out, o, pol_last);  // kept in L2 for the stripe's update
          } else {
            const float4 ww = *reinterpret_cast<const float4*>(st + RG_ARR_BYTES + row * RG_ROW_BYTES + lane * 16);
            o.x = fmaf(ww.x, a.decay, -k4.x * mm.x);
            o.y = fmaf(ww.y, a.decay, -k4.y * mm.y);
            o.z = fmaf(ww.z, a.decay, -k4.z * mm.z);
            o.w = fmaf(ww.w, a.decay, -k4.w * mm.w);
            __stcs(reinterpret_cast<float4*>(out), o);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (++stage == RG_STAGES) {
        stage = 0;
        phase ^= 1u;
      }
      if (p3 || !m.last) continue;
      // the end of a phase-1 tile: this warp's column partial sums (its rows
      // in order) go to the publisher, which adds the warps in order
      if (!hand_over(RG_KIND_P1, m.s, m.rb)) break;
      acc = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  } else {
    // ---- publisher: lane l owns columns 4 l .. 4 l + 3 of each stripe
    for (int k = 0;; ++k) {
      const int slot = k & 1;
      int got = 1;
      if (lane == 0)
        got = wait_bounded(&red_full[slot], static_cast<uint32_t>(k >> 1) & 1u, abort_flag, a.err,
                           FT_WAIT_LIMIT_NS) ? 1 : 0;
      if (!shfl0(got)) break;
      const RgRedMeta rm = red_meta[slot];
      if (rm.kind == RG_KIND_DONE) break;
      // the tile's column partials: the consumer warps' sums in warp order
      float4 sum = *reinterpret_cast<const float4*>(red + slot * RG_CONSUMER_WARPS * FT_COLS + lane * 4);
#pragma unroll
      for (int y = 1; y < RG_CONSUMER_WARPS; ++y)
        sum = add4(sum, *reinterpret_cast<const float4*>(red + (slot * RG_CONSUMER_WARPS + y) * FT_COLS + lane * 4));
      __syncwarp();
      if (lane == 0) mbar_arrive(&red_free[slot]);
      *reinterpret_cast<float4*>(a.partials + (static_cast<int64_t>(rm.s) * a.R + rm.rb) * FT_COLS + lane * 4) =
          sum;
      // The count is one acquire-release atomic: its release orders this
      // tile's momentum stores (which reached this warp through the slot's
      // mbarrier) and the lanes' partial stores (through __syncwarp) before
      // it; for the stripe's last tile its acquire takes in every earlier
      // tile's release along the counter's chain of atomics. (A GPU-scope
      // fence before the atomic and another after it took 2 % longer over
      // the step.)
      __syncwarp();
      int done = 0;
      if (lane == 0) done = atom_add_acq_rel_gpu(a.counters + rm.s, 1) == a.R - 1;
      __syncwarp();
      if (!shfl0(done)) continue;
      // The stripe's last phase-1 tile: inverse column norms. Per column the
      // partials of the even and of the odd row blocks, then their sum (a
      // fixed order, so the result is the same whichever tile comes last).
      // The stripe's updates wait for this, so the loads go out sixteen at a
      // time (eight at a time: 0.7 % slower over the step, a plain loop 3 %).
      const float* pp = a.partials + static_cast<int64_t>(rm.s) * a.R * FT_COLS + lane * 4;
      float4 e = make_float4(0.f, 0.f, 0.f, 0.f), o = e;
      int b = 0;
      for (; b + 16 <= a.R; b += 16) {
        float4 v[16];
#pragma unroll
        for (int u = 0; u < 16; ++u)
          v[u] = __ldcg(reinterpret_cast<const float4*>(pp + static_cast<int64_t>(b + u) * FT_COLS));
#pragma unroll
        for (int u = 0; u < 16; u += 2) {
          e = add4(e, v[u]);
          o = add4(o, v[u + 1]);
        }
      }
      for (; b < a.R; ++b) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(pp + static_cast<int64_t>(b) * FT_COLS));
        if (b & 1)
          o = add4(o, v);
        else
          e = add4(e, v);
      }
      const float4 t = add4(e, o);
      *reinterpret_cast<float4*>(a.inv + static_cast<int64_t>(rm.s) * FT_COLS + lane * 4) =
          make_float4(1.f / fmaxf(sqrtf(t.x), a.eps), 1.f / fmaxf(sqrtf(t.y), a.eps),
                      1.f / fmaxf(sqrtf(t.z), a.eps), 1.f / fmaxf(sqrtf(t.w), a.eps));
      __syncwarp();
      if (lane == 0 && rm.s != a.withhold) st_release_gpu(a.ready + rm.s, 1);
    }
  }
}

template <int THREADS, int NV, bool BF16>
cudaError_t launch_wide_t(const View* d_views, int count, int64_t rows, int64_t cols, bool vec_ok, StepScalars s,
                          cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(rows), static_cast<unsigned>(count));
  constexpr bool kPrefetch = NV >= 6;  // long rows: W via L2 prefetch instead of registers
  if (vec_ok)
    rownorm_wide_kernel<THREADS, NV, BF16, true, kPrefetch><<<grid, THREADS, 0, stream>>>(d_views, cols, s);
  else
    rownorm_wide_kernel<THREADS, NV, BF16, false><<<grid, THREADS, 0, stream>>>(d_views, cols, s);
  return cudaGetLastError();
}

template <bool BF16>
cudaError_t launch_wide_dispatch(const View* d_views, int count, int64_t rows, int64_t cols, bool vec_ok,
                                 StepScalars s, cudaStream_t stream) {
  const int64_t per = (cols + 3) / 4;  // float4 columns (or groups of 4 scalars)
  if (per <= 256 * 1) return launch_wide_t<256, 1, BF16>(d_views, count, rows, cols, vec_ok, s, stream);
  if (per <= 256 * 2) return launch_wide_t<256, 2, BF16>(d_views, count, rows, cols, vec_ok, s, stream);
  if (per <= 256 * 4) return launch_wide_t<256, 4, BF16>(d_views, count, rows, cols, vec_ok, s, stream);
  if (per <= 256 * 6) return launch_wide_t<256, 6, BF16>(d_views, count, rows, cols, vec_ok, s, stream);
  if (per <= 256 * 8) return launch_wide_t<256, 8, BF16>(d_views, count, rows, cols, vec_ok, s, stream);
  if (per <= 256 * 12) return launch_wide_t<256, 12, BF16>(d_views, count, rows, cols, vec_ok, s, stream);
  if (per <= 512 * 10) return launch_wide_t<512, 10, BF16>(d_views, count, rows, cols, vec_ok, s, stream);
  if (per <= 512 * 14) return launch_wide_t<512, 14, BF16>(d_views, count, rows, cols, vec_ok, s, stream);
  const dim3 grid(static_cast<unsigned>(rows), static_cast<unsigned>(count));
  rownorm_wide_long_kernel<BF16><<<grid, 512, 0, stream>>>(d_views, cols, s);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rownorm_wide(const View* d_views, int count, int64_t rows, int64_t cols, bool vec_ok,
                                bool grad_bf16, StepScalars s, cudaStream_t stream) {
  if (count == 0 || rows == 0) return cudaSuccess;
  return grad_bf16 ? launch_wide_dispatch<true>(d_views, count, rows, cols, vec_ok, s, stream)
                   : launch_wide_dispatch<false>(d_views, count, rows, cols, vec_ok, s, stream);
}

int64_t tall_row_blocks(int64_t rows) { return (rows + TALL_RB - 1) / TALL_RB; }

bool tall_fused_fits(int count, int64_t rows, int64_t cols) {
  const int64_t S = static_cast<int64_t>(count) * ((cols + FT_COLS - 1) / FT_COLS);
  const int64_t R = (rows + FT_TILE_ROWS - 1) / FT_TILE_ROWS;
  return 2 * S * R < (int64_t(1) << 31) - 1 && static_cast<int64_t>(FT_TILE_ROWS) * cols < (int64_t(1) << 31);
}

TallFusedScratch tall_fused_scratch(int count, int64_t rows, int64_t cols) {
  TallFusedScratch t;
  const int64_t S = static_cast<int64_t>(count) * ((cols + FT_COLS - 1) / FT_COLS);
  const int64_t R = (rows + FT_TILE_ROWS - 1) / FT_TILE_ROWS;
  t.partials_bytes = static_cast<size_t>(S * R * FT_COLS) * sizeof(float);
  t.inv_bytes = static_cast<size_t>(S * FT_COLS) * sizeof(float);
  t.flag_bytes = sizeof(unsigned long long) + static_cast<size_t>(2 * S) * sizeof(int);
  return t;
}

bool tall_ring_ok(int64_t cols, bool grad_bf16) {
  // TMA coordinates are 32-bit: rows below 2^31 are guaranteed by registration
  return cols % 4 == 0 && (!grad_bf16 || cols % 8 == 0);
}

int tall_ring_box_cols() { return FT_COLS; }
int tall_ring_box_rows() { return RG_SR; }

cudaError_t rownorm_setup_attributes() {
  cudaError_t e = cudaFuncSetAttribute(tall_ring_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(RG_SMEM_BYTES));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(tall_ring_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(RG_SMEM_BYTES));
}

cudaError_t launch_rownorm_tall_fused(const View* d_views, int count, int64_t rows, int64_t cols, bool grad_bf16,
                                      StepScalars s, float* partials, float* inv, void* flags, int* err,
                                      int num_sms, cudaStream_t stream, const CUtensorMap* ring_maps,
                                      int withhold_stripe, uint64_t wait_ns) {
  if (count == 0 || rows == 0) return cudaSuccess;
  const bool ring = ring_maps != nullptr;
  if (ring && !tall_ring_ok(cols, grad_bf16)) return cudaErrorInvalidValue;
  const TallFusedScratch t = tall_fused_scratch(count, rows, cols);
  FusedTall a{};
  a.views = d_views;
  a.rows = rows;
  a.cols = cols;
  a.spv = static_cast<int>((cols + FT_COLS - 1) / FT_COLS);
  a.S = count * a.spv;
  a.R = static_cast<int>((rows + FT_TILE_ROWS - 1) / FT_TILE_ROWS);
  if (!tall_fused_fits(count, rows, cols)) return cudaErrorInvalidValue;
  const int64_t total = 2 * static_cast<int64_t>(a.S) * a.R;
  a.total = static_cast<int>(total);
  const int64_t grid =
      std::min<int64_t>(total, static_cast<int64_t>(std::max(1, num_sms)) * (ring ? RG_CTAS_PER_SM : FT_CTAS_PER_SM));
  // the lag covers the CTAs' window on the queue, so updates rarely wait
  a.D = static_cast<int>(std::min<int64_t>(
      a.S, (ring ? RG_LAG_MUL : FT_LAG_MUL) * ((grid + a.R - 1) / a.R) + (ring ? RG_LAG_ADD : 1)));
  a.beta = s.beta;
  a.decay = s.decay;
  a.eta = s.eta;
  a.eps = s.eps;
  a.partials = partials;
  a.inv = inv;
  a.claim = static_cast<unsigned long long*>(flags);
  a.counters = reinterpret_cast<int*>(static_cast<char*>(flags) + sizeof(unsigned long long));
  a.ready = a.counters + a.S;
  a.err = err;
  a.withhold = withhold_stripe;
  a.maps = ring_maps;
  a.wait_ns = (wait_ns == 0 || wait_ns > FT_WAIT_LIMIT_NS) ? FT_WAIT_LIMIT_NS : wait_ns;
  cudaError_t e = cudaMemsetAsync(flags, 0, t.flag_bytes, stream);
  if (e != cudaSuccess) return e;
  if (ring) {
    if (grad_bf16)
      tall_ring_kernel<true><<<static_cast<unsigned>(grid), RG_THREADS, RG_SMEM_BYTES, stream>>>(a);
    else
      tall_ring_kernel<false><<<static_cast<unsigned>(grid), RG_THREADS, RG_SMEM_BYTES, stream>>>(a);
  } else if (grad_bf16) {
    tall_fused_kernel<true><<<static_cast<unsigned>(grid), FT_THREADS, 0, stream>>>(a);
  } else {
    tall_fused_kernel<false><<<static_cast<unsigned>(grid), FT_THREADS, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_rownorm_tall(const View* d_views, int count, int64_t rows, int64_t cols, bool vec_ok,
                                bool grad_bf16, StepScalars s, float* partials, float* inv,
                                cudaStream_t stream) {
  if (count == 0) return cudaSuccess;
  const int64_t rb = tall_row_blocks(rows);
  const int vw = vec_ok ? 4 : 1;
  const dim3 block(TALL_TX, TALL_TY);
  const dim3 grid(static_cast<unsigned>((cols + TALL_TX * vw - 1) / (TALL_TX * vw)), static_cast<unsigned>(rb),
                  static_cast<unsigned>(count));
  if (grad_bf16) {
    if (vec_ok)
      tall_phase1_kernel<true, true><<<grid, block, 0, stream>>>(d_views, rows, cols, s.beta, partials, rb);
    else
      tall_phase1_kernel<true, false><<<grid, block, 0, stream>>>(d_views, rows, cols, s.beta, partials, rb);
  } else {
    if (vec_ok)
      tall_phase1_kernel<false, true><<<grid, block, 0, stream>>>(d_views, rows, cols, s.beta, partials, rb);
    else
      tall_phase1_kernel<false, false><<<grid, block, 0, stream>>>(d_views, rows, cols, s.beta, partials, rb);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 igrid(static_cast<unsigned>((cols + 255) / 256), static_cast<unsigned>(count));
  tall_inv_kernel<<<igrid, 256, 0, stream>>>(partials, rb, cols, s.eps, inv);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (vec_ok)
    tall_update_kernel<true><<<grid, block, 0, stream>>>(d_views, rows, cols, inv, s.decay, s.eta);
  else
    tall_update_kernel<false><<<grid, block, 0, stream>>>(d_views, rows, cols, inv, s.decay, s.eta);
  return cudaGetLastError();
}

}  // namespace prm
