// NS5 for matrices whose short side r is below NS_SMALL_R (64), on CUDA
// cores in fp32 ("Scaling Muon for Diffusion Transformers", PaperDaily
// walkthrough, section "Periodic Row-wise Muon": on refresh steps the
// direction is five Newton-Schulz rounds of the momentum).
//
// Such matrices fill at most a quarter of the 256 x 256 tile edge of the
// tensor-core GEMMs, and they are where bf16 rounding hurts most: with r x c
// elements that few, the rounding errors of X, C and P do not average out
// and the quintic's slope (up to a = 3.44) carries them through five rounds.
// Here every round keeps X, A = X X^T and P = a I + b A + c A A in fp32,
// evaluated in the plain order of the iteration (no completed square, no
// Gram-space legs):
//
//   prep    : M <- beta M + G (in place), partial sums of A_raw = M M^T over
//             column chunks of the wide orientation
//   poly    : A = s^2 * sum of partials on round 0 (s = 1 / (||M||_F +
//             eps_ns), ||M||_F^2 = trace A_raw), else the plain sum;
//             P = a I + b A + c A A, times s on round 0 (X_0 = s M)
//   combine : X' = P X over each column chunk (round 0 reads M itself),
//             partial sums of X' X'^T for the next round; the last round
//             applies W <- W (1 - lr wd) - eta s D with D = X_5 instead.
//
// All sums run in a fixed order (per chunk, then chunks in index order), so
// the result does not depend on scheduling. X lives in the workspace in
// tile-major order: the r x NS_SMALL_TC values of one column tile
// contiguous, in the element order the tile is loaded in (columns fastest
// for wide views, rows fastest for tall ones), so that every tile moves as
// one coalesced block.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "internal.h"

namespace prm {
namespace {

constexpr int T = NS_SMALL_THREADS;  // 256
constexpr int TC = NS_SMALL_TC;      // columns (wide orientation) per tile
constexpr int LDS = TC + 1;          // shared-memory row pitch of a tile (bank spread)
constexpr int RMAX = NS_SMALL_R - 1; // largest short side on this path (63)
constexpr int PPT = (RMAX * (RMAX + 1) / 2 + T - 1) / T;  // pairs per thread, at most 8
constexpr int OPT = (RMAX * TC + T - 1) / T;              // outputs per thread in a combine, at most 16

__device__ __forceinline__ float grad_value(const void* G, int64_t off, bool bf16) {
  if (bf16) return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(G)[off]) << 16);
  return static_cast<const float*>(G)[off];
}

// Element e of a tile (0 <= e < r * TC) -> row k (short side) and column j
// (long side, within the tile), in the load order: columns fastest for wide
// views (consecutive threads read one storage row), rows fastest for tall
// views (consecutive threads read one storage row of the transposed matrix).
__device__ __forceinline__ void tile_elem(int e, int r, bool tall, int& k, int& j) {
  if (tall) {
    j = e / r;
    k = e - j * r;
  } else {
    k = e / TC;
    j = e - k * TC;
  }
}

// Storage offset of wide-orientation element (k, jj) of a view.
__device__ __forceinline__ int64_t view_off(const View& v, bool tall, int k, int64_t jj) {
  return tall ? jj * v.ld + k : static_cast<int64_t>(k) * v.ld + jj;
}

// Upper-triangle pair p (0 <= p < r (r + 1) / 2) -> (i, k), i <= k, row by row.
__device__ __forceinline__ void pair_ik(int p, int r, int& i, int& k) {
  int row = 0, len = r;
  while (p >= len) {
    p -= len;
    ++row;
    --len;
  }
  i = row;
  k = row + p;
}

// Thread layout of the Gram partial sums: `span` threads per group of
// columns, each thread summing up to PPT pairs (p = lt, lt + span, ...) over
// the columns j = jg, jg + groups, ... of every tile.
struct GramLane {
  int span, groups, jg, lt, npairs;
  int pi[PPT], pk[PPT];
  __device__ __forceinline__ void init(int r) {
    npairs = r * (r + 1) / 2;
    span = npairs < T ? npairs : T;
    groups = T / span;
    jg = threadIdx.x / span;
    lt = threadIdx.x - jg * span;
#pragma unroll
    for (int u = 0; u < PPT; ++u) {
      const int p = lt + u * span;
      if (jg < groups && p < npairs)
        pair_ik(p, r, pi[u], pk[u]);
      else
        pi[u] = pk[u] = -1;
    }
  }
  // acc[u] += sum over this thread's columns of xs[i][j] * xs[k][j]
  __device__ __forceinline__ void accumulate(const float* xs, float (&acc)[PPT]) const {
    if (jg >= groups) return;
    for (int j = jg; j < TC; j += groups) {
#pragma unroll
      for (int u = 0; u < PPT; ++u)
        if (pi[u] >= 0) acc[u] = fmaf(xs[pi[u] * LDS + j], xs[pk[u] * LDS + j], acc[u]);
    }
  }
  // Adds the column groups' sums in group order and writes the chunk's
  // partial for every pair. `red` holds at least T floats.
  __device__ __forceinline__ void store(const float (&acc)[PPT], float* red, float* out) const {
    if (groups == 1) {
#pragma unroll
      for (int u = 0; u < PPT; ++u)
        if (pi[u] >= 0) out[lt + u * span] = acc[u];
      return;
    }
    // groups > 1: npairs < T, one pair per thread (PPT slot 0)
    __syncthreads();
    if (jg < groups) red[jg * span + lt] = acc[0];
    __syncthreads();
    if (threadIdx.x < npairs) {
      float s = 0.f;
      for (int g = 0; g < groups; ++g) s += red[g * span + threadIdx.x];
      out[threadIdx.x] = s;
    }
  }
};

__device__ __forceinline__ void chunk_tiles(const NsSmallArgs& a, int q, int64_t& t0, int64_t& t1) {
  t0 = a.tiles * q / a.chunks;
  t1 = a.tiles * (q + 1) / a.chunks;
}

// grid (chunks, views of one launch set). Momentum update (when UPDATE) and
// the chunk's partial sums of M M^T.
template <bool UPDATE>
__global__ void __launch_bounds__(T) ns_small_prep_kernel(const NsSmallArgs a, const View* __restrict__ views,
                                                          bool tall, bool bf16, float beta) {
  __shared__ float xs[RMAX * LDS];
  __shared__ float red[T];
  const View v = views[blockIdx.y];
  const int r = a.r;
  GramLane gl;
  gl.init(r);
  float acc[PPT];
#pragma unroll
  for (int u = 0; u < PPT; ++u) acc[u] = 0.f;
  int64_t t0, t1;
  chunk_tiles(a, blockIdx.x, t0, t1);
  for (int64_t tile = t0; tile < t1; ++tile) {
    const int64_t j0 = tile * TC;
    for (int e = threadIdx.x; e < r * TC; e += T) {
      int k, j;
      tile_elem(e, r, tall, k, j);
      float m = 0.f;
      if (j0 + j < a.c) {
        const int64_t off = view_off(v, tall, k, j0 + j);
        m = v.M[off];
        if (UPDATE) {
          m = fmaf(beta, m, grad_value(v.G, off, bf16));
          v.M[off] = m;
        }
      }
      xs[k * LDS + j] = m;
    }
    __syncthreads();
    gl.accumulate(xs, acc);
    __syncthreads();
  }
  gl.store(acc, red, a.partials + (static_cast<int64_t>(v.slot) * a.chunks + blockIdx.x) * gl.npairs);
}

// grid (matrices). A from the partial sums (fixed order), then
// P = a I + b A + c A A (times s on round 0).
__global__ void __launch_bounds__(T) ns_small_poly_kernel(const NsSmallArgs a, bool first, float ca, float cb,
                                                          float cc, float ns_eps) {
  __shared__ float A[RMAX * (RMAX + 1)];
  __shared__ float scale_sh;
  const int r = a.r, npairs = r * (r + 1) / 2, lda = r + 1;
  const int64_t slot = blockIdx.x;
  const float* part = a.partials + slot * a.chunks * npairs;
  for (int p = threadIdx.x; p < npairs; p += T) {
    float s = 0.f;
    for (int q = 0; q < a.chunks; ++q) s += part[static_cast<int64_t>(q) * npairs + p];
    int i, k;
    pair_ik(p, r, i, k);
    A[i * lda + k] = s;
    A[k * lda + i] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float sc = 1.f;
    if (first) {
      float tr = 0.f;
      for (int i = 0; i < r; ++i) tr += A[i * lda + i];  // ||M||_F^2
      sc = 1.f / (sqrtf(tr) + ns_eps);
    }
    scale_sh = sc;
  }
  __syncthreads();
  const float s = scale_sh, s2 = s * s;
  if (first) {
    for (int e = threadIdx.x; e < r * r; e += T) {
      const int i = e / r, k = e - i * r;
      A[i * lda + k] *= s2;
    }
    __syncthreads();
  }
  float* P = a.P + slot * r * r;
  for (int e = threadIdx.x; e < r * r; e += T) {
    const int i = e / r, k = e - i * r;
    float aa = 0.f;
    for (int l = 0; l < r; ++l) aa = fmaf(A[i * lda + l], A[l * lda + k], aa);
    float p = fmaf(cb, A[i * lda + k], cc * aa);
    if (i == k) p += ca;
    P[e] = first ? p * s : p;
  }
}

// grid (chunks, views of one launch set). X' = P X for the chunk's tiles.
// FIRST reads X = M from the view, otherwise the workspace copy. LAST
// applies D = X' to W (or writes it to the view's `out`), otherwise X' goes
// back to the workspace and the chunk's partial sums of X' X'^T are written.
template <bool FIRST, bool LAST>
__global__ void __launch_bounds__(T) ns_small_combine_kernel(const NsSmallArgs a, const View* __restrict__ views,
                                                             bool tall, float decay, float eta) {
  __shared__ float xs[RMAX * LDS];
  __shared__ float Ps[RMAX * (RMAX + 1)];
  __shared__ float red[T];
  const View v = views[blockIdx.y];
  const int r = a.r, ldp = r + 1, ne = r * TC;
  const float* P = a.P + static_cast<int64_t>(v.slot) * r * r;
  for (int e = threadIdx.x; e < r * r; e += T) {
    const int i = e / r, k = e - i * r;
    Ps[i * ldp + k] = P[e];
  }
  GramLane gl;
  if (!LAST) gl.init(r);
  float acc[PPT];
#pragma unroll
  for (int u = 0; u < PPT; ++u) acc[u] = 0.f;
  const float step = eta * v.shape_scale;
  float* const dst = v.W != nullptr ? v.W : v.out;
  int64_t t0, t1;
  chunk_tiles(a, blockIdx.x, t0, t1);
  for (int64_t tile = t0; tile < t1; ++tile) {
    const int64_t j0 = tile * TC;
    float* xw = a.X + (static_cast<int64_t>(v.slot) * a.tiles + tile) * ne;
    for (int e = threadIdx.x; e < ne; e += T) {
      int k, j;
      tile_elem(e, r, tall, k, j);
      float x;
      if (FIRST)
        x = j0 + j < a.c ? v.M[view_off(v, tall, k, j0 + j)] : 0.f;
      else
        x = xw[e];
      xs[k * LDS + j] = x;
    }
    __syncthreads();
    float y[OPT];
#pragma unroll
    for (int o = 0; o < OPT; ++o) {
      const int e = threadIdx.x + o * T;
      y[o] = 0.f;
      if (e < ne) {
        int i, j;
        tile_elem(e, r, tall, i, j);
        float s = 0.f;
        for (int k = 0; k < r; ++k) s = fmaf(Ps[i * ldp + k], xs[k * LDS + j], s);
        y[o] = s;
      }
    }
    __syncthreads();  // every thread has read the tile
#pragma unroll
    for (int o = 0; o < OPT; ++o) {
      const int e = threadIdx.x + o * T;
      if (e >= ne) continue;
      int i, j;
      tile_elem(e, r, tall, i, j);
      if (LAST) {
        if (j0 + j < a.c) {
          const int64_t off = view_off(v, tall, i, j0 + j);
          dst[off] = v.W != nullptr ? fmaf(v.W[off], decay, -step * y[o]) : y[o];
        }
      } else {
        // columns beyond c stay zero: P X of a zero column is zero
        xw[e] = y[o];
        xs[i * LDS + j] = y[o];
      }
    }
    if (!LAST) {
      __syncthreads();
      gl.accumulate(xs, acc);
      __syncthreads();
    }
  }
  if (!LAST) gl.store(acc, red, a.partials + (static_cast<int64_t>(v.slot) * a.chunks + blockIdx.x) * gl.npairs);
}

}  // namespace

int64_t ns_small_tiles(int64_t c) { return (c + TC - 1) / TC; }

int ns_small_chunks(int64_t c) { return static_cast<int>(std::min<int64_t>(ns_small_tiles(c), NS_SMALL_MAX_CHUNKS)); }

cudaError_t launch_ns_small_prep(const NsSmallArgs& a, const View* d_views, int count, bool tall, bool grad_bf16,
                                 bool update_momentum, float beta, cudaStream_t stream) {
  if (count == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(a.chunks), static_cast<unsigned>(count));
  if (update_momentum)
    ns_small_prep_kernel<true><<<grid, T, 0, stream>>>(a, d_views, tall, grad_bf16, beta);
  else
    ns_small_prep_kernel<false><<<grid, T, 0, stream>>>(a, d_views, tall, grad_bf16, beta);
  return cudaGetLastError();
}

cudaError_t launch_ns_small_poly(const NsSmallArgs& a, int count, bool first, const float coeffs[3], float ns_eps,
                                 cudaStream_t stream) {
  if (count == 0) return cudaSuccess;
  ns_small_poly_kernel<<<static_cast<unsigned>(count), T, 0, stream>>>(a, first, coeffs[0], coeffs[1], coeffs[2],
                                                                       ns_eps);
  return cudaGetLastError();
}

cudaError_t launch_ns_small_combine(const NsSmallArgs& a, const View* d_views, int count, bool tall, bool first,
                                    bool last, float decay, float eta, cudaStream_t stream) {
  if (count == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(a.chunks), static_cast<unsigned>(count));
#define PRM_NS_SMALL_COMBINE(F, L) \
  ns_small_combine_kernel<F, L><<<grid, T, 0, stream>>>(a, d_views, tall, decay, eta)
  if (first && last) PRM_NS_SMALL_COMBINE(true, true);
  else if (first) PRM_NS_SMALL_COMBINE(true, false);
  else if (last) PRM_NS_SMALL_COMBINE(false, true);
  else PRM_NS_SMALL_COMBINE(false, false);
#undef PRM_NS_SMALL_COMBINE
  return cudaGetLastError();
}

}  // namespace prm
