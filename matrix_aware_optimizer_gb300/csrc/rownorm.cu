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
// Tall matrices: columns span the whole matrix, so the step takes two passes
// over M -- (1) momentum update + per-row-block column partial sums,
// (2) per-column inverse norms, (3) update reading M again.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "internal.h"

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
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
               : "memory");
}

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
