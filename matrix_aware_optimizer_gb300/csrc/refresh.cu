// Memory-bound kernels around the NS5 refresh ("Scaling Muon for Diffusion
// Transformers", PaperDaily walkthrough, section "Periodic Row-wise Muon":
// on steps with t % K == 0 the direction is NS5 of the momentum).
//
//   prep   : M <- beta M + G (in place), X0 = bf16(M) in the wide orientation
//            (tall views are transposed through shared memory), and per-CTA
//            partial sums of M^2 for the Frobenius pre-normalisation. The
//            scale 1 / (||M||_F + eps) is not applied here: the first GRAM
//            epilogue multiplies by its square and the first COMBINE epilogue
//            by the scale itself, which is the same NS5 round on M / ||M||.
//   finish : per-view scale = 1 / (sqrt(sum of partials) + eps_ns).
//   (the update W <- W (1 - lr wd) - eta s D, D = X5, runs in the epilogue
//   of the last NS5 round's COMBINE launch, see ns5_gemm.cu)
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace prm {
namespace {

constexpr int PREP_THREADS = 256;
constexpr int TILE = 64;  // transpose tile edge for tall views

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float block_sum256(float v, float* red) {
  const int t = threadIdx.x;
  const int lane = t & 31, warp = t >> 5;
  v = warp_sum(v);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < PREP_THREADS / 32 ? red[lane] : 0.f;
    v = warp_sum(v);
    if (lane == 0) red[32] = v;
  }
  __syncthreads();
  return red[32];
}

__device__ __forceinline__ uint16_t bf16_bits(float v) {
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  return *reinterpret_cast<const uint16_t*>(&h);
}

__device__ __forceinline__ float bf16_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

template <bool BF16>
__device__ __forceinline__ float grad_at(const void* G, int64_t off) {
  if (BF16) return bf16_to_float(static_cast<const uint16_t*>(G)[off]);
  return static_cast<const float*>(G)[off];
}

// ---------------------------------------------------------------- prep
// Wide views: one CTA per row, X row = same row.
template <bool BF16, bool VEC, bool UPDATE>
__global__ void __launch_bounds__(PREP_THREADS) prep_wide_kernel(const View* __restrict__ views, int64_t cols,
                                                                 float beta, uint16_t* __restrict__ X,
                                                                 int64_t ldc, int64_t x_stride,
                                                                 float* __restrict__ partials, int64_t slots) {
  __shared__ float red[33];
  const View v = views[blockIdx.y];
  const int64_t row = blockIdx.x;
  float* Mr = v.M + row * v.ld;
  uint16_t* Xr = X + v.slot * x_stride + row * ldc;
  float ss = 0.f;
  if constexpr (VEC) {
    for (int64_t c = threadIdx.x * 4; c < cols; c += PREP_THREADS * 4) {
      float4 m = *reinterpret_cast<const float4*>(Mr + c);
      if constexpr (UPDATE) {
        const int64_t go = row * v.ld + c;
        float4 g;
        if constexpr (BF16) {
          const uint2 u = __ldcs(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(v.G) + go));
          g = make_float4(bf16_to_float(u.x & 0xFFFFu), bf16_to_float(u.x >> 16), bf16_to_float(u.y & 0xFFFFu),
                          bf16_to_float(u.y >> 16));
        } else {
          g = __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(v.G) + go));
        }
        m.x = fmaf(beta, m.x, g.x);
        m.y = fmaf(beta, m.y, g.y);
        m.z = fmaf(beta, m.z, g.z);
        m.w = fmaf(beta, m.w, g.w);
        *reinterpret_cast<float4*>(Mr + c) = m;
      }
      ss = fmaf(m.x, m.x, ss);
      ss = fmaf(m.y, m.y, ss);
      ss = fmaf(m.z, m.z, ss);
      ss = fmaf(m.w, m.w, ss);
      uint2 packed;
      packed.x = static_cast<uint32_t>(bf16_bits(m.x)) | (static_cast<uint32_t>(bf16_bits(m.y)) << 16);
      packed.y = static_cast<uint32_t>(bf16_bits(m.z)) | (static_cast<uint32_t>(bf16_bits(m.w)) << 16);
      *reinterpret_cast<uint2*>(Xr + c) = packed;
    }
  } else {
    for (int64_t c = threadIdx.x; c < cols; c += PREP_THREADS) {
      float m = Mr[c];
      if constexpr (UPDATE) {
        m = fmaf(beta, m, grad_at<BF16>(v.G, row * v.ld + c));
        Mr[c] = m;
      }
      ss = fmaf(m, m, ss);
      Xr[c] = bf16_bits(m);
    }
  }
  const float total = block_sum256(ss, red);
  if (threadIdx.x == 0) partials[static_cast<int64_t>(v.slot) * slots + row] = total;
}

// Tall views (rows > cols): 64 x 64 tiles, X[j][i] = bf16(M[i][j]).
// Vector path (cols % 4 == 0, 16-byte aligned rows): 16 x 16 threads, each
// owning 4 rows x 4 columns; all loads of a thread are issued before its first
// store so that they overlap, and the transposed bf16 tile leaves as 32-byte
// row pieces.
template <bool BF16, bool UPDATE, bool VEC>
__global__ void __launch_bounds__(PREP_THREADS) prep_tall_kernel(const View* __restrict__ views, int64_t rows,
                                                                 int64_t cols, float beta,
                                                                 uint16_t* __restrict__ X, int64_t ldc,
                                                                 int64_t x_stride, float* __restrict__ partials,
                                                                 int64_t slots) {
  __shared__ float tile[TILE][TILE + 1];
  __shared__ float red[33];
  const View v = views[blockIdx.z];
  const int tid = threadIdx.x;
  const int64_t i0 = static_cast<int64_t>(blockIdx.y) * TILE;
  const int64_t j0 = static_cast<int64_t>(blockIdx.x) * TILE;
  float ss = 0.f;
  if constexpr (VEC) {
    const int tx = tid & 15, ty = tid >> 4;  // 16 float4 columns x 16 row lanes
    const int64_t j = j0 + tx * 4;
    float4 m[4];
    float4 g[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t i = i0 + ty + 16 * k;
      m[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      g[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < rows && j < cols) {
        m[k] = *reinterpret_cast<const float4*>(v.M + i * v.ld + j);
        if constexpr (UPDATE) {
          if constexpr (BF16) {
            const uint2 u = __ldcs(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(v.G) + i * v.ld + j));
            g[k] = make_float4(bf16_to_float(u.x & 0xFFFFu), bf16_to_float(u.x >> 16),
                               bf16_to_float(u.y & 0xFFFFu), bf16_to_float(u.y >> 16));
          } else {
            g[k] = __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(v.G) + i * v.ld + j));
          }
        }
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t i = i0 + ty + 16 * k;
      if constexpr (UPDATE) {
        m[k].x = fmaf(beta, m[k].x, g[k].x);
        m[k].y = fmaf(beta, m[k].y, g[k].y);
        m[k].z = fmaf(beta, m[k].z, g[k].z);
        m[k].w = fmaf(beta, m[k].w, g[k].w);
        if (i < rows && j < cols) *reinterpret_cast<float4*>(v.M + i * v.ld + j) = m[k];
      }
      ss = fmaf(m[k].x, m[k].x, ss);
      ss = fmaf(m[k].y, m[k].y, ss);
      ss = fmaf(m[k].z, m[k].z, ss);
      ss = fmaf(m[k].w, m[k].w, ss);
      float* t = &tile[ty + 16 * k][tx * 4];
      t[0] = m[k].x;
      t[1] = m[k].y;
      t[2] = m[k].z;
      t[3] = m[k].w;
    }
  } else {
    const int tx = tid & 63, ty = tid >> 6;  // 64 columns x 4 row lanes
    float m[16], g[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const int64_t i = i0 + ty + 4 * k, j = j0 + tx;
      m[k] = 0.f;
      g[k] = 0.f;
      if (i < rows && j < cols) {
        m[k] = v.M[i * v.ld + j];
        if constexpr (UPDATE) g[k] = grad_at<BF16>(v.G, i * v.ld + j);
      }
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const int64_t i = i0 + ty + 4 * k, j = j0 + tx;
      if constexpr (UPDATE) {
        m[k] = fmaf(beta, m[k], g[k]);
        if (i < rows && j < cols) v.M[i * v.ld + j] = m[k];
      }
      ss = fmaf(m[k], m[k], ss);
      tile[ty + 4 * k][tx] = m[k];
    }
  }
  __syncthreads();
  // X row j (= column j of M) gets 64 consecutive i: four threads per row,
  // 16 bf16 (32 bytes) each.
  uint16_t* Xv = X + v.slot * x_stride;
  {
    const int jj = tid >> 2, ic = (tid & 3) * 16;
    const int64_t j = j0 + jj, ib = i0 + ic;
    if (j < cols && ib < rows) {
      uint16_t* dst = Xv + j * ldc + ib;
      if (ib + 16 <= rows) {
        uint32_t w[8];
#pragma unroll
        for (int h = 0; h < 8; ++h)
          w[h] = static_cast<uint32_t>(bf16_bits(tile[ic + 2 * h][jj])) |
                 (static_cast<uint32_t>(bf16_bits(tile[ic + 2 * h + 1][jj])) << 16);
        reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
        reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
      } else {
        for (int k = 0; ib + k < rows; ++k) dst[k] = bf16_bits(tile[ic + k][jj]);
      }
    }
  }
  const float total = block_sum256(ss, red);
  if (tid == 0) partials[static_cast<int64_t>(v.slot) * slots + blockIdx.y * gridDim.x + blockIdx.x] = total;
}

__global__ void __launch_bounds__(256) norm_finish_kernel(const float* __restrict__ partials, int64_t slots,
                                                          float* __restrict__ scale, float ns_eps) {
  __shared__ float red[33];
  const float* p = partials + static_cast<int64_t>(blockIdx.x) * slots;
  float s = 0.f;
  for (int64_t k = threadIdx.x; k < slots; k += 256) s += p[k];
  const float total = block_sum256(s, red);
  if (threadIdx.x == 0) scale[blockIdx.x] = 1.f / (sqrtf(total) + ns_eps);
}

}  // namespace

int64_t prep_slots(int64_t rows, int64_t cols) {
  if (rows <= cols) return rows;
  return ((rows + TILE - 1) / TILE) * ((cols + TILE - 1) / TILE);
}

cudaError_t launch_prep(const View* d_views, int count, int64_t rows, int64_t cols, bool vec_ok, bool grad_bf16,
                        bool update_momentum, float beta, uint16_t* X, int64_t ldc, int64_t x_mat_stride,
                        float* partials, int64_t slots, cudaStream_t stream) {
  if (count == 0) return cudaSuccess;
  if (rows <= cols) {
    const dim3 grid(static_cast<unsigned>(rows), static_cast<unsigned>(count));
#define PRM_PREP_WIDE(B, V, U) \
  prep_wide_kernel<B, V, U><<<grid, PREP_THREADS, 0, stream>>>(d_views, cols, beta, X, ldc, x_mat_stride, partials, slots)
    if (!update_momentum) {
      if (vec_ok) PRM_PREP_WIDE(false, true, false);
      else PRM_PREP_WIDE(false, false, false);
    } else if (grad_bf16) {
      if (vec_ok) PRM_PREP_WIDE(true, true, true);
      else PRM_PREP_WIDE(true, false, true);
    } else {
      if (vec_ok) PRM_PREP_WIDE(false, true, true);
      else PRM_PREP_WIDE(false, false, true);
    }
#undef PRM_PREP_WIDE
  } else {
    const dim3 grid(static_cast<unsigned>((cols + TILE - 1) / TILE), static_cast<unsigned>((rows + TILE - 1) / TILE),
                    static_cast<unsigned>(count));
#define PRM_PREP_TALL(B, U, V) \
  prep_tall_kernel<B, U, V><<<grid, PREP_THREADS, 0, stream>>>(d_views, rows, cols, beta, X, ldc, x_mat_stride, partials, slots)
    if (!update_momentum) {
      if (vec_ok) PRM_PREP_TALL(false, false, true);
      else PRM_PREP_TALL(false, false, false);
    } else if (grad_bf16) {
      if (vec_ok) PRM_PREP_TALL(true, true, true);
      else PRM_PREP_TALL(true, true, false);
    } else {
      if (vec_ok) PRM_PREP_TALL(false, true, true);
      else PRM_PREP_TALL(false, true, false);
    }
#undef PRM_PREP_TALL
  }
  return cudaGetLastError();
}

cudaError_t launch_norm_finish(const float* partials, int64_t slots, float* scale, int count, float ns_eps,
                               cudaStream_t stream) {
  if (count == 0) return cudaSuccess;
  norm_finish_kernel<<<count, 256, 0, stream>>>(partials, slots, scale, ns_eps);
  return cudaGetLastError();
}

}  // namespace prm
