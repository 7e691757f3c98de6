// Fused AdamW step for the non-matrix parameters (biases, normalisation
// parameters) that "Scaling Muon for Diffusion Transformers" keeps on AdamW
// (PaperDaily walkthrough, scaling-study section; decoupled weight decay of
// its reference [3]):
//   m <- b1 m + (1 - b1) g ;  v <- b2 v + (1 - b2) g^2
//   p <- p (1 - lr wd) - (lr / (1 - b1^t)) m / (sqrt(v / (1 - b2^t)) + eps)
// One pass over a flat buffer: reads p, m, v (fp32) and g (bf16 or fp32),
// writes p, m, v: 26 B per parameter with bf16 gradients (28 B with fp32).
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cmath>

#include "prm.h"

namespace prm {
namespace {

struct AdamScalars {
  float b1, b2, one_minus_b1, one_minus_b2;
  float inv_bc2;   // 1 / (1 - b2^t)
  float step;      // lr / (1 - b1^t)
  float decay;     // 1 - lr * wd
  float eps;
};

__device__ __forceinline__ void adam_elem(float& p, float& m, float& v, float g, const AdamScalars& s) {
  m = fmaf(s.b1, m, s.one_minus_b1 * g);
  v = fmaf(s.b2, v, s.one_minus_b2 * g * g);
  const float denom = sqrtf(v * s.inv_bc2) + s.eps;
  p = fmaf(p, s.decay, -s.step * (m / denom));
}

template <bool BF16>
__device__ __forceinline__ float4 load_grad4(const void* g, int64_t k) {
  if constexpr (BF16) {
    const uint2 u = __ldcs(reinterpret_cast<const uint2*>(g) + k);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xFFFF0000u));
  } else {
    return __ldcs(reinterpret_cast<const float4*>(g) + k);
  }
}

// Each thread takes ADAM_UNROLL groups of four elements a grid stride apart
// per iteration, issuing all their loads before any arithmetic, so that more
// bytes are in flight per thread.
constexpr int ADAM_UNROLL = 4;

template <bool BF16>
__global__ void __launch_bounds__(256) adamw_vec_kernel(float* __restrict__ p, float* __restrict__ m,
                                                        float* __restrict__ v, const void* __restrict__ g,
                                                        int64_t n4, AdamScalars s) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t k0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k0 < n4;
       k0 += ADAM_UNROLL * stride) {
    float4 pp[ADAM_UNROLL], mm[ADAM_UNROLL], vv[ADAM_UNROLL], gg[ADAM_UNROLL];
#pragma unroll
    for (int u = 0; u < ADAM_UNROLL; ++u) {
      const int64_t k = k0 + u * stride;
      if (k < n4) {
        pp[u] = __ldcs(reinterpret_cast<const float4*>(p) + k);
        mm[u] = __ldcs(reinterpret_cast<const float4*>(m) + k);
        vv[u] = __ldcs(reinterpret_cast<const float4*>(v) + k);
        gg[u] = load_grad4<BF16>(g, k);
      }
    }
#pragma unroll
    for (int u = 0; u < ADAM_UNROLL; ++u) {
      const int64_t k = k0 + u * stride;
      if (k < n4) {
        adam_elem(pp[u].x, mm[u].x, vv[u].x, gg[u].x, s);
        adam_elem(pp[u].y, mm[u].y, vv[u].y, gg[u].y, s);
        adam_elem(pp[u].z, mm[u].z, vv[u].z, gg[u].z, s);
        adam_elem(pp[u].w, mm[u].w, vv[u].w, gg[u].w, s);
        __stcs(reinterpret_cast<float4*>(p) + k, pp[u]);
        __stcs(reinterpret_cast<float4*>(m) + k, mm[u]);
        __stcs(reinterpret_cast<float4*>(v) + k, vv[u]);
      }
    }
  }
}

// Elements [begin, n): the ragged tail of the vector path, or everything when
// a pointer is not 16-byte aligned.
template <bool BF16>
__global__ void __launch_bounds__(256) adamw_scalar_kernel(float* p, float* m, float* v, const void* g,
                                                           int64_t begin, int64_t n, AdamScalars s) {
  for (int64_t i = begin + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float gi = BF16 ? __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(g)[i]) << 16)
                          : static_cast<const float*>(g)[i];
    float pi = p[i], mi = m[i], vi = v[i];
    adam_elem(pi, mi, vi, gi, s);
    p[i] = pi;
    m[i] = mi;
    v[i] = vi;
  }
}

bool aligned16(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }

}  // namespace
}  // namespace prm

extern "C" int prm_adamw_step(float* param, float* exp_avg, float* exp_avg_sq, const void* grad, int grad_dtype,
                              int64_t n, int64_t t, double lr, double beta1, double beta2, double eps, double wd,
                              void* stream) {
  using namespace prm;
  if (n < 0 || t < 1) return PRM_ERR_INVALID_ARG;
  if (grad_dtype != PRM_FP32 && grad_dtype != PRM_BF16) return PRM_ERR_INVALID_ARG;
  if (!(beta1 >= 0.0 && beta1 < 1.0) || !(beta2 >= 0.0 && beta2 < 1.0) || !(eps > 0.0) || !std::isfinite(lr) ||
      !std::isfinite(wd))
    return PRM_ERR_INVALID_ARG;
  if (n == 0) return PRM_OK;
  if (param == nullptr || exp_avg == nullptr || exp_avg_sq == nullptr || grad == nullptr) return PRM_ERR_INVALID_ARG;
  // Complements and bias corrections are formed in double: 1 - b2 from an
  // fp32 b2 = 0.999 would be off by 1.3e-5 relative (cancellation).
  AdamScalars s;
  s.b1 = static_cast<float>(beta1);
  s.b2 = static_cast<float>(beta2);
  s.one_minus_b1 = static_cast<float>(1.0 - beta1);
  s.one_minus_b2 = static_cast<float>(1.0 - beta2);
  const double bc1 = 1.0 - std::pow(beta1, static_cast<double>(t));
  const double bc2 = 1.0 - std::pow(beta2, static_cast<double>(t));
  s.inv_bc2 = static_cast<float>(1.0 / bc2);
  s.step = static_cast<float>(lr / bc1);
  s.decay = static_cast<float>(1.0 - lr * wd);
  s.eps = static_cast<float>(eps);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool bf16 = grad_dtype == PRM_BF16;
  const bool vec = aligned16(param) && aligned16(exp_avg) && aligned16(exp_avg_sq) &&
                   (bf16 ? (reinterpret_cast<uintptr_t>(grad) & 7u) == 0 : aligned16(grad));
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t n4 = vec ? n / 4 : 0;
  if (n4 > 0) {
    const int64_t blocks = std::min<int64_t>((n4 + 255) / 256, static_cast<int64_t>(sms) * 8);
    if (bf16)
      adamw_vec_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, st>>>(param, exp_avg, exp_avg_sq, grad, n4, s);
    else
      adamw_vec_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, st>>>(param, exp_avg, exp_avg_sq, grad, n4, s);
  }
  const int64_t begin = n4 * 4;
  if (begin < n) {
    const int64_t blocks = std::min<int64_t>((n - begin + 255) / 256, static_cast<int64_t>(sms) * 8);
    if (bf16)
      adamw_scalar_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, st>>>(param, exp_avg, exp_avg_sq, grad,
                                                                                begin, n, s);
    else
      adamw_scalar_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, st>>>(param, exp_avg, exp_avg_sq, grad,
                                                                                 begin, n, s);
  }
  return cudaGetLastError() == cudaSuccess ? PRM_OK : PRM_ERR_CUDA;
}
