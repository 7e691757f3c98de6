// Allocation-free variant of the tall-matrix RowNorm step.
//
// The regular path (prm_step) needs a caller-allocated workspace for the
// column partial sums and inverse column norms of tall matrices. Some callers
// cannot hand one over: code that runs where device allocation is not
// allowed or not possible at that moment -- for example a host process whose
// allocator has reserved all device memory up front and forbids new
// allocations during the update, an integration whose latency budget cannot
// absorb the implicit synchronisation of cudaMalloc / cudaFree, or a plugin
// that only ever receives the tensors it works on. For them this file keeps
// the scratch in a fixed device array that lives in the library itself.
//
// The array (NOALLOC_SCRATCH_FLOATS floats = 4 MiB) is part of the module:
// every GPU that loads the library holds it until the process exits. All
// calls share it and it keeps the last call's contents; the kernels below
// overwrite every element they later read, so nothing needs clearing. Calls
// whose work overlaps on the GPU (different streams, or different host
// threads without ordering) race on the array and must not be issued.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cmath>

#include "internal.h"
#include "prm.h"

namespace prm {
namespace {

constexpr int64_t NOALLOC_SCRATCH_FLOATS = int64_t(1) << 20;
constexpr int NA_TX = 32;   // threads along a row
constexpr int NA_TY = 8;    // thread rows
constexpr int NA_RB = 256;  // rows per row block

// The scratch itself. In host code this name is only a host-side stand-in:
// host code must use the device address from cudaGetSymbolAddress.
static __device__ __align__(256) float g_noalloc_scratch[NOALLOC_SCRATCH_FLOATS];

struct TallArgs {
  float* W;
  float* M;
  const void* G;
  int64_t rows, cols;
  float beta, decay, step, eps;  // step = lr * gamma * shape scale
};

__device__ __forceinline__ float na_grad(const void* G, int64_t off, bool bf16) {
  if (bf16) return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(G)[off]) << 16);
  return static_cast<const float*>(G)[off];
}

// M <- beta M + G over a 256-row block; column partial sums of M^2 into
// partials[row_block][col].
__global__ void __launch_bounds__(NA_TX* NA_TY) na_phase1(TallArgs a, bool bf16, float* partials) {
  __shared__ float red[NA_TY][NA_TX + 1];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int64_t c = static_cast<int64_t>(blockIdx.x) * NA_TX + tx;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * NA_RB;
  const int64_t r1 = (r0 + NA_RB < a.rows) ? r0 + NA_RB : a.rows;
  float acc = 0.f;
  if (c < a.cols) {
    for (int64_t r = r0 + ty; r < r1; r += NA_TY) {
      const int64_t off = r * a.cols + c;
      const float m = fmaf(a.beta, a.M[off], na_grad(a.G, off, bf16));
      a.M[off] = m;
      acc = fmaf(m, m, acc);
    }
  }
  red[ty][tx] = acc;
  __syncthreads();
  if (ty == 0 && c < a.cols) {
    float s = 0.f;
#pragma unroll
    for (int y = 0; y < NA_TY; ++y) s += red[y][tx];
    partials[static_cast<int64_t>(blockIdx.y) * a.cols + c] = s;
  }
}

// inv[col] = 1 / max(sqrt(sum over row blocks), eps).
__global__ void __launch_bounds__(256) na_inv(const float* partials, int64_t row_blocks, int64_t cols, float eps,
                                              float* inv) {
  const int64_t c = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
  if (c >= cols) return;
  float s = 0.f;
  for (int64_t b = 0; b < row_blocks; ++b) s += partials[b * cols + c];
  inv[c] = 1.f / fmaxf(sqrtf(s), eps);
}

// W <- W * decay - step * M * inv[col].
__global__ void __launch_bounds__(NA_TX* NA_TY) na_update(TallArgs a, const float* inv) {
  const int64_t c = static_cast<int64_t>(blockIdx.x) * NA_TX + threadIdx.x;
  if (c >= a.cols) return;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * NA_RB;
  const int64_t r1 = (r0 + NA_RB < a.rows) ? r0 + NA_RB : a.rows;
  const float k = a.step * inv[c];
  for (int64_t r = r0 + threadIdx.y; r < r1; r += NA_TY) {
    const int64_t off = r * a.cols + c;
    a.W[off] = fmaf(a.W[off], a.decay, -k * a.M[off]);
  }
}

// Device address of the scratch array on the current device. Looked up on
// every call rather than cached: the address belongs to the device's
// context, and a context that was torn down and recreated (a device reset in
// the host process) places the array elsewhere. The lookup allocates
// nothing; on the first call on a device it also loads this module there.
int scratch_for_current_device(float** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return PRM_ERR_CUDA;
  *out = static_cast<float*>(p);
  return PRM_OK;
}

}  // namespace
}  // namespace prm

extern "C" int prm_rownorm_tall_step_noalloc(float* param, float* momentum, const void* grad, int grad_dtype,
                                             int64_t rows, int64_t cols, float gamma, float lr, float wd,
                                             float beta, float eps, float shape_scale, void* stream) {
  using namespace prm;
  if (param == nullptr || momentum == nullptr || grad == nullptr) return PRM_ERR_INVALID_ARG;
  if (grad_dtype != PRM_FP32 && grad_dtype != PRM_BF16) return PRM_ERR_INVALID_ARG;
  if (rows < 1 || cols < 1 || rows <= cols) return PRM_ERR_SHAPE;
  if (!(beta >= 0.f && beta < 1.f) || !(eps > 0.f) || !std::isfinite(lr) || !std::isfinite(wd) ||
      !std::isfinite(gamma) || !std::isfinite(shape_scale))
    return PRM_ERR_INVALID_ARG;
  const int64_t row_blocks = (rows + NA_RB - 1) / NA_RB;
  if (row_blocks > 65535 || row_blocks * cols + cols > NOALLOC_SCRATCH_FLOATS) return PRM_ERR_UNSUPPORTED;
  float* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc != PRM_OK) return rc;
  float* partials = scratch;
  float* inv = scratch + row_blocks * cols;
  const float s = shape_scale > 0.f ? shape_scale
                                    : static_cast<float>(std::sqrt(std::max(1.0, double(rows) / double(cols))));
  TallArgs a{param, momentum, grad, rows, cols, beta, 1.f - lr * wd, lr * gamma * s, eps};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const dim3 block(NA_TX, NA_TY);
  const dim3 grid(static_cast<unsigned>((cols + NA_TX - 1) / NA_TX), static_cast<unsigned>(row_blocks));
  na_phase1<<<grid, block, 0, st>>>(a, grad_dtype == PRM_BF16, partials);
  na_inv<<<static_cast<unsigned>((cols + 255) / 256), 256, 0, st>>>(partials, row_blocks, cols, eps, inv);
  na_update<<<grid, block, 0, st>>>(a, inv);
  return cudaGetLastError() == cudaSuccess ? PRM_OK : PRM_ERR_CUDA;
}
