// Declarations shared by the library's translation units: matrix views, the
// kernel launchers and the tensor-map encoder.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace prm {

// A row-major m x n view into caller memory with row pitch `ld` elements (a
// whole matrix has ld == cols; a MuonBP block of a wide matrix has the
// parent's pitch). W and M are fp32; G is fp32 or bf16.
struct View {
  float* W;
  float* M;
  const void* G;
  int64_t rows;
  int64_t cols;
  int64_t ld;
  int32_t grad_bf16;
  float shape_scale;
  int32_t slot;     // index of this view inside its NS5 group (batch index)
  int32_t pad;
  float* out;       // standalone orthogonaliser only (W == nullptr): D is written here
};

// Per-step scalars shared by every kernel of one step.
struct StepScalars {
  float beta;     // momentum coefficient
  float decay;    // 1 - lr * wd
  float eta;      // step size of this branch: lr, or lr * gamma
  float eps;      // RowNorm threshold
};

// ---- RowNorm step (non-refresh branch) --------------------------------
// Fused wide step: one CTA per row, grid (rows, count). All views share
// rows/cols. Returns a cudaError_t from the launch.
cudaError_t launch_rownorm_wide(const View* d_views, int count, int64_t rows, int64_t cols, bool vec_ok,
                                bool grad_bf16, StepScalars s, cudaStream_t stream);

// Tall step in three launches: column partial sums, per-column inverse
// norms, update. `partials` holds count * row_blocks(rows) * cols floats and
// `inv` count * cols floats.
int64_t tall_row_blocks(int64_t rows);
cudaError_t launch_rownorm_tall(const View* d_views, int count, int64_t rows, int64_t cols, bool vec_ok,
                                bool grad_bf16, StepScalars s, float* partials, float* inv,
                                cudaStream_t stream);

// Tall step in one launch (16-byte aligned views with cols % 4 == 0): a
// queue of column-stripe tiles, each stripe's update following its momentum
// pass closely enough to read M back from L2 (see rownorm.cu). Scratch:
// partials, inverse norms and a flag block (zeroed by the launch itself).
// A timed-out wait sets *err to the timeout code. Test aid: withhold_stripe
// >= 0 keeps that stripe's inverse norms unpublished, so its update tiles
// give up after wait_ns (0: the default 2 s limit) and leave W unchanged.
struct TallFusedScratch {
  size_t partials_bytes = 0, inv_bytes = 0, flag_bytes = 0;
};
bool tall_fused_fits(int count, int64_t rows, int64_t cols);  // queue and offsets within 32-bit limits
TallFusedScratch tall_fused_scratch(int count, int64_t rows, int64_t cols);
// ring: the TMA form (tall_ring_kernel, two CTAs per SM, each with a
// producer warp feeding a ring of shared-memory stages, eight consumer warps
// and a publisher warp for the stripe bookkeeping); needs tall_ring_ok.
bool tall_ring_ok(int64_t cols, bool grad_bf16);
cudaError_t rownorm_setup_attributes();
// Ring form: tensor maps of each view's M, G and W (3 per view, device
// memory, in view order), boxes of tall_ring_box_cols() x tall_ring_box_rows().
int tall_ring_box_cols();
int tall_ring_box_rows();
cudaError_t launch_rownorm_tall_fused(const View* d_views, int count, int64_t rows, int64_t cols, bool grad_bf16,
                                      StepScalars s, float* partials, float* inv, void* flags, int* err,
                                      int num_sms, cudaStream_t stream, const CUtensorMap* ring_maps,
                                      int withhold_stripe = -1, uint64_t wait_ns = 0);

// ---- refresh (NS5) branch ---------------------------------------------
// Momentum update + bf16 pack into X (wide: same orientation; tall:
// transposed) + per-view Frobenius partial sums (partials: count * slots).
// With update_momentum false the momentum is read as is (no G).
int64_t prep_slots(int64_t rows, int64_t cols);
cudaError_t launch_prep(const View* d_views, int count, int64_t rows, int64_t cols, bool vec_ok,
                        bool grad_bf16, bool update_momentum, float beta, uint16_t* X, int64_t ldc,
                        int64_t x_mat_stride, float* partials, int64_t slots, cudaStream_t stream);

// scale[slot] = 1 / (sqrt(sum of that slot's partials) + ns_eps).
cudaError_t launch_norm_finish(const float* partials, int64_t slots, float* scale, int count, float ns_eps,
                               cudaStream_t stream);

// ---- NS5 of matrices with a short side below NS_SMALL_R (fp32, CUDA cores)
// One same-shape group (wide orientation r x c); buffers in the workspace,
// indexed by the views' batch slots: X tile-major (slot, tile, r x
// NS_SMALL_TC), Gram partial sums (slot, chunk, r (r + 1) / 2 upper-triangle
// pairs) and P (slot, r x r). Chunk q of a matrix covers its column tiles
// [q tiles / chunks, (q + 1) tiles / chunks).
constexpr int NS_SMALL_R = 64;
constexpr int NS_SMALL_TC = 64;
constexpr int NS_SMALL_THREADS = 256;
constexpr int NS_SMALL_MAX_CHUNKS = 128;
struct NsSmallArgs {
  int r;
  int64_t c;
  int64_t tiles;   // ceil(c / NS_SMALL_TC)
  int chunks;      // CTAs per matrix
  float* X;
  float* partials;
  float* P;
};
int64_t ns_small_tiles(int64_t c);
int ns_small_chunks(int64_t c);
// momentum update (or plain read) and the round-0 Gram partials
cudaError_t launch_ns_small_prep(const NsSmallArgs& a, const View* d_views, int count, bool tall, bool grad_bf16,
                                 bool update_momentum, float beta, cudaStream_t stream);
// P = a I + b A + c A A for every matrix of the group (first: s-scaled)
cudaError_t launch_ns_small_poly(const NsSmallArgs& a, int count, bool first, const float coeffs[3], float ns_eps,
                                 cudaStream_t stream);
// X' = P X; last: the update W <- W decay - eta s X' (or D into the view's out)
cudaError_t launch_ns_small_combine(const NsSmallArgs& a, const View* d_views, int count, bool tall, bool first,
                                    bool last, float decay, float eta, cudaStream_t stream);



// ---- tcgen05 GEMM stages of one NS5 round -------------------------------
enum GemmKind { GEMM_GRAM = 0, GEMM_POLY = 1, GEMM_COMBINE = 2 };

// Tensor maps of one batch of r x c bf16 matrices (X) and r x r matrices
// (A, B), built once per buffer address.
struct NsMaps {
  CUtensorMap x_rows128;   // X as K-major operand, 128-row box
  CUtensorMap x_k64;       // X as MN-major operand, 64 x 64 box
  CUtensorMap store;       // X as a GEMM output, 32 x 32 box (epilogue stores)
};
struct SymMaps {
  CUtensorMap rows128;     // A or B as K-major operand, 128-row box
  CUtensorMap store;       // A or B as a GEMM output, 32 x 32 box
};

int encode_x_maps(NsMaps* maps, const void* X, int batch, int64_t r, int64_t c, int64_t ldc);
// 2-D map over one row-major fp32 or bf16 matrix (no swizzle; box_cols x box_rows boxes)
int encode_rows_2d(CUtensorMap* map, const void* base, bool bf16_elems, int64_t rows, int64_t cols, int64_t ld,
                   uint32_t box_cols, uint32_t box_rows);
int encode_sym_maps(SymMaps* maps, const void* A, int batch, int64_t r, int64_t ldr);

// One same-shape batch of a GEMM launch: `batch` matrices. GRAM: out =
// A B^T over K = c (r x r, symmetric: upper super-blocks computed, the rest
// mirrored; a = b = X rows128 for X X^T); POLY: C C (r x r, K = r); COMBINE:
// out = A B, A r x r rows128, B r x c x_k64 (K = r), out r x c.
struct GemmSegSpec {
  const CUtensorMap* a;
  const CUtensorMap* b;
  const CUtensorMap* out;
  const float* scale;     // per-matrix s or nullptr (GRAM: s^2, COMBINE: s)
  int batch;
  int64_t r, c;
  int out_z0;
  const View* views = nullptr;  // COMBINE: apply D to these device views (by batch slot) instead of storing it
  bool in_fp16 = false;         // operands fp16 (else bf16); A and B always share the type
  bool out_fp16 = false;        // output packed as fp16 (else bf16)
  float gain = 1.f, diag = 0.f;  // GRAM / POLY: out = gain * (scale^2) * acc + diag * [i == j]
  // GRAM / POLY: a second output, fp16(gain2 * scale^2 * acc) with no
  // diagonal shift, written through this map (nullptr: none)
  const CUtensorMap* out2 = nullptr;
  float gain2 = 0.f;
};

// Launch-wide epilogue constants. A COMBINE segment with views applies
// D = X' to them, W <- W * decay - eta * shape_scale * D (transposed back for
// tall views), or writes D into `out` for views without W.
struct GemmEpilogue {
  float decay = 1.f, eta = 0.f;
  int* err = nullptr;     // device error word
  int num_sms = 0;
  bool reverse = false;   // each segment's matrices last to first
};

constexpr int GEMM_MAX_SEGMENTS = 6;  // segments per launch (kernel parameter block within 4 KB)

// Runs the tiles of every segment of one GEMM kind from one queue (in
// launches of up to 6 segments; segments with the longest reduction first).
cudaError_t launch_gemm(GemmKind kind, const GemmSegSpec* segs, int count, const GemmEpilogue& epi,
                        cudaStream_t stream);

// Largest dynamic shared memory the GEMM kernels request (for set-up checks).
size_t gemm_smem_bytes();
cudaError_t gemm_setup_attributes();

}  // namespace prm
