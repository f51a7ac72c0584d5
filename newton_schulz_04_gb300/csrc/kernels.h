// kernels.h -- host-side launchers of the library's kernels (internal interface
// between the engine and the .cu files; not part of the C ABI).
#pragma once
#include <cuda_runtime.h>

#include <utility>

#include "common.cuh"

namespace muon {

// Launch with programmatic stream serialization, so the kernel's prologue may
// overlap the tail of the previous kernel on the stream (every library kernel
// calls pdl_wait() before touching memory).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// A 16-bit operand of the tensor-core GEMM (bf16, or fp16 with TcGemmDesc::f16):
// [batch][rows][ld] row-major, with an optional residual part `lo` of the same
// layout (split operands).
struct TcOperand {
  const void* hi;
  const void* lo;
  long long ld;  // row stride (elements)
  long long bs;  // batch stride (elements)
};

// C[b] (M x N) = A[b] (M x K, row-major) * op(B[b]):
//   b_mn = 0: B stored [N][K] (K-major), C = A B^T      (symmetric right operands, SYRK)
//   b_mn = 1: B stored [K][N] (MN-major), C = A B        (e.g. Q X)
// sym = 1 computes only the tiles touching the lower triangle (M == N) and
// stores the output block-lower (256 x 256 blocks on or below the diagonal).
// a_sym / b_sym mark operands that are symmetric matrices in that storage.
struct TcGemmDesc {
  int B, M, N, K;  // M % 256 == 0, N % 256 == 0, K % 128 == 0 (K % 256 == 0 with symmetric operands)
  int sym;
  int a_sym, b_sym;
  // 1 plain; 2: (A + A_lo) B; 3: A B + A B_lo + A_lo B (bf16 pairs, same scale);
  // 5: fp16 pairs with lo = (v - hi) * 2^11: A B_lo + A_lo B accumulated first,
  // then A B on the accumulator scaled by 2^-11 (tcgen05 scale-input-d)
  int split;
  int b_mn;
  int f16;    // 1: both operands are fp16, 0: both bf16 (one tcgen05 kind::f16 MMA takes one type)
  TcOperand A, Bop;
  // Per-matrix chaining with the previous launch on the stream (optional):
  // every launch adds tc_signals_per_matrix() to done[b] per matrix; with
  // flag_wait a launch starts matrix b once done[b] >= wait_target, instead of
  // waiting for the whole previous grid.
  int* done = nullptr;
  int wait_target = 0;
  int flag_wait = 0;
  // Tile scheduler: one int in global memory, zero before the launch; the
  // CTA pairs take tiles from it in order (atomicAdd), so clusters that start
  // early (while the previous launch drains) take more of them.
  int* tile_ctr = nullptr;
  // Diagonal segment (optional; split 1, b_mn = 1, K == M): a kDiagDim x
  // kDiagDim row-major matrix D = d I of the operand type.  The product is
  // then C = A B + d Bop.lo, the second term computed by the tensor cores as
  // D times the pair's own kDiagDim rows of Bop.lo.
  const void* diag = nullptr;
};
constexpr int kDiagDim = 256;
int tc_signals_per_matrix(int M, int N, int sym);

cudaError_t launch_tc_gemm(const TcGemmDesc& d, const EpiParams& epi, int* status, cudaStream_t st, int num_sms,
                           const char** why);
// Several products in one persistent launch (at most tc_max_products_per_launch()):
// their tiles run as one sequence, and every product after the first waits per
// matrix on the shared completion counters (flag_wait set, one `done` array),
// so the launch overlaps consecutive products without a grid boundary between
// them.  The tile counter is d[0].tile_ctr; at most one product has a final mode.
cudaError_t launch_tc_program(const TcGemmDesc* d, const EpiParams* const* epi, int n, int* status,
                              cudaStream_t st, int num_sms, const char** why);
int tc_max_products_per_launch();
int tc_tiles(int M, int N, int sym);

// fp32 SIMT GEMM with the same conventions (fp32 operands, 128 x 128 tiles).
struct SimtGemmDesc {
  int B, M, N, K;  // multiples of 128 (M, N) and 16 (K)
  int sym;
  int b_mn;
  const float* A;
  long long lda, bsa;
  const float* Bm;
  long long ldb, bsb;
  // A given MN-major: element (m, k) at A[k * lda + m].  For a symmetric A
  // stored in full this is the same buffer as K-major.  With a_mn and b_mn
  // both set, the operand tiles are copied straight into shared memory
  // (cp.async, three stages) instead of through registers.
  int a_mn = 0;
};
cudaError_t launch_simt_gemm(const SimtGemmDesc& d, const EpiParams& epi, cudaStream_t st);

// Momentum + pack + partial norms, then per-matrix 1 / (||M||_F + eps).
cudaError_t launch_pack(const PackArgs& a, int B, cudaStream_t st);
// With `diag` (or nullptr) it also writes the diagonal-segment table D = d I
// (kDiagDim^2 16-bit values, 16-byte aligned; diag_bits = d's bit pattern).
cudaError_t launch_norm_finalize(const float* partial, int tiles, int B, float eps, float* inv_norm, void* diag,
                                 uint16_t diag_bits, cudaStream_t st);
// D = d I on its own (muon_debug_gemm).
cudaError_t launch_fill_diag(void* D, uint16_t bits, cudaStream_t st);
// X = Xf * inv_norm[b] as an fp16 pair (hi, lo = (x - hi) * 2^11), n elements
// per matrix (a multiple of 8; buffers 16-byte aligned), B matrices.
cudaError_t launch_pair_from_f32(const float* Xf, const float* inv_norm, void* Xh, void* Xl, long long n, int B,
                                 int num_sms, cudaStream_t st);
// O = Xf * inv_norm written through a final-mode epilogue (zero NS steps).
cudaError_t launch_final_from_packed(const float* Xf, long long ld, long long bs, int B, const EpiParams& e,
                                     cudaStream_t st);
// Fused AdamW over a list of tensors (the non-matrix tail).
// Tensors per launch: the argument block (49 bytes per tensor) stays inside
// the 32 KB kernel-parameter limit.
constexpr int kMaxTail = 512;
struct AdamwArgs {
  int count;
  float decay;         // 1 - lr * weight_decay
  float beta1, beta2, eps;
  float step_size;     // lr / (1 - beta1^step)
  float inv_sqrt_bc2;  // 1 / sqrt(1 - beta2^step)
  long long gstart[kMaxTail + 1];  // first 8-element group of each tensor; gstart[count] = all groups
  long long numel[kMaxTail];
  void* p[kMaxTail];
  const void* g[kMaxTail];
  float* m[kMaxTail];
  float* v[kMaxTail];
  unsigned char vec_ok[kMaxTail];  // 1: the tensor's four arrays are 16-byte aligned
};
cudaError_t launch_adamw_tail(const AdamwArgs& a, bool bf16_params, int num_sms, cudaStream_t st);

// Failure-detection self test: a bounded wait on a barrier that never completes.
cudaError_t launch_debug_wait(int* status, long long cycles, cudaStream_t st);

}  // namespace muon
