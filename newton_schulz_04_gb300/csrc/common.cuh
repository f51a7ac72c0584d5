// common.cuh -- types shared by the kernels and the host engine: the epilogue
// description every GEMM kernel finishes with, the packing arguments, and the
// per-element epilogue arithmetic.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace muon {

constexpr int kMaxBatch = 256;     // matrices per launch (pointer tables travel as kernel parameters)
constexpr int kStatusTimeout = 1;  // bit set in the workspace status word on a bounded-wait timeout
// An fp16 pair stores v as hi = fp16(v), lo = fp16((v - hi) * kF16LoScale): the
// power-of-two scale keeps the residual out of fp16's subnormal range.
constexpr float kF16LoScale = 2048.f;

typedef __nv_bfloat16 bf16;

enum FinalMode : int { FINAL_NONE = 0, FINAL_STORE = 1, FINAL_APPLY = 2 };

// How a GEMM turns its fp32 accumulator into outputs.  For output element (r, c)
// of matrix b (r, c in the packed, short-side-first orientation):
//
//   v = sc_b * (c_acc * acc + c_res * r_scale * R[b][r][c]) + (r == c && r < rows_valid ? c_id : 0)
//   sc_b = 1, inv_norm[b] or inv_norm[b]^2 (scale_pow = 0, 1, 2)
//
// R is either fp32 (`R`, CUDA-core path) or a 16-bit pair (`Rh` + `Rl`,
// tensor-core path; `Rl` may be absent).  v is then stored into packed buffers
// -- fp32 `Of` (CUDA-core path) or the 16-bit pair `Oh`, `Ol` (tensor-core
// path; `Ol` may be absent) -- or, in a final mode, written (FINAL_STORE) or
// applied as W <- W - lr * v (FINAL_APPLY) to the caller's un-packed matrix
// dst[b].  A 16-bit pair is either bf16, hi = bf16(v) and lo = bf16(v - hi)
// (about 16 significant bits), or fp16, hi = fp16(v) and lo = fp16((v - hi) *
// lo_scale) (about 22 bits; lo_scale is kF16LoScale unless the next product
// folds a coefficient into the stored low part); `r_f16` / `o_f16` select fp16
// for the residual / the output.  On the CUDA-core path, `sym` computes the lower triangle and
// mirrors each element; the tensor-core path stores symmetric outputs
// block-lower.
//
// EpiCore holds the scalars and buffer pointers, EpiFinal the per-matrix
// tables of the final modes; a tensor-core launch that runs several products
// carries one EpiCore per product and a single EpiFinal.
struct EpiCore {
  const float* inv_norm;  // [B] 1 / (||X||_F + eps)
  int scale_pow;
  float c_acc, c_res, c_id;
  const float* R;   // packed fp32 residual or nullptr (CUDA-core path)
  float* Of;        // packed fp32 output or nullptr (CUDA-core path)
  const void* Rh;   // packed 16-bit residual pair or nullptr (tensor-core path)
  const void* Rl;
  void* Oh;         // packed 16-bit output pair (tensor-core path; written through TMA maps)
  void* Ol;         // may be nullptr when only the head is needed
  int r_f16;        // 1: the residual pair is fp16, 0: bf16
  float r_scale;    // multiplies the residual (tensor-core path; e.g. 2^-11 when Rh is the scaled low part of an fp16 pair)
  int o_f16;        // 1: the output pair is fp16, 0: bf16
  float lo_scale;   // an fp16 output pair's low part is stored as (v - hi) * lo_scale (normally 2^11)
  long long ld;     // leading dimension (elements) of the packed residual / outputs
  long long bs;     // batch stride (elements)
  int sym;
  int rows_valid;   // true short side s (padding rows are >= s)
  int cols_valid;   // true long side (or s for square outputs)
  // final-mode fields
  int final_mode;
  int dst_fp32;  // 1: dst is fp32, 0: bf16
  float lr;
};
struct EpiFinal {
  void* dst[kMaxBatch];
  unsigned char tr[kMaxBatch];  // 1: dst[b] is [cols_valid, rows_valid] (the packed matrix transposed)
};
struct EpiParams : EpiCore, EpiFinal {};

__device__ __forceinline__ float epi_scale(const EpiCore& e, int b) {
  if (e.scale_pow == 0) return 1.f;
  const float iv = e.inv_norm[b];
  return e.scale_pow == 2 ? iv * iv : iv;
}

// Final write of one element: packed (p, q) -> caller's matrix.
__device__ __forceinline__ void epi_final_elem(const EpiCore& e, const EpiFinal& f, int b, int p, int q,
                                               float v) {
  if (p >= e.rows_valid || q >= e.cols_valid) return;
  const long long idx =
      f.tr[b] ? (long long)q * e.rows_valid + p : (long long)p * e.cols_valid + q;
  if (e.dst_fp32) {
    float* d = static_cast<float*>(f.dst[b]) + idx;
    if (e.final_mode == FINAL_APPLY) *d = *d - e.lr * v;
    else *d = v;
  } else {
    bf16* d = static_cast<bf16*>(f.dst[b]) + idx;
    if (e.final_mode == FINAL_APPLY) *d = __float2bfloat16_rn(__bfloat162float(*d) - e.lr * v);
    else *d = __float2bfloat16_rn(v);
  }
}

// Full scalar epilogue of one fp32 accumulator element (CUDA-core path).
__device__ __forceinline__ void epi_elem(const EpiParams& e, int b, int r, int c, float acc, float sc) {
  if (e.sym && c > r) return;
  float v = e.c_acc * acc;
  if (e.R) v += e.c_res * e.R[(long long)b * e.bs + (long long)r * e.ld + c];
  v *= sc;
  if (r == c && r < e.rows_valid) v += e.c_id;
  if (e.final_mode != FINAL_NONE) {
    epi_final_elem(e, e, b, r, c, v);
    return;
  }
  const long long base = (long long)b * e.bs;
  e.Of[base + (long long)r * e.ld + c] = v;
  if (e.sym && r > c) e.Of[base + (long long)c * e.ld + r] = v;
}

// Arguments of the momentum / pack / norm kernel.
struct PackArgs {
  int m, n;          // caller's shape of every matrix in this launch
  int sp, lp;        // padded packed shape (short side first)
  int has_mom;       // 1: M = beta*mom + src, written back to mom; 0: M = src
  int src_fp32;      // source dtype: 1 fp32, 0 bf16
  float beta;
  float* Xf;         // packed fp32 copy of M (or nullptr)
  bf16* Xh;          // packed bf16(M) (or nullptr)
  bf16* Xl;          // packed bf16(M - float(Xh)) (or nullptr)
  long long bs;      // batch stride of the packed buffers (elements)
  float* partial;    // [B][tiles] partial sums of squares
  int tiles;         // tiles per matrix
  const void* src[kMaxBatch];
  float* mom[kMaxBatch];
  unsigned char tr[kMaxBatch];
};

}  // namespace muon
