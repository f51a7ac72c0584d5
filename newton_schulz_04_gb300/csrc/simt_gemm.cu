// simt_gemm.cu -- batched fp32 GEMM on the CUDA cores for the fp32 path.
//
// The fp32 path promises a relative error of 1e-4 against the fp64 result.
// Up to 6 steps its products run on the tensor cores as fp16 pairs; beyond
// that the tensor cores' fp32 accumulation error builds up too close to the
// tolerance, and the products run here on FFMA (also on request: the ORIG and
// GRAM schedules for fp32 data).  Same conventions as the tensor-core kernel:
// C[b] = A[b] * op(B[b]), `sym` computes only the lower-triangle tiles and the
// epilogue mirrors them.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace muon {

struct SimtArgs {
  SimtGemmDesc d;
  int nI, nJ, tpm;
  EpiParams epi;
};

constexpr int SB = 128;  // tile edge
constexpr int SK = 16;   // k per smem stage

// Two blocks per SM (at most 128 registers a thread): at 129 registers only one
// block fitted, and 8 warps per SM hid the shared-memory latency poorly (8 x
// 1024x4096 fp32, 10 steps: 24.7 ms per call with one block, 18.8 with two,
// 16.3 once the symmetric-operand products moved to simt_gemm_mn_kernel).
__global__ void __launch_bounds__(256, 2) simt_gemm_kernel(const __grid_constant__ SimtArgs a) {
  __shared__ __align__(16) float As[2][SK][SB];
  __shared__ __align__(16) float Bs[2][SK][SB];
  pdl_launch_dependents();
  pdl_wait();
  const SimtGemmDesc& d = a.d;
  const int b = blockIdx.y;
  const int u = blockIdx.x;
  int i, j;
  if (d.sym) {  // lower-triangular square tiles: row i holds i + 1 tiles
    i = static_cast<int>((sqrtf(8.f * static_cast<float>(u) + 1.f) - 1.f) * 0.5f);
    while (i > 0 && i * (i + 1) / 2 > u) --i;
    while ((i + 1) * (i + 2) / 2 <= u) ++i;
    j = u - i * (i + 1) / 2;
  } else {
    i = u % a.nI;
    j = u / a.nI;
  }
  const int m0 = i * SB, n0 = j * SB;
  const int tid = threadIdx.x;
  const float* A = d.A + static_cast<long long>(b) * d.bsa;
  const float* Bm = d.Bm + static_cast<long long>(b) * d.bsb;

  // global -> register staging
  const int la_r = tid >> 1, la_k = (tid & 1) * 8;    // A (and K-major B): row, k offset
  const int lb_k = tid >> 4, lb_n = (tid & 15) * 8;   // MN-major B: k row, n offset
  float4 ra[2], rb[2];
  auto gload = [&](int k0) {
    const float4* pa = reinterpret_cast<const float4*>(A + static_cast<long long>(m0 + la_r) * d.lda + k0 + la_k);
    ra[0] = pa[0];
    ra[1] = pa[1];
    if (!d.b_mn) {
      const float4* pb =
          reinterpret_cast<const float4*>(Bm + static_cast<long long>(n0 + la_r) * d.ldb + k0 + la_k);
      rb[0] = pb[0];
      rb[1] = pb[1];
    } else {
      const float4* pb =
          reinterpret_cast<const float4*>(Bm + static_cast<long long>(k0 + lb_k) * d.ldb + n0 + lb_n);
      rb[0] = pb[0];
      rb[1] = pb[1];
    }
  };
  auto sstore = [&](int buf) {
    const float av[8] = {ra[0].x, ra[0].y, ra[0].z, ra[0].w, ra[1].x, ra[1].y, ra[1].z, ra[1].w};
#pragma unroll
    for (int q = 0; q < 8; ++q) As[buf][la_k + q][la_r] = av[q];
    if (!d.b_mn) {
      const float bv[8] = {rb[0].x, rb[0].y, rb[0].z, rb[0].w, rb[1].x, rb[1].y, rb[1].z, rb[1].w};
#pragma unroll
      for (int q = 0; q < 8; ++q) Bs[buf][la_k + q][la_r] = bv[q];
    } else {
      *reinterpret_cast<float4*>(&Bs[buf][lb_k][lb_n]) = rb[0];
      *reinterpret_cast<float4*>(&Bs[buf][lb_k][lb_n + 4]) = rb[1];
    }
  };

  const int ty = tid >> 4, tx = tid & 15;
  float acc[8][8];
#pragma unroll
  for (int p = 0; p < 8; ++p)
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[p][q] = 0.f;

  const int nk = d.K / SK;
  gload(0);
  sstore(0);
  __syncthreads();
  for (int kb = 0; kb < nk; ++kb) {
    const int cur = kb & 1;
    if (kb + 1 < nk) gload((kb + 1) * SK);
#pragma unroll
    for (int k = 0; k < SK; ++k) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[cur][k][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[cur][k][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[cur][k][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[cur][k][64 + tx * 4]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int p = 0; p < 8; ++p)
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[p][q] = fmaf(av[p], bv[q], acc[p][q]);
    }
    if (kb + 1 < nk) sstore(cur ^ 1);
    __syncthreads();
  }

  const EpiParams& e = a.epi;
  const float sc = epi_scale(e, b);
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const int r = m0 + (p < 4 ? ty * 4 + p : 64 + ty * 4 + (p - 4));
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int c = n0 + (q < 4 ? tx * 4 + q : 64 + tx * 4 + (q - 4));
      epi_elem(e, b, r, c, acc[p][q], sc);
    }
  }
}

// Both operands MN-major (a_mn and b_mn): every stage is MN_SK rows of 128
// contiguous floats per operand, so each thread copies MN_SK / 8 16-byte
// pieces of each straight into shared memory with cp.async, three stages deep,
// and no registers stage the tiles or transpose them.  The inner product and
// the epilogue are those of simt_gemm_kernel.
constexpr int MN_STAGES = 3;
constexpr int MN_SK = 16;                        // k per stage
constexpr int MN_STAGE_FLOATS = 2 * MN_SK * SB;  // A then B
constexpr size_t MN_SMEM = static_cast<size_t>(MN_STAGES) * MN_STAGE_FLOATS * sizeof(float);
// Within the 48 KB a launch may take without opting in per device.  Deeper or
// wider stages (4 x 16, 3 x 32) timed the same on c5 fp32.
static_assert(MN_SMEM <= 48 * 1024, "dynamic shared memory of simt_gemm_mn_kernel");

__global__ void __launch_bounds__(256, 2) simt_gemm_mn_kernel(const __grid_constant__ SimtArgs a) {
  extern __shared__ __align__(16) float smem[];  // [MN_STAGES][A, B][SK][SB]
  pdl_launch_dependents();
  pdl_wait();
  const SimtGemmDesc& d = a.d;
  const int b = blockIdx.y;
  const int u = blockIdx.x;
  int i, j;
  if (d.sym) {  // lower-triangular square tiles: row i holds i + 1 tiles
    i = static_cast<int>((sqrtf(8.f * static_cast<float>(u) + 1.f) - 1.f) * 0.5f);
    while (i > 0 && i * (i + 1) / 2 > u) --i;
    while ((i + 1) * (i + 2) / 2 <= u) ++i;
    j = u - i * (i + 1) / 2;
  } else {
    i = u % a.nI;
    j = u / a.nI;
  }
  const int m0 = i * SB, n0 = j * SB;
  const int tid = threadIdx.x;
  const float* A = d.A + static_cast<long long>(b) * d.bsa;
  const float* Bm = d.Bm + static_cast<long long>(b) * d.bsb;
  // piece c = tid + 256 h of a stage: row c / 32, floats 4 (c % 32) ..
  auto issue = [&](int kb, int stg) {
    float* As = smem + stg * MN_STAGE_FLOATS;
    float* Bs = As + MN_SK * SB;
    const int k0 = kb * MN_SK;
#pragma unroll
    for (int h = 0; h < MN_SK / 8; ++h) {
      const int c = tid + h * 256, kr = c >> 5, col = (c & 31) * 4;
      cp_async16(As + kr * SB + col, A + static_cast<long long>(k0 + kr) * d.lda + m0 + col);
      cp_async16(Bs + kr * SB + col, Bm + static_cast<long long>(k0 + kr) * d.ldb + n0 + col);
    }
  };

  const int ty = tid >> 4, tx = tid & 15;
  float acc[8][8];
#pragma unroll
  for (int p = 0; p < 8; ++p)
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[p][q] = 0.f;

  const int nk = d.K / MN_SK;
#pragma unroll
  for (int s0 = 0; s0 < MN_STAGES - 1; ++s0) {
    if (s0 < nk) issue(s0, s0);
    cp_async_commit();  // one group per stage, empty past the end, so the counts below hold
  }
  for (int kb = 0; kb < nk; ++kb) {
    cp_async_wait<MN_STAGES - 2>();  // this thread's pieces of stage kb have landed
    __syncthreads();                 // everyone's have, and stage kb - 1 is no longer read
    const int nxt = kb + MN_STAGES - 1;
    if (nxt < nk) issue(nxt, nxt % MN_STAGES);
    cp_async_commit();
    const float* As = smem + (kb % MN_STAGES) * MN_STAGE_FLOATS;
    const float* Bs = As + MN_SK * SB;
#pragma unroll
    for (int k = 0; k < MN_SK; ++k) {
      const float4 a0 = *reinterpret_cast<const float4*>(As + k * SB + ty * 4);
      const float4 a1 = *reinterpret_cast<const float4*>(As + k * SB + 64 + ty * 4);
      const float4 b0 = *reinterpret_cast<const float4*>(Bs + k * SB + tx * 4);
      const float4 b1 = *reinterpret_cast<const float4*>(Bs + k * SB + 64 + tx * 4);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int p = 0; p < 8; ++p)
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[p][q] = fmaf(av[p], bv[q], acc[p][q]);
    }
  }
  cp_async_wait<0>();

  const EpiParams& e = a.epi;
  const float sc = epi_scale(e, b);
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const int r = m0 + (p < 4 ? ty * 4 + p : 64 + ty * 4 + (p - 4));
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int c = n0 + (q < 4 ? tx * 4 + q : 64 + tx * 4 + (q - 4));
      epi_elem(e, b, r, c, acc[p][q], sc);
    }
  }
}

cudaError_t launch_simt_gemm(const SimtGemmDesc& d, const EpiParams& epi, cudaStream_t st) {
  SimtArgs a;
  a.d = d;
  a.nI = d.M / SB;
  a.nJ = d.N / SB;
  a.tpm = d.sym ? a.nI * (a.nI + 1) / 2 : a.nI * a.nJ;
  a.epi = epi;
  a.epi.sym = d.sym;
  if (d.B <= 0 || a.tpm <= 0) return cudaSuccess;
  if (d.a_mn && d.b_mn) return launch_pdl(simt_gemm_mn_kernel, dim3(a.tpm, d.B), dim3(256), MN_SMEM, st, a);
  if (d.a_mn) return cudaErrorInvalidValue;  // an MN-major A is only taken with an MN-major B
  return launch_pdl(simt_gemm_kernel, dim3(a.tpm, d.B), dim3(256), 0, st, a);
}

}  // namespace muon
