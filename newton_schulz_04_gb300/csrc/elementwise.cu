// elementwise.cu -- HBM-bound kernels of the update: momentum accumulate + pack +
// Frobenius partial norms (one pass over grad and momentum), the deterministic
// norm finalisation, the zero-step output, and the bounded-wait self test.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace muon {

constexpr int PT = 64;  // packed tile edge of the pack kernel

// One 64 x 64 tile of the packed (short side first, zero padded) matrix b.
// M = beta * mom + grad (or M = src without momentum) is read with coalesced
// rows of the caller's layout, written back to mom, transposed through shared
// memory when the matrix is stored long side first, and stored packed as fp32
// and/or bf16 head + residual.  Each block leaves one partial sum of M^2.
__global__ void __launch_bounds__(256) pack_kernel(const __grid_constant__ PackArgs a) {
  __shared__ float S[PT][PT + 1];
  __shared__ float red[8];
  pdl_launch_dependents();
  pdl_wait();
  const int b = blockIdx.y;
  const int tile = blockIdx.x;
  const int nq = a.lp / PT;
  const int P0 = (tile / nq) * PT, Q0 = (tile % nq) * PT;
  const bool tr = a.tr[b] != 0;
  const int i0 = tr ? Q0 : P0, j0 = tr ? P0 : Q0;  // origin of the source tile
  const int tid = threadIdx.x;
  float ss = 0.f;
#pragma unroll 4
  for (int rr = 0; rr < (PT * PT) / 256; ++rr) {
    const int idx = rr * 256 + tid;
    const int ri = idx >> 6, cj = idx & 63;
    const int gi = i0 + ri, gj = j0 + cj;
    float x = 0.f;
    if (gi < a.m && gj < a.n) {
      const long long off = static_cast<long long>(gi) * a.n + gj;
      const float g = a.src_fp32 ? static_cast<const float*>(a.src[b])[off]
                                 : __bfloat162float(static_cast<const bf16*>(a.src[b])[off]);
      if (a.has_mom) {
        float* mp = a.mom[b] + off;
        x = fmaf(a.beta, *mp, g);
        *mp = x;
      } else {
        x = g;
      }
    }
    ss = fmaf(x, x, ss);
    S[ri][cj] = x;
  }
  __syncthreads();
  const long long base = static_cast<long long>(b) * a.bs;
#pragma unroll 4
  for (int rr = 0; rr < (PT * PT) / 256; ++rr) {
    const int idx = rr * 256 + tid;
    const int pr = idx >> 6, pc = idx & 63;
    const float x = tr ? S[pc][pr] : S[pr][pc];
    const long long off = base + static_cast<long long>(P0 + pr) * a.lp + (Q0 + pc);
    if (a.Xf) a.Xf[off] = x;
    if (a.Xh) {
      const bf16 h = __float2bfloat16_rn(x);
      a.Xh[off] = h;
      if (a.Xl) a.Xl[off] = __float2bfloat16_rn(x - __bfloat162float(h));
    }
  }
  // fixed-shape reduction: warp shuffle tree, then 8 warp sums in order
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  __syncthreads();
  if (tid == 0) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) t += red[w];
    a.partial[static_cast<long long>(b) * a.tiles + tile] = t;
  }
}

cudaError_t launch_pack(const PackArgs& a, int B, cudaStream_t st) {
  if (B <= 0) return cudaSuccess;
  return launch_pdl(pack_kernel, dim3(a.tiles, B), dim3(256), 0, st, a);
}

// inv_norm[b] = 1 / (sqrt(sum of the partials of b) + eps), summed in a fixed order.
__global__ void __launch_bounds__(256) norm_finalize_kernel(const float* partial, int tiles, float eps,
                                                            float* inv_norm) {
  __shared__ float red[8];
  pdl_launch_dependents();
  pdl_wait();
  const int b = blockIdx.x;
  const float* p = partial + static_cast<long long>(b) * tiles;
  float s = 0.f;
  for (int t = threadIdx.x; t < tiles; t += 256) s += p[t];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) t += red[w];
    inv_norm[b] = 1.f / (sqrtf(t) + eps);
  }
}

cudaError_t launch_norm_finalize(const float* partial, int tiles, int B, float eps, float* inv_norm,
                                 cudaStream_t st) {
  if (B <= 0) return cudaSuccess;
  return launch_pdl(norm_finalize_kernel, dim3(B), dim3(256), 0, st, partial, tiles, eps, inv_norm);
}

struct FinalArgs {
  const float* Xf;
  long long ld, bs;
  EpiParams e;
};

__global__ void __launch_bounds__(256) final_from_packed_kernel(const __grid_constant__ FinalArgs a) {
  pdl_launch_dependents();
  pdl_wait();
  const int b = blockIdx.y;
  const EpiParams& e = a.e;
  const long long n = static_cast<long long>(e.rows_valid) * e.cols_valid;
  const float sc = epi_scale(e, b);
  for (long long t = blockIdx.x * 256LL + threadIdx.x; t < n; t += 256LL * gridDim.x) {
    const int p = static_cast<int>(t / e.cols_valid), q = static_cast<int>(t % e.cols_valid);
    const float v = sc * a.Xf[static_cast<long long>(b) * a.bs + static_cast<long long>(p) * a.ld + q];
    epi_final_elem(e, b, p, q, v);
  }
}

cudaError_t launch_final_from_packed(const float* Xf, long long ld, long long bs, int B, const EpiParams& e,
                                     cudaStream_t st) {
  if (B <= 0) return cudaSuccess;
  FinalArgs a{Xf, ld, bs, e};
  const long long n = static_cast<long long>(e.rows_valid) * e.cols_valid;
  long long blocks = (n + 255) / 256;
  if (blocks > 1024) blocks = 1024;
  if (blocks < 1) blocks = 1;
  return launch_pdl(final_from_packed_kernel, dim3(static_cast<unsigned>(blocks), B), dim3(256), 0, st, a);
}

// Waits on a barrier that nobody arrives at; gives up after `cycles` and records it.
__global__ void debug_wait_kernel(int* status, long long cycles) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, cycles)) atomicOr(status, kStatusTimeout);
}

cudaError_t launch_debug_wait(int* status, long long cycles, cudaStream_t st) {
  debug_wait_kernel<<<1, 32, 0, st>>>(status, cycles);
  return cudaGetLastError();
}

}  // namespace muon
