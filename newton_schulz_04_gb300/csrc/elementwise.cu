// elementwise.cu -- HBM-bound kernels of the update: momentum accumulate + pack +
// Frobenius partial norms (one pass over grad and momentum), the deterministic
// norm finalisation, the zero-step output, and the bounded-wait self test.
#include <cuda_runtime.h>

#include <algorithm>

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
    S[ri][cj] = x;
  }
  __syncthreads();
  const long long base = static_cast<long long>(b) * a.bs;
  // Packed order, 8 consecutive packed elements per thread as in
  // pack_vec_kernel, and the sum of squares taken here in that order: the
  // partial sums (and so the norm) of a packed tile are the same whichever
  // way the matrix is stored and whichever kernel packs it.
#pragma unroll
  for (int rep = 0; rep < 2; ++rep) {
    const int c = rep * 256 + tid;
    const int pr = c >> 3, pc0 = (c & 7) * 8;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int pc = pc0 + k;
      const float x = tr ? S[pc][pr] : S[pr][pc];
      ss = fmaf(x, x, ss);
      const long long off = base + static_cast<long long>(P0 + pr) * a.lp + (Q0 + pc);
      if (a.Xf) a.Xf[off] = x;
      if (a.Xh) {
        const bf16 h = __float2bfloat16_rn(x);
        a.Xh[off] = h;
        if (a.Xl) a.Xl[off] = __float2bfloat16_rn(x - __bfloat162float(h));
      }
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

// Same tile and outputs as pack_kernel, with 8-element (16/32-byte) accesses:
// each thread moves 8 consecutive elements of a source row.  Needs n % 8 == 0
// and 16-byte aligned matrices (the launcher checks).  Matrices stored long
// side first go through a shared-memory transpose; the others are packed
// straight from registers.
template <bool SRC_FP32>
__global__ void __launch_bounds__(256) pack_vec_kernel(const __grid_constant__ PackArgs a) {
  __shared__ float S[PT][PT + 1];
  __shared__ float red[8];
  pdl_launch_dependents();
  pdl_wait();
  const int b = blockIdx.y;
  const int tile = blockIdx.x;
  const int nq = a.lp / PT;
  const int P0 = (tile / nq) * PT, Q0 = (tile % nq) * PT;
  const bool tr = a.tr[b] != 0;
  const int i0 = tr ? Q0 : P0, j0 = tr ? P0 : Q0;
  const int tid = threadIdx.x;
  const long long base = static_cast<long long>(b) * a.bs;
  float ss = 0.f;
  auto store8 = [&](long long off, const float (&x)[8]) {
    if (a.Xf) {
      float4* f = reinterpret_cast<float4*>(a.Xf + off);
      f[0] = make_float4(x[0], x[1], x[2], x[3]);
      f[1] = make_float4(x[4], x[5], x[6], x[7]);
    }
    if (a.Xh) {
      uint32_t h[4], l[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const __nv_bfloat162 hh = __floats2bfloat162_rn(x[2 * u], x[2 * u + 1]);
        h[u] = *reinterpret_cast<const uint32_t*>(&hh);
        const __nv_bfloat162 ll = __floats2bfloat162_rn(x[2 * u] - __low2float(hh), x[2 * u + 1] - __high2float(hh));
        l[u] = *reinterpret_cast<const uint32_t*>(&ll);
      }
      *reinterpret_cast<uint4*>(a.Xh + off) = make_uint4(h[0], h[1], h[2], h[3]);
      if (a.Xl) *reinterpret_cast<uint4*>(a.Xl + off) = make_uint4(l[0], l[1], l[2], l[3]);
    }
  };
#pragma unroll
  for (int rep = 0; rep < 2; ++rep) {
    const int c = rep * 256 + tid;
    const int ri = c >> 3, cj = (c & 7) * 8;
    const int gi = i0 + ri, gj = j0 + cj;
    float x[8];
    if (gi < a.m && gj < a.n) {  // n % 8 == 0: the 8 elements are all inside
      const long long off = static_cast<long long>(gi) * a.n + gj;
      float g[8];
      if (SRC_FP32) {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(a.src[b]) + off);
        const float4 u0 = p[0], u1 = p[1];
        g[0] = u0.x, g[1] = u0.y, g[2] = u0.z, g[3] = u0.w, g[4] = u1.x, g[5] = u1.y, g[6] = u1.z, g[7] = u1.w;
      } else {
        const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const bf16*>(a.src[b]) + off);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          g[2 * k] = __uint_as_float(w[k] << 16);
          g[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        }
      }
      if (a.has_mom) {
        float4* mp = reinterpret_cast<float4*>(a.mom[b] + off);
        const float4 m0 = mp[0], m1 = mp[1];
        const float mo[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = fmaf(a.beta, mo[k], g[k]);
        mp[0] = make_float4(x[0], x[1], x[2], x[3]);
        mp[1] = make_float4(x[4], x[5], x[6], x[7]);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = g[k];
      }
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) x[k] = 0.f;
    }
    if (!tr) {
      // packed order is source order here: the sum of squares goes in that order
#pragma unroll
      for (int k = 0; k < 8; ++k) ss = fmaf(x[k], x[k], ss);
      store8(base + static_cast<long long>(P0 + ri) * a.lp + (Q0 + cj), x);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) S[ri][cj + k] = x[k];
    }
  }
  if (tr) {
    __syncthreads();
#pragma unroll
    for (int rep = 0; rep < 2; ++rep) {
      const int c = rep * 256 + tid;
      const int pr = c >> 3, pc = (c & 7) * 8;  // packed row (= source column), packed column group
      float x[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) x[k] = S[pc + k][pr];
      // in packed order, so the tile's partial sum equals the untransposed one's
#pragma unroll
      for (int k = 0; k < 8; ++k) ss = fmaf(x[k], x[k], ss);
      store8(base + static_cast<long long>(P0 + pr) * a.lp + (Q0 + pc), x);
    }
  }
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
  bool vec = a.n % 8 == 0;
  for (int q = 0; q < B && vec; ++q) {
    if (reinterpret_cast<uintptr_t>(a.src[q]) % 16) vec = false;
    if (a.has_mom && reinterpret_cast<uintptr_t>(a.mom[q]) % 16) vec = false;
  }
  if (vec) {
    if (a.src_fp32) return launch_pdl(pack_vec_kernel<true>, dim3(a.tiles, B), dim3(256), 0, st, a);
    return launch_pdl(pack_vec_kernel<false>, dim3(a.tiles, B), dim3(256), 0, st, a);
  }
  return launch_pdl(pack_kernel, dim3(a.tiles, B), dim3(256), 0, st, a);
}

// D = d I (kDiagDim x kDiagDim 16-bit values, d's bit pattern `bits`) written
// as 16-byte pieces by `nthreads` threads, thread `t` taking pieces t, t + nthreads, ...
__device__ __forceinline__ void fill_diag(uint4* D, uint16_t bits, int t, int nthreads) {
  constexpr int PER_ROW = kDiagDim / 8;
  for (int i = t; i < kDiagDim * PER_ROW; i += nthreads) {
    const int r = i / PER_ROW, c0 = (i % PER_ROW) * 8;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (r >= c0 && r < c0 + 8) w[(r - c0) >> 1] = static_cast<uint32_t>(bits) << (16 * ((r - c0) & 1));
    D[i] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

__global__ void __launch_bounds__(256) fill_diag_kernel(uint4* D, uint16_t bits) {
  pdl_launch_dependents();
  pdl_wait();
  fill_diag(D, bits, blockIdx.x * 256 + threadIdx.x, gridDim.x * 256);
}

cudaError_t launch_fill_diag(void* D, uint16_t bits, cudaStream_t st) {
  return launch_pdl(fill_diag_kernel, dim3(8), dim3(256), 0, st, static_cast<uint4*>(D), bits);
}

// inv_norm[b] = 1 / (sqrt(sum of the partials of b) + eps), summed in a fixed order.
// With `diag`, the blocks also write the table D = d I of the diagonal segment.
__global__ void __launch_bounds__(256) norm_finalize_kernel(const float* partial, int tiles, float eps,
                                                            float* inv_norm, uint4* diag, uint16_t diag_bits) {
  __shared__ float red[8];
  pdl_launch_dependents();
  pdl_wait();
  if (diag) fill_diag(diag, diag_bits, blockIdx.x * 256 + threadIdx.x, gridDim.x * 256);
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

cudaError_t launch_norm_finalize(const float* partial, int tiles, int B, float eps, float* inv_norm, void* diag,
                                 uint16_t diag_bits, cudaStream_t st) {
  if (B <= 0) return cudaSuccess;
  return launch_pdl(norm_finalize_kernel, dim3(B), dim3(256), 0, st, partial, tiles, eps, inv_norm,
                    static_cast<uint4*>(diag), diag_bits);
}

// X (an fp16 pair) = Xf * inv_norm[b], hi = fp16(x), lo = fp16((x - hi) * 2^11),
// 8 elements per thread (n, the elements per matrix, is a multiple of 8 and
// every buffer is 16-byte aligned).
__global__ void __launch_bounds__(256) pair_from_f32_kernel(const float* Xf, const float* inv_norm, __half* Xh,
                                                            __half* Xl, long long n) {
  pdl_launch_dependents();
  pdl_wait();
  const int b = blockIdx.y;
  const float sc = inv_norm[b];
  const long long base = static_cast<long long>(b) * n;
  for (long long i = (static_cast<long long>(blockIdx.x) * 256 + threadIdx.x) * 8; i < n;
       i += static_cast<long long>(gridDim.x) * 256 * 8) {
    const float4* src = reinterpret_cast<const float4*>(Xf + base + i);
    const float4 u0 = src[0], u1 = src[1];
    const float x[8] = {u0.x * sc, u0.y * sc, u0.z * sc, u0.w * sc, u1.x * sc, u1.y * sc, u1.z * sc, u1.w * sc};
    uint32_t h[4], l[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __half2 hh = __floats2half2_rn(x[2 * k], x[2 * k + 1]);
      const float2 hf = __half22float2(hh);
      const __half2 ll = __floats2half2_rn((x[2 * k] - hf.x) * kF16LoScale, (x[2 * k + 1] - hf.y) * kF16LoScale);
      h[k] = *reinterpret_cast<const uint32_t*>(&hh);
      l[k] = *reinterpret_cast<const uint32_t*>(&ll);
    }
    *reinterpret_cast<uint4*>(Xh + base + i) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(Xl + base + i) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

cudaError_t launch_pair_from_f32(const float* Xf, const float* inv_norm, void* Xh, void* Xl, long long n, int B,
                                 int num_sms, cudaStream_t st) {
  if (B <= 0 || n <= 0) return cudaSuccess;
  if (n % 8 || (reinterpret_cast<uintptr_t>(Xf) | reinterpret_cast<uintptr_t>(Xh) | reinterpret_cast<uintptr_t>(Xl)) % 16)
    return cudaErrorInvalidValue;
  long long blocks = (n / 8 + 255) / 256;
  const long long cap = std::max(1LL, 8LL * num_sms / B);  // about 8 blocks per SM over the batch
  if (blocks > cap) blocks = cap;
  return launch_pdl(pair_from_f32_kernel, dim3(static_cast<unsigned>(blocks), B), dim3(256), 0, st, Xf, inv_norm,
                    static_cast<__half*>(Xh), static_cast<__half*>(Xl), n);
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
    epi_final_elem(e, e, b, p, q, v);
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
