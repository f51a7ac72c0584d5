// adamw.cu -- fused AdamW step over the non-matrix "tail" of a model.
//
// MatrixFSDP technical summary (gist.science 2607.05895), "Metodologia" §1:
// 1-D vectors and other non-matrix tensors are packed into a tail that a
// separate owner updates with standard AdamW.  One launch updates up to
// kMaxTail tensors: a persistent grid strides over groups of 8 elements of
// the concatenated tail, finds each group's tensor by binary search over the
// group offsets, and moves parameters, gradients and both moments with
// 16-byte accesses where the tensor's alignment allows.  Every element is
// read and written once (HBM-bound: 22 B per element with bf16 parameters and
// gradients, 28 B with fp32).
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace muon {

__device__ __forceinline__ void adamw_elem(const AdamwArgs& a, float& p, float g, float& m, float& v) {
  p *= a.decay;                                   // decoupled weight decay
  m = a.beta1 * m + (1.f - a.beta1) * g;
  v = a.beta2 * v + (1.f - a.beta2) * g * g;
  const float denom = sqrtf(v) * a.inv_sqrt_bc2 + a.eps;
  p -= a.step_size * m / denom;
}

template <bool BF16>
__global__ void __launch_bounds__(256) adamw_tail_kernel(const __grid_constant__ AdamwArgs a) {
  __shared__ long long gstart[kMaxTail + 1];
  for (int i = threadIdx.x; i <= a.count; i += blockDim.x) gstart[i] = a.gstart[i];
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();
  const long long total = gstart[a.count];
  for (long long gi = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; gi < total;
       gi += static_cast<long long>(gridDim.x) * blockDim.x) {
    int lo = 0, hi = a.count - 1;  // last tensor whose first group is <= gi
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (gstart[mid] <= gi) lo = mid;
      else hi = mid - 1;
    }
    const int t = lo;
    const long long e0 = (gi - gstart[t]) * 8;
    const long long n = a.numel[t];
    float* m = a.m[t] + e0;
    float* v = a.v[t] + e0;
    if (BF16) {
      bf16* p = static_cast<bf16*>(a.p[t]) + e0;
      const bf16* g = static_cast<const bf16*>(a.g[t]) + e0;
      if (e0 + 8 <= n && a.vec_ok[t]) {
        const uint4 pw = *reinterpret_cast<const uint4*>(p);
        const uint4 gw = *reinterpret_cast<const uint4*>(g);
        float4 m0 = reinterpret_cast<float4*>(m)[0], m1 = reinterpret_cast<float4*>(m)[1];
        float4 v0 = reinterpret_cast<float4*>(v)[0], v1 = reinterpret_cast<float4*>(v)[1];
        const __nv_bfloat162* pp = reinterpret_cast<const __nv_bfloat162*>(&pw);
        const __nv_bfloat162* gg = reinterpret_cast<const __nv_bfloat162*>(&gw);
        float pv[8], gv[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 x = __bfloat1622float2(pp[q]), y = __bfloat1622float2(gg[q]);
          pv[2 * q] = x.x, pv[2 * q + 1] = x.y, gv[2 * q] = y.x, gv[2 * q + 1] = y.y;
        }
        float mv[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
        float vv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int q = 0; q < 8; ++q) adamw_elem(a, pv[q], gv[q], mv[q], vv[q]);
        uint4 po;
        __nv_bfloat162* po2 = reinterpret_cast<__nv_bfloat162*>(&po);
#pragma unroll
        for (int q = 0; q < 4; ++q) po2[q] = __floats2bfloat162_rn(pv[2 * q], pv[2 * q + 1]);
        *reinterpret_cast<uint4*>(p) = po;
        reinterpret_cast<float4*>(m)[0] = make_float4(mv[0], mv[1], mv[2], mv[3]);
        reinterpret_cast<float4*>(m)[1] = make_float4(mv[4], mv[5], mv[6], mv[7]);
        reinterpret_cast<float4*>(v)[0] = make_float4(vv[0], vv[1], vv[2], vv[3]);
        reinterpret_cast<float4*>(v)[1] = make_float4(vv[4], vv[5], vv[6], vv[7]);
      } else {
        const int k = static_cast<int>(n - e0 < 8 ? n - e0 : 8);
        for (int q = 0; q < k; ++q) {
          float pv = __bfloat162float(p[q]);
          adamw_elem(a, pv, __bfloat162float(g[q]), m[q], v[q]);
          p[q] = __float2bfloat16_rn(pv);
        }
      }
    } else {
      float* p = static_cast<float*>(a.p[t]) + e0;
      const float* g = static_cast<const float*>(a.g[t]) + e0;
      if (e0 + 8 <= n && a.vec_ok[t]) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float4 pw = reinterpret_cast<float4*>(p)[h];
          const float4 gw = reinterpret_cast<const float4*>(g)[h];
          float4 mw = reinterpret_cast<float4*>(m)[h], vw = reinterpret_cast<float4*>(v)[h];
          adamw_elem(a, pw.x, gw.x, mw.x, vw.x);
          adamw_elem(a, pw.y, gw.y, mw.y, vw.y);
          adamw_elem(a, pw.z, gw.z, mw.z, vw.z);
          adamw_elem(a, pw.w, gw.w, mw.w, vw.w);
          reinterpret_cast<float4*>(p)[h] = pw;
          reinterpret_cast<float4*>(m)[h] = mw;
          reinterpret_cast<float4*>(v)[h] = vw;
        }
      } else {
        const int k = static_cast<int>(n - e0 < 8 ? n - e0 : 8);
        for (int q = 0; q < k; ++q) adamw_elem(a, p[q], g[q], m[q], v[q]);
      }
    }
  }
}

cudaError_t launch_adamw_tail(const AdamwArgs& a, bool bf16_params, int num_sms, cudaStream_t st) {
  const long long total = a.gstart[a.count];
  if (total <= 0) return cudaSuccess;
  // persistent grid: a few 256-thread blocks per SM, never more than the work
  const long long want = (total + 255) / 256;
  const int grid = static_cast<int>(want < 8LL * num_sms ? want : 8LL * num_sms);
  return bf16_params ? launch_pdl(adamw_tail_kernel<true>, dim3(grid), dim3(256), 0, st, a)
                     : launch_pdl(adamw_tail_kernel<false>, dim3(grid), dim3(256), 0, st, a);
}

}  // namespace muon
