// tc_gemm.cu -- batched bf16 tensor-core GEMM / SYRK for sm_103a (tcgen05 + TMEM + TMA).
//
// One persistent CTA per SM walks a list of 128 x 256 output tiles spread over a
// batch of same-shape matrices (DMuon technical summary, §2.2: same-shape
// matrices are batched so small problems still fill the GPU).  For symmetric
// outputs (the Gram matrix G = X X^T and every product of the commuting
// polynomials of G) only tiles that touch the lower triangle are computed; the
// epilogue writes each lower element and its mirror (same section: the
// symmetric products compute only the lower triangle).
//
// Warp roles (192 threads):
//   warp 0      TMA producer: fills a ring of shared-memory stages (mbarrier full/empty)
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer; accumulators are
//               double-buffered in TMEM (2 x 256 fp32 columns) so the epilogue of
//               one tile overlaps the main loop of the next
//   warps 2..5  epilogue: tcgen05.ld of their 32-lane quarter, fused scalar epilogue
//               (EpiParams), global stores
//
// Operand modes (template SPLIT): 1: A*B; 2: Ah*B + Al*B; 3: Ah*Bh + Ah*Bl + Al*Bh where
// X = Xh + Xl is a value split into a bf16 head and a bf16 residual (about 16
// significant bits per operand, fp32 accumulation).  B is read K-major
// ([N, K] row-major, used for symmetric right operands, whose rows are their
// columns) or MN-major ([K, N] row-major, e.g. X in Q X).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace muon {

template <int SPLIT, bool BMN, int SWB>
struct TcCfg {
  static constexpr int BM = 128;
  static constexpr int BN = 256;
  static constexpr int BK = SWB / 2;  // bf16 elements per swizzled row
  static constexpr int A_TILE = BM * BK * 2;
  static constexpr int B_TILE = BN * BK * 2;
  static constexpr int NA = (SPLIT >= 2) ? 2 : 1;
  static constexpr int NB = (SPLIT == 3) ? 2 : 1;
  static constexpr int STAGE = NA * A_TILE + NB * B_TILE;
  static constexpr int STAGES_RAW = (196 * 1024) / STAGE;
  static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM = STAGES * STAGE + BAR_BYTES + 1024;
  static constexpr uint32_t SWZ = (SWB == 128) ? 2u : 4u;  // descriptor swizzle code
  static constexpr int MN_ATOM = SWB / 2;                  // MN elements per swizzle row (MN-major)
  static constexpr int MN_BOX_BYTES = BK * SWB;            // one [BK x MN_ATOM] box
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  static_assert(STAGES >= 2, "need at least two stages");
  static_assert(BAR_BYTES >= (2 * STAGES + 5) * 8 + 8, "barrier area too small");
};

struct TcArgs {
  int M, N, K;  // padded sizes (multiples of 128 / 256 / BK)
  int sym;      // 1: lower-triangle tiles of a symmetric M x M output
  int nI, nJ;   // tile grid of one matrix
  int tpm;      // tiles per matrix
  int total;    // tiles over the batch
  int* status;  // workspace status word
  EpiParams epi;
};

// Tile t of the batch -> (matrix b, row block i, column block j).
__device__ __forceinline__ void decode_tile(const TcArgs& a, int t, int& b, int& i, int& j) {
  b = t / a.tpm;
  const int u = t - b * a.tpm;
  if (a.sym) {
    // Row block i (128 rows) needs column blocks j (256 cols) with 256 j <= 128 i + 127,
    // i.e. j <= i / 2.  Rows 2p and 2p+1 hold p+1 tiles each, starting at p (p + 1).
    int p = static_cast<int>((sqrtf(4.f * static_cast<float>(u) + 1.f) - 1.f) * 0.5f);
    while (p > 0 && p * (p + 1) > u) --p;
    while ((p + 1) * (p + 2) <= u) ++p;
    const int rr = u - p * (p + 1);
    if (rr <= p) {
      i = 2 * p;
      j = rr;
    } else {
      i = 2 * p + 1;
      j = rr - (p + 1);
    }
  } else {
    // Groups of 8 row blocks walked column by column keep a wave's operands in L2.
    constexpr int G = 8;
    const int per = G * a.nJ;
    const int g = u / per;
    const int first = g * G;
    const int gs = min(a.nI - first, G);
    const int w = u - g * per;
    i = first + w % gs;
    j = w / gs;
  }
}

// Epilogue of 32 consecutive accumulator columns of one row.
__device__ __forceinline__ void epi_row32(const EpiParams& e, int b, int r, int c0, float (&v)[32], float sc) {
  if (e.final_mode != FINAL_NONE || (e.sym && !(c0 + 31 < r))) {
#pragma unroll
    for (int j = 0; j < 32; ++j) epi_elem(e, b, r, c0 + j, v[j], sc);
    return;
  }
  const long long base = static_cast<long long>(b) * e.bs;
  const long long roff = base + static_cast<long long>(r) * e.ld + c0;
  if (e.R) {
    const float4* R4 = reinterpret_cast<const float4*>(e.R + roff);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 x = R4[q];
      v[4 * q + 0] = sc * (e.c_acc * v[4 * q + 0] + e.c_res * x.x);
      v[4 * q + 1] = sc * (e.c_acc * v[4 * q + 1] + e.c_res * x.y);
      v[4 * q + 2] = sc * (e.c_acc * v[4 * q + 2] + e.c_res * x.z);
      v[4 * q + 3] = sc * (e.c_acc * v[4 * q + 3] + e.c_res * x.w);
    }
  } else {
    const float f = sc * e.c_acc;
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] *= f;
  }
  if (e.Of) {
    float4* O4 = reinterpret_cast<float4*>(e.Of + roff);
#pragma unroll
    for (int q = 0; q < 8; ++q) O4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  }
  if (e.Oh) {
    uint32_t hw[16], lw[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const bf16 h0 = __float2bfloat16_rn(v[2 * q]);
      const bf16 h1 = __float2bfloat16_rn(v[2 * q + 1]);
      hw[q] = static_cast<uint32_t>(__bfloat16_as_ushort(h0)) |
              (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16);
      const bf16 l0 = __float2bfloat16_rn(v[2 * q] - __bfloat162float(h0));
      const bf16 l1 = __float2bfloat16_rn(v[2 * q + 1] - __bfloat162float(h1));
      lw[q] = static_cast<uint32_t>(__bfloat16_as_ushort(l0)) |
              (static_cast<uint32_t>(__bfloat16_as_ushort(l1)) << 16);
    }
    uint4* H4 = reinterpret_cast<uint4*>(e.Oh + roff);
#pragma unroll
    for (int q = 0; q < 4; ++q) H4[q] = make_uint4(hw[4 * q], hw[4 * q + 1], hw[4 * q + 2], hw[4 * q + 3]);
    if (e.Ol) {
      uint4* L4 = reinterpret_cast<uint4*>(e.Ol + roff);
#pragma unroll
      for (int q = 0; q < 4; ++q) L4[q] = make_uint4(lw[4 * q], lw[4 * q + 1], lw[4 * q + 2], lw[4 * q + 3]);
    }
  }
  if (e.sym) {
    // Mirror: element (r, c0 + j) also goes to (c0 + j, r); across the warp r is
    // consecutive, so each of these stores is one coalesced segment.
#pragma unroll
    for (int j = 0; j < 32; ++j) epi_store_elem(e, base + static_cast<long long>(c0 + j) * e.ld + r, v[j]);
  }
}

template <int SPLIT, bool BMN, int SWB>
__global__ void __launch_bounds__(192, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmAl,
                   const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmBl,
                   const __grid_constant__ TcArgs args) {
  using C = TcCfg<SPLIT, BMN, SWB>;
  extern __shared__ uint8_t smem_raw[];
  // Swizzled tiles must start on a 1024-byte boundary of the shared window.
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* tiles = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;  // [2]
  uint64_t* tempty = tfull + 2;         // [2]
  uint64_t* drain = tempty + 2;         // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (C::NA == 2) tma_prefetch_desc(&tmAl);
    if (C::NB == 2) tma_prefetch_desc(&tmBl);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int nk = args.K / C::BK;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < args.total && ok; t += gridDim.x) {
        int b, i, j;
        decode_tile(args, t, b, i, j);
        const int m0 = i * C::BM, n0 = j * C::BN;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1;
          if (*abort_flag || !mbar_wait(&empty[s], ph ^ 1)) {
            ok = false;
            break;
          }
          uint8_t* st = tiles + s * C::STAGE;
          mbar_arrive_expect_tx(&full[s], C::STAGE);
          const int k0 = kb * C::BK;
          tma_load_3d(&tmA, &full[s], st, k0, m0, b);
          if (C::NA == 2) tma_load_3d(&tmAl, &full[s], st + C::A_TILE, k0, m0, b);
          uint8_t* sb = st + C::NA * C::A_TILE;
          if (!BMN) {
            tma_load_3d(&tmB, &full[s], sb, k0, n0, b);
            if (C::NB == 2) tma_load_3d(&tmBl, &full[s], sb + C::B_TILE, k0, n0, b);
          } else {
#pragma unroll
            for (int q = 0; q < C::BN / C::MN_ATOM; ++q) {
              tma_load_3d(&tmB, &full[s], sb + q * C::MN_BOX_BYTES, n0 + q * C::MN_ATOM, k0, b);
              if (C::NB == 2)
                tma_load_3d(&tmBl, &full[s], sb + C::B_TILE + q * C::MN_BOX_BYTES, n0 + q * C::MN_ATOM, k0, b);
            }
          }
        }
      }
      if (!ok) {
        atomicOr(args.status, kStatusTimeout);
        *abort_flag = 1;
        // Let the copies already issued land before the CTA can exit.
        for (int q = (it > C::STAGES ? it - C::STAGES : 0); q < it; ++q)
          mbar_wait(&full[q % C::STAGES], (q / C::STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = make_idesc_bf16(C::BM, C::BN, BMN);
      constexpr uint32_t SBO = 8 * SWB;
      int it = 0, tcount = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < args.total && ok; t += gridDim.x, ++tcount) {
        const int abuf = tcount & 1;
        const uint32_t aph = (tcount >> 1) & 1;
        if (*abort_flag || !mbar_wait(&tempty[abuf], aph ^ 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + abuf * C::BN;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1;
          if (*abort_flag || !mbar_wait(&full[s], ph)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(tiles + s * C::STAGE);
          const uint32_t al = a0 + C::A_TILE;
          const uint32_t b0 = a0 + C::NA * C::A_TILE;
          const uint32_t bl = b0 + C::B_TILE;
#pragma unroll
          for (int kk = 0; kk < C::BK / 16; ++kk) {
            const uint64_t ad = make_sdesc(a0 + kk * 32, 16, SBO, C::SWZ);
            const uint64_t adl = make_sdesc(al + kk * 32, 16, SBO, C::SWZ);
            const uint64_t bd = BMN ? make_sdesc(b0 + kk * 16 * SWB, C::MN_BOX_BYTES, SBO, C::SWZ)
                                    : make_sdesc(b0 + kk * 32, 16, SBO, C::SWZ);
            const uint64_t bdl = BMN ? make_sdesc(bl + kk * 16 * SWB, C::MN_BOX_BYTES, SBO, C::SWZ)
                                     : make_sdesc(bl + kk * 32, 16, SBO, C::SWZ);
            const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
            tc_mma_bf16(d, ad, bd, idesc, acc);
            if (SPLIT == 2) tc_mma_bf16(d, adl, bd, idesc, 1u);
            if (SPLIT == 3) {
              tc_mma_bf16(d, ad, bdl, idesc, 1u);
              tc_mma_bf16(d, adl, bd, idesc, 1u);
            }
          }
          tc_commit(&empty[s]);  // stage is free once these MMAs have read it
        }
        if (!ok) break;
        tc_commit(&tfull[abuf]);  // accumulator ready for the epilogue
      }
      if (!ok) {
        atomicOr(args.status, kStatusTimeout);
        *abort_flag = 1;
      }
      // Every MMA issued by this thread completes before TMEM is released.
      tc_commit(drain);
      mbar_wait(drain, 0);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM lanes this warp may read
    const EpiParams& e = args.epi;
    int tcount = 0;
    for (int t = blockIdx.x; t < args.total; t += gridDim.x, ++tcount) {
      int b, i, j;
      decode_tile(args, t, b, i, j);
      const int m0 = i * C::BM, n0 = j * C::BN;
      const int abuf = tcount & 1;
      const uint32_t aph = (tcount >> 1) & 1;
      if (*abort_flag || !mbar_wait(&tfull[abuf], aph)) {
        if (lane == 0) atomicOr(args.status, kStatusTimeout);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const int r = m0 + quarter * 32 + lane;
      const int warp_row_max = m0 + quarter * 32 + 31;
      const float sc = epi_scale(e, b);
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + abuf * C::BN;
#pragma unroll 1
      for (int cc = 0; cc < C::BN / 32; ++cc) {
        const int c0 = n0 + cc * 32;
        if (args.sym && c0 > warp_row_max) break;  // rest of the tile is above the diagonal
        float v[32];
        __syncwarp();
        tmem_ld_32x32b_x32(tbase + cc * 32, v);
        epi_row32(e, b, r, c0, v, sc);
      }
      tc_fence_before();
      mbar_arrive(&tempty[abuf]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side

static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 3-D bf16 map over [B][rows][inner] with box {box_inner, box_rows, 1}.
static bool make_map(CUtensorMap* m, const bf16* base, uint64_t inner, uint64_t rows, uint64_t batch,
                     long long ld, long long bs, uint32_t box_inner, uint32_t box_rows, int swb) {
  auto enc = get_encode();
  if (!enc) return false;
  const cuuint64_t dims[3] = {inner, rows, batch};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2, static_cast<cuuint64_t>(bs) * 2};
  const cuuint32_t box[3] = {box_inner, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<bf16*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE,
                         swb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int SPLIT, bool BMN, int SWB>
static cudaError_t launch_impl(const TcGemmDesc& d, const EpiParams& epi, int* status, cudaStream_t st,
                               int num_sms, const char** why) {
  using C = TcCfg<SPLIT, BMN, SWB>;
  {
    const cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<SPLIT, BMN, SWB>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap mA, mAl, mB, mBl;
  bool ok = make_map(&mA, d.A.hi, d.K, d.M, d.B, d.A.ld, d.A.bs, C::BK, C::BM, SWB);
  ok = ok && make_map(&mAl, (C::NA == 2 && d.A.lo) ? d.A.lo : d.A.hi, d.K, d.M, d.B, d.A.ld, d.A.bs, C::BK,
                      C::BM, SWB);
  if (!BMN) {
    ok = ok && make_map(&mB, d.Bop.hi, d.K, d.N, d.B, d.Bop.ld, d.Bop.bs, C::BK, C::BN, SWB);
    ok = ok && make_map(&mBl, (C::NB == 2 && d.Bop.lo) ? d.Bop.lo : d.Bop.hi, d.K, d.N, d.B, d.Bop.ld, d.Bop.bs,
                        C::BK, C::BN, SWB);
  } else {
    ok = ok && make_map(&mB, d.Bop.hi, d.N, d.K, d.B, d.Bop.ld, d.Bop.bs, C::MN_ATOM, C::BK, SWB);
    ok = ok && make_map(&mBl, (C::NB == 2 && d.Bop.lo) ? d.Bop.lo : d.Bop.hi, d.N, d.K, d.B, d.Bop.ld, d.Bop.bs,
                        C::MN_ATOM, C::BK, SWB);
  }
  if (!ok) {
    *why = "cuTensorMapEncodeTiled failed";
    return cudaErrorInvalidValue;
  }
  TcArgs a;
  a.M = d.M;
  a.N = d.N;
  a.K = d.K;
  a.sym = d.sym;
  a.nI = d.M / C::BM;
  a.nJ = d.N / C::BN;
  if (d.sym) {
    const int P = a.nI / 2;
    a.tpm = P * (P + 1);
  } else {
    a.tpm = a.nI * a.nJ;
  }
  a.total = a.tpm * d.B;
  a.status = status;
  a.epi = epi;
  a.epi.sym = d.sym;
  const int grid = a.total < num_sms ? a.total : num_sms;
  if (grid <= 0) return cudaSuccess;
  tc_gemm_kernel<SPLIT, BMN, SWB><<<grid, 192, C::SMEM, st>>>(mA, mAl, mB, mBl, a);
  return cudaGetLastError();
}

cudaError_t launch_tc_gemm(const TcGemmDesc& d, const EpiParams& epi, int* status, cudaStream_t st, int num_sms,
                           const char** why) {
  *why = nullptr;
  if (d.split == 1 && !d.b_mn) return launch_impl<1, false, 128>(d, epi, status, st, num_sms, why);
  if (d.split == 1 && d.b_mn) return launch_impl<1, true, 128>(d, epi, status, st, num_sms, why);
  if (d.split == 2 && d.b_mn) return launch_impl<2, true, 64>(d, epi, status, st, num_sms, why);
  if (d.split == 3 && !d.b_mn) return launch_impl<3, false, 64>(d, epi, status, st, num_sms, why);
  if (d.split == 3 && d.b_mn) return launch_impl<3, true, 64>(d, epi, status, st, num_sms, why);
  *why = "unsupported operand split";
  return cudaErrorInvalidValue;
}

int tc_tiles(int M, int N, int sym) {
  const int nI = M / 128, nJ = N / 256;
  if (sym) return (nI / 2) * (nI / 2 + 1);
  return nI * nJ;
}

}  // namespace muon
