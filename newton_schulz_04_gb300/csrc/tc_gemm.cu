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
  // Epilogue staging: per epilogue warp, NBUF sets of four 32 x 32 bf16 boxes
  // (head, residual, and their mirrors), 2 KB each.
  static constexpr int NBUF = 2;
  static constexpr int BOX = 32 * 32 * 2;
  static constexpr int STG_WARP = NBUF * 4 * BOX;
  static constexpr int STG = 4 * STG_WARP;
  static constexpr int STAGES_RAW = (224 * 1024 - STG) / STAGE;
  static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM = STAGES * STAGE + STG + BAR_BYTES + 1024;
  static constexpr uint32_t SWZ = (SWB == 128) ? 2u : 4u;  // descriptor swizzle code
  static constexpr int MN_ATOM = SWB / 2;                  // MN elements per swizzle row (MN-major)
  static constexpr int MN_BOX_BYTES = BK * SWB;            // one [BK x MN_ATOM] box
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  static_assert(STAGES >= 3, "need at least three stages");
  static_assert(SMEM <= 232448, "shared memory budget");
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

// Byte offset inside a [32 rows x 64 B] box stored with the 64-byte TMA swizzle
// (16-byte chunk index XOR-ed with bits 7..8 of the row address).
__device__ __forceinline__ uint32_t sw64(int row, int byte) {
  return static_cast<uint32_t>(row * 64 + ((((byte >> 4) ^ (row >> 1)) & 3) << 4) + (byte & 15));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(a))) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(b))) << 16);
}

// Stage one thread's 32 values (row `row` of a 32 x 32 box) as bf16 head and residual.
__device__ __forceinline__ void stage_rows(uint8_t* box_h, uint8_t* box_l, int row, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float a = v[8 * q + 2 * t], b = v[8 * q + 2 * t + 1];
      h[t] = pack_bf16x2(a, b);
      if (box_l) {
        const float ra = a - __bfloat162float(__float2bfloat16_rn(a));
        const float rb = b - __bfloat162float(__float2bfloat16_rn(b));
        l[t] = pack_bf16x2(ra, rb);
      }
    }
    *reinterpret_cast<uint4*>(box_h + sw64(row, q * 16)) = make_uint4(h[0], h[1], h[2], h[3]);
    if (box_l) *reinterpret_cast<uint4*>(box_l + sw64(row, q * 16)) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

// Stage the transpose: thread `col` holds column `col` of the mirrored box.
__device__ __forceinline__ void stage_cols(uint8_t* box_h, uint8_t* box_l, int col, const float (&v)[32]) {
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const bf16 h = __float2bfloat16_rn(v[j]);
    *reinterpret_cast<bf16*>(box_h + sw64(j, col * 2)) = h;
    if (box_l) *reinterpret_cast<bf16*>(box_l + sw64(j, col * 2)) = __float2bfloat16_rn(v[j] - __bfloat162float(h));
  }
}

// Residual pair R = Rh + Rl for 32 consecutive columns of one row.
__device__ __forceinline__ void load_residual(const EpiParams& e, long long off, uint4 (&rh)[4], uint4 (&rl)[4]) {
  const uint4* ph = reinterpret_cast<const uint4*>(e.Rh + off);
#pragma unroll
  for (int q = 0; q < 4; ++q) rh[q] = ph[q];
  if (e.Rl) {
    const uint4* pl = reinterpret_cast<const uint4*>(e.Rl + off);
#pragma unroll
    for (int q = 0; q < 4; ++q) rl[q] = pl[q];
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) rl[q] = make_uint4(0, 0, 0, 0);
  }
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <int SPLIT, bool BMN, int SWB>
__global__ void __launch_bounds__(192, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmAl,
                   const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmBl,
                   const __grid_constant__ CUtensorMap tmOh, const __grid_constant__ CUtensorMap tmOl,
                   const __grid_constant__ TcArgs args) {
  using C = TcCfg<SPLIT, BMN, SWB>;
  extern __shared__ uint8_t smem_raw[];
  // Swizzled tiles must start on a 1024-byte boundary of the shared window.
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* tiles = smem;
  uint8_t* staging = smem + C::STAGES * C::STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + C::STG);
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
    // Each warp owns 32 accumulator rows (its TMEM lane quarter).  Per 32-column
    // chunk: residual prefetch, tcgen05.ld, fused arithmetic, then either the
    // final write to the caller's matrix or swizzled staging of 32 x 32 bf16
    // boxes (and their transposes for symmetric outputs) that one lane sends to
    // global memory with TMA bulk-tensor stores.
    const int quarter = warp & 3;  // TMEM lanes this warp may read
    const EpiParams& e = args.epi;
    uint8_t* stg = staging + (warp - 2) * C::STG_WARP;
    const bool has_lo = e.Ol != nullptr;
    int tcount = 0, sbuf = 0;
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
      const int r0 = m0 + quarter * 32;
      const int r = r0 + lane;
      const float sc = epi_scale(e, b);
      const long long base = static_cast<long long>(b) * e.bs;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + abuf * C::BN;
#pragma unroll 1
      for (int cc = 0; cc < C::BN / 32; ++cc) {
        const int c0 = n0 + cc * 32;
        if (args.sym && c0 > r0) break;  // the rest of this warp's rows lies above the diagonal
        uint4 rh[4], rl[4];
        if (e.Rh) load_residual(e, base + static_cast<long long>(r) * e.ld + c0, rh, rl);
        float v[32];
        __syncwarp();
        tmem_ld_32x32b_x32(tbase + cc * 32, v);
        if (e.Rh) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t hw[4] = {rh[q].x, rh[q].y, rh[q].z, rh[q].w};
            const uint32_t lw[4] = {rl[q].x, rl[q].y, rl[q].z, rl[q].w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float r0v = bf_lo(hw[u]) + bf_lo(lw[u]);
              const float r1v = bf_hi(hw[u]) + bf_hi(lw[u]);
              v[8 * q + 2 * u] = sc * (e.c_acc * v[8 * q + 2 * u] + e.c_res * r0v);
              v[8 * q + 2 * u + 1] = sc * (e.c_acc * v[8 * q + 2 * u + 1] + e.c_res * r1v);
            }
          }
        } else {
          const float f = sc * e.c_acc;
#pragma unroll
          for (int u = 0; u < 32; ++u) v[u] *= f;
        }
        if (e.c_id != 0.f && r >= c0 && r < c0 + 32 && r < e.rows_valid) {
#pragma unroll
          for (int u = 0; u < 32; ++u)
            if (c0 + u == r) v[u] += e.c_id;
        }
        if (e.final_mode != FINAL_NONE) {
#pragma unroll
          for (int u = 0; u < 32; ++u) epi_final_elem(e, b, r, c0 + u, v[u]);
          continue;
        }
        const bool mirror = args.sym && c0 < r0;  // strictly-lower 32 x 32 block: also store its transpose
        if (lane == 0) bulk_wait_read<C::NBUF - 1>();  // this staging buffer's previous stores have read it
        __syncwarp();
        uint8_t* sb = stg + sbuf * (4 * C::BOX);
        stage_rows(sb, has_lo ? sb + C::BOX : nullptr, lane, v);
        if (mirror) stage_cols(sb + 2 * C::BOX, has_lo ? sb + 3 * C::BOX : nullptr, lane, v);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&tmOh, sb, c0, r0, b);
          if (has_lo) tma_store_3d(&tmOl, sb + C::BOX, c0, r0, b);
          if (mirror) {
            tma_store_3d(&tmOh, sb + 2 * C::BOX, r0, c0, b);
            if (has_lo) tma_store_3d(&tmOl, sb + 3 * C::BOX, r0, c0, b);
          }
          bulk_commit();
        }
        sbuf = (sbuf + 1) % C::NBUF;
      }
      tc_fence_before();
      mbar_arrive(&tempty[abuf]);
    }
    if (lane == 0) bulk_wait_all();  // stores complete before the CTA retires
    __syncwarp();
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
  // Output maps: 32 x 32 bf16 boxes with the 64-byte swizzle (dummies in final mode).
  CUtensorMap mOh, mOl;
  bf16* oh = epi.Oh ? epi.Oh : const_cast<bf16*>(d.A.hi);
  bf16* ol = epi.Ol ? epi.Ol : oh;
  const long long old_ = epi.Oh ? epi.ld : d.A.ld;
  const long long obs = epi.Oh ? epi.bs : d.A.bs;
  const uint64_t orows = epi.Oh ? static_cast<uint64_t>(d.M) : static_cast<uint64_t>(d.M);
  const uint64_t ocols = epi.Oh ? static_cast<uint64_t>(epi.ld) : static_cast<uint64_t>(d.K);
  ok = ok && make_map(&mOh, oh, ocols, orows, d.B, old_, obs, 32, 32, 64);
  ok = ok && make_map(&mOl, ol, ocols, orows, d.B, old_, obs, 32, 32, 64);
  if (!ok) {
    *why = "cuTensorMapEncodeTiled failed";
    return cudaErrorInvalidValue;
  }
  if (epi.final_mode == FINAL_NONE && !epi.Oh) {
    *why = "tensor-core epilogue needs a bf16 output pair";
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
  tc_gemm_kernel<SPLIT, BMN, SWB><<<grid, 192, C::SMEM, st>>>(mA, mAl, mB, mBl, mOh, mOl, a);
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
