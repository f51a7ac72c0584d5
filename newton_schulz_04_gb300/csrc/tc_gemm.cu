// tc_gemm.cu -- batched bf16 / fp16 tensor-core GEMM / SYRK for sm_103a (tcgen05 + TMEM + TMA).
//
// A persistent grid of CTA pairs works through the 256 x 256 output tiles of a
// batch of same-shape matrices (DMuon technical summary, §2.2: same-shape
// matrices are batched so small problems still fill the GPU).  For symmetric
// outputs (the Gram matrix G = X X^T and every product of the commuting
// polynomials of G) only tiles that touch the lower triangle are computed (same
// section: the symmetric products compute only the lower triangle).
//
// Tile scheduling.  Each pair's leader takes tile indices in order from a
// counter in global memory (atomicAdd) and publishes them to both CTAs through
// a small shared-memory queue, so pairs that start early -- e.g. while the
// previous launch on the stream drains -- take more tiles.
//
// Products per launch.  A launch runs one product, or up to kMaxPhases
// consecutive products ("phases", tc_gemm_kernel<kMaxPhases>) whose tiles form
// one sequence, product by product.  Ordering between products is per matrix
// (TcProgram::done): every epilogue warp adds 1 to its matrix's counter once
// its part of a tile is stored, and a tile of a later product (or of a
// launch chained to the previous one) starts matrix b once the counter shows
// every earlier product finished b -- no grid boundary in between.
//
// Symmetric storage.  A symmetric s x s matrix is stored "block-lower": only
// its 256 x 256 blocks (I, J) with J <= I are written (diagonal blocks in
// full).  When such a matrix is an operand, a 128-deep k-block (one stage)
// that falls in an upper block is read as the transposed (MN-major) boxes of
// the stored lower block and the MMA instruction descriptor switches that operand's major-ness
// for it; so no mirror is ever written.
//
// Warp roles (320 threads):
//   warp 0      TMA producer: fills a ring of shared-memory stages (mbarrier full/empty)
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer; accumulators are
//               double-buffered in TMEM (2 x 256 fp32 columns) so the epilogue of
//               one tile overlaps the main loop of the next
//   warps 2..9  epilogue, WPQ = 2 warps per TMEM lane quarter (warp % 4), each
//               taking every other CH = 32-column chunk of its 32 rows:
//               tcgen05.ld, fused arithmetic (EpiParams) with the residual read
//               coalesced from global memory one chunk ahead, then 32 x 32
//               blocks of 16-bit values (bf16 or fp16 pairs) passed through a
//               padded shared-memory box and written with row-contiguous
//               16-byte stores.  With one warp per scheduler the epilogue ran
//               at a fraction of the issue rate and, at K = 1024, took as long
//               as the main loop
//
// Split operands.  A value X carried as a bf16 head Xh and a bf16 residual Xl
// (X ~ Xh + Xl to ~16 significant bits) is multiplied as a sum of plain bf16
// products: Ah Bh + Ah Bl + Al Bh (three "K segments", the lo*lo term dropped)
// or Ah B + Al B (two).  Each segment is an ordinary pass over K with its own
// pair of tensor maps, all accumulating into the same TMEM tile, so split
// products run on the same 128-byte-swizzled pipeline as plain ones.
//
// Scaled fp16 pairs (split 5).  A value carried as an fp16 pair, hi = fp16(v)
// and lo = fp16((v - hi) * 2^11) (about 22 significant bits), is multiplied as
// hi*lo + lo*hi (two K segments, accumulated at 2^11 times their true scale)
// followed by hi*hi, whose first MMA scales the accumulator by 2^-11 on input
// (tcgen05 scale-input-d): D = hi*hi + (hi*lo + lo*hi) / 2^11 in one TMEM tile.
//
// Diagonal segment.  For C = A B + d B_lo with A square (K == M), B MN-major
// and d a scalar, the term d B_lo runs on the tensor cores too: rows 256 p ..
// 256 p + 255 of d B_lo are D B_lo[256 p .. 256 p + 255, :] with D = d I (256
// x 256), so a CTA pair appends two 128-deep k-blocks to its tile whose A
// operand is its 128 rows of D (loaded from a small table) and whose B
// operand is the pair's own 256 rows of B_lo.  This costs 256 more of K per
// tile and takes the residual out of the epilogue, which at K ~ 1024 sets the
// pace (the main loop is short).

// B is read K-major ([N, K] row-major: symmetric right operands, whose rows are
// their columns) or MN-major ([K, N] row-major, e.g. X in B X or Q X).
//
// CTA pairs (2-SM MMA).  CTAs run in clusters of two that compute one 256 x 256
// output tile together: row blocks 2p (leader, rank 0) and 2p + 1 (rank 1).
// Each CTA loads its own 128 rows of A and one half (128 columns) of B into its
// own shared memory, signalling the leader's stage barrier; the leader issues
// tcgen05.mma.cta_group::2 (M = 256), which reads A from each CTA and B from
// both, and leaves each CTA's 128 rows of the accumulator in that CTA's TMEM.
// Per SM this is 8 KB of operands per 256 x 256 x 16 step instead of 12 KB for a
// single-CTA 128 x 256 x 16 step, which ran at about half the tensor rate.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <memory>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace muon {

struct TcCfg {
  static constexpr int BM = 128;
  static constexpr int BN = 256;
  // A stage covers 128 of K as two 64-element (128-byte) swizzle atoms, i.e.
  // 8 MMAs per stage barrier: with 64-wide stages the per-stage wait / commit
  // round trip left the tensor pipe idle ~45 % of the time.
  static constexpr int KA = 64;           // bf16 elements per 128-byte swizzled row
  static constexpr int BK = 128;          // K per stage
  static constexpr int KATOMS = BK / KA;  // K-major swizzle atoms per operand per stage
  static constexpr int BNH = BN / 2;      // B columns held by each CTA of the pair
  static constexpr int KATOM_BYTES = 128 * KA * 2;  // one K-major atom of 128 rows
  static constexpr int A_TILE = BM * BK * 2;
  static constexpr int B_TILE = BNH * BK * 2;  // this CTA's half of the B tile
  static constexpr int STAGE = A_TILE + B_TILE;
  static constexpr int STAGES = 3;
  // Epilogue: WPQ warps per TMEM lane quarter; warp q of a quarter takes the
  // chunks q, q + WPQ, ... of CH columns of its 32 rows.  Each warp stages
  // its outputs through one padded 32-row box (rows of 2 CH bytes, 16 bytes
  // of padding), which it writes and reads back itself.
  static constexpr int CH = 32;
  static constexpr int WPQ = 2;
  static constexpr int EPI_WARPS = 4 * WPQ;
  static constexpr int NCHT = BN / CH;  // chunks per tile row
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int ROWBOX = 32 * (2 * CH + 16);
  static constexpr int STG = EPI_WARPS * ROWBOX;
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM = STAGES * STAGE + STG + BAR_BYTES + 1024;
  static constexpr uint32_t SWZ = 2u;            // descriptor code for the 128-byte swizzle
  static constexpr int MN_ATOM = 64;             // MN elements per swizzled row (MN-major)
  static constexpr int MN_BOX_BYTES = BK * 128;  // one [BK x MN_ATOM] box (MN-major atom)
  static_assert(BM == 128 && BNH == 128, "K-major atoms hold 128 rows");
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  static constexpr uint32_t EPI_ARRIVALS = 2 * EPI_WARPS;  // epilogue warps of both CTAs release a TMEM buffer
  // Tile queue: the leader's producer fetches tile indices from a counter in
  // global memory and publishes them to both CTAs; QD slots deep.  A slot is
  // free again once the peer producer, the MMA issuer and the epilogue warps
  // of both CTAs have read it.
  static constexpr int QD = 4;
  static constexpr uint32_t Q_ARRIVALS = 2 + 2 * EPI_WARPS;
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(BAR_BYTES >= (2 * STAGES + 5 + 2 * QD) * 8 + 4 * QD + 8, "barrier area too small");
  static_assert((CH == 16 || CH == 32) && WPQ >= 1 && NCHT >= WPQ, "epilogue chunking");
};

// One product of a launch.  A launch runs up to NPH products ("phases") on
// one persistent grid: their tile pairs form one sequence, phase by phase and
// within a phase matrix by matrix, which the CTA pairs take in order from
// tile_ctr.  A tile of a phase with `wait` starts once its matrix's counter
// shows that every earlier product of that matrix has finished.
struct TcPhase {
  CUtensorMap tm[9];  // see TcMap
  int M, N, K;    // padded sizes (multiples of 256 / 256 / 128)
  int sym;        // 1: lower-triangle tiles of a symmetric M x M output
  int nI, nJ;     // tile grid of one matrix
  int tpm;        // tile pairs per matrix
  int first;      // index of this phase's first tile pair in the launch's sequence
  int nseg;       // K segments (1 plain, 2 or 3 split)
  int a_sym;      // A is a symmetric matrix in block-lower storage (upper k-blocks read transposed)
  int b_sym;      // same for B (K-major B only)
  int bmn;        // 1: B is MN-major ([K, N] row-major), 0: K-major ([N, K])
  int seg_lo;     // bit 2s: segment s reads A's residual map; bit 2s+1: B's residual map
  int diag_kb;    // k-blocks of the diagonal segment (0, or 256 / BK: D times B's residual rows)
  int final_vec;    // final mode may use 16-byte accesses to the caller's rows (matrices stored as packed)
  int final_vec_t;  // the same for matrices stored transposed (rows of length rows_valid)
  int f16;        // operands are fp16 (else bf16)
  int pair_scale; // 1: the last segment's first MMA scales the accumulator by 2^-11 (split 5)
  int rgroup;     // rectangular products: row-block pairs per column-major group of tiles
  // With `wait`, a tile of matrix b starts once done[b] >= wait_target
  // instead of after the whole previous grid (griddepcontrol.wait).
  int wait;
  int wait_target;
  EpiCore epi;
};
// Tensor maps of a phase: A's K-major boxes, its residual's, A's transposed
// (MN-major) boxes and its residual's; the same four for B (for an MN-major B
// the transposed maps repeat the plain ones); D of the diagonal segment.
enum TcMap { kMapA = 0, kMapAl, kMapAt, kMapAtl, kMapB, kMapBl, kMapBt, kMapBtl, kMapD };

template <int NPH>
struct TcProgram {
  int nph;        // phases in use
  int total;      // tile pairs over all phases
  int* status;    // workspace status word
  // Per-matrix completion counters (or nullptr).  Every epilogue warp adds 1
  // to done[b] once its part of a tile of matrix b is stored.
  int* done;
  int* tile_ctr;  // zeroed before the launch; tiles are taken in order by atomicAdd
  EpiFinal fin;   // the final modes' per-matrix tables (one final product per launch)
  TcPhase ph[NPH];
};
constexpr int kMaxPhases = 16;
static_assert(sizeof(TcProgram<kMaxPhases>) <= 32000, "kernel parameter space");

// Tile pair t of the batch -> (matrix b, row-block pair p, column block j); the
// CTA of rank r in the cluster computes row block i = 2 p + r.
__device__ __forceinline__ void decode_pair(const TcPhase& a, int t, int& b, int& p, int& j) {
  b = t / a.tpm;
  const int u = t - b * a.tpm;
  if (a.sym) {
    // Row blocks 2p and 2p+1 (256 rows) need column blocks j <= p: p + 1 pairs,
    // starting at p (p + 1) / 2.
    int q = static_cast<int>((sqrtf(8.f * static_cast<float>(u) + 1.f) - 1.f) * 0.5f);
    while (q > 0 && q * (q + 1) / 2 > u) --q;
    while ((q + 1) * (q + 2) / 2 <= u) ++q;
    p = q;
    j = u - q * (q + 1) / 2;
  } else {
    // Groups of rgroup row-block pairs walked column by column: the group's
    // rows of A stay in L2 while each column block of B is read once per group.
    const int G = a.rgroup;
    const int nP = a.nI / 2;
    const int per = G * a.nJ;
    const int g = u / per;
    const int first = g * G;
    const int gs = min(nP - first, G);
    const int w = u - g * per;
    p = first + w % gs;
    j = w / gs;
  }
}


__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // a in the low half
  return *reinterpret_cast<const uint32_t*>(&h);
}

// One chunk of 32 accumulator rows (this warp's lane quarter) from TMEM.
__device__ __forceinline__ void tmem_ld_rows(uint32_t taddr, float (&v)[32]) { tmem_ld_32x32b_x32(taddr, v); }
__device__ __forceinline__ void tmem_ld_rows(uint32_t taddr, float (&v)[16]) { tmem_ld_32x32b_x16(taddr, v); }

__device__ __forceinline__ uint32_t pack2_h(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);  // a in the low half
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack2_h(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

// Split N values into packed 16-bit pairs: bf16 head hw = bf16(v), residual
// lw = bf16(v - head); or fp16 head hw = fp16(v), residual lw = fp16((v - head) * lo_scale).
template <int N>
__device__ __forceinline__ void split_words(const float (&v)[N], uint32_t (&hw)[N / 2], uint32_t (&lw)[N / 2],
                                            bool want_lo, bool f16, float lo_scale) {
  if (f16) {
#pragma unroll
    for (int k = 0; k < N / 2; ++k) {
      hw[k] = pack2_h(v[2 * k], v[2 * k + 1]);
      if (want_lo) {
        const float2 h = unpack2_h(hw[k]);
        lw[k] = pack2_h((v[2 * k] - h.x) * lo_scale, (v[2 * k + 1] - h.y) * lo_scale);
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < N / 2; ++k) {
      hw[k] = pack2(v[2 * k], v[2 * k + 1]);
      if (want_lo) lw[k] = pack2(v[2 * k] - bf_lo(hw[k]), v[2 * k + 1] - bf_hi(hw[k]));
    }
  }
}

// Store a 32 x CH block of 16-bit values to dst (row stride ld elements):
// lane t holds row t as CH / 2 packed words.  The rows go through the warp's
// padded box (row stride 2 CH + 16 bytes: the 16-byte accesses of a phase of
// 8 lanes hit distinct banks), then each warp-wide 16-byte store covers whole
// row segments of 2 CH bytes.
template <int CH>
__device__ __forceinline__ void store_block16(uint16_t* dst, long long ld, int lane, const uint32_t (&w)[CH / 2],
                                              uint8_t* box) {
  constexpr int STRIDE = 2 * CH + 16, P = 2 * CH / 16, RPI = 32 / P;
#pragma unroll
  for (int q = 0; q < P; ++q)
    *reinterpret_cast<uint4*>(box + lane * STRIDE + q * 16) =
        make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
  __syncwarp();
#pragma unroll
  for (int it = 0; it < P; ++it) {
    const int row = it * RPI + lane / P, pc = lane % P;
    *reinterpret_cast<uint4*>(dst + row * ld + pc * 8) = *reinterpret_cast<const uint4*>(box + row * STRIDE + pc * 16);
  }
  __syncwarp();
}

// Final write of a full 32 x CH block to a caller's row-major matrix (not
// transposed): global memory is read and written a warp-wide few rows at a time
// through a padded shared-memory box, lane t owning row t in between.
template <typename T, int CH>
__device__ __forceinline__ void final_block_rows(const EpiCore& e, const EpiFinal& f, int b, int r0, int c0,
                                                 int lane, const float (&v)[CH], uint8_t* box) {
  constexpr int ROWB = CH * static_cast<int>(sizeof(T));  // bytes of one block row
  constexpr int STRIDE = ROWB + 16;                        // padded row stride in shared memory
  constexpr int PIECES = ROWB / 16;                        // 16-byte pieces per row
  constexpr int ROWS_PER = 32 / PIECES;                    // rows covered by one warp-wide access
  constexpr int EPP = 16 / static_cast<int>(sizeof(T));    // elements per piece
  const long long cols = e.cols_valid;
  T* dst = static_cast<T*>(f.dst[b]);
  const bool apply = e.final_mode == FINAL_APPLY;
  if (apply) {
#pragma unroll
    for (int it = 0; it < PIECES; ++it) {
      const int row = it * ROWS_PER + lane / PIECES, pc = lane % PIECES;
      const uint4 x = *reinterpret_cast<const uint4*>(dst + (r0 + row) * cols + c0 + pc * EPP);
      *reinterpret_cast<uint4*>(box + row * STRIDE + pc * 16) = x;
    }
    __syncwarp();
  }
  // lane owns row `lane`
#pragma unroll
  for (int pc = 0; pc < PIECES; ++pc) {
    uint4* p = reinterpret_cast<uint4*>(box + lane * STRIDE + pc * 16);
    if (sizeof(T) == 2) {
      uint32_t w[4];
      if (apply) {
        const uint4 x = *p;
        const uint32_t in[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int u = 0; u < 4; ++u)
          w[u] = pack2(bf_lo(in[u]) - e.lr * v[pc * 8 + 2 * u], bf_hi(in[u]) - e.lr * v[pc * 8 + 2 * u + 1]);
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) w[u] = pack2(v[pc * 8 + 2 * u], v[pc * 8 + 2 * u + 1]);
      }
      *p = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      float4 y;
      if (apply) {
        const float4 x = *reinterpret_cast<const float4*>(p);
        y = make_float4(x.x - e.lr * v[pc * 4], x.y - e.lr * v[pc * 4 + 1], x.z - e.lr * v[pc * 4 + 2],
                        x.w - e.lr * v[pc * 4 + 3]);
      } else {
        y = make_float4(v[pc * 4], v[pc * 4 + 1], v[pc * 4 + 2], v[pc * 4 + 3]);
      }
      *reinterpret_cast<float4*>(p) = y;
    }
  }
  __syncwarp();
#pragma unroll
  for (int it = 0; it < PIECES; ++it) {
    const int row = it * ROWS_PER + lane / PIECES, pc = lane % PIECES;
    *reinterpret_cast<uint4*>(dst + (r0 + row) * cols + c0 + pc * EPP) =
        *reinterpret_cast<const uint4*>(box + row * STRIDE + pc * 16);
  }
  __syncwarp();
}

// Final write of a full 32 x CH block to a caller's bf16 matrix stored
// transposed (dst[b] is [cols_valid, rows_valid]): the block is CH rows of dst
// (packed columns c0 ..) by 32 columns (packed rows r0 .., one per lane).
// Rows of dst are read and written 16 bytes at a time through the warp's box
// (CH rows of 64 bytes, 16 bytes of padding each); in between, lane t updates
// column t of the box, 2 bytes per row (lanes t and t + 1 share a 4-byte word,
// so a warp's accesses fall in 16 distinct banks).
template <int CH>
__device__ __forceinline__ void final_block_cols(const EpiCore& e, const EpiFinal& f, int b, int r0, int c0,
                                                 int lane, const float (&v)[CH], uint8_t* box) {
  constexpr int STRIDE = 32 * 2 + 16;         // one dst row of the block: 32 bf16 values, padded
  constexpr int PIECES = CH * 4;              // 16-byte pieces of the block (4 per row)
  static_assert(PIECES % 32 == 0 && CH * STRIDE <= 32 * (2 * CH + 16), "block fits the warp's box");
  const long long ldd = e.rows_valid;         // dst row length
  uint16_t* dst = static_cast<uint16_t*>(f.dst[b]);
  const bool apply = e.final_mode == FINAL_APPLY;
  if (apply) {
#pragma unroll
    for (int it = 0; it < PIECES / 32; ++it) {
      const int k = it * 32 + lane, row = k >> 2, pc = k & 3;
      *reinterpret_cast<uint4*>(box + row * STRIDE + pc * 16) =
          *reinterpret_cast<const uint4*>(dst + (c0 + row) * ldd + r0 + pc * 8);
    }
    __syncwarp();
  }
#pragma unroll
  for (int u = 0; u < CH; ++u) {
    uint16_t* q = reinterpret_cast<uint16_t*>(box + u * STRIDE) + lane;
    float w = v[u];
    if (apply) w = __uint_as_float(static_cast<uint32_t>(*q) << 16) - e.lr * v[u];
    const bf16 h = __float2bfloat16_rn(w);
    *q = *reinterpret_cast<const uint16_t*>(&h);
  }
  __syncwarp();
#pragma unroll
  for (int it = 0; it < PIECES / 32; ++it) {
    const int k = it * 32 + lane, row = k >> 2, pc = k & 3;
    *reinterpret_cast<uint4*>(dst + (c0 + row) * ldd + r0 + pc * 8) =
        *reinterpret_cast<const uint4*>(box + row * STRIDE + pc * 16);
  }
  __syncwarp();
}

template <int NPH>
__global__ void __launch_bounds__(TcCfg::THREADS, 1) tc_gemm_kernel(const __grid_constant__ TcProgram<NPH> prog) {
  using C = TcCfg;
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
  uint64_t* qfull = drain + 1;          // [QD] tile index published
  uint64_t* qempty = qfull + C::QD;     // [QD] (leader) slot read by every consumer
  volatile int* tq = reinterpret_cast<volatile int*>(qempty + C::QD);  // [QD] tile indices (-1: no more)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(const_cast<int*>(tq) + C::QD);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);   // leader: its arrive + the bytes of both CTAs
      mbar_init(&empty[s], 1);  // the leader's MMA commit, multicast to both CTAs
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], C::EPI_ARRIVALS);
    }
    mbar_init(drain, 1);
    for (int q = 0; q < C::QD; ++q) {
      mbar_init(&qfull[q], 1);
      mbar_init(&qempty[q], C::Q_ARRIVALS);
    }
    *abort_flag = 0;
    fence_mbar_init();
    for (int pi = 0; pi < prog.nph; ++pi) {
      const TcPhase& phs = prog.ph[pi];
      tma_prefetch_desc(&phs.tm[kMapA]);
      tma_prefetch_desc(&phs.tm[kMapB]);
      if (phs.nseg > 1 || phs.diag_kb) {
        tma_prefetch_desc(&phs.tm[kMapAl]);
        tma_prefetch_desc(&phs.tm[kMapBl]);
      }
      if (phs.diag_kb) tma_prefetch_desc(&phs.tm[kMapD]);
    }
  }
  if (warp == 1) {  // both CTAs: the pair's TMEM is allocated collectively
    tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncwarp();
  cluster_sync();  // the peer's barriers exist before any multicast reaches them
  tc_fence_after();
  pdl_launch_dependents();
  // Inputs are written by earlier kernels on the stream: wait for the whole
  // previous grid, or, chained per matrix, for that matrix's counter below.
  if (!prog.ph[0].wait) pdl_wait();
  const int rank = static_cast<int>(cluster_ctarank());
  const uint32_t tmem_base = *tmem_slot;
  // Tile k of this cluster's sequence (every role reads the same sequence):
  // returns the tile index, -1 at the end, -2 on a timeout.
  auto take_tile = [&](int k) -> int {
    const int slot = k % C::QD;
    if (*abort_flag || !mbar_wait_cluster(&qfull[slot], (k / C::QD) & 1)) return -2;
    return tq[slot];
  };
  auto release_tile = [&](int k) { mbar_arrive_cluster(mapa_cluster(&qempty[k % C::QD], 0)); };
  // phase of tile pair t of the sequence
  auto phase_of = [&](int t) -> int {
    int pi = 0;
    if (NPH > 1)
      while (pi + 1 < prog.nph && t >= prog.ph[pi + 1].first) ++pi;
    return pi;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int it = 0;
      bool ok = true;
      int ready_b = -1, ready_pi = -1;  // last (phase, matrix) whose inputs are known to be complete
      // Leader: take tiles from the counter and publish them to both CTAs.
      // Tile k + 1 is fetched when tile k starts (the atomic's result is
      // only read after tile k's loads are issued, so its round trip overlaps
      // them) and published once those loads are out.
      int pub = 0;         // tiles published so far (the last may be the -1 end mark)
      bool ended = false;  // the end mark is published
      auto publish = [&](int t) -> bool {
        const int slot = pub % C::QD;
        const bool live = !*abort_flag && mbar_wait(&qempty[slot], ((pub / C::QD) & 1) ^ 1);
        if (!live || t >= prog.total) t = -1;
        tq[slot] = t;
        st_shared_cluster(mapa_cluster(const_cast<int*>(&tq[slot]), 1), t);
        mbar_arrive_cluster(mapa_cluster(&qfull[slot], 0));
        mbar_arrive_cluster(mapa_cluster(&qfull[slot], 1));
        ++pub;
        ended = t < 0;
        return live;
      };
      if (rank == 0 && !publish(atomicAdd(prog.tile_ctr, 1))) ok = false;
      for (int k = 0; ok; ++k) {
        int t;
        int fetched = -1;  // the next tile (leader), in flight during this tile's loads
        if (rank == 0) {
          t = tq[k % C::QD];  // this thread published it
          if (t >= 0 && !ended) fetched = atomicAdd(prog.tile_ctr, 1);
        } else {
          t = take_tile(k);
          if (t == -2) {
            ok = false;
            break;
          }
          release_tile(k);
        }
        if (t < 0) break;
        const int pi = phase_of(t);
        const TcPhase& phs = prog.ph[pi];
        int b, p, j;
        decode_pair(phs, t - phs.first, b, p, j);
        const int m0 = (2 * p + rank) * C::BM, n0 = j * C::BN;
        if (phs.wait && (b != ready_b || pi != ready_pi)) {
          if (!wait_counter(&prog.done[b], phs.wait_target)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();  // the TMA loads below read what that matrix's writers stored
          ready_b = b;
          ready_pi = pi;
        }
        const int nk = phs.K / C::BK;         // k-blocks per segment
        const int nks = nk * phs.nseg;        // k-blocks of the segments over K
        const int nkb = nks + phs.diag_kb;    // k-blocks of this tile
        const CUtensorMap* tm = phs.tm;
        // the phase's flags, read once per tile from the kernel-parameter block
        const int seg_lo = phs.seg_lo, pa_sym = phs.a_sym, pb_sym = phs.b_sym, pbmn = phs.bmn;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1;
          if (*abort_flag || !mbar_wait(&empty[s], ph ^ 1)) {
            ok = false;
            break;
          }
          uint8_t* st = tiles + s * C::STAGE;
          // both CTAs' copies complete on the leader's barrier for this stage
          const uint32_t fbar = mapa_cluster(&full[s], 0);
          if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * C::STAGE);
          uint8_t* sb = st + C::A_TILE;
          const int nb0 = n0 + rank * C::BNH;  // this CTA's half of the B tile: columns nb0 .. nb0 + 127
          if (kb >= nks) {
            // diagonal segment: this CTA's 128 rows of D, and the pair's own
            // rows of B's residual (256 p + 128 dk ..), MN-major
            const int dk = (kb - nks) * C::BK;
#pragma unroll
            for (int g = 0; g < C::KATOMS; ++g)
              tma_load_3d_pair(&tm[kMapD], fbar, st + g * C::KATOM_BYTES, dk + g * C::KA, rank * C::BM, 0);
#pragma unroll
            for (int q = 0; q < C::BNH / C::MN_ATOM; ++q)
              tma_load_3d_pair(&tm[kMapBl], fbar, sb + q * C::MN_BOX_BYTES, nb0 + q * C::MN_ATOM,
                               2 * p * C::BM + dk, b);
            continue;
          }
          const int seg = kb / nk;
          const int k0 = (kb - seg * nk) * C::BK;
          const bool alo = (seg_lo >> (2 * seg)) & 1;
          const bool blo = (seg_lo >> (2 * seg + 1)) & 1;
          // k-blocks above the diagonal of a block-lower symmetric operand come
          // from the stored lower block, read transposed
          const bool a_up = pa_sym && (k0 >> 8) > (m0 >> 8);
          const bool b_up = !pbmn && pb_sym && (k0 >> 8) > (n0 >> 8);
          if (!a_up) {
#pragma unroll
            for (int g = 0; g < C::KATOMS; ++g)
              tma_load_3d_pair(&tm[alo ? kMapAl : kMapA], fbar, st + g * C::KATOM_BYTES, k0 + g * C::KA, m0, b);
          } else {
#pragma unroll
            for (int q = 0; q < C::BM / C::MN_ATOM; ++q)
              tma_load_3d_pair(&tm[alo ? kMapAtl : kMapAt], fbar, st + q * C::MN_BOX_BYTES, m0 + q * C::MN_ATOM,
                               k0, b);
          }
          if (!pbmn && !b_up) {
#pragma unroll
            for (int g = 0; g < C::KATOMS; ++g)
              tma_load_3d_pair(&tm[blo ? kMapBl : kMapB], fbar, sb + g * C::KATOM_BYTES, k0 + g * C::KA, nb0, b);
          } else {
            const CUtensorMap* mb = &tm[pbmn ? (blo ? kMapBl : kMapB) : (blo ? kMapBtl : kMapBt)];
#pragma unroll
            for (int q = 0; q < C::BNH / C::MN_ATOM; ++q)
              tma_load_3d_pair(mb, fbar, sb + q * C::MN_BOX_BYTES, nb0 + q * C::MN_ATOM, k0, b);
          }
        }
        if (rank == 0 && ok && !ended && !publish(fetched)) ok = false;
      }
      if (!ok) {
        atomicOr(prog.status, kStatusTimeout);
        *abort_flag = 1;
        // Let the copies already issued land before the CTAs can exit (the
        // leader's barriers count the bytes of both CTAs).
        if (rank == 0)
          for (int q = (it > C::STAGES ? it - C::STAGES : 0); q < it; ++q)
            mbar_wait(&full[q % C::STAGES], (q / C::STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ------------------------------------------------------------ MMA issuer (leader)
      constexpr uint32_t SBO = 8 * 128;
      int it = 0, tcount = 0;
      bool ok = true;
      for (int k = 0; ok; ++k, ++tcount) {
        const int t = take_tile(k);
        if (t == -2) {
          ok = false;
          break;
        }
        release_tile(k);
        if (t < 0) break;
        const TcPhase& phs = prog.ph[phase_of(t)];
        int b, p, j;
        decode_pair(phs, t - phs.first, b, p, j);
        const int m0 = (2 * p + rank) * C::BM, n0 = j * C::BN;
        const int nk = phs.K / C::BK;
        const int nks = nk * phs.nseg;
        const int nkb = nks + phs.diag_kb;
        // the phase's flags, read once per tile from the kernel-parameter block
        const int pa_sym = phs.a_sym, pb_sym = phs.b_sym, pbmn = phs.bmn, pf16 = phs.f16;
        const int pscale = phs.pair_scale;
        const int abuf = tcount & 1;
        const uint32_t aph = (tcount >> 1) & 1;
        if (*abort_flag || !mbar_wait(&tempty[abuf], aph ^ 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + abuf * C::BN;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1;
          if (*abort_flag || !mbar_wait(&full[s], ph)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // the diagonal segment's A (D) is K-major and its B MN-major
          const bool dseg = kb >= nks;
          const int k0 = dseg ? 0 : (kb % nk) * C::BK;
          const bool a_mn = !dseg && pa_sym && (k0 >> 8) > (m0 >> 8);
          const bool b_mn = pbmn || (!dseg && pb_sym && (k0 >> 8) > (n0 >> 8));
          const uint32_t idesc =
              make_idesc_f16kind(2 * C::BM, C::BN, b_mn, pf16 == 0) | (a_mn ? (1u << 15) : 0u);
          const uint32_t a0 = smem_u32(tiles + s * C::STAGE);
          const uint32_t b0 = a0 + C::A_TILE;
#pragma unroll
          for (int kk = 0; kk < C::BK / 16; ++kk) {
            // K-major: atom kk / 4, 32 bytes per 16 of K inside it; MN-major: 16 rows of 128 B
            const uint32_t koff = (kk / 4) * C::KATOM_BYTES + (kk % 4) * 32;
            const uint64_t ad = a_mn ? make_sdesc(a0 + kk * 16 * 128, C::MN_BOX_BYTES, SBO, C::SWZ)
                                     : make_sdesc(a0 + koff, 16, SBO, C::SWZ);
            const uint64_t bd = b_mn ? make_sdesc(b0 + kk * 16 * 128, C::MN_BOX_BYTES, SBO, C::SWZ)
                                     : make_sdesc(b0 + koff, 16, SBO, C::SWZ);
            if (pscale && kb == nks - nk && kk == 0)
              tc_mma_pair_scale_d<11>(d, ad, bd, idesc);  // hi*hi + (cross terms) * 2^-11
            else
              tc_mma_pair(d, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit_pair(&empty[s], 0x3);  // both CTAs' stage s is free once these MMAs have read it
        }
        if (!ok) break;
        tc_commit_pair(&tfull[abuf], 0x3);  // both CTAs' accumulators ready for their epilogues
      }
      if (!ok) {
        atomicOr(prog.status, kStatusTimeout);
        *abort_flag = 1;
      }
      // Every MMA issued by this thread completes before TMEM is released.
      tc_commit_pair(drain, 0x1);
      mbar_wait(drain, 0);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    constexpr int CH = C::CH;
    constexpr int P = 2 * CH / 16;  // 16-byte pieces per row of a chunk
    constexpr int RPI = 32 / P;     // rows covered by one warp-wide coalesced access
    const int quarter = warp & 3;   // TMEM lanes this warp may read
    const int ew = warp - 2;
    const int jq = ew >> 2;         // this warp's index among the WPQ warps of its quarter
    const EpiFinal& f = prog.fin;
    uint8_t* box = staging + ew * C::ROWBOX;
    const uint4 zero4 = make_uint4(0, 0, 0, 0);
    int tcount = 0;
    bool ok = true;
    for (int k = 0; ok; ++k, ++tcount) {
      int t = 0;
      if (lane == 0) t = take_tile(k);
      t = __shfl_sync(0xffffffffu, t, 0);
      if (t == -2) {
        ok = false;
        break;
      }
      __syncwarp();
      if (lane == 0) release_tile(k);
      if (t < 0) break;
      const TcPhase& phs = prog.ph[phase_of(t)];
      const EpiCore& e = phs.epi;
      const bool has_lo = e.Ol != nullptr;
      const bool has_r = e.Rh != nullptr;
      const bool has_rl = e.Rl != nullptr;
      int b, p, j;
      decode_pair(phs, t - phs.first, b, p, j);
      const int m0 = (2 * p + rank) * C::BM;
      const int r0 = m0 + quarter * 32;
      const int r = r0 + lane;
      const int cb = j * C::BN;  // first column of the tile
      if (phs.wait && has_r) {
        // the residual may be an earlier product's output: acquire its
        // counter before the first residual load below
        if (lane == 0 && !wait_counter(&prog.done[b], phs.wait_target)) ok = false;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
      // While the main loop runs, pull this lane's rows of the residual (and,
      // in the final apply, of the caller's W) into L2 (one warp per quarter).
      const long long roff = static_cast<long long>(b) * e.bs + static_cast<long long>(r) * e.ld + cb;
      if (jq == 0) {
        if (has_r) bulk_prefetch_l2(static_cast<const uint16_t*>(e.Rh) + roff, C::BN * 2);
        if (has_rl) bulk_prefetch_l2(static_cast<const uint16_t*>(e.Rl) + roff, C::BN * 2);
        if (e.final_mode == FINAL_APPLY && !f.tr[b] && phs.final_vec && r < e.rows_valid &&
            cb + C::BN <= e.cols_valid) {
          const int esz = e.dst_fp32 ? 4 : 2;
          bulk_prefetch_l2(
              static_cast<const uint8_t*>(f.dst[b]) + (static_cast<long long>(r) * e.cols_valid + cb) * esz,
              C::BN * esz);
        }
      }
      // Residual loads: through the read-only cache, unless the previous launch
      // may still be writing other matrices (chained), then from L2.
      const bool coherent = phs.wait != 0;
      auto ld16 = [&](const uint16_t* q) {
        return coherent ? __ldcg(reinterpret_cast<const uint4*>(q)) : __ldg(reinterpret_cast<const uint4*>(q));
      };
      // Each chunk of the residual (32 rows x 2 CH bytes per part) is read
      // coalesced: load `it` of lane `lane` is row it * RPI + lane / P, 16
      // bytes at column (lane % P) * 8; the rows are turned back into one row
      // per lane through the warp's box when the chunk is used.
      const long long rrow0 = static_cast<long long>(b) * e.bs + static_cast<long long>(r0) * e.ld + cb;
      const long long cpiece = static_cast<long long>(lane / P) * e.ld + (lane % P) * 8;
      const uint16_t* rh0 = has_r ? static_cast<const uint16_t*>(e.Rh) + rrow0 + cpiece : nullptr;
      const uint16_t* rl0 = has_rl ? static_cast<const uint16_t*>(e.Rl) + rrow0 + cpiece : nullptr;
      const long long rows_it = static_cast<long long>(RPI) * e.ld;
      uint4 nh[P], nl[P];  // this lane's coalesced pieces of the next chunk
#pragma unroll
      for (int q = 0; q < P; ++q) {
        nh[q] = has_r ? ld16(rh0 + q * rows_it + jq * CH) : zero4;
        nl[q] = has_rl ? ld16(rl0 + q * rows_it + jq * CH) : zero4;
      }
      // coalesced pieces -> this lane's row (CH values as CH / 2 words)
      auto to_rows = [&](const uint4 (&piece)[P], uint32_t (&w)[CH / 2]) {
        constexpr int STRIDE = 2 * CH + 16;
#pragma unroll
        for (int it = 0; it < P; ++it)
          *reinterpret_cast<uint4*>(box + (it * RPI + lane / P) * STRIDE + (lane % P) * 16) = piece[it];
        __syncwarp();
#pragma unroll
        for (int q = 0; q < P; ++q) {
          const uint4 x = *reinterpret_cast<const uint4*>(box + lane * STRIDE + q * 16);
          w[4 * q] = x.x, w[4 * q + 1] = x.y, w[4 * q + 2] = x.z, w[4 * q + 3] = x.w;
        }
        __syncwarp();
      };
      const int abuf = tcount & 1;
      const uint32_t aph = (tcount >> 1) & 1;
      if (*abort_flag || !mbar_wait(&tfull[abuf], aph)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float sc = epi_scale(e, b);
      const float ka = sc * e.c_acc, kr = sc * e.c_res * e.r_scale;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + abuf * C::BN;
      constexpr int MAXIT = C::NCHT / C::WPQ;  // chunks of each warp of a quarter
      static_assert(C::NCHT % C::WPQ == 0 && CH == 32, "every warp takes the same number of 32-column chunks");
      // The TMEM load of chunk i + 1 is issued once chunk i's values are in
      // their output form, so it runs while chunk i is stored (one buffer of
      // registers: two would not fit this kernel's 168 per thread)
      uint32_t tb[CH];
      tmem_ld_32x32b_x32_issue(tbase + jq * CH, tb);
#pragma unroll
      for (int i = 0; i < MAXIT; ++i) {
        const int cc = jq + i * C::WPQ;
        const int c0 = cb + cc * CH;
        const bool more = i + 1 < MAXIT;
        const uint32_t tnext = tbase + (cc + C::WPQ) * CH;
        __syncwarp();
        tmem_ld_wait_x32(tb);
        float v[CH];
#pragma unroll
        for (int u = 0; u < CH; ++u) v[u] = __uint_as_float(tb[u]);
        uint32_t rhw[CH / 2], rlw[CH / 2];
        if (has_r) to_rows(nh, rhw);
        if (has_rl) {
          to_rows(nl, rlw);
        } else {
#pragma unroll
          for (int u = 0; u < CH / 2; ++u) rlw[u] = 0u;
        }
        if (cc + C::WPQ < C::NCHT) {
#pragma unroll
          for (int q = 0; q < P; ++q) {
            nh[q] = has_r ? ld16(rh0 + q * rows_it + (cc + C::WPQ) * CH) : zero4;
            nl[q] = has_rl ? ld16(rl0 + q * rows_it + (cc + C::WPQ) * CH) : zero4;
          }
        }
        if (has_r) {
          if (e.r_f16) {
#pragma unroll
            for (int u = 0; u < CH / 2; ++u) {
              const float2 h = unpack2_h(rhw[u]), l = unpack2_h(rlw[u]);  // rlw = 0 without a residual part
              v[2 * u] = ka * v[2 * u] + kr * (h.x + l.x * (1.f / kF16LoScale));
              v[2 * u + 1] = ka * v[2 * u + 1] + kr * (h.y + l.y * (1.f / kF16LoScale));
            }
          } else {
#pragma unroll
            for (int u = 0; u < CH / 2; ++u) {
              v[2 * u] = ka * v[2 * u] + kr * (bf_lo(rhw[u]) + bf_lo(rlw[u]));
              v[2 * u + 1] = ka * v[2 * u + 1] + kr * (bf_hi(rhw[u]) + bf_hi(rlw[u]));
            }
          }
        } else if (ka != 1.f) {
#pragma unroll
          for (int u = 0; u < CH; ++u) v[u] *= ka;
        }
        if (e.c_id != 0.f && r >= c0 && r < c0 + CH && r < e.rows_valid) {
#pragma unroll
          for (int u = 0; u < CH; ++u)
            if (c0 + u == r) v[u] += e.c_id;
        }
        if (e.final_mode != FINAL_NONE) {
          const bool full_block = r0 + 32 <= e.rows_valid && c0 + CH <= e.cols_valid;
          if (!f.tr[b] && !e.dst_fp32 && phs.final_vec && full_block) {
            final_block_rows<bf16, CH>(e, f, b, r0, c0, lane, v, box);
          } else if (f.tr[b] && !e.dst_fp32 && phs.final_vec_t && full_block) {
            final_block_cols<CH>(e, f, b, r0, c0, lane, v, box);
          } else {
#pragma unroll
            for (int u = 0; u < CH; ++u) epi_final_elem(e, f, b, r, c0 + u, v[u]);
          }
          __syncwarp();  // tcgen05.ld is warp-aligned: reconverge after the per-lane branches
          if (more) tmem_ld_32x32b_x32_issue(tnext, tb);
        } else {
          uint32_t hw[CH / 2], lw[CH / 2];
          split_words<CH>(v, hw, lw, has_lo, e.o_f16 != 0, e.lo_scale);
          __syncwarp();  // tcgen05.ld is warp-aligned: reconverge after the per-lane branches
          if (more) tmem_ld_32x32b_x32_issue(tnext, tb);
          const long long off = static_cast<long long>(b) * e.bs + static_cast<long long>(r0) * e.ld + c0;
          store_block16<CH>(static_cast<uint16_t*>(e.Oh) + off, e.ld, lane, hw, box);
          if (has_lo) store_block16<CH>(static_cast<uint16_t*>(e.Ol) + off, e.ld, lane, lw, box);
        }
      }
      // this warp's TMEM rows are read: release the buffer to the leader's MMA issuer
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_cluster(&tempty[abuf], 0));
      if (prog.done) {
        // this warp's part of the tile is stored: publish it for the later
        // products, whose TMA (async proxy) and L2 loads read it.  The warp
        // barrier orders every lane's stores before lane 0's release, which
        // is cumulative over them (no per-lane membar.gl).
        fence_proxy_async_global();
        __syncwarp();
        if (lane == 0) red_release_gpu_add(&prog.done[b], 1);
      }
    }
    if (!ok) {
      if (lane == 0) atomicOr(prog.status, kStatusTimeout);
      *abort_flag = 1;
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncwarp();
  cluster_sync();  // neither CTA leaves while its peer may still write into it
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
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

// 3-D map of 16-bit elements (bf16, or fp16 with f16) over [B][rows][inner]
// with box {box_inner, box_rows, 1}.
static bool make_map(CUtensorMap* m, const void* base, bool f16, uint64_t inner, uint64_t rows, uint64_t batch,
                     long long ld, long long bs, uint32_t box_inner, uint32_t box_rows, int swb) {
  auto enc = get_encode();
  if (!enc) return false;
  const cuuint64_t dims[3] = {inner, rows, batch};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2, static_cast<cuuint64_t>(bs) * 2};
  const cuuint32_t box[3] = {box_inner, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                         const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE,
                         swb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Launch `ncl` clusters of two CTAs with programmatic stream serialization.
template <typename... KArgs, typename... Args>
static cudaError_t launch_pair(void (*kernel)(KArgs...), int ncl, cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * ncl);
  cfg.blockDim = dim3(TcCfg::THREADS);
  cfg.dynamicSmemBytes = TcCfg::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The dynamic shared-memory limit is raised once per device and kernel, so a
// later call (e.g. under stream capture) only enqueues launches.
template <int NPH>
static cudaError_t ensure_smem_attr() {
  static std::mutex mu;
  static bool done[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(mu);
  if (!done[dev]) {
    e = cudaFuncSetAttribute(tc_gemm_kernel<NPH>, cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg::SMEM);
    if (e != cudaSuccess) return e;
    done[dev] = true;
  }
  return cudaSuccess;
}

// Clusters of two that can be resident at once (queried once per device), so
// the persistent grid never waits for a second wave of clusters.
template <int NPH>
static int max_clusters(int num_sms) {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms / 2;
  std::lock_guard<std::mutex> lk(mu);
  if (!cached[dev]) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(TcCfg::THREADS);
    cfg.dynamicSmemBytes = TcCfg::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tc_gemm_kernel<NPH>, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = num_sms / 2;
    }
    cached[dev] = std::min(n, num_sms / 2);
  }
  return cached[dev];
}

// Validates one product and fills its phase (tiles from `first` on).
static bool build_phase(TcPhase& ph, const TcGemmDesc& d, const EpiParams& epi, int first, const char** why) {
  using C = TcCfg;
  if (d.split < 1 || d.split > 5 || d.split == 4 || (d.split == 2 && !d.b_mn)) {
    *why = "unsupported operand split";
    return false;
  }
  if (d.split == 5 && (!d.f16 || !d.A.lo || !d.Bop.lo || d.diag)) {
    *why = "scaled fp16-pair products need fp16 operands with both residuals and no diagonal segment";
    return false;
  }
  if (d.M % 256 || d.N % 256 || d.K % 128) {
    *why = "tensor-core GEMM needs M and N multiples of 256 (CTA pairs) and K a multiple of 128";
    return false;
  }
  if ((d.split >= 2 && !d.A.lo) || (d.split >= 3 && !d.Bop.lo)) {
    *why = "split products need the residual operands";
    return false;
  }
  if ((d.a_sym && d.K != d.M) || (d.b_sym && (d.b_mn || d.K != d.N)) || ((d.a_sym || d.b_sym) && d.K % 256)) {
    *why = "symmetric operands must be square with K a multiple of 256";
    return false;
  }
  if (d.diag && (d.split != 1 || !d.b_mn || d.K != d.M || !d.Bop.lo ||
                 reinterpret_cast<uintptr_t>(d.diag) % 16)) {
    *why = "a diagonal segment needs split 1, an MN-major B with its residual, K == M and an aligned D";
    return false;
  }
  const void* alo = d.A.lo ? d.A.lo : d.A.hi;
  const void* blo = d.Bop.lo ? d.Bop.lo : d.Bop.hi;
  const bool f = d.f16 != 0;
  CUtensorMap* tm = ph.tm;
  // K-major boxes {64 k, rows}; transposed boxes {64 mn, 64 k} (symmetric operands: K == rows)
  bool ok = make_map(&tm[kMapA], d.A.hi, f, d.K, d.M, d.B, d.A.ld, d.A.bs, C::KA, C::BM, 128);
  ok = ok && make_map(&tm[kMapAl], alo, f, d.K, d.M, d.B, d.A.ld, d.A.bs, C::KA, C::BM, 128);
  ok = ok && make_map(&tm[kMapAt], d.A.hi, f, d.K, d.M, d.B, d.A.ld, d.A.bs, C::MN_ATOM, C::BK, 128);
  ok = ok && make_map(&tm[kMapAtl], alo, f, d.K, d.M, d.B, d.A.ld, d.A.bs, C::MN_ATOM, C::BK, 128);
  if (!d.b_mn) {
    ok = ok && make_map(&tm[kMapB], d.Bop.hi, f, d.K, d.N, d.B, d.Bop.ld, d.Bop.bs, C::KA, C::BNH, 128);
    ok = ok && make_map(&tm[kMapBl], blo, f, d.K, d.N, d.B, d.Bop.ld, d.Bop.bs, C::KA, C::BNH, 128);
    ok = ok && make_map(&tm[kMapBt], d.Bop.hi, f, d.K, d.N, d.B, d.Bop.ld, d.Bop.bs, C::MN_ATOM, C::BK, 128);
    ok = ok && make_map(&tm[kMapBtl], blo, f, d.K, d.N, d.B, d.Bop.ld, d.Bop.bs, C::MN_ATOM, C::BK, 128);
  } else {
    ok = ok && make_map(&tm[kMapB], d.Bop.hi, f, d.N, d.K, d.B, d.Bop.ld, d.Bop.bs, C::MN_ATOM, C::BK, 128);
    ok = ok && make_map(&tm[kMapBl], blo, f, d.N, d.K, d.B, d.Bop.ld, d.Bop.bs, C::MN_ATOM, C::BK, 128);
    tm[kMapBt] = tm[kMapB];
    tm[kMapBtl] = tm[kMapBl];
  }
  // D (the diagonal segment's A): one 256 x 256 matrix, K-major boxes like A's
  tm[kMapD] = tm[kMapA];
  if (d.diag)
    ok = ok && make_map(&tm[kMapD], d.diag, f, kDiagDim, kDiagDim, 1, kDiagDim, kDiagDim * kDiagDim, C::KA, C::BM,
                        128);
  if (!ok) {
    *why = "cuTensorMapEncodeTiled failed";
    return false;
  }
  const bool has_out = epi.Oh != nullptr;
  if (epi.final_mode == FINAL_NONE && !has_out) {
    *why = "tensor-core epilogue needs a 16-bit output pair";
    return false;
  }
  // packed outputs and residuals are accessed with 16-byte row accesses
  if ((has_out || epi.Rh) && ((reinterpret_cast<uintptr_t>(epi.Oh) | reinterpret_cast<uintptr_t>(epi.Ol) |
                               reinterpret_cast<uintptr_t>(epi.Rh) | reinterpret_cast<uintptr_t>(epi.Rl)) %
                                  16 ||
                              epi.ld % 8 || epi.bs % 8)) {
    *why = "tensor-core outputs and residuals need 16-byte aligned rows";
    return false;
  }
  ph.M = d.M;
  ph.N = d.N;
  ph.K = d.K;
  ph.sym = d.sym;
  ph.nI = d.M / C::BM;
  ph.nJ = d.N / C::BN;
  if (d.sym) {
    const int P = ph.nI / 2;
    ph.tpm = P * (P + 1) / 2;
  } else {
    ph.tpm = (ph.nI / 2) * ph.nJ;
  }
  ph.first = first;
  // K segments of the split products (bit 2s: A residual, bit 2s+1: B residual)
  if (d.split == 1) {
    ph.nseg = 1;
    ph.seg_lo = 0;
  } else if (d.split == 2) {  // Ah B + Al B
    ph.nseg = 2;
    ph.seg_lo = 1 << 2;
  } else if (d.split == 3) {  // Ah Bh + Ah Bl + Al Bh
    ph.nseg = 3;
    ph.seg_lo = (1 << 3) | (1 << 4);
  } else {  // split 5: Ah Bl + Al Bh (scaled by 2^11), then Ah Bh on a 2^-11-scaled accumulator
    ph.nseg = 3;
    ph.seg_lo = (1 << 1) | (1 << 2);
  }
  ph.pair_scale = d.split == 5 ? 1 : 0;
  // A rectangular product walks its tiles column by column within groups of
  // row-block pairs, so that a group's rows of A (rgroup * 256 rows x K) stay
  // in L2 while every column block of B is fetched once per group: as many
  // pairs as keep that panel within 32 MiB of the 126 MiB L2, at least 4.
  ph.rgroup = std::min(std::max(ph.nI / 2, 1), std::max(4, static_cast<int>((32LL << 20) / (512LL * d.K))));
  ph.diag_kb = d.diag ? kDiagDim / C::BK : 0;
  ph.a_sym = d.a_sym;
  ph.b_sym = d.b_mn ? 0 : d.b_sym;
  ph.bmn = d.b_mn ? 1 : 0;
  ph.f16 = d.f16 ? 1 : 0;
  ph.wait = d.done && d.flag_wait ? 1 : 0;
  ph.wait_target = d.wait_target;
  ph.epi = epi;  // the scalars; the final tables travel once per launch
  ph.epi.sym = d.sym;
  // 16-byte row accesses to the caller's matrices in final mode need aligned rows
  ph.final_vec = 1;
  ph.final_vec_t = 1;
  if (epi.final_mode != FINAL_NONE) {
    const int esz = epi.dst_fp32 ? 4 : 2;
    if ((static_cast<long long>(epi.cols_valid) * esz) % 16) ph.final_vec = 0;
    if ((static_cast<long long>(epi.rows_valid) * esz) % 16) ph.final_vec_t = 0;
    for (int q = 0; q < d.B; ++q)
      if (reinterpret_cast<uintptr_t>(epi.dst[q]) % 16) ph.final_vec = ph.final_vec_t = 0;
  }
  return true;
}

// One launch over n products (n <= NPH) that share the batch's counters.
template <int NPH>
static cudaError_t launch_program(const TcGemmDesc* d, const EpiParams* const* epi, int n, int* status,
                                  cudaStream_t st, int num_sms, const char** why) {
  if (n < 1 || n > NPH) {
    *why = "too many products for one launch";
    return cudaErrorInvalidValue;
  }
  if (!d[0].tile_ctr) {
    *why = "tensor-core GEMM needs a zeroed tile counter";
    return cudaErrorInvalidValue;
  }
  {
    const cudaError_t e = ensure_smem_attr<NPH>();
    if (e != cudaSuccess) return e;
  }
  // The argument block is large (NPH tensor-map sets); build it on the heap,
  // once per thread (the launch copies it).
  static thread_local std::unique_ptr<TcProgram<NPH>> prog;
  if (!prog) prog.reset(new TcProgram<NPH>());
  TcProgram<NPH>& a = *prog;
  memset(&a, 0, sizeof(a));
  const EpiParams* fin = nullptr;
  int total = 0;
  for (int q = 0; q < n; ++q) {
    if (d[q].done != d[0].done) {
      *why = "the products of one launch share one set of completion counters";
      return cudaErrorInvalidValue;
    }
    if (q > 0 && !(d[q].done && d[q].flag_wait)) {
      *why = "every product after a launch's first waits on the completion counters";
      return cudaErrorInvalidValue;
    }
    if (epi[q]->final_mode != FINAL_NONE) {
      if (fin) {
        *why = "one final product per launch";
        return cudaErrorInvalidValue;
      }
      fin = epi[q];
    }
    if (!build_phase(a.ph[q], d[q], *epi[q], total, why)) return cudaErrorInvalidValue;
    total += a.ph[q].tpm * d[q].B;
  }
  a.nph = n;
  a.total = total;
  a.status = status;
  a.done = d[0].done;
  a.tile_ctr = d[0].tile_ctr;
  if (fin) a.fin = static_cast<const EpiFinal&>(*fin);
  const int nclusters = std::min(a.total, max_clusters<NPH>(num_sms));
  if (nclusters <= 0) return a.total > 0 ? cudaErrorLaunchOutOfResources : cudaSuccess;
  return launch_pair(tc_gemm_kernel<NPH>, nclusters, st, a);
}

cudaError_t launch_tc_gemm(const TcGemmDesc& d, const EpiParams& epi, int* status, cudaStream_t st, int num_sms,
                           const char** why) {
  *why = nullptr;
  const EpiParams* e = &epi;
  return launch_program<1>(&d, &e, 1, status, st, num_sms, why);
}

cudaError_t launch_tc_program(const TcGemmDesc* d, const EpiParams* const* epi, int n, int* status,
                              cudaStream_t st, int num_sms, const char** why) {
  *why = nullptr;
  if (n == 1) return launch_program<1>(d, epi, 1, status, st, num_sms, why);
  return launch_program<kMaxPhases>(d, epi, n, status, st, num_sms, why);
}

int tc_max_products_per_launch() { return kMaxPhases; }

int tc_signals_per_matrix(int M, int N, int sym) {
  const int P = M / 256;
  return static_cast<int>(TcCfg::EPI_ARRIVALS) * (sym ? P * (P + 1) / 2 : P * (N / 256));
}

int tc_tiles(int M, int N, int sym) {
  const int nI = M / 128, nJ = N / 256;
  if (sym) return (nI / 2) * (nI / 2 + 1);
  return nI * nJ;
}

}  // namespace muon
