// engine.cu -- host engine and C ABI of the owner-side Muon update.
//
// Per call: validate every argument (no launch before that), group the matrices
// by (short side, long side) (DMuon technical summary, §2.2: same-shape matrices
// run the Gram recurrence jointly), carve the caller's workspace, and enqueue one
// schedule per group on the caller's stream:
//
//   ORIG       original space.  Step 0 multiplies the packed bf16 copy of M;
//              later products take fp16 operands, with X carried between steps
//              as an fp16 pair (hi + lo / 2^11):
//              A = X X^T (SYRK), B' = a I + b A + c A^2, X <- B' X_hi + a X_lo
//   GRAM_R2    the Gram recurrence (DMuon technical summary, §2.2) restarted
//              from X every two steps: step 0 as in ORIG, then segments
//              A = X_hi X_hi^T; P_0 = a I + b A + c A^2; G_1 = P_0 (P_0 A);
//              P_1 = a I + b G_1 + c G_1^2; X <- (P_1 P_0) X_hi + a^2 X_lo,
//              on fp16 operands (the bf16 default where it saves work)
//   ORIG_BF16  ORIG on bf16 operands only, X carried as a bf16 pair, with
//              split products in the last steps (the fallback for coefficients
//              outside fp16's range)
//   ORIG_F16X3 ORIG on fp16 pairs, three MMAs per product (fp32 data, up to
//              6 steps)
//   GRAM_X3    Gram space for all steps, split-bf16 operands (hi*hi + hi*lo +
//              lo*hi): G0 = X0 X0^T; P_k = a I + b G_k + c G_k^2; Q <- P_k Q;
//              G_{k+1} = P_k (P_k G_k); O = Q X0
//   GRAM_X1    the same recurrence with plain bf16 operands
//   fp32       ORIG, GRAM_R2 or the Gram recurrence with fp32 FFMA products
//
// Why these: the Gram recurrence squares the condition number, and without
// restarts the rounding of G grows in the directions of small singular values
// (GRAM_X1 diverges on rank-deficient inputs, GRAM_X3 reaches ~2e-2).
// Re-forming G from X every two steps keeps it within a third of the bf16
// tolerance.  fp16 operands (11 significant bits) in original space need no
// splits.  GRAM_X3 and GRAM_X1 are kept on request for comparison.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "muon_ns.h"
#include "common.cuh"
#include "kernels.h"

namespace muon {

static thread_local std::string g_last_error;

muon_status fail(muon_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

// ------------------------------------------------------------------ profiling
// Optional per-launch CUDA-event timing on the caller's stream (off by default).
struct ProfRec {
  const char* kind;
  cudaEvent_t a, b;
  double flops;  // algorithmic flops of the launch (symmetric products counted once)
  double bytes;  // algorithmic HBM bytes of the launch
};
static bool g_prof_on = false;
static std::vector<ProfRec> g_prof;
static std::vector<cudaEvent_t> g_event_pool;
static size_t g_event_next = 0;

static cudaEvent_t prof_event() {
  if (g_event_next == g_event_pool.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    g_event_pool.push_back(e);
  }
  return g_event_pool[g_event_next++];
}

struct ProfScope {
  bool on;
  cudaStream_t st;
  size_t idx;
  ProfScope(const char* kind, double flops, double bytes, cudaStream_t s) : on(g_prof_on), st(s), idx(0) {
    if (!on) return;
    ProfRec r{kind, prof_event(), prof_event(), flops, bytes};
    if (!r.a || !r.b) {
      on = false;
      return;
    }
    cudaEventRecord(r.a, st);
    idx = g_prof.size();
    g_prof.push_back(r);
  }
  ~ProfScope() {
    if (on) cudaEventRecord(g_prof[idx].b, st);
  }
};

static const float kQuintic[3] = {3.4445f, -4.7750f, 2.0315f};
static const float kEps = 1e-7f;
// ORIG_BF16: number of final NS steps whose A*A (resp. B*X) products use split
// operands.  The error of plain bf16 products comes from the last steps; an
// fp32-exact CPU emulation over Gaussian inputs of aspect 1:1 to 1:3 gives a
// worst relative error of 2.3e-2 with no splits, 1.04e-2 with both splits in
// the last two steps, 0.97e-2 in the last three, and 1.3e-2 / 2.1e-2 with only
// A*A / only B*X split.  The ORIG schedule's fp16 operands (11 significant
// bits) need no splits: the same emulation gives at most 1.8e-3 with X carried
// as an fp16 pair, including rank-8 and row-scaled inputs.
#ifndef MUON_SPLIT_A_STEPS
#define MUON_SPLIT_A_STEPS 2
#endif
#ifndef MUON_SPLIT_B_STEPS
#define MUON_SPLIT_B_STEPS 2
#endif
static const int kSplitA = MUON_SPLIT_A_STEPS;
static const int kSplitB = MUON_SPLIT_B_STEPS;
// Beyond five steps the rounding of the unsplit steps builds up (same
// emulation, 256 x 512 Gaussian, quintic: 7 steps reach 3.0e-2 with two split
// steps and 1.5e-2 with four), so every step from the fourth on is split.
static int split_steps(int T, int base) { return std::max(base, T - 3); }

static inline long long round_up(long long x, long long m) { return (x + m - 1) / m * m; }

// One matrix of a call, in the caller's layout.
struct Mat {
  const void* src;  // gradient (step) or X (ns only)
  float* mom;       // momentum or nullptr
  void* dst;        // W (apply) or out (store)
  int m, n;
};

// ------------------------------------------------------------------ bucketing
// Groups by (short, long) key in increasing key order; members keep input order.
static int bucket_plan(const std::vector<std::pair<long long, long long>>& shapes, std::vector<int>& order,
                       std::vector<int>& start) {
  const int count = static_cast<int>(shapes.size());
  order.resize(count);
  for (int i = 0; i < count; ++i) order[i] = i;
  auto key = [&](int i) {
    const long long a = shapes[i].first, b = shapes[i].second;
    return std::make_pair(std::min(a, b), std::max(a, b));
  };
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return key(x) < key(y); });
  start.clear();
  for (int t = 0; t < count; ++t)
    if (t == 0 || key(order[t]) != key(order[t - 1])) start.push_back(t);
  const int groups = static_cast<int>(start.size());
  start.push_back(count);
  return groups;
}

// ------------------------------------------------------------------ schedules
// Lengths of the segments the steps run in (ORIG: every step alone; GRAM_R2:
// step 0 alone, on the packed bf16 copy of M, then two steps per segment,
// and a last single step when T - 1 is odd).
static std::vector<int> segment_plan(int T, muon_sched sc) {
  std::vector<int> plan;
  if (T <= 0) return plan;
  plan.push_back(1);
  int left = T - 1;
  if (sc == MUON_SCHED_GRAM_R2)
    for (; left >= 2; left -= 2) plan.push_back(2);
  for (; left > 0; --left) plan.push_back(1);
  return plan;
}

static float ipow(float x, int k) {
  float r = 1.f;
  for (int i = 0; i < k; ++i) r *= x;
  return r;
}

// ORIG on bf16 data multiplies fp16 operands from step 1 on.  That is safe when
// every iterate keeps its singular values <= 1.25: X0 has sigma <= 1 (Frobenius
// normalisation), and the singular values of the next X are |p(sigma)|, so it
// suffices that p(s) = a s + b s^3 + c s^5 maps [0, 1.25] into [-1.25, 1.25].
// That is checked on a grid, widened by half a grid step times a bound on |p'|.
// Then |A| <= 1.5625, and B = b A + c A^2 stays far inside fp16's range when
// 1.5625 |b| + 2.4414 |c| <= 1e4.
static bool f16_coefficients_safe(float a, float b, float c) {
  const double A = std::fabs(a), B = std::fabs(b), C = std::fabs(c);
  if (!(1.5625 * B + 2.44140625 * C <= 1e4)) return false;
  const double dmax = A + 3.0 * B * 1.5625 + 5.0 * C * 2.44140625;  // |p'(s)| on [0, 1.25]
  const int n = 5000;
  const double h = 1.25 / n;
  double pmax = 0.0;
  for (int i = 0; i <= n; ++i) {
    const double x = i * h, x2 = x * x;
    pmax = std::max(pmax, std::fabs(x * (a + x2 * (b + x2 * c))));
  }
  return pmax + 0.5 * h * dmax <= 1.25;
}


// The coefficients as the schedules need them (the fp16 range check above).
struct Coef {
  float a, b, c;
  bool f16_ok;
};

static Coef coef_of(const float* coeffs) {
  const float* cf = coeffs ? coeffs : kQuintic;
  return Coef{cf[0], cf[1], cf[2], f16_coefficients_safe(cf[0], cf[1], cf[2])};
}

static bool pair_sched(muon_sched sc) { return sc == MUON_SCHED_ORIG_F16X3; }

// Tensor-core (or FFMA) work of a schedule's segment plan, with the padded
// sizes: per segment of k steps one SYRK (S^2 L, lower tiles), 4k - 3
// symmetric s x s products (S^3 each) and the update (2 S^2 L).
static double plan_work(long long s, long long l, int steps, muon_sched sc) {
  const double S = static_cast<double>(round_up(s, 256)), L = static_cast<double>(round_up(l, 256));
  double w = 0.0;
  for (int k : segment_plan(steps, sc)) w += 3.0 * S * S * L + (4.0 * k - 3.0) * S * S * S;
  return w;
}

// fp32 runs up to this many steps take the tensor-core fp16-pair schedule:
// measured on Gaussian and row-scaled fp32 inputs it stays within 3e-5 of
// the fp64 result at 5 steps, but reaches about 9e-5 at 10 (the tensor cores'
// fp32 accumulation, about 1e-6 of the sum of |products| per product, builds
// up), too close to the 1e-4 tolerance; longer runs use FFMA.  (Gram space
// without restarts is not used for them either: rounding leaves G with small
// negative eigenvalues that the recurrence lambda <- (a + b lambda + c
// lambda^2)^2 lambda grows by about a^2 per step until they overflow,
// measured on rank-deficient fp32 inputs at 10 steps.)
constexpr int kFp32PairMaxSteps = 6;

// bf16 runs up to this many steps take single fp16 operands (ORIG, GRAM_R2);
// longer ones take fp16 pairs (ORIG_F16X3).  The quintic does not contract
// inside the band it maps the singular values into, so each step's operand
// rounding (fp16: 2^-11) is carried forward and the error grows with the step
// count.  Measured on Gaussian, row-scaled and rank-8 inputs: at most 8.9e-3
// at 10 steps, 1.3e-2 at 12, 2.1e-2 at 15 and 2.3-3.7e-2 at 20 to 100, where
// the fp16 pairs stay at the bf16 output rounding (1.7e-3; 4.7e-3 at most).
constexpr int kBf16SingleMaxSteps = 10;

static muon_sched resolve(long long s, long long l, int steps, muon_dtype dt, muon_sched sc, const Coef& k) {
  sc = static_cast<muon_sched>(sc & MUON_SCHED_MASK);  // launch-mode flags are the Group's
  if (steps == 0) return MUON_SCHED_ORIG;  // only the packed fp32 copy is needed
  // two-step Gram segments where they save at least a tenth of the work
  const bool r2_pays = plan_work(s, l, steps, MUON_SCHED_GRAM_R2) <= 0.9 * plan_work(s, l, steps, MUON_SCHED_ORIG);
  if (sc == MUON_SCHED_AUTO) {
    if (dt == MUON_FP32) {
      // short runs: tensor-core fp16 pairs (FFMA Gram space if the
      // coefficients leave fp16's range); long runs: FFMA in two-step Gram
      // segments where they save work, else original space
      if (steps <= kFp32PairMaxSteps)
        sc = k.f16_ok ? MUON_SCHED_ORIG_F16X3 : (l > s ? MUON_SCHED_GRAM_X3 : MUON_SCHED_ORIG);
      else
        sc = r2_pays ? MUON_SCHED_GRAM_R2 : MUON_SCHED_ORIG;
    } else if (steps > kBf16SingleMaxSteps && k.f16_ok) {
      // bf16, long runs: fp16 pairs
      sc = MUON_SCHED_ORIG_F16X3;
    } else {
      // bf16: the Gram recurrence restarted every two steps (GRAM_R2) where it
      // saves at least a tenth of the tensor-core work, else original space
      sc = r2_pays ? MUON_SCHED_GRAM_R2 : MUON_SCHED_ORIG;
    }
  }
  // fp16 pairs need coefficients that keep every operand in fp16's range
  if (pair_sched(sc)) return k.f16_ok ? sc : (dt == MUON_FP32 ? MUON_SCHED_ORIG : MUON_SCHED_ORIG_BF16);
  if (dt == MUON_FP32) {
    if (sc == MUON_SCHED_ORIG || sc == MUON_SCHED_ORIG_BF16) return MUON_SCHED_ORIG;  // one fp32 form
    return sc == MUON_SCHED_GRAM_R2 ? MUON_SCHED_GRAM_R2 : MUON_SCHED_GRAM_X3;       // both Gram modes: FFMA
  }
  return sc;
}

// Bump allocator over the workspace; with base == nullptr it only measures.
struct Carve {
  char* base;
  size_t off;
  void* take(size_t bytes) {
    off = static_cast<size_t>(round_up(static_cast<long long>(off), 1024));
    void* p = base ? base + off : nullptr;
    off += bytes;
    return p;
  }
};

constexpr size_t kHeader = 1024;  // status word + reserved
constexpr size_t kDebugTileCtr = 512;  // header offset of muon_debug_gemm's tile counter
// tensor-core launches in one chunk: at most 3 per NS step (ORIG) or 5 (Gram) plus 2
constexpr int kMaxTcLaunches = 5 * MUON_MAX_STEPS + 8;

struct Buffers {
  float* inv_norm = nullptr;
  float* partial = nullptr;
  int* done = nullptr;  // per-matrix completion counters chaining consecutive tensor-core launches
  int* tile_ctr = nullptr;  // one tile-scheduler counter per tensor-core launch of the chunk
  // packed X
  float* Xf = nullptr;
  float* Xf2 = nullptr;
  bf16* Xb[2] = {nullptr, nullptr};
  bf16* Xlo[2] = {nullptr, nullptr};
  bf16* Xl = nullptr;
  // s x s
  float* Gf = nullptr;
  bf16* Gh = nullptr;
  bf16* Gl = nullptr;
  bf16* Bh = nullptr;
  bf16* Bl = nullptr;
  bf16* Ph[2] = {nullptr, nullptr};
  bf16* Pl[2] = {nullptr, nullptr};
  bf16* Qh[2] = {nullptr, nullptr};
  bf16* Ql[2] = {nullptr, nullptr};
  bf16* Hh = nullptr;
  bf16* Hl = nullptr;
  float* Pf[2] = {nullptr, nullptr};
  float* Qf[2] = {nullptr, nullptr};
  float* Hf = nullptr;
  float* Af = nullptr;
  float* Bf = nullptr;
  void* diag = nullptr;  // D = 2^-11 I (fp16) for the update's diagonal segment (ORIG)
};

static size_t carve_buffers(char* base, int Bc, long long sp, long long lp, int tiles, muon_dtype dt,
                            muon_sched sc, int steps, Buffers& bf) {
  Carve c{base, kHeader};
  const size_t nx = static_cast<size_t>(Bc) * sp * lp;
  const size_t ns = static_cast<size_t>(Bc) * sp * sp;
  bf.inv_norm = static_cast<float*>(c.take(sizeof(float) * Bc));
  bf.partial = static_cast<float*>(c.take(sizeof(float) * Bc * static_cast<size_t>(tiles)));
  bf.done = static_cast<int*>(c.take(sizeof(int) * Bc));
  bf.tile_ctr = static_cast<int*>(c.take(sizeof(int) * kMaxTcLaunches));
  if (steps > 0 && pair_sched(sc)) {
    // fp32 copy of M, then fp16 pairs (stored in 16-bit buffers) of X (ping-pong), A and B'
    bf.Xf = static_cast<float*>(c.take(4 * nx));
    for (int q = 0; q < 2; ++q) {
      bf.Xb[q] = static_cast<bf16*>(c.take(2 * nx));
      bf.Xlo[q] = static_cast<bf16*>(c.take(2 * nx));
    }
    bf.Gh = static_cast<bf16*>(c.take(2 * ns));
    bf.Gl = static_cast<bf16*>(c.take(2 * ns));
    bf.Bh = static_cast<bf16*>(c.take(2 * ns));
    bf.Bl = static_cast<bf16*>(c.take(2 * ns));
    return c.off;
  }
  if (dt == MUON_FP32 || steps == 0) {
    bf.Xf = static_cast<float*>(c.take(4 * nx));
    if (steps == 0) return c.off;
    if (sc == MUON_SCHED_ORIG || sc == MUON_SCHED_GRAM_R2) {
      bf.Xf2 = static_cast<float*>(c.take(4 * nx));
      bf.Af = static_cast<float*>(c.take(4 * ns));
      bf.Bf = static_cast<float*>(c.take(4 * ns));
      if (sc == MUON_SCHED_GRAM_R2) {  // the two-step segments' H and P_1
        bf.Hf = static_cast<float*>(c.take(4 * ns));
        bf.Pf[0] = static_cast<float*>(c.take(4 * ns));
      }
    } else {
      bf.Gf = static_cast<float*>(c.take(4 * ns));
      for (int q = 0; q < 2; ++q) bf.Pf[q] = static_cast<float*>(c.take(4 * ns));
      for (int q = 0; q < 2; ++q) bf.Qf[q] = static_cast<float*>(c.take(4 * ns));
      bf.Hf = static_cast<float*>(c.take(4 * ns));
    }
    return c.off;
  }
  if (sc == MUON_SCHED_ORIG || sc == MUON_SCHED_ORIG_BF16 || sc == MUON_SCHED_GRAM_R2) {
    // X carried as a 16-bit pair (bf16 pair ~16 significant bits, fp16 pair ~22), ping-ponged
    for (int q = 0; q < 2; ++q) {
      bf.Xb[q] = static_cast<bf16*>(c.take(2 * nx));
      bf.Xlo[q] = static_cast<bf16*>(c.take(2 * nx));
    }
    bf.Gh = static_cast<bf16*>(c.take(2 * ns));
    bf.Gl = static_cast<bf16*>(c.take(2 * ns));
    bf.Bh = static_cast<bf16*>(c.take(2 * ns));
    bf.Bl = static_cast<bf16*>(c.take(2 * ns));
    bf.diag = c.take(2 * kDiagDim * kDiagDim);
    return c.off;
  }
  const bool x3 = (sc == MUON_SCHED_GRAM_X3);
  bf.Xb[0] = static_cast<bf16*>(c.take(2 * nx));
  if (x3) bf.Xl = static_cast<bf16*>(c.take(2 * nx));
  bf.Gh = static_cast<bf16*>(c.take(2 * ns));
  bf.Gl = static_cast<bf16*>(c.take(2 * ns));  // kept in both modes: G = Gh + Gl feeds the P epilogue
  for (int q = 0; q < 2; ++q) {
    bf.Ph[q] = static_cast<bf16*>(c.take(2 * ns));
    if (x3) bf.Pl[q] = static_cast<bf16*>(c.take(2 * ns));
    bf.Qh[q] = static_cast<bf16*>(c.take(2 * ns));
    if (x3) bf.Ql[q] = static_cast<bf16*>(c.take(2 * ns));
  }
  bf.Hh = static_cast<bf16*>(c.take(2 * ns));
  if (x3) bf.Hl = static_cast<bf16*>(c.take(2 * ns));
  return c.off;
}

struct Group {
  long long s, l, sp, lp;
  int tiles;  // pack tiles per matrix
  muon_sched sc;
  int steps;
  int launch;  // 0: shared launches for small chunks, else one per product; or the forcing flag
};

static Group make_group(long long m, long long n, int steps, muon_dtype dt, muon_sched sc,
                        const Coef& k = coef_of(nullptr)) {
  Group g;
  g.s = std::min(m, n);
  g.l = std::max(m, n);
  g.sp = round_up(g.s, 256);
  g.lp = round_up(g.l, 256);
  g.tiles = static_cast<int>((g.sp / 64) * (g.lp / 64));
  g.sc = resolve(g.s, g.l, steps, dt, sc, k);
  g.launch = sc & ~MUON_SCHED_MASK;
  g.steps = steps;
  return g;
}

static size_t group_bytes(const Group& g, int Bc, muon_dtype dt) {
  Buffers bf;
  return carve_buffers(nullptr, Bc, g.sp, g.lp, g.tiles, dt, g.sc, g.steps, bf);
}

// Largest batch width that fits in ws_bytes (0 if none).
static int fit_batch(const Group& g, int want, muon_dtype dt, size_t ws_bytes) {
  want = std::min(want, kMaxBatch);
  if (want <= 0) return 0;
  if (group_bytes(g, want, dt) <= ws_bytes) return want;
  const size_t one = group_bytes(g, 1, dt);
  if (one > ws_bytes) return 0;
  const size_t per = group_bytes(g, 2, dt) - one;
  int bc = static_cast<int>(std::min<size_t>(want, 1 + (ws_bytes - one) / std::max<size_t>(per, 1)));
  while (bc > 1 && group_bytes(g, bc, dt) > ws_bytes) --bc;
  return bc;
}

// ------------------------------------------------------------------ device info
static int device_sms(int* major, int* minor, muon_status* st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    *st = fail(MUON_ERR_CUDA, "no CUDA device available");
    return 0;
  }
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(minor, cudaDevAttrComputeCapabilityMinor, dev);
  *st = MUON_OK;
  return sms;
}

// ------------------------------------------------------------------ one group
struct Ctx {
  cudaStream_t st;
  int sms;
  int* status;
  muon_dtype dt;
  int steps;
  float a, b, c;
  float beta, lr;
  bool apply;   // W <- W - lr O (else out = O)
  bool has_mom;
  bool f16_ok;  // the coefficients allow ORIG's fp16 operands
};

#define CK(expr)                                                                                  \
  do {                                                                                            \
    cudaError_t e_ = (expr);                                                                      \
    if (e_ != cudaSuccess)                                                                        \
      return fail(MUON_ERR_CUDA, "%s failed: %s%s%s", #expr, cudaGetErrorString(e_), why ? ": " : "", \
                  why ? why : "");                                                                \
  } while (0)

// fp32 (CUDA-core) epilogue: residual R and output Of.
static EpiParams epi_packed(const Group& g, const Buffers& bf, int scale_pow, float c_acc, float c_res, float c_id,
                            const float* R, float* Of, long long ld, long long bs) {
  EpiParams e;
  memset(&e, 0, sizeof(e));
  e.inv_norm = bf.inv_norm;
  e.scale_pow = scale_pow;
  e.c_acc = c_acc;
  e.c_res = c_res;
  e.c_id = c_id;
  e.R = R;
  e.Of = Of;
  e.r_scale = 1.f;
  e.lo_scale = kF16LoScale;
  e.ld = ld;
  e.bs = bs;
  e.rows_valid = static_cast<int>(g.s);
  e.cols_valid = static_cast<int>(g.s);
  e.final_mode = FINAL_NONE;
  return e;
}

// bf16-pair (tensor-core) epilogue: residual Rh + Rl and outputs Oh (+ Ol).
static EpiParams epi_pair(const Group& g, const Buffers& bf, int scale_pow, float c_acc, float c_res, float c_id,
                          const void* Rh, const void* Rl, void* Oh, void* Ol, long long ld, long long bs) {
  EpiParams e = epi_packed(g, bf, scale_pow, c_acc, c_res, c_id, nullptr, nullptr, ld, bs);
  e.Rh = Rh;
  e.Rl = Rl;
  e.Oh = Oh;
  e.Ol = Ol;
  return e;
}

static void epi_set_final(EpiParams& e, const Ctx& cx, const Group& g, const Mat* mats, int Bc) {
  e.Of = nullptr;
  e.Oh = nullptr;
  e.Ol = nullptr;
  e.final_mode = cx.apply ? FINAL_APPLY : FINAL_STORE;
  e.dst_fp32 = cx.dt == MUON_FP32 ? 1 : 0;
  e.lr = cx.lr;
  e.rows_valid = static_cast<int>(g.s);
  e.cols_valid = static_cast<int>(g.l);
  for (int q = 0; q < Bc; ++q) {
    e.dst[q] = mats[q].dst;
    e.tr[q] = mats[q].m > mats[q].n ? 1 : 0;
  }
}

// The ORIG update on fp16 operands, X <- B' X_hi + a X_lo, runs the a X_lo
// term as a diagonal segment of the product (D = 2^-11 I times the low part,
// stored as a 2^11 (X - X_hi)) when its K (the padded short side) is at most
// this: 256 more of K per tile is at most 12.5 % more MMA work there, and it
// takes the residual out of an epilogue that sets the pace at K ~ 1024.  At
// larger K the main loop already hides the epilogue.
constexpr long long kDiagMaxK = 2048;

static uint16_t f16_bits(float x) {
  const __half h = __float2half_rn(x);
  uint16_t u;
  memcpy(&u, &h, sizeof(u));
  return u;
}

static muon_status run_chunk(const Ctx& cx, const Group& g, const Mat* mats, int Bc, char* ws) {
  const char* why = nullptr;
  Buffers bf;
  carve_buffers(ws, Bc, g.sp, g.lp, g.tiles, cx.dt, g.sc, cx.steps, bf);
  // Chaining (and the shared launches below) pays when each product is a few
  // waves of tiles: then one product's ragged last wave overlaps the next
  // one's first, and a grid's fill and drain is a large part of a product.
  // On longer products the overlap only adds power next to a tail it cannot
  // shorten, and the per-tile signals cost more than it gains.  Measured
  // with shared launches, against separate ones: 8 x 1024 x 4096 (7 pair-tiles
  // per cluster in the update) 287 -> 360 TFLOP/s, 8 x 1024 x 8192 (13.5)
  // 234 -> 270; the 512 small matrices of shapes 256 x 1024 .. 768 x 3072
  // (10 to 75 per cluster) 293 -> 286 when every bucket shares launches.
  // Also when the s x s products alone are about a wave (at most 4 tile pairs
  // per CTA pair, e.g. 8 x 1024 x 16384): each is then a short launch whose
  // fill and drain dominate, and the SYRK's last partial wave leaves most of
  // the GPU idle; sharing launches overlaps them across matrices.  Measured on
  // 8 x 1024 x 16384: 1.95 -> 1.77 ms per step.
  const long long pairs_rect = static_cast<long long>(Bc) * (g.sp / 256) * (g.lp / 256);
  const long long nbs = g.sp / 256;
  const long long pairs_sym = static_cast<long long>(Bc) * nbs * (nbs + 1) / 2;
  const bool pairs = cx.steps > 0 && pair_sched(g.sc);  // fp16-pair operands (either dtype)
  const bool tensor = cx.dt == MUON_BF16 || pairs;       // the NS products run on the tensor cores
  const bool small = pairs_rect <= 16LL * (cx.sms / 2) || pairs_sym <= 4LL * (cx.sms / 2);
  const bool chain = tensor && (g.launch == MUON_SCHED_SHARED_LAUNCH || (g.launch == 0 && small));
  // stream-ordered: runs after everything before this chunk, before its pack
  if (chain) CK(cudaMemsetAsync(bf.done, 0, sizeof(int) * Bc, cx.st));
  if (tensor && cx.steps > 0) CK(cudaMemsetAsync(bf.tile_ctr, 0, sizeof(int) * kMaxTcLaunches, cx.st));
  const long long sp = g.sp, lp = g.lp;
  const long long bsx = sp * lp, bss = sp * sp;
  const bool fp32 = cx.dt == MUON_FP32;
  const bool x3 = g.sc == MUON_SCHED_GRAM_X3;
  const bool h16 = !fp32 && (g.sc == MUON_SCHED_ORIG || g.sc == MUON_SCHED_GRAM_R2) && cx.f16_ok;
  const bool use_diag = h16 && cx.steps >= 2 && sp <= kDiagMaxK;

  // ---- momentum + pack + norm
  PackArgs pa;
  memset(&pa, 0, sizeof(pa));
  pa.m = mats[0].m;
  pa.n = mats[0].n;
  pa.sp = static_cast<int>(sp);
  pa.lp = static_cast<int>(lp);
  pa.has_mom = cx.has_mom ? 1 : 0;
  pa.src_fp32 = fp32 ? 1 : 0;
  pa.beta = cx.beta;
  pa.bs = bsx;
  pa.partial = bf.partial;
  pa.tiles = g.tiles;
  pa.Xf = bf.Xf;  // fp32 path, pair schedules, or zero steps
  if (!fp32 && !pairs && cx.steps > 0) {
    pa.Xh = bf.Xb[0];
    pa.Xl = (g.sc == MUON_SCHED_ORIG || g.sc == MUON_SCHED_ORIG_BF16 || g.sc == MUON_SCHED_GRAM_R2)
                ? bf.Xlo[0]
                : (x3 ? bf.Xl : nullptr);
  }
  for (int q = 0; q < Bc; ++q) {
    // a bucket can mix m x n and n x m members: the pack kernel transposes per member
    pa.src[q] = mats[q].src;
    pa.mom[q] = mats[q].mom;
    pa.tr[q] = mats[q].m > mats[q].n ? 1 : 0;
  }
  {
    // One pack launch covers members stored the same way round (the chunk is
    // ordered m x n before n x m); a mixed chunk takes two launches.
    int q = 1;
    while (q < Bc && mats[q].m == pa.m) ++q;
    const double el = static_cast<double>(g.s) * g.l;
    const double esz = fp32 ? 4.0 : 2.0;
    const double pbytes = el * (esz + (cx.has_mom ? 8.0 : 0.0) + (pa.Xf ? 4.0 : 0.0) + (pa.Xh ? 2.0 : 0.0) +
                                (pa.Xl ? 2.0 : 0.0));
    {
      ProfScope ps("pack", 0.0, pbytes * q, cx.st);
      CK(launch_pack(pa, q, cx.st));
    }
    if (q < Bc) {
      ProfScope ps("pack", 0.0, pbytes * (Bc - q), cx.st);
      PackArgs pb = pa;
      pb.m = mats[q].m;
      pb.n = mats[q].n;
      for (int r = q; r < Bc; ++r) {
        pb.src[r - q] = mats[r].src;
        pb.mom[r - q] = mats[r].mom;
        pb.tr[r - q] = pa.tr[r];
      }
      if (pb.Xf) pb.Xf += q * bsx;
      if (pb.Xh) pb.Xh += q * bsx;
      if (pb.Xl) pb.Xl += q * bsx;
      pb.partial += static_cast<long long>(q) * g.tiles;
      CK(launch_pack(pb, Bc - q, cx.st));
    }
  }
  {
    ProfScope ps("norm_finalize", 0.0, 4.0 * g.tiles * Bc, cx.st);
    CK(launch_norm_finalize(bf.partial, g.tiles, Bc, kEps, bf.inv_norm, use_diag ? bf.diag : nullptr,
                            f16_bits(1.f / kF16LoScale), cx.st));
  }

  if (cx.steps == 0) {
    EpiParams e = epi_packed(g, bf, 1, 1.f, 0.f, 0.f, nullptr, nullptr, lp, bsx);
    epi_set_final(e, cx, g, mats, Bc);
    ProfScope ps("final_from_packed", 0.0, Bc * static_cast<double>(g.s) * g.l * (fp32 ? 12.0 : 8.0), cx.st);
    CK(launch_final_from_packed(bf.Xf, lp, bsx, Bc, e, cx.st));
    return MUON_OK;
  }
  const int T = cx.steps;
  const int S = static_cast<int>(sp), L = static_cast<int>(lp);

  if (pairs) {
    ProfScope ps("pair_split", 0.0, 12.0 * Bc * static_cast<double>(bsx), cx.st);
    CK(launch_pair_from_f32(bf.Xf, bf.inv_norm, bf.Xb[0], g.sc == MUON_SCHED_ORIG_F16X3 ? bf.Xlo[0] : bf.Xl, bsx, Bc,
                            cx.sms, cx.st));
  }
  if (fp32 && !pairs) {
    // Every operand here but the SYRK's X is symmetric and stored in full (the
    // symmetric products mirror their lower tiles), so it is read MN-major
    // (`sym_ops`): both operands then go straight into shared memory.
    auto simt = [&](const float* A, long long lda, long long bsa, const float* Bm, long long ldb, long long bsb,
                    int M, int N, int K, int sym, int b_mn, const EpiParams& e, bool sym_ops = false) {
      SimtGemmDesc d{Bc, M, N, K, sym, sym_ops ? 1 : b_mn, A, lda, bsa, Bm, ldb, bsb};
      d.a_mn = sym_ops ? 1 : 0;
      const double Kt = K == S ? static_cast<double>(g.s) : static_cast<double>(g.l);
      const double fl = sym ? Bc * static_cast<double>(g.s) * g.s * Kt : 2.0 * Bc * g.s * g.l * Kt;
      ProfScope ps(sym ? "simt_sym" : "simt_rect", fl, 0.0, cx.st);
      return launch_simt_gemm(d, e, cx.st);
    };
    if (g.sc == MUON_SCHED_ORIG || g.sc == MUON_SCHED_GRAM_R2) {
      // Segments of one step (ORIG) or, after step 0, of two Gram steps
      // (GRAM_R2): A = X X^T; then Q' = Q - a^k I with Q the segment's
      // polynomial product (k = 1: b A + c A^2; k = 2: P_1 P_0 - a^2 I with
      // P_j = a I + b G_j + c G_j^2, G_0 = A, G_1 = P_0 A P_0); X <- Q' X + a^k X.
      float* cur = bf.Xf;
      float* nxt = bf.Xf2;
      const std::vector<int> plan = segment_plan(T, g.sc);
      for (size_t si = 0; si < plan.size(); ++si) {
        const int k = plan[si];
        const bool first = si == 0, last = si + 1 == plan.size();
        EpiParams e1 = epi_packed(g, bf, first ? 2 : 0, 1.f, 0.f, 0.f, nullptr, bf.Af, sp, bss);
        CK(simt(cur, lp, bsx, cur, lp, bsx, S, S, L, 1, 0, e1));
        const float* Qp = bf.Bf;
        if (k == 1) {
          EpiParams e2 = epi_packed(g, bf, 0, cx.c, cx.b, 0.f, bf.Af, bf.Bf, sp, bss);
          CK(simt(bf.Af, sp, bss, bf.Af, sp, bss, S, S, S, 1, 0, e2, true));
        } else {
          // A in Af -> P_0 in Bf, H in Hf, G_1 in Af, P_1 in Pf[0], Q' in Af
          EpiParams p0 = epi_packed(g, bf, 0, cx.c, cx.b, cx.a, bf.Af, bf.Bf, sp, bss);
          CK(simt(bf.Af, sp, bss, bf.Af, sp, bss, S, S, S, 1, 0, p0, true));
          EpiParams eh = epi_packed(g, bf, 0, 1.f, 0.f, 0.f, nullptr, bf.Hf, sp, bss);
          CK(simt(bf.Bf, sp, bss, bf.Af, sp, bss, S, S, S, 1, 0, eh, true));
          EpiParams eg = epi_packed(g, bf, 0, 1.f, 0.f, 0.f, nullptr, bf.Af, sp, bss);
          CK(simt(bf.Bf, sp, bss, bf.Hf, sp, bss, S, S, S, 1, 0, eg, true));
          EpiParams p1 = epi_packed(g, bf, 0, cx.c, cx.b, cx.a, bf.Af, bf.Pf[0], sp, bss);
          CK(simt(bf.Af, sp, bss, bf.Af, sp, bss, S, S, S, 1, 0, p1, true));
          EpiParams eq = epi_packed(g, bf, 0, 1.f, 0.f, -cx.a * cx.a, nullptr, bf.Af, sp, bss);
          CK(simt(bf.Pf[0], sp, bss, bf.Bf, sp, bss, S, S, S, 1, 0, eq, true));
          Qp = bf.Af;
        }
        EpiParams e3 = epi_packed(g, bf, first ? 1 : 0, 1.f, ipow(cx.a, k), 0.f, cur, nxt, lp, bsx);
        e3.cols_valid = static_cast<int>(g.l);
        if (last) epi_set_final(e3, cx, g, mats, Bc);
        CK(simt(Qp, sp, bss, cur, lp, bsx, S, L, S, 0, 1, e3, true));
        std::swap(cur, nxt);
      }
      return MUON_OK;
    }
    // fp32 Gram
    EpiParams e0 = epi_packed(g, bf, 2, 1.f, 0.f, 0.f, nullptr, bf.Gf, sp, bss);
    CK(simt(bf.Xf, lp, bsx, bf.Xf, lp, bsx, S, S, L, 1, 0, e0));
    const float* Q = nullptr;
    int qi = 0;
    for (int k = 0; k < T; ++k) {
      float* P = bf.Pf[k & 1];
      EpiParams ep = epi_packed(g, bf, 0, cx.c, cx.b, cx.a, bf.Gf, P, sp, bss);
      CK(simt(bf.Gf, sp, bss, bf.Gf, sp, bss, S, S, S, 1, 0, ep, true));
      if (k == 0) {
        Q = P;
      } else {
        float* Qn = bf.Qf[qi];
        qi ^= 1;
        EpiParams eq = epi_packed(g, bf, 0, 1.f, 0.f, 0.f, nullptr, Qn, sp, bss);
        CK(simt(P, sp, bss, Q, sp, bss, S, S, S, 1, 0, eq, true));
        Q = Qn;
      }
      if (k + 1 < T) {
        EpiParams eh = epi_packed(g, bf, 0, 1.f, 0.f, 0.f, nullptr, bf.Hf, sp, bss);
        CK(simt(P, sp, bss, bf.Gf, sp, bss, S, S, S, 1, 0, eh, true));
        EpiParams eg = epi_packed(g, bf, 0, 1.f, 0.f, 0.f, nullptr, bf.Gf, sp, bss);
        CK(simt(P, sp, bss, bf.Hf, sp, bss, S, S, S, 1, 0, eg, true));
      }
    }
    EpiParams ef = epi_packed(g, bf, 1, 1.f, 0.f, 0.f, nullptr, nullptr, lp, bsx);
    epi_set_final(ef, cx, g, mats, Bc);
    CK(simt(Q, sp, bss, bf.Xf, lp, bsx, S, L, S, 0, 1, ef, true));
    return MUON_OK;
  }

  // Consecutive tensor-core launches are chained per matrix: each adds to
  // done[b] as it finishes matrix b's tiles, and every launch after the first
  // starts matrix b as soon as done[b] reaches the total of all launches
  // before it, rather than waiting for the whole previous grid.  By induction
  // every earlier launch has then finished matrix b, so all read-after-write
  // and write-after-read hazards on b's buffers are covered.  (The counters
  // are zeroed at the top of the chunk.)
  // On those short chunks the products also share launches: up to
  // tc_max_products_per_launch() consecutive products run on one persistent
  // grid, their tiles in one sequence, so the per-launch fill and drain (the
  // ramp of a grid, its ragged last wave) is paid once per launch instead of
  // once per product.
  const bool program = chain;
  std::vector<TcGemmDesc> pend_d;
  std::vector<EpiParams> pend_e;
  double pend_fl = 0.0;
  auto flush = [&]() -> cudaError_t {
    if (pend_d.empty()) return cudaSuccess;
    std::vector<const EpiParams*> ep;
    for (const EpiParams& x : pend_e) ep.push_back(&x);
    cudaError_t err;
    {
      ProfScope ps("tc_program", pend_fl, 0.0, cx.st);
      err = launch_tc_program(pend_d.data(), ep.data(), static_cast<int>(pend_d.size()), cx.status, cx.st,
                              cx.sms, &why);
    }
    pend_d.clear();
    pend_e.clear();
    pend_fl = 0.0;
    return err;
  };
  int tc_launches = 0;  // products so far (each has its own tile counter slot)
  int tc_cum = 0;
  // sym: bit 0 = symmetric output (lower tiles, block-lower storage); bits 1 / 2 =
  // A / B is a symmetric operand in that storage.
  auto tc = [&](int split, int b_mn, int sym, int f16, int M, int N, int K, const void* Ah, const void* Al,
                long long lda, long long bsa, const void* Bh, const void* Bl, long long ldb, long long bsb,
                const EpiParams& e, const void* diag = nullptr) {
    TcGemmDesc d;
    d.B = Bc;
    d.M = M;
    d.N = N;
    d.K = K;
    d.sym = sym & 1;
    d.a_sym = (sym >> 1) & 1;
    d.b_sym = (sym >> 2) & 1;
    d.split = split;
    d.b_mn = b_mn;
    d.f16 = f16;
    d.A = TcOperand{Ah, Al, lda, bsa};
    d.Bop = TcOperand{Bh, Bl, ldb, bsb};
    d.diag = diag;
    const double Kt = K == S ? static_cast<double>(g.s) : static_cast<double>(g.l);
    const double fl = d.sym ? Bc * static_cast<double>(g.s) * g.s * Kt : 2.0 * Bc * g.s * g.l * Kt;
    static const char* const kSym[6] = {"", "tc_sym", "tc_sym_x2", "tc_sym_x3", "", "tc_sym_p3"};
    static const char* const kSyrk[6] = {"", "tc_syrk", "tc_syrk_x2", "tc_syrk_x3", "", "tc_syrk_p3"};
    static const char* const kRect[6] = {"", "tc_rect", "tc_rect_x2", "tc_rect_x3", "", "tc_rect_p3"};
    const char* kind = d.sym ? (K == S ? kSym[split] : kSyrk[split]) : kRect[split];
    d.done = chain ? bf.done : nullptr;
    d.flag_wait = tc_launches > 0 ? 1 : 0;
    if (tc_launches >= kMaxTcLaunches) return cudaErrorInvalidValue;
    d.tile_ctr = bf.tile_ctr + tc_launches;
    d.wait_target = tc_cum;
    tc_cum += tc_signals_per_matrix(M, N, d.sym);
    ++tc_launches;
    if (program) {
      pend_d.push_back(d);
      pend_e.push_back(e);
      pend_fl += fl;
      return static_cast<int>(pend_d.size()) == tc_max_products_per_launch() ? flush() : cudaSuccess;
    }
    ProfScope ps(kind, fl, 0.0, cx.st);
    return launch_tc_gemm(d, e, cx.status, cx.st, cx.sms, &why);
  };

  if (pairs) {
    // Original space on fp16 pairs: X0 (normalised, fp32) was split above; A,
    // B' = a I + b A + c A^2 and X are pairs, every product split 5.
    int cur = 0;
    for (int k = 0; k < T; ++k) {
      const int nxt = cur ^ 1;
      EpiParams e1 = epi_pair(g, bf, 0, 1.f, 0.f, 0.f, nullptr, nullptr, bf.Gh, bf.Gl, sp, bss);
      e1.o_f16 = 1;
      CK(tc(5, 0, 1, 1, S, S, L, bf.Xb[cur], bf.Xlo[cur], lp, bsx, bf.Xb[cur], bf.Xlo[cur], lp, bsx, e1));
      EpiParams e2 = epi_pair(g, bf, 0, cx.c, cx.b, cx.a, bf.Gh, bf.Gl, bf.Bh, bf.Bl, sp, bss);
      e2.r_f16 = 1;
      e2.o_f16 = 1;
      CK(tc(5, 0, 7, 1, S, S, S, bf.Gh, bf.Gl, sp, bss, bf.Gh, bf.Gl, sp, bss, e2));
      EpiParams e3 = epi_pair(g, bf, 0, 1.f, 0.f, 0.f, nullptr, nullptr, bf.Xb[nxt], bf.Xlo[nxt], lp, bsx);
      e3.o_f16 = 1;
      e3.cols_valid = static_cast<int>(g.l);
      if (k == T - 1) epi_set_final(e3, cx, g, mats, Bc);
      CK(tc(5, 1, 2, 1, S, L, S, bf.Bh, bf.Bl, sp, bss, bf.Xb[cur], bf.Xlo[cur], lp, bsx, e3));
      cur = nxt;
    }
    CK(flush());
    return MUON_OK;
  }
  if (h16) {
    // Step 0 multiplies the packed bf16 copy of M (slot 0: hi, and lo for
    // the residual); A is stored as fp16, and B in the type of this step's X.
    // From step 1 on, X lives in the ping-pong slots as an fp16 pair and
    // every product takes fp16 operands.  Slot 0's bf16 copy is dead after
    // step 0, so step 1 writes its fp16 X there.
    // The steps run in segments (segment_plan): ORIG's are all one step long;
    // GRAM_R2's are step 0 and then two steps each.  A segment of k steps
    // starts from A = X_hi X_hi^T and ends with X <- Q X_hi + a^k X_lo, where
    // Q = a^k I + ... is the product of the segment's polynomials: for k = 1
    // Q = B' = a I + b A + c A^2, for k = 2 the Gram recurrence
    //   P_0 = a I + b A + c A^2, G_1 = P_0 (P_0 A), P_1 = a I + b G_1 + c G_1^2,
    //   Q = P_1 P_0
    // on fp16 operands (all of them polynomials in A, so symmetric and stored
    // block-lower).  Restarting from X every two steps keeps the Gram
    // recurrence's fp16 rounding from building up in the directions of small
    // singular values.  The a^k X_lo term keeps X's low part, which the
    // products do not see: with the diagonal segment (use_diag) the low part
    // written for the next segment is 2^11 a^k' (X - X_hi) (k' the next
    // segment's length) and the next update adds 2^-11 I times it on the
    // tensor cores; otherwise the epilogue reads it as a residual.
    const std::vector<int> plan = segment_plan(T, g.sc);
    int cur = 0;
    for (size_t si = 0; si < plan.size(); ++si) {
      const int k = plan[si];
      const bool first = si == 0, last = si + 1 == plan.size();
      const float ak = ipow(cx.a, k), ak_next = last ? 1.f : ipow(cx.a, plan[si + 1]);
      const int nxt = cur ^ 1;
      const int xf = first ? 0 : 1;  // 1: X (and so Q) are fp16 in this segment
      // A = X X^T (first segment: X = M / s, so scale by inv_norm^2), fp16 out
      EpiParams e1 = epi_pair(g, bf, first ? 2 : 0, 1.f, 0.f, 0.f, nullptr, nullptr, bf.Gh, nullptr, sp, bss);
      e1.o_f16 = 1;
      CK(tc(1, 0, 1, xf, S, S, L, bf.Xb[cur], nullptr, lp, bsx, bf.Xb[cur], nullptr, lp, bsx, e1));
      const bf16* Q = bf.Bh;
      if (k == 1) {
        // B' = a I + b A + c A^2 on fp16 operands
        EpiParams e2 = epi_pair(g, bf, 0, cx.c, cx.b, cx.a, bf.Gh, nullptr, bf.Bh, nullptr, sp, bss);
        e2.r_f16 = 1;
        e2.o_f16 = xf;
        CK(tc(1, 0, 7, 1, S, S, S, bf.Gh, nullptr, sp, bss, bf.Gh, nullptr, sp, bss, e2));
      } else {
        // two Gram steps; buffers: A and G_1 in Gh, P_0 in Bh, H = P_0 A in
        // Gl, P_1 in Bl, Q in Gh (each written after its last reader)
        auto poly = [&](const bf16* G, bf16* P) {
          EpiParams e = epi_pair(g, bf, 0, cx.c, cx.b, cx.a, G, nullptr, P, nullptr, sp, bss);
          e.r_f16 = 1;
          e.o_f16 = 1;
          return tc(1, 0, 7, 1, S, S, S, G, nullptr, sp, bss, G, nullptr, sp, bss, e);
        };
        auto mul = [&](const bf16* X1, const bf16* X2, bf16* out) {
          EpiParams e = epi_pair(g, bf, 0, 1.f, 0.f, 0.f, nullptr, nullptr, out, nullptr, sp, bss);
          e.o_f16 = 1;
          return tc(1, 0, 7, 1, S, S, S, X1, nullptr, sp, bss, X2, nullptr, sp, bss, e);
        };
        CK(poly(bf.Gh, bf.Bh));        // P_0
        CK(mul(bf.Bh, bf.Gh, bf.Gl));  // H = P_0 A
        CK(mul(bf.Bh, bf.Gl, bf.Gh));  // G_1 = P_0 H
        CK(poly(bf.Gh, bf.Bl));        // P_1
        CK(mul(bf.Bl, bf.Bh, bf.Gh));  // Q = P_1 P_0
        Q = bf.Gh;
      }
      // X <- Q X_hi + a^k X_lo (first segment: both terms carry 1 / s), fp16 pair out
      const bool dseg = use_diag && !first;
      EpiParams e3 = epi_pair(g, bf, first ? 1 : 0, 1.f, ak, 0.f, dseg ? nullptr : bf.Xlo[cur], nullptr,
                              bf.Xb[nxt], bf.Xlo[nxt], lp, bsx);
      e3.r_f16 = xf;
      e3.r_scale = xf ? 1.f / kF16LoScale : 1.f;  // an fp16 pair's low part is stored scaled by 2^11
      e3.o_f16 = 1;
      if (use_diag) e3.lo_scale = kF16LoScale * ak_next;
      e3.cols_valid = static_cast<int>(g.l);
      if (last) epi_set_final(e3, cx, g, mats, Bc);
      CK(tc(1, 1, 2, xf, S, L, S, Q, nullptr, sp, bss, bf.Xb[cur], dseg ? bf.Xlo[cur] : nullptr, lp, bsx, e3,
            dseg ? bf.diag : nullptr));
      cur = nxt;
    }
    CK(flush());
    return MUON_OK;
  }

  if (g.sc == MUON_SCHED_ORIG || g.sc == MUON_SCHED_ORIG_BF16 || g.sc == MUON_SCHED_GRAM_R2) {
    // (GRAM_R2 with coefficients outside fp16's range runs this bf16 form.)
    // Operand splits (see kSplitA / kSplitB): plain bf16 products miss a 2e-2
    // relative error on Gaussian inputs of aspect >= 1:2, mostly through the
    // rounding of the last steps, where sigma ~ 1 and the b, c terms are large.
    int cur = 0;
    for (int k = 0; k < T; ++k) {
      const bool split_a = k >= T - split_steps(T, kSplitA);
      const bool split = k >= T - split_steps(T, kSplitB);
      const int nxt = cur ^ 1;
      // A = X X^T (k = 0: X = M / s, so scale by inv_norm^2)
      EpiParams e1 = epi_pair(g, bf, k == 0 ? 2 : 0, 1.f, 0.f, 0.f, nullptr, nullptr, bf.Gh, bf.Gl, sp, bss);
      CK(tc(1, 0, 1, 0, S, S, L, bf.Xb[cur], nullptr, lp, bsx, bf.Xb[cur], nullptr, lp, bsx, e1));
      // B = b A + c A^2 with A = Ah + Al in the epilogue
      EpiParams e2 =
          epi_pair(g, bf, 0, cx.c, cx.b, 0.f, bf.Gh, bf.Gl, bf.Bh, split ? bf.Bl : nullptr, sp, bss);
      CK(tc(split_a ? 3 : 1, 0, 7, 0, S, S, S, bf.Gh, bf.Gl, sp, bss, bf.Gh, bf.Gl, sp, bss, e2));
      // X <- a X + B X (k = 0: both terms carry 1 / s); X kept as a bf16 pair
      EpiParams e3 = epi_pair(g, bf, k == 0 ? 1 : 0, 1.f, cx.a, 0.f, bf.Xb[cur], bf.Xlo[cur], bf.Xb[nxt],
                              bf.Xlo[nxt], lp, bsx);
      e3.cols_valid = static_cast<int>(g.l);
      if (k == T - 1) epi_set_final(e3, cx, g, mats, Bc);
      CK(tc(split ? 2 : 1, 1, 2, 0, S, L, S, bf.Bh, bf.Bl, sp, bss, bf.Xb[cur], nullptr, lp, bsx, e3));
      cur = nxt;
    }
    CK(flush());
    return MUON_OK;
  }

  // Gram space (split 3 or 1)
  const int sp3 = x3 ? 3 : 1;
  EpiParams e0 = epi_pair(g, bf, 2, 1.f, 0.f, 0.f, nullptr, nullptr, bf.Gh, bf.Gl, sp, bss);
  CK(tc(sp3, 0, 1, 0, S, S, L, bf.Xb[0], bf.Xl, lp, bsx, bf.Xb[0], bf.Xl, lp, bsx, e0));
  const bf16* Qh = nullptr;
  const bf16* Ql = nullptr;
  int qi = 0;
  for (int k = 0; k < T; ++k) {
    bf16* Ph = bf.Ph[k & 1];
    bf16* Pl = bf.Pl[k & 1];
    // P = a I + b G + c G^2
    EpiParams ep = epi_pair(g, bf, 0, cx.c, cx.b, cx.a, bf.Gh, bf.Gl, Ph, Pl, sp, bss);
    CK(tc(sp3, 0, 7, 0, S, S, S, bf.Gh, bf.Gl, sp, bss, bf.Gh, bf.Gl, sp, bss, ep));
    if (k == 0) {
      Qh = Ph;
      Ql = Pl;
    } else {
      bf16* Qnh = bf.Qh[qi];
      bf16* Qnl = bf.Ql[qi];
      qi ^= 1;
      EpiParams eq = epi_pair(g, bf, 0, 1.f, 0.f, 0.f, nullptr, nullptr, Qnh, Qnl, sp, bss);
      CK(tc(sp3, 0, 7, 0, S, S, S, Ph, Pl, sp, bss, Qh, Ql, sp, bss, eq));
      Qh = Qnh;
      Ql = Qnl;
    }
    if (k + 1 < T) {
      EpiParams eh = epi_pair(g, bf, 0, 1.f, 0.f, 0.f, nullptr, nullptr, bf.Hh, bf.Hl, sp, bss);
      CK(tc(sp3, 0, 7, 0, S, S, S, Ph, Pl, sp, bss, bf.Gh, bf.Gl, sp, bss, eh));
      EpiParams eg = epi_pair(g, bf, 0, 1.f, 0.f, 0.f, nullptr, nullptr, bf.Gh, bf.Gl, sp, bss);
      CK(tc(sp3, 0, 7, 0, S, S, S, Ph, Pl, sp, bss, bf.Hh, bf.Hl, sp, bss, eg));
    }
  }
  // O = Q X0 = Q X / s
  EpiParams ef = epi_pair(g, bf, 1, 1.f, 0.f, 0.f, nullptr, nullptr, nullptr, nullptr, lp, bsx);
  epi_set_final(ef, cx, g, mats, Bc);
  CK(tc(sp3, 1, 2, 0, S, L, S, Qh, Ql, sp, bss, bf.Xb[0], bf.Xl, lp, bsx, ef));
  CK(flush());
  return MUON_OK;
}
#undef CK

// ------------------------------------------------------------------ validation
static bool valid_dt(int dt) { return dt == MUON_BF16 || dt == MUON_FP32; }
static bool valid_sc(int sc) {
  const int base = sc & MUON_SCHED_MASK, flags = sc & ~MUON_SCHED_MASK;
  return base >= MUON_SCHED_AUTO && base <= MUON_SCHED_GRAM_R2 &&
         (flags == 0 || flags == MUON_SCHED_SHARED_LAUNCH || flags == MUON_SCHED_SEPARATE_LAUNCH);
}

static muon_status check_common(int steps, const float* coeffs, int dt, int sc, void* ws, size_t ws_bytes) {
  if (steps < 0 || steps > MUON_MAX_STEPS) return fail(MUON_ERR_ARG, "steps=%d out of [0, %d]", steps, MUON_MAX_STEPS);
  if (!valid_dt(dt)) return fail(MUON_ERR_ARG, "bad dtype %d", dt);
  if (!valid_sc(sc)) return fail(MUON_ERR_ARG, "bad schedule %d", sc);
  if (coeffs && !(std::isfinite(coeffs[0]) && std::isfinite(coeffs[1]) && std::isfinite(coeffs[2])))
    return fail(MUON_ERR_ARG, "coefficients must be finite");
  if (!ws) return fail(MUON_ERR_ARG, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(ws) % MUON_WS_ALIGN) return fail(MUON_ERR_ALIGN, "workspace not %d-byte aligned", MUON_WS_ALIGN);
  if (ws_bytes < kHeader) return fail(MUON_ERR_WORKSPACE, "workspace smaller than its %zu-byte header", kHeader);
  return MUON_OK;
}

static muon_status run_all(std::vector<Mat>& mats, int steps, const float* coeffs, muon_dtype dt, muon_sched sc,
                           float beta, float lr, bool apply, bool has_mom, void* ws, size_t ws_bytes,
                           void* stream) {
  const int count = static_cast<int>(mats.size());
  std::vector<std::pair<long long, long long>> shapes(count);
  for (int i = 0; i < count; ++i) shapes[i] = {mats[i].m, mats[i].n};
  std::vector<int> order, start;
  const int groups = bucket_plan(shapes, order, start);
  // plan every group before launching anything
  const Coef kc = coef_of(coeffs);
  std::vector<Group> gs(groups);
  std::vector<int> widths(groups);
  for (int gi = 0; gi < groups; ++gi) {
    const Mat& m0 = mats[order[start[gi]]];
    gs[gi] = make_group(m0.m, m0.n, steps, dt, sc, kc);
    widths[gi] = fit_batch(gs[gi], start[gi + 1] - start[gi], dt, ws_bytes);
    if (widths[gi] <= 0)
      return fail(MUON_ERR_WORKSPACE, "workspace of %zu bytes cannot hold one %lldx%lld matrix (needs %zu)", ws_bytes,
                  gs[gi].s, gs[gi].l, group_bytes(gs[gi], 1, dt));
  }
  if (count == 0) return MUON_OK;
  int major = 0, minor = 0;
  muon_status dst;
  const int sms = device_sms(&major, &minor, &dst);
  if (dst != MUON_OK) return dst;
  if (major != 10 || minor != 3)
    return fail(MUON_ERR_UNSUPPORTED, "this library is built for sm_103a (GB300); device is sm_%d%d", major, minor);
  Ctx cx;
  cx.st = static_cast<cudaStream_t>(stream);
  cx.sms = sms;
  cx.status = static_cast<int*>(ws);
  cx.dt = dt;
  cx.steps = steps;
  const float* cf = coeffs ? coeffs : kQuintic;
  cx.a = cf[0];
  cx.b = cf[1];
  cx.c = cf[2];
  cx.beta = beta;
  cx.lr = lr;
  cx.apply = apply;
  cx.has_mom = has_mom;
  cx.f16_ok = kc.f16_ok;
  std::vector<Mat> chunk;
  for (int gi = 0; gi < groups; ++gi) {
    const int n = start[gi + 1] - start[gi];
    for (int c0 = 0; c0 < n; c0 += widths[gi]) {
      const int bc = std::min(widths[gi], n - c0);
      chunk.clear();
      for (int q = 0; q < bc; ++q) chunk.push_back(mats[order[start[gi] + c0 + q]]);
      // pack requires equal caller shapes in one launch: order m x n before n x m
      std::stable_sort(chunk.begin(), chunk.end(), [](const Mat& x, const Mat& y) { return x.m < y.m; });
      const muon_status r = run_chunk(cx, gs[gi], chunk.data(), bc, static_cast<char*>(ws));
      if (r != MUON_OK) return r;
    }
  }
  return MUON_OK;
}

// ------------------------------------------------------------------ cost model
// Predicted device seconds of one matrix's update (pack, norm, the NS products
// and the apply), counted launch by launch as run_chunk issues them: executed
// flops over the padded 256-blocks (lower blocks only for symmetric outputs,
// x2 / x3 for split operands) and HBM bytes, each launch taking the larger of
// flops / rate and bytes / bandwidth.  The rates are nominal figures for this
// library's kernels on GB300 under the power cap.
constexpr double kRateTensor = 1.3e15;  // executed bf16 tensor-core flop/s
constexpr double kRateSimt = 4.0e13;    // fp32 FFMA flop/s
constexpr double kRateHbm = 6.0e12;     // byte/s

static double estimate_seconds(long long m, long long n, int steps, muon_dtype dt, muon_sched sc) {
  const Group g = make_group(m, n, steps, dt, sc);
  const double S = static_cast<double>(g.sp), L = static_cast<double>(g.lp);
  const double el = static_cast<double>(g.s) * g.l;
  const bool pairs = steps > 0 && pair_sched(g.sc);
  const bool fp32 = dt == MUON_FP32;
  const double rate = fp32 && !pairs ? kRateSimt : kRateTensor;
  const double nb = S / 256.0, nl = L / 256.0;
  const double sym_tiles = nb * (nb + 1) / 2, rect_tiles = nb * nl, tile = 2.0 * 256.0 * 256.0;
  const double ssz = 4.0;  // bytes of a packed element: fp32, or a bf16 pair
  double t = 0.0;
  auto launch = [&](double flops, double bytes) { t += std::max(flops / rate, bytes / kRateHbm); };
  // pack: read grad + momentum, write momentum + packed copy
  const bool x1 = !fp32 && g.sc == MUON_SCHED_GRAM_X1;
  launch(0.0, el * ((fp32 ? 4.0 : 2.0) + 8.0 + (steps == 0 ? 4.0 : (x1 ? 2.0 : 4.0))));
  const double apply = el * 2.0 * (fp32 ? 4.0 : 2.0);  // W read + write
  if (steps == 0) {
    launch(0.0, el * 4.0 + apply);
    return t;
  }
  const double sym_out = sym_tiles * 256.0 * 256.0 * ssz;  // a block-lower s x s output
  if (pairs) {
    // fp16 pairs: every product three times the tensor-core work, 4-byte operands
    launch(0.0, S * L * 12.0);  // X0 split into its pair
    for (int k = 0; k < steps; ++k) {
      launch(3.0 * sym_tiles * tile * L, S * L * 4.0 + sym_out);
      launch(3.0 * sym_tiles * tile * S, 2.0 * sym_out);
      launch(3.0 * rect_tiles * tile * S, sym_out + S * L * 4.0 + (k == steps - 1 ? apply : S * L * 4.0));
    }
    return t;
  }
  if (g.sc == MUON_SCHED_GRAM_R2) {
    // segments: SYRK, then A*A (one step) or five s x s products (two steps), then the update
    const double sym1 = sym_out / 2;  // single fp16 values
    const std::vector<int> plan = segment_plan(steps, g.sc);
    for (size_t si = 0; si < plan.size(); ++si) {
      launch(sym_tiles * tile * L, S * L * 2.0 + sym1);
      for (int p = 0; p < 4 * plan[si] - 3; ++p) launch(sym_tiles * tile * S, 3.0 * sym1);
      const double out = si + 1 == plan.size() ? apply : S * L * 4.0;
      launch(rect_tiles * tile * S, sym1 + S * L * 4.0 + out);
    }
    return t;
  }
  if (g.sc == MUON_SCHED_ORIG || g.sc == MUON_SCHED_ORIG_BF16) {
    // ORIG on bf16 data: fp16 operands, no splits, A and B single 16-bit values
    // (the default coefficients pass the fp16 range check)
    const bool h16 = !fp32 && g.sc == MUON_SCHED_ORIG;
    const double sym1 = h16 ? sym_out / 2 : sym_out;
    for (int k = 0; k < steps; ++k) {
      const double fa = (!fp32 && !h16 && k >= steps - split_steps(steps, kSplitA)) ? 3.0 : 1.0;
      const double fb = (!fp32 && !h16 && k >= steps - split_steps(steps, kSplitB)) ? 2.0 : 1.0;
      launch(sym_tiles * tile * L, S * L * (fp32 ? 4.0 : 2.0) + sym1);
      launch(fa * sym_tiles * tile * S, 2.0 * sym1);
      const double out = k == steps - 1 ? apply : S * L * ssz;
      launch(fb * rect_tiles * tile * S, sym1 + S * L * (fp32 ? 8.0 : 6.0) + out);
    }
    return t;
  }
  const double f3 = (!fp32 && g.sc == MUON_SCHED_GRAM_X3) ? 3.0 : 1.0;
  launch(f3 * sym_tiles * tile * L, S * L * ssz + sym_out);
  for (int k = 0; k < steps; ++k) {
    launch(f3 * sym_tiles * tile * S, 2.0 * sym_out);
    const int prods = (k > 0 ? 1 : 0) + (k + 1 < steps ? 2 : 0);
    for (int p = 0; p < prods; ++p) launch(f3 * sym_tiles * tile * S, 3.0 * sym_out);
  }
  launch(f3 * rect_tiles * tile * S, sym_out + S * L * ssz + apply);
  return t;
}

static bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace muon

using namespace muon;

extern "C" {

muon_status muon_adamw_tail(void* const* params, const void* const* grads, float* const* exp_avg,
                            float* const* exp_avg_sq, const int64_t* numel, int count, float lr, float beta1,
                            float beta2, float eps, float weight_decay, int step, muon_dtype dt, void* stream) {
  g_last_error.clear();
  if (count < 0) return fail(MUON_ERR_ARG, "count=%d < 0", count);
  if (count == 0) return MUON_OK;
  if (!params || !grads || !exp_avg || !exp_avg_sq || !numel) return fail(MUON_ERR_ARG, "NULL array");
  if (!valid_dt(dt)) return fail(MUON_ERR_ARG, "bad dtype %d", dt);
  if (step < 1) return fail(MUON_ERR_ARG, "step=%d: steps count from 1", step);
  if (!(std::isfinite(lr) && std::isfinite(eps) && std::isfinite(weight_decay) && beta1 >= 0.f && beta1 < 1.f &&
        beta2 >= 0.f && beta2 < 1.f && eps >= 0.f))
    return fail(MUON_ERR_ARG, "need finite lr, eps >= 0, weight_decay and betas in [0, 1)");
  const size_t esz = dt == MUON_FP32 ? 4 : 2;
  long long total = 0;
  for (int i = 0; i < count; ++i) {
    if (numel[i] < 0) return fail(MUON_ERR_SHAPE, "numel[%d] < 0", i);
    if (numel[i] > 0 && (!params[i] || !grads[i] || !exp_avg[i] || !exp_avg_sq[i]))
      return fail(MUON_ERR_ARG, "tensor %d has a NULL pointer", i);
    if ((reinterpret_cast<uintptr_t>(params[i]) | reinterpret_cast<uintptr_t>(grads[i])) % esz ||
        (reinterpret_cast<uintptr_t>(exp_avg[i]) | reinterpret_cast<uintptr_t>(exp_avg_sq[i])) % 4)
      return fail(MUON_ERR_ALIGN, "tensor %d is not aligned to its element size", i);
    total += numel[i];
  }
  if (total == 0) return MUON_OK;
  int major = 0, minor = 0;
  muon_status dst;
  const int sms = device_sms(&major, &minor, &dst);
  if (dst != MUON_OK) return dst;
  if (major != 10 || minor != 3)
    return fail(MUON_ERR_UNSUPPORTED, "this library is built for sm_103a (GB300); device is sm_%d%d", major, minor);
  static_assert(sizeof(AdamwArgs) < 32000, "AdamW arguments must fit the kernel parameter space");
  AdamwArgs a;
  memset(&a, 0, sizeof(a));
  a.decay = static_cast<float>(1.0 - static_cast<double>(lr) * weight_decay);
  a.beta1 = beta1;
  a.beta2 = beta2;
  a.eps = eps;
  const double bc1 = 1.0 - std::pow(static_cast<double>(beta1), step);
  const double bc2 = 1.0 - std::pow(static_cast<double>(beta2), step);
  a.step_size = static_cast<float>(lr / bc1);
  a.inv_sqrt_bc2 = static_cast<float>(1.0 / std::sqrt(bc2));
  const char* why = nullptr;
  for (int c0 = 0; c0 < count; c0 += kMaxTail) {
    const int n = std::min(kMaxTail, count - c0);
    a.count = n;
    long long gs = 0;
    for (int i = 0; i < n; ++i) {
      const int k = c0 + i;
      a.gstart[i] = gs;
      gs += (numel[k] + 7) / 8;
      a.numel[i] = numel[k];
      a.p[i] = params[k];
      a.g[i] = grads[k];
      a.m[i] = exp_avg[k];
      a.v[i] = exp_avg_sq[k];
      a.vec_ok[i] = ((reinterpret_cast<uintptr_t>(params[k]) | reinterpret_cast<uintptr_t>(grads[k]) |
                      reinterpret_cast<uintptr_t>(exp_avg[k]) | reinterpret_cast<uintptr_t>(exp_avg_sq[k])) % 16) == 0;
    }
    a.gstart[n] = gs;
    ProfScope ps("adamw_tail", 0.0, static_cast<double>(gs) * 8.0 * (dt == MUON_FP32 ? 28.0 : 22.0),
                 static_cast<cudaStream_t>(stream));
    const cudaError_t e = launch_adamw_tail(a, dt == MUON_BF16, sms, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
      return fail(MUON_ERR_CUDA, "launch_adamw_tail failed: %s%s%s", cudaGetErrorString(e), why ? ": " : "",
                  why ? why : "");
  }
  return MUON_OK;
}

muon_status muon_cost_estimate(const int64_t* shapes, int count, int steps, muon_dtype dt, muon_sched sc,
                               double* seconds) {
  if (count < 0) return fail(MUON_ERR_ARG, "count=%d < 0", count);
  if (count > 0 && (!shapes || !seconds)) return fail(MUON_ERR_ARG, "shapes and seconds must not be NULL");
  if (steps < 0 || steps > MUON_MAX_STEPS) return fail(MUON_ERR_ARG, "steps=%d out of [0, %d]", steps, MUON_MAX_STEPS);
  if (!valid_dt(dt)) return fail(MUON_ERR_ARG, "bad dtype %d", dt);
  if (!valid_sc(sc)) return fail(MUON_ERR_ARG, "bad schedule %d", sc);
  for (int i = 0; i < count; ++i) {
    const int64_t m = shapes[2 * i], n = shapes[2 * i + 1];
    if (m < 1 || n < 1 || m > MUON_MAX_DIM || n > MUON_MAX_DIM)
      return fail(MUON_ERR_SHAPE, "matrix %d has shape %lldx%lld", i, static_cast<long long>(m),
                  static_cast<long long>(n));
  }
  for (int i = 0; i < count; ++i) seconds[i] = estimate_seconds(shapes[2 * i], shapes[2 * i + 1], steps, dt, sc);
  return MUON_OK;
}

muon_status muon_ns_batched(const void* X, int B, int m, int n, int steps, const float* coeffs, void* out,
                            muon_dtype dt, muon_sched sc, void* ws, size_t ws_bytes, void* stream) {
  g_last_error.clear();
  try {
    if (B < 0) return fail(MUON_ERR_ARG, "B=%d < 0", B);
    if (B > 0 && (!X || !out)) return fail(MUON_ERR_ARG, "X or out is NULL");
    if (m <= 0 || n <= 0 || m > MUON_MAX_DIM || n > MUON_MAX_DIM)
      return fail(MUON_ERR_SHAPE, "bad shape %dx%d", m, n);
    muon_status s = check_common(steps, coeffs, dt, sc, ws, ws_bytes);
    if (s != MUON_OK) return s;
    const size_t esz = dt == MUON_FP32 ? 4 : 2;
    if (reinterpret_cast<uintptr_t>(X) % esz || reinterpret_cast<uintptr_t>(out) % esz)
      return fail(MUON_ERR_ALIGN, "X/out not aligned to the element size");
    const size_t bytes = static_cast<size_t>(B) * m * n * esz;
    if (B > 0 && overlaps(X, bytes, out, bytes)) return fail(MUON_ERR_ARG, "out overlaps X");
    if (B > 0 && overlaps(ws, ws_bytes, out, bytes)) return fail(MUON_ERR_ARG, "out overlaps the workspace");
    if (B > 0 && overlaps(ws, ws_bytes, X, bytes)) return fail(MUON_ERR_ARG, "X overlaps the workspace");
    std::vector<Mat> mats(B);
    for (int i = 0; i < B; ++i) {
      mats[i].src = static_cast<const char*>(X) + static_cast<size_t>(i) * m * n * esz;
      mats[i].mom = nullptr;
      mats[i].dst = static_cast<char*>(out) + static_cast<size_t>(i) * m * n * esz;
      mats[i].m = m;
      mats[i].n = n;
    }
    return run_all(mats, steps, coeffs, dt, sc, 0.f, 0.f, false, false, ws, ws_bytes, stream);
  } catch (...) {
    return fail(MUON_ERR_ARG, "internal exception");
  }
}

muon_status muon_step(void* const* W, const void* const* grad, float* const* mom, const int64_t* shapes, int count,
                      float beta, float lr, int steps, const float* coeffs, muon_dtype dt, muon_sched sc, void* ws,
                      size_t ws_bytes, void* stream) {
  g_last_error.clear();
  try {
    if (count < 0) return fail(MUON_ERR_ARG, "count=%d < 0", count);
    if (count > 0 && (!W || !grad || !mom || !shapes)) return fail(MUON_ERR_ARG, "a pointer array is NULL");
    if (!std::isfinite(beta) || !std::isfinite(lr)) return fail(MUON_ERR_ARG, "beta and lr must be finite");
    muon_status s = check_common(steps, coeffs, dt, sc, ws, ws_bytes);
    if (s != MUON_OK) return s;
    const size_t esz = dt == MUON_FP32 ? 4 : 2;
    std::vector<Mat> mats(count);
    for (int i = 0; i < count; ++i) {
      const int64_t m = shapes[2 * i], n = shapes[2 * i + 1];
      if (m <= 0 || n <= 0 || m > MUON_MAX_DIM || n > MUON_MAX_DIM)
        return fail(MUON_ERR_SHAPE, "matrix %d has bad shape %lldx%lld", i, (long long)m, (long long)n);
      if (!W[i] || !grad[i] || !mom[i]) return fail(MUON_ERR_ARG, "matrix %d has a NULL pointer", i);
      if (reinterpret_cast<uintptr_t>(W[i]) % esz || reinterpret_cast<uintptr_t>(grad[i]) % esz ||
          reinterpret_cast<uintptr_t>(mom[i]) % 4)
        return fail(MUON_ERR_ALIGN, "matrix %d: pointer not aligned to its element size", i);
      const size_t nel = static_cast<size_t>(m) * n;
      if (overlaps(W[i], nel * esz, mom[i], nel * 4) || overlaps(W[i], nel * esz, grad[i], nel * esz) ||
          overlaps(grad[i], nel * esz, mom[i], nel * 4))
        return fail(MUON_ERR_ARG, "matrix %d: W, grad and mom overlap", i);
      if (overlaps(ws, ws_bytes, W[i], nel * esz) || overlaps(ws, ws_bytes, mom[i], nel * 4))
        return fail(MUON_ERR_ARG, "matrix %d overlaps the workspace", i);
      mats[i].src = grad[i];
      mats[i].mom = mom[i];
      mats[i].dst = W[i];
      mats[i].m = static_cast<int>(m);
      mats[i].n = static_cast<int>(n);
    }
    return run_all(mats, steps, coeffs, dt, sc, beta, lr, true, true, ws, ws_bytes, stream);
  } catch (...) {
    return fail(MUON_ERR_ARG, "internal exception");
  }
}

size_t muon_workspace_bytes(const int64_t* shapes, int count, int steps, muon_dtype dt, muon_sched sc) {
  g_last_error.clear();
  if (count < 0 || (count > 0 && !shapes) || !valid_dt(dt) || !valid_sc(sc) || steps < 0 || steps > MUON_MAX_STEPS) {
    fail(MUON_ERR_ARG, "bad arguments to muon_workspace_bytes");
    return 0;
  }
  std::vector<std::pair<long long, long long>> sh(count);
  for (int i = 0; i < count; ++i) {
    if (shapes[2 * i] <= 0 || shapes[2 * i + 1] <= 0 || shapes[2 * i] > MUON_MAX_DIM ||
        shapes[2 * i + 1] > MUON_MAX_DIM) {
      fail(MUON_ERR_SHAPE, "matrix %d has a bad shape", i);
      return 0;
    }
    sh[i] = {shapes[2 * i], shapes[2 * i + 1]};
  }
  std::vector<int> order, start;
  const int groups = bucket_plan(sh, order, start);
  size_t best = kHeader;
  for (int gi = 0; gi < groups; ++gi) {
    const auto& s0 = sh[order[start[gi]]];
    const Group g = make_group(s0.first, s0.second, steps, dt, sc);
    const int w = std::min(start[gi + 1] - start[gi], kMaxBatch);
    best = std::max(best, group_bytes(g, w, dt));
  }
  return best;
}

muon_sched muon_resolve_schedule(int64_t m, int64_t n, int steps, muon_dtype dt, muon_sched sc) {
  return resolve(std::min<long long>(m, n), std::max<long long>(m, n), steps, dt, sc, coef_of(nullptr));
}

int muon_bucket_plan(const int64_t* shapes, int count, int* order, int* group_start) {
  if (count < 0 || (count > 0 && (!shapes || !order || !group_start))) return -1;
  std::vector<std::pair<long long, long long>> sh(count);
  for (int i = 0; i < count; ++i) sh[i] = {shapes[2 * i], shapes[2 * i + 1]};
  std::vector<int> ord, st;
  const int groups = bucket_plan(sh, ord, st);
  for (int i = 0; i < count; ++i) order[i] = ord[i];
  for (int gi = 0; gi <= groups; ++gi) group_start[gi] = st[gi];
  return groups;
}

muon_status muon_device_status(void* ws, void* stream) {
  g_last_error.clear();
  if (!ws) return fail(MUON_ERR_ARG, "workspace is NULL");
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(MUON_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
  int word = 0;
  e = cudaMemcpy(&word, ws, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(MUON_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
  if (word) {
    const int zero = 0;
    cudaMemcpy(ws, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (word & kStatusTimeout) return fail(MUON_ERR_TIMEOUT, "a kernel gave up on a bounded wait");
  }
  return MUON_OK;
}

muon_status muon_debug_bounded_wait(void* ws, long long max_cycles, void* stream) {
  g_last_error.clear();
  if (!ws) return fail(MUON_ERR_ARG, "workspace is NULL");
  if (max_cycles <= 0 || max_cycles > 10000000000LL) return fail(MUON_ERR_ARG, "max_cycles out of range");
  const cudaError_t e = launch_debug_wait(static_cast<int*>(ws), max_cycles, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(MUON_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
  return MUON_OK;
}

muon_status muon_debug_gemm(const void* A, const void* A_lo, const void* B, const void* B_lo, int batch, int M,
                            int N, int K, int split, int b_mn, int sym, muon_dtype dt, void* out, void* out_lo,
                            void* ws, size_t ws_bytes, void* stream) {
  g_last_error.clear();
  if (!A || !B || !out || !ws || batch <= 0 || batch > kMaxBatch) return fail(MUON_ERR_ARG, "bad pointers or batch");
  if (ws_bytes < kHeader || reinterpret_cast<uintptr_t>(ws) % MUON_WS_ALIGN)
    return fail(MUON_ERR_WORKSPACE, "workspace must hold the %zu-byte header", kHeader);
  if ((sym & 1) && M != N) return fail(MUON_ERR_SHAPE, "sym needs M == N");
  if (b_mn != 0 && b_mn != 1) return fail(MUON_ERR_ARG, "b_mn must be 0 or 1");
  EpiParams e;
  memset(&e, 0, sizeof(e));
  e.c_acc = 1.f;
  e.r_scale = 1.f;
  e.lo_scale = kF16LoScale;
  if (dt == MUON_FP32) {
    e.Of = static_cast<float*>(out);
  } else {
    e.Oh = out;
    e.Ol = out_lo;
    e.o_f16 = dt == MUON_FP16 ? 1 : 0;
  }
  e.ld = N;
  e.bs = static_cast<long long>(M) * N;
  e.rows_valid = M;
  e.cols_valid = N;
  const long long bsb = static_cast<long long>(N) * K;
  cudaError_t err;
  const char* why = nullptr;
  if (dt == MUON_BF16 || dt == MUON_FP16) {
    if (M <= 0 || N <= 0 || K <= 0 || M % 256 || N % 256 || K % 128) return fail(MUON_ERR_SHAPE, "16-bit sizes");
    if (split < 1 || split > 5) return fail(MUON_ERR_ARG, "split must be 1, 2, 3, 4 or 5");
    if ((split == 2 || split == 3 || split == 5) && !A_lo) return fail(MUON_ERR_ARG, "split 2, 3 and 5 need A_lo");
    if (split >= 3 && !B_lo) return fail(MUON_ERR_ARG, "split 3, 4 and 5 need B_lo");
    if (split == 5 && dt != MUON_FP16) return fail(MUON_ERR_ARG, "split 5 needs fp16 operands");
    if (split == 4 && (dt != MUON_FP16 || !b_mn || M != K || (sym & 1)))
      return fail(MUON_ERR_ARG, "split 4 needs fp16, b_mn = 1, M == K and a full output");
    if (split == 4 && ws_bytes < kHeader + 2 * kDiagDim * kDiagDim)
      return fail(MUON_ERR_WORKSPACE, "split 4 needs a %zu-byte workspace", kHeader + 2 * kDiagDim * kDiagDim);
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(A_lo) |
         reinterpret_cast<uintptr_t>(B_lo)) % 16)
      return fail(MUON_ERR_ALIGN, "16-bit operands must be 16-byte aligned");
    int major = 0, minor = 0;
    muon_status ds;
    const int sms = device_sms(&major, &minor, &ds);
    if (ds != MUON_OK) return ds;
    if (major != 10 || minor != 3) return fail(MUON_ERR_UNSUPPORTED, "needs sm_103a");
    TcGemmDesc d;
    d.B = batch;
    d.M = M;
    d.N = N;
    d.K = K;
    d.sym = sym & 1;
    d.a_sym = (sym >> 1) & 1;
    d.b_sym = (sym >> 2) & 1;
    d.split = split == 4 ? 1 : split;
    d.b_mn = b_mn;
    d.f16 = dt == MUON_FP16 ? 1 : 0;
    d.A = TcOperand{A, split == 4 ? nullptr : A_lo, K, static_cast<long long>(M) * K};
    d.Bop = TcOperand{B, B_lo, b_mn ? N : K, bsb};
    d.tile_ctr = reinterpret_cast<int*>(static_cast<char*>(ws) + kDebugTileCtr);
    if (cudaMemsetAsync(d.tile_ctr, 0, sizeof(int), static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return fail(MUON_ERR_CUDA, "memset of the tile counter failed");
    if (split == 4) {  // D = 2^-11 I after the header
      d.diag = static_cast<char*>(ws) + kHeader;
      if (launch_fill_diag(const_cast<void*>(d.diag), f16_bits(1.f / kF16LoScale),
                           static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return fail(MUON_ERR_CUDA, "launch of the diagonal fill failed");
    }
    err = launch_tc_gemm(d, e, static_cast<int*>(ws), static_cast<cudaStream_t>(stream), sms, &why);
    if (err == cudaErrorInvalidValue && why) return fail(MUON_ERR_ARG, "%s", why);
  } else if (dt == MUON_FP32) {
    if (M <= 0 || N <= 0 || K <= 0 || M % 128 || N % 128 || K % 16) return fail(MUON_ERR_SHAPE, "fp32 sizes");
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B)) % 16)
      return fail(MUON_ERR_ALIGN, "fp32 operands must be 16-byte aligned");
    SimtGemmDesc d{batch, M, N, K, sym & 1, b_mn, static_cast<const float*>(A), K, static_cast<long long>(M) * K,
                   static_cast<const float*>(B), b_mn ? N : K, bsb};
    err = launch_simt_gemm(d, e, static_cast<cudaStream_t>(stream));
  } else {
    return fail(MUON_ERR_ARG, "bad dtype");
  }
  if (err != cudaSuccess)
    return fail(MUON_ERR_CUDA, "launch: %s%s%s", cudaGetErrorString(err), why ? ": " : "", why ? why : "");
  return MUON_OK;
}

void muon_profile_enable(int on) {
  g_prof_on = on != 0;
  if (g_prof_on) {  // a new recording replaces the old one; stopping keeps it readable
    g_prof.clear();
    g_event_next = 0;
  }
}

int muon_profile_count(void) { return static_cast<int>(g_prof.size()); }

muon_status muon_profile_get(int i, const char** kind, float* ms, double* flops, double* bytes) {
  g_last_error.clear();
  if (i < 0 || i >= static_cast<int>(g_prof.size())) return fail(MUON_ERR_ARG, "no record %d", i);
  const ProfRec& r = g_prof[i];
  if (cudaEventSynchronize(r.b) != cudaSuccess) return fail(MUON_ERR_CUDA, "event synchronize failed");
  float t = 0.f;
  if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) return fail(MUON_ERR_CUDA, "elapsed time failed");
  if (kind) *kind = r.kind;
  if (ms) *ms = t;
  if (flops) *flops = r.flops;
  if (bytes) *bytes = r.bytes;
  return MUON_OK;
}

// ------------------------------------------------------------------ static scratch
// Device scratch for muon_ns_batched_static: one file-scope array, present on
// every GPU that loads this library until the process exits.  Host code only
// sees a host-side stand-in for this symbol, so its device address is looked
// up (cudaGetSymbolAddress, on the current device) by every call that needs
// it and passed to the kernels like any caller workspace.  The array starts
// zeroed when the module loads; its first word is the status word, which
// kernels set on a bounded-wait timeout and muon_static_status reads and
// clears.
static constexpr size_t kStaticScratchBytes = size_t(64) << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

static muon_status static_scratch_addr(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
  if (e != cudaSuccess || !p) {
    cudaGetLastError();
    return fail(MUON_ERR_CUDA, "cudaGetSymbolAddress of the static scratch: %s", cudaGetErrorString(e));
  }
  *out = p;
  return MUON_OK;
}

muon_status muon_ns_batched_static(const void* X, int B, int m, int n, int steps, const float* coeffs, void* out,
                                   muon_dtype dt, muon_sched sc, void* stream) {
  g_last_error.clear();
  try {
    if (B < 0) return fail(MUON_ERR_ARG, "B=%d < 0", B);
    if (B > 0 && (!X || !out)) return fail(MUON_ERR_ARG, "X or out is NULL");
    if (m <= 0 || n <= 0 || m > MUON_MAX_DIM || n > MUON_MAX_DIM)
      return fail(MUON_ERR_SHAPE, "bad shape %dx%d", m, n);
    if (steps < 0 || steps > MUON_MAX_STEPS)
      return fail(MUON_ERR_ARG, "steps=%d out of [0, %d]", steps, MUON_MAX_STEPS);
    if (!valid_dt(dt) || !valid_sc(sc)) return fail(MUON_ERR_ARG, "bad dtype or schedule");
    // Reject problems whose single matrix does not fit the fixed scratch, before any CUDA call.
    const Group g = make_group(m, n, steps, dt, sc, coef_of(coeffs));
    const size_t need = group_bytes(g, 1, dt);
    if (need > kStaticScratchBytes)
      return fail(MUON_ERR_WORKSPACE,
                  "a %dx%d matrix needs %zu bytes of scratch; the static scratch of muon_ns_batched_static holds "
                  "%zu bytes (use muon_ns_batched with a caller workspace)",
                  m, n, need, kStaticScratchBytes);
    if (B == 0) return MUON_OK;
    void* scratch = nullptr;
    const muon_status st = static_scratch_addr(&scratch);
    if (st != MUON_OK) return st;
    return muon_ns_batched(X, B, m, n, steps, coeffs, out, dt, sc, scratch, kStaticScratchBytes, stream);
  } catch (...) {
    return fail(MUON_ERR_ARG, "internal exception");
  }
}

muon_status muon_static_status(void* stream) {
  g_last_error.clear();
  try {
    void* scratch = nullptr;
    const muon_status st = static_scratch_addr(&scratch);
    if (st != MUON_OK) return st;
    return muon_device_status(scratch, stream);
  } catch (...) {
    return fail(MUON_ERR_ARG, "internal exception");
  }
}

muon_status muon_debug_bounded_wait_static(long long max_cycles, void* stream) {
  g_last_error.clear();
  try {
    void* scratch = nullptr;
    const muon_status st = static_scratch_addr(&scratch);
    if (st != MUON_OK) return st;
    return muon_debug_bounded_wait(scratch, max_cycles, stream);
  } catch (...) {
    return fail(MUON_ERR_ARG, "internal exception");
  }
}

size_t muon_static_scratch_bytes(void) { return kStaticScratchBytes; }

const char* muon_last_error(void) { return g_last_error.c_str(); }

const char* muon_version(void) { return "muon-ns-gb300 0.1 (sm_103a)"; }

}  // extern "C"
