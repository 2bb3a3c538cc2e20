// C ABI of the DyRA linear layer (include/dyra.h): offline preparation and the online
// forward, which enqueues the CUDA kernels of this library on the caller's stream.
//
// bf16 low-rank forward, per sample s (every contraction on tcgen05 through tc_gemm), as one
// chain of kernels on the caller's stream:
//   1. T = X [U | P]                     -> [X U | L]                 (static branch, L = X P)
//   2. [C^T ; G] = [X | L]^T L           -> C^T = X^T L (fp32), G = L^T L
//   3. C~ = (G + lambda I)^-1 C          (block sweeps for r <= 64, Newton-Schulz otherwise)
//   4. R = C~ W_res                      one [batch r x d] [d x m] GEMM
//   5. Y = [X U | L] [V ; R] + b         (the bias in the epilogue)
// R = G^-1 (C W_res) = (G^-1 C) W_res is the R-update of the one-step ALS; solving on C
// before the residual product keeps the solve at r x d per sample. The Monarch static branch
// replaces step 1 by X BD1, X P and the stride permutation, and step 5's static chunks by BD2.
#include "../../include/dyra.h"
#include "fit.h"
#include "kernels.cuh"
#include "monarch.cuh"
#include "tc_gemm.cuh"

#include <cuda_bf16.h>

#include <algorithm>
#include <array>
#include <cmath>
#include <cstring>
#include <memory>
#include <mutex>
#include <new>
#include <string>
#include <vector>

struct dyra_layer {
  int d = 0, m = 0, k = 0, r = 0, kp = 0;
  dyra_static_kind kind = DYRA_STATIC_LOWRANK;
  dyra_dtype dtype = DYRA_BF16;
  dyra_solver solver = DYRA_SOLVE_CHOLESKY;
  dyra_activation activation = DYRA_ACT_NONE;
  int ns_iters = 8;
  int als_half = 2;        // ALS half-steps: 2 t (t = 1: one L-update, one R-update)
  double ridge = 0.0;
  int device = 0;
  std::vector<double> W_hat, W_res, P, R0, F1, F2, F3, bias;
  int blast_t = 0;
  // device copies. kp = the static columns of T: roundup(k, 64) (low rank) or d (Monarch).
  // bf16 low rank: w1 = [U^T (padded to kp rows); P^T] [kp + r, d], v = V^T [m, kp];
  // bf16 Monarch: w1 = P^T [r, d], bd1 / bd2 = the block-diagonal factors as K-major tiles
  // [d][256] / [m][256] (row = output column, K local to the output's 256-column tile);
  // wres = W_res^T [m, d] (bf16); f32: w1 = [U | P] [d, k + r], v = V [k, m], wres = W_res [d, m]
  void *w1 = nullptr, *v = nullptr, *wres = nullptr, *bd1 = nullptr, *bd2 = nullptr;
  float *bias_d = nullptr;
  mutable std::mutex mu;                 // plan cache
  mutable std::vector<std::pair<std::array<uintptr_t, 5>, std::shared_ptr<void>>> plans;
  // the host-buffer forward's copy streams and events (created on first use)
  mutable std::mutex host_mu;
  mutable cudaStream_t copy_in = nullptr, copy_out = nullptr;
  mutable std::vector<cudaEvent_t> host_ev;
};

namespace {

thread_local std::string g_last_error;

dyra_status cuda_fail(cudaError_t e, const char *where) {
  g_last_error = std::string(where) + ": " + cudaGetErrorString(e);
  return DYRA_ERR_CUDA;
}

#define DY_CUDA(call)                                   \
  do {                                                  \
    cudaError_t e_ = (call);                            \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
  } while (0)

inline long long cdiv(long long a, long long b) { return (a + b - 1) / b; }
inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
inline int roundup(int x, int q) { return (x + q - 1) / q * q; }

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

// ------------------------------------------------------------------------ workspace

struct WsLayout {
  size_t T = 0, C = 0, G = 0, Ginv = 0, EX0 = 0, EX1 = 0, G32 = 0, B = 0, R = 0, Cs = 0,
         total = 0;
  size_t clear = 16;   // bytes at the start cleared before a forward (status and flags)
  size_t ready = 0;    // [2][batch] ints: the fused Gram / solve kernel's per-sample flags
  int ldT = 0;
};

// The R-update's Gram GEMM takes the SPD solve into its epilogue (one kernel instead of
// three) for the Cholesky branch.
inline bool fused_gram_solve(const dyra_layer *L) {
  return L->dtype == DYRA_BF16 && L->solver == DYRA_SOLVE_CHOLESKY && L->r <= 64 && L->r % 4 == 0;
}

WsLayout layout_of(const dyra_layer *L, int batch, int n) {
  WsLayout w;
  size_t off = 256;   // status words: [0] not-SPD samples, [1] bounded waits that gave up
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align256(off + bytes);
    return at;
  };
  const size_t B = (size_t)batch, N = (size_t)n, d = L->d, m = L->m, r = L->r;
  if (L->dtype == DYRA_BF16) {
    if (fused_gram_solve(L)) {   // right after the status words: one memset clears both
      w.ready = take(B * 2 * 4);
      w.clear = w.ready + B * 2 * 4;
    }
    w.ldT = L->kp + L->r;
    w.T = take(B * N * (size_t)w.ldT * 2);
    w.C = take(B * d * r * 4);   // C^T, fp32
    w.G = take(B * r * r * 4);
    w.Ginv = take(B * r * r * 2);
    w.G32 = take(B * r * r * 4);         // fp32 G^-1, read by the apply step
    if (L->solver == DYRA_SOLVE_NEWTON_SCHULZ) {
      w.EX0 = take(B * 2 * r * r * 4);   // [E ; X] iterate, two buffers
      w.EX1 = take(B * 2 * r * r * 4);
    }
    w.Cs = take(B * r * d * 2);
    w.R = take(B * r * m * 2);
  } else {
    w.ldT = L->k + L->r;
    w.T = take(B * N * (size_t)w.ldT * 4);
    w.G = take(B * r * r * 8);
    w.Ginv = take(B * r * r * 8);
    w.C = take(B * r * d * 4);
    w.B = take(B * r * m * 4);
    w.R = take(B * r * m * 4);
  }
  w.total = off;
  return w;
}

// ------------------------------------------------------------------------ launch plans
//
// A plan is the list of launches of one forward for a fixed (X, Y, workspace, batch, n):
// tensor maps and kernel parameters are encoded once and reused by later calls with the
// same buffers, so a steady-state forward costs only its launches on the host.

struct Step {
  enum Kind { GEMM, SPD_INVERT, SPD_APPLY, NS_FUSED, PERMUTE } kind = GEMM;
  const char *name = nullptr;   // the kernel's name in dyra_kernel_name
  dyra::TcGemmParams p;
  CUtensorMap a0, a1, b0, b1, out;
  CUtensorMap ns_maps[2][2];
  const float *G = nullptr;
  float *X0 = nullptr, *X1 = nullptr;
  __nv_bfloat16 *Ginv = nullptr;
  __nv_bfloat16 *T = nullptr;
  const float *Ct = nullptr;
  float *G32 = nullptr;
  __nv_bfloat16 *Cs = nullptr;
  int *status = nullptr;
  int batch = 0, r = 0, d = 0, ldT = 0, nb = 0;
  long long rows = 0;
  float ridge = 0.f;
};

struct Plan {
  std::vector<Step> steps;
  size_t clear = 16;   // bytes of the workspace cleared before a forward
};

// Records an event pair around each kernel, on the stream that kernel runs on. Under stream
// capture the records become event-record nodes of the graph (external records), so the
// graph's replays time the kernels too.
struct Recorder {
  cudaEvent_t *ev = nullptr;
  int max = 0, count = 0;
  void mark(cudaStream_t s) {
    if (ev && count < max) {
      cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
      if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(ev[count], s, cudaEventRecordExternal);
      else
        cudaEventRecord(ev[count], s);
    }
    ++count;
  }
};

#define DY_TIMED(rec, stream, call) \
  do {                              \
    (rec).mark(stream);             \
    DY_CUDA(call);                  \
    (rec).mark(stream);             \
  } while (0)

bool make_map(CUtensorMap *map, const void *base, int eb, long long inner, long long rows,
              long long batch, long long row_stride_el, long long batch_stride_el, int box_rows) {
  dyra::TcOperand op{base, eb, inner, rows, batch, row_stride_el * eb, batch_stride_el * eb};
  return dyra::tc_make_map(map, op, box_rows);
}

bool make_store_map(CUtensorMap *map, const void *base, long long inner, long long rows,
                    long long batch, long long row_stride_el, long long batch_stride_el) {
  dyra::TcOperand op{base, 2, inner, rows, batch, row_stride_el * 2, batch_stride_el * 2};
  return dyra::tc_make_store_map(map, op);
}

// GEMMs whose A operand is K-major run as cta_group::2 pair MMAs (M = 256 per CTA pair, B
// split between the pair, each CTA loading its own half), which cuts each SM's shared-memory
// traffic per MMA by a third.
constexpr bool kPairMma = true;
constexpr int kBDiv = kPairMma ? 2 : 1;   // K-major B box rows = BN / kBDiv

void set_pair(dyra::TcGemmParams &p, int elem_bytes, int b_major1) {
  if (!kPairMma) return;
  p.pair_mma = 1;
  p.idesc = dyra::tc_idesc(elem_bytes, 0, 0, p.BN, 256);
  p.idesc1 = dyra::tc_idesc(elem_bytes, 0, b_major1, p.BN, 256);
}

// The output GEMM tiles the flat batch * n rows (its rank chunks then repeat for every
// sample that a tile's rows touch) when per-sample tiles would leave part of each sample's
// last tile empty. Below 64 rows per sample a tile would touch too many samples.
bool use_flat_rows(int batch, int n) {
  const int unit = kPairMma ? 256 : 128;
  return batch > 1 && n >= 64 && n % unit != 0;
}

// Switches the output GEMM `p` (per-sample maps a0 / o over [batch][n]) to flat rows:
// a0 and o become [batch * n] views, a1 keeps the per-sample view for the rank chunks.
dyra_status set_flat_rows(dyra::TcGemmParams &p, CUtensorMap &a0, CUtensorMap &o,
                          const void *T, int ldT, void *Y, int m, int batch, int n) {
  const long long rows = (long long)batch * n;
  if (!make_map(&a0, T, 2, ldT, rows, 1, ldT, 0, 128) ||
      !make_store_map(&o, Y, m, rows, 1, m, 0)) {
    g_last_error = "cuTensorMapEncodeTiled failed: flat output maps";
    return DYRA_ERR_CUDA;
  }
  p.m_tiles = (int)cdiv(rows, 128);
  p.batch = 1;
  p.a_split = p.m_tiles;
  p.a_batched0 = 0;
  p.seg_n = n;
  p.seg_count = batch;
  p.out_batched = 0;
  p.rows_valid = (int)rows;
  return DYRA_OK;
}

dyra::TcGemmParams base_params() {
  dyra::TcGemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.alpha = 1.f;
  p.cluster = 1;
  p.a_k1 = -1;
  return p;
}

Step gemm_step(const dyra::TcGemmParams &p, const CUtensorMap &a0, const CUtensorMap &a1,
               const CUtensorMap &b0, const CUtensorMap &b1) {
  Step st;
  st.kind = Step::GEMM;
  st.p = p;
  st.a0 = a0;
  st.a1 = a1;
  st.b0 = b0;
  st.b1 = b1;
  st.out = a0;
  return st;
}

#define DY_MAP(expr)                                               \
  do {                                                             \
    if (!(expr)) {                                                 \
      g_last_error = "cuTensorMapEncodeTiled failed: " #expr;      \
      return DYRA_ERR_CUDA;                                        \
    }                                                              \
  } while (0)

// ------------------------------------------------------------------------ bf16 low-rank path

// N width of a GEMM tile (multiple of `q`, <= 256) for an M x N output on a persistent grid
// of one CTA per SM: fewest rounds of tiles, weighed by a tile's main-loop time (which grows
// with its width plus a fixed per-chunk issue cost).
int pick_bn(long long M, int N, int q) {
  int best = 256, sms = 148, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = 148;
  double best_cost = 1e300;
  for (int bn = 256; bn >= 64; bn -= q) {
    if (bn % q) continue;
    const long long tiles = cdiv(M, 128) * cdiv(N, bn);
    const double cost = (double)cdiv(tiles, sms) * (bn + 96);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

// L = X P (P^T [r, d] is the layer's w1) into T[:, col : col + r], over the flat batch * n
// rows (X and T are dense row blocks).
dyra_status plan_l_projection(const dyra_layer *L, const void *X, int batch, int n,
                              __nv_bfloat16 *T, int ldT, int col, int *status, Plan &plan) {
  using namespace dyra;
  const int d = L->d, r = L->r;
  const long long rows = (long long)batch * n;
  CUtensorMap a, b, o;
  const int BN = roundup(r, kPairMma ? 32 : 16);
  DY_MAP(make_map(&a, X, 2, d, rows, 1, d, 0, 128));
  DY_MAP(make_map(&b, L->w1, 2, d, r, 1, d, 0, BN / kBDiv));
  DY_MAP(make_store_map(&o, T + col, r, rows, 1, ldT, 0));
  TcGemmParams p = base_params();
  p.m_tiles = (int)cdiv(rows, 128);
  p.n_tiles = 1;
  p.batch = 1;
  p.BN = BN;
  p.k_chunks = (int)cdiv(d, 64);
  p.elem_bytes = 2;
  p.a_split = p.m_tiles;
  p.b_split = p.k_chunks;
  p.idesc = p.idesc1 = tc_idesc(2, 0, 0, BN);
  set_pair(p, 2, 0);
  p.epi = EPI_ROW_BF16;
  p.tma_store = 1;
  p.rows_valid = (int)rows;
  p.cols_valid = r;
  p.timeouts = status + 1;
  Step st = gemm_step(p, a, a, b, b);
  st.out = o;
  st.name = "xproj_L";
  plan.steps.push_back(st);
  return DYRA_OK;
}

// BLAST static branch, front half ([S] Appendix B; blog structured-methods section): stage 1,
// Z[:, i t : (i + 1) t] = X[:, i p : (i + 1) p] U_i for every block row i, as one GEMM whose
// N tile i contracts only with input block i; then L = X P into T[:, kp : kp + r]. The
// middle matrices and the column bases are folded into the output GEMM's static factor.
dyra_status plan_blast_front(const dyra_layer *L, const void *X, int batch, int n,
                             __nv_bfloat16 *T, int ldT, int *status, Plan &plan) {
  using namespace dyra;
  const int d = L->d, nb = L->k, t = L->blast_t, pb = d / nb;
  const long long rows = (long long)batch * n;
  {
    CUtensorMap a, b, o;
    const int BN = t;
    DY_MAP(make_map(&a, X, 2, d, rows, 1, d, 0, 128));
    DY_MAP(make_map(&b, L->bd1, 2, pb, (long long)nb * t, 1, pb, 0, BN / kBDiv));
    DY_MAP(make_store_map(&o, T, (long long)nb * t, rows, 1, ldT, 0));
    TcGemmParams p = base_params();
    p.m_tiles = (int)cdiv(rows, 128);
    p.n_tiles = nb;
    p.batch = 1;
    p.BN = BN;
    p.k_chunks = pb / 64;
    p.elem_bytes = 2;
    p.a_split = p.m_tiles;
    p.a_kdiag = pb;
    p.b_split = p.k_chunks;
    p.idesc = p.idesc1 = tc_idesc(2, 0, 0, BN);
    set_pair(p, 2, 0);
    p.epi = EPI_ROW_BF16;
    p.tma_store = 1;
    p.rows_valid = (int)rows;
    p.cols_valid = nb * t;
    p.timeouts = status + 1;
    Step st = gemm_step(p, a, a, b, b);
    st.out = o;
    st.name = "blast_stage1";
    plan.steps.push_back(st);
  }
  return plan_l_projection(L, X, batch, n, T, ldT, L->kp, status, plan);
}

// Monarch static branch, front half: T[:, 0:d] = the permuted X BD1, T[:, d:d+r] = L = X P.
dyra_status plan_monarch_front(const dyra_layer *L, const void *X, int batch, int n,
                               __nv_bfloat16 *T, int ldT, int *status, Plan &plan) {
  using namespace dyra;
  const int d = L->d, nb = L->k;
  // Z = X BD1: 256-column tiles, each contracting with its own 256 input columns
  {
    CUtensorMap a, b, o;
    const int BN = 256;
    DY_MAP(make_map(&a, X, 2, d, n, batch, d, (long long)n * d, 128));
    DY_MAP(make_map(&b, L->bd1, 2, 256, d, 1, 256, 0, BN / kBDiv));
    DY_MAP(make_store_map(&o, T, d, n, batch, ldT, (long long)n * ldT));
    TcGemmParams p = base_params();
    p.m_tiles = (int)cdiv(n, 128);
    p.n_tiles = d / BN;
    p.batch = batch;
    p.BN = BN;
    p.k_chunks = BN / 64;
    p.elem_bytes = 2;
    p.a_split = p.m_tiles;
    p.a_batched0 = 1;
    p.a_kdiag = BN;
    p.b_split = p.k_chunks;
    p.idesc = p.idesc1 = tc_idesc(2, 0, 0, BN);
    set_pair(p, 2, 0);
    p.epi = EPI_ROW_BF16;
    p.tma_store = 1;
    p.out_batched = 1;
    p.rows_valid = n;
    p.cols_valid = d;
    p.timeouts = status + 1;
    Step st = gemm_step(p, a, a, b, b);
    st.out = o;
    st.name = "monarch_bd1";
    plan.steps.push_back(st);
  }
  // L = X P into T[:, d:d+r]
  const dyra_status ls = plan_l_projection(L, X, batch, n, T, ldT, d, status, plan);
  if (ls != DYRA_OK) return ls;
  // the stride permutation between the two factors, in place
  {
    Step st;
    st.kind = Step::PERMUTE;
    st.T = T;
    st.rows = (long long)batch * n;
    st.ldT = ldT;
    st.nb = nb;
    st.name = "monarch_permute";
    plan.steps.push_back(st);
  }
  return DYRA_OK;
}

// [C^T ; G] = [X | L]^T L per sample, from the L columns of T (both operands MN-major: the
// reduction runs over tokens). C^T [batch, d, r] and G [batch, r, r], fp32.
dyra_status plan_gram_c(const dyra_layer *L, const void *X, int batch, int n,
                        const __nv_bfloat16 *T, int ldT, float *Ct, float *G, int *status,
                        Plan &plan) {
  using namespace dyra;
  const int d = L->d, r = L->r, kp = L->kp;
  {
    CUtensorMap ax, al;
    DY_MAP(make_map(&ax, X, 2, d, n, batch, d, (long long)n * d, 64));
    DY_MAP(make_map(&al, T + kp, 2, r, n, batch, ldT, (long long)n * ldT, 64));
    TcGemmParams p = base_params();
    p.a_split = (int)cdiv(d, 128);
    p.m_tiles = p.a_split + (int)cdiv(r, 128);
    p.n_tiles = 1;
    p.batch = batch;
    p.BN = roundup(r, 64);
    p.k_chunks = (int)cdiv(n, 64);
    p.elem_bytes = 2;
    p.a_major = 1;
    p.b_major = 1;
    p.a_batched0 = p.a_batched1 = 1;
    p.b_split = p.k_chunks;
    p.b_batched0 = 1;
    p.idesc = tc_idesc(2, 1, 1, p.BN);
    p.epi = EPI_CG;
    p.out = Ct;                      // C^T [batch, d, r], fp32
    p.out_bstride = (long long)d * r;
    p.out_ld = r;
    p.rows_valid = d;
    p.cols_valid = r;
    p.out2 = G;
    p.out2_bstride = (long long)r * r;
    p.out2_ld = r;
    p.rows2_valid = r;
    p.cols2_valid = r;
    p.timeouts = status + 1;
    plan.steps.push_back(gemm_step(p, ax, al, al, al));
    plan.steps.back().name = "cg_c_gram";
  }
  return DYRA_OK;
}

// The R-update's Gram GEMM with the solve in its epilogue (r <= 64, Cholesky branch): per
// sample, the G tile [r, r] comes first in the walk and is inverted by its CTA's epilogue
// warps, which publish (G + lambda I)^-1 (G32 fp32, Ginv bf16) and a flag; each 128-feature
// C^T tile waits for its sample's flag and writes C~ = (G + lambda I)^-1 C (Cs, bf16
// [batch, r, d]). C^T and G also go out (fp32) for checks of the intermediates.
dyra_status plan_gram_solve(const dyra_layer *L, const void *X, int batch, int n,
                            const __nv_bfloat16 *T, int ldT, float *Ct, float *G,
                            __nv_bfloat16 *Cs, uint8_t *ws, const WsLayout &w, int *status,
                            Plan &plan) {
  using namespace dyra;
  const int d = L->d, r = L->r, kp = L->kp;
  CUtensorMap ax, al;
  DY_MAP(make_map(&ax, X, 2, d, n, batch, d, (long long)n * d, 64));
  DY_MAP(make_map(&al, T + kp, 2, r, n, batch, ldT, (long long)n * ldT, 64));
  TcGemmParams p = base_params();
  p.a_split = (int)cdiv(d, 128);
  p.m_tiles = p.a_split + 1;
  p.n_tiles = 1;
  p.batch = batch;
  p.BN = roundup(r, 64);
  p.k_chunks = (int)cdiv(n, 64);
  p.elem_bytes = 2;
  p.a_major = 1;
  p.b_major = 1;
  p.a_batched0 = p.a_batched1 = 1;
  p.b_split = p.k_chunks;
  p.b_batched0 = 1;
  p.idesc = tc_idesc(2, 1, 1, p.BN);
  p.epi = EPI_CG_SOLVE;
  p.g_first = 1;
  p.solve_r = r;
  p.ridge = (float)L->ridge;
  p.ginv32 = reinterpret_cast<float *>(ws + w.G32);
  p.ginv16 = reinterpret_cast<__nv_bfloat16 *>(ws + w.Ginv);
  p.cs = Cs;
  p.cs_d = d;
  p.ready = reinterpret_cast<int *>(ws + w.ready);
  p.nspd = status;
  p.out = Ct;
  p.out_bstride = (long long)d * r;
  p.out_ld = r;
  p.rows_valid = d;
  p.cols_valid = r;
  p.out2 = G;
  p.timeouts = status + 1;
  plan.steps.push_back(gemm_step(p, ax, al, al, al));
  plan.steps.back().name = "cg_solve";
  return DYRA_OK;
}

// Cs = (Gs + lambda I)^-1 Cs_src^T per sample: Gs [batch, r, r] fp32 (consumed), the operand
// given as its transpose Ct [batch, d, r] fp32, the result bf16 [batch, r, d]; G^-1 also to
// Ginv (bf16) and G32 (fp32). r <= 64 (Cholesky branch): one CTA per sample inverts G, then
// a wide kernel applies the inverse; larger r: Newton-Schulz (ns_iterate), then a
// tf32 GEMM applies the inverse.
dyra_status plan_solve(const dyra_layer *L, int batch, float *G, float ridge, const float *Ct,
                       __nv_bfloat16 *Cs, uint8_t *ws, const WsLayout &w, int *status,
                       Plan &plan) {
  using namespace dyra;
  const int d = L->d, r = L->r;
  __nv_bfloat16 *Ginv = reinterpret_cast<__nv_bfloat16 *>(ws + w.Ginv);
  float *G32 = reinterpret_cast<float *>(ws + w.G32);
  if (L->solver == DYRA_SOLVE_CHOLESKY) {
    Step st;
    st.kind = Step::SPD_INVERT;
    st.G = G;
    st.batch = batch;
    st.r = r;
    st.d = d;
    st.ridge = ridge;
    st.Ct = Ct;
    st.Cs = Cs;
    st.Ginv = Ginv;
    st.G32 = G32;
    st.status = status;
    st.name = "spd_invert";
    plan.steps.push_back(st);
    st.kind = Step::SPD_APPLY;
    st.name = "spd_apply_c";
    plan.steps.push_back(st);
  } else {
    // Newton-Schulz in residual form, start to finish in one cluster kernel: EX = [E ; X]
    // per sample ([2r][r] fp32, two buffers used in turn); each iteration forms
    // X' = X + X E and E' = E E.
    float *EXa = reinterpret_cast<float *>(ws + w.EX0);
    float *EXb = reinterpret_cast<float *>(ws + w.EX1);
    const long long ex_bs = 2LL * r * r;   // elements between samples of EX
    {
      Step st;
      st.kind = Step::NS_FUSED;
      float *bufs[2] = {EXa, EXb};
      for (int bi = 0; bi < 2; ++bi)
        for (int blk = 0; blk < 2; ++blk)
          DY_MAP(make_map(&st.ns_maps[bi][blk], bufs[bi] + (size_t)blk * r * r, 4, r, r, batch, r,
                          ex_bs, 128));
      st.G = G;
      st.ridge = ridge;
      st.X0 = EXa;
      st.X1 = EXb;
      st.batch = batch;
      st.r = r;
      st.nb = L->ns_iters;
      st.Ginv = Ginv;
      st.G32 = G32;
      st.status = status;
      st.name = "ns_iterate";
      plan.steps.push_back(st);
    }
    // C~ = G^-1 C as a tf32 GEMM: M = r rows of G^-1 (fp32, K-major), N = d, K = r, with
    // B = C^T [d, r] (K-major); bf16 result [batch, r, d]
    {
      CUtensorMap a, b, o;
      const int BN = pick_bn((long long)batch * cdiv(r, 128) * 128, d, 32);
      DY_MAP(make_map(&a, G32, 4, r, r, batch, r, (long long)r * r, 128));
      DY_MAP(make_map(&b, Ct, 4, r, d, batch, r, (long long)d * r, BN / kBDiv));
      DY_MAP(make_store_map(&o, Cs, d, r, batch, d, (long long)r * d));
      TcGemmParams p = base_params();
      p.m_tiles = (int)cdiv(r, 128);
      p.n_tiles = (int)cdiv(d, BN);
      p.batch = batch;
      p.BN = BN;
      p.k_chunks = (int)cdiv(r, 32);
      p.elem_bytes = 4;
      p.a_split = p.m_tiles;
      p.a_batched0 = 1;
      p.b_split = p.k_chunks;
      p.b_batched0 = 1;
      p.idesc = p.idesc1 = tc_idesc(4, 0, 0, BN);
      set_pair(p, 4, 0);
      p.epi = EPI_ROW_BF16;
      p.tma_store = 1;
      p.out_batched = 1;
      p.rows_valid = r;
      p.cols_valid = d;
      p.timeouts = status + 1;
      Step st = gemm_step(p, a, a, b, b);
      st.out = o;
      st.name = "ginv_c";
      plan.steps.push_back(st);
    }
  }
  return DYRA_OK;
}

// R = C~ W_res, one [batch * r, d] x [d, m] GEMM, row-major [batch * r, m].
dyra_status plan_residual(const dyra_layer *L, int batch, const __nv_bfloat16 *Cs,
                          __nv_bfloat16 *Rm, int *status, Plan &plan) {
  using namespace dyra;
  const int d = L->d, m = L->m, r = L->r;
  {
    CUtensorMap a, b, o;
    const long long rows = (long long)batch * r;
    const int BN = pick_bn(rows, m, 32);
    DY_MAP(make_map(&a, Cs, 2, d, rows, 1, d, 0, 128));
    DY_MAP(make_map(&b, L->wres, 2, d, m, 1, d, 0, BN / kBDiv));
    DY_MAP(make_store_map(&o, Rm, m, rows, 1, m, 0));
    TcGemmParams p = base_params();
    p.m_tiles = (int)cdiv(rows, 128);
    p.n_tiles = (int)cdiv(m, BN);
    p.m_fast = 1;   // W_res is the large operand: each column block read once from HBM
    p.batch = 1;
    p.BN = BN;
    p.k_chunks = (int)cdiv(d, 64);
    p.elem_bytes = 2;
    p.a_split = p.m_tiles;
    p.b_split = p.k_chunks;
    p.idesc = p.idesc1 = tc_idesc(2, 0, 0, BN);
    set_pair(p, 2, 0);
    p.epi = EPI_ROW_BF16;
    p.tma_store = 1;
    p.rows_valid = (int)rows;
    p.cols_valid = m;
    p.timeouts = status + 1;
    Step st = gemm_step(p, a, a, b, b);
    st.out = o;
    st.name = "residual_product";
    plan.steps.push_back(st);
  }
  return DYRA_OK;
}

// L-update of ALS with R held fixed (t > 1; blog section "残差乘积的低秩优化目标是什么": with R
// fixed, L is the least-squares solution, computed by reducing the output dimension to r
// first): from R [batch, r, m] (bf16),
//   H = R R^T,   Q = W_res R^T,   P_s^T = H^-1 Q^T,   L = X P_s,
// the new L written into the L columns of T. H, Q and P_s^T reuse the G, C^T and C~ buffers.
dyra_status plan_l_update(const dyra_layer *L, const void *X, int batch, int n,
                          __nv_bfloat16 *T, int ldT, const __nv_bfloat16 *Rm, float *H, float *Q,
                          __nv_bfloat16 *PsT, uint8_t *ws, const WsLayout &w, int *status,
                          Plan &plan) {
  using namespace dyra;
  const int d = L->d, m = L->m, r = L->r, kp = L->kp;
  {   // H = R R^T: K = m, both operands rows of R (K-major)
    CUtensorMap a, b;
    const int BN = roundup(r, 16);
    DY_MAP(make_map(&a, Rm, 2, m, r, batch, m, (long long)r * m, 128));
    DY_MAP(make_map(&b, Rm, 2, m, r, batch, m, (long long)r * m, BN));
    TcGemmParams p = base_params();
    p.m_tiles = (int)cdiv(r, 128);
    p.n_tiles = 1;
    p.batch = batch;
    p.BN = BN;
    p.k_chunks = (int)cdiv(m, 64);
    p.elem_bytes = 2;
    p.a_split = p.m_tiles;
    p.a_batched0 = 1;
    p.b_split = p.k_chunks;
    p.b_batched0 = 1;
    p.idesc = p.idesc1 = tc_idesc(2, 0, 0, BN);
    p.epi = EPI_ROW_F32;
    p.out = H;
    p.out_bstride = (long long)r * r;
    p.out_ld = r;
    p.rows_valid = r;
    p.cols_valid = r;
    p.timeouts = status + 1;
    plan.steps.push_back(gemm_step(p, a, a, b, b));
    plan.steps.back().name = "als_gram_r";
  }
  {   // Q = W_res R^T [batch, d, r]: A = W_res read MN-major from W_res^T [m, d]
    CUtensorMap a, b;
    const int BN = roundup(r, 16);
    DY_MAP(make_map(&a, L->wres, 2, d, m, 1, d, 0, 64));
    DY_MAP(make_map(&b, Rm, 2, m, r, batch, m, (long long)r * m, BN));
    TcGemmParams p = base_params();
    p.m_tiles = (int)cdiv(d, 128);
    p.n_tiles = 1;
    p.batch = batch;
    p.BN = BN;
    p.k_chunks = (int)cdiv(m, 64);
    p.elem_bytes = 2;
    p.a_major = 1;
    p.a_split = p.m_tiles;
    p.b_split = p.k_chunks;
    p.b_batched0 = 1;
    p.idesc = p.idesc1 = tc_idesc(2, 1, 0, BN);
    p.epi = EPI_ROW_F32;
    p.out = Q;
    p.out_bstride = (long long)d * r;
    p.out_ld = r;
    p.rows_valid = d;
    p.cols_valid = r;
    p.timeouts = status + 1;
    plan.steps.push_back(gemm_step(p, a, a, b, b));
    plan.steps.back().name = "als_q";
  }
  // P_s^T = H^-1 Q^T (no ridge: the L-update is the plain least-squares step)
  dyra_status st = plan_solve(L, batch, H, 0.f, Q, PsT, ws, w, status, plan);
  if (st != DYRA_OK) return st;
  {   // L = X P_s per sample, into T's L columns
    CUtensorMap a, b, o;
    const int BN = roundup(r, kPairMma ? 32 : 16);
    DY_MAP(make_map(&a, X, 2, d, n, batch, d, (long long)n * d, 128));
    DY_MAP(make_map(&b, PsT, 2, d, r, batch, d, (long long)r * d, BN / kBDiv));
    DY_MAP(make_store_map(&o, T + kp, r, n, batch, ldT, (long long)n * ldT));
    TcGemmParams p = base_params();
    p.m_tiles = (int)cdiv(n, 128);
    p.n_tiles = 1;
    p.batch = batch;
    p.BN = BN;
    p.k_chunks = (int)cdiv(d, 64);
    p.elem_bytes = 2;
    p.a_split = p.m_tiles;
    p.a_batched0 = 1;
    p.b_split = p.k_chunks;
    p.b_batched0 = 1;
    p.idesc = p.idesc1 = tc_idesc(2, 0, 0, BN);
    set_pair(p, 2, 0);
    p.epi = EPI_ROW_BF16;
    p.tma_store = 1;
    p.out_batched = 1;
    p.rows_valid = n;
    p.cols_valid = r;
    p.timeouts = status + 1;
    Step stp = gemm_step(p, a, a, b, b);
    stp.out = o;
    stp.name = "als_l_update";
    plan.steps.push_back(stp);
  }
  return DYRA_OK;
}

dyra_status plan_bf16(const dyra_layer *L, const void *X, int batch, int n, void *Y,
                      uint8_t *ws, const WsLayout &w, Plan &plan) {
  using namespace dyra;
  const int d = L->d, m = L->m, r = L->r, kp = L->kp, ldT = w.ldT;
  int *status = reinterpret_cast<int *>(ws);
  __nv_bfloat16 *T = reinterpret_cast<__nv_bfloat16 *>(ws + w.T);
  float *Ct = reinterpret_cast<float *>(ws + w.C);   // C^T [batch, d, r]
  float *G = reinterpret_cast<float *>(ws + w.G);
  __nv_bfloat16 *Cs = reinterpret_cast<__nv_bfloat16 *>(ws + w.Cs);
  __nv_bfloat16 *Rm = reinterpret_cast<__nv_bfloat16 *>(ws + w.R);

  // 1. T = X [U | P]   (Monarch: permuted X BD1 and L)
  if (L->kind == DYRA_STATIC_MONARCH) {
    const dyra_status fs = plan_monarch_front(L, X, batch, n, T, ldT, status, plan);
    if (fs != DYRA_OK) return fs;
  } else if (L->kind == DYRA_STATIC_BLAST) {
    const dyra_status fs = plan_blast_front(L, X, batch, n, T, ldT, status, plan);
    if (fs != DYRA_OK) return fs;
  } else {
    // X and T are dense [batch * n] row blocks: the static and L columns of every token are
    // independent of its sample, so the GEMM tiles the flat rows (no per-sample tail tiles)
    CUtensorMap a, b, o;
    const int N = ldT;
    const long long rows = (long long)batch * n;
    const int BN = pick_bn(rows, N, 32);
    DY_MAP(make_map(&a, X, 2, d, rows, 1, d, 0, 128));
    DY_MAP(make_map(&b, L->w1, 2, d, N, 1, d, 0, BN / kBDiv));
    DY_MAP(make_store_map(&o, T, N, rows, 1, ldT, 0));
    TcGemmParams p = base_params();
    p.m_tiles = (int)cdiv(rows, 128);
    p.n_tiles = (int)cdiv(N, BN);
    p.batch = 1;
    p.BN = BN;
    p.k_chunks = (int)cdiv(d, 64);
    p.elem_bytes = 2;
    p.a_split = p.m_tiles;
    p.b_split = p.k_chunks;
    p.idesc = p.idesc1 = tc_idesc(2, 0, 0, BN);
    set_pair(p, 2, 0);
    p.epi = EPI_ROW_BF16;
    p.tma_store = 1;
    p.rows_valid = (int)rows;
    p.cols_valid = N;
    p.timeouts = status + 1;
    Step st = gemm_step(p, a, a, b, b);
    st.out = o;
    st.name = "xproj_static_L";
    plan.steps.push_back(st);
  }
  // 2-4. the R-update: [C^T ; G] = [X | L]^T L, C~ = (G + lambda I)^-1 C, R = C~ W_res
  auto r_update = [&]() {
    dyra_status e;
    if (fused_gram_solve(L)) {
      e = plan_gram_solve(L, X, batch, n, T, ldT, Ct, G, Cs, ws, w, status, plan);
    } else {
      e = plan_gram_c(L, X, batch, n, T, ldT, Ct, G, status, plan);
      if (e == DYRA_OK) e = plan_solve(L, batch, G, (float)L->ridge, Ct, Cs, ws, w, status, plan);
    }
    if (e == DYRA_OK) e = plan_residual(L, batch, Cs, Rm, status, plan);
    return e;
  };
  dyra_status st2 = r_update();
  if (st2 != DYRA_OK) return st2;
  // further ALS half-steps (t > 1): an L-update from the current R, then (t >= 2) another
  // R-update from the new L, and so on; the workspace buffers are reused
  for (int hs = 2; hs < L->als_half; ++hs) {
    if (hs % 2 == 0)
      st2 = plan_l_update(L, X, batch, n, T, ldT, Rm, G, Ct, Cs, ws, w, status, plan);
    else
      st2 = r_update();
    if (st2 != DYRA_OK) return st2;
  }
  // 5. Y = [X U | L] [V ; R] + b: K chunks of V^T (K-major, shared by all samples), then
  //    the sample's R (MN-major, [r, m] with m contiguous). Monarch: the first chunks are
  //    Zp BD2 on 256-column tiles (each contracting with its own 256 columns of Zp).
  if (L->kind == DYRA_STATIC_MONARCH) {
    CUtensorMap a, b0, b1, o;
    const int BN = 256;
    DY_MAP(make_map(&a, T, 2, ldT, n, batch, ldT, (long long)n * ldT, 128));
    DY_MAP(make_map(&b1, Rm, 2, m, r, batch, m, (long long)r * m, 64));
    DY_MAP(make_map(&b0, L->bd2, 2, 256, m, 1, 256, 0, BN / kBDiv));
    DY_MAP(make_store_map(&o, Y, m, n, batch, m, (long long)n * m));
    TcGemmParams p = base_params();
    p.m_tiles = (int)cdiv(n, 128);
    p.n_tiles = m / BN;
    p.batch = batch;
    p.BN = BN;
    p.b_split = BN / 64;
    p.k_chunks = p.b_split + (int)cdiv(r, 64);
    p.elem_bytes = 2;
    p.a_split = p.m_tiles;
    p.a_batched0 = 1;
    p.a_kdiag = BN;
    p.a_k1 = kp;
    p.b_batched0 = 0;
    p.b_batched1 = 1;
    p.b_major1 = 1;
    p.idesc = tc_idesc(2, 0, 0, BN);
    p.idesc1 = tc_idesc(2, 0, 1, BN);
    set_pair(p, 2, 1);
    p.epi = EPI_ROW_BF16;
    p.tma_store = 1;
    p.out_batched = 1;
    p.rows_valid = n;
    p.cols_valid = m;
    p.bias = L->bias_d;
    p.act = L->activation == DYRA_ACT_GELU ? 1 : 0;
    p.timeouts = status + 1;
    CUtensorMap a0 = a;
    if (use_flat_rows(batch, n)) {
      const dyra_status fs = set_flat_rows(p, a0, o, T, ldT, Y, m, batch, n);
      if (fs != DYRA_OK) return fs;
    }
    Step st = gemm_step(p, a0, a, b0, b1);
    st.out = o;
    st.name = "fused_output";
    plan.steps.push_back(st);
    return DYRA_OK;
  }
  {
    CUtensorMap a, b0, b1, o;
    const bool flat = use_flat_rows(batch, n);
    const int BN = pick_bn(flat ? (long long)batch * n : (long long)batch * cdiv(n, 128) * 128, m,
                           kPairMma ? 128 : 64);
    DY_MAP(make_map(&a, T, 2, ldT, n, batch, ldT, (long long)n * ldT, 128));
    DY_MAP(make_map(&b1, Rm, 2, m, r, batch, m, (long long)r * m, 64));
    if (kp > 0)
      DY_MAP(make_map(&b0, L->v, 2, kp, m, 1, kp, 0, BN / kBDiv));
    else
      b0 = b1;
    DY_MAP(make_store_map(&o, Y, m, n, batch, m, (long long)n * m));
    TcGemmParams p = base_params();
    p.m_tiles = (int)cdiv(n, 128);
    p.n_tiles = (int)cdiv(m, BN);
    p.batch = batch;
    p.BN = BN;
    p.b_split = kp / 64;
    p.k_chunks = p.b_split + (int)cdiv(r, 64);
    p.elem_bytes = 2;
    p.a_split = p.m_tiles;
    p.a_batched0 = 1;
    p.b_batched0 = 0;
    p.b_batched1 = 1;
    p.b_major1 = 1;
    p.idesc = tc_idesc(2, 0, 0, BN);
    p.idesc1 = tc_idesc(2, 0, 1, BN);
    set_pair(p, 2, 1);
    p.epi = EPI_ROW_BF16;
    p.tma_store = 1;
    p.out_batched = 1;
    p.rows_valid = n;
    p.cols_valid = m;
    p.bias = L->bias_d;
    p.act = L->activation == DYRA_ACT_GELU ? 1 : 0;
    p.timeouts = status + 1;
    CUtensorMap a0 = a;
    if (flat) {
      const dyra_status fs = set_flat_rows(p, a0, o, T, ldT, Y, m, batch, n);
      if (fs != DYRA_OK) return fs;
    }
    Step st = gemm_step(p, a0, a, b0, b1);
    st.out = o;
    st.name = "fused_output";
    plan.steps.push_back(st);
  }
  return DYRA_OK;
}

dyra_status run_plan(const dyra_layer *L, const Plan &plan, void *ws, cudaStream_t s,
                     Recorder &rec, bool clear_status) {
  using namespace dyra;
  // the fused Gram / solve kernel's flags are cleared even when the status words are kept
  // (a chained layer's flags may share bytes with the previous layer's buffers)
  if (clear_status)
    DY_CUDA(cudaMemsetAsync(ws, 0, plan.clear, s));
  else if (plan.clear > 16)
    DY_CUDA(cudaMemsetAsync(static_cast<uint8_t *>(ws) + 16, 0, plan.clear - 16, s));
  for (const Step &st : plan.steps) {
    const cudaStream_t ks = s;
    switch (st.kind) {
      case Step::GEMM:
        DY_TIMED(rec, ks, tc_gemm_launch(st.p, st.a0, st.a1, st.b0, st.b1, st.out, ks));
        break;
      case Step::SPD_INVERT:
        DY_TIMED(rec, ks, launch_spd_invert(st.G, st.batch, st.r, st.ridge, st.G32, st.Ginv,
                                             st.status, ks));
        break;
      case Step::SPD_APPLY:
        DY_TIMED(rec, ks, launch_spd_apply(st.G32, st.batch, st.r, st.Ct, st.d, st.Cs, ks));
        break;
      case Step::PERMUTE:
        DY_TIMED(rec, ks, launch_monarch_permute(st.T, st.rows, st.ldT, st.nb, ks));
        break;
      case Step::NS_FUSED:
        DY_TIMED(rec, ks, launch_ns_fused(st.ns_maps, st.batch, st.r, st.nb, st.ridge, st.G, st.X0,
                                          st.X1, st.G32, st.Ginv, st.status, ks));
        break;
      default:
        break;
    }
  }
  return DYRA_OK;
}

// ------------------------------------------------------------------------ fp32 path

dyra_status forward_f32(const dyra_layer *L, const float *X, int batch, int n, float *Y,
                        uint8_t *ws, const WsLayout &w, cudaStream_t s, Recorder &rec,
                        bool clear_status) {
  using namespace dyra;
  const int d = L->d, m = L->m, k = L->k, r = L->r, ldT = w.ldT;
  int *status = reinterpret_cast<int *>(ws);
  float *T = reinterpret_cast<float *>(ws + w.T);
  double *G = reinterpret_cast<double *>(ws + w.G);
  double *Gi = reinterpret_cast<double *>(ws + w.Ginv);
  float *C = reinterpret_cast<float *>(ws + w.C);
  float *Bm = reinterpret_cast<float *>(ws + w.B);
  float *R = reinterpret_cast<float *>(ws + w.R);
  const float *Wcat = static_cast<const float *>(L->w1);
  const float *V = static_cast<const float *>(L->v);
  const float *Wr = static_cast<const float *>(L->wres);
  const long long nT = (long long)n * ldT;
  if (clear_status) DY_CUDA(cudaMemsetAsync(ws, 0, 16, s));
  // T = X [U | P]
  DY_TIMED(rec, s, launch_sgemm(batch, n, ldT, d, X, (long long)n * d, d, 1, Wcat, 0, ldT, 1, T,
                                nT, ldT, 1, false, nullptr, s));
  // G = L^T L (fp64)
  DY_TIMED(rec, s, launch_gram_f64(T, batch, n, ldT, k, r, nT, G, s));
  // C = L^T X
  DY_TIMED(rec, s, launch_sgemm(batch, r, d, n, T + k, nT, 1, ldT, X, (long long)n * d, d, 1, C,
                                (long long)r * d, d, 1, false, nullptr, s));
  // B = C W_res
  DY_TIMED(rec, s, launch_sgemm(batch, r, m, d, C, (long long)r * d, d, 1, Wr, 0, m, 1, Bm,
                                (long long)r * m, m, 1, false, nullptr, s));
  // (G + lambda I)^-1
  DY_TIMED(rec, s, launch_inverse_f64(G, batch, r, L->ridge, L->solver == DYRA_SOLVE_NEWTON_SCHULZ,
                                      L->ns_iters, Gi, status, s));
  // R = G^-1 B
  DY_TIMED(rec, s, launch_apply_inverse(Gi, Bm, batch, r, m, R, s));
  // Y = (X U) V + b
  DY_TIMED(rec, s, launch_sgemm(batch, n, m, k, T, nT, ldT, 1, V, 0, m, 1, Y, (long long)n * m, m,
                                1, false, L->bias_d, s));
  // Y += L R
  DY_TIMED(rec, s, launch_sgemm(batch, n, m, r, T + k, nT, ldT, 1, R, (long long)r * m, m, 1, Y,
                                (long long)n * m, m, 1, true, nullptr, s));
  return DYRA_OK;
}

const char *const kNamesF32[] = {"f32_xproj", "f32_gram_f64", "f32_c", "f32_b",
                                 "f32_inverse_f64", "f32_apply_inverse", "f32_static_out",
                                 "f32_correction_out"};

// The kernels one forward launches, in order (the plan builders push them in this order).
std::vector<const char *> forward_kernel_names(const dyra_layer *L) {
  std::vector<const char *> v;
  if (L->dtype == DYRA_F32) {
    v.assign(std::begin(kNamesF32), std::end(kNamesF32));
    return v;
  }
  if (L->kind == DYRA_STATIC_MONARCH)
    v.insert(v.end(), {"monarch_bd1", "xproj_L", "monarch_permute"});
  else if (L->kind == DYRA_STATIC_BLAST)
    v.insert(v.end(), {"blast_stage1", "xproj_L"});
  else
    v.push_back("xproj_static_L");
  auto solve = [&]() {
    if (L->solver == DYRA_SOLVE_CHOLESKY)
      v.insert(v.end(), {"spd_invert", "spd_apply_c"});
    else
      v.insert(v.end(), {"ns_iterate", "ginv_c"});
  };
  auto r_update = [&]() {
    if (fused_gram_solve(L)) {
      v.push_back("cg_solve");
    } else {
      v.push_back("cg_c_gram");
      solve();
    }
    v.push_back("residual_product");
  };
  r_update();
  for (int hs = 2; hs < L->als_half; ++hs) {
    if (hs % 2 == 0) {
      v.insert(v.end(), {"als_gram_r", "als_q"});
      solve();
      v.push_back("als_l_update");
    } else {
      r_update();
    }
  }
  v.push_back("fused_output");
  return v;
}

int kernels_per_forward(const dyra_layer *L) { return (int)forward_kernel_names(L).size(); }

const char *kernel_name(const dyra_layer *L, int i) {
  const std::vector<const char *> v = forward_kernel_names(L);
  if (i < 0 || i >= (int)v.size()) return nullptr;
  return v[i];
}

dyra_status forward_impl(const dyra_layer *L, const void *X, int batch, int n, void *Y,
                         void *workspace, size_t ws_bytes, cudaStream_t s, Recorder &rec,
                         bool clear_status = true) {
  if (!L) return DYRA_ERR_INVALID_ARG;
  if (batch < 0 || n < 0) return DYRA_ERR_INVALID_ARG;
  if (batch == 0 || n == 0) return DYRA_OK;
  if (!X || !Y || !workspace) return DYRA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(X) & 15) || (reinterpret_cast<uintptr_t>(Y) & 15))
    return DYRA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return DYRA_ERR_WORKSPACE;
  const WsLayout w = layout_of(L, batch, n);
  if (ws_bytes < w.total) return DYRA_ERR_WORKSPACE;
  DeviceGuard guard(L->device);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  if (L->dtype == DYRA_F32)
    return forward_f32(L, static_cast<const float *>(X), batch, n, static_cast<float *>(Y), ws, w,
                       s, rec, clear_status);
  const std::array<uintptr_t, 5> key = {reinterpret_cast<uintptr_t>(X),
                                         reinterpret_cast<uintptr_t>(Y),
                                         reinterpret_cast<uintptr_t>(workspace), (uintptr_t)batch,
                                         (uintptr_t)n};
  std::lock_guard<std::mutex> lock(L->mu);
  std::shared_ptr<Plan> plan;
  for (auto &kv : L->plans)
    if (kv.first == key) plan = std::static_pointer_cast<Plan>(kv.second);
  if (!plan) {
    plan = std::make_shared<Plan>();
    dyra_status ps = plan_bf16(L, X, batch, n, Y, ws, w, *plan);
    if (ps != DYRA_OK) return ps;
    plan->clear = w.clear;
    if (plan->steps.size() != (size_t)kernels_per_forward(L)) {
      g_last_error = "internal: the launch plan does not match the kernel list";
      return DYRA_ERR_INVALID_ARG;
    }
    if (L->plans.size() >= 64) L->plans.erase(L->plans.begin());
    L->plans.emplace_back(key, plan);
  }
  return run_plan(L, *plan, ws, s, rec, clear_status);
}

// ------------------------------------------------------------------------ preparation

void to_bf16(const double *src, size_t count, std::vector<__nv_bfloat16> &dst) {
  dst.resize(count);
  for (size_t i = 0; i < count; ++i) dst[i] = __float2bfloat16_rn((float)src[i]);
}

template <typename T>
dyra_status upload(void **dptr, const std::vector<T> &host) {
  const size_t bytes = host.size() * sizeof(T);
  cudaError_t e = cudaMalloc(dptr, bytes ? bytes : 16);
  if (e != cudaSuccess) {
    g_last_error = std::string("cudaMalloc: ") + cudaGetErrorString(e);
    return DYRA_ERR_OOM;
  }
  if (bytes) DY_CUDA(cudaMemcpy(*dptr, host.data(), bytes, cudaMemcpyHostToDevice));
  return DYRA_OK;
}

void free_device(dyra_layer *L) {
  if (L->w1) cudaFree(L->w1);
  if (L->v) cudaFree(L->v);
  if (L->wres) cudaFree(L->wres);
  if (L->bd1) cudaFree(L->bd1);
  if (L->bd2) cudaFree(L->bd2);
  if (L->bias_d) cudaFree(L->bias_d);
  L->w1 = L->v = L->wres = L->bd1 = L->bd2 = nullptr;
  L->bias_d = nullptr;
}

// Monarch fit: each (a, c) block of W gets its leading singular triplet.
void fit_monarch(const std::vector<double> &W, int d, int m, int nb, std::vector<double> &B1,
                 std::vector<double> &B2, int threads) {
  const int bi = d / nb, bo = m / nb;
  B1.assign((size_t)nb * bi * nb, 0.0);
  B2.assign((size_t)nb * nb * bo, 0.0);
  struct Ctx {
    const double *W;
    int d, m, nb, bi, bo;
    double *B1, *B2;
  } ctx{W.data(), d, m, nb, bi, bo, B1.data(), B2.data()};
  dyra::fit::parallel_for(nb * nb, threads, &ctx, [](const void *vc, int t) {
    const Ctx &c = *static_cast<const Ctx *>(vc);
    const int a = t / c.nb, cc = t % c.nb;
    std::vector<double> blk((size_t)c.bi * c.bo);
    for (int i = 0; i < c.bi; ++i)
      for (int j = 0; j < c.bo; ++j)
        blk[(size_t)i * c.bo + j] = c.W[(size_t)(a * c.bi + i) * c.m + (size_t)cc * c.bo + j];
    std::vector<double> U((size_t)c.bi), S(1), Vt((size_t)c.bo);
    dyra::fit::top_svd(c.bi, c.bo, blk.data(), 1, U.data(), S.data(), Vt.data(), 1);
    const double root = std::sqrt(std::max(S[0], 0.0));
    for (int i = 0; i < c.bi; ++i) c.B1[((size_t)a * c.bi + i) * c.nb + cc] = root * U[i];
    for (int j = 0; j < c.bo; ++j) c.B2[((size_t)cc * c.nb + a) * c.bo + j] = root * Vt[j];
  });
}

void monarch_dense(const std::vector<double> &B1, const std::vector<double> &B2, int d, int m,
                   int nb, std::vector<double> &Wh) {
  const int bi = d / nb, bo = m / nb;
  Wh.assign((size_t)d * m, 0.0);
  for (int a = 0; a < nb; ++a)
    for (int i = 0; i < bi; ++i)
      for (int c = 0; c < nb; ++c) {
        const double u = B1[((size_t)a * bi + i) * nb + c];
        if (u == 0.0) continue;
        const double *v = &B2[((size_t)c * nb + a) * bo];
        double *row = &Wh[(size_t)(a * bi + i) * m + (size_t)c * bo];
        for (int j = 0; j < bo; ++j) row[j] = u * v[j];
      }
}

// BLAST with nb x nb blocks of rank t: U [nb][p][t], V [nb][q][t], S [nb][nb][t][t],
// block (i, j) = U_i S_ij V_j^T. Fit (alternating exact minimisations of ||W - W_hat||_F with
// orthonormal bases): U_i, V_j start as the top-t singular vectors of block row i / block
// column j; each sweep sets U_i to the top-t left singular vectors of [W_i1 V_1 .. W_i,nb V_nb]
// and then V_j to those of [W_1j^T U_1 .. W_nb,j^T U_nb]; finally S_ij = U_i^T W_ij V_j.
constexpr int kBlastSweeps = 10;

bool fit_blast(const std::vector<double> &W, int d, int m, int nb, int t, std::vector<double> &U,
               std::vector<double> &V, std::vector<double> &S, int threads) {
  const int p = d / nb, q = m / nb;
  U.assign((size_t)nb * p * t, 0.0);
  V.assign((size_t)nb * q * t, 0.0);
  S.assign((size_t)nb * nb * t * t, 0.0);
  auto block = [&](int i, int j, std::vector<double> &out) {   // W_ij [p x q]
    out.resize((size_t)p * q);
    for (int a = 0; a < p; ++a)
      std::memcpy(&out[(size_t)a * q], &W[(size_t)(i * p + a) * m + (size_t)j * q],
                  sizeof(double) * q);
  };
  std::vector<double> Uo, Sv, Vt, Wij, K, tmp;
  // left singular vectors of a rows x cols matrix into dst [rows x t]
  auto left = [&](int rows, int cols, const double *A, double *dst) {
    Uo.resize((size_t)rows * t);
    Sv.resize(t);
    Vt.resize((size_t)t * cols);
    if (!dyra::fit::top_svd(rows, cols, A, t, Uo.data(), Sv.data(), Vt.data(), threads)) return false;
    std::copy(Uo.begin(), Uo.end(), dst);
    return true;
  };
  for (int i = 0; i < nb; ++i)
    if (!left(p, m, &W[(size_t)i * p * m], &U[(size_t)i * p * t])) return false;
  for (int j = 0; j < nb; ++j) {   // column block j transposed: [q x d]
    K.resize((size_t)q * d);
    for (int c = 0; c < q; ++c)
      for (int a = 0; a < d; ++a) K[(size_t)c * d + a] = W[(size_t)a * m + (size_t)j * q + c];
    if (!left(q, d, K.data(), &V[(size_t)j * q * t])) return false;
  }
  for (int sw = 0; sw < kBlastSweeps; ++sw) {
    for (int i = 0; i < nb; ++i) {   // K = [W_i1 V_1 .. W_i,nb V_nb], p x (nb t)
      K.assign((size_t)p * nb * t, 0.0);
      for (int j = 0; j < nb; ++j) {
        block(i, j, Wij);
        tmp.resize((size_t)p * t);
        dyra::fit::gemm(p, t, q, Wij.data(), false, &V[(size_t)j * q * t], false, tmp.data(), 1);
        for (int a = 0; a < p; ++a)
          std::memcpy(&K[(size_t)a * nb * t + (size_t)j * t], &tmp[(size_t)a * t], sizeof(double) * t);
      }
      if (!left(p, nb * t, K.data(), &U[(size_t)i * p * t])) return false;
    }
    for (int j = 0; j < nb; ++j) {   // K = [W_1j^T U_1 .. W_nb,j^T U_nb], q x (nb t)
      K.assign((size_t)q * nb * t, 0.0);
      for (int i = 0; i < nb; ++i) {
        block(i, j, Wij);
        tmp.resize((size_t)q * t);
        dyra::fit::gemm(q, t, p, Wij.data(), true, &U[(size_t)i * p * t], false, tmp.data(), 1);
        for (int c = 0; c < q; ++c)
          std::memcpy(&K[(size_t)c * nb * t + (size_t)i * t], &tmp[(size_t)c * t], sizeof(double) * t);
      }
      if (!left(q, nb * t, K.data(), &V[(size_t)j * q * t])) return false;
    }
  }
  for (int i = 0; i < nb; ++i)
    for (int j = 0; j < nb; ++j) {   // S_ij = U_i^T W_ij V_j
      block(i, j, Wij);
      tmp.resize((size_t)p * t);
      dyra::fit::gemm(p, t, q, Wij.data(), false, &V[(size_t)j * q * t], false, tmp.data(), 1);
      dyra::fit::gemm(t, t, p, &U[(size_t)i * p * t], true, tmp.data(), false,
                      &S[((size_t)i * nb + j) * t * t], 1);
    }
  return true;
}

void blast_dense(const std::vector<double> &U, const std::vector<double> &V,
                 const std::vector<double> &S, int d, int m, int nb, int t,
                 std::vector<double> &Wh) {
  const int p = d / nb, q = m / nb;
  Wh.assign((size_t)d * m, 0.0);
  std::vector<double> US((size_t)p * t), blk((size_t)p * q);
  for (int i = 0; i < nb; ++i)
    for (int j = 0; j < nb; ++j) {
      dyra::fit::gemm(p, t, t, &U[(size_t)i * p * t], false, &S[((size_t)i * nb + j) * t * t],
                      false, US.data(), 1);
      dyra::fit::gemm(p, q, t, US.data(), false, &V[(size_t)j * q * t], true, blk.data(), 1);
      for (int a = 0; a < p; ++a)
        std::memcpy(&Wh[(size_t)(i * p + a) * m + (size_t)j * q], &blk[(size_t)a * q],
                    sizeof(double) * q);
    }
}

// Argument checks shared by dyra_fit and dyra_prepare.
dyra_status validate(const dyra_prepare_args *a, dyra_solver *solver_out, int *ns_out,
                     bool device_checks) {
  if (!a || !a->W) return DYRA_ERR_INVALID_ARG;
  const int d = a->d, m = a->m, k = a->k, r = a->r;
  if (d <= 0 || m <= 0 || r <= 0 || k < 0) return DYRA_ERR_INVALID_ARG;
  if ((a->F1 == nullptr) != (a->F2 == nullptr)) return DYRA_ERR_INVALID_ARG;
  if (!(a->ridge >= 0.0) || !std::isfinite(a->ridge)) return DYRA_ERR_INVALID_ARG;
  if (a->input_aware != DYRA_INPUT_AWARE_NONE) {
    if (a->input_aware != DYRA_INPUT_AWARE_DIAG && a->input_aware != DYRA_INPUT_AWARE_CHOLESKY)
      return DYRA_ERR_INVALID_ARG;
    if (a->kind != DYRA_STATIC_LOWRANK || (!a->F1 && (!a->calib || a->n_calib <= 0)))
      return DYRA_ERR_INVALID_ARG;
  }
  if (a->dtype != DYRA_F32 && a->dtype != DYRA_BF16) return DYRA_ERR_INVALID_ARG;
  if (a->activation != DYRA_ACT_NONE && a->activation != DYRA_ACT_GELU) return DYRA_ERR_INVALID_ARG;
  if (a->als_t != 0.0) {   // t in {1, 1.5, 2, ..., 8}
    const double h = 2.0 * a->als_t;
    if (!(a->als_t >= 1.0 && a->als_t <= 8.0) || h != std::floor(h)) return DYRA_ERR_INVALID_ARG;
  }
  if (a->kind == DYRA_STATIC_LOWRANK) {
    if (k >= std::min(d, m) || r > std::min(d, m)) return DYRA_ERR_INVALID_ARG;
    if (!a->R0 && k + r > std::min(d, m)) return DYRA_ERR_INVALID_ARG;
  } else if (a->kind == DYRA_STATIC_MONARCH) {
    if (k <= 0 || d % k || m % k) return DYRA_ERR_INVALID_ARG;
    if (r > std::min(d, m)) return DYRA_ERR_INVALID_ARG;
  } else if (a->kind == DYRA_STATIC_BLAST) {
    if (k <= 0 || d % k || m % k) return DYRA_ERR_INVALID_ARG;
    if (a->blast_t < 1 || a->blast_t > std::min(d / k, m / k)) return DYRA_ERR_INVALID_ARG;
    if (r > std::min(d, m) || (a->F1 && !a->F3)) return DYRA_ERR_INVALID_ARG;
  } else {
    return DYRA_ERR_INVALID_ARG;
  }
  dyra_solver solver = a->solver;
  if (solver == DYRA_SOLVE_AUTO) solver = r <= 64 ? DYRA_SOLVE_CHOLESKY : DYRA_SOLVE_NEWTON_SCHULZ;
  if (solver != DYRA_SOLVE_CHOLESKY && solver != DYRA_SOLVE_NEWTON_SCHULZ) return DYRA_ERR_INVALID_ARG;
  *solver_out = solver;
  *ns_out = a->ns_iters > 0 ? a->ns_iters : 8;
  if (!device_checks) return DYRA_OK;
  if (a->dtype == DYRA_F32) {
    if (r > 64) return DYRA_ERR_UNSUPPORTED;
    if (a->kind == DYRA_STATIC_BLAST) return DYRA_ERR_UNSUPPORTED;
    if (a->activation != DYRA_ACT_NONE) return DYRA_ERR_UNSUPPORTED;
    if (a->als_t != 0.0 && a->als_t != 1.0) return DYRA_ERR_UNSUPPORTED;
    if (a->kind != DYRA_STATIC_LOWRANK) return DYRA_ERR_UNSUPPORTED;
  } else {
    if (r > 256 || r % 8 || d % 8 || m % 8) return DYRA_ERR_UNSUPPORTED;
    if (solver == DYRA_SOLVE_CHOLESKY && r > 64) return DYRA_ERR_UNSUPPORTED;
    if (a->kind == DYRA_STATIC_MONARCH && !dyra::monarch_supported(d, m, k, r))
      return DYRA_ERR_UNSUPPORTED;
    if (a->kind == DYRA_STATIC_BLAST &&
        ((d / k) % 64 || a->blast_t % 32 || a->blast_t > 256))
      return DYRA_ERR_UNSUPPORTED;
  }
  return DYRA_OK;
}

// Input-aware truncated SVD: W_hat = S^-T TSVD_k(S^T W) with S from the calibration rows
// (diag: channel rms; cholesky: lower Cholesky factor of calib^T calib / n_calib). Stores the
// factors F1 = S^-T U_k sqrt(S_k), F2 = sqrt(S_k) V_k^T.
dyra_status fit_input_aware(const dyra_prepare_args *a, const std::vector<double> &W,
                            dyra_layer *L) {
  const int d = a->d, m = a->m, k = a->k, N = a->n_calib, th = a->fit_threads;
  std::vector<double> A(W);   // S^T W
  std::vector<double> Lc;     // Cholesky factor (cholesky mode)
  std::vector<double> s;      // channel rms (diag mode)
  if (a->input_aware == DYRA_INPUT_AWARE_DIAG) {
    s.assign(d, 0.0);
    for (int n = 0; n < N; ++n)
      for (int i = 0; i < d; ++i) s[i] += a->calib[(size_t)n * d + i] * a->calib[(size_t)n * d + i];
    for (int i = 0; i < d; ++i) {
      s[i] = std::sqrt(s[i] / N);
      if (!(s[i] > 0.0)) {
        g_last_error = "input-aware fit: an input channel is zero on every calibration row";
        return DYRA_ERR_INVALID_ARG;
      }
      for (int j = 0; j < m; ++j) A[(size_t)i * m + j] *= s[i];
    }
  } else {
    Lc.assign((size_t)d * d, 0.0);
    dyra::fit::gemm(d, d, N, a->calib, true, a->calib, false, Lc.data(), th);   // calib^T calib
    for (double &x : Lc) x /= N;
    if (!dyra::fit::cholesky(d, Lc.data())) {
      g_last_error = "input-aware fit: the calibration covariance is not positive definite";
      return DYRA_ERR_INVALID_ARG;
    }
    for (int i = 0; i < d; ++i)   // keep the lower triangle only
      for (int j = i + 1; j < d; ++j) Lc[(size_t)i * d + j] = 0.0;
    dyra::fit::gemm(d, m, d, Lc.data(), true, W.data(), false, A.data(), th);   // L^T W
  }
  std::vector<double> U((size_t)d * k), S(k), Vt((size_t)k * m);
  if (k > 0 && !dyra::fit::top_svd(d, m, A.data(), k, U.data(), S.data(), Vt.data(), th)) {
    g_last_error = "eigen-decomposition did not converge";
    return DYRA_ERR_INVALID_ARG;
  }
  L->F1.assign((size_t)d * k, 0.0);
  L->F2.assign((size_t)k * m, 0.0);
  for (int j = 0; j < k; ++j) {
    const double root = std::sqrt(S[j]);
    for (int i = 0; i < d; ++i) L->F1[(size_t)i * k + j] = U[(size_t)i * k + j] * root;
    for (int i = 0; i < m; ++i) L->F2[(size_t)j * m + i] = Vt[(size_t)j * m + i] * root;
  }
  if (a->input_aware == DYRA_INPUT_AWARE_DIAG) {
    for (int i = 0; i < d; ++i)
      for (int j = 0; j < k; ++j) L->F1[(size_t)i * k + j] /= s[i];
  } else if (k > 0) {
    dyra::fit::lower_transpose_solve(d, Lc.data(), L->F1.data(), k);   // S^-T (U_k sqrt(S_k))
  }
  return DYRA_OK;
}

// Host fp64 offline step: static fit, W_res, R0, P (no device needed).
dyra_status fit_host(const dyra_prepare_args *a, dyra_layer *L) {
  const int d = a->d, m = a->m, k = a->k, r = a->r;
  const int th = a->fit_threads;
  const std::vector<double> W(a->W, a->W + (size_t)d * m);
  L->bias.assign(m, 0.0);
  if (a->b) std::copy(a->b, a->b + m, L->bias.begin());
  if (a->kind == DYRA_STATIC_LOWRANK) {
    if (a->F1) {
      L->F1.assign(a->F1, a->F1 + (size_t)d * k);
      L->F2.assign(a->F2, a->F2 + (size_t)k * m);
    } else if (a->input_aware != DYRA_INPUT_AWARE_NONE) {
      const dyra_status st = fit_input_aware(a, W, L);
      if (st != DYRA_OK) return st;
    } else {
      const int cnt = k + (a->R0 ? 0 : r);
      std::vector<double> U((size_t)d * cnt), S(cnt), Vt((size_t)cnt * m);
      if (!dyra::fit::top_svd(d, m, W.data(), cnt, U.data(), S.data(), Vt.data(), th)) {
        g_last_error = "eigen-decomposition did not converge";
        return DYRA_ERR_INVALID_ARG;
      }
      L->F1.assign((size_t)d * k, 0.0);
      L->F2.assign((size_t)k * m, 0.0);
      for (int j = 0; j < k; ++j) {
        const double root = std::sqrt(S[j]);
        for (int i = 0; i < d; ++i) L->F1[(size_t)i * k + j] = U[(size_t)i * cnt + j] * root;
        for (int i = 0; i < m; ++i) L->F2[(size_t)j * m + i] = Vt[(size_t)j * m + i] * root;
      }
      // for a truncated-SVD W_hat, the residual's top right singular vectors are W's
      // singular vectors k+1..k+r
      if (!a->R0) L->R0.assign(Vt.begin() + (size_t)k * m, Vt.begin() + (size_t)(k + r) * m);
    }
    L->W_hat.assign((size_t)d * m, 0.0);
    if (k > 0) dyra::fit::gemm(d, m, k, L->F1.data(), false, L->F2.data(), false, L->W_hat.data(), th);
  } else if (a->kind == DYRA_STATIC_BLAST) {
    const int nb = k, t = a->blast_t;
    if (a->F1) {
      L->F1.assign(a->F1, a->F1 + (size_t)d * t);
      L->F2.assign(a->F2, a->F2 + (size_t)m * t);
      L->F3.assign(a->F3, a->F3 + (size_t)nb * nb * t * t);
    } else if (!fit_blast(W, d, m, nb, t, L->F1, L->F2, L->F3, th)) {
      g_last_error = "eigen-decomposition did not converge";
      return DYRA_ERR_INVALID_ARG;
    }
    blast_dense(L->F1, L->F2, L->F3, d, m, nb, t, L->W_hat);
  } else {
    const int nb = k;
    if (a->F1) {
      L->F1.assign(a->F1, a->F1 + (size_t)d * nb);
      L->F2.assign(a->F2, a->F2 + (size_t)nb * m);
    } else {
      fit_monarch(W, d, m, nb, L->F1, L->F2, th);
    }
    monarch_dense(L->F1, L->F2, d, m, nb, L->W_hat);
  }
  L->W_res.resize((size_t)d * m);
  for (size_t i = 0; i < L->W_res.size(); ++i) L->W_res[i] = W[i] - L->W_hat[i];
  if (a->R0) {
    L->R0.assign(a->R0, a->R0 + (size_t)r * m);
  } else if (L->R0.empty()) {
    std::vector<double> U((size_t)d * r), S(r), Vt((size_t)r * m);
    if (!dyra::fit::top_svd(d, m, L->W_res.data(), r, U.data(), S.data(), Vt.data(), th)) {
      g_last_error = "eigen-decomposition did not converge";
      return DYRA_ERR_INVALID_ARG;
    }
    L->R0 = Vt;
  }
  // P = W_res R0^T (R0 R0^T)^-1
  std::vector<double> gram((size_t)r * r), WR((size_t)r * d);
  dyra::fit::gemm(r, r, m, L->R0.data(), false, L->R0.data(), true, gram.data(), th);
  if (!dyra::fit::cholesky(r, gram.data())) {
    g_last_error = "R0 R0^T is not positive definite (R0 rank deficient)";
    return DYRA_ERR_INVALID_ARG;
  }
  dyra::fit::gemm(r, d, m, L->R0.data(), false, L->W_res.data(), true, WR.data(), th);   // R0 W_res^T
  dyra::fit::cholesky_solve(r, gram.data(), WR.data(), d);
  L->P.resize((size_t)d * r);
  for (int i = 0; i < d; ++i)
    for (int j = 0; j < r; ++j) L->P[(size_t)i * r + j] = WR[(size_t)j * d + i];
  return DYRA_OK;
}

dyra_layer *new_layer(const dyra_prepare_args *a, dyra_solver solver, int ns_iters) {
  dyra_layer *L = new (std::nothrow) dyra_layer();
  if (!L) return nullptr;
  L->d = a->d; L->m = a->m; L->k = a->k; L->r = a->r;
  L->kp = (a->kind == DYRA_STATIC_LOWRANK) ? roundup(a->k, 64)
          : (a->kind == DYRA_STATIC_BLAST) ? roundup(a->k * a->blast_t, 64) : a->d;
  L->blast_t = a->kind == DYRA_STATIC_BLAST ? a->blast_t : 0;
  L->kind = a->kind; L->dtype = a->dtype; L->solver = solver; L->ns_iters = ns_iters;
  L->ridge = a->ridge; L->device = a->device; L->activation = a->activation;
  L->als_half = a->als_t > 0.0 ? (int)std::lround(2.0 * a->als_t) : 2;
  return L;
}

dyra_status upload_layer(const dyra_prepare_args *a, dyra_layer *L) {
  const int d = L->d, m = L->m, k = L->k, r = L->r;
  dyra_status st = DYRA_OK;
  // the bias in fp32, zero-padded by 256 columns: an output epilogue reads the bias of its
  // whole last tile, which may reach past column m
  std::vector<float> bias32(L->bias.begin(), L->bias.end());
  bias32.resize((size_t)m + 256, 0.f);
  if (a->dtype == DYRA_BF16 && L->kind == DYRA_STATIC_MONARCH) {
    const int nb = k, T0 = 256;
    std::vector<double> pt((size_t)r * d), b1((size_t)d * T0, 0.0), b2((size_t)m * T0, 0.0),
        wrt((size_t)m * d);
    for (int j = 0; j < r; ++j)
      for (int i = 0; i < d; ++i) pt[(size_t)j * d + i] = L->P[(size_t)i * r + j];
    // Z[:, a*nb + c] = sum_i X[:, a*nb + i] B1[a][i][c]
    for (int n = 0; n < d; ++n) {
      const int a_ = n / nb, c = n % nb, n0 = n / T0 * T0;
      for (int i = 0; i < nb; ++i)
        b1[(size_t)n * T0 + (a_ * nb + i - n0)] = L->F1[((size_t)a_ * nb + i) * nb + c];
    }
    // Y[:, c*nb + j] = sum_a Zp[:, c*nb + a] B2[c][a][j]
    for (int o = 0; o < m; ++o) {
      const int c = o / nb, j = o % nb, n0 = o / T0 * T0;
      for (int a_ = 0; a_ < nb; ++a_)
        b2[(size_t)o * T0 + (c * nb + a_ - n0)] = L->F2[((size_t)c * nb + a_) * nb + j];
    }
    for (int i = 0; i < d; ++i)
      for (int j = 0; j < m; ++j) wrt[(size_t)j * d + i] = L->W_res[(size_t)i * m + j];
    std::vector<__nv_bfloat16> h;
    to_bf16(pt.data(), pt.size(), h);
    if (st == DYRA_OK) st = upload(&L->w1, h);
    to_bf16(b1.data(), b1.size(), h);
    if (st == DYRA_OK) st = upload(&L->bd1, h);
    to_bf16(b2.data(), b2.size(), h);
    if (st == DYRA_OK) st = upload(&L->bd2, h);
    to_bf16(wrt.data(), wrt.size(), h);
    if (st == DYRA_OK) st = upload(&L->wres, h);
  } else if (a->dtype == DYRA_BF16 && L->kind == DYRA_STATIC_BLAST) {
    // w1 = P^T [r, d]; bd1 = the stage-1 factor [nb t, p]: row i t + x is column x of U_i;
    // v = the output GEMM's static factor [m, kp]: v[j q + c][i t + x] = (S_ij V_j^T)[x][c]
    const int nb = k, t = L->blast_t, pb = d / nb, qb = m / nb, kp = L->kp;
    std::vector<double> pt((size_t)r * d), b1((size_t)nb * t * pb), vt((size_t)m * kp, 0.0),
        wrt((size_t)m * d);
    for (int j = 0; j < r; ++j)
      for (int i = 0; i < d; ++i) pt[(size_t)j * d + i] = L->P[(size_t)i * r + j];
    for (int i = 0; i < nb; ++i)
      for (int x = 0; x < t; ++x)
        for (int a_ = 0; a_ < pb; ++a_)
          b1[((size_t)i * t + x) * pb + a_] = L->F1[((size_t)i * pb + a_) * t + x];
    for (int i = 0; i < nb; ++i)
      for (int j = 0; j < nb; ++j) {
        const double *S = &L->F3[((size_t)i * nb + j) * t * t];
        for (int c = 0; c < qb; ++c) {
          const double *vr = &L->F2[((size_t)j * qb + c) * t];
          for (int x = 0; x < t; ++x) {
            double acc = 0.0;
            for (int y = 0; y < t; ++y) acc += S[(size_t)x * t + y] * vr[y];
            vt[((size_t)j * qb + c) * kp + (size_t)i * t + x] = acc;
          }
        }
      }
    for (int i = 0; i < d; ++i)
      for (int j = 0; j < m; ++j) wrt[(size_t)j * d + i] = L->W_res[(size_t)i * m + j];
    std::vector<__nv_bfloat16> h;
    to_bf16(pt.data(), pt.size(), h);
    if (st == DYRA_OK) st = upload(&L->w1, h);
    to_bf16(b1.data(), b1.size(), h);
    if (st == DYRA_OK) st = upload(&L->bd1, h);
    to_bf16(vt.data(), vt.size(), h);
    if (st == DYRA_OK) st = upload(&L->v, h);
    to_bf16(wrt.data(), wrt.size(), h);
    if (st == DYRA_OK) st = upload(&L->wres, h);
  } else if (a->dtype == DYRA_BF16) {
    const int kp = L->kp, N1 = kp + r;
    std::vector<double> w1((size_t)N1 * d, 0.0), vt((size_t)m * std::max(kp, 1), 0.0),
        wrt((size_t)m * d);
    for (int j = 0; j < k; ++j)
      for (int i = 0; i < d; ++i) w1[(size_t)j * d + i] = L->F1[(size_t)i * k + j];
    for (int j = 0; j < r; ++j)
      for (int i = 0; i < d; ++i) w1[(size_t)(kp + j) * d + i] = L->P[(size_t)i * r + j];
    for (int i = 0; i < k; ++i)
      for (int j = 0; j < m; ++j) vt[(size_t)j * kp + i] = L->F2[(size_t)i * m + j];
    for (int i = 0; i < d; ++i)
      for (int j = 0; j < m; ++j) wrt[(size_t)j * d + i] = L->W_res[(size_t)i * m + j];
    std::vector<__nv_bfloat16> h;
    to_bf16(w1.data(), w1.size(), h);
    if (st == DYRA_OK) st = upload(&L->w1, h);
    to_bf16(vt.data(), vt.size(), h);
    if (st == DYRA_OK) st = upload(&L->v, h);
    to_bf16(wrt.data(), wrt.size(), h);
    if (st == DYRA_OK) st = upload(&L->wres, h);
  } else {
    const int N1 = k + r;
    std::vector<float> wc((size_t)d * N1), vv((size_t)std::max(k, 1) * m, 0.f), wr((size_t)d * m);
    for (int i = 0; i < d; ++i) {
      for (int j = 0; j < k; ++j) wc[(size_t)i * N1 + j] = (float)L->F1[(size_t)i * k + j];
      for (int j = 0; j < r; ++j) wc[(size_t)i * N1 + k + j] = (float)L->P[(size_t)i * r + j];
    }
    for (size_t i = 0; i < L->F2.size(); ++i) vv[i] = (float)L->F2[i];
    for (size_t i = 0; i < wr.size(); ++i) wr[i] = (float)L->W_res[i];
    if (st == DYRA_OK) st = upload(&L->w1, wc);
    if (st == DYRA_OK) st = upload(&L->v, vv);
    if (st == DYRA_OK) st = upload(&L->wres, wr);
  }
  if (st == DYRA_OK) {
    void *bp = nullptr;
    st = upload(&bp, bias32);
    L->bias_d = static_cast<float *>(bp);
  }
  return st;
}

dyra_status prepare_impl(const dyra_prepare_args *a, dyra_layer **out) {
  if (!out) return DYRA_ERR_INVALID_ARG;
  *out = nullptr;
  dyra_solver solver;
  int ns_iters;
  dyra_status vs = validate(a, &solver, &ns_iters, true);
  if (vs != DYRA_OK) return vs;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || a->device < 0 || a->device >= ndev)
    return DYRA_ERR_NO_DEVICE;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, a->device) != cudaSuccess) return DYRA_ERR_NO_DEVICE;
  if (prop.major != 10 || prop.minor != 3) {
    g_last_error = "device is not sm_103";
    return DYRA_ERR_NO_DEVICE;
  }
  dyra_layer *L = new_layer(a, solver, ns_iters);
  if (!L) return DYRA_ERR_OOM;
  dyra_status st = fit_host(a, L);
  if (st == DYRA_OK) {
    DeviceGuard guard(L->device);
    st = upload_layer(a, L);
    if (st != DYRA_OK) free_device(L);
  }
  if (st != DYRA_OK) {
    delete L;
    return st;
  }
  *out = L;
  return DYRA_OK;
}

}  // namespace

// ------------------------------------------------------------------------ static scratch
//
// Device scratch for dyra_linear_forward_static: a fixed array in the library's own device
// image, so that entry point needs no allocation. Host code may not use the symbol as a
// device address (it names a host-side stand-in); the device address is queried once per
// device with cudaGetSymbolAddress while that device is current.
static __device__ __align__(256) unsigned char g_static_scratch[DYRA_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void *g_static_ptr[kMaxDevices] = {};
void *g_static_ctx[kMaxDevices] = {};   // the context g_static_ptr[device] belongs to

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);

// The current CUDA context of the calling thread (the device's primary context once the
// runtime has used it), or nullptr if the driver entry point is unavailable.
void *current_context() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
  });
  CUcontext c = nullptr;
  if (fn && fn(&c) == CUDA_SUCCESS) return c;
  return nullptr;
}

// Device address of g_static_scratch on the current device. Looked up on the first call on a
// device and again whenever the device's context has changed since (a cudaDeviceReset
// destroys the primary context and the module image that holds the array).
dyra_status static_scratch(int device, void **out) {
  if (device < 0 || device >= kMaxDevices) return DYRA_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(g_static_mu);
  // cudaSetDevice (the caller's DeviceGuard) has made the device's primary context current
  void *ptr = g_static_ptr[device];
  void *ctx = current_context();
  if (!ptr || !ctx || ctx != g_static_ctx[device]) {
    ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess || !ptr) return cuda_fail(e, "cudaGetSymbolAddress(g_static_scratch)");
    g_static_ptr[device] = ptr;
    g_static_ctx[device] = current_context();
  }
  *out = g_static_ptr[device];
  return DYRA_OK;
}

}  // namespace

// ============================================================================ C ABI

extern "C" {

dyra_status dyra_prepare(const dyra_prepare_args *args, dyra_layer **out) {
  try {
    return prepare_impl(args, out);
  } catch (const std::bad_alloc &) {
    return DYRA_ERR_OOM;
  } catch (...) {
    g_last_error = "unexpected host exception in dyra_prepare";
    return DYRA_ERR_INVALID_ARG;
  }
}

dyra_status dyra_fit(const dyra_prepare_args *args, double *W_hat, double *W_res, double *P,
                     double *R0, double *F1, double *F2) {
  try {
    dyra_solver solver;
    int ns_iters;
    dyra_status vs = validate(args, &solver, &ns_iters, false);
    if (vs != DYRA_OK) return vs;
    std::unique_ptr<dyra_layer> L(new_layer(args, solver, ns_iters));
    if (!L) return DYRA_ERR_OOM;
    dyra_status fs = fit_host(args, L.get());
    if (fs == DYRA_OK) {
      if (W_hat) std::copy(L->W_hat.begin(), L->W_hat.end(), W_hat);
      if (W_res) std::copy(L->W_res.begin(), L->W_res.end(), W_res);
      if (P) std::copy(L->P.begin(), L->P.end(), P);
      if (R0) std::copy(L->R0.begin(), L->R0.end(), R0);
      if (F1) std::copy(L->F1.begin(), L->F1.end(), F1);
      if (F2) std::copy(L->F2.begin(), L->F2.end(), F2);
    }
    return fs;
  } catch (const std::bad_alloc &) {
    return DYRA_ERR_OOM;
  } catch (...) {
    g_last_error = "unexpected host exception in dyra_fit";
    return DYRA_ERR_INVALID_ARG;
  }
}

void dyra_layer_destroy(dyra_layer *layer) {
  if (!layer) return;
  {
    DeviceGuard guard(layer->device);
    cudaDeviceSynchronize();   // no forward of this layer may still read its weights
    free_device(layer);
    for (cudaEvent_t e : layer->host_ev) cudaEventDestroy(e);
    if (layer->copy_in) cudaStreamDestroy(layer->copy_in);
    if (layer->copy_out) cudaStreamDestroy(layer->copy_out);
  }
  delete layer;
}

dyra_status dyra_layer_info(const dyra_layer *L, dyra_layer_desc *out) {
  if (!L || !out) return DYRA_ERR_INVALID_ARG;
  out->d = L->d; out->m = L->m; out->k = L->k; out->r = L->r;
  out->kind = L->kind; out->dtype = L->dtype; out->solver = L->solver;
  out->ns_iters = L->ns_iters; out->ridge = L->ridge; out->device = L->device;
  out->kernels_per_forward = kernels_per_forward(L);
  out->activation = L->activation;
  out->als_t = 0.5 * L->als_half;
  return DYRA_OK;
}

dyra_status dyra_export(const dyra_layer *L, double *W_hat, double *W_res, double *P, double *R0) {
  if (!L) return DYRA_ERR_INVALID_ARG;
  if (W_hat) std::copy(L->W_hat.begin(), L->W_hat.end(), W_hat);
  if (W_res) std::copy(L->W_res.begin(), L->W_res.end(), W_res);
  if (P) std::copy(L->P.begin(), L->P.end(), P);
  if (R0) std::copy(L->R0.begin(), L->R0.end(), R0);
  return DYRA_OK;
}

dyra_status dyra_export_factors(const dyra_layer *L, double *F1, double *F2) {
  if (!L) return DYRA_ERR_INVALID_ARG;
  if (F1) std::copy(L->F1.begin(), L->F1.end(), F1);
  if (F2) std::copy(L->F2.begin(), L->F2.end(), F2);
  return DYRA_OK;
}

dyra_status dyra_workspace_size(const dyra_layer *L, int batch, int n, size_t *bytes) {
  if (!L || !bytes || batch < 0 || n < 0) return DYRA_ERR_INVALID_ARG;
  *bytes = layout_of(L, batch, n).total;
  return DYRA_OK;
}

dyra_status dyra_linear_forward(const dyra_layer *L, const void *X, int batch, int n, void *Y,
                                void *workspace, size_t workspace_bytes, cudaStream_t stream) {
  Recorder rec;
  return forward_impl(L, X, batch, n, Y, workspace, workspace_bytes, stream, rec);
}

dyra_status dyra_linear_forward_profiled(const dyra_layer *L, const void *X, int batch, int n,
                                         void *Y, void *workspace, size_t workspace_bytes,
                                         cudaStream_t stream, cudaEvent_t *events, int max_events,
                                         int *recorded) {
  if (!L || !events || max_events < 2 * kernels_per_forward(L)) return DYRA_ERR_INVALID_ARG;
  Recorder rec;
  rec.ev = events;
  rec.max = max_events;
  dyra_status st = forward_impl(L, X, batch, n, Y, workspace, workspace_bytes, stream, rec);
  if (recorded) *recorded = rec.count;
  return st;
}

dyra_status dyra_mlp_forward(const dyra_layer *fc1, const dyra_layer *fc2, const void *X,
                             int batch, int n, void *H, void *Y, void *workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
  if (!fc1 || !fc2 || batch < 0 || n < 0) return DYRA_ERR_INVALID_ARG;
  if (fc1->m != fc2->d || fc1->dtype != fc2->dtype || fc1->device != fc2->device)
    return DYRA_ERR_INVALID_ARG;
  if (batch == 0 || n == 0) return DYRA_OK;
  if (!X || !H || !Y || !workspace) return DYRA_ERR_INVALID_ARG;
  const size_t need = std::max(layout_of(fc1, batch, n).total, layout_of(fc2, batch, n).total);
  if (workspace_bytes < need) return DYRA_ERR_WORKSPACE;
  Recorder rec;
  dyra_status st = forward_impl(fc1, X, batch, n, H, workspace, workspace_bytes, stream, rec);
  if (st != DYRA_OK) return st;
  // the second layer keeps the status words the first one counted into
  return forward_impl(fc2, H, batch, n, Y, workspace, workspace_bytes, stream, rec, false);
}

dyra_status dyra_linear_forward_host(const dyra_layer *L, const void *X_host, int batch, int n,
                                     void *Y_host, void *X_dev, void *Y_dev, void *workspace,
                                     size_t workspace_bytes, cudaStream_t stream) {
  if (!L || batch < 0 || n < 0) return DYRA_ERR_INVALID_ARG;
  if (batch == 0 || n == 0) return DYRA_OK;
  if (!X_host || !Y_host || !X_dev || !Y_dev || !workspace) return DYRA_ERR_INVALID_ARG;
  const size_t eb = L->dtype == DYRA_F32 ? 4 : 2;
  const size_t xb = (size_t)batch * n * L->d * eb, yb = (size_t)batch * n * L->m * eb;
  if (workspace_bytes < layout_of(L, batch, n).total) return DYRA_ERR_WORKSPACE;
  DeviceGuard guard(L->device);
  Recorder rec;
  // groups of whole samples, each at least 8 MB of X and Y, at most 8 of them
  const int groups = (int)std::min<size_t>({(size_t)batch, 8, std::max<size_t>(1, (xb + yb) >> 23)});
  if (groups <= 1) {
    DY_CUDA(cudaMemcpyAsync(X_dev, X_host, xb, cudaMemcpyHostToDevice, stream));
    dyra_status st = forward_impl(L, X_dev, batch, n, Y_dev, workspace, workspace_bytes, stream, rec);
    if (st != DYRA_OK) return st;
    DY_CUDA(cudaMemcpyAsync(Y_host, Y_dev, yb, cudaMemcpyDeviceToHost, stream));
    return DYRA_OK;
  }
  std::lock_guard<std::mutex> lock(L->host_mu);
  if (!L->copy_in) DY_CUDA(cudaStreamCreateWithFlags(&L->copy_in, cudaStreamNonBlocking));
  if (!L->copy_out) DY_CUDA(cudaStreamCreateWithFlags(&L->copy_out, cudaStreamNonBlocking));
  const size_t need = 2 + 2 * (size_t)groups;
  while (L->host_ev.size() < need) {
    cudaEvent_t e;
    DY_CUDA(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    L->host_ev.push_back(e);
  }
  cudaEvent_t *ev = L->host_ev.data();
  // the copies start after the work already on `stream` (earlier users of X_dev / Y_dev)
  DY_CUDA(cudaEventRecord(ev[0], stream));
  DY_CUDA(cudaStreamWaitEvent(L->copy_in, ev[0], 0));
  DY_CUDA(cudaStreamWaitEvent(L->copy_out, ev[0], 0));
  DY_CUDA(cudaMemsetAsync(workspace, 0, 16, stream));   // status words, counted over all groups
  const size_t xs = xb / (size_t)batch, ys = yb / (size_t)batch;
  for (int gi = 0; gi < groups; ++gi) {
    const int b0 = (int)((long long)batch * gi / groups), b1 = (int)((long long)batch * (gi + 1) / groups);
    const size_t xo = xs * (size_t)b0, yo = ys * (size_t)b0;
    const size_t xn = xs * (size_t)(b1 - b0), yn = ys * (size_t)(b1 - b0);
    cudaEvent_t in_done = ev[2 + 2 * gi], fwd_done = ev[3 + 2 * gi];
    DY_CUDA(cudaMemcpyAsync(static_cast<uint8_t *>(X_dev) + xo,
                            static_cast<const uint8_t *>(X_host) + xo, xn, cudaMemcpyHostToDevice,
                            L->copy_in));
    DY_CUDA(cudaEventRecord(in_done, L->copy_in));
    DY_CUDA(cudaStreamWaitEvent(stream, in_done, 0));
    dyra_status st = forward_impl(L, static_cast<const uint8_t *>(X_dev) + xo, b1 - b0, n,
                                  static_cast<uint8_t *>(Y_dev) + yo, workspace, workspace_bytes,
                                  stream, rec, false);
    if (st != DYRA_OK) {   // `stream` still ends after the copies already enqueued
      cudaEventRecord(ev[1], L->copy_out);
      cudaStreamWaitEvent(stream, ev[1], 0);
      cudaStreamWaitEvent(stream, in_done, 0);
      return st;
    }
    DY_CUDA(cudaEventRecord(fwd_done, stream));
    DY_CUDA(cudaStreamWaitEvent(L->copy_out, fwd_done, 0));
    DY_CUDA(cudaMemcpyAsync(static_cast<uint8_t *>(Y_host) + yo,
                            static_cast<const uint8_t *>(Y_dev) + yo, yn, cudaMemcpyDeviceToHost,
                            L->copy_out));
  }
  // `stream` completes after the last copy out
  DY_CUDA(cudaEventRecord(ev[1], L->copy_out));
  DY_CUDA(cudaStreamWaitEvent(stream, ev[1], 0));
  return DYRA_OK;
}

const char *dyra_kernel_name(const dyra_layer *L, int i) {
  if (!L) return nullptr;
  return kernel_name(L, i);
}

dyra_status dyra_workspace_status(const dyra_layer *L, const void *workspace, cudaStream_t stream,
                                  int *not_spd_samples, int *timeouts) {
  if (!L || !workspace) return DYRA_ERR_INVALID_ARG;
  DeviceGuard guard(L->device);
  int h[2] = {0, 0};
  DY_CUDA(cudaStreamSynchronize(stream));
  DY_CUDA(cudaMemcpy(h, workspace, sizeof(h), cudaMemcpyDeviceToHost));
  if (not_spd_samples) *not_spd_samples = h[0];
  if (timeouts) *timeouts = h[1];
  if (h[1] > 0) return DYRA_ERR_TIMEOUT;
  if (h[0] > 0) return DYRA_ERR_NOT_SPD;
  return DYRA_OK;
}

dyra_status dyra_workspace_tensor(const dyra_layer *L, int batch, int n, int which,
                                  size_t *offset_bytes, int *ld) {
  if (!L || !offset_bytes || !ld || batch < 0 || n < 0) return DYRA_ERR_INVALID_ARG;
  const WsLayout w = layout_of(L, batch, n);
  const bool bf = L->dtype == DYRA_BF16;
  size_t off = 0;
  int l = 0;
  switch (which) {
    case DYRA_BUF_T: off = w.T; l = w.ldT; break;
    case DYRA_BUF_C: off = w.C; l = L->d; break;
    case DYRA_BUF_G: off = w.G; l = L->r; break;
    case DYRA_BUF_GINV: off = w.Ginv; l = L->r; break;
    case DYRA_BUF_B: if (bf) return DYRA_ERR_UNSUPPORTED; off = w.B; l = L->m; break;
    case DYRA_BUF_R: off = w.R; l = L->m; break;
    case DYRA_BUF_CS: if (!bf) return DYRA_ERR_UNSUPPORTED; off = w.Cs; l = L->d; break;
    default: return DYRA_ERR_INVALID_ARG;
  }
  *offset_bytes = off;
  *ld = l;
  return DYRA_OK;
}

dyra_status dyra_linear_forward_static(const dyra_layer *L, const void *X, int batch, int n,
                                       void *Y, cudaStream_t stream) {
  if (!L || batch < 0 || n < 0) return DYRA_ERR_INVALID_ARG;
  if (batch == 0 || n == 0) return DYRA_OK;
  const size_t need = layout_of(L, batch, n).total;
  if (need > (size_t)DYRA_STATIC_SCRATCH_BYTES) {
    g_last_error = "dyra_linear_forward_static: batch " + std::to_string(batch) + " x n " +
                   std::to_string(n) + " needs " + std::to_string(need) +
                   " bytes of scratch, more than the static " +
                   std::to_string((size_t)DYRA_STATIC_SCRATCH_BYTES) + " bytes";
    return DYRA_ERR_WORKSPACE;
  }
  DeviceGuard guard(L->device);
  void *ws = nullptr;
  const dyra_status ss = static_scratch(L->device, &ws);
  if (ss != DYRA_OK) return ss;
  Recorder rec;
  return forward_impl(L, X, batch, n, Y, ws, (size_t)DYRA_STATIC_SCRATCH_BYTES, stream, rec);
}

dyra_status dyra_selftest_bounded_wait(int limit_us, int *status_words, cudaStream_t stream) {
  if (!status_words || limit_us < 1 || limit_us > 2000000) return DYRA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(status_words) & 3) return DYRA_ERR_INVALID_ARG;
  DY_CUDA(cudaMemsetAsync(status_words, 0, 2 * sizeof(int), stream));
  DY_CUDA(dyra::launch_bounded_wait_probe(status_words, 1000ull * (unsigned long long)limit_us,
                                          stream));
  DY_CUDA(cudaStreamSynchronize(stream));
  int h[2] = {0, 0};
  DY_CUDA(cudaMemcpy(h, status_words, sizeof(h), cudaMemcpyDeviceToHost));
  return h[1] > 0 ? DYRA_ERR_TIMEOUT : DYRA_OK;
}

const char *dyra_status_string(dyra_status s) {
  switch (s) {
    case DYRA_OK: return "ok";
    case DYRA_ERR_INVALID_ARG: return "invalid argument";
    case DYRA_ERR_UNSUPPORTED: return "unsupported shape or option";
    case DYRA_ERR_CUDA: return "CUDA error";
    case DYRA_ERR_OOM: return "out of memory";
    case DYRA_ERR_NOT_SPD: return "L^T L + lambda I not positive definite for some sample";
    case DYRA_ERR_TIMEOUT: return "bounded in-kernel wait timed out";
    case DYRA_ERR_WORKSPACE: return "workspace too small or misaligned";
    case DYRA_ERR_NO_DEVICE: return "no usable sm_103 device";
  }
  return "unknown status";
}

const char *dyra_last_error(void) { return g_last_error.c_str(); }

int dyra_abi_version(void) { return DYRA_ABI_VERSION; }

}  // extern "C"
