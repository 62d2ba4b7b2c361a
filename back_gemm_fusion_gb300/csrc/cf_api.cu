// cf_api.cu -- the C ABI (include/cf.h): argument validation, TMA tensor-map
// encoding, device checks, grid sizing and launch of the fused kernels.
//
// Validation runs entirely on the host before any CUDA call, so every
// argument error is reported synchronously and nothing is enqueued.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "cf_internal.h"

// Device status word written by bounded waits that give up.
__device__ unsigned int g_cf_status_word;

namespace cf {
namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool init = false;
  cudaError_t err = cudaSuccess;
  int sms = 0;
  int major = 0, minor = 0;
  unsigned* status = nullptr;
  // Indexed [row code (row_code(first, last row op))][kernel variant][...].
  bool prepared[kRowCodes][kNumVariants][3][2] = {};
  int max_clusters[kRowCodes][kNumVariants][kMaxClusterCtas + 1] = {};  // resident clusters per size (-1: none fit)
  int max_pairs[kRowCodes][kNumVariants][3] = {};                        // resident 2-CTA clusters per xmode
  int blocks_per_sm[kRowCodes][kNumVariants][3] = {};                    // 0 = unknown
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Returns the current device's cached info, or an error status.
cf_status current_device(DeviceInfo** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return CF_ERR_NO_DEVICE;
  }
  if (dev >= kMaxDevices) return CF_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.init) {
    cudaDeviceProp prop;
    d.err = cudaGetDeviceProperties(&prop, dev);
    if (d.err == cudaSuccess) {
      d.sms = prop.multiProcessorCount;
      d.major = prop.major;
      d.minor = prop.minor;
      void* sp = nullptr;
      d.err = cudaGetSymbolAddress(&sp, g_cf_status_word);
      d.status = static_cast<unsigned*>(sp);
    }
    d.init = true;
  }
  if (d.err != cudaSuccess) return CF_ERR_CUDA;
  if (!(d.major == 10 && d.minor == 3)) return CF_ERR_UNSUPPORTED_DEVICE;
  *out = &d;
  return CF_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t elem_size(int dtype) { return dtype == CF_BF16 ? 2 : 4; }

// Logical rows x cols view checks shared by every operand.
cf_status check_matrix(const cf_matrix* m, int dtype, bool allow_trans) {
  if (!m || !m->ptr) return CF_ERR_INVALID_ARG;
  if (m->dtype != dtype) return CF_ERR_INVALID_ARG;
  if (m->trans != 0 && !(allow_trans && m->trans == 1)) return CF_ERR_INVALID_ARG;
  if (m->rows < 0 || m->cols < 0) return CF_ERR_INVALID_ARG;
  const int64_t inner = m->trans ? m->rows : m->cols;
  if (m->ld < inner || m->ld < 1) return CF_ERR_INVALID_ARG;
  if (!aligned16(m->ptr) || ((m->ld * (int64_t)elem_size(dtype)) % 16) != 0) return CF_ERR_MISALIGNED;
  return CF_OK;
}

cf_status encode_2d(CUtensorMap* map, CUtensorMapDataType dt, void* ptr, uint64_t inner, uint64_t outer,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                    CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return CF_ERR_CUDA;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(map, dt, 2, ptr, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CF_OK : CF_ERR_CUDA;
}


struct EpiPlan {
  int rowop = ROW_NONE;
  float eps = 0.0f;
  int rowop0 = ROW_NONE;  // first of two chained reductions
  float eps0 = 0.0f;
  int n_elem0 = 0;        // elementwise ops before it
  int code() const { return row_code(rowop0, rowop); }
  int n_elem = 0;
  int kinds[CF_EPI_MAX_OPS] = {};
  float scalars[CF_EPI_MAX_OPS] = {};
  bool need_bias = false, need_gamma = false, need_beta = false, need_residual = false;
  bool cols = false;      // reductions down the columns (the kernel runs on P^T)
};

cf_status parse_epi(const cf_epi_desc* epi, EpiPlan* plan) {
  if (!epi || epi->version < 1 || epi->version > 3 || epi->n_ops > CF_EPI_MAX_OPS) return CF_ERR_INVALID_ARG;
  if (epi->exchange < CF_XCHG_AUTO || epi->exchange > CF_XCHG_GLOBAL_DYNAMIC) return CF_ERR_INVALID_ARG;
  for (uint32_t i = 0; i < epi->n_ops; ++i) {
    const cf_op& op = epi->ops[i];
    if (!std::isfinite(op.scalar)) return CF_ERR_INVALID_ARG;
    switch (op.kind) {
      case CF_OP_BIAS: plan->need_bias = true; break;
      case CF_OP_ADD_RESIDUAL:
        if (epi->version < 2) return CF_ERR_INVALID_ARG;  // the residual view exists from version 2
        plan->need_residual = true;
        break;
      case CF_OP_SCALE: case CF_OP_RELU: case CF_OP_GELU_TANH: break;
      case CF_OP_ROW_LAYERNORM: case CF_OP_ROW_RMSNORM: case CF_OP_ROW_SOFTMAX: {
        if (op.kind != CF_OP_ROW_SOFTMAX && op.scalar < 0.0f) return CF_ERR_INVALID_ARG;
        const int r = op.kind == CF_OP_ROW_LAYERNORM ? ROW_LAYERNORM
                      : op.kind == CF_OP_ROW_RMSNORM ? ROW_RMSNORM : ROW_SOFTMAX;
        if (i + 1 != epi->n_ops) {
          // A first reduction stage: version 2, a norm, at most one of them.
          if (epi->version < 2 || plan->rowop0 != ROW_NONE || r == ROW_SOFTMAX) return CF_ERR_INVALID_ARG;
          plan->rowop0 = r;
          plan->eps0 = op.scalar;
          plan->n_elem0 = plan->n_elem;
          continue;
        }
        plan->rowop = r;
        plan->eps = op.scalar;
        plan->need_gamma = op.kind != CF_OP_ROW_SOFTMAX;
        plan->need_beta = op.kind == CF_OP_ROW_LAYERNORM;
        continue;
      }
      default: return CF_ERR_INVALID_ARG;
    }
    plan->kinds[plan->n_elem] = op.kind;
    plan->scalars[plan->n_elem] = op.scalar;
    plan->n_elem++;
  }
  // The axis field exists from version 3 (never read from a shorter struct).
  if (epi->version >= 3) {
    if (epi->axis != CF_AXIS_ROWS && epi->axis != CF_AXIS_COLS) return CF_ERR_INVALID_ARG;
    plan->cols = epi->axis == CF_AXIS_COLS && plan->rowop != ROW_NONE;
  }
  return CF_OK;
}

// Exchange mode the fused kernel will use (host-only decision).
int choose_xmode(const EpiPlan& plan, const cf_epi_desc* epi, int64_t tiles_n) {
  if (plan.rowop == ROW_NONE || tiles_n == 1) return X_NONE;
  if (plan.rowop0 != ROW_NONE) return X_GLOBAL;  // chained stages: workspace exchange only
  if (epi->exchange == CF_XCHG_GLOBAL || epi->exchange == CF_XCHG_GLOBAL_DYNAMIC) return X_GLOBAL;
  if (epi->exchange == CF_XCHG_CLUSTER) return X_CLUSTER;
  return tiles_n <= kMaxClusterCtas ? X_CLUSTER : X_GLOBAL;
}

// Workspace of one reduction stage: per-tile partial statistics, then the
// per-(strip, quarter) arrival counters and the work-item ticket counter.
size_t ws_bytes_for(int64_t strips, int64_t tiles_n) {
  const size_t stats = (size_t)strips * (size_t)tiles_n * kBM * sizeof(float2);
  const size_t counters = ((size_t)strips * 4 + 1) * sizeof(unsigned);
  return ((stats + 255) & ~size_t(255)) + ((counters + 255) & ~size_t(255));
}

struct GemmShape {
  int64_t M, N, K;   // the user's problem: P = A . B is M x N
  int64_t kM, kN;    // the kernel's: M x N, or N x M for column reductions (P^T)
};

cf_status validate_gemm_epi(const cf_matrix* A, const cf_matrix* B, const float* bias, const float* gamma,
                            const float* beta, const cf_epi_desc* epi, const cf_matrix* out,
                            EpiPlan* plan, GemmShape* sh) {
  cf_status s;
  if ((s = check_matrix(A, CF_BF16, false)) != CF_OK) return s;
  if ((s = check_matrix(B, CF_BF16, true)) != CF_OK) return s;
  if ((s = parse_epi(epi, plan)) != CF_OK) return s;
  if (epi->out_dtype != CF_FP32 && epi->out_dtype != CF_BF16) return CF_ERR_INVALID_ARG;
  if ((s = check_matrix(out, epi->out_dtype, false)) != CF_OK) return s;
  const int64_t M = A->rows, K = A->cols, N = B->cols;
  if (B->rows != K || out->rows != M || out->cols != N) return CF_ERR_INVALID_ARG;
  if ((plan->need_bias && !bias) || (plan->need_gamma && !gamma) || (plan->need_beta && !beta))
    return CF_ERR_INVALID_ARG;
  if ((bias && !aligned16(bias)) || (gamma && !aligned16(gamma)) || (beta && !aligned16(beta)))
    return CF_ERR_MISALIGNED;
  const int64_t kN = plan->cols ? M : N;  // the kernel's row length
  if (plan->rowop0 != ROW_NONE && epi->exchange == CF_XCHG_CLUSTER && kN > kBN) return CF_ERR_UNSUPPORTED_SHAPE;
  // Chained stages keep the static order (no claimed work items).
  if (plan->rowop0 != ROW_NONE && epi->exchange == CF_XCHG_GLOBAL_DYNAMIC) return CF_ERR_UNSUPPORTED_SHAPE;
  if (plan->rowop0 != ROW_NONE &&
      ((epi->stage0_gamma && !aligned16(epi->stage0_gamma)) || (epi->stage0_beta && !aligned16(epi->stage0_beta))))
    return CF_ERR_MISALIGNED;
  if (plan->need_residual) {
    const cf_matrix& r = epi->residual;
    if (!r.ptr || r.trans || r.rows != M || r.cols != N || r.ld < N || (r.dtype != CF_FP32 && r.dtype != CF_BF16))
      return CF_ERR_INVALID_ARG;
    if (!aligned16(r.ptr) || (r.ld * (r.dtype == CF_FP32 ? 4 : 2)) % 16 != 0) return CF_ERR_MISALIGNED;
  }
  sh->M = M;
  sh->N = N;
  sh->K = K;
  sh->kM = plan->cols ? N : M;
  sh->kN = kN;
  if (M == 0 || N == 0) return CF_OK;
  // Column reductions run on P^T = B^T A^T: the kernel's A operand is B's
  // N x K transpose (K-major), so B must be given that way.
  if (plan->cols && B->trans != 1) return CF_ERR_UNSUPPORTED_SHAPE;
  // Any M >= 1: rows past M are zero-filled by the TMA loads and clipped by
  // the TMA stores of the last (ragged) 128-row strip; rows are independent.
  // K >= 8 with K % 8 == 0: the last (or only) 64-wide K block reads zeros
  // past K
  // (TMA out-of-bounds fill), which add nothing to the products.
  // Any N >= 1: the last 256-column tile of a row may be ragged; its B
  // columns past N load as zeros, the epilogue keeps them out of the row
  // statistics and never reads a vector past N, and the TMA stores clip them.
  if (K % 8 != 0 || K < 8) return CF_ERR_UNSUPPORTED_SHAPE;
  if (M > (int64_t)1 << 31 || N > (int64_t)1 << 31 || K > (int64_t)1 << 31) return CF_ERR_UNSUPPORTED_SHAPE;
  const int64_t tiles_n = (kN + kBN - 1) / kBN;
  if (epi->exchange == CF_XCHG_CLUSTER && plan->rowop != ROW_NONE && tiles_n > kMaxClusterCtas)
    return CF_ERR_UNSUPPORTED_SHAPE;
  return CF_OK;
}

}  // namespace

long long wait_timeout_cycles() {
  const char* e = std::getenv("CF_WAIT_TIMEOUT_CYCLES");
  if (e && *e) {
    long long v = std::atoll(e);
    if (v > 0) return v;
  }
  return 4000000000LL;  // about two seconds at the maximum SM clock
}

cf_status device_query(int* sms, unsigned** status) {
  DeviceInfo* d = nullptr;
  cf_status s = current_device(&d);
  if (s != CF_OK) return s;
  *sms = d->sms;
  *status = d->status;
  return CF_OK;
}

cf_status encode_tmap(CUtensorMap* map, CUtensorMapDataType dt, int rank, void* ptr, const uint64_t* dims,
                      const uint64_t* strides_bytes, const uint32_t* box) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc || rank < 1 || rank > 5) return CF_ERR_CUDA;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides_bytes[i];
  }
  CUresult r = enc(map, dt, (cuuint32_t)rank, ptr, d, st, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CF_OK : CF_ERR_CUDA;
}

}  // namespace cf

using namespace cf;

extern "C" {

int cf_abi_version(void) { return CF_ABI_VERSION; }

const char* cf_status_string(cf_status s) {
  switch (s) {
    case CF_OK: return "CF_OK";
    case CF_ERR_INVALID_ARG: return "CF_ERR_INVALID_ARG";
    case CF_ERR_UNSUPPORTED_SHAPE: return "CF_ERR_UNSUPPORTED_SHAPE";
    case CF_ERR_MISALIGNED: return "CF_ERR_MISALIGNED";
    case CF_ERR_UNSUPPORTED_DEVICE: return "CF_ERR_UNSUPPORTED_DEVICE";
    case CF_ERR_CUDA: return "CF_ERR_CUDA";
    case CF_ERR_TIMEOUT: return "CF_ERR_TIMEOUT";
    case CF_ERR_WORKSPACE: return "CF_ERR_WORKSPACE";
    case CF_ERR_NO_DEVICE: return "CF_ERR_NO_DEVICE";
  }
  return "CF_ERR_UNKNOWN";
}

size_t cf_workspace_size(const cf_matrix* A, const cf_matrix* B, const cf_epi_desc* epi) {
  if (!A || !B || !epi) return 0;
  EpiPlan plan;
  if (parse_epi(epi, &plan) != CF_OK) return 0;
  const int64_t M = plan.cols ? B->cols : A->rows, N = plan.cols ? A->rows : B->cols;  // the kernel's
  if (M <= 0 || N <= 0) return 0;
  const int64_t tiles_n = (N + kBN - 1) / kBN;
  // The cluster path may fall back to the workspace path when no cluster of
  // that size can be resident, so AUTO/CLUSTER strips that fit a cluster
  // still report the (small) fallback workspace.
  if (plan.rowop == ROW_NONE || tiles_n == 1) return 0;
  // Chained reductions: one statistics region per stage.
  return (plan.rowop0 != ROW_NONE ? 2 : 1) * ws_bytes_for((M + kBM - 1) / kBM, tiles_n);
}

cf_status cf_gemm_epilogue(const cf_matrix* A, const cf_matrix* B, const float* bias, const float* gamma,
                           const float* beta, const cf_epi_desc* epi, cf_matrix* out, void* workspace,
                           size_t workspace_bytes, void* stream) {
  EpiPlan plan;
  GemmShape sh;
  cf_status s = validate_gemm_epi(A, B, bias, gamma, beta, epi, out, &plan, &sh);
  if (s != CF_OK) return s;
  if (sh.M == 0 || sh.N == 0) return CF_OK;
  // The kernel's operands: P^T = B^T A^T for column reductions (B given as
  // N x K is the K-major A operand, A the K-major B operand).
  const cf_matrix* KA = plan.cols ? B : A;
  const cf_matrix* KB = plan.cols ? A : B;
  const bool kb_k_major = plan.cols || B->trans == 1;
  const int64_t tiles_n = (sh.kN + kBN - 1) / kBN, strips = (sh.kM + kBM - 1) / kBM;
  int xmode = choose_xmode(plan, epi, tiles_n);
  const int code = plan.code();
  const size_t ws_stage = (plan.rowop != ROW_NONE && tiles_n > 1) ? ws_bytes_for(strips, tiles_n) : 0;
  const size_t need_ws = (plan.rowop0 != ROW_NONE ? 2 : 1) * ws_stage;
  if (xmode == X_GLOBAL && (!workspace || workspace_bytes < need_ws || !aligned16(workspace)))
    return CF_ERR_WORKSPACE;

  DeviceInfo* dev = nullptr;
  if ((s = current_device(&dev)) != CF_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  GemmEpiLaunch L;
  std::memset(&L, 0, sizeof(L));
  GemmEpiParams& p = L.p;
  if ((s = encode_2d(&p.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, KA->ptr, sh.K, sh.kM, KA->ld * 2, kBK, kBM)) != CF_OK)
    return s;
  p.b_mn_major = kb_k_major ? 0 : 1;
  // fp32 out: 32 x 32 blocks of 128-byte rows, 128-byte swizzle; bf16 out:
  // 32 x 32 blocks of 64-byte rows, unswizzled; column reductions stage
  // transposed blocks, unswizzled.  The map always describes the user's
  // M x N output.
  p.out_bf16 = epi->out_dtype == CF_BF16 ? 1 : 0;
  if ((s = p.out_bf16 ? encode_2d(&p.tmOut, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, out->ptr, sh.N, sh.M, out->ld * 2, 32,
                                  32, CU_TENSOR_MAP_SWIZZLE_NONE)
                      : encode_2d(&p.tmOut, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, out->ptr, sh.N, sh.M, out->ld * 4, 32,
                                  32, plan.cols ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B)) != CF_OK)
    return s;
  p.M = (int)sh.kM;
  p.N = (int)sh.kN;
  p.K = (int)sh.K;
  p.tiles_n = (int)tiles_n;
  p.strips = (int)strips;
  p.num_items = (int)(strips * tiles_n);
  p.n_ops = plan.n_elem;
  for (int i = 0; i < plan.n_elem; ++i) {
    p.op_kind[i] = plan.kinds[i];
    p.op_scalar[i] = plan.scalars[i];
  }
  p.eps = plan.eps;
  p.n_ops0 = plan.n_elem0;
  p.eps0 = plan.eps0;
  if (plan.rowop0 != ROW_NONE) {
    p.gamma0 = epi->stage0_gamma;
    p.beta0 = epi->stage0_beta;
  }
  p.bias = bias;
  p.gamma = gamma;
  p.beta = beta;
  if (plan.need_residual) {
    p.res = epi->residual.ptr;
    p.res_ld = epi->residual.ld;
    p.res_bf16 = epi->residual.dtype == CF_BF16 ? 1 : 0;
  }
  p.status = dev->status;
  p.timeout_cycles = wait_timeout_cycles();

  const int variant = (sh.kN % kBN != 0 ? 1 : 0) + (plan.cols ? 2 : 0);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    for (int x = X_NONE; x <= X_GLOBAL; ++x) {
      if (plan.rowop == ROW_NONE && x != X_NONE) continue;
      if (plan.rowop0 != ROW_NONE && x == X_CLUSTER) continue;  // not instantiated for chained stages
      for (int pr = 0; pr < 2; ++pr) {
        if (pr == 1 && x == X_CLUSTER) continue;
        if (!dev->prepared[code][variant][x][pr]) {
          if (gemm_epi_prepare(code, x, pr == 1, variant) != cudaSuccess) return CF_ERR_CUDA;
          dev->prepared[code][variant][x][pr] = true;
        }
      }
    }
  }

  if (xmode == X_CLUSTER) {
    int maxc = 0;
    {
      std::lock_guard<std::mutex> lk(g_mu);
      int& cached = dev->max_clusters[code][variant][tiles_n];
      if (cached == 0) {
        int q = 0;
        if (gemm_epi_max_clusters(code, X_CLUSTER, false, variant, (int)tiles_n, &q) != cudaSuccess) {
          cudaGetLastError();
          q = 0;
        }
        cached = q > 0 ? q : -1;
      }
      maxc = cached > 0 ? cached : 0;
    }
    // The review leaves the choice of inter-CTA aggregation mode open (its
    // threshold C_N).  Here the DSMEM exchange is used on AUTO only when the
    // resident clusters keep at least 90% of the SMs busy; otherwise the
    // per-tile partial-statistics exchange over a persistent grid of every SM
    // is faster (measured: 16-CTA clusters fill only 112 of 152 GB300 SMs).
    const bool fills_gpu = (int64_t)maxc * tiles_n * 10 >= (int64_t)dev->sms * 9;
    if (maxc <= 0 || (epi->exchange == CF_XCHG_AUTO && !fills_gpu)) {
      if (epi->exchange == CF_XCHG_CLUSTER) return CF_ERR_UNSUPPORTED_SHAPE;
      xmode = X_GLOBAL;
      if (!workspace || workspace_bytes < need_ws || !aligned16(workspace)) return CF_ERR_WORKSPACE;
    } else {
      const int64_t nclusters = strips < maxc ? strips : maxc;
      L.cluster = (int)tiles_n;
      L.grid = (int)(nclusters * tiles_n);
    }
  }
  // Pair mode (decided once the exchange mode is final): CTA pairs (2-CTA
  // clusters along M) run 256 x 256 tiles with cta_group::2 MMAs; each CTA
  // loads its A rows and half of the B tile, halving per-SM shared-memory
  // traffic per MMA.  Needs an even number of strips; the cluster (DSMEM)
  // exchange keeps 1-CTA tiles.
  //
  // The workspace exchange makes every tile of a strip (pair) wait for all of
  // its strip-mates, and each worker (a CTA pair, or a CTA) holds two tiles at
  // a time (two TMEM accumulators).  In the static order a worker's epilogue
  // publishes its tiles' statistics one after another, so a worker holding
  // two tiles of one strip would wait for itself: a strip's tiles must not
  // outnumber the workers.  Single-stage programs may instead claim tiles
  // as tickets and publish a worker's next tile while the current one waits
  // (see the kernel): then a strip's tiles must fit in twice the workers
  // that run.  Tickets are used for strips wider than the workers and when
  // the caller asks for them (CF_XCHG_GLOBAL_DYNAMIC); the static order is
  // faster on a GPU of its own.  Strips too wide for the pairs run on 1-CTA
  // tiles (twice the workers); wider still they are refused below.
  const int64_t per_worker = plan.rowop0 != ROW_NONE ? 1 : 2;
  bool want_pair = xmode != X_CLUSTER && strips % 2 == 0;
  int maxp = 0;
  if (want_pair) {
    {
      std::lock_guard<std::mutex> lk(g_mu);
      int& cached = dev->max_pairs[code][variant][xmode];
      if (cached == 0) {
        int q = 0;
        if (gemm_epi_max_clusters(code, xmode, true, variant, 2, &q) != cudaSuccess) {
          cudaGetLastError();
          q = 0;
        }
        cached = q > 0 ? q : -1;
      }
      maxp = cached > 0 ? cached : 0;
    }
    const int64_t pair_items = strips / 2 * tiles_n;
    const int64_t pairs = pair_items < maxp ? pair_items : maxp;
    if (maxp <= 0 || (xmode == X_GLOBAL && tiles_n > per_worker * pairs)) want_pair = false;
  }
  if (p.b_mn_major)
    s = encode_2d(&p.tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, KB->ptr, sh.kN, sh.K, KB->ld * 2, 64, kBK);
  else
    s = encode_2d(&p.tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, KB->ptr, sh.K, sh.kN, KB->ld * 2, kBK,
                  want_pair ? kBN / 2 : kBN);  // pair mode: each CTA loads 128 of the 256 N rows
  if (s != CF_OK) return s;
  if (want_pair) {
    p.pair = 1;
    p.pair_items = (int)(strips / 2 * tiles_n);
    L.grid = 2 * (p.pair_items < maxp ? p.pair_items : maxp);
    L.cluster = 2;
  } else if (xmode != X_CLUSTER) {
    int per_sm = 0;
    {
      std::lock_guard<std::mutex> lk(g_mu);
      int& cached = dev->blocks_per_sm[code][variant][xmode];
      if (cached == 0 && gemm_epi_max_blocks_per_sm(code, xmode, variant, &cached) != cudaSuccess) cached = 0;
      per_sm = cached;
    }
    if (per_sm < 1) return CF_ERR_CUDA;
    const int64_t cap = (int64_t)per_sm * dev->sms;
    L.grid = (int)(p.num_items < cap ? p.num_items : cap);
    L.cluster = 1;
    if (xmode == X_GLOBAL && tiles_n > per_worker * (int64_t)L.grid) return CF_ERR_UNSUPPORTED_SHAPE;  // see above
  }
  if (xmode == X_GLOBAL) {
    const int64_t workers = p.pair ? L.grid / 2 : L.grid;
    p.tickets = (plan.rowop0 == ROW_NONE && (epi->exchange == CF_XCHG_GLOBAL_DYNAMIC || tiles_n > workers)) ? 1 : 0;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const size_t stats = ((size_t)strips * tiles_n * kBM * sizeof(float2) + 255) & ~size_t(255);
    p.ws_stats = reinterpret_cast<float2*>(ws);
    p.ws_count = reinterpret_cast<unsigned*>(ws + stats);
    p.ws_ticket = p.ws_count + strips * 4;
    if (cudaMemsetAsync(p.ws_count, 0, ((size_t)strips * 4 + 1) * sizeof(unsigned), st) != cudaSuccess)
      return CF_ERR_CUDA;
    if (plan.rowop0 != ROW_NONE) {  // the first stage's region follows the last stage's
      p.ws_stats0 = reinterpret_cast<float2*>(ws + ws_stage);
      p.ws_count0 = reinterpret_cast<unsigned*>(ws + ws_stage + stats);
      if (cudaMemsetAsync(p.ws_count0, 0, (size_t)strips * 4 * sizeof(unsigned), st) != cudaSuccess)
        return CF_ERR_CUDA;
    }
  }
  L.rowop = code;
  L.xmode = xmode;
  L.variant = variant;
  if (gemm_epi_launch(L, st) != cudaSuccess) {
    cudaGetLastError();
    return CF_ERR_CUDA;
  }
  return CF_OK;
}

cf_status cf_last_device_status(void* stream) {
  DeviceInfo* dev = nullptr;
  cf_status s = current_device(&dev);
  if (s != CF_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return CF_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, dev->status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return CF_ERR_CUDA;
  if (v != 0) {
    const unsigned zero = 0;
    if (cudaMemcpy(dev->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return CF_ERR_CUDA;
    return CF_ERR_TIMEOUT;
  }
  return CF_OK;
}

}  // extern "C"
