// cf_unfused.cu -- the unfused comparison path: a cuBLASLt GEMM writes the
// intermediate to HBM, then separate kernels read it back.
//
// This is the baseline the fused kernels are measured against (the
// materialisation boundary the ComFuse review describes in "The reading":
// compute-intensive and memory-intensive operators as separate kernels, with
// the intermediate tensor written to global memory and re-read).  The
// epilogue kernels here are plain row-per-CTA kernels; the GEMMs are
// cuBLASLt (bf16 inputs, fp32 accumulate and output).
#include <cublasLt.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "cf_internal.h"

namespace cf {
namespace {

constexpr int kMaxDev = 64;
constexpr size_t kLtWorkspace = 64u << 20;  // cuBLASLt scratch, one per device (comparison path only)

struct LtState {
  cublasLtHandle_t h = nullptr;
  void* ws = nullptr;
  bool init = false;
};
std::mutex g_mu;
LtState g_lt[kMaxDev];

cf_status lt_state(LtState** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    cudaGetLastError();
    return CF_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  LtState& s = g_lt[dev];
  if (!s.init) {
    if (cublasLtCreate(&s.h) != CUBLAS_STATUS_SUCCESS) return CF_ERR_CUDA;
    if (cudaMalloc(&s.ws, kLtWorkspace) != cudaSuccess) return CF_ERR_CUDA;
    s.init = true;
  }
  *out = &s;
  return CF_OK;
}

// Row-major C[M x N] (fp32) = A[M x K] (bf16, row-major) . B (bf16, K x N
// row-major if !b_trans, else stored N x K), `batch` problems with element
// strides.  Expressed column-major as C^T = B^T A^T.
cf_status lt_gemm(const void* A, int64_t lda, const void* B, int64_t ldb, bool b_trans, void* C, int64_t ldc,
                  cudaDataType_t ctype, int64_t M, int64_t N, int64_t K, int64_t batch, int64_t sA, int64_t sB,
                  int64_t sC, cudaStream_t stream) {
  LtState* lt = nullptr;
  cf_status st = lt_state(&lt);
  if (st != CF_OK) return st;
  cublasLtMatmulDesc_t op = nullptr;
  cublasLtMatrixLayout_t la = nullptr, lb = nullptr, lc = nullptr;
  cublasLtMatmulPreference_t pref = nullptr;
  cf_status rs = CF_ERR_CUDA;
  do {
    if (cublasLtMatmulDescCreate(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS) break;
    cublasOperation_t ta = b_trans ? CUBLAS_OP_T : CUBLAS_OP_N, tb = CUBLAS_OP_N;
    cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSA, &ta, sizeof(ta));
    cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSB, &tb, sizeof(tb));
    // cuBLAS "A" = B memory: N x K (col-major, ld ldb) or K x N when stored N x K.
    if (cublasLtMatrixLayoutCreate(&la, CUDA_R_16BF, b_trans ? K : N, b_trans ? N : K, ldb) != CUBLAS_STATUS_SUCCESS)
      break;
    if (cublasLtMatrixLayoutCreate(&lb, CUDA_R_16BF, K, M, lda) != CUBLAS_STATUS_SUCCESS) break;
    if (cublasLtMatrixLayoutCreate(&lc, ctype, N, M, ldc) != CUBLAS_STATUS_SUCCESS) break;
    if (batch > 1) {
      int32_t b32 = (int32_t)batch;
      cublasLtMatrixLayoutSetAttribute(la, CUBLASLT_MATRIX_LAYOUT_BATCH_COUNT, &b32, sizeof(b32));
      cublasLtMatrixLayoutSetAttribute(lb, CUBLASLT_MATRIX_LAYOUT_BATCH_COUNT, &b32, sizeof(b32));
      cublasLtMatrixLayoutSetAttribute(lc, CUBLASLT_MATRIX_LAYOUT_BATCH_COUNT, &b32, sizeof(b32));
      cublasLtMatrixLayoutSetAttribute(la, CUBLASLT_MATRIX_LAYOUT_STRIDED_BATCH_OFFSET, &sB, sizeof(sB));
      cublasLtMatrixLayoutSetAttribute(lb, CUBLASLT_MATRIX_LAYOUT_STRIDED_BATCH_OFFSET, &sA, sizeof(sA));
      cublasLtMatrixLayoutSetAttribute(lc, CUBLASLT_MATRIX_LAYOUT_STRIDED_BATCH_OFFSET, &sC, sizeof(sC));
    }
    if (cublasLtMatmulPreferenceCreate(&pref) != CUBLAS_STATUS_SUCCESS) break;
    size_t wsb = kLtWorkspace;
    cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &wsb, sizeof(wsb));
    cublasLtMatmulHeuristicResult_t heur;
    int found = 0;
    if (cublasLtMatmulAlgoGetHeuristic(lt->h, op, la, lb, lc, lc, pref, 1, &heur, &found) !=
            CUBLAS_STATUS_SUCCESS ||
        found == 0)
      break;
    const float alpha = 1.0f, beta = 0.0f;
    if (cublasLtMatmul(lt->h, op, &alpha, B, la, A, lb, &beta, C, lc, C, lc, &heur.algo, lt->ws, kLtWorkspace,
                       stream) != CUBLAS_STATUS_SUCCESS)
      break;
    rs = CF_OK;
  } while (false);
  if (pref) cublasLtMatmulPreferenceDestroy(pref);
  if (lc) cublasLtMatrixLayoutDestroy(lc);
  if (lb) cublasLtMatrixLayoutDestroy(lb);
  if (la) cublasLtMatrixLayoutDestroy(la);
  if (op) cublasLtMatmulDescDestroy(op);
  return rs;
}

struct RowProgram {
  int n_ops;
  int kind[CF_EPI_MAX_OPS];
  float scalar[CF_EPI_MAX_OPS];
  int rowop;  // 0 none, CF_OP_ROW_* otherwise
  float eps;
};

// The CF_OP_ADD_RESIDUAL matrix (fp32 or bf16) of a program; passed to the
// kernels apart from RowProgram so that the program stays in parameter space.
struct ResView {
  const void* ptr;
  long long ld;
  int bf16;
};

// Residual value of element (m, n) (0 when the program has no residual op).
__device__ __forceinline__ float res_at(const void* res, long long ld, int bf16, int m, int n) {
  if (!res) return 0.0f;
  return bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(res)[(long long)m * ld + n])
              : static_cast<const float*>(res)[(long long)m * ld + n];
}

// tanh-GELU as 0.5 x (1 + tanh(u)) = x / (1 + exp(-2u)), u = sqrt(2/pi) (x +
// 0.044715 x^3), with the fast exponential (the fused kernel's arithmetic).
__device__ __forceinline__ float gelu_fast(float x) {
  const float u = 0.7978845608028654f * fmaf(0.044715f * x, x * x, x);
  return __fdividef(x, 1.0f + __expf(-2.0f * u));
}

// The first of two chained row reductions of a program (LayerNorm or
// RMSNorm); ops [0, n_ops0) precede it.
struct ChainStage {
  int rowop;
  float eps;
  int n_ops0;
  const float* gamma;  // may be null (no affine transform)
  const float* beta;
};

// Block-wide sum or max of one value per thread (blockDim.x == 256).
template <bool kMax>
__device__ float block_reduce(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    v = kMax ? fmaxf(v, w) : v + w;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
  for (int i = 1; i < (int)(blockDim.x >> 5); ++i) r = kMax ? fmaxf(r, red[i]) : r + red[i];
  return r;
}

// Ops [o0, o1) of the program over this thread's elements of row m (held in
// shared memory; every pass visits the same elements with the same thread,
// so no barrier is needed between passes), one dispatch per op.
__device__ __forceinline__ void apply_ops_smem(const RowProgram& pg, float* row, int N, const float* bias,
                                               const ResView& rv, int m, int o0, int o1) {
  for (int op = o0; op < o1; ++op) {
    const int kind = pg.kind[op];
    const float sc = pg.scalar[op];
    if (kind == CF_OP_BIAS) {
      for (int n = threadIdx.x; n < N; n += blockDim.x) row[n] += bias[n];
    } else if (kind == CF_OP_ADD_RESIDUAL) {
      for (int n = threadIdx.x; n < N; n += blockDim.x) row[n] += res_at(rv.ptr, rv.ld, rv.bf16, m, n);
    } else if (kind == CF_OP_SCALE) {
      for (int n = threadIdx.x; n < N; n += blockDim.x) row[n] *= sc;
    } else if (kind == CF_OP_RELU) {
      for (int n = threadIdx.x; n < N; n += blockDim.x) row[n] = fmaxf(row[n], 0.0f);
    } else if (kind == CF_OP_GELU_TANH) {
      for (int n = threadIdx.x; n < N; n += blockDim.x) row[n] = gelu_fast(row[n]);
    }
  }
}

// One CTA per row: read P back from HBM, elementwise program, row statistic,
// normalise, write out.  The activated row is kept in shared memory.
__global__ void __launch_bounds__(256) row_epilogue_kernel(const float* __restrict__ P, int64_t ldp,
                                                           float* __restrict__ out, int64_t ldo, int N,
                                                           RowProgram pg, const float* __restrict__ bias,
                                                           const float* __restrict__ gamma,
                                                           const float* __restrict__ beta, ResView rv) {
  extern __shared__ float row[];
  __shared__ float red[32];
  const float* p = P + (int64_t)blockIdx.x * ldp;
  float* o = out + (int64_t)blockIdx.x * ldo;
  for (int n = threadIdx.x; n < N; n += blockDim.x) row[n] = p[n];
  apply_ops_smem(pg, row, N, bias, rv, (int)blockIdx.x, 0, pg.n_ops);
  float acc = 0.0f, mx = -INFINITY;
  for (int n = threadIdx.x; n < N; n += blockDim.x) {
    const float x = row[n];
    acc += x;
    mx = fmaxf(mx, x);
  }
  if (pg.rowop == 0) {
    for (int n = threadIdx.x; n < N; n += blockDim.x) o[n] = row[n];
    return;
  }
  if (pg.rowop == CF_OP_ROW_LAYERNORM) {
    const float mean = block_reduce<false>(acc, red) / N;
    float ss = 0.0f;
    for (int n = threadIdx.x; n < N; n += blockDim.x) {
      const float d = row[n] - mean;
      ss += d * d;
    }
    const float rstd = rsqrtf(block_reduce<false>(ss, red) / N + pg.eps);
    for (int n = threadIdx.x; n < N; n += blockDim.x) o[n] = gamma[n] * (row[n] - mean) * rstd + beta[n];
  } else if (pg.rowop == CF_OP_ROW_RMSNORM) {
    float ss = 0.0f;
    for (int n = threadIdx.x; n < N; n += blockDim.x) ss += row[n] * row[n];
    const float rstd = rsqrtf(block_reduce<false>(ss, red) / N + pg.eps);
    for (int n = threadIdx.x; n < N; n += blockDim.x) o[n] = gamma[n] * row[n] * rstd;
  } else {
    const float m = block_reduce<true>(mx, red);
    float s = 0.0f;
    for (int n = threadIdx.x; n < N; n += blockDim.x) s += __expf(row[n] - m);
    const float inv = 1.0f / block_reduce<false>(s, red);
    for (int n = threadIdx.x; n < N; n += blockDim.x) o[n] = __expf(row[n] - m) * inv;
  }
}

// Chained programs, one CTA per row: first stage (ops, reduction, affine),
// then the remaining ops and the last reduction; the row stays in shared
// memory between the stages.
__global__ void __launch_bounds__(256) row_epilogue_chain_kernel(const float* __restrict__ P, int64_t ldp,
                                                                 float* __restrict__ out, int64_t ldo, int N,
                                                                 RowProgram pg, ChainStage c0,
                                                                 const float* __restrict__ bias,
                                                                 const float* __restrict__ gamma,
                                                                 const float* __restrict__ beta, ResView rv) {
  extern __shared__ float row[];
  __shared__ float red[32];
  const int m = (int)blockIdx.x;
  const float* p = P + (int64_t)m * ldp;
  float* o = out + (int64_t)m * ldo;
  for (int n = threadIdx.x; n < N; n += blockDim.x) row[n] = p[n];
  apply_ops_smem(pg, row, N, bias, rv, m, 0, c0.n_ops0);
  float acc = 0.0f;
  for (int n = threadIdx.x; n < N; n += blockDim.x) {
    const float x = row[n];
    acc += (c0.rowop == CF_OP_ROW_RMSNORM) ? x * x : x;
  }
  float sc, sh = 0.0f;
  if (c0.rowop == CF_OP_ROW_LAYERNORM) {
    const float mean = block_reduce<false>(acc, red) / N;
    float ss = 0.0f;
    for (int n = threadIdx.x; n < N; n += blockDim.x) {
      const float d = row[n] - mean;
      ss += d * d;
    }
    sc = rsqrtf(block_reduce<false>(ss, red) / N + c0.eps);
    sh = -mean * sc;
  } else {
    sc = rsqrtf(block_reduce<false>(acc, red) / N + c0.eps);
  }
  for (int n = threadIdx.x; n < N; n += blockDim.x) {
    float x = row[n] * sc + sh;
    if (c0.gamma) x *= c0.gamma[n];
    if (c0.rowop == CF_OP_ROW_LAYERNORM && c0.beta) x += c0.beta[n];
    row[n] = x;
  }
  apply_ops_smem(pg, row, N, bias, rv, m, c0.n_ops0, pg.n_ops);
  acc = 0.0f;
  float mx = -INFINITY;
  for (int n = threadIdx.x; n < N; n += blockDim.x) {
    const float x = row[n];
    acc += x;
    mx = fmaxf(mx, x);
  }
  if (pg.rowop == CF_OP_ROW_LAYERNORM) {
    const float mean = block_reduce<false>(acc, red) / N;
    float ss = 0.0f;
    for (int n = threadIdx.x; n < N; n += blockDim.x) {
      const float d = row[n] - mean;
      ss += d * d;
    }
    const float rstd = rsqrtf(block_reduce<false>(ss, red) / N + pg.eps);
    for (int n = threadIdx.x; n < N; n += blockDim.x) o[n] = gamma[n] * (row[n] - mean) * rstd + beta[n];
  } else if (pg.rowop == CF_OP_ROW_RMSNORM) {
    float ss = 0.0f;
    for (int n = threadIdx.x; n < N; n += blockDim.x) ss += row[n] * row[n];
    const float rstd = rsqrtf(block_reduce<false>(ss, red) / N + pg.eps);
    for (int n = threadIdx.x; n < N; n += blockDim.x) o[n] = gamma[n] * row[n] * rstd;
  } else {
    const float mm = block_reduce<true>(mx, red);
    float sum = 0.0f;
    for (int n = threadIdx.x; n < N; n += blockDim.x) sum += __expf(row[n] - mm);
    const float inv = 1.0f / block_reduce<false>(sum, red);
    for (int n = threadIdx.x; n < N; n += blockDim.x) o[n] = __expf(row[n] - mm) * inv;
  }
}

// Ops [o0, o1) of the program over a thread's VPT float4 vectors of row m
// (float4 index c = i * 256 + threadIdx.x), one dispatch per op, 16-byte
// loads of the bias and the residual.
template <int VPT>
__device__ __forceinline__ void apply_ops_vec(const RowProgram& pg, float4 (&v)[VPT], const float* bias,
                                              const ResView& rv, int m, int o0, int o1) {
  for (int op = o0; op < o1; ++op) {
    const int kind = pg.kind[op];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int c = i * 256 + threadIdx.x;  // float4 index
      float4 x = v[i];
      if (kind == CF_OP_BIAS) {
        const float4 b = reinterpret_cast<const float4*>(bias)[c];
        x = make_float4(x.x + b.x, x.y + b.y, x.z + b.z, x.w + b.w);
      } else if (kind == CF_OP_ADD_RESIDUAL) {
        float4 r;
        if (rv.bf16) {
          const uint2 w = reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(rv.ptr) +
                                                         (long long)m * rv.ld)[c];
          r = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                          __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
        } else {
          r = reinterpret_cast<const float4*>(static_cast<const float*>(rv.ptr) + (long long)m * rv.ld)[c];
        }
        x = make_float4(x.x + r.x, x.y + r.y, x.z + r.z, x.w + r.w);
      } else if (kind == CF_OP_SCALE) {
        const float sc = pg.scalar[op];
        x = make_float4(x.x * sc, x.y * sc, x.z * sc, x.w * sc);
      } else if (kind == CF_OP_RELU) {
        x = make_float4(fmaxf(x.x, 0.0f), fmaxf(x.y, 0.0f), fmaxf(x.z, 0.0f), fmaxf(x.w, 0.0f));
      } else if (kind == CF_OP_GELU_TANH) {
        x = make_float4(gelu_fast(x.x), gelu_fast(x.y), gelu_fast(x.z), gelu_fast(x.w));
      }
      v[i] = x;
    }
  }
}

// Normalisation constants (y = x * mul + add) of a LayerNorm or RMSNorm over
// the row held in the block's vectors.
template <int VPT>
__device__ __forceinline__ void norm_consts_vec(int rowop, float eps, const float4 (&v)[VPT], int N, float* red,
                                                float& mul, float& add) {
  add = 0.0f;
  if (rowop == CF_OP_ROW_LAYERNORM) {
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) s += v[i].x + v[i].y + v[i].z + v[i].w;
    const float mean = block_reduce<false>(s, red) / N;
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const float a = v[i].x - mean, b = v[i].y - mean, c = v[i].z - mean, d = v[i].w - mean;
      ss += a * a + b * b + c * c + d * d;
    }
    mul = rsqrtf(block_reduce<false>(ss, red) / N + eps);
    add = -mean * mul;
  } else {
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
    mul = rsqrtf(block_reduce<false>(ss, red) / N + eps);
  }
}

// Bandwidth-oriented row epilogue for N = 1024 * VPT: each of 256 threads
// keeps VPT float4 vectors of the row in registers, so P is read once and
// the output written once; chained programs (c0.rowop != 0) run both stages
// on the same registers.
template <int VPT>
__global__ void __launch_bounds__(256) row_epilogue_reg_kernel(const float* __restrict__ P, int64_t ldp,
                                                               float* __restrict__ out, int64_t ldo, int N,
                                                               RowProgram pg, ChainStage c0,
                                                               const float* __restrict__ bias,
                                                               const float* __restrict__ gamma,
                                                               const float* __restrict__ beta, ResView rv) {
  __shared__ float red[32];
  const float4* p = reinterpret_cast<const float4*>(P + (int64_t)blockIdx.x * ldp);
  float4* o = reinterpret_cast<float4*>(out + (int64_t)blockIdx.x * ldo);
  float4 v[VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i) v[i] = p[i * 256 + threadIdx.x];
  if (c0.rowop != 0) {
    // A first (chained) reduction: its ops, its normalisation and affine
    // vectors, then the ops that follow it.
    apply_ops_vec<VPT>(pg, v, bias, rv, (int)blockIdx.x, 0, c0.n_ops0);
    float mul0, add0;
    norm_consts_vec<VPT>(c0.rowop, c0.eps, v, N, red, mul0, add0);
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int c = i * 256 + threadIdx.x;
      float4 x = make_float4(fmaf(v[i].x, mul0, add0), fmaf(v[i].y, mul0, add0), fmaf(v[i].z, mul0, add0),
                             fmaf(v[i].w, mul0, add0));
      if (c0.gamma) {
        const float4 g = reinterpret_cast<const float4*>(c0.gamma)[c];
        x = make_float4(x.x * g.x, x.y * g.y, x.z * g.z, x.w * g.w);
      }
      if (c0.rowop == CF_OP_ROW_LAYERNORM && c0.beta) {
        const float4 b = reinterpret_cast<const float4*>(c0.beta)[c];
        x = make_float4(x.x + b.x, x.y + b.y, x.z + b.z, x.w + b.w);
      }
      v[i] = x;
    }
    apply_ops_vec<VPT>(pg, v, bias, rv, (int)blockIdx.x, c0.n_ops0, pg.n_ops);
  } else {
    apply_ops_vec<VPT>(pg, v, bias, rv, (int)blockIdx.x, 0, pg.n_ops);
  }
  float mul = 1.0f, add = 0.0f;  // y = (x * mul + add) [* gamma + beta]
  if (pg.rowop == CF_OP_ROW_LAYERNORM) {
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) s += v[i].x + v[i].y + v[i].z + v[i].w;
    const float mean = block_reduce<false>(s, red) / N;
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const float a = v[i].x - mean, b = v[i].y - mean, c = v[i].z - mean, d = v[i].w - mean;
      ss += a * a + b * b + c * c + d * d;
    }
    mul = rsqrtf(block_reduce<false>(ss, red) / N + pg.eps);
    add = -mean * mul;
  } else if (pg.rowop == CF_OP_ROW_RMSNORM) {
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
    mul = rsqrtf(block_reduce<false>(ss, red) / N + pg.eps);
  } else if (pg.rowop == CF_OP_ROW_SOFTMAX) {
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < VPT; ++i) mx = fmaxf(fmaxf(mx, fmaxf(v[i].x, v[i].y)), fmaxf(v[i].z, v[i].w));
    const float m = block_reduce<true>(mx, red);
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      v[i].x = __expf(v[i].x - m);
      v[i].y = __expf(v[i].y - m);
      v[i].z = __expf(v[i].z - m);
      v[i].w = __expf(v[i].w - m);
      s += v[i].x + v[i].y + v[i].z + v[i].w;
    }
    mul = 1.0f / block_reduce<false>(s, red);
  }
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = i * 256 + threadIdx.x;
    float4 y = make_float4(fmaf(v[i].x, mul, add), fmaf(v[i].y, mul, add), fmaf(v[i].z, mul, add),
                           fmaf(v[i].w, mul, add));
    if (pg.rowop == CF_OP_ROW_LAYERNORM || pg.rowop == CF_OP_ROW_RMSNORM) {
      const float4 g = reinterpret_cast<const float4*>(gamma)[c];
      y.x *= g.x; y.y *= g.y; y.z *= g.z; y.w *= g.w;
      if (pg.rowop == CF_OP_ROW_LAYERNORM) {
        const float4 b = reinterpret_cast<const float4*>(beta)[c];
        y.x += b.x; y.y += b.y; y.z += b.z; y.w += b.w;
      }
    }
    o[c] = y;
  }
}

// Column reductions for the unfused comparison path, three kinds of
// kernels over a grid of (32-column block, row chunk) CTAs of 32 x 16
// threads (lane x = column, y = row group: every row read is a coalesced
// 128-byte segment):
//   col_stats_kernel     per-chunk statistics of one reduction stage,
//   col_finalize_kernel  per-column merge of the chunks -> (mul, add),
//   col_write_kernel     the normalised output.
// The elementwise stages are recomputed from P on every pass.  Norm
// statistics are sums shifted by the column's row-0 value (robust to large
// means, identical in every chunk); softmax keeps an online (max, sum) pair.
// Scratch (partials and constants) is a static device array of the library.
constexpr int kColGroups = 16;
constexpr int kColMaxN = 65536;
constexpr size_t kColPartCap = (size_t)6 << 17;  // ColStat entries (6 MB)

struct ColStat {
  float a, b;  // norms: shifted sum, shifted sum of squares; softmax: max, sum exp
};

__device__ ColStat g_col_part[kColPartCap];   // [chunk][column]
__device__ float2 g_col_consts[2][kColMaxN];  // [stage][column]: y = x * mul + add

struct ColArgs {
  const float* P;
  int M, N, rows_per, chunks;
  RowProgram pg;
  ChainStage c0;
  const float* bias;
  ResView rv;
};

__device__ __forceinline__ float col_ops(const RowProgram& pg, float x, const float* bias, const ResView& rv, int m,
                                         int n, int o0, int o1) {
  for (int op = o0; op < o1; ++op) {
    switch (pg.kind[op]) {
      case CF_OP_BIAS: x += bias[n]; break;
      case CF_OP_ADD_RESIDUAL: x += res_at(rv.ptr, rv.ld, rv.bf16, m, n); break;
      case CF_OP_SCALE: x *= pg.scalar[op]; break;
      case CF_OP_RELU: x = fmaxf(x, 0.0f); break;
      case CF_OP_GELU_TANH: x = gelu_fast(x); break;
    }
  }
  return x;
}

// Value of element (m, n) at the input of reduction stage `second` (0: the
// first or only reduction, 1: the second of a chain).
__device__ __forceinline__ float col_stage(const ColArgs& a, int m, int n, bool second) {
  const bool chain = a.c0.rowop != 0;
  float x = col_ops(a.pg, a.P[(int64_t)m * a.N + n], a.bias, a.rv, m, n, 0, chain ? a.c0.n_ops0 : a.pg.n_ops);
  if (!second) return x;
  const float2 k0 = g_col_consts[0][n];
  x = fmaf(x, k0.x, k0.y);
  if (a.c0.gamma) x *= a.c0.gamma[n];
  if (a.c0.rowop == CF_OP_ROW_LAYERNORM && a.c0.beta) x += a.c0.beta[n];
  return col_ops(a.pg, x, a.bias, a.rv, m, n, a.c0.n_ops0, a.pg.n_ops);
}

__global__ void __launch_bounds__(32 * kColGroups) col_stats_kernel(ColArgs a, int rowop, int second) {
  __shared__ ColStat sh[kColGroups][32];
  const int n = blockIdx.x * 32 + threadIdx.x;
  const int nn = n < a.N ? n : a.N - 1;
  const float shift = col_stage(a, 0, nn, second);
  ColStat st = rowop == CF_OP_ROW_SOFTMAX ? ColStat{-INFINITY, 0.0f} : ColStat{0.0f, 0.0f};
  const int r0 = blockIdx.y * a.rows_per, r1 = min(a.M, r0 + a.rows_per);
  for (int m = r0 + threadIdx.y; m < r1; m += kColGroups) {
    const float x = col_stage(a, m, nn, second);
    if (rowop == CF_OP_ROW_SOFTMAX) {
      const float mm = fmaxf(st.a, x);
      st.b = st.b * __expf(st.a - mm) + __expf(x - mm);
      st.a = mm;
    } else {
      const float d = x - shift;
      st.a += d;
      st.b = fmaf(d, d, st.b);
    }
  }
  sh[threadIdx.y][threadIdx.x] = st;
  __syncthreads();
  if (threadIdx.y != 0 || n >= a.N) return;
  for (int g = 1; g < kColGroups; ++g) {
    const ColStat u = sh[g][threadIdx.x];
    if (rowop == CF_OP_ROW_SOFTMAX) {
      const float mm = fmaxf(st.a, u.a);
      st.b = (st.b == 0.0f ? 0.0f : st.b * __expf(st.a - mm)) + (u.b == 0.0f ? 0.0f : u.b * __expf(u.a - mm));
      st.a = mm;
    } else {
      st.a += u.a;
      st.b += u.b;
    }
  }
  g_col_part[(size_t)blockIdx.y * a.N + n] = st;
}

// Constants of the stage whose input is col_stage(second) into slot `slot`.
__global__ void col_finalize_kernel(ColArgs a, int rowop, float eps, int second, int slot) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= a.N) return;
  ColStat t = g_col_part[n];
  for (int r = 1; r < a.chunks; ++r) {
    const ColStat u = g_col_part[(size_t)r * a.N + n];
    if (rowop == CF_OP_ROW_SOFTMAX) {
      const float mm = fmaxf(t.a, u.a);
      t.b = (t.b == 0.0f ? 0.0f : t.b * __expf(t.a - mm)) + (u.b == 0.0f ? 0.0f : u.b * __expf(u.a - mm));
      t.a = mm;
    } else {
      t.a += u.a;
      t.b += u.b;
    }
  }
  float mul, add;
  if (rowop == CF_OP_ROW_SOFTMAX) {  // y = exp(x - max) / sum: kept as (1 / sum, max)
    mul = 1.0f / t.b;
    add = t.a;
  } else {
    const float shift = col_stage(a, 0, n, second);
    const float m1 = t.a / a.M, m2 = t.b / a.M;
    if (rowop == CF_OP_ROW_LAYERNORM) {
      mul = rsqrtf(fmaxf(m2 - m1 * m1, 0.0f) + eps);
      add = -(shift + m1) * mul;
    } else {  // mean of x^2 = mean of (d + shift)^2 with d = x - shift
      mul = rsqrtf(m2 + 2.0f * shift * m1 + shift * shift + eps);
      add = 0.0f;
    }
  }
  g_col_consts[slot][n] = make_float2(mul, add);
}

__global__ void __launch_bounds__(32 * kColGroups) col_write_kernel(ColArgs a, float* __restrict__ out, int64_t ldo,
                                                                     const float* __restrict__ gamma,
                                                                     const float* __restrict__ beta) {
  const int n = blockIdx.x * 32 + threadIdx.x;
  if (n >= a.N) return;
  const bool chain = a.c0.rowop != 0;
  const int rowop = a.pg.rowop;
  const float2 k = g_col_consts[1][n];
  const float g = rowop == CF_OP_ROW_SOFTMAX ? 1.0f : gamma[n];
  const float b = rowop == CF_OP_ROW_LAYERNORM ? beta[n] : 0.0f;
  const int r0 = blockIdx.y * a.rows_per, r1 = min(a.M, r0 + a.rows_per);
  for (int m = r0 + threadIdx.y; m < r1; m += kColGroups) {
    const float x = col_stage(a, m, n, chain);
    out[(int64_t)m * ldo + n] = rowop == CF_OP_ROW_SOFTMAX ? __expf(x - k.y) * k.x : fmaf(x, k.x, k.y) * g + b;
  }
}

// Register-resident mid op for N1 = 1024 * VPT (one CTA of 256 threads per row).
template <int VPT>
__global__ void __launch_bounds__(256) mid_op_reg_kernel(const float* __restrict__ S, __nv_bfloat16* __restrict__ Pout,
                                                         int N1, int op, float scale) {
  __shared__ float red[32];
  const float4* s = reinterpret_cast<const float4*>(S + (int64_t)blockIdx.x * N1);
  uint2* o = reinterpret_cast<uint2*>(Pout + (int64_t)blockIdx.x * N1);
  float4 v[VPT];
  const float sc = op == CF_MID_RELU ? 1.0f : scale;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    float4 x = s[i * 256 + threadIdx.x];
    v[i] = make_float4(x.x * sc, x.y * sc, x.z * sc, x.w * sc);
  }
  float mul = 1.0f;
  if (op == CF_MID_SCALE_SOFTMAX) {
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < VPT; ++i) mx = fmaxf(fmaxf(mx, fmaxf(v[i].x, v[i].y)), fmaxf(v[i].z, v[i].w));
    const float m = block_reduce<true>(mx, red);
    float sum = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      v[i].x = __expf(v[i].x - m);
      v[i].y = __expf(v[i].y - m);
      v[i].z = __expf(v[i].z - m);
      v[i].w = __expf(v[i].w - m);
      sum += v[i].x + v[i].y + v[i].z + v[i].w;
    }
    mul = 1.0f / block_reduce<false>(sum, red);
  }
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    float4 y = v[i];
    if (op == CF_MID_SCALE_SOFTMAX) {
      y.x *= mul; y.y *= mul; y.z *= mul; y.w *= mul;
    } else {
      y.x = fmaxf(y.x, 0.0f); y.y = fmaxf(y.y, 0.0f); y.z = fmaxf(y.z, 0.0f); y.w = fmaxf(y.w, 0.0f);
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(y.x, y.y), hi = __floats2bfloat162_rn(y.z, y.w);
    o[i * 256 + threadIdx.x] = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
  }
}

// Mid op of the unfused B2BGEMM: S (fp32) -> bf16 S' = F(S), one CTA per row.
__global__ void __launch_bounds__(256) mid_op_kernel(const float* __restrict__ S, __nv_bfloat16* __restrict__ Pout,
                                                     int N1, int op, float scale) {
  extern __shared__ float row[];
  __shared__ float red[32];
  const float* s = S + (int64_t)blockIdx.x * N1;
  __nv_bfloat16* p = Pout + (int64_t)blockIdx.x * N1;
  if (op != CF_MID_SCALE_SOFTMAX) {
    const float sc = op == CF_MID_RELU ? 1.0f : scale;
    for (int n = threadIdx.x; n < N1; n += blockDim.x) p[n] = __float2bfloat16_rn(fmaxf(sc * s[n], 0.0f));
    return;
  }
  float mx = -INFINITY;
  for (int n = threadIdx.x; n < N1; n += blockDim.x) {
    row[n] = scale * s[n];
    mx = fmaxf(mx, row[n]);
  }
  const float m = block_reduce<true>(mx, red);
  float sum = 0.0f;
  for (int n = threadIdx.x; n < N1; n += blockDim.x) sum += __expf(row[n] - m);
  const float inv = 1.0f / block_reduce<false>(sum, red);
  for (int n = threadIdx.x; n < N1; n += blockDim.x) p[n] = __float2bfloat16_rn(__expf(row[n] - m) * inv);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace cf

using namespace cf;

extern "C" cf_status cf_unfused_gemm_epilogue(const cf_matrix* A, const cf_matrix* B, const float* bias,
                                              const float* gamma, const float* beta, const cf_epi_desc* epi,
                                              cf_matrix* out, float* intermediate, void* stream) {
  if (!A || !B || !epi || !out || !intermediate || !A->ptr || !B->ptr || !out->ptr) return CF_ERR_INVALID_ARG;
  if (A->dtype != CF_BF16 || B->dtype != CF_BF16 || out->dtype != CF_FP32 || A->trans || out->trans)
    return CF_ERR_INVALID_ARG;
  if (epi->version < 1 || epi->version > 3 || epi->n_ops > CF_EPI_MAX_OPS) return CF_ERR_INVALID_ARG;
  bool cols = false;  // reductions down the columns (col_epilogue_kernel)
  if (epi->version >= 3) {
    if (epi->axis != CF_AXIS_ROWS && epi->axis != CF_AXIS_COLS) return CF_ERR_INVALID_ARG;
    for (uint32_t i = 0; i < epi->n_ops; ++i)
      if (epi->ops[i].kind >= CF_OP_ROW_LAYERNORM && epi->ops[i].kind <= CF_OP_ROW_SOFTMAX)
        cols = epi->axis == CF_AXIS_COLS;
  }
  const int64_t M = A->rows, K = A->cols, N = B->cols;
  if (B->rows != K || out->rows != M || out->cols != N) return CF_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return CF_OK;
  if (N > 16384) return CF_ERR_UNSUPPORTED_SHAPE;  // the row must fit the epilogue's shared memory
  if (!aligned16(A->ptr) || !aligned16(B->ptr) || !aligned16(intermediate)) return CF_ERR_MISALIGNED;
  RowProgram pg;
  std::memset(&pg, 0, sizeof(pg));
  ResView rv = {nullptr, 0, 0};
  ChainStage c0 = {0, 0.0f, 0, nullptr, nullptr};
  for (uint32_t i = 0; i < epi->n_ops; ++i) {
    const int k = epi->ops[i].kind;
    if (k >= CF_OP_ROW_LAYERNORM && i + 1 != epi->n_ops) {  // first of two chained reductions
      if (epi->version < 2 || c0.rowop != 0 || k == CF_OP_ROW_SOFTMAX) return CF_ERR_INVALID_ARG;
      c0.rowop = k;
      c0.eps = epi->ops[i].scalar;
      c0.n_ops0 = pg.n_ops;
      c0.gamma = epi->stage0_gamma;
      c0.beta = epi->stage0_beta;
      continue;
    }
    if (k == CF_OP_ADD_RESIDUAL) {
      const cf_matrix& r = epi->residual;
      if (epi->version < 2 || !r.ptr || r.trans || r.rows != M || r.cols != N || r.ld < N ||
          (r.dtype != CF_FP32 && r.dtype != CF_BF16))
        return CF_ERR_INVALID_ARG;
      // The row kernels read the residual with vector loads (same rule as
      // the fused call).
      if (!aligned16(r.ptr) || (r.ld * (r.dtype == CF_FP32 ? 4 : 2)) % 16 != 0) return CF_ERR_MISALIGNED;
      rv.ptr = r.ptr;
      rv.ld = r.ld;
      rv.bf16 = r.dtype == CF_BF16;
    }
    if (k >= CF_OP_ROW_LAYERNORM) {
      if (i + 1 != epi->n_ops) return CF_ERR_INVALID_ARG;
      pg.rowop = k;
      pg.eps = epi->ops[i].scalar;
    } else {
      pg.kind[pg.n_ops] = k;
      pg.scalar[pg.n_ops] = epi->ops[i].scalar;
      pg.n_ops++;
    }
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cf_status s = lt_gemm(A->ptr, A->ld, B->ptr, B->ld, B->trans != 0, intermediate, N, CUDA_R_32F, M, N, K, 1, 0,
                        0, 0, st);
  if (s != CF_OK) return s;
  float* o = static_cast<float*>(out->ptr);
  if (cols) {
    if (N > kColMaxN) return CF_ERR_UNSUPPORTED_SHAPE;
    ColArgs ca;
    ca.P = intermediate;
    ca.M = (int)M;
    ca.N = (int)N;
    // Row chunks of >= 256 rows, as many as the partial-statistics array holds.
    const int64_t max_chunks = (int64_t)(kColPartCap / (size_t)N);
    int64_t rows_per = 256;
    while ((M + rows_per - 1) / rows_per > max_chunks) rows_per *= 2;
    ca.rows_per = (int)rows_per;
    ca.chunks = (int)((M + rows_per - 1) / rows_per);
    ca.pg = pg;
    ca.c0 = c0;
    ca.bias = bias;
    ca.rv = rv;
    const dim3 grid((unsigned)((N + 31) / 32), (unsigned)ca.chunks), block(32, kColGroups);
    const unsigned fin_grid = (unsigned)((N + 255) / 256);
    // Slot 0: a chain's first reduction (read by col_stage for the second);
    // slot 1: the last reduction (read by the write kernel).
    if (c0.rowop != 0) {
      col_stats_kernel<<<grid, block, 0, st>>>(ca, c0.rowop, 0);
      col_finalize_kernel<<<fin_grid, 256, 0, st>>>(ca, c0.rowop, c0.eps, 0, 0);
    }
    const int second = c0.rowop != 0 ? 1 : 0;
    col_stats_kernel<<<grid, block, 0, st>>>(ca, pg.rowop, second);
    col_finalize_kernel<<<fin_grid, 256, 0, st>>>(ca, pg.rowop, pg.eps, second, 1);
    col_write_kernel<<<grid, block, 0, st>>>(ca, o, out->ld, gamma, beta);
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
  }
  const bool vec = N % 1024 == 0 && (out->ld % 4) == 0 && aligned16(out->ptr) && (!bias || aligned16(bias)) &&
                   (!gamma || aligned16(gamma)) && (!beta || aligned16(beta));
  const bool vec_chain = vec && (!c0.gamma || aligned16(c0.gamma)) && (!c0.beta || aligned16(c0.beta));
  if (c0.rowop != 0 && !vec_chain) {
    const size_t smem = (size_t)N * sizeof(float);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(row_epilogue_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
      return CF_ERR_CUDA;
    row_epilogue_chain_kernel<<<(unsigned)M, 256, smem, st>>>(intermediate, N, o, out->ld, (int)N, pg, c0, bias,
                                                              gamma, beta, rv);
    return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
  }
  switch (vec ? N / 1024 : 0) {
    case 1: row_epilogue_reg_kernel<1><<<(unsigned)M, 256, 0, st>>>(intermediate, N, o, out->ld, (int)N, pg, c0, bias, gamma, beta, rv); break;
    case 2: row_epilogue_reg_kernel<2><<<(unsigned)M, 256, 0, st>>>(intermediate, N, o, out->ld, (int)N, pg, c0, bias, gamma, beta, rv); break;
    case 4: row_epilogue_reg_kernel<4><<<(unsigned)M, 256, 0, st>>>(intermediate, N, o, out->ld, (int)N, pg, c0, bias, gamma, beta, rv); break;
    case 8: row_epilogue_reg_kernel<8><<<(unsigned)M, 256, 0, st>>>(intermediate, N, o, out->ld, (int)N, pg, c0, bias, gamma, beta, rv); break;
    case 16: row_epilogue_reg_kernel<16><<<(unsigned)M, 256, 0, st>>>(intermediate, N, o, out->ld, (int)N, pg, c0, bias, gamma, beta, rv); break;
    default: {
      const size_t smem = (size_t)N * sizeof(float);
      if (smem > 48 * 1024 &&
          cudaFuncSetAttribute(row_epilogue_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
              cudaSuccess)
        return CF_ERR_CUDA;
      row_epilogue_kernel<<<(unsigned)M, 256, smem, st>>>(intermediate, N, o, out->ld, (int)N, pg, bias, gamma, beta, rv);
    }
  }
  return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

extern "C" cf_status cf_unfused_b2bgemm(const cf_matrix* A, const cf_matrix* W1, const cf_matrix* W2,
                                        const cf_b2b_desc* d, cf_matrix* out, float* s_buf, void* p_buf,
                                        void* stream) {
  if (!A || !W1 || !W2 || !d || !out || !s_buf || !p_buf) return CF_ERR_INVALID_ARG;
  if (d->version < 1 || d->version > CF_B2B_VERSION || d->batch < 1) return CF_ERR_INVALID_ARG;
  if (d->mid_op < CF_MID_RELU || d->mid_op > CF_MID_SCALE_SOFTMAX) return CF_ERR_INVALID_ARG;
  if (d->mid_op == CF_MID_SCALE_SOFTMAX && !(d->mid_scale > 0.0f)) return CF_ERR_INVALID_ARG;
  if ((d->out_dtype != CF_FP32 && d->out_dtype != CF_BF16) || out->dtype != d->out_dtype) return CF_ERR_INVALID_ARG;
  const int64_t M = A->rows, K = A->cols, N1 = W1->cols, N2 = W2->cols;
  if (W1->rows != K || W2->rows != N1 || out->rows != M || out->cols != N2) return CF_ERR_INVALID_ARG;
  if (N1 > 16384) return CF_ERR_UNSUPPORTED_SHAPE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t batch = d->batch;
  cf_status s = lt_gemm(A->ptr, A->ld, W1->ptr, W1->ld, W1->trans != 0, s_buf, N1, CUDA_R_32F, M, N1, K, batch,
                        d->strideA, d->strideW1, M * N1, st);
  if (s != CF_OK) return s;
  __nv_bfloat16* pb = static_cast<__nv_bfloat16*>(p_buf);
  const unsigned rows = (unsigned)(M * batch);
  switch (N1 % 1024 == 0 && aligned16(p_buf) && aligned16(s_buf) ? N1 / 1024 : 0) {
    case 1: mid_op_reg_kernel<1><<<rows, 256, 0, st>>>(s_buf, pb, (int)N1, d->mid_op, d->mid_scale); break;
    case 2: mid_op_reg_kernel<2><<<rows, 256, 0, st>>>(s_buf, pb, (int)N1, d->mid_op, d->mid_scale); break;
    case 4: mid_op_reg_kernel<4><<<rows, 256, 0, st>>>(s_buf, pb, (int)N1, d->mid_op, d->mid_scale); break;
    case 8: mid_op_reg_kernel<8><<<rows, 256, 0, st>>>(s_buf, pb, (int)N1, d->mid_op, d->mid_scale); break;
    case 16: mid_op_reg_kernel<16><<<rows, 256, 0, st>>>(s_buf, pb, (int)N1, d->mid_op, d->mid_scale); break;
    default: {
      const size_t smem = (size_t)N1 * sizeof(float);
      if (smem > 48 * 1024 &&
          cudaFuncSetAttribute(mid_op_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return CF_ERR_CUDA;
      mid_op_kernel<<<rows, 256, smem, st>>>(s_buf, pb, (int)N1, d->mid_op, d->mid_scale);
    }
  }
  if (cudaGetLastError() != cudaSuccess) return CF_ERR_CUDA;
  return lt_gemm(p_buf, N1, W2->ptr, W2->ld, W2->trans != 0, out->ptr, out->ld,
                 out->dtype == CF_BF16 ? CUDA_R_16BF : CUDA_R_32F, M, N2, N1, batch,
                 M * N1, d->strideW2, d->strideOut, st);
}
