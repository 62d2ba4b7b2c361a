// cf_gemm_epi_kernel.cuh -- the fused GEMM + epilogue kernel template (sm_103a),
// included by the translation units that instantiate it.
//
// The Stage-Stream Execution Model of the ComFuse review ("What carries the
// argument"): the GEMM's accumulator tile streams through the elementwise
// nodes while still on chip, and the trailing row reduction (LayerNorm,
// RMSNorm, softmax) is a stage boundary whose statistics are aggregated
// hierarchically.  Tile-strip locality (referee report, major comment 1
// [Sec. III, Eq. (1)]) means one output row depends only on the CTAs that
// share its 128-row strip.
//
// GB300 design (not the pages' Hopper/CUTLASS one):
//   * warp 0   : TMA producer -- A [128 x 64] and B [256 x 64] bf16 tiles,
//                128-byte swizzle, into a 4-stage shared-memory ring.
//   * warp 1   : TMEM allocator and single-thread tcgen05.mma issuer,
//                128 x 256 x 16 bf16 MMAs accumulating fp32 in TMEM; two
//                256-column accumulators so tile t+1's main loop overlaps
//                tile t's epilogue (the review's PingPong overlap, Sec. III-C).
//   * warps 2-5: epilogue.  tcgen05.ld's 32x32b shape gives each thread one
//                accumulator row, so the "intra-warp" level of the review's
//                three-level reduction is a register loop over the thread's
//                own columns; the activated values are written back to TMEM
//                so the normalisation pass does not recompute them.
//   * level 3  : CTAs sharing a row strip exchange per-row partial statistics
//                either through distributed shared memory inside one
//                thread-block cluster (<= 16 CTAs; peer-to-peer all-gather,
//                the review's "cross-broadcast" mode, Sec. III-A) or, when
//                the strip is wider than a cluster, through a small global
//                workspace of per-tile partials with bounded waits.
//   * output   : each epilogue warp stages a 32 x 32 fp32 block in swizzled
//                shared memory and writes it with a TMA store.
// The pre-normalisation tile never leaves the SM: only A, B, the vectors,
// the output and (for the wide-row fallback) 8 bytes per row per tile of
// statistics touch global memory.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "cf_internal.h"
#include "cf_ptx.cuh"

namespace cf {
namespace {

constexpr int kEpiWarps = 4;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kAStageBytes = kBM * kBK * 2;              // 16 KB
constexpr int kOutStageBytes = 32 * 32 * 4;              // 4 KB per epilogue warp
constexpr int kTmemCols = 2 * kBN;                       // two accumulators
constexpr int kNumVec = 5;                               // staged vector slices per tile

// Per-mode geometry.  CTA2: a CTA pair runs 256 x 256 MMAs (cta_group::2),
// each CTA holding its 128 rows of A and half (128 columns) of the B tile,
// so a stage is 32 KB and six fit; otherwise 48 KB stages, four of them.
template <bool CTA2>
struct Geo {
  static constexpr int kStages = CTA2 ? 6 : 4;
  static constexpr int kBStageBytes = (CTA2 ? kBN / 2 : kBN) * kBK * 2;
  static constexpr int kStageBytes = kAStageBytes + kBStageBytes;
  static constexpr int kOffOut = kStages * kStageBytes;
  static constexpr int kOffSlots = kOffOut + kEpiWarps * kOutStageBytes;  // float2 [2][128]
  static constexpr int kOffVec = kOffSlots + 2 * kBM * 8;                 // float [kNumVec][kBN]
  static constexpr int kOffEarly = kOffVec + kNumVec * kBN * 4;           // float [kEpiWarps][kBN]: early bias slices
  static constexpr int kOffBars = kOffEarly + kEpiWarps * kBN * 4;
  // barriers: full[S], empty[S], tfull[2], tempty[2], sfull[2][4], sempty[2][4], drain
  // ..., vec_free, vec_full, item[4], xdone[2]
  static constexpr int kNumBars = 2 * kStages + 2 + 2 + 8 + 8 + 1 + 2 + 4 + 2;
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;  // tmem base (u32), abort flag (i32), item slots (i32 [4])
  static constexpr int kSmemBytes = kOffMisc + 32 + 1024;   // + slack for the 1024-byte alignment
};

constexpr float kLog2e = 1.4426950408889634f;

// The tile's slices of the epilogue vectors, staged in shared memory once per
// tile: bias, gamma, beta, and the first reduction stage's gamma0, beta0.
enum VecSlot : int { VEC_BIAS = 0, VEC_GAMMA = 1, VEC_BETA = 2, VEC_GAMMA0 = 3, VEC_BETA0 = 4 };

enum OpKind : int { OP_BIAS = 1, OP_SCALE = 2, OP_RELU = 3, OP_GELU_TANH = 4, OP_ADD_RESIDUAL = 5 };

// tanh-GELU of two values: 0.5 x (1 + tanh(u)) == x * sigmoid(2u) ==
// x / (1 + exp(-2u)), u = sqrt(2/pi) (x + 0.044715 x^3); the polynomial and
// the scalings two per packed instruction.
__device__ __forceinline__ void gelu_tanh2(float& x0, float& x1) {
  float sq0 = x0, sq1 = x1, c0 = x0, c1 = x1;
  fmul2(sq0, sq1, x0, x1);                   // x^2
  fmul2(c0, c1, 0.044715f, 0.044715f);       // 0.044715 x
  ffma2(c0, c1, c0, c1, sq0, sq1, x0, x1);   // x + 0.044715 x^3
  fmul2(c0, c1, 0.7978845608028654f, 0.7978845608028654f);
  const float m = -2.0f * kLog2e;
  fmul2(c0, c1, m, m);
  float e0 = ex2_approx(c0), e1 = ex2_approx(c1);
  fadd2(e0, e1, 1.0f, 1.0f);
  x0 = __fdividef(x0, e0);
  x1 = __fdividef(x1, e1);
}

// Entries i..i+3 of a length-N fp32 vector (i a multiple of 4, x 16-byte
// aligned).  GUARD: the 32-column chunk holding them crosses column N (the
// ragged last tile of a row); entries at or past N read as zero and are
// never dereferenced.
template <bool GUARD>
__device__ __forceinline__ float4 ld4(const float* x, int i, int N) {
  if (!GUARD || i + 4 <= N) return __ldg(reinterpret_cast<const float4*>(x + i));
  float4 r = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  if (i < N) r.x = __ldg(x + i);
  if (i + 1 < N) r.y = __ldg(x + i + 1);
  if (i + 2 < N) r.z = __ldg(x + i + 2);
  return r;
}

// Columns j >= cv of a 32-column chunk lie past N: give them the value that
// leaves a row statistic unchanged (0 for sums, -inf for a max, the
// segment's reference for sums of squared deviations).
__device__ __forceinline__ void mask_tail(float (&v)[32], int cv, float fill) {
#pragma unroll
  for (int j = 0; j < 32; ++j)
    if (j >= cv) v[j] = fill;
}

// v[j] *= x[j] and v[j] += x[j] over a 32-column chunk, x the chunk's slice
// of a staged vector in shared memory (every lane reads the same address).
// Two columns per packed fp32x2 instruction: one epilogue warp runs per SM
// sub-partition, so the epilogue's time is its instruction count.
__device__ __forceinline__ void mul_vec(float (&v)[32], const float* x) {
  const float4* x4 = reinterpret_cast<const float4*>(x);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float4 g = x4[j];
    fmul2(v[4 * j + 0], v[4 * j + 1], g.x, g.y);
    fmul2(v[4 * j + 2], v[4 * j + 3], g.z, g.w);
  }
}
__device__ __forceinline__ void add_vec(float (&v)[32], const float* x) {
  const float4* x4 = reinterpret_cast<const float4*>(x);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float4 b = x4[j];
    fadd2(v[4 * j + 0], v[4 * j + 1], b.x, b.y);
    fadd2(v[4 * j + 2], v[4 * j + 3], b.z, b.w);
  }
}
// v[j] = v[j] * s + t for the whole chunk (s, t scalars).
__device__ __forceinline__ void scale_shift(float (&v)[32], float s, float t) {
#pragma unroll
  for (int j = 0; j < 32; j += 2) ffma2(v[j], v[j + 1], v[j], v[j + 1], s, s, t, t);
}

// Normalisation with the affine vectors: v = gamma (v sa + sh) (+ beta),
// two columns per packed instruction (the gamma product and the beta add
// in one fused multiply-add).
template <bool BETA>
__device__ __forceinline__ void norm_affine(float (&v)[32], const float* gamma, const float* beta, float sa,
                                            float sh) {
  const float4* g4 = reinterpret_cast<const float4*>(gamma);
  const float4* b4 = reinterpret_cast<const float4*>(beta);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float4 g = g4[j];
    const float4 b = BETA ? b4[j] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    ffma2(v[4 * j + 0], v[4 * j + 1], v[4 * j + 0], v[4 * j + 1], sa, sa, sh, sh);
    ffma2(v[4 * j + 2], v[4 * j + 3], v[4 * j + 2], v[4 * j + 3], sa, sa, sh, sh);
    if (BETA) {
      ffma2(v[4 * j + 0], v[4 * j + 1], v[4 * j + 0], v[4 * j + 1], g.x, g.y, b.x, b.y);
      ffma2(v[4 * j + 2], v[4 * j + 3], v[4 * j + 2], v[4 * j + 3], g.z, g.w, b.z, b.w);
    } else {
      fmul2(v[4 * j + 0], v[4 * j + 1], g.x, g.y);
      fmul2(v[4 * j + 2], v[4 * j + 3], g.z, g.w);
    }
  }
}

// Elementwise ops [o0, o1) of the program on 32 consecutive columns n.. of
// row m of the tile; bias_s: the chunk's slice of the staged bias.  GUARD:
// the chunk crosses column N (see ld4; the staged slices hold zeros there).
// COLS: the tile is a tile of P^T (column reductions): row m is column m of
// the output, the 32 columns are output rows n.., the bias is the row's own
// scalar bias_r and the residual is read transposed (R[n + j][m]; the lanes
// of a warp hold consecutive m, so each read is coalesced across the warp).
template <bool GUARD, bool COLS>
__device__ __forceinline__ void apply_program(const GemmEpiParams& p, float (&v)[32], int n, int m, int o0, int o1,
                                              const float* bias_s, float bias_r) {
  for (int o = o0; o < o1; ++o) {
    const int kind = p.op_kind[o];
    if (COLS && kind == OP_ADD_RESIDUAL) {
      if (m < p.M) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (!GUARD || n + j < p.N) {
            const long long idx = (long long)(n + j) * p.res_ld + m;
            v[j] += p.res_bf16 ? __uint_as_float((uint32_t)__ldg(static_cast<const uint16_t*>(p.res) + idx) << 16)
                               : __ldg(static_cast<const float*>(p.res) + idx);
          }
        }
      }
    } else if (kind == OP_ADD_RESIDUAL) {
      // Each thread owns one row: 128 (fp32) or 64 (bf16) contiguous bytes of
      // the residual row, read with 16-byte loads.  Rows past M (a ragged
      // last strip) are never stored, so they skip the read.
      if (m < p.M) {
        if (GUARD && p.res_bf16) {
          const uint16_t* rr = static_cast<const uint16_t*>(p.res) + (long long)m * p.res_ld;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (n + j < p.N) v[j] += __uint_as_float((uint32_t)__ldg(rr + n + j) << 16);
        } else if (GUARD) {
          const float* rr = static_cast<const float*>(p.res) + (long long)m * p.res_ld;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 r = ld4<true>(rr, n + 4 * j, p.N);
            v[4 * j + 0] += r.x;
            v[4 * j + 1] += r.y;
            v[4 * j + 2] += r.z;
            v[4 * j + 3] += r.w;
          }
        } else if (p.res_bf16) {
          const uint4* r4 = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.res) +
                                                           (long long)m * p.res_ld + n);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 w = __ldg(r4 + j);
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              fadd2(v[8 * j + 2 * e], v[8 * j + 2 * e + 1], __uint_as_float(ww[e] << 16),
                    __uint_as_float(ww[e] & 0xffff0000u));
          }
        } else {
          const float4* r4 = reinterpret_cast<const float4*>(static_cast<const float*>(p.res) +
                                                             (long long)m * p.res_ld + n);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 r = __ldg(r4 + j);
            fadd2(v[4 * j + 0], v[4 * j + 1], r.x, r.y);
            fadd2(v[4 * j + 2], v[4 * j + 3], r.z, r.w);
          }
        }
      }
    } else if (kind == OP_BIAS) {
      if (COLS) {
#pragma unroll
        for (int j = 0; j < 32; j += 2) fadd2(v[j], v[j + 1], bias_r, bias_r);
      } else {
        add_vec(v, bias_s);
      }
    } else if (kind == OP_SCALE) {
      const float s = p.op_scalar[o];
#pragma unroll
      for (int j = 0; j < 32; j += 2) fmul2(v[j], v[j + 1], s, s);
    } else if (kind == OP_RELU) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = fmaxf(v[j], 0.0f);
    } else if (kind == OP_GELU_TANH) {
#pragma unroll
      for (int j = 0; j < 32; j += 2) gelu_tanh2(v[j], v[j + 1]);
    }
  }
}

// Per-row statistics of a row segment and their merge (fixed order in every
// CTA, so all CTAs of a strip derive bit-identical row statistics).
//   LayerNorm: (mean, M2) over the segment's columns, merged with Chan et
//              al.'s pairwise update (counts: kBN, or fewer for the ragged
//              last tile of a row).
//   RMSNorm:   (sum x^2, 0), merged by addition.
//   softmax:   (max, sum exp(x - max)), merged by rescaling to the new max.
template <int ROWOP>
struct Stat {
  __device__ static float2 identity() {
    if (ROWOP == ROW_SOFTMAX) return make_float2(-INFINITY, 0.0f);
    return make_float2(0.0f, 0.0f);
  }
  // Merge segment b (of n_b columns) into a (of n_a columns).
  __device__ static float2 merge(float2 a, float2 b, float n_a, float n_b) {
    if (ROWOP == ROW_RMSNORM) return make_float2(a.x + b.x, 0.0f);
    if (ROWOP == ROW_SOFTMAX) {
      const float m = fmaxf(a.x, b.x);
      const float la = (a.y == 0.0f) ? 0.0f : a.y * ex2_approx((a.x - m) * kLog2e);
      const float lb = (b.y == 0.0f) ? 0.0f : b.y * ex2_approx((b.x - m) * kLog2e);
      return make_float2(m, la + lb);
    }
    // LayerNorm
    const float n = n_a + n_b;
    const float d = b.x - a.x;
    return make_float2(a.x + d * (n_b / n), a.y + b.y + d * d * (n_a * n_b / n));
  }
};

// Valid columns of N tile j: kBN, or N - j kBN for the ragged last tile.
template <bool RAG>
__device__ __forceinline__ float tile_cols(const GemmEpiParams& p, int j) {
  return RAG ? (float)min(kBN, p.N - j * kBN) : (float)kBN;
}

// Strip-wide merge of per-tile row statistics `st` through the workspace
// (the fallback exchange): publish, count arrivals (release), wait (bounded,
// acquire) for every tile of the strip, merge in tile order.
template <int R, bool RAG>
__device__ __forceinline__ bool global_exchange(const GemmEpiParams& p, float2* ws_stats, unsigned* ws_count,
                                                int strip, int tile, int row, int q, int lane,
                                                volatile int* abort_flag, const WaitCtx& wc, float2& st) {
  float2* wsrow = ws_stats + (size_t)strip * p.tiles_n * kBM + row;
  __stcg(wsrow + (size_t)tile * kBM, st);
  __threadfence();
  __syncwarp();
  unsigned* cnt = ws_count + strip * 4 + q;
  if (lane == 0) red_release_gpu_add(cnt, 1u);
  bool ok = true;
  if (ld_acquire_gpu(cnt) < (unsigned)p.tiles_n) {
    const long long t0 = clock64();
    while (ld_acquire_gpu(cnt) < (unsigned)p.tiles_n) {
      __nanosleep(64);
      if (*abort_flag) { ok = false; break; }
      if (clock64() - t0 > p.timeout_cycles) { record_timeout(wc); ok = false; break; }
    }
  }
  if (!__all_sync(0xffffffffu, ok)) return false;
  float2 tot = __ldcg(wsrow);
  float n_acc = tile_cols<RAG>(p, 0);
  for (int j = 1; j < p.tiles_n; ++j) {
    const float nb = tile_cols<RAG>(p, j);
    tot = Stat<R>::merge(tot, __ldcg(wsrow + (size_t)j * kBM), n_acc, nb);
    n_acc += nb;
  }
  st = tot;
  return true;
}

// Pass 1 (the elementwise program applied and written back to TMEM, the
// first local statistic) and pass 2 (the second statistic about the
// segment's own mean or max) over one tile row segment: the tile's row
// statistics.  vsm: the tile's staged vector slices [kNumVec][kBN] (only the
// bias slice, VEC_BIAS = 0, is read when ROWOP0 == ROW_NONE); m: the row of
// P (of P^T with COLS).  Chained programs (ROWOP0) first normalise with the
// first stage's (sc0, sh0) and affine vectors.
template <int ROWOP, bool RAG, bool COLS, int ROWOP0>
__device__ __forceinline__ float2 tile_stats(const GemmEpiParams& p, uint32_t taddr, int nch, int nv, int n0, int m,
                                             const float* vsm, float r_bias, float r_gamma0, float r_beta0,
                                             float sc0, float sh0) {
  // One pass: the elementwise program (its result kept in TMEM) and the
  // segment's statistics together, so a tile publishes them after a single
  // walk over its columns.  LayerNorm: sums of x - k and (x - k)^2 about a
  // shift k, the segment's first value (the shifted-data form of the
  // variance, exact for any k and accurate while k is near the mean);
  // softmax: the online maximum and the sum of exp(x - max), rescaled when
  // the maximum grows; RMSNorm: the sum of squares.  Each sum is kept in four
  // partial accumulators (element j in accumulator j mod 4, two per packed
  // fp32x2 instruction): one epilogue warp runs per SM sub-partition, so a
  // single chain of dependent adds would expose its latency.
  float s1p[4] = {0.0f, 0.0f, 0.0f, 0.0f}, s2p[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  float shift = 0.0f;                         // LayerNorm: k
  float run_max = -INFINITY, run_sum = 0.0f;  // softmax
#pragma unroll 1
  for (int c = 0; c < nch; ++c) {
    float v[32];
    tmem_ld32(taddr + c * 32, v);
    tmem_wait_ld();
    const int n = n0 + c * 32;
    const bool tail = RAG && n + 32 > p.N;
    if constexpr (ROWOP0 != ROW_NONE) {
      scale_shift(v, sc0, sh0);
      if (COLS) {
        scale_shift(v, r_gamma0, ROWOP0 == ROW_LAYERNORM ? r_beta0 : 0.0f);
      } else {
        if (p.gamma0) mul_vec(v, vsm + VEC_GAMMA0 * kBN + c * 32);
        if (ROWOP0 == ROW_LAYERNORM && p.beta0) add_vec(v, vsm + VEC_BETA0 * kBN + c * 32);
      }
    }
    if (ROWOP0 != ROW_NONE || p.n_ops > 0) {
      const int o0 = ROWOP0 != ROW_NONE ? p.n_ops0 : 0;
      const float* bs = vsm + VEC_BIAS * kBN + c * 32;
      if (tail) apply_program<true, COLS>(p, v, n, m, o0, p.n_ops, bs, r_bias);
      else apply_program<false, COLS>(p, v, n, m, o0, p.n_ops, bs, r_bias);
      tmem_st32(taddr + c * 32, v);
    }
    if (ROWOP == ROW_LAYERNORM && c == 0) shift = v[0];  // column n0 < N: always valid
    // Columns past N leave every statistic unchanged.
    if (tail) mask_tail(v, p.N - n, ROWOP == ROW_SOFTMAX ? -INFINITY : ROWOP == ROW_LAYERNORM ? shift : 0.0f);
    if (ROWOP == ROW_RMSNORM) {
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        ffma2(s1p[0], s1p[1], v[j], v[j + 1], v[j], v[j + 1], s1p[0], s1p[1]);
        ffma2(s1p[2], s1p[3], v[j + 2], v[j + 3], v[j + 2], v[j + 3], s1p[2], s1p[3]);
      }
    } else if (ROWOP == ROW_LAYERNORM) {
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        float d0 = v[j], d1 = v[j + 1], d2 = v[j + 2], d3 = v[j + 3];
        fadd2(d0, d1, -shift, -shift);
        fadd2(d2, d3, -shift, -shift);
        fadd2(s1p[0], s1p[1], d0, d1);
        fadd2(s1p[2], s1p[3], d2, d3);
        ffma2(s2p[0], s2p[1], d0, d1, d0, d1, s2p[0], s2p[1]);
        ffma2(s2p[2], s2p[3], d2, d3, d2, d3, s2p[2], s2p[3]);
      }
    } else {  // softmax
      float cm[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
      for (int j = 4; j < 32; j += 4) {
#pragma unroll
        for (int k = 0; k < 4; ++k) cm[k] = fmaxf(cm[k], v[j + k]);
      }
      const float m_new = fmaxf(run_max, fmaxf(fmaxf(cm[0], cm[1]), fmaxf(cm[2], cm[3])));
      if (m_new > run_max) run_sum *= ex2_approx((run_max - m_new) * kLog2e);  // 0 while run_max is -inf
      const float sh = -m_new * kLog2e;
      float cs[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        float d0 = v[j], d1 = v[j + 1], d2 = v[j + 2], d3 = v[j + 3];
        ffma2(d0, d1, d0, d1, kLog2e, kLog2e, sh, sh);
        ffma2(d2, d3, d2, d3, kLog2e, kLog2e, sh, sh);
        fadd2(cs[0], cs[1], ex2_approx(d0), ex2_approx(d1));
        fadd2(cs[2], cs[3], ex2_approx(d2), ex2_approx(d3));
      }
      run_sum += (cs[0] + cs[1]) + (cs[2] + cs[3]);
      run_max = m_new;
    }
  }
  if (ROWOP0 != ROW_NONE || p.n_ops > 0) tmem_wait_st();
  float2 st;
  if (ROWOP == ROW_RMSNORM) {
    st = make_float2((s1p[0] + s1p[1]) + (s1p[2] + s1p[3]), 0.0f);
  } else if (ROWOP == ROW_LAYERNORM) {
    const float cnt = RAG ? (float)nv : (float)kBN;
    const float s1 = (s1p[0] + s1p[1]) + (s1p[2] + s1p[3]);
    const float s2 = (s2p[0] + s2p[1]) + (s2p[2] + s2p[3]);
    const float dm = s1 / cnt;                                     // mean - k
    st = make_float2(shift + dm, fmaxf(s2 - s1 * dm, 0.0f));      // (mean, sum of squared deviations)
  } else {
    st = make_float2(run_max, run_sum);
  }
  return st;
}

struct Work {
  int i, step, end, rank, tiles_n;
  __device__ bool valid() const { return i < end; }
  __device__ void next() { i += step; }
};

template <int XMODE>
__device__ __forceinline__ Work make_work(const GemmEpiParams& p) {
  Work w;
  w.tiles_n = p.tiles_n;
  if (XMODE == X_CLUSTER) {
    w.i = (int)cluster_id_x();
    w.step = (int)num_clusters_x();
    w.end = p.strips;
    w.rank = (int)cluster_ctarank();
  } else if (p.pair) {
    // A pair of CTAs takes strips (2 sp, 2 sp + 1) of the same N tile.
    w.i = (int)cluster_id_x();
    w.step = (int)num_clusters_x();
    w.end = p.pair_items;
    w.rank = (int)cluster_ctarank();
  } else {
    w.i = blockIdx.x;
    w.step = gridDim.x;
    w.end = p.num_items;
    w.rank = 0;
  }
  return w;
}

template <int XMODE>
__device__ __forceinline__ void item_coords(const GemmEpiParams& p, const Work& w, int& strip, int& tile) {
  if (XMODE == X_CLUSTER) {
    strip = w.i;
    tile = w.rank;
  } else if (p.pair) {
    const int sp = w.i / w.tiles_n;
    tile = w.i - sp * w.tiles_n;
    if (sp & 1) tile = w.tiles_n - 1 - tile;  // serpentine, see below
    strip = 2 * sp + w.rank;
  } else {
    strip = w.i / w.tiles_n;
    tile = w.i - strip * w.tiles_n;
    if (strip & 1) tile = w.tiles_n - 1 - tile;
  }
}
// Serpentine tile order: consecutive (pairs of) strips walk the N tiles in
// opposite directions, so a strip starts on the B tiles its predecessor read
// last, while they are still in L2.  When B is about the size of L2 (the
// 4096 x 16384 softmax head: 128 MB), a plain order re-reads all of B from
// DRAM for every strip.  Items of a strip stay contiguous, so the row
// statistics exchange keeps its strip-major schedule.

// Workspace exchange (single-stage programs), when the host asks for it:
// work items are claimed in the strip-major order above as tickets from a
// global counter, so only CTAs that are running ever hold items (a
// statically assigned item of a CTA that is not resident -- another kernel
// holds its SM -- stalls its strip-mates until that CTA starts, or until
// the bounded waits give up).  The static assignment is faster on a GPU of
// its own (its rounds keep the tiles of a strip in lockstep; claims made as
// strips complete drift off the strip boundaries), so it stays the default.  A worker claims an item
// once its item two back has finished its strip exchange, and while an item
// waits for its strip the epilogue publishes the statistics of the worker's
// next item (see the epilogue), so a worker holding two tiles of one strip
// never waits for itself; a strip's tiles then fit in twice the workers
// that run, whatever the launched grid.
__device__ __forceinline__ void ticket_coords(const GemmEpiParams& p, int idx, int rank, int& strip, int& tile) {
  const int T = p.tiles_n;
  const int u = idx / T;  // row-strip unit: a strip, or a strip pair with CTA pairs
  tile = idx - u * T;
  if (u & 1) tile = T - 1 - tile;
  strip = p.pair ? 2 * u + rank : u;
}

// ROWOP0 != ROW_NONE: the program has two chained row reductions, ROWOP0
// (LayerNorm or RMSNorm) then ROWOP; only the per-tile and workspace
// exchanges are instantiated for it.
//
// RAG: N is not a multiple of kBN, so the last tile of each row is ragged.
// The full-tile instantiations compile every ragged-column guard away.
//
// COLS: column reductions (over the first dimension of the user's P).  The
// host swaps the operands, so the kernel computes tiles of P^T = B^T A^T and
// runs the same row machinery over them (the complementary strip: all tiles
// of one column block of P share a row strip of P^T); the vectors become
// per-row scalars and the output tiles are stored transposed.
template <int ROWOP, int XMODE, bool CTA2, bool RAG, bool COLS, int ROWOP0 = ROW_NONE>
__global__ void __launch_bounds__(kThreads, 1) gemm_epi_kernel(const __grid_constant__ GemmEpiParams p) {
  using G = Geo<CTA2>;
  constexpr int kStages = G::kStages, kStageBytes = G::kStageBytes, kOffOut = G::kOffOut,
                kOffSlots = G::kOffSlots, kOffBars = G::kOffBars, kOffMisc = G::kOffMisc;
  constexpr int kOffStages = 0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // CTA2: rank 0 of the pair issues every MMA ("leader").
  const uint32_t pair_rank = CTA2 ? cluster_ctarank() : 0u;
  const bool leader = pair_rank == 0;

  auto bar = [&](int idx) -> uint32_t { return sbase + kOffBars + 8 * idx; };
  const int BAR_FULL = 0, BAR_EMPTY = kStages, BAR_TFULL = 2 * kStages, BAR_TEMPTY = 2 * kStages + 2;
  const int BAR_SFULL = 2 * kStages + 4, BAR_SEMPTY = 2 * kStages + 12, BAR_DRAIN = 2 * kStages + 20;
  const int BAR_VFREE = 2 * kStages + 21, BAR_VFULL = 2 * kStages + 22, BAR_ITEM = 2 * kStages + 23,
            BAR_XDONE = 2 * kStages + 27;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  // Tickets: the claimed ticket of local item t sits in slot t & 3 (filled
  // when item t - 2 has finished its exchange, read by every role of both
  // CTAs of a pair before item t - 2 releases its accumulator).
  volatile int* item_slot = reinterpret_cast<volatile int*>(smem + kOffMisc + 8);
  const int sched_items = p.pair ? p.pair_items : p.num_items;
  const Work w0 = make_work<XMODE>(p);
  // Work items from tickets (the workspace exchange of single-stage
  // programs, when the host asks for them: see its launch rules); otherwise
  // the static strip-major assignment.
  constexpr bool kTicketsOk = XMODE == X_GLOBAL && ROWOP0 == ROW_NONE;
  const bool tickets = kTicketsOk && p.tickets != 0;
  const WaitCtx wc{p.timeout_cycles, abort_flag, p.status};

  int cn = 1;
  if (XMODE == X_CLUSTER) cn = p.tiles_n;

  // The tensor-map fetches start before the barrier set-up, which they
  // overlap (the first TMA load waits for its map).
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmA);
    tma_prefetch_desc(&p.tmB);
    tma_prefetch_desc(&p.tmOut);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(BAR_FULL + s), 1);
      mbar_init(bar(BAR_EMPTY + s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar(BAR_TFULL + a), 1);
      // CTA2: the leader's barrier collects both CTAs' epilogue warps.
      mbar_init(bar(BAR_TEMPTY + a), CTA2 ? 2 * kEpiWarps : kEpiWarps);
    }
    for (int k = 0; k < 8; ++k) {
      mbar_init(bar(BAR_SFULL + k), cn);
      mbar_init(bar(BAR_SEMPTY + k), cn);
    }
    mbar_init(bar(BAR_DRAIN), 1);
    mbar_init(bar(BAR_VFREE), kEpiWarps);
    mbar_init(bar(BAR_VFULL), kEpiWarps);
    for (int i = 0; i < 4; ++i) mbar_init(bar(BAR_ITEM + i), 1);
    mbar_init(bar(BAR_XDONE), kEpiWarps);  // this CTA's epilogue warps
    mbar_init(bar(BAR_XDONE + 1), kEpiWarps);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    if (CTA2) {
      tmem_alloc_pair(smem_u32(tmem_holder), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_holder), kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (XMODE == X_CLUSTER || CTA2) cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int kblocks = (p.K + kBK - 1) / kBK;  // the last block is zero-filled past K

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, issued = 0;
      bool ok = true;
      // B tiles are reread by every strip: keep them in L2 ahead of the
      // streamed output.
      const uint64_t b_policy = l2_policy_evict_last();
      // Tickets (the leader of a pair claims for both CTAs): claim local item
      // tn once item tn - 2 (the last item on accumulator tn & 1) has
      // finished its strip exchange -- every tile of its strip has been
      // claimed by then, so item tn belongs to another strip and item tn - 2
      // never waits for it -- and hand it to this CTA's MMA and epilogue
      // roles (and to the pair's peer).  Claims are made as late as that:
      // claiming earlier spreads the start of a strip's tiles over time and
      // lengthens the exchange waits (measured: claiming the next item while
      // the current one's stages were still being issued cut GELU + RMSNorm
      // 8192 x 4096 x 4096 from ~1490 to ~1020 TFLOP/s).
      int claimed = -1;  // the last local item claimed
      auto claim = [&](int tn) {
        int v = (int)atomicAdd(p.ws_ticket, 1u);
        if (v >= sched_items) v = -1;  // no work left
        item_slot[tn & 3] = v;
        if (CTA2) {
          st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<int*>(item_slot) + (tn & 3)), 1u), (uint32_t)v);
          mbar_arrive_cluster(bar(BAR_ITEM + (tn & 3)), 1u);
        }
        mbar_arrive(bar(BAR_ITEM + (tn & 3)));
        claimed = tn;
      };
      for (int t = 0; ok; ++t) {
        int strip, tile;
        if (tickets) {
          int idx;
          if (leader) {
            if (claimed < t) {
              if (!mbar_wait(bar(BAR_XDONE + (t & 1)), ((t >> 1) & 1) ^ 1, wc)) { ok = false; break; }
              claim(t);
            }
            idx = item_slot[t & 3];
          } else {
            if (!mbar_wait<true>(bar(BAR_ITEM + (t & 3)), (t >> 2) & 1, wc)) { ok = false; break; }
            idx = item_slot[t & 3];
          }
          if (idx < 0) break;
          ticket_coords(p, idx, (int)pair_rank, strip, tile);
        } else {
          Work w = w0;
          w.i += t * w.step;
          if (!w.valid()) break;
          item_coords<XMODE>(p, w, strip, tile);
        }
        const int m0 = strip * kBM, n0 = tile * kBN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(bar(BAR_EMPTY + stage), phase ^ 1, wc)) { ok = false; break; }
          const uint32_t sa = sbase + kOffStages + stage * kStageBytes;
          const uint32_t sb = sa + kAStageBytes;
          const uint32_t fb = bar(BAR_FULL + stage);
          if (CTA2) {
            // Both CTAs' bytes land on the leader's "full" barrier.
            const uint32_t fbl = mapa_shared(fb, 0);
            if (leader) mbar_arrive_expect_tx(fb, 2 * kStageBytes);
            tma_load_2d_pair(sa, &p.tmA, fbl, kb * kBK, m0);
            const int nb0 = n0 + (kBN / 2) * (int)pair_rank;  // this CTA's half of the B tile
            if (p.b_mn_major) {
              tma_load_2d_pair_hint(sb, &p.tmB, fbl, nb0, kb * kBK, b_policy);
              tma_load_2d_pair_hint(sb + 64 * kBK * 2, &p.tmB, fbl, nb0 + 64, kb * kBK, b_policy);
            } else {
              tma_load_2d_pair_hint(sb, &p.tmB, fbl, kb * kBK, nb0, b_policy);
            }
          } else {
            mbar_arrive_expect_tx(fb, kStageBytes);
            tma_load_2d(sa, &p.tmA, fb, kb * kBK, m0);
            if (p.b_mn_major) {
#pragma unroll
              for (int i = 0; i < kBN / 64; ++i)
                tma_load_2d(sb + i * (64 * kBK * 2), &p.tmB, fb, n0 + 64 * i, kb * kBK);
            } else {
              tma_load_2d(sb, &p.tmB, fb, kb * kBK, n0);
            }
          }
          ++issued;
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
      if (CTA2) {
        // The leader's MMA releases reach this CTA's barriers asynchronously:
        // wait until every stage's last release has landed before exiting
        // (after an abort they may never come: stop at the abort flag).
        for (int s2 = 0; s2 < kStages; ++s2) {
          if (!mbar_wait<false, true>(bar(BAR_EMPTY + stage), phase ^ 1, wc)) break;
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        // A pair's loads complete on the leader's barrier only, so after an
        // abort they are waited for at the end of the kernel (settle).
      } else {
        drain_ring(bar(BAR_FULL), kStages, issued, wc);  // no load of this CTA is still in flight
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && leader) {
      const uint32_t idesc = idesc_bf16_f32(CTA2 ? 2 * kBM : kBM, kBN, (uint32_t)p.b_mn_major);
      // Stage-0 descriptors; per 16 K elements A advances 32 bytes, B 32
      // bytes (K-major) or 16 rows = 2048 bytes (MN-major: 64-column atoms
      // 8 KB apart, 8-row groups 1 KB apart).
      const SDesc da = sdesc_sw128(sbase + kOffStages, 16, 1024);
      const SDesc db = sdesc_sw128(sbase + kOffStages + kAStageBytes, p.b_mn_major ? 64 * kBK * 2 : 16, 1024);
      const uint32_t b_step = p.b_mn_major ? (2048u >> 4) : (32u >> 4);
      uint32_t stage = 0, phase = 0;
      int t = 0;
      bool ok = true;
      for (;; ++t) {
        const int acc = t & 1;
        // CTA2: the peer's epilogue arrives remotely, so acquire at cluster scope.
        if (!mbar_wait<CTA2>(bar(BAR_TEMPTY + acc), ((t >> 1) & 1) ^ 1, wc)) { ok = false; break; }
        if (tickets) {
          if (!mbar_wait(bar(BAR_ITEM + (t & 3)), (t >> 2) & 1, wc)) { ok = false; break; }
          if (item_slot[t & 3] < 0) break;  // no work left
        } else {
          if (w0.i + t * w0.step >= w0.end) break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * kBN);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(bar(BAR_FULL + stage), phase, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_lo = da.lo + stage * (kStageBytes >> 4);
          const uint32_t b_lo = db.lo + stage * (kStageBytes >> 4);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            if (CTA2) mma_ss_pair(d, a_lo + kk * 2, da.hi, b_lo + kk * b_step, db.hi, idesc, (kb | kk) != 0 ? 1u : 0u);
            else mma_ss(d, a_lo + kk * 2, da.hi, b_lo + kk * b_step, db.hi, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          if (CTA2) mma_commit_pair(bar(BAR_EMPTY + stage), 0x3);  // frees the stage in both CTAs
          else mma_commit(bar(BAR_EMPTY + stage));
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        if (CTA2) mma_commit_pair(bar(BAR_TFULL + acc), 0x3);
        else mma_commit(bar(BAR_TFULL + acc));
      }
      // Drain: every MMA issued above has completed before TMEM is freed.
      if (CTA2) mma_commit_pair(bar(BAR_DRAIN), 0x1);
      else mma_commit(bar(BAR_DRAIN));
      mbar_wait<false, false>(bar(BAR_DRAIN), 0, wc);
      if (CTA2 && ok) {
        // Every remote "accumulator empty" arrival from the peer has landed.
        for (int t2 = t; t2 < t + 2; ++t2)
          if (!mbar_wait<true, true>(bar(BAR_TEMPTY + (t2 & 1)), ((t2 >> 1) & 1) ^ 1, wc)) break;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;             // TMEM lane quarter this warp may access
    const int row = 32 * q + lane;      // row within the tile
    const uint32_t out_buf = sbase + kOffOut + (warp - 2) * kOutStageBytes;
    // The output is streamed out once: let it leave L2 first, keeping the
    // operand tiles the next items reread.
    const uint64_t out_policy = l2_policy_evict_first();
    uint8_t* out_ptr = smem + kOffOut + (warp - 2) * kOutStageBytes;
    float2* slots = reinterpret_cast<float2*>(smem + kOffSlots);
    float* vsm = reinterpret_cast<float*>(smem + G::kOffVec);  // [kNumVec][kBN] this tile's vector slices
    const bool stage_vec = !COLS && (p.bias || p.gamma || p.beta || p.gamma0 || p.beta0);
    // Workspace exchange: publishing an item's statistics to its strip.
    auto publish = [&](int strip_, int tile_, float2 st_) {
      float2* wsr = p.ws_stats + (size_t)strip_ * p.tiles_n * kBM + row;
      __stcg(wsr + (size_t)tile_ * kBM, st_);
      __threadfence();
      __syncwarp();
      if (lane == 0) red_release_gpu_add(p.ws_count + strip_ * 4 + q, 1u);
    };
    // Tickets: while item t waits for its strip, this warp publishes the
    // statistics of its next item t + 1 as soon as that item's main loop is
    // done, when t + 1 is a tile of the same strip.  The epilogue handles a
    // worker's items in order: without this the first tile would wait for
    // the second's statistics, which are published only after the first
    // finishes.  Item t + 1's main loop needs only the accumulator that
    // item t - 1 has released, so its statistics never wait on an exchange.
    // (A next item of another strip is never needed: along any chain of
    // waits between different strips the strips only go down in the
    // strip-major ticket order, and the lowest incomplete strip waits for
    // nobody.)  The bias slice comes from the global vector into this warp's
    // own buffer (the shared staging belongs to item t).  The barriers are
    // probed without blocking (test_wait), so the wait keeps watching its
    // strip's counter.
    int early_t = -1;
    float2 early_st = make_float2(0.0f, 0.0f);
    int checked_t = -1;  // the next item was looked at and needs no early statistics
    float* ebuf = reinterpret_cast<float*>(smem + G::kOffEarly) + (warp - 2) * kBN;
    auto try_early = [&](int tn, int strip_now) {
      const int an = tn & 1;
      const uint32_t par = (uint32_t)((tn >> 1) & 1), ipar = (uint32_t)((tn >> 2) & 1);
      if (!__all_sync(0xffffffffu, CTA2 ? mbar_test_wait_cluster(bar(BAR_ITEM + (tn & 3)), ipar)
                                        : mbar_test_wait(bar(BAR_ITEM + (tn & 3)), ipar)))
        return;
      const int idx = item_slot[tn & 3];
      int strip1, tile1;
      if (idx >= 0) ticket_coords(p, idx, (int)pair_rank, strip1, tile1);
      if (idx < 0 || strip1 != strip_now) {
        checked_t = tn;  // no next item, or one of another strip
        return;
      }
      if (!__all_sync(0xffffffffu, mbar_test_wait(bar(BAR_TFULL + an), par))) return;
      tc_fence_after();
      const int m1 = strip1 * kBM, n1 = tile1 * kBN;
      const int nv1 = RAG ? min(kBN, p.N - n1) : kBN;
      const int nch1 = RAG ? (nv1 + 31) >> 5 : kBN / 32;
      float rb = 0.0f;
      if (COLS) {
        if (p.bias && m1 + row < p.M) rb = __ldg(p.bias + m1 + row);
      } else if (p.bias) {
        for (int c4 = 4 * lane; c4 < kBN; c4 += 128) *reinterpret_cast<float4*>(ebuf + c4) = ld4<RAG>(p.bias, n1 + c4, p.N);
        __syncwarp();
      }
      const uint32_t taddr1 = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(an * kBN);
      const float2 st1 = tile_stats<ROWOP, RAG, COLS, ROW_NONE>(p, taddr1, nch1, nv1, n1, m1 + row, ebuf, rb, 1.0f,
                                                                0.0f, 1.0f, 0.0f);
      publish(strip1, tile1, st1);
      early_t = tn;
      early_st = st1;
    };
    int t = 0;
    for (;; ++t) {
      int strip, tile;
      if (tickets) {
        // CTA2: the leader fills the peer's slot remotely (cluster scope).
        if (!__all_sync(0xffffffffu, mbar_wait<CTA2>(bar(BAR_ITEM + (t & 3)), (t >> 2) & 1, wc))) break;
        const int idx = item_slot[t & 3];
        if (idx < 0) break;
        ticket_coords(p, idx, (int)pair_rank, strip, tile);
      } else {
        Work w = w0;
        w.i += t * w.step;
        if (!w.valid()) break;
        item_coords<XMODE>(p, w, strip, tile);
      }
      const int m0 = strip * kBM, n0 = tile * kBN;
      const int nv = RAG ? min(kBN, p.N - n0) : kBN;  // valid columns: fewer in a ragged last tile
      const int nch = RAG ? (nv + 31) >> 5 : kBN / 32;  // 32-column chunks holding them
      const int acc = t & 1;
      // Stage the tile's vector slices (zeros past N) while its main loop
      // runs: one round trip to L2 per tile instead of one per chunk and
      // pass.  Every epilogue warp must be done with the previous tile's
      // slices first (vec_free); all four fill, then wait for vec_full.
      // (Programs without vectors, e.g. scale + softmax, skip all of it.)
      if (stage_vec) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar(BAR_VFREE), (t & 1) ^ 1, wc))) break;
        for (int i = lane + 32 * (warp - 2); i < kNumVec * (kBN / 4); i += 32 * kEpiWarps) {
          const int vi = i / (kBN / 4), c4 = 4 * (i - vi * (kBN / 4));
          const float* src = vi == VEC_BIAS ? p.bias : vi == VEC_GAMMA ? p.gamma : vi == VEC_BETA ? p.beta
                           : vi == VEC_GAMMA0 ? p.gamma0 : p.beta0;
          if (src) *reinterpret_cast<float4*>(vsm + vi * kBN + c4) = ld4<RAG>(src, n0 + c4, p.N);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_VFULL));
        if (!__all_sync(0xffffffffu, mbar_wait(bar(BAR_VFULL), t & 1, wc))) break;
      }
      // COLS: this thread's row is one column of the output; its vector
      // entries are scalars (rows past M keep the neutral values).
      float r_bias = 0.0f, r_gamma = 1.0f, r_beta = 0.0f, r_gamma0 = 1.0f, r_beta0 = 0.0f;
      if (COLS && m0 + row < p.M) {
        const int i = m0 + row;
        if (p.bias) r_bias = __ldg(p.bias + i);
        if (p.gamma) r_gamma = __ldg(p.gamma + i);
        if (p.beta) r_beta = __ldg(p.beta + i);
        if (p.gamma0) r_gamma0 = __ldg(p.gamma0 + i);
        if (p.beta0) r_beta0 = __ldg(p.beta0 + i);
      }
      if (!__all_sync(0xffffffffu, mbar_wait(bar(BAR_TFULL + acc), (t >> 1) & 1, wc))) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * kBN);

      // Chained programs: the first reduction stage.  Its elementwise ops
      // [0, n_ops0) are applied and written back to TMEM, its statistics
      // are merged across the strip (same exchange as the last stage), and
      // pass 1 below normalises with (sc0, sh0) and its affine vectors
      // before the ops that follow it.
      float sc0 = 1.0f, sh0 = 0.0f;
      if constexpr (ROWOP0 != ROW_NONE) {
        // One pass, as in tile_stats: the sum of squares (RMSNorm), or the
        // sums of x - k and (x - k)^2 about the segment's first value k
        // (LayerNorm), in four partial accumulators.
        float s1p[4] = {0.0f, 0.0f, 0.0f, 0.0f}, s2p[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        float shift = 0.0f;
#pragma unroll 1
        for (int c = 0; c < nch; ++c) {
          float v[32];
          tmem_ld32(taddr + c * 32, v);
          tmem_wait_ld();
          const int n = n0 + c * 32;
          const bool tail = RAG && n + 32 > p.N;
          if (p.n_ops0 > 0) {
            const float* bs = vsm + VEC_BIAS * kBN + c * 32;
            if (tail) apply_program<true, COLS>(p, v, n, m0 + row, 0, p.n_ops0, bs, r_bias);
            else apply_program<false, COLS>(p, v, n, m0 + row, 0, p.n_ops0, bs, r_bias);
            tmem_st32(taddr + c * 32, v);
          }
          if (ROWOP0 == ROW_LAYERNORM && c == 0) shift = v[0];
          if (tail) mask_tail(v, p.N - n, ROWOP0 == ROW_LAYERNORM ? shift : 0.0f);
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            if (ROWOP0 == ROW_RMSNORM) {
              ffma2(s1p[0], s1p[1], v[j], v[j + 1], v[j], v[j + 1], s1p[0], s1p[1]);
              ffma2(s1p[2], s1p[3], v[j + 2], v[j + 3], v[j + 2], v[j + 3], s1p[2], s1p[3]);
            } else {
              float d0 = v[j], d1 = v[j + 1], d2 = v[j + 2], d3 = v[j + 3];
              fadd2(d0, d1, -shift, -shift);
              fadd2(d2, d3, -shift, -shift);
              fadd2(s1p[0], s1p[1], d0, d1);
              fadd2(s1p[2], s1p[3], d2, d3);
              ffma2(s2p[0], s2p[1], d0, d1, d0, d1, s2p[0], s2p[1]);
              ffma2(s2p[2], s2p[3], d2, d3, d2, d3, s2p[2], s2p[3]);
            }
          }
        }
        const float s1 = (s1p[0] + s1p[1]) + (s1p[2] + s1p[3]);
        if (p.n_ops0 > 0) tmem_wait_st();
        float2 st0;
        if (ROWOP0 == ROW_RMSNORM) {
          st0 = make_float2(s1, 0.0f);
        } else {
          const float s2 = (s2p[0] + s2p[1]) + (s2p[2] + s2p[3]);
          const float dm = s1 / (RAG ? (float)nv : (float)kBN);
          st0 = make_float2(shift + dm, fmaxf(s2 - s1 * dm, 0.0f));
        }
        if (XMODE == X_GLOBAL &&
            !global_exchange<ROWOP0, RAG>(p, p.ws_stats0, p.ws_count0, strip, tile, row, q, lane, abort_flag, wc, st0))
          break;
        if (ROWOP0 == ROW_RMSNORM) {
          sc0 = rsqrtf(st0.x / (float)p.N + p.eps0);
        } else {
          sc0 = rsqrtf(st0.y / (float)p.N + p.eps0);
          sh0 = -st0.x * sc0;
        }
      }

      float2 st = Stat<ROWOP>::identity();
      float scale_a = 1.0f, shift_a = 0.0f;  // y = gamma * (x * scale_a + shift_a) (+ beta)
      if (ROWOP != ROW_NONE) {
        const bool pre = tickets && early_t == t;  // published while the previous item waited
        if (pre) st = early_st;
        else st = tile_stats<ROWOP, RAG, COLS, ROWOP0>(p, taddr, nch, nv, n0, m0 + row, vsm, r_bias, r_gamma0, r_beta0,
                                                       sc0, sh0);

        // Level 3: statistics of the whole row across the CTAs of the strip.
        if (XMODE == X_CLUSTER) {
          const int b = t & 1;
          const uint32_t u = (uint32_t)(t >> 1);
          const uint32_t slot_addr = smem_u32(slots + b * kBM + row);
          if (!__all_sync(0xffffffffu, mbar_wait<true>(bar(BAR_SEMPTY + b * 4 + q), (u & 1) ^ 1, wc))) break;
          slots[b * kBM + row] = st;
          __syncwarp();
          if (lane == 0) {
            fence_acq_rel_cluster();
            for (int r = 0; r < cn; ++r) mbar_arrive_cluster(bar(BAR_SFULL + b * 4 + q), (uint32_t)r);
          }
          if (!__all_sync(0xffffffffu, mbar_wait<true>(bar(BAR_SFULL + b * 4 + q), u & 1, wc))) break;
          float2 tot = ld_shared_cluster_f2(mapa_shared(slot_addr, 0));
          float n_acc = tile_cols<RAG>(p, 0);  // CTA r of the cluster holds N tile r
          for (int r = 1; r < cn; ++r) {
            const float nb = tile_cols<RAG>(p, r);
            tot = Stat<ROWOP>::merge(tot, ld_shared_cluster_f2(mapa_shared(slot_addr, (uint32_t)r)), n_acc, nb);
            n_acc += nb;
          }
          st = tot;
          __syncwarp();
          if (lane == 0) {
            for (int r = 0; r < cn; ++r) mbar_arrive_cluster(bar(BAR_SEMPTY + b * 4 + q), (uint32_t)r);
          }
        } else if (XMODE == X_GLOBAL) {
          if (!pre) publish(strip, tile, st);
          // Wait (bounded, acquire) until every tile of the strip has
          // published; the loop's control flow is uniform across the warp.
          const unsigned* cnt = p.ws_count + strip * 4 + q;
          bool ok = true;
          const long long t0 = clock64();
          while (!__all_sync(0xffffffffu, ld_acquire_gpu(cnt) >= (unsigned)p.tiles_n)) {
            if constexpr (kTicketsOk) {
              if (tickets && early_t != t + 1 && checked_t != t + 1) try_early(t + 1, strip);
            }
            __nanosleep(64);
            if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
            if (__any_sync(0xffffffffu, clock64() - t0 > p.timeout_cycles)) {
              if (lane == 0) record_timeout(wc);
              ok = false;
              break;
            }
          }
          if (!ok) break;
          // The strip is complete: the producer may claim this warp's item
          // t + 2 (the leader's warps signal for a CTA pair).
          if (tickets) {
            __syncwarp();
            if (lane == 0 && leader) mbar_arrive(bar(BAR_XDONE + (t & 1)));
          }
          const float2* wsrow = p.ws_stats + (size_t)strip * p.tiles_n * kBM + row;
          float2 tot = __ldcg(wsrow);
          float n_acc = tile_cols<RAG>(p, 0);
          for (int j = 1; j < p.tiles_n; ++j) {
            const float nb = tile_cols<RAG>(p, j);
            tot = Stat<ROWOP>::merge(tot, __ldcg(wsrow + (size_t)j * kBM), n_acc, nb);
            n_acc += nb;
          }
          st = tot;
        }

        // Row normalisation constants.
        if (ROWOP == ROW_RMSNORM) {
          scale_a = rsqrtf(st.x / (float)p.N + p.eps);
        } else if (ROWOP == ROW_LAYERNORM) {
          scale_a = rsqrtf(st.y / (float)p.N + p.eps);
          shift_a = -st.x * scale_a;
        } else {  // softmax: y = exp(x - max) / sum = exp2(x*log2e - max*log2e) / sum
          scale_a = kLog2e;
          shift_a = -st.x * kLog2e;
        }
      }
      const float inv_sum = (ROWOP == ROW_SOFTMAX) ? 1.0f / st.y : 1.0f;

      // Final pass: normalise, stage through swizzled smem, TMA store.
      // Columns past N in a ragged last chunk are computed but clipped by the
      // TMA store.
#pragma unroll 1
      for (int c = 0; c < nch; ++c) {
        float v[32];
        tmem_ld32(taddr + c * 32, v);
        tmem_wait_ld();
        const int n = n0 + c * 32;
        const bool tail = RAG && n + 32 > p.N;
        if (ROWOP == ROW_NONE) {
          const float* bs = vsm + VEC_BIAS * kBN + c * 32;
          if (tail) apply_program<true, COLS>(p, v, n, m0 + row, 0, p.n_ops, bs, r_bias);
          else apply_program<false, COLS>(p, v, n, m0 + row, 0, p.n_ops, bs, r_bias);
        } else if (ROWOP == ROW_SOFTMAX) {
          scale_shift(v, scale_a, shift_a);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = ex2_approx(v[j]);
#pragma unroll
          for (int j = 0; j < 32; j += 2) fmul2(v[j], v[j + 1], inv_sum, inv_sum);
        } else {
          if (COLS) {
            scale_shift(v, scale_a, shift_a);
            scale_shift(v, r_gamma, ROWOP == ROW_LAYERNORM ? r_beta : 0.0f);
          } else {
            norm_affine<ROWOP == ROW_LAYERNORM>(v, vsm + VEC_GAMMA * kBN + c * 32, vsm + VEC_BETA * kBN + c * 32,
                                                scale_a, shift_a);
          }
        }
        // The previous TMA store from this buffer must have read it.
        if (lane == 0) bulk_wait_read0();
        __syncwarp();
        if (COLS) {
          // Transposed block: staging row j holds output row n + j, whose 32
          // columns are this warp's 32 tile rows (one per lane), unswizzled;
          // the lanes write consecutive elements of a row.
          if (p.out_bf16) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              reinterpret_cast<__nv_bfloat16*>(out_ptr)[j * 32 + lane] = __float2bfloat16_rn(v[j]);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) reinterpret_cast<float*>(out_ptr)[j * 32 + lane] = v[j];
          }
        } else if (p.out_bf16) {
          // bf16: 64-byte rows, unswizzled; lane l writes its 16-byte chunks
          // starting at chunk l & 3 to spread them over the banks.
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
            w[e] = *reinterpret_cast<const uint32_t*>(&h2);
          }
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int j = (jj + lane) & 3;
            uint4 val;
            switch (j) {  // constant register indices for each case
              case 0: val = make_uint4(w[0], w[1], w[2], w[3]); break;
              case 1: val = make_uint4(w[4], w[5], w[6], w[7]); break;
              case 2: val = make_uint4(w[8], w[9], w[10], w[11]); break;
              default: val = make_uint4(w[12], w[13], w[14], w[15]); break;
            }
            *reinterpret_cast<uint4*>(out_ptr + lane * 64 + j * 16) = val;
          }
        } else {
          // 128-byte swizzle: 16-byte chunk j of row r lands at chunk j ^ (r & 7).
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            float4* dst = reinterpret_cast<float4*>(out_ptr + lane * 128 + ((j ^ (lane & 7)) * 16));
            *dst = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (COLS) tma_store_2d_hint(&p.tmOut, out_buf, m0 + 32 * q, n, out_policy);
          else tma_store_2d_hint(&p.tmOut, out_buf, n, m0 + 32 * q, out_policy);
          bulk_commit();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (CTA2 && !leader) mbar_arrive_cluster(bar(BAR_TEMPTY + acc), 0);  // the leader issues the MMAs
        else mbar_arrive(bar(BAR_TEMPTY + acc));
        if (stage_vec) mbar_arrive(bar(BAR_VFREE));  // this warp no longer reads the tile's vector slices
      }
    }
    if (lane == 0) bulk_wait0();
  }

  tc_fence_before();
  __syncthreads();
  if (CTA2) {
    cluster_sync_all();  // the peer's TMEM and smem are in use until the leader is done
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc_pair(tmem_base, kTmemCols);
    }
    // After an abort (any bounded wait gave up: the status word is set),
    // loads of the pair may still be in flight into this CTA's shared
    // memory or onto the leader's barrier; both CTAs stop issuing before
    // the cluster barrier above, so both wait here before leaving.
    if (threadIdx.x == 0 && *reinterpret_cast<volatile unsigned*>(p.status) != 0u) settle_after_abort();
  } else {
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem_base, kTmemCols);
    }
    if (XMODE == X_CLUSTER) cluster_sync_all();
  }
}

template <int R, int X, bool P, bool RAG, bool COLS, int R0 = ROW_NONE>
const void* kernel_ptr() {
  return reinterpret_cast<const void*>(&gemm_epi_kernel<R, X, P, RAG, COLS, R0>);
}

// The instantiations one translation unit holds, one (RAG, COLS) variant per
// unit: cf_gemm_epi.cu (full tiles), cf_gemm_epi_ragged.cu (ragged last
// tile), cf_gemm_epi_cols.cu and cf_gemm_epi_cols_ragged.cu (column
// reductions), compiled in parallel.  Column variants exist for programs with
// a reduction only (without one the two axes are the same program).
template <bool RAG, bool COLS>
const void* select_kernel_t(int rowop, int xmode, bool pair) {
#define CF_CASE(R, X, P) \
  if (rowop == R && xmode == X && pair == P) return kernel_ptr<R, X, P, RAG, COLS>();
  if constexpr (!COLS) {
    CF_CASE(ROW_NONE, X_NONE, false)
    CF_CASE(ROW_NONE, X_NONE, true)
  }
  CF_CASE(ROW_LAYERNORM, X_NONE, false)
  CF_CASE(ROW_LAYERNORM, X_NONE, true)
  CF_CASE(ROW_LAYERNORM, X_CLUSTER, false)
  CF_CASE(ROW_LAYERNORM, X_GLOBAL, false)
  CF_CASE(ROW_LAYERNORM, X_GLOBAL, true)
  CF_CASE(ROW_RMSNORM, X_NONE, false)
  CF_CASE(ROW_RMSNORM, X_NONE, true)
  CF_CASE(ROW_RMSNORM, X_CLUSTER, false)
  CF_CASE(ROW_RMSNORM, X_GLOBAL, false)
  CF_CASE(ROW_RMSNORM, X_GLOBAL, true)
  CF_CASE(ROW_SOFTMAX, X_NONE, false)
  CF_CASE(ROW_SOFTMAX, X_NONE, true)
  CF_CASE(ROW_SOFTMAX, X_CLUSTER, false)
  CF_CASE(ROW_SOFTMAX, X_GLOBAL, false)
  CF_CASE(ROW_SOFTMAX, X_GLOBAL, true)
#undef CF_CASE
  // Two chained reductions (per-tile or workspace exchange only).
#define CF_CASE2(R0, R)                                                                                   \
  if (rowop == row_code(R0, R)) {                                                                         \
    if (xmode == X_NONE)                                                                                  \
      return pair ? kernel_ptr<R, X_NONE, true, RAG, COLS, R0>() : kernel_ptr<R, X_NONE, false, RAG, COLS, R0>(); \
    if (xmode == X_GLOBAL)                                                                                \
      return pair ? kernel_ptr<R, X_GLOBAL, true, RAG, COLS, R0>()                                        \
                  : kernel_ptr<R, X_GLOBAL, false, RAG, COLS, R0>();                                      \
    return nullptr;                                                                                       \
  }
  CF_CASE2(ROW_LAYERNORM, ROW_LAYERNORM)
  CF_CASE2(ROW_LAYERNORM, ROW_RMSNORM)
  CF_CASE2(ROW_LAYERNORM, ROW_SOFTMAX)
  CF_CASE2(ROW_RMSNORM, ROW_LAYERNORM)
  CF_CASE2(ROW_RMSNORM, ROW_RMSNORM)
  CF_CASE2(ROW_RMSNORM, ROW_SOFTMAX)
#undef CF_CASE2
  return nullptr;
}

int smem_for(bool pair) { return pair ? Geo<true>::kSmemBytes : Geo<false>::kSmemBytes; }

}  // namespace
}  // namespace cf
