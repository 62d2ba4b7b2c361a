// cf_b2b.cu -- fused back-to-back GEMM: O = bf16(F(A . W1)) . W2 with the
// intermediate S' never written to global memory.
//
// ComFuse review, "What carries the argument": the B2BGEMM schedule keeps the
// post-processed intermediate tile S_tile on chip and accumulates the second
// GEMM's output from it; referee report, major comment 2 [Sec. IV-A,
// Eqs. (3)-(5)]: the intermediate tile transform F and the segmented
// accumulation over the co-scheduled CTAs.  The page's "four-stage pipeline"
// is cut off; it is read here as load -> GEMM1 -> F -> GEMM2, overlapped
// across intermediate chunks.
//
// Two sm_103a kernels:
//
// attn_kernel (W1 given as its transpose, head dims K, N2 <= 128 computed
// as 128 with zero padding, any N1; the attention shape S = Q K^T):  one CTA
// owns a 128-row block of A for one batch entry and
// walks the N1 dimension in 128-wide chunks.  Per chunk j: S_j = A . W1_j in
// TMEM (two S buffers, so S_{j+1} is computed while F runs on S_j), F on
// TMEM rows in registers, S'_j rounded to bf16 into a swizzled shared-memory
// tile, then O += S'_j . W2_j in TMEM.  For the softmax op the row
// statistics use the online form (running max m and sum l, O rescaled when
// the max grows; the rescale is skipped while the max grows by less than
// 2^8, since exp2(x - m) <= 256 stays exact enough in bf16 and fp32), and O
// is divided by l at the end.  This is the C = 1 (single-CTA) case of the
// review's Eq. (5) merge.
//
// mlp_kernel (general K, N1; N2 <= 256 * C): a cluster of C CTAs shares one
// 128-row strip.  CTA c owns O[:, 256c .. 256c+255] in TMEM (the whole
// 128 x N2 fp32 strip does not fit one SM's TMEM).  For each round of C
// chunks of N1, CTA c computes the 128 x 128 chunk S_c = A . W1[:, chunk],
// applies F, rounds to bf16 and writes it into the same shared-memory slot of
// every CTA of the cluster (distributed shared memory), so GEMM1 work is never
// repeated; each CTA then accumulates O_c += [S'_0 .. S'_{C-1}] . W2[round
// rows, its columns].  This is the review's cluster-cooperative dataflow:
// the second GEMM's output accumulation is distributed across the cluster.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "cf_internal.h"
#include "cf_ptx.cuh"

namespace cf {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// Pack 32 fp32 values into 16 bf16x2 words (round to nearest even, one
// packed conversion per pair).
__device__ __forceinline__ void pack_bf16(const float (&v)[32], uint32_t (&w)[16]) {
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
    w[e] = *reinterpret_cast<uint32_t*>(&h);
  }
}

// Three-input maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// v[e] = v[e] * s + t for 32 values, two per packed fp32x2 FMA; s2 and t2
// hold {s, s} and {t, t}.
__device__ __forceinline__ void fma2_32(float (&v)[32], uint64_t s2, uint64_t t2) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    asm("{\n\t.reg .b64 x;\n\tmov.b64 x, {%0, %1};\n\tfma.rn.f32x2 x, x, %2, %3;\n\tmov.b64 {%0, %1}, x;\n\t}"
        : "+f"(v[e]), "+f"(v[e + 1])
        : "l"(s2), "l"(t2));
  }
}

__device__ __forceinline__ uint64_t pack2f(float a) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(a));
  return r;
}

// Sum of the 32 bf16 values held in 16 packed words (exact widening).
// Sum of the 32 bf16 values held in 16 packed words: mixed-precision adds
// (each bf16 half widens exactly into an fp32 accumulator), four independent
// accumulators to keep the dependency chains short.
__device__ __forceinline__ float sum_packed_bf16(const uint32_t (&w)[16]) {
  float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    float& a = acc[(e & 1) * 2];
    float& b = acc[(e & 1) * 2 + 1];
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tadd.rn.f32.bf16 %0, lo, %0;\n\t"
        "add.rn.f32.bf16 %1, hi, %1;\n\t}"
        : "+f"(a), "+f"(b)
        : "r"(w[e]));
  }
  return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// Write 32 packed bf16 values of row `r` (columns c0..c0+31 of a 128-column
// K-major tile) into a 128-byte-swizzled smem tile of two 64-column regions.
__device__ __forceinline__ void store_row_packed_sw128(uint8_t* tile, int r, int c0, const uint32_t (&w)[16]) {
  uint8_t* base = tile + (c0 >> 6) * 16384 + r * 128;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int chunk = ((c0 & 63) >> 3) + q;
    *reinterpret_cast<uint4*>(base + ((chunk ^ (r & 7)) << 4)) =
        make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
  }
}

// One 32-byte store (a whole 32-byte sector of the memory system).
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
               "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// Store W values v[i] * s of one output row at element offset `off` of
// `out`: fp32 or bf16 rounded to nearest even.  W is a multiple of 16.
// V8: `out + off` is 32-byte aligned, so every store writes one whole
// 32-byte sector (8 fp32 or 16 bf16 values); otherwise 16-byte stores (row
// pitch and column offsets keep those aligned; checked on the host).  Each
// thread writes its own row, so 16-byte stores would leave every sector
// half-written per request.
template <int W>
__device__ __forceinline__ void store_row(void* out, int bf16, long long off, const float* v, float s, bool v8) {
  if (v8) {
    if (bf16) {
#pragma unroll
      for (int j = 0; j < W / 16; ++j) {
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const __nv_bfloat162 h = __floats2bfloat162_rn(v[16 * j + 2 * e] * s, v[16 * j + 2 * e + 1] * s);
          w[e] = *reinterpret_cast<const uint32_t*>(&h);
        }
        st_global_v8(static_cast<uint16_t*>(out) + off + 16 * j, w);
      }
    } else {
#pragma unroll
      for (int j = 0; j < W / 8; ++j) {
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = __float_as_uint(v[8 * j + e] * s);
        st_global_v8(static_cast<float*>(out) + off + 8 * j, w);
      }
    }
    return;
  }
  if (bf16) {
    uint4* d = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + off);
#pragma unroll
    for (int j = 0; j < W / 8; ++j) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(v[8 * j + 2 * e] * s, v[8 * j + 2 * e + 1] * s);
        w[e] = *reinterpret_cast<const uint32_t*>(&h);
      }
      d[j] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
    float4* d = reinterpret_cast<float4*>(static_cast<float*>(out) + off);
#pragma unroll
    for (int j = 0; j < W / 4; ++j) d[j] = make_float4(v[4 * j] * s, v[4 * j + 1] * s, v[4 * j + 2] * s, v[4 * j + 3] * s);
  }
}

// store_row for an output row that ends inside these W columns: only the
// first `valid` (< W) values are stored, one element at a time.
template <int W>
__device__ __forceinline__ void store_row_part(void* out, int bf16, long long off, const float* v, float s,
                                               int valid) {
#pragma unroll
  for (int j = 0; j < W; ++j) {
    if (j < valid) {
      if (bf16) static_cast<__nv_bfloat16*>(out)[off + j] = __float2bfloat16_rn(v[j] * s);
      else static_cast<float*>(out)[off + j] = v[j] * s;
    }
  }
}

// ======================================================================
// Attention-shaped B2BGEMM
// ======================================================================
namespace attn {

constexpr int kTile = 128;                  // rows of A per CTA, N1 chunk, K and N2
constexpr int kTileBytes = 128 * 128 * 2;   // one bf16 128 x 128 tile (two 64-column regions)
constexpr int kRing1 = 3;                   // W1 tiles in flight (GEMM1 operand ring)
constexpr int kRing2 = 2;                   // W2 tiles in flight (GEMM2 operand ring)
constexpr int kFWarps = 8;                  // two warpgroups; group G takes the chunks g with g % 2 == G
// Warps: 0 loads A and W1, 1 issues GEMM1 (and owns TMEM), 2..9 run F,
// 10 loads W2, 11 issues GEMM2.
constexpr int kWarpLoad2 = 2 + kFWarps, kWarpMma2 = 3 + kFWarps;
constexpr int kThreads = 32 * (4 + kFWarps);
constexpr int kOffQ = 0;                    // the A tile (reloaded once the item's last GEMM1 is done)
constexpr int kOffW1 = kOffQ + kTileBytes;
constexpr int kOffW2 = kOffW1 + kRing1 * kTileBytes;
constexpr int kOffM = kOffW2 + kRing2 * kTileBytes;   // float [2 chunk parities][128]: running max hand-off
constexpr int kOffL = kOffM + 2 * 128 * 4;            // float2 [2 item parities][128]: (l, m) of a group
constexpr int kOffBars = kOffL + 2 * 128 * 8;
// q_full, q_empty, W1 ring full/empty, W2 ring full/empty, and per S buffer
// b (= chunk parity = F group): s_full, s_free (group b holds S_b in
// registers), p_full, pv_done; then o_full, o_empty, one drain barrier per
// MMA issuer, running-max hand-off [2 chunk parities][4 quarters], (l, m)
// hand-off [2 item parities][4 quarters]; key split only: the cluster's
// published row statistics [4 quarters] and staged output rows [4 quarters].
constexpr int BAR_QF = 0, BAR_QE = 1, BAR_RF1 = 2, BAR_RE1 = BAR_RF1 + kRing1, BAR_RF2 = BAR_RE1 + kRing1,
              BAR_RE2 = BAR_RF2 + kRing2, BAR_SF = BAR_RE2 + kRing2, BAR_SFREE = BAR_SF + 2, BAR_PF = BAR_SFREE + 2,
              BAR_PV = BAR_PF + 2, BAR_OF = BAR_PV + 2, BAR_OE = BAR_OF + 1, BAR_DRAIN1 = BAR_OE + 1,
              BAR_DRAIN2 = BAR_DRAIN1 + 1, BAR_MB = BAR_DRAIN2 + 1, BAR_XL = BAR_MB + 8, BAR_MLF = BAR_XL + 8,
              BAR_STG = BAR_MLF + 4, kNumBars = BAR_STG + 4;
constexpr int kOffMisc = kOffBars + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
constexpr int kTmemCols = 512;  // S0 [0,128), S1 [128,256), O [256,384), S'0 [384,448), S'1 [448,512)
constexpr int kTmemO = 256;
constexpr int kTmemP = 384;     // S' buffer b (bf16 pairs, 64 columns) at kTmemP + 64 b
constexpr float kRescaleLog2 = 8.0f;

struct Params {
  CUtensorMap tmA, tmW1, tmW2;  // 3-D: {128 cols, rows, batch}
  void* out;        // fp32 or bf16 (out_bf16), element offsets below
  long long ldo, stride_out;
  int out_bf16;
  int M;             // rows of A per batch entry (the last 128-row block may be ragged)
  int batch, m_blocks, n1_blocks, items;
  int kv_last;       // valid columns of S in the last N1 chunk (1..128; < 128: ragged N1)
  int n2;            // valid output columns (N2 <= 128)
  int softmax;       // 1: scaled softmax (scale > 0), 0: ReLU (optionally scaled)
  float scale;       // multiplies S before F
  int out_v8;        // the output base, row pitch and batch stride are 32-byte aligned
  int split;         // key split: CTAs per query block (the cluster size); 1 without the split
  int nb_per;        // key split: 128-key chunks per CTA (the last CTA's range may be shorter)
  unsigned* status;
  long long timeout_cycles;
};

// Four output values of one row at element offset `off`: fp32 (one 16-byte
// store) or bf16 rounded to nearest even (one 8-byte store); only the first
// `valid` are stored when the row ends inside them.
template <bool OBF16>
__device__ __forceinline__ void store4(void* out, long long off, float4 v, int valid) {
  if (valid >= 4) {
    if (OBF16) {
      const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + off) =
          make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
    } else {
      *reinterpret_cast<float4*>(static_cast<float*>(out) + off) = v;
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    if (j < valid) {
      const float e = j == 0 ? v.x : j == 1 ? v.y : v.z;
      if (OBF16) static_cast<__nv_bfloat16*>(out)[off + j] = __float2bfloat16_rn(e);
      else static_cast<float*>(out)[off + j] = e;
    }
  }
}

__device__ __forceinline__ float (&part32(float (&v)[128], int c))[32] {
  return *reinterpret_cast<float(*)[32]>(&v[32 * c]);
}

// tcgen05.ld of a row's 128 columns that also returns the maximum of the
// 128 values the thread loads (the reducing TMEM load of sm_103a).  Like the
// loaded registers, the maximum is valid only after tcgen05.wait::ld.
__device__ __forceinline__ void tmem_ld128_max(uint32_t taddr, float (&v)[128], float& mx) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x128.max.f32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, %128, [%129];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127]), "=f"(mx)
      : "r"(taddr)
      : "memory");
}

// Two MMA-issuing threads: a 128 x 128 x 16 MMA lasts only 64 cycles and the
// tensor pipe runs barely one instruction ahead of its issuing thread, so a
// single thread that also waits on barriers between GEMM1 and GEMM2 bursts
// leaves the pipe idle for every wait.  With GEMM1 and GEMM2 issued from
// different warps, one keeps the pipe fed while the other waits.
// RAG: the softmax masks the last chunk's keys past N1 (N1 not a multiple
// of 128), or the output has fewer than 128 columns; OBF16: bf16 output.
// Both are compile-time so that the common instantiation (full chunks,
// fp32 output) carries neither the masking nor a second store path in the F
// warps, which bound the softmax variant.
//
// SPLIT: the key range of each query block is split across the CTAs of a
// thread-block cluster (the co-scheduled CTA set C of the review's Eq. (5)):
// CTA r of the cluster runs the same pipeline over its own chunks
// [r nb_per, min(N1 chunks, (r + 1) nb_per)) and keeps its running
// (m_r, l_r, O_r); at the end the cluster merges them through distributed
// shared memory, m = max_r m_r, l = sum_r l_r 2^(m_r - m),
// O = sum_r O_r 2^(m_r - m) / l (for ReLU, O = sum_r O_r).  Each cluster takes
// exactly one query block (no persistence), so the key rings are idle when
// the merge stages O in them.  Used when there are fewer query blocks than
// SMs, where one CTA per block would leave most of the GPU idle.
template <bool RAG, bool OBF16, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1) attn_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) -> uint32_t { return sbase + kOffBars + 8 * i; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  const WaitCtx wc{p.timeout_cycles, abort_flag, p.status};
  const int nb = p.n1_blocks;
  // Items (query blocks) of this CTA and its key chunks [j0, j1) of each.
  int item0 = blockIdx.x, istep = gridDim.x, j0 = 0, j1 = nb;
  uint32_t crank = 0;
  if constexpr (SPLIT) {
    crank = cluster_ctarank();
    item0 = (int)cluster_id_x();
    istep = (int)num_clusters_x();
    j0 = (int)crank * p.nb_per;
    j1 = min(nb, j0 + p.nb_per);
  }
  const int nbl = j1 - j0;  // >= 1: the host sizes the split so that no range is empty

  // The tensor-map fetches start before the barrier set-up, which they
  // overlap (the first TMA load waits for its map).
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmA);
    tma_prefetch_desc(&p.tmW1);
    tma_prefetch_desc(&p.tmW2);
  }
  if (threadIdx.x == 0) {
    mbar_init(bar(BAR_QF), 1);
    mbar_init(bar(BAR_QE), 1);
    for (int i = 0; i < kRing1; ++i) {
      mbar_init(bar(BAR_RF1 + i), 1);
      mbar_init(bar(BAR_RE1 + i), 1);
    }
    for (int i = 0; i < kRing2; ++i) {
      mbar_init(bar(BAR_RF2 + i), 1);
      mbar_init(bar(BAR_RE2 + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(BAR_SF + i), 1);
      mbar_init(bar(BAR_SFREE + i), 4);  // the four warps of F group i
      mbar_init(bar(BAR_PF + i), 4);
      mbar_init(bar(BAR_PV + i), 1);
    }
    mbar_init(bar(BAR_OF), 1);
    mbar_init(bar(BAR_OE), 4);  // the group that writes the item's output
    mbar_init(bar(BAR_DRAIN1), 1);
    mbar_init(bar(BAR_DRAIN2), 1);
    for (int i = 0; i < 16; ++i) mbar_init(bar(BAR_MB + i), 1);  // MB[8] then XL[8]: one publishing warp
    for (int i = 0; i < 8; ++i) mbar_init(bar(BAR_MLF + i), SPLIT ? p.split : 1);  // one warp of each CTA
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0 || warp == kWarpLoad2) {
    // ----------------------------------------------------------- producers
    // Warp 0: the A tile and the W1 ring; warp 10: the W2 ring.  Each ring is
    // consumed in load order by one MMA issuer.
    if (lane == 0) {
      const bool w1 = warp == 0;
      const int depth = w1 ? kRing1 : kRing2;
      const int off = w1 ? kOffW1 : kOffW2;
      const int rf = w1 ? BAR_RF1 : BAR_RF2, re = w1 ? BAR_RE1 : BAR_RE2;
      const CUtensorMap* m = w1 ? &p.tmW1 : &p.tmW2;
      uint32_t rs = 0, rph = 0, issued = 0, q_issued = 0;
      int it = 0;
      bool ok = true;
      for (int item = item0; ok && item < p.items; item += istep, ++it) {
        const int b = item / p.m_blocks, mb = item - b * p.m_blocks;
        if (w1) {
          if (!mbar_wait(bar(BAR_QE), (it & 1) ^ 1, wc)) break;
          mbar_arrive_expect_tx(bar(BAR_QF), kTileBytes);
          tma_load_3d(sbase + kOffQ, &p.tmA, bar(BAR_QF), 0, mb * kTile, b);
          tma_load_3d(sbase + kOffQ + 16384, &p.tmA, bar(BAR_QF), 64, mb * kTile, b);
          ++q_issued;
        }
        for (int j = j0; j < j1; ++j) {
          if (!mbar_wait(bar(re + rs), rph ^ 1, wc)) { ok = false; break; }
          const uint32_t dst = sbase + off + rs * kTileBytes;
          mbar_arrive_expect_tx(bar(rf + rs), kTileBytes);
          tma_load_3d(dst, m, bar(rf + rs), 0, j * kTile, b);
          tma_load_3d(dst + 16384, m, bar(rf + rs), 64, j * kTile, b);
          ++issued;
          if (++rs == (uint32_t)depth) { rs = 0; rph ^= 1; }
        }
      }
      // No load of this CTA is still in flight when it exits.
      drain_ring(bar(rf), (uint32_t)depth, issued, wc);
      if (w1) drain_ring(bar(BAR_QF), 1u, q_issued, wc);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- GEMM1 issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(128, 128, 0);   // W1 tile is K-major (rows = N1)
      const SDesc dq = sdesc_sw128(sbase + kOffQ, 16, 1024);
      const SDesc dk = sdesc_sw128(sbase + kOffW1, 16, 1024);
      constexpr uint32_t kTileStep = kTileBytes >> 4;
      uint32_t rs = 0, rph = 0;
      uint32_t g = 0;  // global chunk counter (S buffer and F group = g & 1)
      int it = 0;
      bool ok = true;
      for (int item = item0; ok && item < p.items; item += istep, ++it) {
        if (!mbar_wait(bar(BAR_QF), it & 1, wc)) break;
        for (int j = j0; j < j1; ++j, ++g) {
          // S buffer g & 1 is free once F group g & 1 holds S_{g-2} in registers.
          if (g >= 2 && !mbar_wait(bar(BAR_SFREE + (g & 1)), ((g - 2) >> 1) & 1, wc)) { ok = false; break; }
          if (!mbar_wait(bar(BAR_RF1 + rs), rph, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t k_lo = dk.lo + rs * kTileStep;
          const uint32_t d = tmem_base + (g & 1) * 128;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t koff = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
            mma_ss(d, dq.lo + koff, dq.hi, k_lo + koff, dk.hi, id_s, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(BAR_RE1 + rs));
          mma_commit(bar(BAR_SF + (g & 1)));
          if (++rs == kRing1) { rs = 0; rph ^= 1; }
        }
        if (!ok) break;
        mma_commit(bar(BAR_QE));  // every GEMM1 of this item has read the A tile
      }
      mma_commit(bar(BAR_DRAIN1));
      mbar_wait<false, false>(bar(BAR_DRAIN1), 0, wc);
    }
  } else if (warp == kWarpMma2) {
    // ------------------------------------------------------- GEMM2 issuer
    if (lane == 0) {
      const uint32_t id_o = idesc_bf16_f32(128, 128, 1);   // W2 tile is MN-major (rows = K of GEMM2)
      const SDesc dv = sdesc_sw128(sbase + kOffW2, 16384, 1024);
      constexpr uint32_t kTileStep = kTileBytes >> 4;
      uint32_t rs = 0, rph = 0;
      uint32_t g = 0;
      int it = 0;
      bool ok = true;
      for (int item = item0; ok && item < p.items; item += istep, ++it) {
        for (int j = j0; j < j1; ++j, ++g) {
          if (!mbar_wait(bar(BAR_PF + (g & 1)), (g >> 1) & 1, wc)) { ok = false; break; }
          if (j == j0 && !mbar_wait(bar(BAR_OE), (it & 1) ^ 1, wc)) { ok = false; break; }
          if (!mbar_wait(bar(BAR_RF2 + rs), rph, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t v_lo = dv.lo + rs * kTileStep;
          const uint32_t p_col = tmem_base + kTmemP + 64 * (g & 1);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // A = S' from TMEM (16 K elements = 8 packed columns per step);
            // B = W2 rows 16 kk .. 16 kk + 15 (2048 bytes per step).
            mma_ts(tmem_base + kTmemO, p_col + 8 * kk, v_lo + kk * (2048 >> 4), dv.hi, id_o,
                   (j > j0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(bar(BAR_RE2 + rs));
          mma_commit(bar(BAR_PV + (g & 1)));
          if (++rs == kRing2) { rs = 0; rph ^= 1; }
        }
        if (!ok) break;
        mma_commit(bar(BAR_OF));
      }
      mma_commit(bar(BAR_DRAIN2));
      mbar_wait<false, false>(bar(BAR_DRAIN2), 0, wc);
    }
  } else {
    // -------------------------------------- F (softmax / ReLU) and epilogue
    // F group G = 0, 1 takes the chunks g with g % 2 == G: a thread owns one
    // S row (TMEM lane) and all 128 columns of the chunk, so two chunks are
    // in F at once.  Softmax keeps one running max per row for both groups:
    // the owner of chunk g receives the max in use after chunk g-1 from the
    // other group (shared memory + a per-quarter mbarrier), decides the max
    // for chunk g, and passes it on at once, before its exponentials.  Each
    // group keeps its own running sum l in the scale of the last max it used;
    // the group that owns an item's last chunk merges both sums and writes
    // the output rows.
    const int grp = (warp - 2) >> 2;
    const int q = warp & 3;
    const int row = 32 * q + lane;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    float* mrun = reinterpret_cast<float*>(smem + kOffM);   // [chunk parity][row]
    float2* lm = reinterpret_cast<float2*>(smem + kOffL);   // [item parity][row]
    const float sl2 = p.scale * kLog2e;
    uint32_t g = 0;
    int it = 0;
    bool ok = true;
    for (int item = item0; ok && item < p.items; item += istep, ++it) {
      const int b = item / p.m_blocks, mb = item - b * p.m_blocks;
      const uint32_t g0 = g;
      const uint32_t g_last = g0 + (uint32_t)nbl - 1;
      float l = 0.0f, m_last = -INFINITY;   // this group's sum, and the max it is scaled to
      for (uint32_t gg = g0 + ((g0 & 1) != (uint32_t)grp ? 1u : 0u); gg <= g_last; gg += 2) {
        const int j = (int)(gg - g0);
        const uint32_t sb = gg & 1, u = gg >> 1;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(BAR_SF + sb), u & 1, wc))) { ok = false; break; }
        tc_fence_after();
        float v[128];
        // Full chunks of the softmax take the row maximum from the reducing
        // TMEM load itself; a ragged last chunk masks its keys past N1 first
        // and takes the maximum below.
        const bool ragged_chunk = RAG && j0 + j == nb - 1 && p.kv_last < kTile;
        const bool ld_max = p.softmax && !ragged_chunk;
        float rmax_ld = 0.0f;
        if (ld_max) {
          tmem_ld128_max(tmem_base + lane_off + sb * 128, v, rmax_ld);
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(tmem_base + lane_off + sb * 128 + 32 * c, part32(v, c));
        }
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_SFREE + sb));  // S_sb may be overwritten now
        if (p.softmax) {
          if (ragged_chunk) {
            // Ragged N1: keys past N1 were loaded as zero rows; their logits
            // leave the max and the sum (exp2(-inf) = 0).  The V rows past
            // N1 are zero as well.
#pragma unroll
            for (int e = 0; e < 128; ++e)
              if (e >= p.kv_last) v[e] = -INFINITY;
          }
          float rmax;
          if (ld_max) {
            rmax = rmax_ld;
          } else {
            // Row max with three-input max instructions: 128 -> 16 -> 1.
            float mx[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              mx[e] = max3f(max3f(v[e], v[e + 16], v[e + 32]), max3f(v[e + 48], v[e + 64], v[e + 80]),
                            fmaxf(v[e + 96], v[e + 112]));
            const float mxa =
                max3f(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], mx[5]), max3f(mx[6], mx[7], mx[8]));
            const float mxb = max3f(max3f(mx[9], mx[10], mx[11]), max3f(mx[12], mx[13], mx[14]), mx[15]);
            rmax = fmaxf(mxa, mxb);
          }
          const float bmax = rmax * sl2;
          // Max in use after chunk gg-1 (every chunk but the CTA's first
          // waits, so hand-offs alternate strictly between the groups).
          float m_prev = -INFINITY;
          if (gg > 0) {
            const uint32_t pg = gg - 1;
            if (!__all_sync(0xffffffffu, mbar_wait(bar(BAR_MB + (pg & 1) * 4 + q), (pg >> 1) & 1, wc))) {
              ok = false;
              break;
            }
            if (j > 0) m_prev = mrun[(pg & 1) * 128 + row];
          }
          // Lazy rescale: the max in use moves only when the block max
          // exceeds it by more than 2^8 (in exp2 units).
          const bool need = bmax > m_prev + kRescaleLog2;
          const float m_new = need ? bmax : m_prev;
          mrun[sb * 128 + row] = m_new;
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(BAR_MB + sb * 4 + q));
          if (j > 0 && __any_sync(0xffffffffu, need)) {
            // O must hold every earlier S' . W2 product before it is rescaled.
            const uint32_t pg = gg - 1;
            if (!__all_sync(0xffffffffu, mbar_wait(bar(BAR_PV + (pg & 1)), (pg >> 1) & 1, wc))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const float f = ex2_approx(m_prev - m_new);
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {  // 16 columns at a time: v[] stays in registers
              float o[16];
              tmem_ld16(tmem_base + lane_off + kTmemO + c * 16, o);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 16; ++e) o[e] *= f;
              tmem_st16(tmem_base + lane_off + kTmemO + c * 16, o);
            }
            tmem_wait_st();
          }
          l *= ex2_approx(m_last - m_new);  // 0 on this group's first chunk of the item
          m_last = m_new;
        }
        // F, bf16 rounding and (softmax) the row sum of exactly what GEMM2
        // consumes, 32 columns at a time, into registers: all of it before
        // the wait for the S' buffer, so that this work overlaps the S' . W2
        // product two chunks back instead of following it.
        uint32_t w[4][16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float(&vc)[32] = part32(v, c);
          if (p.softmax) {
            fma2_32(vc, pack2f(sl2), pack2f(-m_last));  // the exp2 arguments, two per instruction
#pragma unroll
            for (int e = 0; e < 32; ++e) vc[e] = ex2_approx(vc[e]);
            pack_bf16(vc, w[c]);
            l += sum_packed_bf16(w[c]);
          } else {
            // relu(bf16(scale s)) == bf16(relu(scale s)) (rounding is monotonic
            // and keeps 0): scale two per packed FMA, round, then a bf16x2 max.
            fma2_32(vc, pack2f(p.scale), pack2f(0.0f));
            pack_bf16(vc, w[c]);
#pragma unroll
            for (int e = 0; e < 16; ++e) asm("max.bf16x2 %0, %0, %1;" : "+r"(w[c][e]) : "r"(0u));
          }
        }
        // S' buffer sb was last read by the S' . W2 product two chunks back.
        if (!__all_sync(0xffffffffu, mbar_wait(bar(BAR_PV + sb), (u & 1) ^ 1, wc))) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_st16(tmem_base + lane_off + kTmemP + 64 * sb + 16 * c, *reinterpret_cast<float(*)[16]>(&w[c][0]));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_PF + sb));
      }
      g = g_last + 1;
      if (!ok) break;
      const bool writer = (g_last & 1) == (uint32_t)grp;
      const uint32_t xl = (uint32_t)(it & 1);
      if (!writer) {
        // Hand this group's (l, max) to the writer of the item's output.
        if (p.softmax && nbl >= 2) {
          lm[xl * 128 + row] = make_float2(l, m_last);
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(BAR_XL + xl * 4 + q));
        }
        continue;
      }
      // Writer: O / l -> fp32 output rows (all 128 columns of its rows).
      float inv = 1.0f, lt = 1.0f;
      if (p.softmax) {
        lt = l;
        if (nbl >= 2) {
          if (!__all_sync(0xffffffffu, mbar_wait(bar(BAR_XL + xl * 4 + q), (it >> 1) & 1, wc))) break;
          const float2 o = lm[xl * 128 + row];
          // m_last is the final max (the max in use never decreases).
          lt = l + o.x * ex2_approx(o.y - m_last);
        }
        inv = 1.0f / lt;
      }
      if (!__all_sync(0xffffffffu, mbar_wait(bar(BAR_OF), it & 1, wc))) break;
      tc_fence_after();
      const long long orow = (long long)b * p.stride_out + (long long)(mb * kTile + row) * p.ldo;
      if constexpr (SPLIT) {
        // The review's Eq. (5) over the cluster.  Each CTA publishes its
        // rows' (m_r, l_r), derives the block's (m, l) from all of them in
        // rank order, stages O_r 2^(m_r - m) / l in shared memory, and sums
        // its own slice of the 32 four-column chunks of every CTA's staged
        // row, in rank order, into the output.  Only this CTA's warp of the
        // same TMEM quarter reads a row, so the barriers are per quarter.
        const int C = p.split;
        float2* mlx = lm + 128;  // one item per CTA: the second item slot is free
        mlx[row] = make_float2(m_last, lt);
        __syncwarp();
        if (lane == 0) {
          fence_acq_rel_cluster();
          for (int r = 0; r < C; ++r) mbar_arrive_cluster(bar(BAR_MLF + q), (uint32_t)r);
        }
        if (!__all_sync(0xffffffffu, mbar_wait<true>(bar(BAR_MLF + q), 0, wc))) break;
        float f = 1.0f;
        if (p.softmax) {
          const uint32_t a = smem_u32(mlx + row);
          float mx = -INFINITY;
          for (int r = 0; r < C; ++r) mx = fmaxf(mx, ld_shared_cluster_f2(mapa_shared(a, (uint32_t)r)).x);
          float lsum = 0.0f;
          for (int r = 0; r < C; ++r) {
            const float2 v = ld_shared_cluster_f2(mapa_shared(a, (uint32_t)r));
            lsum += v.y * ex2_approx(v.x - mx);
          }
          f = ex2_approx(m_last - mx) / lsum;
        }
        // Stage the scaled O rows in the W1 ring: its last tile was consumed
        // by a GEMM1 that completed before this item's last GEMM2.  Row r is
        // 512 bytes; its 16-byte chunk k sits at chunk k ^ (r & 31), so a
        // warp's 32 rows hit distinct bank groups.
        fence_proxy_async_smem();
        uint8_t* srow = smem + kOffW1 + row * 512;
#pragma unroll 1
        for (int h = 0; h < 4; ++h) {
          float o[32];
          tmem_ld32(tmem_base + lane_off + kTmemO + 32 * h, o);
          tmem_wait_ld();
#pragma unroll
          for (int k4 = 0; k4 < 8; ++k4) {
            const int k = 8 * h + k4;
            *reinterpret_cast<float4*>(srow + ((k ^ (row & 31)) << 4)) =
                make_float4(o[4 * k4] * f, o[4 * k4 + 1] * f, o[4 * k4 + 2] * f, o[4 * k4 + 3] * f);
          }
        }
        __syncwarp();
        if (lane == 0) {
          fence_acq_rel_cluster();
          for (int r = 0; r < C; ++r) mbar_arrive_cluster(bar(BAR_STG + q), (uint32_t)r);
        }
        if (!__all_sync(0xffffffffu, mbar_wait<true>(bar(BAR_STG + q), 0, wc))) break;
        // This CTA's slice: eight-column units (32 bytes of fp32 output, one
        // whole sector per store when the rows are 32-byte aligned).
        const int ub = (16 * (int)crank) / C, ue = (16 * ((int)crank + 1)) / C;
        const uint32_t srow_addr = sbase + kOffW1 + row * 512;
        const bool live = mb * kTile + row < p.M;  // rows past M (ragged last block) are not stored
#pragma unroll 1
        for (int u8 = ub; u8 < ue; ++u8) {
          float4 acc[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int k = 2 * u8 + h;
            const uint32_t a = srow_addr + ((uint32_t)(k ^ (row & 31)) << 4);
            acc[h] = ld_shared_cluster_f4(mapa_shared(a, 0));
            for (int r = 1; r < C; ++r) {
              const float4 v = ld_shared_cluster_f4(mapa_shared(a, (uint32_t)r));
              acc[h].x += v.x;
              acc[h].y += v.y;
              acc[h].z += v.z;
              acc[h].w += v.w;
            }
          }
          const int col = 8 * u8;
          if (!live || col >= p.n2) continue;
          if (p.out_v8 && col + 8 <= p.n2) {
            uint32_t w[8];
            if (OBF16) {
              // 8 bf16 values: half a sector (16 bytes), still one store.
              const float e[8] = {acc[0].x, acc[0].y, acc[0].z, acc[0].w, acc[1].x, acc[1].y, acc[1].z, acc[1].w};
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(e[2 * j], e[2 * j + 1]);
                w[j] = *reinterpret_cast<const uint32_t*>(&h2);
              }
              *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + orow + col) = make_uint4(w[0], w[1], w[2], w[3]);
            } else {
              w[0] = __float_as_uint(acc[0].x); w[1] = __float_as_uint(acc[0].y);
              w[2] = __float_as_uint(acc[0].z); w[3] = __float_as_uint(acc[0].w);
              w[4] = __float_as_uint(acc[1].x); w[5] = __float_as_uint(acc[1].y);
              w[6] = __float_as_uint(acc[1].z); w[7] = __float_as_uint(acc[1].w);
              st_global_v8(static_cast<float*>(p.out) + orow + col, w);
            }
          } else {
            store4<OBF16>(p.out, orow + col, acc[0], p.n2 - col);
            if (col + 4 < p.n2) store4<OBF16>(p.out, orow + col + 4, acc[1], p.n2 - col - 4);
          }
        }
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float o[64];
          tmem_ld32(tmem_base + lane_off + kTmemO + 64 * h, *reinterpret_cast<float(*)[32]>(&o[0]));
          tmem_ld32(tmem_base + lane_off + kTmemO + 64 * h + 32, *reinterpret_cast<float(*)[32]>(&o[32]));
          tmem_wait_ld();
          if (h == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(BAR_OE));  // O may be overwritten by the next item
          }
          if (mb * kTile + row < p.M) {  // rows past M (ragged last block) are not stored
            if (!RAG || p.n2 >= 64 * (h + 1)) store_row<64>(p.out, OBF16, orow + 64 * h, o, inv, p.out_v8);
            else if (p.n2 > 64 * h) store_row_part<64>(p.out, OBF16, orow + 64 * h, o, inv, p.n2 - 64 * h);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  // Key split: no CTA leaves while a peer may still read its shared memory.
  if constexpr (SPLIT) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace attn


// ======================================================================
// MLP-shaped B2BGEMM (cluster-cooperative)
// ======================================================================
namespace mlp {

constexpr int kStageBytes = 32768;              // one ring stage
constexpr int kMaxRing = 6;
constexpr int kSlotBytes = 128 * 128 * 2;       // one 128 x 128 bf16 S' chunk
constexpr int kMaxC = 4;                        // CTAs per cluster (N2 / 256)
constexpr int kEpiWarps = 4;
constexpr int kThreads = 64 + 32 * kEpiWarps;
// Shared memory: the C slots, the barriers, then as many ring stages as fit
// (C = 1: 6, C = 2: 5, C = 4: 3); the host computes the ring depth.
// ring_full[6], ring_empty[6], s_full[2], s_free[2], slot_full[4] (slot k holds CTA k's chunk;
// a peer's slot fills with its bulk copy), slot_empty (this CTA's own slot is free: every CTA
// consumed it), o_full, o_empty, drain, slot_written (the F warps finished writing this CTA's S' chunk)
constexpr int BAR_RF = 0, BAR_RE = 6, BAR_SF = 12, BAR_SFREE = 14, BAR_SLF = 16, BAR_SLE = 20, BAR_OF = 21,
              BAR_OE = 22, BAR_DRAIN = 23, BAR_SLW = 24, kNumBars = 25;
constexpr int kSmemLimit = 232448;
constexpr int kFixedBytes = 1024 + kNumBars * 8 + 16;  // alignment slack, barriers, misc
__host__ __device__ constexpr int ring_for(int C) {
  return (kSmemLimit - kFixedBytes - C * kSlotBytes) / kStageBytes > kMaxRing
             ? kMaxRing
             : (kSmemLimit - kFixedBytes - C * kSlotBytes) / kStageBytes;
}
__host__ __device__ constexpr int smem_for(int C) { return ring_for(C) * kStageBytes + C * kSlotBytes + kFixedBytes; }
constexpr int kTmemCols = 512;  // S0 [0,128), S1 [128,256), O [256,512)

struct Params {
  CUtensorMap tmA;   // {K, M, batch}, box {64, 128, 1}
  CUtensorMap tmW1;  // MN-major: {N1, K, batch} box {64, 64, 1}; K-major: {K, N1, batch} box {64, 128, 1}
  CUtensorMap tmW2;  // {N2, N1, batch}, box {64, 64, 1}
  void* out;        // fp32 or bf16 (out_bf16), element offsets below
  long long ldo, stride_out;
  int out_bf16;
  int M;             // rows of A per batch entry (the last 128-row strip may be ragged)
  int w1_k_major;
  int C;             // CTAs per cluster = ceil(N2 / 256)
  int n2;            // output columns (the last CTA's block may be ragged)
  int ring;          // ring stages (ring_for(C))
  int out_v8;        // the output base, row pitch and batch stride are 32-byte aligned
  int kblocks;       // ceil(K / 64): the last block's columns past K are zero-filled
  int rounds;        // ceil(N1 / (128 C)): chunks past N1 are zero (W1 and W2 zero-filled)
  int strips, items; // M / 128, batch * strips
  float scale;       // F(S) = max(scale S, 0)
  unsigned* status;
  long long timeout_cycles;
};

// OBF16: bf16 output (compile-time, one store path in the epilogue warps).
template <bool OBF16>
__global__ void __launch_bounds__(kThreads, 1) mlp_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kRing = p.ring;
  const int kOffRing = 0;
  const int kOffSlots = kRing * kStageBytes;
  const int kOffBars = kOffSlots + p.C * kSlotBytes;
  const int kOffMisc = kOffBars + kNumBars * 8;
  auto bar = [&](int i) -> uint32_t { return sbase + kOffBars + 8 * i; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  const WaitCtx wc{p.timeout_cycles, abort_flag, p.status};
  const int C = p.C;
  const uint32_t rank = cluster_ctarank();
  const int cid = (int)cluster_id_x(), ncl = (int)num_clusters_x();
  const int R = p.rounds;

  // The tensor-map fetches start before the barrier set-up, which they
  // overlap (the first TMA load waits for its map).
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmA);
    tma_prefetch_desc(&p.tmW1);
    tma_prefetch_desc(&p.tmW2);
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRing; ++i) {
      mbar_init(bar(BAR_RF + i), 1);
      mbar_init(bar(BAR_RE + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(BAR_SF + i), 1);
      mbar_init(bar(BAR_SFREE + i), kEpiWarps);
    }
    // A peer's slot: one arrival by this CTA's GEMM2 issuer (expecting the
    // copy's bytes) per round, armed for the first round here.
    for (int k = 0; k < C; ++k) {
      mbar_init(bar(BAR_SLF + k), 1);
      if (k != (int)rank) mbar_arrive_expect_tx(bar(BAR_SLF + k), kSlotBytes);
    }
    mbar_init(bar(BAR_SLE), C);   // one commit from every CTA's second GEMM on this CTA's chunk
    mbar_init(bar(BAR_OF), 1);
    mbar_init(bar(BAR_OE), kEpiWarps);
    mbar_init(bar(BAR_DRAIN), 1);
    mbar_init(bar(BAR_SLW), kEpiWarps);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t rs = 0, rph = 0, issued = 0;
      bool ok = true;
      auto acquire = [&]() -> uint32_t {
        if (!mbar_wait(bar(BAR_RE + rs), rph ^ 1, wc)) return 0;
        return 1;
      };
      auto advance = [&]() {
        ++issued;
        if (++rs == kRing) { rs = 0; rph ^= 1; }
      };
      auto load_g1 = [&](int strip, int b, int r) -> bool {
        const int h = r * C + (int)rank;  // this CTA's N1 chunk
        for (int kb = 0; kb < p.kblocks; ++kb) {
          if (!acquire()) return false;
          const uint32_t dst = sbase + kOffRing + rs * kStageBytes;
          const uint32_t fb = bar(BAR_RF + rs);
          mbar_arrive_expect_tx(fb, kStageBytes);
          tma_load_3d(dst, &p.tmA, fb, kb * 64, strip * 128, b);
          if (p.w1_k_major) {
            tma_load_3d(dst + 16384, &p.tmW1, fb, kb * 64, h * 128, b);
          } else {
            tma_load_3d(dst + 16384, &p.tmW1, fb, h * 128, kb * 64, b);
            tma_load_3d(dst + 16384 + 8192, &p.tmW1, fb, h * 128 + 64, kb * 64, b);
          }
          advance();
        }
        return true;
      };
      auto load_g2 = [&](int b, int r) -> bool {
        for (int i2 = 0; i2 < C; ++i2) {
          const int c2 = ((int)rank + i2) % C;  // the MMA issuer's chunk order: its own chunk first
          for (int kh = 0; kh < 2; ++kh) {
            if (!acquire()) return false;
            const uint32_t dst = sbase + kOffRing + rs * kStageBytes;
            const uint32_t fb = bar(BAR_RF + rs);
            const int row0 = (r * C + c2) * 128 + kh * 64;
            mbar_arrive_expect_tx(fb, kStageBytes);
#pragma unroll
            for (int i = 0; i < 4; ++i) tma_load_3d(dst + i * 8192, &p.tmW2, fb, (int)rank * 256 + 64 * i, row0, b);
            advance();
          }
        }
        return true;
      };
      for (int item = cid; ok && item < p.items; item += ncl) {
        const int b = item / p.strips, strip = item - b * p.strips;
        ok = load_g1(strip, b, 0) && (R < 2 || load_g1(strip, b, 1));
        for (int r = 0; ok && r < R; ++r) {
          if (r + 2 < R) ok = load_g1(strip, b, r + 2);  // same order as the MMA issuer
          if (ok) ok = load_g2(b, r);
        }
      }
      drain_ring(bar(BAR_RF), (uint32_t)kRing, issued, wc);  // no load of this CTA is still in flight
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(128, 128, p.w1_k_major ? 0u : 1u);
      const uint32_t id_o = idesc_bf16_f32(128, 256, 1u);
      uint32_t rs = 0, rph = 0;
      uint32_t g = 0;  // global round counter
      int t = 0;
      bool ok = true;
      // Stage-0 descriptors: A (X) tile, W1 tile (K- or MN-major), W2 tile
      // (MN-major, 64-column atoms 8 KB apart), and S' slot 0.
      constexpr uint32_t kStageStep = kStageBytes >> 4;
      const SDesc dx = sdesc_sw128(sbase + kOffRing, 16, 1024);
      const SDesc dw1 = sdesc_sw128(sbase + kOffRing + 16384, p.w1_k_major ? 16u : 8192u, 1024);
      const uint32_t w1_step = p.w1_k_major ? (32u >> 4) : (2048u >> 4);  // per 16 K elements
      const SDesc dw2 = sdesc_sw128(sbase + kOffRing, 8192, 1024);
      const SDesc dsl = sdesc_sw128(sbase + kOffSlots, 16, 1024);
      auto g1 = [&](uint32_t gg) -> bool {
        // The F warps must be done reading the S buffer's previous contents.
        if (!mbar_wait(bar(BAR_SFREE + (gg & 1)), ((gg >> 1) & 1) ^ 1, wc)) return false;
        tc_fence_after();
        const uint32_t d = tmem_base + (gg & 1) * 128;
        for (int kb = 0; kb < p.kblocks; ++kb) {
          if (!mbar_wait(bar(BAR_RF + rs), rph, wc)) return false;
          tc_fence_after();
          const uint32_t x_lo = dx.lo + rs * kStageStep, w_lo = dw1.lo + rs * kStageStep;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(d, x_lo + kk * (32u >> 4), dx.hi, w_lo + kk * w1_step, dw1.hi, id_s, (kb | kk) ? 1u : 0u);
          mma_commit(bar(BAR_RE + rs));
          if (++rs == kRing) { rs = 0; rph ^= 1; }
        }
        mma_commit(bar(BAR_SF + (gg & 1)));
        return true;
      };
      for (int item = cid; ok && item < p.items; item += ncl, ++t) {
        const uint32_t g0 = g;
        ok = g1(g0) && (R < 2 || g1(g0 + 1));
        for (int r = 0; ok && r < R; ++r, ++g) {
          // The next-but-one S chunk only needs the F warps to have read S(r):
          // issue it first so it overlaps the S' exchange of round r.
          if (r + 2 < R && !(ok = g1(g + 2))) break;
          if (r == 0 && !mbar_wait(bar(BAR_OE), (t & 1) ^ 1, wc)) { ok = false; break; }
          // The round's chunks, this CTA's own first (its F warps wrote it
          // locally), then the peers' in turn as their copies land, so the
          // second GEMM starts before the whole exchange is done.
          for (int i2 = 0; ok && i2 < C; ++i2) {
            const int c2 = ((int)rank + i2) % C;
            if (c2 == (int)rank) {
              if (!mbar_wait(bar(BAR_SLW), g & 1, wc)) { ok = false; break; }
            } else {
              if (!mbar_wait(bar(BAR_SLF + c2), g & 1, wc)) { ok = false; break; }
              mbar_arrive_expect_tx(bar(BAR_SLF + c2), kSlotBytes);  // arm the next round's copy
            }
            tc_fence_after();
            for (int kh = 0; kh < 2; ++kh) {
              if (!mbar_wait(bar(BAR_RF + rs), rph, wc)) { ok = false; break; }
              tc_fence_after();
              const uint32_t w_lo = dw2.lo + rs * kStageStep;
              const uint32_t a_lo = dsl.lo + ((uint32_t)(c2 * kSlotBytes + kh * 16384) >> 4);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_ss(tmem_base + 256, a_lo + kk * (32u >> 4), dsl.hi, w_lo + kk * (2048u >> 4), dw2.hi, id_o,
                       (r | i2 | kh | kk) ? 1u : 0u);
              mma_commit(bar(BAR_RE + rs));
              if (++rs == kRing) { rs = 0; rph ^= 1; }
            }
            // CTA c2 may refill its slot once every CTA has consumed it.
            if (ok) mma_commit_multicast(bar(BAR_SLE), (uint16_t)(1u << c2));
          }
          if (!ok) break;
        }
        if (!ok) break;
        mma_commit(bar(BAR_OF));
      }
      mma_commit(bar(BAR_DRAIN));
      mbar_wait<false, false>(bar(BAR_DRAIN), 0, wc);
      // All peers' multicast arrivals for the last round have landed here
      // (after an abort they may never come: stop at the abort flag).
      if (ok && g > 0) mbar_wait<false, true>(bar(BAR_SLE), (g - 1) & 1, wc);
    }
  } else {
    // ------------------------------------------------ F warps and epilogue
    const int q = warp & 3;
    const int row = 32 * q + lane;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    uint8_t* my_slot = smem + kOffSlots + rank * kSlotBytes;
    const uint32_t my_slot_addr = sbase + kOffSlots + rank * kSlotBytes;
    uint32_t g = 0;
    int t = 0;
    bool ok = true;
    for (int item = cid; ok && item < p.items; item += ncl, ++t) {
      const int b = item / p.strips, strip = item - b * p.strips;
      for (int r = 0; r < R; ++r, ++g) {
        const uint32_t sb = g & 1, u = g >> 1;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(BAR_SF + sb), u & 1, wc))) { ok = false; break; }
        tc_fence_after();
        // Read this S chunk into registers (F applied, packed to bf16) and
        // release its TMEM buffer at once, so the next-but-one chunk's GEMM1
        // can start while the slots are still being exchanged.
        uint32_t w[4][16];
        {
          float v[4][32];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(tmem_base + lane_off + sb * 128 + c * 32, v[c]);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[c][e] = fmaxf(v[c][e] * p.scale, 0.0f);
            pack_bf16(v[c], w[c]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_SFREE + sb));
        // This CTA's slot may be overwritten once every CTA consumed its previous chunk.
        if (!__all_sync(0xffffffffu, mbar_wait(bar(BAR_SLE), (g & 1) ^ 1, wc))) { ok = false; break; }
#pragma unroll
        for (int c = 0; c < 4; ++c) store_row_packed_sw128(my_slot, row, c * 32, w[c]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_SLW));
        if (warp == 2) {
          // The whole chunk is in this CTA's slot: publish it to the peers.
          if (!__all_sync(0xffffffffu, mbar_wait(bar(BAR_SLW), g & 1, wc))) { ok = false; break; }
          if (lane == 0) {
            // Each copy completes on the peer's barrier for this CTA's slot.
            for (int pr = 1; pr < C; ++pr) {
              const uint32_t peer = (rank + pr) % C;
              bulk_copy_to_peer(my_slot_addr, my_slot_addr, kSlotBytes, bar(BAR_SLF + (int)rank), peer);
            }
          }
        }
      }
      if (!ok) break;
      // Epilogue: this CTA's 128 x 256 block of O, straight from TMEM to HBM.
      if (!__all_sync(0xffffffffu, mbar_wait(bar(BAR_OF), t & 1, wc))) break;
      tc_fence_after();
      const long long orow = (long long)b * p.stride_out + (long long)(strip * 128 + row) * p.ldo + rank * 256;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        float v[32];
        tmem_ld32(tmem_base + lane_off + 256 + c * 32, v);
        tmem_wait_ld();
        const int col = (int)rank * 256 + c * 32;  // columns past N2 (ragged last block) are not stored
        if (strip * 128 + row < p.M && col < p.n2) {  // nor rows past M (ragged last strip)
          if (col + 32 <= p.n2) store_row<32>(p.out, OBF16, orow + c * 32, v, 1.0f, p.out_v8);
          else store_row_part<32>(p.out, OBF16, orow + c * 32, v, 1.0f, p.n2 - col);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_OE));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
  cluster_sync_all();
  // S' slots travel between the CTAs as bulk copies that complete on the
  // receiver's barrier.  After an abort (any bounded wait gave up: the
  // status word is set) some may still be in flight; every CTA has stopped
  // issuing them at the cluster barrier above, so all wait here before
  // leaving (the copies' sources and destinations both stay allocated).
  if (C > 1 && threadIdx.x == 0 && *reinterpret_cast<volatile unsigned*>(p.status) != 0u) settle_after_abort();
}

}  // namespace mlp


std::mutex g_mu;
bool g_prepared[64][10] = {};  // [device][MLP fp32 / bf16 out, attention variants 0..7]
// Resident clusters of C CTAs of the key-split attention kernel, by device,
// kernel variant and C (0: not queried yet, -1: none fit).
int g_attn_clusters[64][8][CF_MAX_KEY_SPLIT + 1] = {};

// Clusters of C CTAs of `fn` (a key-split attention variant) that fit on
// the current device at once; 0 if none (cached per device and variant).
int attn_max_clusters(const void* fn, int variant, int C) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  int& cached = g_attn_clusters[dev][variant][C];
  if (cached == 0) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)C, 1, 1);
    cfg.blockDim = dim3(attn::kThreads, 1, 1);
    cfg.dynamicSmemBytes = attn::kSmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int q = 0;
    if (cudaOccupancyMaxActiveClusters(&q, fn, &cfg) != cudaSuccess) {
      cudaGetLastError();
      q = 0;
    }
    cached = q > 0 ? q : -1;
  }
  return cached > 0 ? cached : 0;
}

cf_status prepare(int slot, const void* fn, int smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return CF_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_prepared[dev][slot]) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
      cudaGetLastError();
      return CF_ERR_CUDA;
    }
    g_prepared[dev][slot] = true;
  }
  return CF_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Every output row (and batch entry) starts on a 32-byte boundary.
bool out_aligned32(const cf_matrix* out, long long stride_out) {
  const long long es = out->dtype == CF_BF16 ? 2 : 4;
  return (reinterpret_cast<uintptr_t>(out->ptr) & 31u) == 0 && (out->ld * es) % 32 == 0 && (stride_out * es) % 32 == 0;
}

cf_status check_bf16_view(const cf_matrix* m, bool allow_trans) {
  if (!m || !m->ptr || m->dtype != CF_BF16) return CF_ERR_INVALID_ARG;
  if (m->trans != 0 && !(allow_trans && m->trans == 1)) return CF_ERR_INVALID_ARG;
  if (m->rows < 0 || m->cols < 0) return CF_ERR_INVALID_ARG;
  if (m->ld < (m->trans ? m->rows : m->cols)) return CF_ERR_INVALID_ARG;
  if (!aligned16(m->ptr) || (m->ld * 2) % 16 != 0) return CF_ERR_MISALIGNED;
  return CF_OK;
}



cf_status launch_mlp(const cf_matrix* A, const cf_matrix* W1, const cf_matrix* W2, const cf_b2b_desc* d,
                     cf_matrix* out, int64_t C, int sms, unsigned* status, cudaStream_t stream) {
  const int64_t M = A->rows, K = A->cols, N1 = W1->cols, N2 = W2->cols, batch = d->batch;
  const uint64_t bs = (uint64_t)batch;
  mlp::Params p;
  std::memset(&p, 0, sizeof(p));
  cf_status s;
  {
    const uint64_t dims[3] = {(uint64_t)K, (uint64_t)M, bs};
    const uint64_t st[2] = {(uint64_t)A->ld * 2, (uint64_t)(batch > 1 ? d->strideA : M * A->ld) * 2};
    const uint32_t box[3] = {64, 128, 1};
    if ((s = encode_tmap(&p.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, A->ptr, dims, st, box)) != CF_OK) return s;
  }
  p.w1_k_major = W1->trans;
  if (W1->trans) {  // stored N1 x K
    const uint64_t dims[3] = {(uint64_t)K, (uint64_t)N1, bs};
    const uint64_t st[2] = {(uint64_t)W1->ld * 2, (uint64_t)(batch > 1 ? d->strideW1 : N1 * W1->ld) * 2};
    const uint32_t box[3] = {64, 128, 1};
    if ((s = encode_tmap(&p.tmW1, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, W1->ptr, dims, st, box)) != CF_OK) return s;
  } else {          // stored K x N1
    const uint64_t dims[3] = {(uint64_t)N1, (uint64_t)K, bs};
    const uint64_t st[2] = {(uint64_t)W1->ld * 2, (uint64_t)(batch > 1 ? d->strideW1 : K * W1->ld) * 2};
    const uint32_t box[3] = {64, 64, 1};
    if ((s = encode_tmap(&p.tmW1, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, W1->ptr, dims, st, box)) != CF_OK) return s;
  }
  {
    const uint64_t dims[3] = {(uint64_t)N2, (uint64_t)N1, bs};
    const uint64_t st[2] = {(uint64_t)W2->ld * 2, (uint64_t)(batch > 1 ? d->strideW2 : N1 * W2->ld) * 2};
    const uint32_t box[3] = {64, 64, 1};
    if ((s = encode_tmap(&p.tmW2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, W2->ptr, dims, st, box)) != CF_OK) return s;
  }
  p.out = out->ptr;
  p.out_bf16 = out->dtype == CF_BF16 ? 1 : 0;
  p.ldo = out->ld;
  p.stride_out = batch > 1 ? d->strideOut : 0;
  p.out_v8 = out_aligned32(out, p.stride_out) ? 1 : 0;
  p.C = (int)C;
  p.n2 = (int)N2;
  p.ring = mlp::ring_for((int)C);
  p.kblocks = (int)((K + 63) / 64);
  p.rounds = (int)((N1 + 128 * C - 1) / (128 * C));
  p.M = (int)M;
  p.strips = (int)((M + 127) / 128);
  p.items = (int)(batch * p.strips);
  p.scale = d->mid_op == CF_MID_RELU ? 1.0f : d->mid_scale;
  p.status = status;
  p.timeout_cycles = wait_timeout_cycles();
  const void* fn = p.out_bf16 ? reinterpret_cast<const void*>(&mlp::mlp_kernel<true>)
                              : reinterpret_cast<const void*>(&mlp::mlp_kernel<false>);
  const int smem = mlp::smem_for((int)C);
  if ((s = prepare(p.out_bf16 ? 1 : 0, fn, mlp::smem_for(1))) != CF_OK) return s;  // the largest layout
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(mlp::kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3((unsigned)C, 1, 1);
  int maxc = 0;
  if (cudaOccupancyMaxActiveClusters(&maxc, fn, &cfg) != cudaSuccess || maxc < 1) {
    cudaGetLastError();
    return CF_ERR_CUDA;
  }
  const int64_t ncl = p.items < maxc ? p.items : maxc;
  cfg.gridDim = dim3((unsigned)(ncl * C), 1, 1);
  void* args[] = {&p};
  if (cudaLaunchKernelExC(&cfg, fn, args) != cudaSuccess) {
    cudaGetLastError();
    return CF_ERR_CUDA;
  }
  return CF_OK;
}
}  // namespace
}  // namespace cf

using namespace cf;

extern "C" cf_status cf_b2bgemm(const cf_matrix* A, const cf_matrix* W1, const cf_matrix* W2, const cf_b2b_desc* d,
                                cf_matrix* out, void* stream) {
  cf_status s;
  if (!d || d->version < 1 || d->version > CF_B2B_VERSION || d->batch < 1) return CF_ERR_INVALID_ARG;
  if (d->mid_op < CF_MID_RELU || d->mid_op > CF_MID_SCALE_SOFTMAX || !std::isfinite(d->mid_scale))
    return CF_ERR_INVALID_ARG;
  // The key_split field exists from version 2 (never read from a version-1 struct).
  const int key_split = d->version >= 2 ? d->key_split : 0;
  if (key_split < 0 || key_split > CF_MAX_KEY_SPLIT) return CF_ERR_INVALID_ARG;
  // The softmax's running max is taken on the unscaled logits: its scale
  // must be positive (a temperature).
  if (d->mid_op == CF_MID_SCALE_SOFTMAX && !(d->mid_scale > 0.0f)) return CF_ERR_INVALID_ARG;
  if (d->out_dtype != CF_FP32 && d->out_dtype != CF_BF16) return CF_ERR_INVALID_ARG;
  if ((s = check_bf16_view(A, false)) != CF_OK) return s;
  if ((s = check_bf16_view(W1, true)) != CF_OK) return s;
  if ((s = check_bf16_view(W2, false)) != CF_OK) return s;
  if (!out || !out->ptr || out->dtype != d->out_dtype || out->trans) return CF_ERR_INVALID_ARG;
  if (out->ld < out->cols) return CF_ERR_INVALID_ARG;
  const int64_t out_elem = out->dtype == CF_BF16 ? 2 : 4;
  if (!aligned16(out->ptr) || (out->ld * out_elem) % 16 != 0) return CF_ERR_MISALIGNED;
  const int64_t M = A->rows, K = A->cols, N1 = W1->cols, N2 = W2->cols, batch = d->batch;
  if (W1->rows != K || W2->rows != N1 || out->rows != M || out->cols != N2) return CF_ERR_INVALID_ARG;
  if (d->strideA < 0 || d->strideW1 < 0 || d->strideW2 < 0 || d->strideOut < 0) return CF_ERR_INVALID_ARG;
  // Inputs may overlap between batch entries (they are only read); outputs
  // must not, or the entries' stores would race.
  if (batch > 1 && M > 0 && d->strideOut < (M - 1) * out->ld + N2) return CF_ERR_INVALID_ARG;
  if (batch > 1 && ((d->strideA * 2) % 16 || (d->strideW1 * 2) % 16 || (d->strideW2 * 2) % 16 ||
                    (d->strideOut * out_elem) % 16))
    return CF_ERR_MISALIGNED;
  if (M == 0 || N2 == 0) return CF_OK;

  // Attention shape: W1 stored transposed (N1 x K), head dims K, N2 <= 128
  // (K % 8 == 0), any N1 >= 1 (a ragged last 128-key chunk is masked).
  const bool attn_shape = W1->trans == 1 && K % 8 == 0 && K >= 8 && K <= 128 && N2 >= 1 && N2 <= 128 && N1 >= 1;
  // MLP shape: N2 <= 256 C with C <= 4 CTAs per cluster (the last CTA's
  // block may be ragged), any N1 >= 1, K >= 8 (a K below 64 is one
  // zero-filled 64-wide block), elementwise F only.
  const int64_t C = (N2 + 255) / 256;
  const bool mlp_shape = !attn_shape && d->mid_op != CF_MID_SCALE_SOFTMAX && K % 8 == 0 && K >= 8 && C >= 1 &&
                         C <= mlp::kMaxC && N1 >= 1;
  if (!attn_shape && !mlp_shape) return CF_ERR_UNSUPPORTED_SHAPE;

  int sms = 0;
  unsigned* status = nullptr;
  if ((s = device_query(&sms, &status)) != CF_OK) return s;
  if (mlp_shape) return launch_mlp(A, W1, W2, d, out, C, sms, status, static_cast<cudaStream_t>(stream));
  attn::Params p;
  std::memset(&p, 0, sizeof(p));
  const uint64_t bs = (uint64_t)(batch > 1 ? batch : 1);
  // K < 128 or N2 < 128 (head dims below 128): the columns past K of Q and
  // K, and past N2 of V, load as zeros, adding nothing to S and giving O
  // zero columns that are not stored; rows of K and V past N1 load as zeros.
  {
    const uint64_t dims[3] = {(uint64_t)K, (uint64_t)M, bs};
    const uint64_t st[2] = {(uint64_t)A->ld * 2, (uint64_t)(batch > 1 ? d->strideA : M * A->ld) * 2};
    const uint32_t box[3] = {64, 128, 1};
    if ((s = encode_tmap(&p.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, A->ptr, dims, st, box)) != CF_OK) return s;
  }
  {
    const uint64_t dims[3] = {(uint64_t)K, (uint64_t)N1, bs};
    const uint64_t st[2] = {(uint64_t)W1->ld * 2, (uint64_t)(batch > 1 ? d->strideW1 : N1 * W1->ld) * 2};
    const uint32_t box[3] = {64, 128, 1};
    if ((s = encode_tmap(&p.tmW1, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, W1->ptr, dims, st, box)) != CF_OK) return s;
  }
  {
    const uint64_t dims[3] = {(uint64_t)N2, (uint64_t)N1, bs};
    const uint64_t st[2] = {(uint64_t)W2->ld * 2, (uint64_t)(batch > 1 ? d->strideW2 : N1 * W2->ld) * 2};
    const uint32_t box[3] = {64, 128, 1};
    if ((s = encode_tmap(&p.tmW2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, W2->ptr, dims, st, box)) != CF_OK) return s;
  }
  p.out = out->ptr;
  p.out_bf16 = out->dtype == CF_BF16 ? 1 : 0;
  p.ldo = out->ld;
  p.stride_out = batch > 1 ? d->strideOut : 0;
  p.out_v8 = out_aligned32(out, p.stride_out) ? 1 : 0;
  p.batch = (int)bs;
  p.M = (int)M;
  p.m_blocks = (int)((M + 127) / 128);
  p.n1_blocks = (int)((N1 + 127) / 128);
  p.kv_last = (int)(N1 - 128 * (p.n1_blocks - 1));
  p.n2 = (int)N2;
  p.items = p.batch * p.m_blocks;
  p.softmax = d->mid_op == CF_MID_SCALE_SOFTMAX ? 1 : 0;
  p.scale = d->mid_op == CF_MID_RELU ? 1.0f : d->mid_scale;
  p.status = status;
  p.timeout_cycles = wait_timeout_cycles();
  // Key split (the review's Eq. (5) over a cluster).  AUTO splits only
  // when the query blocks are fewer than the SMs (one CTA per block would
  // leave SMs idle), every CTA keeps at least kSplitMinChunks 128-key
  // chunks (measured on GB300: the merge and the cluster launch cost about
  // as much as 6-7 chunks of one CTA's pipeline, so a 2-chunk row loses
  // 13.5 -> 19.6 us when split), and all the clusters are resident at once
  // (a second wave of clusters doubles the time); it takes the largest such
  // cluster.  Otherwise one CTA per block walks all keys (the C = 1 online
  // form).  The chunk count per CTA is rounded up and the CTA count
  // recomputed from it, so that no CTA's key range is empty.
  constexpr int kSplitMinChunks = 8;
  const bool rag = (p.softmax && p.kv_last < attn::kTile) || p.n2 < attn::kTile;
  const int base_variant = (rag ? 1 : 0) + (p.out_bf16 ? 2 : 0);
  const void* fns[8] = {reinterpret_cast<const void*>(&attn::attn_kernel<false, false, false>),
                        reinterpret_cast<const void*>(&attn::attn_kernel<true, false, false>),
                        reinterpret_cast<const void*>(&attn::attn_kernel<false, true, false>),
                        reinterpret_cast<const void*>(&attn::attn_kernel<true, true, false>),
                        reinterpret_cast<const void*>(&attn::attn_kernel<false, false, true>),
                        reinterpret_cast<const void*>(&attn::attn_kernel<true, false, true>),
                        reinterpret_cast<const void*>(&attn::attn_kernel<false, true, true>),
                        reinterpret_cast<const void*>(&attn::attn_kernel<true, true, true>)};
  int split = key_split == 0 ? 1 : key_split;
  if (key_split == 0 && p.items < sms && p.n1_blocks >= 2 * kSplitMinChunks) {
    if ((s = prepare(2 + base_variant + 4, fns[base_variant + 4], attn::kSmemBytes)) != CF_OK) return s;
    int cmax = p.n1_blocks / kSplitMinChunks;
    if (cmax > CF_MAX_KEY_SPLIT) cmax = CF_MAX_KEY_SPLIT;
    for (int c = cmax; c >= 2; --c) {
      if (p.items <= attn_max_clusters(fns[base_variant + 4], base_variant + 4, c)) {
        split = c;
        break;
      }
    }
  }
  if (split > p.n1_blocks) split = p.n1_blocks;
  if (split >= 2) {
    p.nb_per = (p.n1_blocks + split - 1) / split;
    split = (p.n1_blocks + p.nb_per - 1) / p.nb_per;
  }
  p.split = split >= 2 ? split : 1;
  const int variant = base_variant + (p.split > 1 ? 4 : 0);
  if ((s = prepare(2 + variant, fns[variant], attn::kSmemBytes)) != CF_OK) return s;
  void* args[] = {&p};
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(attn::kThreads, 1, 1);
  cfg.dynamicSmemBytes = attn::kSmemBytes;
  cfg.stream = static_cast<cudaStream_t>(stream);
  if (p.split > 1) {
    // One cluster of `split` CTAs per query block, not persistent: clusters
    // do not wait on each other, so any number of them may queue.
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.split;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (attn_max_clusters(fns[variant], variant, p.split) < 1) return CF_ERR_UNSUPPORTED_SHAPE;  // none fits
    if ((int64_t)p.items * p.split > INT32_MAX) return CF_ERR_UNSUPPORTED_SHAPE;
    cfg.gridDim = dim3((unsigned)(p.items * p.split), 1, 1);
  } else {
    cfg.gridDim = dim3((unsigned)(p.items < sms ? p.items : sms), 1, 1);  // persistent
  }
  if (cudaLaunchKernelExC(&cfg, fns[variant], args) != cudaSuccess) {
    cudaGetLastError();
    return CF_ERR_CUDA;
  }
  return CF_OK;
}
