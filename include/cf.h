/*
 * cf.h -- C ABI of the GB300 (sm_103a) fused GEMM-epilogue / B2BGEMM library.
 *
 * What the library computes comes from the Pith review of "ComFuse: Fusing
 * Complex Memory-Intensive Subgraphs with Compute-Intensive Kernels For
 * Modern GPU Architectures" (arXiv 2608.03537):
 *   - "What carries the argument" (Stage-Stream Execution Model): the GEMM's
 *     output tiles stream, while still on chip, through elementwise nodes at
 *     fragment granularity; each reduction is a stage boundary aggregated
 *     hierarchically (within a thread/warp, across warps in shared memory,
 *     across CTAs of a thread-block cluster through distributed shared memory).
 *   - Referee report, major comment 1 [Sec. III, Eq. (1)]: a reduction along
 *     the column dimension of P only needs the row strip {T_{m,n}}_n; when the
 *     strip is wider than one cluster a multi-cluster fallback is required
 *     (this library exchanges per-tile partial statistics through a small
 *     caller-provided workspace).
 *   - "What carries the argument" and major comment 2 [Sec. IV-A,
 *     Eqs. (3)-(5)]: back-to-back GEMM (B2BGEMM) keeps the post-processed
 *     intermediate tile on chip and accumulates the second GEMM from it, so
 *     the intermediate matrix never reaches global memory.
 *
 * Conventions for every entry point:
 *   - Matrices are described by cf_matrix: element (r, c) of the logical
 *     rows x cols matrix is at ptr[r * ld + c] when trans == 0 and at
 *     ptr[c * ld + r] when trans == 1 (ld in elements).  All data pointers
 *     are DEVICE pointers of the current CUDA device, owned by the caller;
 *     the library never frees or retains them after the call returns.
 *   - Calls enqueue work on `stream` (a cudaStream_t, NULL = legacy default
 *     stream) and return without synchronising.  Errors found on the host
 *     are returned synchronously and nothing is enqueued.  A device-side
 *     bounded wait that gives up is reported by cf_last_device_status().
 *   - There is no CPU fallback: without an sm_103 device every compute entry
 *     point returns CF_ERR_UNSUPPORTED_DEVICE (or CF_ERR_NO_DEVICE).
 *   - Entry points are thread-safe for distinct streams; tensor-map encoding
 *     is done per call on the host.  Host-side state: a per-device cache
 *     (device properties, kernel attributes, occupancy answers and the
 *     device addresses of the library's __device__ variables).  Device-side
 *     state: the status word (all entry points), the 4 MiB scratch array of
 *     cf_gemm_epilogue_noalloc, and the per-chunk statistics arrays of the
 *     unfused column path; each of the last two is shared by every call of
 *     its entry point (see there).
 *   - The cache assumes a device's context lives as long as the process:
 *     after cudaDeviceReset() on a device, the library must not be used on
 *     that device again in the same process (its cached device addresses
 *     would point into the destroyed context).
 */
#ifndef CF_GB300_H
#define CF_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CF_API __attribute__((visibility("default")))
#else
#define CF_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define CF_ABI_VERSION 1

typedef enum {
  CF_OK = 0,
  CF_ERR_INVALID_ARG = 1,        /* null pointer, bad enum, inconsistent dims     */
  CF_ERR_UNSUPPORTED_SHAPE = 2,  /* shape outside a call's shape rules (below)   */
  CF_ERR_MISALIGNED = 3,         /* pointer or leading dim not 16-byte aligned   */
  CF_ERR_UNSUPPORTED_DEVICE = 4, /* current device is not compute capability 10.3 */
  CF_ERR_CUDA = 5,               /* a CUDA runtime/driver call failed            */
  CF_ERR_TIMEOUT = 6,            /* a device-side bounded wait gave up           */
  CF_ERR_WORKSPACE = 7,          /* workspace missing or smaller than required   */
  CF_ERR_NO_DEVICE = 8           /* no CUDA device visible                       */
} cf_status;

typedef enum { CF_BF16 = 0, CF_FP32 = 1 } cf_dtype;

/* A strided 2-D view of caller-owned device memory (see conventions above). */
typedef struct {
  void* ptr;
  int32_t dtype; /* cf_dtype */
  int32_t trans; /* 0: row-major view, 1: the stored matrix is the transpose */
  int64_t rows;
  int64_t cols;
  int64_t ld;    /* leading dimension of the stored matrix, in elements */
} cf_matrix;

/* Epilogue operations.  Elementwise ops (kind < 16) are applied in order to
 * every element of P = A.B; reductions (kind >= 16) are stage boundaries,
 * along each row (over n) or, with descriptor version 3 and CF_AXIS_COLS,
 * down each column (over m; the formulas below then reduce over m and the
 * vectors stay indexed by n).  A program has at most two reductions, and if
 * it has any it ends with one: [elementwise...] [R0 [elementwise...]] R1.  A
 * first reduction R0 (descriptor version 2) must be LayerNorm or RMSNorm;
 * its affine vectors are stage0_gamma / stage0_beta, the last reduction's
 * are the gamma / beta arguments. */
typedef enum {
  CF_OP_BIAS = 1,            /* x += bias[n]                                        */
  CF_OP_SCALE = 2,           /* x *= scalar                                         */
  CF_OP_RELU = 3,            /* x = max(x, 0)                                       */
  CF_OP_GELU_TANH = 4,       /* x = 0.5 x (1 + tanh(sqrt(2/pi)(x + 0.044715 x^3)))  */
  CF_OP_ADD_RESIDUAL = 5,    /* x += residual[m][n] (descriptor version 2)          */
  CF_OP_ROW_LAYERNORM = 16,  /* y = gamma[n] (x - mean) / sqrt(var + scalar) + beta[n], biased var */
  CF_OP_ROW_RMSNORM = 17,    /* y = gamma[n] x / sqrt(mean(x^2) + scalar)           */
  CF_OP_ROW_SOFTMAX = 18     /* y = exp(x - max) / sum(exp(x - max))                */
} cf_op_kind;

typedef struct {
  int32_t kind;  /* cf_op_kind */
  float scalar;  /* the scale for CF_OP_SCALE, eps for the norms, unused otherwise */
} cf_op;

#define CF_EPI_VERSION 3  /* versions 1 (no residual) and 2 (no axis) are still accepted */

/* Axis of an epilogue program's reductions (descriptor version 3). */
typedef enum {
  CF_AXIS_ROWS = 0, /* along each row of P = A.B (over n) */
  CF_AXIS_COLS = 1  /* down each column of P (over m): the complementary strip */
} cf_axis;
#define CF_EPI_MAX_OPS 8

/* Row-statistics exchange used when a row spans several CTAs. */
typedef enum {
  CF_XCHG_AUTO = 0,    /* cluster DSMEM when the strip fits one cluster, else workspace */
  CF_XCHG_CLUSTER = 1, /* force the thread-block-cluster DSMEM exchange (<= 16 CTAs)  */
  CF_XCHG_GLOBAL = 2,  /* force per-tile partial statistics through the workspace    */
  /* The workspace exchange with work items claimed from a counter by the
   * CTAs that run (one reduction stage only): for a GPU shared with other
   * work (other streams, MPS), where not every CTA of the launch may become
   * resident.  Slower on a GPU of its own (about 4-25% on the measured
   * shapes). */
  CF_XCHG_GLOBAL_DYNAMIC = 3
} cf_exchange;

/* A tiny epilogue program: a linear chain of ops (the Stage-Stream model:
 * elementwise nodes, then up to two reduction stages, the last one ending
 * the program; see cf_op_kind). */
typedef struct {
  uint32_t version;  /* 1, 2 or 3 (CF_EPI_VERSION); version 1 ends after `exchange`,
                        version 2 after `stage0_beta` */
  uint32_t n_ops;    /* 0..CF_EPI_MAX_OPS */
  cf_op ops[CF_EPI_MAX_OPS];
  int32_t out_dtype; /* cf_dtype of `out`: CF_FP32, or CF_BF16 (each value
                        rounded to nearest even from the fp32 epilogue
                        result; the fused entry points only) */
  int32_t exchange;  /* cf_exchange */
  /* Version 2: the matrix read by CF_OP_ADD_RESIDUAL (the residual stream of
   * a post-norm block): M x N, fp32 or bf16, trans == 0, pointer and leading
   * dim 16-byte aligned, caller-owned.  Ignored (may be all zero) when the
   * program has no CF_OP_ADD_RESIDUAL; the fused kernel reads it once. */
  cf_matrix residual;
  /* Version 2: affine vectors (fp32 [N], 16-byte aligned) of the first of two
   * row reductions; NULL means gamma = 1 / beta = 0 (no affine transform). */
  const float* stage0_gamma;
  const float* stage0_beta;
  /* Version 3: cf_axis of the program's reductions.  CF_AXIS_COLS reduces
   * down each column of P (LayerNorm / RMSNorm / softmax over m, e.g. a
   * batch normalisation); every vector (bias, gamma, beta, stage0_*) stays
   * indexed by the column n, so for columns gamma/beta are constant along
   * the reduction.  CF_AXIS_COLS needs B given as its N x K transpose
   * (trans == 1); the cluster exchange then takes M <= 4096.  Programs
   * without a reduction ignore the axis. */
  int32_t axis;
} cf_epi_desc;

/*
 * cf_gemm_epilogue -- out = epilogue(A . B), fused in one kernel.
 *
 * Passages: the Stage-Stream Execution Model (ComFuse review, "What carries
 * the argument": accumulator tiles stream on chip through elementwise nodes,
 * each reduction is a stage boundary aggregated hierarchically) and the
 * tile-strip locality of a row reduction (referee report, major comment 1
 * [Sec. III, Eq. (1)]: a row depends only on its strip {T_{m,n}}_n, and a
 * strip wider than one cluster needs a multi-cluster fallback; column
 * reductions use the complementary strip).
 *
 *   A    : M x K, bf16, trans == 0 (K contiguous).
 *   B    : K x N, bf16; trans == 0 (stored K x N, N contiguous) or
 *          trans == 1 (stored N x K, K contiguous, e.g. a Linear weight).
 *   bias, gamma, beta : device fp32 vectors of length N; required only when
 *          the program uses CF_OP_BIAS / a norm (beta only for LayerNorm);
 *          may be NULL otherwise.
 *   out  : M x N, trans == 0, dtype == epi->out_dtype (fp32 or bf16).
 *   workspace : device memory of at least cf_workspace_size(...) bytes when
 *          that is non-zero (per-tile partial row statistics and arrival
 *          counters; the call clears the counters on `stream`).  Its contents
 *          are scratch; concurrent calls must use distinct workspaces.
 *
 * Shape rules (this version): any M >= 0 (a ragged last 128-row strip is
 * handled), any N >= 0 (a ragged last 256-column tile is handled: its
 * columns past N stay out of the row statistics and are not stored), K % 8
 * == 0 with K >= 8 (a ragged last, or only, 64-wide K block reads zeros
 * past K), all
 * pointers and leading dims 16-byte aligned; the cluster exchange takes rows
 * of at most 16 tiles (N <= 4096).  Through the workspace every tile of a
 * row strip waits for its strip-mates and each CTA (or CTA pair) holds two
 * tiles.  By default a CTA takes fixed tiles in a strip-major order, which
 * needs every CTA of the launch to become resident (the grid never exceeds
 * what fits on the device; kernels running beside it only delay it) and a
 * row of at most as many tiles as CTAs: a CTA must not hold two tiles of
 * one row.  With one reduction stage, wider rows (up to twice the CTAs) and
 * CF_XCHG_GLOBAL_DYNAMIC take tiles from a counter in the workspace instead,
 * claimed by the CTAs that run, so a row may span at most twice the CTAs
 * that run: N <= 77,824 on a 152-SM GB300 (CTA pairs up to N <= 38,912,
 * wider rows on 1-CTA tiles).  With two chained stages rows are limited to
 * N <= 38,912 (CTA pairs up to N <= 19,456) and CF_XCHG_GLOBAL_DYNAMIC
 * returns CF_ERR_UNSUPPORTED_SHAPE.  Wider rows return
 * CF_ERR_UNSUPPORTED_SHAPE.  Violations return CF_ERR_UNSUPPORTED_SHAPE /
 * CF_ERR_MISALIGNED without launching anything.  M == 0 or N == 0 returns
 * CF_OK without launching.
 */
CF_API cf_status cf_gemm_epilogue(const cf_matrix* A, const cf_matrix* B,
                           const float* bias, const float* gamma, const float* beta,
                           const cf_epi_desc* epi, cf_matrix* out,
                           void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace cf_gemm_epilogue needs for these operands (0 if none). */
CF_API size_t cf_workspace_size(const cf_matrix* A, const cf_matrix* B, const cf_epi_desc* epi);

/* Size of the library-owned scratch array used by cf_gemm_epilogue_noalloc. */
#define CF_NOALLOC_WORKSPACE_BYTES (4u << 20)

/*
 * cf_gemm_epilogue_noalloc -- cf_gemm_epilogue for callers that cannot
 * allocate device memory.  (The paper has no counterpart; this is a library
 * convenience.)
 *
 * Who needs it: callers that must not call cudaMalloc or any other
 * allocator where they run this kernel -- code with latency bounds (an
 * allocation may synchronise the device), plugins whose host framework owns
 * all device memory and offers no allocator, and steady-state loops that
 * must not allocate.  Rows wider than one 256-column tile need scratch for
 * partial row statistics; this call takes it from a static device array of
 * CF_NOALLOC_WORKSPACE_BYTES (4 MiB) inside the library instead of a
 * caller-provided workspace.  It calls no allocator.
 *
 * Arguments and results are those of cf_gemm_epilogue without the workspace.
 * Problems needing more scratch than the array holds (cf_workspace_size >
 * CF_NOALLOC_WORKSPACE_BYTES: roughly M * N > 2^27 with one reduction
 * stage, M * N > 2^26 with two chained stages, which need one statistics
 * region each; cf_workspace_size is the exact test) return
 * CF_ERR_WORKSPACE and enqueue nothing.
 *
 * Sharing: all calls in the process share the one array per device, which
 * keeps the last call's contents; each call clears the part that must start
 * at zero on its own stream.  Calls whose executions overlap on the GPU race
 * on the array and must be serialised by the caller.  Every GPU that loads
 * the library holds the array until the process exits.  The first call on a
 * device looks up the array's address on that device (which must be
 * current); make that first call before any stream capture.
 */
CF_API cf_status cf_gemm_epilogue_noalloc(const cf_matrix* A, const cf_matrix* B,
                                          const float* bias, const float* gamma, const float* beta,
                                          const cf_epi_desc* epi, cf_matrix* out, void* stream);

/* Intermediate ops of a B2BGEMM. */
typedef enum {
  CF_MID_RELU = 1,          /* S' = max(S, 0)                    */
  CF_MID_SCALE_RELU = 2,    /* S' = max(scale S, 0)              */
  CF_MID_SCALE_SOFTMAX = 3  /* S' = row softmax of (scale S)     */
} cf_mid_op;

#define CF_B2B_VERSION 2  /* version 1 (no key_split) is still accepted */

/* Largest key split (CTAs per query block) of the attention shape. */
#define CF_MAX_KEY_SPLIT 8

typedef struct {
  uint32_t version;  /* 1 or 2 (CF_B2B_VERSION); version 1 ends after strideOut */
  int32_t mid_op;    /* cf_mid_op */
  float mid_scale;   /* scale for the SCALE_* ops */
  int32_t out_dtype; /* cf_dtype of `out`: CF_FP32, or CF_BF16 (rounded to
                        nearest even from the fp32 accumulator; cf_b2bgemm
                        only) */
  int64_t batch;     /* number of independent problems (>= 1) */
  int64_t strideA, strideW1, strideW2, strideOut; /* elements between problems; inputs may
                                                     overlap (read only), outputs must not:
                                                     strideOut >= (M - 1) * ld + N2 */
  /* Version 2, attention shape only (ignored by the MLP shape): how many
   * CTAs share the N1 (key) range of one 128-row block of A.  0: chosen per
   * shape (split only when the row blocks are fewer than the SMs, into as
   * many CTAs as keep every SM busy); 1: one CTA walks all of N1;
   * 2..CF_MAX_KEY_SPLIT: that many CTAs of a thread-block cluster (fewer
   * when N1 has fewer 128-key chunks, or when the count must shrink so that
   * every CTA gets at least one chunk), each over its own key range,
   * merged on chip (see cf_b2bgemm).  Other values: CF_ERR_INVALID_ARG. */
  int32_t key_split;
} cf_b2b_desc;

/*
 * cf_b2bgemm -- out = bf16_rne(F(A . W1)) . W2 per batch entry, fused: the
 * intermediate S' never reaches global memory.
 *
 * Passages: the B2BGEMM schedule (ComFuse review, "What carries the
 * argument": the post-processed intermediate tile stays on chip and the
 * second GEMM's output accumulation is distributed across the cluster) and
 * referee report, major comment 2 [Sec. IV-A, Eqs. (3)-(5)] (S = A W1, the
 * tile transform F, O accumulated over the set C of co-scheduled CTAs, with
 * partial results aggregated across C).
 *
 *   A   : M x K bf16, trans == 0.
 *   W1  : K x N1 bf16; trans == 0 (stored K x N1) or trans == 1 (stored
 *         N1 x K, e.g. the key matrix of attention, giving S = Q K^T).
 *   W2  : N1 x N2 bf16, trans == 0 (stored N1 x N2, e.g. the value matrix).
 *   out : M x N2, trans == 0, dtype == desc->out_dtype (fp32 or bf16).
 *   The softmax mid op normalises each row of S over all N1 columns.
 *
 * Attention shape, key split (desc->key_split): the CTAs of a cluster each
 * run GEMM1 -> F -> GEMM2 over their own key range with the online softmax
 * statistics (m_c, l_c) and partial output O_c, then merge them through
 * distributed shared memory as in Eq. (5): m = max_c m_c,
 * l = sum_c l_c exp(m_c - m), O = sum_c O_c exp(m_c - m) / l (for ReLU,
 * O = sum_c O_c), summed in cluster-rank order.  Nothing of S, S' or the
 * partial outputs reaches global memory.  A forced split whose cluster
 * cannot be resident returns CF_ERR_UNSUPPORTED_SHAPE.
 *
 * Shape rules (this version), two kernels:
 *   attention shape: W1 given transposed (trans == 1), head dims K <= 128
 *     (K % 8 == 0) and N2 <= 128 (both computed as 128 with zero padding),
 *     any N1 >= 1 (keys past N1 in the last 128-key chunk are masked); any
 *     mid op (the softmax normalises over all N1);
 *   MLP shape: mid op ReLU or scaled ReLU, K % 8 == 0 with K >= 8,
 *     N2 <= 1024 (C = ceil(N2 / 256) CTAs per cluster), any N1 >= 1.
 *   The softmax mid op needs mid_scale > 0 (CF_ERR_INVALID_ARG otherwise).
 *   Both: any M >= 0 (a ragged last 128-row block is handled), pointers and
 *   leading dims 16-byte aligned.  Other shapes return
 *   CF_ERR_UNSUPPORTED_SHAPE without launching anything.
 */
CF_API cf_status cf_b2bgemm(const cf_matrix* A, const cf_matrix* W1, const cf_matrix* W2,
                     const cf_b2b_desc* desc, cf_matrix* out, void* stream);

/*
 * cf_unfused_gemm_epilogue -- the unfused comparison path: a cuBLASLt GEMM
 * writes P (M x N fp32) to `intermediate`, then a separate row-epilogue
 * kernel reads it back and writes `out`.  Same program semantics as
 * cf_gemm_epilogue (row or column reductions), fp32 `out` only.
 * `intermediate` is caller-owned device memory of M * N * 4 bytes.  Column
 * reductions (N <= 65536) keep per-chunk statistics in a static device array
 * of the library (6 MB + 0.5 MB per device, held until the process exits):
 * column calls whose executions overlap on the GPU race on it and must be
 * serialised by the caller.
 */
CF_API cf_status cf_unfused_gemm_epilogue(const cf_matrix* A, const cf_matrix* B,
                                   const float* bias, const float* gamma, const float* beta,
                                   const cf_epi_desc* epi, cf_matrix* out,
                                   float* intermediate, void* stream);

/*
 * cf_unfused_b2bgemm -- unfused comparison path for B2BGEMM: cuBLASLt GEMM1
 * to `s_buf` (M x N1 fp32), a mid-op kernel writing bf16 S' to `p_buf`
 * (M x N1 bf16), cuBLASLt GEMM2 to `out` (fp32 or bf16).  Same semantics
 * as cf_b2bgemm.
 */
CF_API cf_status cf_unfused_b2bgemm(const cf_matrix* A, const cf_matrix* W1, const cf_matrix* W2,
                             const cf_b2b_desc* desc, cf_matrix* out,
                             float* s_buf, void* p_buf, void* stream);

/*
 * Cost model (host only, no device access): predicts whether fusing pays.
 *
 * The ComFuse review's suggested extension ("If this is right", third
 * bullet): compare the predicted GEMM time with the predicted epilogue time
 * and fuse only when the GEMM is heavy enough to hide the epilogue.  The
 * fused kernel's main loop and epilogue overlap tile by tile (two TMEM
 * accumulators), so a fused tile costs max(main loop, epilogue + exchange);
 * the unfused path pays the GEMM, then a second kernel that reads the
 * intermediate back from HBM.  Efficiencies are calibrated on a GB300 (the
 * fused kernels' measured fractions of the tensor peak, cuBLASLt's, and the
 * copy bandwidth); the numbers are estimates, not guarantees.
 */
typedef struct {
  double tensor_tflops; /* dense bf16 tensor peak (TFLOP/s); <= 0: 1908 (a measured GB300 burst) */
  double hbm_gbs;       /* HBM copy bandwidth (GB/s); <= 0: 7000 */
  int32_t sms;          /* streaming multiprocessors; <= 0: 152 */
  double clock_ghz;     /* SM clock (GHz); <= 0: 2.07 */
  double launch_us;     /* fixed cost of one kernel launch on the device (us); < 0: 4 */
} cf_device_model;

typedef struct {
  double flops;            /* algorithmic flops: 2 M N K per GEMM */
  double fused_bytes;      /* compulsory HBM bytes of the fused call */
  double unfused_bytes;    /* HBM bytes of the unfused path (the intermediate written and read back) */
  double mainloop_us;      /* fused: predicted main-loop time of one tile */
  double epilogue_us;      /* fused: predicted epilogue (+ statistics exchange) time of one tile */
  double fused_us;         /* predicted time of the fused call */
  double unfused_us;       /* predicted time of the unfused path */
  int32_t fused_preferred; /* 1 when fused_us <= unfused_us */
  int32_t epilogue_hidden; /* 1 when a tile's epilogue fits inside a tile's main loop */
} cf_cost;

/* Same validation as cf_gemm_epilogue / cf_b2bgemm (pointers are not
 * dereferenced; NULL data pointers are allowed here).  `dev` may be NULL
 * (GB300 defaults).  Returns CF_ERR_UNSUPPORTED_SHAPE where the fused call
 * would. */
CF_API cf_status cf_cost_gemm_epilogue(const cf_matrix* A, const cf_matrix* B, const cf_epi_desc* epi,
                                       const cf_device_model* dev, cf_cost* out);
CF_API cf_status cf_cost_b2bgemm(const cf_matrix* A, const cf_matrix* W1, const cf_matrix* W2,
                                 const cf_b2b_desc* desc, const cf_device_model* dev, cf_cost* out);

/* Reads and clears the device status word written by bounded waits
 * (synchronises the stream first).  CF_OK or CF_ERR_TIMEOUT. */
CF_API cf_status cf_last_device_status(void* stream);

/* Human-readable name of a status code (static string). */
CF_API const char* cf_status_string(cf_status s);

/* ABI version (CF_ABI_VERSION) of the loaded library. */
CF_API int cf_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CF_GB300_H */
