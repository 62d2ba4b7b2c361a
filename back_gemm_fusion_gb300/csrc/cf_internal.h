// cf_internal.h -- host-side structures shared by the C-ABI layer and the
// kernel translation units (not part of the public ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/cf.h"

namespace cf {

// Row reduction that ends the epilogue program.
enum RowOp : int { ROW_NONE = 0, ROW_LAYERNORM = 1, ROW_RMSNORM = 2, ROW_SOFTMAX = 3 };
// How row statistics cross CTAs.
enum XMode : int { X_NONE = 0, X_CLUSTER = 1, X_GLOBAL = 2 };

// Tile shape of the fused GEMM-epilogue kernel.
constexpr int kBM = 128;     // rows per tile = TMEM lanes
constexpr int kBN = 256;     // columns per tile = one TMEM accumulator
constexpr int kBK = 64;      // K per pipeline stage (one 128-byte swizzle row of bf16)
constexpr int kMaxClusterCtas = 16;
// Kernel variant of a program: the last row op plus 4 x the first of two
// chained row ops (ROW_NONE, ROW_LAYERNORM or ROW_RMSNORM).
constexpr int kRowCodes = 12;
constexpr int row_code(int rowop0, int rowop) { return rowop + 4 * rowop0; }

// Kernel parameters (passed by value as a __grid_constant__).
struct GemmEpiParams {
  CUtensorMap tmA;    // A: bf16 [M][K], box {64, 128}, 128B swizzle
  CUtensorMap tmB;    // B: K-major [N][K] box {64, 256} or MN-major [K][N] box {64, 64}
  CUtensorMap tmOut;  // out: fp32 [M][N], box {32, 32}, 128B swizzle; or bf16, box {32, 32}, no swizzle
  int M, N, K;
  int tiles_n;        // ceil(N / kBN); the last tile may be ragged
  int strips;         // M / kBM
  int num_items;      // strips * tiles_n
  int b_mn_major;     // 1: B stored K x N (N contiguous)
  int pair;           // 1: CTA pairs run 256 x 256 tiles with cta_group::2 MMAs
  int pair_items;     // (strips / 2) * tiles_n when pair == 1
  int n_ops;          // elementwise ops (row op excluded)
  int op_kind[CF_EPI_MAX_OPS];
  float op_scalar[CF_EPI_MAX_OPS];
  float eps;
  const float* bias;
  const float* gamma;
  const float* beta;
  // First of two chained row reductions (row op code / 4; see row_code):
  // elementwise ops [0, n_ops0) precede it, ops [n_ops0, n_ops) follow it.
  int n_ops0;
  float eps0;
  const float* gamma0;    // may be null: no affine transform
  const float* beta0;
  float2* ws_stats0;      // its partial statistics and arrival counters (workspace exchange)
  unsigned* ws_count0;
  const void* res;        // residual matrix (CF_OP_ADD_RESIDUAL), M x N, leading dim res_ld
  long long res_ld;
  int res_bf16;           // 1: bf16 residual, 0: fp32
  int out_bf16;           // 1: bf16 output (rounded to nearest even), 0: fp32
  float2* ws_stats;       // [strips][tiles_n][kBM] partial row statistics
  unsigned* ws_count;     // [strips][4] arrival counters (cleared by the host)
  unsigned* ws_ticket;    // workspace exchange: the next work item to claim (cleared by the host)
  int tickets;            // 1: work items from ws_ticket (single-stage programs), 0: static assignment
  unsigned* status;       // device status word
  long long timeout_cycles;
};

struct GemmEpiLaunch {
  GemmEpiParams p;
  int rowop;
  int xmode;
  int grid;          // CTAs
  int cluster;       // CTAs per cluster (X_CLUSTER: tiles_n; pair mode: 2), else 1
  int variant;       // kernel variant: ragged last tile (+1), column reductions (+2)
};

// Host helpers implemented in cf_api.cu and shared by the kernel launchers.
// Current device's SM count and status-word address; fails unless sm_103.
cf_status device_query(int* sms, unsigned** status);
// Tiled tensor map with 128-byte swizzle: `rank` dims (innermost first),
// rank-1 byte strides, box sizes.
cf_status encode_tmap(CUtensorMap* map, CUtensorMapDataType dt, int rank, void* ptr, const uint64_t* dims,
                      const uint64_t* strides_bytes, const uint32_t* box);
long long wait_timeout_cycles();

size_t gemm_epi_smem_bytes();
// variant: 1 if the kernel's N % kBN != 0 (its last tile per row is ragged),
// + 2 for column reductions (the kernel runs on P^T).
constexpr int kNumVariants = 4;
cudaError_t gemm_epi_prepare(int rowop, int xmode, bool pair, int variant);  // set function attributes
cudaError_t gemm_epi_launch(const GemmEpiLaunch& L, cudaStream_t s);
cudaError_t gemm_epi_max_clusters(int rowop, int xmode, bool pair, int variant, int cluster, int* out);
cudaError_t gemm_epi_max_blocks_per_sm(int rowop, int xmode, int variant, int* out);

}  // namespace cf
