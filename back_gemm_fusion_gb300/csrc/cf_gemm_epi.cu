// cf_gemm_epi.cu -- host side of the fused GEMM + epilogue kernel: kernel
// selection, function attributes, occupancy queries and the launch.  This
// unit instantiates the full-tile row-reduction kernels (variant 0); the
// other variants live in their own units: 1 ragged last tile
// (cf_gemm_epi_ragged.cu), 2 column reductions (cf_gemm_epi_cols.cu), 3 both
// (cf_gemm_epi_cols_ragged.cu).
#include "cf_gemm_epi_kernel.cuh"

namespace cf {

const void* gemm_epi_select_variant1(int rowop, int xmode, bool pair);
const void* gemm_epi_select_variant2(int rowop, int xmode, bool pair);
const void* gemm_epi_select_variant3(int rowop, int xmode, bool pair);

namespace {
const void* select_kernel(int rowop, int xmode, bool pair, int variant) {
  switch (variant) {
    case 0: return select_kernel_t<false, false>(rowop, xmode, pair);
    case 1: return gemm_epi_select_variant1(rowop, xmode, pair);
    case 2: return gemm_epi_select_variant2(rowop, xmode, pair);
    case 3: return gemm_epi_select_variant3(rowop, xmode, pair);
    default: return nullptr;
  }
}
}  // namespace

size_t gemm_epi_smem_bytes() { return (size_t)smem_for(false); }

cudaError_t gemm_epi_prepare(int rowop, int xmode, bool pair, int variant) {
  const void* k = select_kernel(rowop, xmode, pair, variant);
  if (!k) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_for(pair));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

cudaError_t gemm_epi_max_clusters(int rowop, int xmode, bool pair, int variant, int cluster, int* out) {
  const void* k = select_kernel(rowop, xmode, pair, variant);
  if (!k) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(cluster, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_for(pair);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(out, k, &cfg);
}

cudaError_t gemm_epi_max_blocks_per_sm(int rowop, int xmode, int variant, int* out) {
  const void* k = select_kernel(rowop, xmode, false, variant);
  if (!k) return cudaErrorInvalidValue;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, k, kThreads, smem_for(false));
}

cudaError_t gemm_epi_launch(const GemmEpiLaunch& L, cudaStream_t s) {
  const void* k = select_kernel(L.rowop, L.xmode, L.p.pair != 0, L.variant);
  if (!k) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  int na = 0;
  if (L.cluster > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = L.cluster;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  // The workspace exchange needs no co-residency guarantee: tiles of a strip
  // wait for one another, but items are claimed as tickets by running CTAs
  // only (see the kernel), so CTAs that start late find the work taken.
  cfg.gridDim = dim3(L.grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_for(L.p.pair != 0);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = na;
  void* args[] = {const_cast<GemmEpiParams*>(&L.p)};
  return cudaLaunchKernelExC(&cfg, k, args);
}

}  // namespace cf
