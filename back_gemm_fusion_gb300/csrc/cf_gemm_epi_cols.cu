// cf_gemm_epi_cols.cu -- the fused GEMM + epilogue kernels for reductions
// down the columns of P (the complementary strip), full tiles.
#include "cf_gemm_epi_kernel.cuh"

namespace cf {

const void* gemm_epi_select_variant2(int rowop, int xmode, bool pair) {
  return select_kernel_t<false, true>(rowop, xmode, pair);
}

}  // namespace cf
