// cf_gemm_epi_cols_ragged.cu -- column-reduction kernels whose reduced
// dimension (M of P) is not a multiple of the 256-wide tile.
#include "cf_gemm_epi_kernel.cuh"

namespace cf {

const void* gemm_epi_select_variant3(int rowop, int xmode, bool pair) {
  return select_kernel_t<true, true>(rowop, xmode, pair);
}

}  // namespace cf
