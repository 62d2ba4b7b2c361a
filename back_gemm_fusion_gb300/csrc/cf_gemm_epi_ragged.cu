// cf_gemm_epi_ragged.cu -- the fused GEMM + epilogue kernels for N not a
// multiple of the 256-column tile (the last tile of each row is ragged),
// instantiated apart from the full-tile ones so both compile in parallel.
#include "cf_gemm_epi_kernel.cuh"

namespace cf {

const void* gemm_epi_select_variant1(int rowop, int xmode, bool pair) {
  return select_kernel_t<true, false>(rowop, xmode, pair);
}

}  // namespace cf
