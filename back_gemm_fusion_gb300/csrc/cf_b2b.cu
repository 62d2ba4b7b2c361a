// cf_b2b.cu -- fused back-to-back GEMM (placeholder until the kernel lands).
#include "cf_internal.h"

extern "C" cf_status cf_b2bgemm(const cf_matrix*, const cf_matrix*, const cf_matrix*, const cf_b2b_desc*,
                                cf_matrix*, void*) {
  return CF_ERR_UNSUPPORTED_SHAPE;
}
