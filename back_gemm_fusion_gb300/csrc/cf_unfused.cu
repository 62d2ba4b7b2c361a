// cf_unfused.cu -- unfused comparison path (placeholder).
#include "cf_internal.h"

extern "C" cf_status cf_unfused_gemm_epilogue(const cf_matrix*, const cf_matrix*, const float*, const float*,
                                              const float*, const cf_epi_desc*, cf_matrix*, float*, void*) {
  return CF_ERR_UNSUPPORTED_SHAPE;
}
extern "C" cf_status cf_unfused_b2bgemm(const cf_matrix*, const cf_matrix*, const cf_matrix*, const cf_b2b_desc*,
                                        cf_matrix*, float*, void*, void*) {
  return CF_ERR_UNSUPPORTED_SHAPE;
}
