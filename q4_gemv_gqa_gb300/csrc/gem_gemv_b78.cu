// gem_gemv_b78.cu — Q4_0 GEMV kernels for batch sizes 7 and 8.
#include "gem_gemv_kernels.cuh"

GEM_GEMV_DEFINE_BATCH(7)
GEM_GEMV_DEFINE_BATCH(8)
