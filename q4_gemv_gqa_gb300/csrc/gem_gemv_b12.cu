// gem_gemv_b12.cu — Q4_0 GEMV kernels for batch sizes 1 and 2.
#include "gem_gemv_kernels.cuh"

GEM_GEMV_DEFINE_BATCH(1)
GEM_GEMV_DEFINE_BATCH(2)
