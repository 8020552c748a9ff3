// gem_gemv_b56.cu — Q4_0 GEMV kernels for batch sizes 5 and 6.
#include "gem_gemv_kernels.cuh"

GEM_GEMV_DEFINE_BATCH(5)
GEM_GEMV_DEFINE_BATCH(6)
