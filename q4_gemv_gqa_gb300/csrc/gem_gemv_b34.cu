// gem_gemv_b34.cu — Q4_0 GEMV kernels for batch sizes 3 and 4.
#include "gem_gemv_kernels.cuh"

GEM_GEMV_DEFINE_BATCH(3)
GEM_GEMV_DEFINE_BATCH(4)
