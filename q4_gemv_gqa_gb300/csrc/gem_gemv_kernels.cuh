// gem_gemv_kernels.cuh — the general-path Q4_0 GEMV (any K % 32 == 0, any alignment), used
// where the tensor-core kernel (gem_gemv_mma.cuh) cannot stream the matrix with TMA.
// Included by the gem_gemv_b*.cu files, each of which instantiates it for two batch sizes
// so the library's translation units compile in parallel.
#pragma once

#include "gem_device.cuh"

namespace gem {
namespace gemv_detail {

struct GemvParams {
    const float* x;
    int64_t ldx;
    float* y;
    int64_t ldy;
    const float* residual;
    int64_t ldr;
    const float* gamma;
    float eps;
    int act;
    unsigned* clear;     // words zeroed after the wait (see GemvOp)
    int nclear;
};

__device__ __forceinline__ float act_fn(float g, int act) {
    if (act == 0) return g / (1.0f + __expf(-g));
    const float c = 0.7978845608028654f;  // sqrt(2/pi)
    return 0.5f * g * (1.0f + tanhf(c * (g + 0.044715f * g * g * g)));
}

// General path: any K % 32 == 0 and any alignment.  One warp per output row; plain
// byte loads.  Same arithmetic definition, simpler schedule.
template <int BATCH, int NMAT>
__global__ void __launch_bounds__(256) q4_0_gemv_generic_kernel(const uint8_t* __restrict__ W0,
                                                                const uint8_t* __restrict__ W1,
                                                                int64_t N, int64_t K, GemvParams p) {
    __shared__ float rstd[8];
    __shared__ float red[8][8];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    pdl_wait_trigger();
    clear_words(p.clear, p.nclear, static_cast<int>(threadIdx.x), static_cast<int>(blockDim.x));
    if (p.gamma) {
        for (int b = 0; b < BATCH; ++b) {
            float part = 0.f;
            for (int64_t k = threadIdx.x; k < K; k += blockDim.x) {
                const float v = p.x[b * p.ldx + k];
                part = fmaf(v, v, part);
            }
            part = warp_sum(part);
            if (lane == 0) red[wid][b] = part;
        }
        __syncthreads();
        if (threadIdx.x < BATCH) {
            float s = 0.f;
            for (int i = 0; i < (int)(blockDim.x / 32); ++i) s += red[i][threadIdx.x];
            rstd[threadIdx.x] = rsqrtf(s / static_cast<float>(K) + p.eps);
        }
        __syncthreads();
    }
    const int64_t n = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + wid;
    if (n >= N) return;
    const int64_t nb = K / 32;
    float acc[NMAT][BATCH];
    for (int m = 0; m < NMAT; ++m)
        for (int b = 0; b < BATCH; ++b) acc[m][b] = 0.f;
    for (int m = 0; m < NMAT; ++m) {
        const uint8_t* row = (m ? W1 : W0) + n * nb * 18;
        for (int64_t blk = lane; blk < nb; blk += 32) {
            const uint8_t* q = row + blk * 18;
            const float d = half_bits_to_float(static_cast<uint32_t>(q[0]) | (static_cast<uint32_t>(q[1]) << 8));
            for (int b = 0; b < BATCH; ++b) {
                float s = 0.f;
                for (int j = 0; j < 16; ++j) {
                    const int64_t k0 = blk * 32 + j;
                    float x0 = p.x[b * p.ldx + k0], x1 = p.x[b * p.ldx + k0 + 16];
                    if (p.gamma) {
                        x0 = x0 * rstd[b] * p.gamma[k0];
                        x1 = x1 * rstd[b] * p.gamma[k0 + 16];
                    }
                    s = fmaf(static_cast<float>((q[2 + j] & 15) - 8), x0, s);
                    s = fmaf(static_cast<float>((q[2 + j] >> 4) - 8), x1, s);
                }
                acc[m][b] = fmaf(d, s, acc[m][b]);
            }
        }
    }
    for (int b = 0; b < BATCH; ++b) {
        float v = warp_sum(acc[0][b]);
        float u = NMAT == 2 ? warp_sum(acc[NMAT - 1][b]) : 0.f;
        if (lane == 0) {
            if (NMAT == 1) {
                if (p.residual) v += p.residual[b * p.ldr + n];
            } else {
                v = act_fn(v, p.act) * u;
            }
            p.y[b * p.ldy + n] = v;
        }
    }
}

}  // namespace gemv_detail
}  // namespace gem

// Kernel entry points of batch size B for NMAT = 1 and 2, defined in gem_gemv_b*.cu.
#define GEM_GEMV_DECLARE_BATCH(B)                                          \
    namespace gem {                                                        \
    const void* gemv_generic_kernel_b##B(int nmat);                        \
    }
#define GEM_GEMV_DEFINE_BATCH(B)                                                                       \
    namespace gem {                                                                                    \
    const void* gemv_generic_kernel_b##B(int nmat) {                                                   \
        return nmat == 2 ? reinterpret_cast<const void*>(gemv_detail::q4_0_gemv_generic_kernel<B, 2>)  \
                         : reinterpret_cast<const void*>(gemv_detail::q4_0_gemv_generic_kernel<B, 1>); \
    }                                                                                                  \
    }
