// gem_gemv_kernels.cuh — device code of the Q4_0 GEMV (see gem_gemv.cu for the design).
// Included by the gem_gemv_b*.cu files, each of which instantiates the kernels for two
// batch sizes so the library's translation units compile in parallel.
#pragma once

#include "gem_device.cuh"

namespace gem {
namespace gemv_detail {

constexpr int kGroupBytes = 144;                 // 8 blocks, 256 weights
constexpr int kUnitRows = 16;                    // rows per TMA box
constexpr int kBoxBytes = kGroupBytes * kUnitRows;
constexpr int kMaxThreads = 640;
constexpr int kPartsPerGroup = 4;               // a task covers 2 of a group's 8 blocks
constexpr size_t kSmemBudget = 112 * 1024;       // leaves room for a neighbouring kernel's CTA

struct GemvParams {
    int64_t N;
    int G;            // groups (of 256 weights) per row
    const float* x;
    int64_t ldx;
    float* y;
    int64_t ldy;
    const float* residual;
    int64_t ldr;
    const float* gamma;
    float eps;
    int act;
    int U;            // 16-row units per matrix
    int up;           // units per pass
    int gps;          // groups per stage
    int ns;           // ring stages
    int spp;          // stages per pass
    int tasks;        // nmat * up * 16 * gps * kPartsPerGroup
    uint32_t stage_bytes;
    uint32_t bar_off, raw_off, xs_off, rstd_off, red_off;
    int* status;
};

__device__ __forceinline__ float act_fn(float g, int act) {
    if (act == 0) return g / (1.0f + __expf(-g));
    const float c = 0.7978845608028654f;  // sqrt(2/pi)
    return 0.5f * g * (1.0f + tanhf(c * (g + 0.044715f * g * g * g)));
}

// 32-bit little-endian word of the group at byte offset OFF (OFF even, compile-time).
template <int OFF>
__device__ __forceinline__ uint32_t word_at(const uint32_t (&w)[9]) {
    if constexpr ((OFF & 3) == 0) return w[OFF >> 2];
    else return __funnelshift_r(w[OFF >> 2], w[(OFF >> 2) + 1], 16);
}
// word_at<OFF>() << 3 and >> 1, with any bits that the 0x78 byte mask discards left as
// they fall; only bits 3..6 of each byte are used afterwards.
template <int OFF>
__device__ __forceinline__ uint32_t word_shl3(const uint32_t (&w)[9]) {
    if constexpr ((OFF & 3) == 0) return w[OFF >> 2] << 3;
    else return __funnelshift_r(w[OFF >> 2], w[(OFF >> 2) + 1], 13);
}
template <int OFF>
__device__ __forceinline__ uint32_t word_shr1(const uint32_t (&w)[9]) {
    if constexpr ((OFF & 3) == 0) return w[OFF >> 2] >> 1;
    else return __funnelshift_r(w[OFF >> 2], w[(OFF >> 2) + 1], 17);
}

// float 1 + q/16 from byte m of v, where v's bytes are 0x80 | (q << 3).
template <int M>
__device__ __forceinline__ float nib_float(uint32_t v) {
    return __uint_as_float(__byte_perm(v, 0x3Fu, 0x4055u | (M << 8)));
}

// Accumulate block BLK (0 or 1) of a 36-byte task (two Q4_0 blocks of one row, held in
// w[0..8]) against BATCH activation chunks: xc points at the task's 64 activations, batch b
// at xc + b * xstride.
template <int BATCH, int BLK>
__device__ __forceinline__ void dot_block(const uint32_t (&w)[9], const float* __restrict__ xc,
                                          int xstride, float (&acc)[BATCH]) {
    constexpr int O = 18 * BLK;
    const uint32_t dbits = (O & 2) ? (w[O >> 2] >> 16) : (w[O >> 2] & 0xffffu);
    const float d = half_bits_to_float(dbits);
    float f[32];
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
        uint32_t lo, hi;
        if (wi == 0) { lo = word_shl3<O + 2>(w); hi = word_shr1<O + 2>(w); }
        if (wi == 1) { lo = word_shl3<O + 6>(w); hi = word_shr1<O + 6>(w); }
        if (wi == 2) { lo = word_shl3<O + 10>(w); hi = word_shr1<O + 10>(w); }
        if (wi == 3) { lo = word_shl3<O + 14>(w); hi = word_shr1<O + 14>(w); }
        lo = (lo & 0x78787878u) | 0x80808080u;
        hi = (hi & 0x78787878u) | 0x80808080u;
        f[4 * wi + 0] = nib_float<0>(lo);
        f[4 * wi + 1] = nib_float<1>(lo);
        f[4 * wi + 2] = nib_float<2>(lo);
        f[4 * wi + 3] = nib_float<3>(lo);
        f[16 + 4 * wi + 0] = nib_float<0>(hi);
        f[16 + 4 * wi + 1] = nib_float<1>(hi);
        f[16 + 4 * wi + 2] = nib_float<2>(hi);
        f[16 + 4 * wi + 3] = nib_float<3>(hi);
    }
    // (1 + q/16) - 1.5 = (q - 8)/16 exactly: every product below is of an exact weight code
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float2 e = fadd2(make_float2(f[2 * i], f[2 * i + 1]), make_float2(-1.5f, -1.5f));
        f[2 * i] = e.x;
        f[2 * i + 1] = e.y;
    }
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
        const float4* xv = reinterpret_cast<const float4*>(xc + b * xstride + 32 * BLK);
        float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
            const float4 xx = xv[q4];
            s0 = ffma2(make_float2(f[4 * q4 + 0], f[4 * q4 + 1]), make_float2(xx.x, xx.y), s0);
            s1 = ffma2(make_float2(f[4 * q4 + 2], f[4 * q4 + 3]), make_float2(xx.z, xx.w), s1);
        }
        acc[b] = fmaf(d, (s0.x + s0.y) + (s1.x + s1.y), acc[b]);
    }
}

template <int BATCH>
__device__ __forceinline__ void dot_task(const uint8_t* __restrict__ src, const float* __restrict__ xc,
                                         int xstride, float (&acc)[BATCH]) {
    uint32_t w[9];
    const uint32_t* s4 = reinterpret_cast<const uint32_t*>(src);
#pragma unroll
    for (int i = 0; i < 9; ++i) w[i] = s4[i];
    dot_block<BATCH, 0>(w, xc, xstride, acc);
    dot_block<BATCH, 1>(w, xc, xstride, acc);
}

__device__ __forceinline__ void cp_async_16(void* dst, const void* src, bool valid) {
    const uint32_t n = valid ? 16u : 0u;  // 0 source bytes: the 16 destination bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(n)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int BATCH, int NMAT>
__global__ void __launch_bounds__(kMaxThreads) q4_0_gemv_tma_kernel(const __grid_constant__ CUtensorMap tm0,
                                                                    const __grid_constant__ CUtensorMap tm1,
                                                                    const GemvParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_off);
    float* raw = reinterpret_cast<float*>(smem + p.raw_off);   // 3 x (BATCH + 1) x chunk
    float* xs = reinterpret_cast<float*>(smem + p.xs_off);     // 2 x BATCH x chunk
    float* rstd = reinterpret_cast<float*>(smem + p.rstd_off);
    float* red = reinterpret_cast<float*>(smem + p.red_off);
    __shared__ int abort_flag;

    const int t = threadIdx.x;
    const int nthr = blockDim.x;
    const int C = gridDim.x;
    const int c = blockIdx.x;
    const int u0 = static_cast<int>((static_cast<int64_t>(c) * p.U) / C);
    const int u1 = static_cast<int>((static_cast<int64_t>(c + 1) * p.U) / C);
    const int npass = (u1 - u0 + p.up - 1) / p.up;
    const int S = npass * p.spp;                       // stages this CTA streams
    const int chunk = p.gps * 256;                     // activation floats per stage and batch
    const int rawsz = (BATCH + 1) * chunk;             // x rows + gamma
    const int rows_in_pass = NMAT * p.up * kUnitRows;  // task slots per group phase

    // task of this thread: group phase phi, part pi (blocks 2pi, 2pi+1), row slot rem
    const int psi = t / rows_in_pass;
    const int phi = psi / kPartsPerGroup, pi = psi % kPartsPerGroup;
    const int rem = t - psi * rows_in_pass;
    const int mat = rem / (p.up * kUnitRows);
    const int uu = (rem >> 4) % p.up;
    const int r = rem & 15;

    uint64_t policy = 0;
    if (t == 0) {
        abort_flag = 0;
        for (int i = 0; i < p.ns; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        prefetch_tensormap(&tm0);
        if (NMAT == 2) prefetch_tensormap(&tm1);
    }
    __syncthreads();

    auto issue = [&](int s) {
        const int pass = s / p.spp, ks = s - pass * p.spp;
        const int ub = u0 + pass * p.up;
        const int nup = min(p.up, u1 - ub);
        const int g0 = ks * p.gps;
        const int ng = min(p.gps, p.G - g0);
        const int slot = s % p.ns;
        uint8_t* dst = smem + static_cast<size_t>(slot) * p.stage_bytes;
        mbar_arrive_expect_tx(&bars[slot], static_cast<uint32_t>(NMAT * nup * ng * kBoxBytes));
        for (int ph = 0; ph < ng; ++ph)
            for (int m = 0; m < NMAT; ++m)
                for (int u = 0; u < nup; ++u)
                    tma_load_2d(dst + ((ph * NMAT + m) * p.up + u) * kBoxBytes, m ? &tm1 : &tm0,
                                (g0 + ph) * kGroupBytes, (ub + u) * kUnitRows, &bars[slot], policy);
    };

    if (t == 0) {
        policy = l2_policy_evict_first();
        const int pre = min(p.ns, S);
        for (int s = 0; s < pre; ++s) issue(s);
    }
    pdl_trigger();
    pdl_wait();  // activations (and residual) come from the previous kernel

    // Activation staging, per stage: cp.async of the raw x chunk (and gamma) into a
    // 3-deep ring.  A chunk is waited for (each thread its own copies) and published by the
    // end-of-iteration barrier one iteration before it is transformed (x * gamma, per-block
    // sums) into the double-buffered operand chunk.
    const int nf4 = (BATCH + (p.gamma ? 1 : 0)) * chunk / 4;
    auto copy_raw = [&](int s) {
        if (s < S) {
            const int ks = s % p.spp;
            const int g0 = ks * p.gps;
            const int lim = min(p.gps, p.G - g0) * 256;
            float* rd = raw + static_cast<size_t>(s % 3) * rawsz;
            for (int f = t; f < nf4; f += nthr) {
                const int b = f / (chunk / 4);
                const int i = (f - b * (chunk / 4)) * 4;
                const bool valid = i < lim;
                const int64_t k = static_cast<int64_t>(g0) * 256 + (valid ? i : 0);
                const float* src = b < BATCH ? p.x + b * p.ldx + k : p.gamma + k;
                cp_async_16(rd + b * chunk + i, src, valid);
            }
        }
        cp_async_commit();
    };
    float ssq[BATCH];
#pragma unroll
    for (int b = 0; b < BATCH; ++b) ssq[b] = 0.f;
    auto transform = [&](int s) {  // raw(s) -> xs[s & 1]
        if (s >= S) return;
        const float* rd = raw + static_cast<size_t>(s % 3) * rawsz;
        float* xd = xs + static_cast<size_t>(s & 1) * BATCH * chunk;
        const bool first_pass = s < p.spp;
        for (int f = t; f < BATCH * chunk / 4; f += nthr) {
            const int b = f / (chunk / 4);
            const int i = (f - b * (chunk / 4)) * 4;
            float4 v = *reinterpret_cast<const float4*>(rd + b * chunk + i);
            if (p.gamma) {
                if (first_pass) {
#pragma unroll
                    for (int bb = 0; bb < BATCH; ++bb)
                        if (bb == b) ssq[bb] += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
                }
                const float4 g = *reinterpret_cast<const float4*>(rd + BATCH * chunk + i);
                v.x *= g.x; v.y *= g.y; v.z *= g.z; v.w *= g.w;
            }
            *reinterpret_cast<float4*>(xd + b * chunk + i) = v;
        }
    };

    float acc[BATCH];
#pragma unroll
    for (int b = 0; b < BATCH; ++b) acc[b] = 0.f;

    copy_raw(0);
    copy_raw(1);
    copy_raw(2);
    cp_async_wait<2>();
    __syncthreads();
    transform(0);
    cp_async_wait<1>();
    __syncthreads();

    for (int s = 0; s < S; ++s) {
        const int pass = s / p.spp, ks = s - pass * p.spp;
        const int ub = u0 + pass * p.up;
        const int nup = min(p.up, u1 - ub);
        const int ng = min(p.gps, p.G - ks * p.gps);
        const int slot = s % p.ns;
        const int buf = s & 1;
        transform(s + 1);

        if (!mbar_wait(&bars[slot], static_cast<uint32_t>((s / p.ns) & 1), p.status)) abort_flag = 1;
        if (t < p.tasks && phi < ng && uu < nup) {
            const uint8_t* src = smem + static_cast<size_t>(slot) * p.stage_bytes +
                                 ((phi * NMAT + mat) * p.up + uu) * kBoxBytes + r * kGroupBytes + pi * 36;
            const float* xc = xs + static_cast<size_t>(buf) * BATCH * chunk + phi * 256 + pi * 64;
            dot_task<BATCH>(src, xc, chunk, acc);
        }

        if (ks == p.spp - 1) {  // end of pass: combine the group phases of every row
            if (pass == 0 && p.gamma) {  // 1 / rms of each activation row, from pass 0's staging
#pragma unroll
                for (int b = 0; b < BATCH; ++b) {
                    const float v = warp_sum(ssq[b]);
                    if ((t & 31) == 0) red[(t >> 5) * BATCH + b] = v;
                }
                __syncthreads();
                if (t < BATCH) {
                    float sum = 0.f;
                    for (int wv = 0; wv < nthr / 32; ++wv) sum += red[wv * BATCH + t];
                    rstd[t] = rsqrtf(sum / static_cast<float>(p.G * 256) + p.eps);
                }
                __syncthreads();
            }
            const int nph = p.gps * kPartsPerGroup;
            if (t < p.tasks) {
#pragma unroll
                for (int b = 0; b < BATCH; ++b) red[(rem * nph + psi) * BATCH + b] = acc[b];
            }
#pragma unroll
            for (int b = 0; b < BATCH; ++b) acc[b] = 0.f;
            __syncthreads();
            if (t < rows_in_pass && (NMAT == 1 || mat == 0)) {
                const int64_t n = static_cast<int64_t>(ub + uu) * kUnitRows + r;
                if (uu < nup && n < p.N) {
#pragma unroll
                    for (int b = 0; b < BATCH; ++b) {
                        const float scale = 16.f * (p.gamma ? rstd[b] : 1.f);
                        float v = 0.f;
                        for (int ph = 0; ph < nph; ++ph) v += red[(t * nph + ph) * BATCH + b];
                        v *= scale;
                        if (NMAT == 1) {
                            if (p.residual) v += p.residual[b * p.ldr + n];
                        } else {
                            float uv = 0.f;
                            const int srow = p.up * kUnitRows + t;
                            for (int ph = 0; ph < nph; ++ph) uv += red[(srow * nph + ph) * BATCH + b];
                            v = act_fn(v, p.act) * (uv * scale);
                        }
                        p.y[b * p.ldy + n] = v;
                    }
                }
            }
        }
        copy_raw(s + 3);
        cp_async_wait<1>();
        __syncthreads();
        if (abort_flag) {  // stages s .. s + ns - 1 may still be in flight
            if (t == 0) drain_stages(bars, p.ns, s, min(s + p.ns - 1, S - 1));
            break;
        }
        if (t == 0 && s + p.ns < S) issue(s + p.ns);
    }
    cp_async_wait<0>();
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
    pdl_trigger();
    pdl_wait();
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
    const void* gemv_tma_kernel_b##B(int nmat);                            \
    const void* gemv_generic_kernel_b##B(int nmat);                        \
    }
#define GEM_GEMV_DEFINE_BATCH(B)                                                                       \
    namespace gem {                                                                                    \
    const void* gemv_tma_kernel_b##B(int nmat) {                                                       \
        return nmat == 2 ? reinterpret_cast<const void*>(gemv_detail::q4_0_gemv_tma_kernel<B, 2>)      \
                         : reinterpret_cast<const void*>(gemv_detail::q4_0_gemv_tma_kernel<B, 1>);     \
    }                                                                                                  \
    const void* gemv_generic_kernel_b##B(int nmat) {                                                   \
        return nmat == 2 ? reinterpret_cast<const void*>(gemv_detail::q4_0_gemv_generic_kernel<B, 2>)  \
                         : reinterpret_cast<const void*>(gemv_detail::q4_0_gemv_generic_kernel<B, 1>); \
    }                                                                                                  \
    }
