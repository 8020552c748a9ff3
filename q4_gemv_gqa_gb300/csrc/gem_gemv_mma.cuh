// gem_gemv_mma.cuh — Q4_0 GEMV on mma.sync tensor-core instructions (see gem_gemv.cu).
//
// Why tensor cores for a matvec: at ~7 TB/s a GB300 must consume ~12e12 Q4_0 weights per
// second, and the SM issue rate leaves ~2.7 thread-instructions per weight.  A CUDA-core
// unpack-and-FMA inner loop needs >= 3 (measured), so it cannot reach the HBM roof.  With
// m16n8k16 (binary16 operands, fp32 accumulate) one lop3 turns two 4-bit codes into a
// binary16 pair (exponent-magic 0x6400) and one hsub2/hfma2 makes them the exact codes
// q - 8; the tensor op does the 16 x 8 x 16 multiply-adds.  Activations enter as hi + lo
// binary16 pairs (two columns of B, or two mma per k-step for B > 4), scaled per 128
// elements by a power of two so any fp32 range is safe, so products keep ~22 bits.
//
// Work split.  A CTA owns 16-row units; a consumer warp owns one (group phase, matrix,
// unit, half group) task: 16 rows x 4 blocks (128 weights) of every stage.  A producer warp
// streams 16-row x 144-byte TMA boxes into a ring guarded by full / empty mbarriers, so
// consumer warps never wait on each other except at the (few) activation-phase switches.
// Activations for a K-phase are converted once per CTA into mma B fragments in shared
// memory; the next phase's raw activations are prefetched into registers meanwhile.
#pragma once

#include "gem_device.cuh"

namespace gem {
namespace gemv_mma {

constexpr int kGroupBytes = 144;
constexpr int kUnitRows = 16;
constexpr int kBoxBytes = kGroupBytes * kUnitRows;
constexpr int kMaxConsumerWarps = 20;
constexpr int kMaxThreads = (kMaxConsumerWarps + 1) * 32;
constexpr int kPrefetchF4 = 2;                    // raw activation float4s per thread per phase
constexpr size_t kSmemBudget = 112 * 1024;

struct Params {
    int64_t N;
    int G;               // 256-weight groups per row
    int B;
    const float* x;
    int64_t ldx;
    float* y;
    int64_t ldy;
    const float* residual;
    int64_t ldr;
    const float* gamma;
    float eps;
    int act;
    int U, up, gps, ns, spp;
    int nphase;          // K-phases per pass
    int kp;              // activations per phase (multiple of 256 * gps)
    int ncw;             // consumer warps = gps * NMAT * up * 2
    uint32_t stage_bytes;
    uint32_t full_off, empty_off, xf_off, xsc_off, rstd_off, red_off, ssq_off;
    int* status;
};

__device__ __forceinline__ float act_fn(float g, int act) {
    if (act == 0) return g / (1.0f + __expf(-g));
    const float c = 0.7978845608028654f;  // sqrt(2/pi)
    return 0.5f * g * (1.0f + tanhf(c * (g + 0.044715f * g * g * g)));
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void consumer_sync(int nthreads) {
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
    uint16_t v;
    asm volatile("ld.shared.b16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lop3_mask_or(uint32_t a, uint32_t mask, uint32_t orv) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(orv));  // (a & mask) | orv
    return d;
}

__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t hfma2_bits(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// The 4-byte code word t (qs bytes 4t .. 4t+3) of block jj of a row starting at `row`
// (shared address).  Block jj starts at byte 18 * jj; its codes at 18 * jj + 2.
template <int JPAR>
__device__ __forceinline__ uint32_t code_word(uint32_t row, int jj, int t) {
    const uint32_t off = 18u * jj + 2u + 4u * t;
    if constexpr (JPAR == 1) return lds32(row + off);        // odd block: 4-byte aligned
    else return __funnelshift_r(lds32(row + off - 2), lds32(row + off + 2), 16);
}

// A fragments (tile 0: low nibbles = elements 0..15, tile 1: high nibbles = 16..31) of one
// row's code word.  Pair order inside a fragment register: elements (4t, 4t+2) and
// (4t+1, 4t+3); the activation fragments use the same order.
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t& t0a, uint32_t& t0b, uint32_t& t1a,
                                             uint32_t& t1b) {
    const uint32_t w8 = w >> 8;
    const uint32_t lo_off = 0x64086408u;   // binary16 1032.0 twice: (1024 + q) - 1032 = q - 8
    const uint32_t sixteenth = 0x2C002C00u; // binary16 1/16 twice
    const uint32_t m72 = 0xD480D480u;      // binary16 -72 twice: (1024 + 16q)/16 - 72 = q - 8
    t0a = hsub2_bits(lop3_mask_or(w, 0x000F000Fu, 0x64006400u), lo_off);
    t0b = hsub2_bits(lop3_mask_or(w8, 0x000F000Fu, 0x64006400u), lo_off);
    t1a = hfma2_bits(lop3_mask_or(w, 0x00F000F0u, 0x64006400u), sixteenth, m72);
    t1b = hfma2_bits(lop3_mask_or(w8, 0x00F000F0u, 0x64006400u), sixteenth, m72);
}

// Activation fragment layout (one K-phase, per 128-element half group hg, block j 0..3,
// lane quad t 0..3, column n): 16 bytes = {tile0 b0, tile0 b1, tile1 b0, tile1 b1}, each
// a binary16 pair.  PACKED (B <= 4): columns n = 2b (hi), 2b + 1 (lo), NCOL = 2B.
// Otherwise columns n = b with hi and lo entries adjacent (32 bytes), NCOL = B.
template <bool PACKED>
__device__ __forceinline__ uint32_t xf_entry(int hg, int j, int t, int n, int B) {
    if constexpr (PACKED) return static_cast<uint32_t>((((hg * 4 + j) * 4 + t) * (2 * B) + n) * 16);
    else return static_cast<uint32_t>((((hg * 4 + j) * 4 + t) * B + n) * 32);
}

template <bool PACKED, int NMAT>
__global__ void __launch_bounds__(kMaxThreads, 1) q4_0_gemv_mma_kernel(const __grid_constant__ CUtensorMap tm0,
                                                                       const __grid_constant__ CUtensorMap tm1,
                                                                       const Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.full_off);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + p.empty_off);
    float* xsc = reinterpret_cast<float*>(smem + p.xsc_off);   // [hg][B] scale back (2^e)
    float* rstd = reinterpret_cast<float*>(smem + p.rstd_off);
    float* red = reinterpret_cast<float*>(smem + p.red_off);
    float* ssqb = reinterpret_cast<float*>(smem + p.ssq_off);  // [B][K/128] sums of x^2
    const uint32_t xf = smem_u32(smem + p.xf_off);
    const uint32_t ring = smem_u32(smem);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ncw = p.ncw, nct = ncw * 32;
    const int C = gridDim.x, c = blockIdx.x;
    const int u0 = static_cast<int>((static_cast<int64_t>(c) * p.U) / C);
    const int u1 = static_cast<int>((static_cast<int64_t>(c + 1) * p.U) / C);
    const int npass = (u1 - u0 + p.up - 1) / p.up;
    const int S = npass * p.spp;
    const int B = p.B;

    if (tid == 0) {
        for (int i = 0; i < p.ns; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], ncw);
        }
        fence_mbar_init();
        prefetch_tensormap(&tm0);
        if (NMAT == 2) prefetch_tensormap(&tm1);
    }
    __syncthreads();

    // ---------------- producer warp ----------------
    if (warp == ncw) {
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_first();
            auto issue = [&](int s) {
                const int pass = s / p.spp, ks = s - pass * p.spp;
                const int ub = u0 + pass * p.up;
                const int nup = min(p.up, u1 - ub);
                const int g0 = ks * p.gps;
                const int ng = min(p.gps, p.G - g0);
                const int slot = s % p.ns;
                uint8_t* dst = smem + static_cast<size_t>(slot) * p.stage_bytes;
                mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(NMAT * nup * ng * kBoxBytes));
                for (int ph = 0; ph < ng; ++ph)
                    for (int m = 0; m < NMAT; ++m)
                        for (int u = 0; u < nup; ++u)
                            tma_load_2d(dst + ((ph * NMAT + m) * p.up + u) * kBoxBytes, m ? &tm1 : &tm0,
                                        (g0 + ph) * kGroupBytes, (ub + u) * kUnitRows, &full[slot], policy);
            };
            const int pre = min(p.ns, S);
            for (int s = 0; s < pre; ++s) issue(s);  // weights only: before the dependency wait
            pdl_trigger();
            bool ok = true;
            for (int s = pre; s < S && ok; ++s) {
                const int slot = s % p.ns;
                ok = mbar_wait(&empty[slot], static_cast<uint32_t>(((s / p.ns) + 1) & 1), p.status);
                if (ok) issue(s);
            }
        } else {
            pdl_trigger();
        }
        return;
    }

    // ---------------- consumer warps ----------------
    pdl_trigger();
    pdl_wait();  // activations and residual come from the previous kernel

    const int g = lane >> 2, t = lane & 3;
    const int rows_in_pass = NMAT * p.up * kUnitRows;
    // task: (phase phi, matrix, unit uu, half group eta)
    const int eta = warp & 1;
    const int tw = warp >> 1;
    const int uu = tw % p.up;
    const int mat = (tw / p.up) % NMAT;
    const int phi = tw / (p.up * NMAT);
    const int nph = 2 * p.gps;  // partial sums per row
    const int psi = phi * 2 + eta;
    const bool col_ok = PACKED ? (g < 2 * B) : (g < B);

    // Raw activations of a K-phase: slot f covers float4 e4 of batch row b (f = b * kp4 + e4).
    // Thread tid owns slots tid + i * nct; the first kPrefetchF4 are prefetched into
    // registers (with the matching norm weights) during the previous phase's compute.
    const int kp4 = p.kp / 4;
    const int nslots = B * kp4;
    float4 pf[kPrefetchF4], pg[kPrefetchF4];
    auto load_slot = [&](int phase, int f, float4& xv, float4& gv) {
        const int k0 = phase * p.kp;
        const int lim = min(p.kp, p.G * 256 - k0);
        const int b = f / kp4, e = (f - b * kp4) * 4;
        xv = make_float4(0.f, 0.f, 0.f, 0.f);
        gv = make_float4(1.f, 1.f, 1.f, 1.f);
        if (e < lim) {
            xv = *reinterpret_cast<const float4*>(p.x + b * p.ldx + k0 + e);
            if (p.gamma) gv = *reinterpret_cast<const float4*>(p.gamma + k0 + e);
        }
    };
    auto prefetch = [&](int phase) {
#pragma unroll
        for (int i = 0; i < kPrefetchF4; ++i) {
            const int f = tid + i * nct;
            if (f < nslots) load_slot(phase, f, pf[i], pg[i]);
        }
    };
    // One slot -> binary16 hi/lo B fragments.  The 32 lanes of a warp hold one 128-element
    // half group of one row (nslots, kp4 and nct are multiples of 32), so the power-of-two
    // scale and the sum of squares are warp reductions.
    auto convert_slot = [&](int phase, int f, float4 v, float4 gm, bool first_pass) {
        const int b = f / kp4, e4 = f - b * kp4;
        if (p.gamma) {
            const int hgk = (phase * p.kp) / 128 + (e4 >> 5);   // half group inside the row
            if (first_pass && hgk < 2 * p.G) {  // one fixed slot per (row, half group)
                const float ps = warp_sum(v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w);
                if (lane == 0) ssqb[b * (2 * p.G) + hgk] = ps;
            }
            v.x *= gm.x; v.y *= gm.y; v.z *= gm.z; v.w *= gm.w;
        }
        float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
        m = warp_max(m);
        int ex = 0;
        if (m > 0.f) ex = ((__float_as_int(m) >> 23) & 0xff) - 127 - 13;  // m * 2^-ex in [2^13, 2^14)
        ex = max(-100, min(100, ex));
        const float sc = __int_as_float((127 - ex) << 23);
        const int hg = e4 >> 5, ln = e4 & 31;
        const int j = ln >> 3, tile = (ln >> 2) & 1, tt = ln & 3;
        __half h0, l0, h1, l1, h2, l2, h3, l3;
        split_hi_lo(v.x * sc, h0, l0);
        split_hi_lo(v.y * sc, h1, l1);
        split_hi_lo(v.z * sc, h2, l2);
        split_hi_lo(v.w * sc, h3, l3);
        const __half2 hb0 = __halves2half2(h0, h2), hb1 = __halves2half2(h1, h3);  // b0 = {x0, x2}
        const __half2 lb0 = __halves2half2(l0, l2), lb1 = __halves2half2(l1, l3);  // b1 = {x1, x3}
        const uint2 hv = make_uint2(*reinterpret_cast<const uint32_t*>(&hb0), *reinterpret_cast<const uint32_t*>(&hb1));
        const uint2 lv = make_uint2(*reinterpret_cast<const uint32_t*>(&lb0), *reinterpret_cast<const uint32_t*>(&lb1));
        uint8_t* xfp = smem + p.xf_off;
        if constexpr (PACKED) {
            *reinterpret_cast<uint2*>(xfp + xf_entry<true>(hg, j, tt, 2 * b, B) + tile * 8) = hv;
            *reinterpret_cast<uint2*>(xfp + xf_entry<true>(hg, j, tt, 2 * b + 1, B) + tile * 8) = lv;
        } else {
            uint8_t* base = xfp + xf_entry<false>(hg, j, tt, b, B);
            *reinterpret_cast<uint2*>(base + tile * 8) = hv;
            *reinterpret_cast<uint2*>(base + 16 + tile * 8) = lv;
        }
        if (lane == 0) xsc[hg * B + b] = __int_as_float((127 + ex) << 23);
    };
    auto convert = [&](int phase, bool first_pass) {
#pragma unroll
        for (int i = 0; i < kPrefetchF4; ++i) {
            const int f = tid + i * nct;
            if (f < nslots) convert_slot(phase, f, pf[i], pg[i], first_pass);
        }
        for (int f = tid + kPrefetchF4 * nct; f < nslots; f += nct) {  // beyond the prefetch
            float4 xv, gv;
            load_slot(phase, f, xv, gv);
            convert_slot(phase, f, xv, gv, first_pass);
        }
    };

    float acc[4] = {0.f, 0.f, 0.f, 0.f};   // PACKED: [row g, row g+8] of batch t; else [g: 2t, 2t+1; g+8: 2t, 2t+1]
    int s = 0;
    bool ok = true;
    prefetch(0);
    // Every consumer warp runs the same sequence of named barriers whatever happens: after a
    // timed-out wait (ok == false) the remaining waits are skipped, never the barriers.
    for (int pass = 0; pass < npass; ++pass) {
        const int ub = u0 + pass * p.up;
        const int nup = min(p.up, u1 - ub);
        for (int ph = 0; ph < p.nphase; ++ph) {
            consumer_sync(nct);                 // previous phase's fragments are no longer read
            convert(ph, pass == 0);
            const int nxt = ph + 1 < p.nphase ? ph + 1 : (pass + 1 < npass ? 0 : -1);
            consumer_sync(nct);                 // fragments (and scales) published
            if (nxt >= 0) prefetch(nxt);
            const int st_lo = ph * (p.kp / (256 * p.gps));
            const int st_hi = min(p.spp, st_lo + p.kp / (256 * p.gps));
            for (int ks = st_lo; ks < st_hi; ++ks, ++s) {
                const int slot = s % p.ns;
                if (ok) ok = mbar_wait(&full[slot], static_cast<uint32_t>((s / p.ns) & 1), p.status);
                const int gidx = ks * p.gps + phi;          // group index of this task
                if (gidx < p.G && uu < nup) {
                    const uint32_t box = ring + slot * p.stage_bytes + ((phi * NMAT + mat) * p.up + uu) * kBoxBytes;
                    const uint32_t rg = box + g * kGroupBytes, rg8 = box + (g + 8) * kGroupBytes;
                    const int hg = (gidx * 256 - ph * p.kp) / 128 + eta;   // half group inside the phase
                    float blk[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int jj = eta * 4 + j;
                        uint32_t wg, wg8;
                        if (j & 1) {
                            wg = code_word<1>(rg, jj, t);
                            wg8 = code_word<1>(rg8, jj, t);
                        } else {
                            wg = code_word<0>(rg, jj, t);
                            wg8 = code_word<0>(rg8, jj, t);
                        }
                        const float dg = half_bits_to_float(lds16(rg + 18u * jj));
                        const float dg8 = half_bits_to_float(lds16(rg8 + 18u * jj));
                        uint32_t a0, a2, a4, a6, a1, a3, a5, a7;
                        dequant_word(wg, a0, a2, a4, a6);
                        dequant_word(wg8, a1, a3, a5, a7);
                        float cf[4] = {0.f, 0.f, 0.f, 0.f};
                        if constexpr (PACKED) {
                            uint4 bx = make_uint4(0, 0, 0, 0);
                            if (col_ok) bx = lds128(xf + xf_entry<true>(hg, j, t, g, B));
                            mma_16816(cf, a0, a1, a2, a3, bx.x, bx.y);
                            mma_16816(cf, a4, a5, a6, a7, bx.z, bx.w);
                            blk[0] = fmaf(dg, cf[0] + cf[1], blk[0]);
                            blk[1] = fmaf(dg8, cf[2] + cf[3], blk[1]);
                        } else {
                            uint4 bh = make_uint4(0, 0, 0, 0), bl = make_uint4(0, 0, 0, 0);
                            if (col_ok) {
                                bh = lds128(xf + xf_entry<false>(hg, j, t, g, B));
                                bl = lds128(xf + xf_entry<false>(hg, j, t, g, B) + 16);
                            }
                            mma_16816(cf, a0, a1, a2, a3, bh.x, bh.y);
                            mma_16816(cf, a4, a5, a6, a7, bh.z, bh.w);
                            mma_16816(cf, a0, a1, a2, a3, bl.x, bl.y);
                            mma_16816(cf, a4, a5, a6, a7, bl.z, bl.w);
                            blk[0] = fmaf(dg, cf[0], blk[0]);
                            blk[1] = fmaf(dg, cf[1], blk[1]);
                            blk[2] = fmaf(dg8, cf[2], blk[2]);
                            blk[3] = fmaf(dg8, cf[3], blk[3]);
                        }
                    }
                    if constexpr (PACKED) {
                        const float sc = t < B ? xsc[hg * B + t] : 0.f;
                        acc[0] = fmaf(sc, blk[0], acc[0]);
                        acc[1] = fmaf(sc, blk[1], acc[1]);
                    } else {
                        const float sc0 = 2 * t < B ? xsc[hg * B + 2 * t] : 0.f;
                        const float sc1 = 2 * t + 1 < B ? xsc[hg * B + 2 * t + 1] : 0.f;
                        acc[0] = fmaf(sc0, blk[0], acc[0]);
                        acc[1] = fmaf(sc1, blk[1], acc[1]);
                        acc[2] = fmaf(sc0, blk[2], acc[2]);
                        acc[3] = fmaf(sc1, blk[3], acc[3]);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[slot]);
            }
        }
        // ---- end of pass: combine the 2 * gps partial sums of every row, write outputs ----
        consumer_sync(nct);
        if (pass == 0 && p.gamma) {   // 1 / rms of every activation row (pass 0 saw all of K)
            if (tid < B) {
                float sum = 0.f;
                for (int i = 0; i < 2 * p.G; ++i) sum += ssqb[tid * (2 * p.G) + i];
                rstd[tid] = rsqrtf(sum / static_cast<float>(p.G * 256) + p.eps);
            }
            consumer_sync(nct);
        }
        {
            // partial sums: red[(slotrow * nph + psi) * B + b]
            const int slotrow = (mat * p.up + uu) * kUnitRows;
            if (uu < nup) {
                if constexpr (PACKED) {
                    if (t < B) {
                        red[((slotrow + g) * nph + psi) * B + t] = acc[0];
                        red[((slotrow + g + 8) * nph + psi) * B + t] = acc[1];
                    }
                } else {
                    if (2 * t < B) {
                        red[((slotrow + g) * nph + psi) * B + 2 * t] = acc[0];
                        red[((slotrow + g + 8) * nph + psi) * B + 2 * t] = acc[2];
                    }
                    if (2 * t + 1 < B) {
                        red[((slotrow + g) * nph + psi) * B + 2 * t + 1] = acc[1];
                        red[((slotrow + g + 8) * nph + psi) * B + 2 * t + 1] = acc[3];
                    }
                }
            }
            acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
            consumer_sync(nct);
            for (int idx = tid; idx < rows_in_pass * B; idx += nct) {
                const int row = idx / B, b = idx - row * B;
                const int m = row / (p.up * kUnitRows);
                const int rr = row - m * p.up * kUnitRows;
                const int64_t n = static_cast<int64_t>(ub) * kUnitRows + rr;
                if (NMAT == 2 && m == 1) continue;
                if (rr / kUnitRows >= nup || n >= p.N) continue;
                float v = 0.f;
                for (int q = 0; q < nph; ++q) v += red[(row * nph + q) * B + b];
                if (p.gamma) v *= rstd[b];
                if (NMAT == 1) {
                    if (p.residual) v += p.residual[b * p.ldr + n];
                } else {
                    float uv = 0.f;
                    const int urow = p.up * kUnitRows + rr;
                    for (int q = 0; q < nph; ++q) uv += red[(urow * nph + q) * B + b];
                    if (p.gamma) uv *= rstd[b];
                    v = act_fn(v, p.act) * uv;
                }
                p.y[b * p.ldy + n] = v;
            }
        }
    }
    // a copy never landed: give whatever the producer still had in flight a bounded chance to
    // land before the CTA exits
    __shared__ int any_failed;
    if (tid == 0) any_failed = 0;
    consumer_sync(nct);
    if (!ok) atomicOr(&any_failed, 1);
    consumer_sync(nct);
    if (any_failed && tid == 0) drain_stages(full, p.ns, max(0, S - p.ns), S - 1);
}

}  // namespace gemv_mma
}  // namespace gem
