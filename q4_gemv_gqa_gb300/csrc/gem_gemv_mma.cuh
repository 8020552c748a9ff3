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
// Work split.  A CTA owns a contiguous range of 16-row units; one matrix's 16 rows of one
// unit form a "row block".  K is walked in phases of `gps` groups (gps * 256 weights).  A
// ring stage holds one row block's `gps` consecutive groups (gps TMA boxes of 16 rows x
// 144 bytes): every row is read in runs of gps * 144 bytes (about 1 KB), which the HBM
// streams near its copy rate, where runs of 144 bytes per row reach less than half of it.
// The producer warp issues stages in (pass, phase, unit, matrix) order into a circular
// ring of `ns` slots.  Consumer warp w owns half group w of every stage (group w / 2,
// half w % 2: 16 rows x 128 weights), so all 2 * gps consumer warps walk the ring in
// order, and it adds its two per-row partial sums into a shared-memory slot of its own
// after each stage.  Activations of a phase are converted once per CTA into mma B
// fragments, double-buffered: phase ph + 1 is converted while phase ph's stages stream,
// so the warps meet at one barrier per phase.
#pragma once

#include "gem_device.cuh"

namespace gem {
namespace gemv_mma {

constexpr int kGroupBytes = 144;
constexpr int kUnitRows = 16;
constexpr int kBoxBytes = kGroupBytes * kUnitRows;
constexpr int kMaxConsumerWarps = 18;
constexpr int kMaxSlots = 32;                     // ring slots
constexpr int kMaxThreads = (kMaxConsumerWarps + 1) * 32;
constexpr int kPrefetchF4 = 2;                    // raw activation float4s per thread per phase
constexpr size_t kSmemBudget = 220 * 1024;
constexpr size_t kResidentX = 48 * 1024;         // activation fragments kept for all of K up to this size

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
    int U;               // 16-row units
    int up;              // units per pass (row blocks per pass = NMAT * up)
    int gps;             // groups per phase (one stage = one row block x gps groups)
    int nphase;          // phases per pass = ceil(G / gps)
    int ns;              // ring slots
    int ncw;             // consumer warps = 2 * gps
    int nbuf;            // activation fragment buffers: nphase (all resident) or 2 (double-buffered)
    uint32_t stage_bytes;
    uint32_t full_off, empty_off, xf_off, xf_bytes, xsc_off, rstd_off, red_off, ssq_off;
    int* status;
    unsigned* clear;     // words zeroed after the wait (see GemvOp)
    int nclear;
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

// Shared-memory loads at 32-bit shared addresses (the ring is read only after its full
// barrier, whose wait is a volatile asm with a memory clobber, so these stay after it).
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

// The 4-byte code word of a block whose codes for this lane start at shared address `ca`
// (block start + 2 + 4t): 4-byte aligned in odd blocks, two aligned words and a funnel
// shift in even ones (blocks are 18 bytes).
template <int JPAR>
__device__ __forceinline__ uint32_t code_word(uint32_t ca) {
    if constexpr (JPAR == 1) return lds32(ca);
    else return __funnelshift_r(lds32(ca - 2), lds32(ca + 2), 16);
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
    float* rstd = reinterpret_cast<float*>(smem + p.rstd_off);
    float* red = reinterpret_cast<float*>(smem + p.red_off);   // [row of pass][warp][B]
    float* ssqb = reinterpret_cast<float*>(smem + p.ssq_off);  // [B][K/128] sums of x^2

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ncw = p.ncw, nct = ncw * 32;
    const int C = gridDim.x, c = blockIdx.x;
    const int u0 = static_cast<int>((static_cast<int64_t>(c) * p.U) / C);
    const int u1 = static_cast<int>((static_cast<int64_t>(c + 1) * p.U) / C);
    const int npass = (u1 - u0 + p.up - 1) / p.up;
    const int B = p.B;

    __shared__ int any_failed;
    if (tid == 0) {
        any_failed = 0;
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
    // Stage s (order: pass, phase, unit, matrix) goes to slot s % ns.
    if (warp == ncw) {
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_first();
            bool ok = true;
            int s = 0, slot = 0;
            uint32_t par = 1;   // parity of the empty-barrier phase to wait for (from the second lap)
            for (int pass = 0; pass < npass && ok; ++pass) {
                const int ub = u0 + pass * p.up;
                const int nup = min(p.up, u1 - ub);
                // resident activations: row-block-major (every K-phase of a row block in turn);
                // otherwise phase-major, as the consumers convert one K-phase at a time
                const bool rbmajor = p.nbuf == p.nphase;
                const int nrb = nup * NMAT;
                for (int i = 0; i < p.nphase * nrb && ok; ++i) {
                    const int ph = rbmajor ? i % p.nphase : i / nrb;
                    const int rb = rbmajor ? i / p.nphase : i % nrb;
                    const int ul = rb / NMAT, m = rb % NMAT;
                    const int g0 = ph * p.gps;
                    const int ng = min(p.gps, p.G - g0);
                    if (s >= p.ns) {
                        ok = mbar_wait(&empty[slot], par, p.status);
                        if (!ok) break;
                    }
                    uint8_t* dst = smem + static_cast<size_t>(slot) * p.stage_bytes;
                    mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(ng * kBoxBytes));
                    for (int j = 0; j < ng; ++j)
                        tma_load_2d(dst + j * kBoxBytes, m ? &tm1 : &tm0, (g0 + j) * kGroupBytes,
                                    (ub + ul) * kUnitRows, &full[slot], policy);
                    ++s;
                    if (++slot == p.ns) {
                        slot = 0;
                        par ^= 1u;
                    }
                }
            }
            if (!ok) drain_stages(full, p.ns, max(0, s - p.ns), s - 1);
        }
        return;   // the producer warp never triggers: the consumers do, after their wait
    }

    // ---------------- consumer warps ----------------
    pdl_wait_trigger();  // activations and residual come from the previous kernel
    clear_words(p.clear, p.nclear, tid, nct);

    const int g = lane >> 2, t = lane & 3;
    const int jg = warp >> 1, eta = warp & 1;   // my half group inside every stage
    const bool col_ok = PACKED ? (g < 2 * B) : (g < B);
    const int kp = p.gps * 256;          // activations per phase
    const int nhg = kp / 128;            // half groups per phase
    const int hg = jg * 2 + eta;         // my half group inside the phase

    // Raw activations of a phase: slot f covers float4 e4 of batch row b (f = b * kp4 + e4).
    // Thread tid owns slots tid + i * nct; the first kPrefetchF4 are prefetched into
    // registers (with the matching norm weights) ahead of their conversion.
    const int kp4 = kp / 4;
    const int nslots = B * kp4;
    float4 pf[kPrefetchF4], pg[kPrefetchF4];
    auto load_slot = [&](int phase, int f, float4& xv, float4& gv) {
        const int k0 = phase * kp;
        const int lim = min(kp, p.G * 256 - k0);
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
    // One slot -> binary16 hi/lo B fragments in buffer `buf`.  The 32 lanes of a warp hold
    // one 128-element half group of one row (kp4 is a multiple of 32), so the power-of-two
    // scale and the sum of squares are warp reductions.
    auto convert_slot = [&](int phase, int buf, int f, float4 v, float4 gm, bool first_pass) {
        const int b = f / kp4, e4 = f - b * kp4;
        if (p.gamma) {
            const int hgk = phase * nhg + (e4 >> 5);   // half group inside the row
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
        const int hgi = e4 >> 5, ln = e4 & 31;
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
        uint8_t* xfp = smem + p.xf_off + buf * p.xf_bytes;
        if constexpr (PACKED) {
            *reinterpret_cast<uint2*>(xfp + xf_entry<true>(hgi, j, tt, 2 * b, B) + tile * 8) = hv;
            *reinterpret_cast<uint2*>(xfp + xf_entry<true>(hgi, j, tt, 2 * b + 1, B) + tile * 8) = lv;
        } else {
            uint8_t* base = xfp + xf_entry<false>(hgi, j, tt, b, B);
            *reinterpret_cast<uint2*>(base + tile * 8) = hv;
            *reinterpret_cast<uint2*>(base + 16 + tile * 8) = lv;
        }
        float* xsc = reinterpret_cast<float*>(smem + p.xsc_off) + buf * nhg * B;
        if (lane == 0) xsc[hgi * B + b] = __int_as_float((127 + ex) << 23);
    };
    auto convert = [&](int phase, int buf, bool first_pass) {
#pragma unroll
        for (int i = 0; i < kPrefetchF4; ++i) {
            const int f = tid + i * nct;
            if (f < nslots) convert_slot(phase, buf, f, pf[i], pg[i], first_pass);
        }
        for (int f = tid + kPrefetchF4 * nct; f < nslots; f += nct) {  // beyond the prefetch
            float4 xv, gv;
            load_slot(phase, f, xv, gv);
            convert_slot(phase, buf, f, xv, gv, first_pass);
        }
    };

    // All phases at once (resident fragments, converted in pass 0 only): my slots
    // f = tid + i * nct over (phase, row, float4), loaded two at a time before converting.
    auto convert_all = [&]() {
        const int per_phase = B * kp4;
        const int total = p.nphase * per_phase;
        for (int f0 = tid; f0 < total; f0 += 2 * nct) {
            float4 xv[2], gv[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int f = f0 + i * nct;
                if (f < total) load_slot(f / per_phase, f % per_phase, xv[i], gv[i]);
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int f = f0 + i * nct;
                if (f < total) convert_slot(f / per_phase, f / per_phase, f % per_phase, xv[i], gv[i], true);
            }
        }
    };

    bool ok = true;
    int s = 0, slot = 0;
    uint32_t par = 0;                      // parity of the full-barrier phase to wait for
    const bool resident = p.nbuf == p.nphase;
    const int nq = npass * p.nphase;       // phases over all passes (the same activations each pass)
    if (!resident) prefetch(0);
    // Every consumer warp runs the same sequence of named barriers whatever happens: after a
    // timed-out wait (ok == false) the remaining waits are skipped, never the barriers.
    for (int pass = 0; pass < npass; ++pass) {
        const int ub = u0 + pass * p.up;
        const int nup = min(p.up, u1 - ub);
        const int q0 = pass * p.nphase;
        consumer_sync(nct);                 // the previous pass is done with the buffers
        if (resident) {
            if (pass == 0) convert_all();
        } else {
            convert(0, q0 & 1, pass == 0);
            if (q0 + 1 < nq) prefetch((q0 + 1) % p.nphase);
        }
        consumer_sync(nct);                 // fragments published
        if (resident) {
            // Row-block-major: all K-phases of one row block in turn, running sums in registers,
            // one store per row block (no read-modify-write of shared partial sums per stage).
            const uint32_t soff = static_cast<uint32_t>(jg * kBoxBytes + g * kGroupBytes + eta * 72);
            const uint32_t ring0 = smem_u32(smem);
            const int nrb = nup * NMAT;
            for (int rb = 0; rb < nrb; ++rb) {
                float tot[4] = {0.f, 0.f, 0.f, 0.f};
                for (int ph = 0; ph < p.nphase; ++ph) {
                    const int ng = min(p.gps, p.G - ph * p.gps);
                    const bool mine = jg < ng;
                    if (ok) ok = mbar_wait(&full[slot], par, p.status);
                    if (mine) {
                        const uint8_t* xfb = smem + p.xf_off + ph * p.xf_bytes;
                        const float* xsc = reinterpret_cast<const float*>(smem + p.xsc_off) + ph * nhg * B;
                        float sc0, sc1 = 0.f;
                        if constexpr (PACKED) {
                            sc0 = t < B ? xsc[hg * B + t] : 0.f;
                        } else {
                            sc0 = 2 * t < B ? xsc[hg * B + 2 * t] : 0.f;
                            sc1 = 2 * t + 1 < B ? xsc[hg * B + 2 * t + 1] : 0.f;
                        }
                        const uint32_t sa = ring0 + static_cast<uint32_t>(slot) * p.stage_bytes + soff;  // scales
                        const uint32_t ca = sa + 2 + 4 * t;                                               // codes
                        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            uint4 bh = make_uint4(0, 0, 0, 0), bl = make_uint4(0, 0, 0, 0);
                            if (col_ok) {
                                bh = *reinterpret_cast<const uint4*>(xfb + xf_entry<PACKED>(hg, j, t, g, B));
                                if constexpr (!PACKED) bl = *reinterpret_cast<const uint4*>(xfb + xf_entry<false>(hg, j, t, g, B) + 16);
                            }
                            uint32_t wg, wg8;
                            if ((j & 1) != 0) {
                                wg = code_word<1>(ca + 18 * j);
                                wg8 = code_word<1>(ca + 18 * j + 8 * kGroupBytes);
                            } else {
                                wg = code_word<0>(ca + 18 * j);
                                wg8 = code_word<0>(ca + 18 * j + 8 * kGroupBytes);
                            }
                            const float dg = half_bits_to_float(lds16(sa + 18 * j));
                            const float dg8 = half_bits_to_float(lds16(sa + 18 * j + 8 * kGroupBytes));
                            uint32_t a0, a2, a4, a6, a1, a3, a5, a7;
                            dequant_word(wg, a0, a2, a4, a6);
                            dequant_word(wg8, a1, a3, a5, a7);
                            float cf[4] = {0.f, 0.f, 0.f, 0.f};
                            mma_16816(cf, a0, a1, a2, a3, bh.x, bh.y);
                            mma_16816(cf, a4, a5, a6, a7, bh.z, bh.w);
                            if constexpr (PACKED) {
                                acc[0] = fmaf(dg, cf[0] + cf[1], acc[0]);
                                acc[1] = fmaf(dg8, cf[2] + cf[3], acc[1]);
                            } else {
                                mma_16816(cf, a0, a1, a2, a3, bl.x, bl.y);
                                mma_16816(cf, a4, a5, a6, a7, bl.z, bl.w);
                                acc[0] = fmaf(dg, cf[0], acc[0]);
                                acc[1] = fmaf(dg, cf[1], acc[1]);
                                acc[2] = fmaf(dg8, cf[2], acc[2]);
                                acc[3] = fmaf(dg8, cf[3], acc[3]);
                            }
                        }
                        if constexpr (PACKED) {
                            tot[0] = fmaf(sc0, acc[0], tot[0]);
                            tot[1] = fmaf(sc0, acc[1], tot[1]);
                        } else {
                            tot[0] = fmaf(sc0, acc[0], tot[0]);
                            tot[1] = fmaf(sc1, acc[1], tot[1]);
                            tot[2] = fmaf(sc0, acc[2], tot[2]);
                            tot[3] = fmaf(sc1, acc[3], tot[3]);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[slot]);
                    if (++slot == p.ns) {
                        slot = 0;
                        par ^= 1u;
                    }
                    ++s;
                }
                if (jg < min(p.gps, p.G)) {   // owned a half group in phase 0: my slots of this row block
                    float* rr = red + ((rb * kUnitRows + g) * ncw + warp) * B;
                    float* rr8 = rr + 8 * ncw * B;
                    if constexpr (PACKED) {
                        if (t < B) {
                            rr[t] = tot[0];
                            rr8[t] = tot[1];
                        }
                    } else {
                        if (2 * t < B) {
                            rr[2 * t] = tot[0];
                            rr8[2 * t] = tot[2];
                        }
                        if (2 * t + 1 < B) {
                            rr[2 * t + 1] = tot[1];
                            rr8[2 * t + 1] = tot[3];
                        }
                    }
                }
            }
        }
        for (int ph = 0; ph < (resident ? 0 : p.nphase); ++ph) {
            const int q = q0 + ph;
            if (!resident && ph + 1 < p.nphase) {   // next phase into the other buffer
                convert(ph + 1, (q + 1) & 1, pass == 0);
                if (q + 2 < nq) prefetch((q + 2) % p.nphase);
            }
            const int buf = resident ? ph : (q & 1);
            const int ng = min(p.gps, p.G - ph * p.gps);
            const bool mine = jg < ng;
            const uint8_t* xfb = smem + p.xf_off + buf * p.xf_bytes;
            const float* xsc = reinterpret_cast<const float*>(smem + p.xsc_off) + buf * nhg * B;
            float sc0 = 0.f, sc1 = 0.f;     // power-of-two activation scales of my half group
            if constexpr (PACKED) {
                sc0 = t < B ? xsc[hg * B + t] : 0.f;
            } else {
                sc0 = 2 * t < B ? xsc[hg * B + 2 * t] : 0.f;
                sc1 = 2 * t + 1 < B ? xsc[hg * B + 2 * t + 1] : 0.f;
            }
            uint4 xh[4];                    // B <= 4: my activation fragments, the same for every stage
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                xh[j] = make_uint4(0, 0, 0, 0);
                if (PACKED && col_ok) xh[j] = *reinterpret_cast<const uint4*>(xfb + xf_entry<true>(hg, j, t, g, B));
            }
            float* rr = red + (g * ncw + warp) * B;   // my partial-sum slots, row g of row block 0
            // my half group inside a stage: row g, blocks 4 eta .. 4 eta + 3 of group jg
            const uint32_t soff = static_cast<uint32_t>(jg * kBoxBytes + g * kGroupBytes + eta * 72);
            const uint32_t ring0 = smem_u32(smem);
            for (int ul = 0; ul < nup; ++ul) {
                for (int m = 0; m < NMAT; ++m, rr += kUnitRows * ncw * B) {
                    if (ok) ok = mbar_wait(&full[slot], par, p.status);
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
                    if (mine) {
                        const uint32_t sa = ring0 + static_cast<uint32_t>(slot) * p.stage_bytes + soff;  // scales
                        const uint32_t ca = sa + 2 + 4 * t;                                               // codes
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            uint32_t wg, wg8;
                            if (((eta * 4 + j) & 1) != 0) {   // eta * 4 is even: parity of j
                                wg = code_word<1>(ca + 18 * j);
                                wg8 = code_word<1>(ca + 18 * j + 8 * kGroupBytes);
                            } else {
                                wg = code_word<0>(ca + 18 * j);
                                wg8 = code_word<0>(ca + 18 * j + 8 * kGroupBytes);
                            }
                            const float dg = half_bits_to_float(lds16(sa + 18 * j));
                            const float dg8 = half_bits_to_float(lds16(sa + 18 * j + 8 * kGroupBytes));
                            uint32_t a0, a2, a4, a6, a1, a3, a5, a7;
                            dequant_word(wg, a0, a2, a4, a6);
                            dequant_word(wg8, a1, a3, a5, a7);
                            float cf[4] = {0.f, 0.f, 0.f, 0.f};
                            if constexpr (PACKED) {
                                mma_16816(cf, a0, a1, a2, a3, xh[j].x, xh[j].y);
                                mma_16816(cf, a4, a5, a6, a7, xh[j].z, xh[j].w);
                                acc[0] = fmaf(dg, cf[0] + cf[1], acc[0]);
                                acc[1] = fmaf(dg8, cf[2] + cf[3], acc[1]);
                            } else {
                                uint4 bh = make_uint4(0, 0, 0, 0), bl = make_uint4(0, 0, 0, 0);
                                if (col_ok) {
                                    bh = *reinterpret_cast<const uint4*>(xfb + xf_entry<false>(hg, j, t, g, B));
                                    bl = *reinterpret_cast<const uint4*>(xfb + xf_entry<false>(hg, j, t, g, B) + 16);
                                }
                                mma_16816(cf, a0, a1, a2, a3, bh.x, bh.y);
                                mma_16816(cf, a4, a5, a6, a7, bh.z, bh.w);
                                mma_16816(cf, a0, a1, a2, a3, bl.x, bl.y);
                                mma_16816(cf, a4, a5, a6, a7, bl.z, bl.w);
                                acc[0] = fmaf(dg, cf[0], acc[0]);
                                acc[1] = fmaf(dg, cf[1], acc[1]);
                                acc[2] = fmaf(dg8, cf[2], acc[2]);
                                acc[3] = fmaf(dg8, cf[3], acc[3]);
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[slot]);
                    if (++slot == p.ns) {
                        slot = 0;
                        par ^= 1u;
                    }
                    ++s;
                    // my partial sums of this row block: red[(row * ncw + warp) * B + b]
                    if (mine) {
                        float* rr8 = rr + 8 * ncw * B;
                        if constexpr (PACKED) {
                            if (t < B) {
                                rr[t] = (ph ? rr[t] : 0.f) + sc0 * acc[0];
                                rr8[t] = (ph ? rr8[t] : 0.f) + sc0 * acc[1];
                            }
                        } else {
                            if (2 * t < B) {
                                rr[2 * t] = (ph ? rr[2 * t] : 0.f) + sc0 * acc[0];
                                rr8[2 * t] = (ph ? rr8[2 * t] : 0.f) + sc0 * acc[2];
                            }
                            if (2 * t + 1 < B) {
                                rr[2 * t + 1] = (ph ? rr[2 * t + 1] : 0.f) + sc1 * acc[1];
                                rr8[2 * t + 1] = (ph ? rr8[2 * t + 1] : 0.f) + sc1 * acc[3];
                            }
                        }
                    }
                }
            }
            if (!resident) consumer_sync(nct);   // next buffer published; this one free again
        }
        if (resident) consumer_sync(nct);        // every partial sum written
        // ---- end of pass: combine the per-warp partial sums of every row, write outputs ----
        if (pass == 0 && p.gamma) {   // 1 / rms of every activation row (pass 0 saw all of K)
            if (tid < B) {
                float sum = 0.f;
                for (int i = 0; i < 2 * p.G; ++i) sum += ssqb[tid * (2 * p.G) + i];
                rstd[tid] = rsqrtf(sum / static_cast<float>(p.G * 256) + p.eps);
            }
            consumer_sync(nct);
        }
        // warps that own no half group of the first phase never wrote their slots
        const int nw = min(ncw, 2 * min(p.gps, p.G));
        const int rows_in_pass = nup * NMAT * kUnitRows;
        for (int idx = tid; idx < rows_in_pass * B; idx += nct) {
            const int row = idx / B, b = idx - row * B;
            const int rb = row / kUnitRows, r16 = row - rb * kUnitRows;
            const int u = rb / NMAT, m = rb - u * NMAT;
            const int64_t n = static_cast<int64_t>(ub + u) * kUnitRows + r16;
            if (NMAT == 2 && m == 1) continue;
            if (n >= p.N) continue;
            float v = 0.f;
            for (int w = 0; w < nw; ++w) v += red[(row * ncw + w) * B + b];
            if (p.gamma) v *= rstd[b];
            if (NMAT == 1) {
                if (p.residual) v += p.residual[b * p.ldr + n];
            } else {
                float uv = 0.f;
                const int urow = row + kUnitRows;   // same unit, matrix 1
                for (int w = 0; w < nw; ++w) uv += red[(urow * ncw + w) * B + b];
                if (p.gamma) uv *= rstd[b];
                v = act_fn(v, p.act) * uv;
            }
            p.y[b * p.ldy + n] = v;
        }
    }
    // a copy never landed: give the copies the producer may still have in flight a bounded
    // chance to land before the CTA exits
    if (!ok) atomicOr(&any_failed, 1);
    consumer_sync(nct);
    if (any_failed && tid == 0) drain_stages(full, p.ns, max(0, s - p.ns), s - 1);
}

}  // namespace gemv_mma
}  // namespace gem
