// gem_gemv_b1.cuh — Q4_0 GEMV for one activation row (B = 1) on mma.sync, block-diagonal form.
//
// Same staging as the general tensor-core kernel (gem_gemv_mma.cuh): a TMA producer warp streams
// row blocks (16 rows of one matrix) x `gps` consecutive 256-weight groups into a ring, rows read
// in ~1 KB runs; consumer warp w owns half group w of every stage.  What differs is how a warp
// maps its 16 rows x 128 weights onto m16n8k16:
//
// * A half group is not 4 consecutive blocks but the 4 even (w even) or the 4 odd (w odd) blocks
//   of a 256-weight group, and lane quad position t owns block 2t (+1) entirely: all 8 k-tiles of
//   the task take lane t's four k-slots from that one block, so each lane reads its block's 16
//   code bytes as 4-byte words with one scale, instead of 4 bytes of 4 blocks with 4 scales.
//   Even blocks start 4-byte aligned (scale in the low half of the first word, codes in words
//   1-3 plus two 2-byte tails joined by one byte permute), odd blocks 2 bytes past (scale in the
//   high half of the first word, codes in 4 aligned words).
// * The activation operand is block diagonal: B column n = 2t + h holds block t's activations
//   (h = 0 the binary16 high part, h = 1 the low remainder) in lane t's k-slots and zero
//   elsewhere, so D[row][2t + h] is the dot product of the row's block t with the hi or lo part.
//   Lane (g, t) ends a task holding rows g and g + 8 of its own block in hi and lo: one
//   d * (hi + lo) per row.  All 8 columns are used, where a plain layout would use 2 of 8.
// * Each 32-weight block of the activation vector is scaled by its own power of two (its largest
//   magnitude to [2^13, 2^14)), undone exactly by folding the inverse into the block's scale d.
//   The records are therefore built straight from the loads: one CTA-wide barrier between the
//   activation loads and the first task; a fused RMSNorm's 1/rms only scales the epilogue.
//
// Reference: "Q4_0 dequant-matvec" (GGML block: fp16 d, 16 bytes of codes, value (q - 8) * d).
#pragma once

#include <cuda_fp16.h>

#include <type_traits>

#include "gem_gemv_mma.cuh"

namespace gem {
namespace gemv_b1 {

using gemv_mma::kBoxBytes;
using gemv_mma::kGroupBytes;
using gemv_mma::kMaxSlots;
using gemv_mma::kUnitRows;

constexpr int kMaxConsumerWarps = 18;
constexpr int kMaxThreads = (kMaxConsumerWarps + 1) * 32;
constexpr int kRecBytes = 512;   // activation record of one half group: 8 columns x 8 tiles x 8 B
constexpr int kZeroBytes = 96;   // the operand of lanes off the block diagonal (bytes 32..95)
constexpr int kPro = 4;          // float4s of the activation row kept per consumer thread
constexpr int kProSplit = 6;     // the same for a CTA of a K split (its range only)
constexpr int kMaxRps = 3;       // row blocks per stage at most

struct Params {
    int64_t N;
    int G;               // 256-weight groups per row
    const float* x;
    float* y;
    const float* residual;
    const float* gamma;
    float eps;
    int act;
    int U;               // 16-row units
    int up;              // units per pass
    int gps;             // groups per phase (stage = rps row blocks x gps groups)
    int rps;             // row blocks per stage (1..kMaxRps): as many as the CTAs' units allow
    int ks;              // K split (the kernel's KS): the CTAs of a ks-CTA cluster take K ranges of the same units
    int nphase;
    int ns;
    int ncw;             // consumer warps = 2 * gps
    uint32_t stage_bytes, full_off, empty_off, xf_off, red_off, misc_off, bsc_off;
    int* status;
    unsigned* clear;     // words zeroed after the wait (see GemvOp)
    int nclear;
};

// qs byte held in byte j of code word i of a lane's block.  Odd blocks: word i = bytes 4i..4i+3.
// Even blocks: word i = bytes 4i-2 .. 4i+1 mod 16 (word 0 = {14, 15, 0, 1}: the two 2-byte tails).
__device__ __forceinline__ int code_byte(bool odd, int i, int j) {
    return odd ? 4 * i + j : (4 * i + j + 14) & 15;
}
// The inverse: code word and byte of qs byte m.
__device__ __forceinline__ void code_slot(bool odd, int m, int& i, int& j) {
    const int mm = odd ? m : (m + 2) & 15;
    i = mm >> 2;
    j = mm & 3;
}

// Every thread of every CTA of the cluster arrives, then waits (release / acquire).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ float ld_cluster_f32(const void* local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// One task: rows g and g + 8 of one block per lane in each of NR row blocks (the same K range,
// so they share the activation operand), 8 mma per row block.  a = shared offset of the lane's
// 5 words in row g of row block 0 (row g + 8 is 8 rows further, row block r is r * rstride
// further); xr = shared offset of the lane's 64-byte activation operand.
template <bool ODD, int NR>
__device__ __forceinline__ void task(const uint8_t* smem, uint32_t a, uint32_t rstride, uint32_t xr, float bs,
                                     float (&t0)[kMaxRps], float (&t1)[kMaxRps]) {
    const uint4* xp = reinterpret_cast<const uint4*>(smem + xr);
    uint4 xb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) xb[i] = xp[i];
    uint32_t ca[NR][4], cb[NR][4];
    float da[NR], db[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        const uint32_t* wa = reinterpret_cast<const uint32_t*>(smem + a + r * rstride);
        const uint32_t* wb = reinterpret_cast<const uint32_t*>(smem + a + r * rstride + 8 * kGroupBytes);
        uint32_t ra[5], rb[5];
#pragma unroll
        for (int i = 0; i < 5; ++i) {
            ra[i] = wa[i];
            rb[i] = wb[i];
        }
        if constexpr (ODD) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                ca[r][i] = ra[i + 1];
                cb[r][i] = rb[i + 1];
            }
            da[r] = __high2float(*reinterpret_cast<const __half2*>(&ra[0]));
            db[r] = __high2float(*reinterpret_cast<const __half2*>(&rb[0]));
        } else {
            ca[r][0] = __byte_perm(ra[0], ra[4], 0x3254);   // qs 14, 15 (word 4), qs 0, 1 (word 0)
            cb[r][0] = __byte_perm(rb[0], rb[4], 0x3254);
#pragma unroll
            for (int i = 1; i < 4; ++i) {
                ca[r][i] = ra[i];
                cb[r][i] = rb[i];
            }
            da[r] = __low2float(*reinterpret_cast<const __half2*>(&ra[0]));
            db[r] = __low2float(*reinterpret_cast<const __half2*>(&rb[0]));
        }
    }
    float d[NR][4];
#pragma unroll
    for (int r = 0; r < NR; ++r) d[r][0] = d[r][1] = d[r][2] = d[r][3] = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            uint32_t l02, l13, h02, h13, m02, m13, n02, n13;
            gemv_mma::dequant_word(ca[r][i], l02, l13, h02, h13);   // row g: low nibbles (b0,b2) (b1,b3), high nibbles
            gemv_mma::dequant_word(cb[r][i], m02, m13, n02, n13);   // row g + 8
            mma_16816(d[r], l02, m02, l13, m13, xb[i].x, xb[i].y);  // k-tile 2i: low nibbles of word i
            mma_16816(d[r], h02, n02, h13, n13, xb[i].z, xb[i].w);  // k-tile 2i + 1: high nibbles
        }
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) {   // bs: 2^-e of the block's operand scale (exact)
        t0[r] = fmaf(da[r] * bs, d[r][0] + d[r][1], t0[r]);
        t1[r] = fmaf(db[r] * bs, d[r][2] + d[r][3], t1[r]);
    }
}

// KS = 1, or 2 for the form whose CTA pairs (thread-block clusters) split K (a separate
// instantiation, so the plain form carries none of the split's code).
template <int NMAT, int KS>
__global__ void __launch_bounds__(kMaxThreads, 1) q4_0_gemv_b1_kernel(const __grid_constant__ CUtensorMap tm0,
                                                                      const __grid_constant__ CUtensorMap tm1,
                                                                      const Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.full_off);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + p.empty_off);
    float* red = reinterpret_cast<float*>(smem + p.red_off);    // [row of pass][warp]
    float* misc = reinterpret_cast<float*>(smem + p.misc_off);  // [warp]: partial sums of squares

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ncw = p.ncw, nct = ncw * 32;
    const int G = p.G, gps = p.gps, nphase = p.nphase, ns = p.ns, rps = p.rps;
    const uint32_t stage_bytes = p.stage_bytes;
    const uint32_t rstride = static_cast<uint32_t>(gps * kBoxBytes);   // second row block of a stage
    // K split: cluster cid (of ncl) owns a unit range; its CTA `rank` owns groups [gk0, gk0 + Gr)
    constexpr int ks = KS;
    const int rank = static_cast<int>(blockIdx.x) % ks, cid = static_cast<int>(blockIdx.x) / ks;
    const int ncl = static_cast<int>(gridDim.x) / ks;
    const int gk0 = KS == 1 ? 0 : rank * G / ks;
    const int Gr = KS == 1 ? G : (rank + 1) * G / ks - gk0;
    const int nphr = KS == 1 ? nphase : (Gr + gps - 1) / gps;   // this CTA's phases
    const int u0 = static_cast<int>((static_cast<int64_t>(cid) * p.U) / ncl);
    const int u1 = static_cast<int>((static_cast<int64_t>(cid + 1) * p.U) / ncl);
    const int npass = (u1 - u0 + p.up - 1) / p.up;   // 1 whenever ks > 1

    __shared__ int any_failed;
    if (tid == 0) {
        any_failed = 0;
        for (int i = 0; i < ns; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], ncw);
        }
        fence_mbar_init();
        prefetch_tensormap(&tm0);
        if (NMAT == 2) prefetch_tensormap(&tm1);
    }
    __syncthreads();

    // ---------------- producer warp: stages (pass, row-block tuple, phase) ----------------
    // Row blocks of a pass: rb = unit * NMAT + matrix; stage v holds rb v * rps .. v * rps + rps - 1
    // (those that exist) x the phase's groups.
    if (warp == ncw) {
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_first();
            bool ok = true;
            int s = 0, slot = 0;
            uint32_t par = 1;
            for (int pass = 0; pass < npass && ok; ++pass) {
                const int ub = u0 + pass * p.up;
                const int nrb = min(p.up, u1 - ub) * NMAT;
                for (int v = 0; v * rps < nrb && ok; ++v) {
                    const int nr = min(rps, nrb - v * rps);
                    for (int ph = 0; ph < nphr; ++ph) {
                        const int g0 = ph * gps;
                        const int ng = min(gps, Gr - g0);
                        if (s >= ns) {
                            ok = mbar_wait(&empty[slot], par, p.status);
                            if (!ok) break;
                        }
                        uint8_t* dst = smem + static_cast<size_t>(slot) * stage_bytes;
                        // Test hook (GEM_INJECT_RING_SHORTFALL): CTA 0 expects 16 bytes more than
                        // its last stage copies, so the consumers' wait on it runs out.  The last
                        // stage's slot is never refilled, and every copy still lands.
                        uint32_t extra = 0;
                        if (KS == 1 && blockIdx.x == 0 && pass == npass - 1 && (v + 1) * rps >= nrb &&
                            ph == nphr - 1 && (test_inject() & GEM_INJECT_RING_SHORTFALL))
                            extra = 16;
                        mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(nr * ng * kBoxBytes) + extra);
                        for (int r = 0; r < nr; ++r) {
                            const int rb = v * rps + r;
                            const int row0 = (ub + rb / NMAT) * kUnitRows;
                            const CUtensorMap* tm = (NMAT == 2 && (rb & 1)) ? &tm1 : &tm0;
                            for (int j = 0; j < ng; ++j)
                                tma_load_2d(dst + r * rstride + j * kBoxBytes, tm, (gk0 + g0 + j) * kGroupBytes,
                                            row0, &full[slot], policy);
                        }
                        ++s;
                        if (++slot == ns) {
                            slot = 0;
                            par ^= 1u;
                        }
                    }
                }
            }
            if (!ok) drain_stages(full, ns, max(0, s - ns), s - 1);
        }
        // the producer warp never triggers dependents: the consumers do, after their wait
        if constexpr (KS > 1) {   // the consumers' combine: two cluster barriers per pass (one pass)
            __syncwarp();
            for (int i = 0; i < 2 * npass; ++i) cluster_sync_all();
        }
        return;
    }

    // ---------------- consumer warps ----------------
    pdl_wait_trigger();   // the activations (and residual) come from the previous kernel
    clear_words(p.clear, p.nclear, tid, nct);

    const int K = G * 256, K4 = K / 4;
    // this CTA's records cover groups [gk0, gk0 + Gr): float4s [kr0, kr1) of the row
    const int kr0 = gk0 * 64, kr1 = (gk0 + Gr) * 64;
    float* bsc = reinterpret_cast<float*>(smem + p.bsc_off);   // [local block]: 2^-e of its operand scale
    uint8_t* xf = smem + p.xf_off;
    const float4* x4 = reinterpret_cast<const float4*>(p.x);
    const float4* g4 = reinterpret_cast<const float4*>(p.gamma);
    float ss = 0.f;   // sum of x^2 for a fused RMSNorm (whole row), needed only by the epilogue
    // Every 32-weight block gets its own power of two taking its largest |gamma x| to
    // [2^13, 2^14) (exact), undone by folding 2^-e into the block's scale d in the tasks, so the
    // records are built straight from the loads with no CTA-wide reduction first.  The 8 float4
    // of a block are held by 8 consecutive lanes: their maximum takes 3 shuffles.  Every lane
    // of the warp calls this (valid or not); it returns 2^e.
    auto block_scale = [&](float4 v, bool valid, int lb) -> float {
        float m = valid ? fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))) : 0.f;
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
        int e = 0;
        if (m > 0.f) e = 13 - (((__float_as_int(m) >> 23) & 0xff) - 127);
        e = max(-126, min(126, e));
        if (valid && (lane & 7) == 0) bsc[lb] = __int_as_float((127 - e) << 23);
        return __int_as_float((127 + e) << 23);
    };
    // activation records: record (hg, column 2t + h), tile tau, register r holds the h part of
    // the two elements of block 2t + (hg & 1) of group hg / 2 that lane t's k-slots of that
    // register meet in the A operand (bytes j = r and r + 2 of code word tau / 2, nibble tau & 1).
    // Float4 i of the row, scaled by sc, into its slots (element m of a block's nibble half goes
    // to the slot of qs byte m).
    auto scatter4 = [&](float4 v, float sc, int i) {
        const int k0 = 4 * i;
        const int blk = (k0 >> 5) & 7, e0 = k0 & 31;
        const bool odd = blk & 1;
        const uint32_t rec = static_cast<uint32_t>((2 * ((k0 >> 8) - gk0) + (odd ? 1 : 0)) * kRecBytes +
                                                   (blk >> 1) * 128 + (e0 >> 4) * 8);
        const float v4[4] = {v.x * sc, v.y * sc, v.z * sc, v.w * sc};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            int ci, cj;
            code_slot(odd, (e0 & 15) + e, ci, cj);
            const uint32_t off = rec + ci * 16 + (cj & 1) * 4 + (cj >> 1) * 2;
            __half h, l;
            split_hi_lo(v4[e], h, l);
            *reinterpret_cast<__half*>(xf + off) = h;
            *reinterpret_cast<__half*>(xf + off + 64) = l;
        }
    };
    // Up to kProN float4 per consumer thread are read once (loads first) and converted from
    // registers; longer ranges are read twice (block scales, then a gather of the records).
    constexpr int kProN = KS > 1 ? kProSplit : kPro;
    if (kr1 - kr0 <= kProN * nct) {
        float4 xv[kProN], gv[kProN];
#pragma unroll
        for (int u = 0; u < kProN; ++u) {
            const int i = kr0 + tid + u * nct;
            xv[u] = i < kr1 ? __ldg(x4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            gv[u] = p.gamma && i < kr1 ? __ldg(g4 + i) : make_float4(1.f, 1.f, 1.f, 1.f);
        }
#pragma unroll
        for (int u = 0; u < kProN; ++u) {
            if (kr0 + u * nct >= kr1) break;   // uniform over the CTA
            const int i = kr0 + tid + u * nct;
            const bool valid = i < kr1;
            float4 v = xv[u];
            ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
            v.x *= gv[u].x; v.y *= gv[u].y; v.z *= gv[u].z; v.w *= gv[u].w;
            const float sc = block_scale(v, valid, (i - kr0) >> 3);
            if (valid) scatter4(v, sc, i);
        }
    } else {
        for (int i0 = kr0; i0 < kr1; i0 += nct) {   // block scales (uniform trip count)
            const int i = i0 + tid;
            const bool valid = i < kr1;
            float4 v = valid ? __ldg(x4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
            if (p.gamma && valid) {
                const float4 gm = __ldg(g4 + i);
                v.x *= gm.x; v.y *= gm.y; v.z *= gm.z; v.w *= gm.w;
            }
            (void)block_scale(v, valid, (i - kr0) >> 3);
        }
        gemv_mma::consumer_sync(nct);   // block scales visible
        // gather: four registers per thread and round, their loads issued before converting
        const int nreg = 2 * Gr * 64;   // (local hg, t, tau, r)
        for (int i0 = tid; i0 < nreg; i0 += 4 * nct) {
            float v0[4], v1[4], sc[4];
            uint32_t off[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * nct;
                v0[u] = v1[u] = 0.f;
                sc[u] = 1.f;
                off[u] = 0;
                if (i < nreg) {
                    const int hg = i >> 6, t = (i >> 4) & 3, tau = (i >> 1) & 7, r = i & 1;
                    const bool odd = hg & 1;
                    const int lb = (hg >> 1) * 8 + 2 * t + (odd ? 1 : 0);
                    const int base = ((hg >> 1) + gk0) * 256 + (2 * t + (odd ? 1 : 0)) * 32 + (tau & 1) * 16;
                    const int k0 = base + code_byte(odd, tau >> 1, r);
                    const int k1 = base + code_byte(odd, tau >> 1, r + 2);
                    v0[u] = __ldg(p.x + k0);
                    v1[u] = __ldg(p.x + k1);
                    if (p.gamma) {
                        v0[u] *= __ldg(p.gamma + k0);
                        v1[u] *= __ldg(p.gamma + k1);
                    }
                    sc[u] = __int_as_float(0x7F000000 - __float_as_int(bsc[lb]));   // 2^e, exact
                    off[u] = static_cast<uint32_t>(hg * kRecBytes + (2 * t) * 64 + tau * 8 + r * 4);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (i0 + u * nct < nreg) {
                    __half h0, l0, h1, l1;
                    split_hi_lo(v0[u] * sc[u], h0, l0);
                    split_hi_lo(v1[u] * sc[u], h1, l1);
                    *reinterpret_cast<__half2*>(xf + off[u]) = __halves2half2(h0, h1);
                    *reinterpret_cast<__half2*>(xf + off[u] + 64) = __halves2half2(l0, l1);
                }
            }
        }
    }
    if (KS > 1 && p.gamma)   // the norm needs the whole row: the sum of squares outside this range
        for (int i = tid; i < K4; i += nct)
            if (i < kr0 || i >= kr1) {
                const float4 v = __ldg(x4 + i);
                ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
            }
    ss = warp_sum(ss);
    if (lane == 0) misc[warp] = ss;
    if (tid < kZeroBytes / 4) reinterpret_cast<uint32_t*>(xf + 2 * Gr * kRecBytes)[tid] = 0u;
    gemv_mma::consumer_sync(nct);   // records, block scales and partial sums of squares complete
    // the fused RMSNorm's 1 / rms, summed in the same order in every thread
    float out = 1.f;
    if (p.gamma) {
        float q = 0.f;
        for (int w = 0; w < ncw; ++w) q += misc[w];
        out = rsqrtf(q / static_cast<float>(K) + p.eps);
    }

    const int g = lane >> 2, t = lane & 3;
    const int jg = warp >> 1;
    const bool odd = warp & 1;
    // my 5 words of row g inside a stage (group jg, block 2t (+1)); my activation operand (the
    // zero block, 32 bytes past its start, sits on other banks than the records read with it)
    const uint32_t aoff = static_cast<uint32_t>(jg * kBoxBytes + g * kGroupBytes + 36 * t + (odd ? 16 : 0));
    const bool diag = (g >> 1) == t;
    const uint32_t xbase = diag ? p.xf_off + static_cast<uint32_t>(warp * kRecBytes + g * 64)
                                : p.xf_off + static_cast<uint32_t>(2 * Gr * kRecBytes + 32);
    const uint32_t xstep = diag ? static_cast<uint32_t>(2 * gps * kRecBytes) : 0u;   // per phase

    bool ok = true;
    int s = 0, slot = 0;
    uint32_t par = 0;
    auto run = [&](auto odd_tag) {
        constexpr bool ODD = decltype(odd_tag)::value;
        for (int pass = 0; pass < npass; ++pass) {
            const int ub = u0 + pass * p.up;
            const int nrb = min(p.up, u1 - ub) * NMAT;
            gemv_mma::consumer_sync(nct);   // the previous pass has read `red`
            for (int v = 0; v * rps < nrb; ++v) {
                const int nr = min(rps, nrb - v * rps);
                float t0[kMaxRps], t1[kMaxRps];
#pragma unroll
                for (int r = 0; r < kMaxRps; ++r) t0[r] = t1[r] = 0.f;
                uint32_t xr = xbase;
                for (int ph = 0; ph < nphr; ++ph, xr += xstep) {
                    const bool mine = jg < min(gps, Gr - ph * gps);
                    if (ok) ok = mbar_wait(&full[slot], par, p.status);
                    if (mine && ok) {
                        const uint32_t a = static_cast<uint32_t>(slot) * stage_bytes + aoff;
                        const float bs = bsc[(ph * gps + jg) * 8 + 2 * t + (ODD ? 1 : 0)];
                        if (nr == 3) task<ODD, 3>(smem, a, rstride, xr, bs, t0, t1);
                        else if (nr == 2) task<ODD, 2>(smem, a, rstride, xr, bs, t0, t1);
                        else task<ODD, 1>(smem, a, rstride, xr, bs, t0, t1);
                    }
                    __syncwarp();
                    if (lane == 0) gemv_mma::mbar_arrive(&empty[slot]);
                    ++s;
                    if (++slot == ns) {
                        slot = 0;
                        par ^= 1u;
                    }
                }
                // rows g and g + 8 of the stage's row blocks: sum the quad's four blocks, one
                // value per (row, warp)
#pragma unroll
                for (int r = 0; r < kMaxRps; ++r) {
                    t0[r] += __shfl_xor_sync(0xffffffffu, t0[r], 1);
                    t1[r] += __shfl_xor_sync(0xffffffffu, t1[r], 1);
                    t0[r] += __shfl_xor_sync(0xffffffffu, t0[r], 2);
                    t1[r] += __shfl_xor_sync(0xffffffffu, t1[r], 2);
                }
                if (t == 0) {
#pragma unroll
                    for (int r = 0; r < kMaxRps; ++r) {
                        if (r < nr) {
                            const int rb = v * rps + r;
                            red[(rb * kUnitRows + g) * ncw + warp] = t0[r];
                            red[(rb * kUnitRows + g + 8) * ncw + warp] = t1[r];
                        }
                    }
                }
            }
            gemv_mma::consumer_sync(nct);   // every partial sum of the pass written
            const int rows_in_pass = nrb * kUnitRows;
            if constexpr (KS > 1) {
                // this CTA's sums over its K range per row, into the (now idle) records; the
                // cluster then adds its ks ranges in rank order
                float* part = reinterpret_cast<float*>(smem + p.xf_off);
                for (int row = tid; row < rows_in_pass; row += nct) {
                    float v = 0.f;
                    for (int w = 0; w < ncw; ++w) v += red[row * ncw + w];
                    part[row] = v;
                }
                cluster_sync_all();
                const int nout = nrb / NMAT * kUnitRows;   // output rows of the pass
                const int chunk = (nout + ks - 1) / ks;
                for (int oi = rank * chunk + tid; oi < min(nout, (rank + 1) * chunk); oi += nct) {
                    const int u = oi / kUnitRows, r16 = oi - u * kUnitRows;
                    const int64_t n = static_cast<int64_t>(ub + u) * kUnitRows + r16;
                    if (n >= p.N) continue;
                    const int row = (u * NMAT) * kUnitRows + r16;
                    float v = 0.f, uv = 0.f;
                    for (int r = 0; r < ks; ++r) v += ld_cluster_f32(part + row, static_cast<uint32_t>(r));
                    if (NMAT == 2)
                        for (int r = 0; r < ks; ++r) uv += ld_cluster_f32(part + row + kUnitRows, static_cast<uint32_t>(r));
                    const float cs = out;
                    v *= cs;
                    if (NMAT == 1) {
                        if (p.residual) v += p.residual[n];
                    } else {
                        v = gemv_mma::act_fn(v, p.act) * (uv * cs);
                    }
                    p.y[n] = v;
                }
                cluster_sync_all();   // the peers have read this CTA's sums
            } else {
                for (int row = tid; row < rows_in_pass; row += nct) {
                    const int rb = row / kUnitRows, r16 = row - rb * kUnitRows;
                    if (NMAT == 2 && (rb & 1)) continue;
                    const int64_t n = static_cast<int64_t>(ub + rb / NMAT) * kUnitRows + r16;
                    if (n >= p.N) continue;
                    float v = 0.f;
                    for (int w = 0; w < ncw; ++w) v += red[row * ncw + w];
                    v *= out;
                    if (NMAT == 1) {
                        if (p.residual) v += p.residual[n];
                    } else {
                        float uv = 0.f;
                        for (int w = 0; w < ncw; ++w) uv += red[(row + kUnitRows) * ncw + w];
                        v = gemv_mma::act_fn(v, p.act) * (uv * out);
                    }
                    p.y[n] = v;
                }
            }
        }
    };
    if (odd) run(std::true_type{});
    else run(std::false_type{});
    if (!ok) atomicOr(&any_failed, 1);
    gemv_mma::consumer_sync(nct);
    if (any_failed && tid == 0) drain_stages(full, ns, max(0, s - ns), s - 1);
}

}  // namespace gemv_b1
}  // namespace gem
