// gem_gemv_bn.cuh — Q4_0 GEMV for 2..32 activation rows on mma.sync, with the activations
// converted once per call into mma operand records (not once per CTA).  2..8 rows are the
// batched-decode form; 9..32 rows (column tiles of 8 activation rows, NT = 2 or 4) the batched
// prefill GEMM, where each weight is reused by up to 32 rows.
//
// act_prep_kernel turns x (optionally RMSNorm-weighted: gamma * x, the 1/rms factor being applied
// to the output) into binary16 hi + lo operand records in global memory, with one power of two per
// row that takes its largest magnitude to [2^13, 2^14).  The GEMV kernel then walks K phase by
// phase: at the start of a phase each consumer warp takes its half group's operands (32 registers)
// from a record buffer in shared memory and keeps them for every row block of the phase; the
// producer bulk-copies the next phase's records into the buffer as soon as every warp has taken
// its operands (long before they are needed), and streams weights through the usual TMA ring.
//
// MMA mapping (m16n8k16, f16 x f16 -> f32): A = 16 weight rows x 16 codes of one block (low
// nibbles: k-tile 0, high nibbles: k-tile 1), B = the same 16 codes' activations x 8 columns (the
// activation rows, hi and lo parts in two separate mma), so D[row][b] of one block is scaled by
// the row's block scale d before it is summed.  With NT column tiles (8 activation rows each) a
// block's dequantised A fragments serve NT x 4 mma, and each warp owns 4 / NT of its half
// group's blocks, so its operand registers stay at 32 whatever the row count.  A half group is the 4 even or the 4 odd blocks of
// a 256-weight group (as in the one-row kernel): odd blocks give each lane an aligned code word,
// even ones one byte permute of two words.
//
// Reference: "Q4_0 dequant-matvec" (GGML block: fp16 d, 16 bytes of codes, value (q - 8) * d).
#pragma once

#include <cuda_fp16.h>

#include "gem_gemv_b1.cuh"

namespace gem {
namespace gemv_bn {

using gemv_mma::kBoxBytes;
using gemv_mma::kGroupBytes;
using gemv_mma::kMaxSlots;
using gemv_mma::kUnitRows;

constexpr int kMaxConsumerWarps = 18;
constexpr int kMaxThreads = (kMaxConsumerWarps + 1) * 32;
constexpr int kEntryBytes = 32;                    // one lane's hi (16 B) and lo (16 B) operands of one block
constexpr int kHgBytes = 4 * 32 * kEntryBytes;     // one half group: 4 blocks x 32 lanes
constexpr int kPrepThreads = 256;

// Records: [hg][j][ct][lane][hi uint4, lo uint4]; lane (g, t) = activation row 8 ct + g, k-slot t.  For block
// 2j + (hg & 1) of group hg / 2, register r of k-tile tau holds the two elements whose codes sit in
// bytes r and r + 2 of code word t (nibble tau): the operand layout the weights' A fragments meet.
// rowinfo[b] = {2^e_b, 2^-e_b (* 1/rms of row b when gamma is given)}.
constexpr int kMaxRows = 32;
struct PrepParams {
    const float* x;
    int64_t ldx;
    const float* gamma;
    float eps;
    int G;
    int B;
    int nt;              // column tiles of 8 activation rows in the record layout
    int nchunk;          // CTAs per activation row
    uint8_t* rec;
    float2* rowinfo;
    unsigned* clear;     // words zeroed after the wait (see GemvOp)
    int nclear;
};

__global__ void __launch_bounds__(kPrepThreads) act_prep_kernel(const PrepParams p) {
    pdl_wait_trigger();
    clear_words(p.clear, p.nclear, static_cast<int>(threadIdx.x), kPrepThreads);
    __shared__ float red_m[kPrepThreads / 32], red_s[kPrepThreads / 32];
    __shared__ float sc_sh;
    const int b = blockIdx.y, chunk = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = p.G * 256;
    const float* xr = p.x + b * p.ldx;
    float mx = 0.f, ss = 0.f;
    for (int i = tid; i < K / 4; i += kPrepThreads) {
        float4 v = __ldg(reinterpret_cast<const float4*>(xr) + i);
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        if (p.gamma) {
            const float4 gm = __ldg(reinterpret_cast<const float4*>(p.gamma) + i);
            v.x *= gm.x; v.y *= gm.y; v.z *= gm.z; v.w *= gm.w;
        }
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    mx = warp_max(mx);
    ss = warp_sum(ss);
    if (lane == 0) {
        red_m[warp] = mx;
        red_s[warp] = ss;
    }
    __syncthreads();
    if (tid == 0) {
        float m = 0.f, q = 0.f;
        for (int w = 0; w < kPrepThreads / 32; ++w) {
            m = fmaxf(m, red_m[w]);
            q += red_s[w];
        }
        int e = 0;
        if (m > 0.f) e = 13 - (((__float_as_int(m) >> 23) & 0xff) - 127);
        e = max(-126, min(126, e));
        sc_sh = __int_as_float((127 + e) << 23);
        if (chunk == 0) {
            float out = __int_as_float((127 - e) << 23);
            if (p.gamma) out *= rsqrtf(q / static_cast<float>(K) + p.eps);
            p.rowinfo[b] = make_float2(__int_as_float((127 + e) << 23), out);
        }
    }
    __syncthreads();
    const float sc = sc_sh;
    // entries (hg, j, t) of row b, this CTA's contiguous share
    const int nent = 2 * p.G * 16;
    const int e0 = static_cast<int>((static_cast<int64_t>(chunk) * nent) / p.nchunk);
    const int e1 = static_cast<int>((static_cast<int64_t>(chunk + 1) * nent) / p.nchunk);
    for (int e = e0 + tid; e < e1; e += kPrepThreads) {
        const int hg = e >> 4, j = (e >> 2) & 3, t = e & 3;
        const bool odd = hg & 1;
        const int base = (hg >> 1) * 256 + (2 * j + (odd ? 1 : 0)) * 32;
        float v[8];   // tile 0: bytes 0, 2, 1, 3 of code word t; tile 1: the same + 16
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int jj = (u & 3) == 1 ? 2 : ((u & 3) == 2 ? 1 : (u & 3));
            const int k = base + gemv_b1::code_byte(odd, t, jj) + (u >> 2) * 16;
            v[u] = __ldg(xr + k) * (p.gamma ? __ldg(p.gamma + k) : 1.f) * sc;
        }
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            __half h0, l0, h1, l1;
            split_hi_lo(v[2 * r], h0, l0);
            split_hi_lo(v[2 * r + 1], h1, l1);
            const __half2 hh = __halves2half2(h0, h1), ll = __halves2half2(l0, l1);
            hw[r] = *reinterpret_cast<const uint32_t*>(&hh);
            lw[r] = *reinterpret_cast<const uint32_t*>(&ll);
        }
        const size_t ent = (static_cast<size_t>(hg * 4 + j) * p.nt + (b >> 3)) * 32 + ((b & 7) * 4 + t);
        uint4* dst = reinterpret_cast<uint4*>(p.rec + ent * kEntryBytes);
        dst[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        dst[1] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
}

struct Params {
    int64_t N;
    int G;
    int B;
    float* y;
    int64_t ldy;
    const float* residual;
    int64_t ldr;
    const uint8_t* rec;
    const float2* rowinfo;
    int act;
    int U, up, gps, nphase, ns, ncw, rps;
    int ks;              // K split: CTAs of a ks-CTA cluster take K ranges of the same units (1: none)
    uint32_t stage_bytes, full_off, empty_off, rfull_off, rempty_off, xf_off, red_off;
    int* status;
};

// One task: blocks j0 .. j0 + BPW - 1 of my half group in rows g and g + 8 of one row block, all
// NT column tiles.  a = shared offset of row g, group jg, plus 16 for odd blocks; acc += d * D.
template <bool ODD, int BPW, int NT>
__device__ __forceinline__ void task_bn(const uint8_t* smem, uint32_t a, int j0, int t, uint32_t sel,
                                        const uint4 (&xh)[BPW][NT], const uint4 (&xl)[BPW][NT],
                                        float (&acc)[NT][4]) {
#pragma unroll
    for (int jj = 0; jj < BPW; ++jj) {
        const int j = j0 + jj;
        uint32_t w[2];
        float dsc[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint8_t* rg = smem + a + h * 8 * kGroupBytes + 36 * j;
            const uint32_t d0 = *reinterpret_cast<const uint32_t*>(rg);
            if constexpr (ODD) {
                w[h] = *reinterpret_cast<const uint32_t*>(rg + 4 + 4 * t);
                dsc[h] = __high2float(*reinterpret_cast<const __half2*>(&d0));
            } else {
                const uint32_t wa = *reinterpret_cast<const uint32_t*>(rg + 4 * t);
                const uint32_t wb = *reinterpret_cast<const uint32_t*>(rg + 16);
                w[h] = __byte_perm(wa, wb, sel);
                dsc[h] = __low2float(*reinterpret_cast<const __half2*>(&d0));
            }
        }
        uint32_t l02, l13, h02, h13, m02, m13, n02, n13;
        gemv_mma::dequant_word(w[0], l02, l13, h02, h13);
        gemv_mma::dequant_word(w[1], m02, m13, n02, n13);
#pragma unroll
        for (int ct = 0; ct < NT; ++ct) {
            float c[4] = {0.f, 0.f, 0.f, 0.f};
            mma_16816(c, l02, m02, l13, m13, xh[jj][ct].x, xh[jj][ct].y);
            mma_16816(c, h02, n02, h13, n13, xh[jj][ct].z, xh[jj][ct].w);
            mma_16816(c, l02, m02, l13, m13, xl[jj][ct].x, xl[jj][ct].y);
            mma_16816(c, h02, n02, h13, n13, xl[jj][ct].z, xl[jj][ct].w);
            acc[ct][0] = fmaf(dsc[0], c[0], acc[ct][0]);
            acc[ct][1] = fmaf(dsc[0], c[1], acc[ct][1]);
            acc[ct][2] = fmaf(dsc[1], c[2], acc[ct][2]);
            acc[ct][3] = fmaf(dsc[1], c[3], acc[ct][3]);
        }
    }
}

// The reduction area: per (row block, consumer warp, column tile) the lanes' float4 partial sums;
// (row r16 of the unit, activation row b) sits at lane (r16 & 7) * 4 + (b & 7) / 2, component
// (r16 >> 3) * 2 + (b & 1) of column tile b / 8.
template <int NT>
__device__ __forceinline__ int red_index(int rb, int w, int ncw, int r16, int b) {
    const int ct = b >> 3, gb = b & 7;
    return ((((rb * ncw + w) * NT + ct) * 32 + (r16 & 7) * 4 + (gb >> 1)) * 4) + (r16 >> 3) * 2 + (gb & 1);
}

using gemv_b1::cluster_sync_all;
using gemv_b1::ld_cluster_f32;

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

template <int NMAT, int NT>
__global__ void __launch_bounds__(kMaxThreads, 1) q4_0_gemv_bn_kernel(const __grid_constant__ CUtensorMap tm0,
                                                                      const __grid_constant__ CUtensorMap tm1,
                                                                      const Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.full_off);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + p.empty_off);
    uint64_t* rfull = reinterpret_cast<uint64_t*>(smem + p.rfull_off);
    uint64_t* rempty = reinterpret_cast<uint64_t*>(smem + p.rempty_off);
    float* red = reinterpret_cast<float*>(smem + p.red_off);   // [rb][warp][ct][lane][4]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ncw = p.ncw, nct = ncw * 32;
    const int gps = p.gps, ns = p.ns, rps = p.rps;
    const uint32_t stage_bytes = p.stage_bytes;
    const uint32_t rstride = static_cast<uint32_t>(gps * kBoxBytes);
    const uint32_t rec_phase = static_cast<uint32_t>(2 * gps * kHgBytes * NT);   // one record buffer
    // K split: cluster cid (of ncl) owns a unit range; its CTA `rank` owns groups [gk0, gk0 + Gr)
    const int ks = p.ks, rank = static_cast<int>(blockIdx.x) % ks, cid = static_cast<int>(blockIdx.x) / ks;
    const int ncl = static_cast<int>(gridDim.x) / ks;
    const int gk0 = rank * p.G / ks, Gr = (rank + 1) * p.G / ks - gk0;
    const int nphr = (Gr + gps - 1) / gps;   // this CTA's phases
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
        mbar_init(rfull, 1);
        mbar_init(rempty, ncw);
        fence_mbar_init();
        prefetch_tensormap(&tm0);
        if (NMAT == 2) prefetch_tensormap(&tm1);
    }
    __syncthreads();

    // ---------------- producer warp ----------------
    // Order: (pass, phase, row-block tuple).  Each phase's records go out before its weight
    // stages; the first stages of the first phase go out before griddepcontrol.wait (the weights
    // are not written by earlier kernels, the records are).
    if (warp == ncw) {
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_first();
            bool ok = true;
            int s = 0, slot = 0;
            uint32_t par = 1;
            int pre = 0;   // stages issued before the wait
            auto issue = [&](int pass, int ph, int v) -> bool {
                const int ub = u0 + pass * p.up;
                const int nrb = min(p.up, u1 - ub) * NMAT;
                const int nr = min(rps, nrb - v * rps);
                const int g0 = ph * gps;
                const int ng = min(gps, Gr - g0);
                if (s >= ns && !mbar_wait(&empty[slot], par, p.status)) return false;
                uint8_t* dst = smem + static_cast<size_t>(slot) * stage_bytes;
                mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(nr * ng * kBoxBytes));
                for (int r = 0; r < nr; ++r) {
                    const int rb = v * rps + r;
                    const int row0 = (ub + rb / NMAT) * kUnitRows;
                    const CUtensorMap* tm = (NMAT == 2 && (rb & 1)) ? &tm1 : &tm0;
                    for (int j = 0; j < ng; ++j)
                        tma_load_2d(dst + r * rstride + j * kBoxBytes, tm, (gk0 + g0 + j) * kGroupBytes, row0,
                                    &full[slot], policy);
                }
                ++s;
                if (++slot == ns) {
                    slot = 0;
                    par ^= 1u;
                }
                return true;
            };
            {
                const int nrb0 = min(p.up, u1 - u0) * NMAT;
                const int nv0 = (nrb0 + rps - 1) / rps;
                for (int v = 0; v < nv0 && pre < ns; ++v, ++pre) (void)issue(0, 0, v);
            }
            pdl_wait();
            int q = 0;
            for (int pass = 0; pass < npass && ok; ++pass) {
                const int ub = u0 + pass * p.up;
                const int nrb = min(p.up, u1 - ub) * NMAT;
                const int nv = (nrb + rps - 1) / rps;
                for (int ph = 0; ph < nphr && ok; ++ph, ++q) {
                    // the buffer is free once every warp holds phase q - 1's operands
                    if (q >= 1 && !(ok = mbar_wait(rempty, (q - 1) & 1, p.status))) break;
                    const int ng = min(gps, Gr - ph * gps);
                    const uint32_t bytes = static_cast<uint32_t>(2 * ng * kHgBytes * NT);
                    mbar_arrive_expect_tx(rfull, bytes);
                    bulk_load(smem + p.xf_off,
                              p.rec + static_cast<size_t>(2 * gk0) * kHgBytes * NT + static_cast<size_t>(ph) * rec_phase,
                              bytes, rfull);
                    for (int v = (q == 0 ? pre : 0); v < nv && ok; ++v) ok = issue(pass, ph, v);
                }
            }
            if (!ok) drain_stages(full, ns, max(0, s - ns), s - 1);
        }
        // the producer warp never triggers dependents: the consumers do, after their wait
        __syncwarp();
        if (ks > 1) {   // the consumers' combine: two cluster barriers per pass (one pass)
            for (int i = 0; i < 2 * npass; ++i) cluster_sync_all();
        }
        return;
    }

    // ---------------- consumer warps ----------------
    pdl_wait_trigger();   // row scales (and the residual) come from earlier kernels

    constexpr int BPW = 4 / NT;   // blocks of the half group per warp
    const int g = lane >> 2, t = lane & 3;
    const int hgl = warp / NT, j0 = (warp % NT) * BPW;   // half group of the phase, first block
    const int jg = hgl >> 1;
    const bool odd = hgl & 1;
    const uint32_t aoff = static_cast<uint32_t>(jg * kBoxBytes + g * kGroupBytes + (odd ? 16 : 0));
    const uint32_t sel = t == 0 ? 0x3254u : 0x3210u;   // even blocks: word 0 joins the two tails

    bool ok = true;
    int s = 0, slot = 0;
    uint32_t par = 0;
    auto run = [&](auto odd_tag) {
        constexpr bool ODD = decltype(odd_tag)::value;
        int q = 0;
        for (int pass = 0; pass < npass; ++pass) {
            const int ub = u0 + pass * p.up;
            const int nrb = min(p.up, u1 - ub) * NMAT;
            const int nv = (nrb + rps - 1) / rps;
            gemv_mma::consumer_sync(nct);   // the previous pass has read `red`
            for (int ph = 0; ph < nphr; ++ph, ++q) {
                const bool mine = jg < min(gps, Gr - ph * gps);
                if (ok) ok = mbar_wait(rfull, q & 1, p.status);
                uint4 xh[BPW][NT], xl[BPW][NT];
#pragma unroll
                for (int jj = 0; jj < BPW; ++jj)
#pragma unroll
                    for (int ct = 0; ct < NT; ++ct) {
                        xh[jj][ct] = xl[jj][ct] = make_uint4(0u, 0u, 0u, 0u);
                        if (mine && ok && ct * 8 + g < p.B) {   // activation row 8 ct + g exists
                            const uint4* e = reinterpret_cast<const uint4*>(
                                smem + p.xf_off + (((hgl * 4 + j0 + jj) * NT + ct) * 32 + lane) * kEntryBytes);
                            xh[jj][ct] = e[0];
                            xl[jj][ct] = e[1];
                        }
                    }
                // The next bulk copy into the buffer (async proxy) may follow the arrive at once:
                // order my reads of it (generic proxy) before that write.
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) gemv_mma::mbar_arrive(rempty);   // operands now in registers
                for (int v = 0; v < nv; ++v) {
                    if (ok) ok = mbar_wait(&full[slot], par, p.status);
                    if (mine && ok) {
                        const int nr = min(rps, nrb - v * rps);
                        for (int r = 0; r < nr; ++r) {
                            float acc[NT][4];
#pragma unroll
                            for (int ct = 0; ct < NT; ++ct) acc[ct][0] = acc[ct][1] = acc[ct][2] = acc[ct][3] = 0.f;
                            task_bn<ODD, BPW, NT>(smem, static_cast<uint32_t>(slot) * stage_bytes + r * rstride + aoff,
                                                  j0, t, sel, xh, xl, acc);
#pragma unroll
                            for (int ct = 0; ct < NT; ++ct) {
                                float4* rr = reinterpret_cast<float4*>(red) + (((v * rps + r) * ncw + warp) * NT + ct) * 32 + lane;
                                if (ph) {
                                    const float4 o = *rr;
                                    acc[ct][0] += o.x; acc[ct][1] += o.y; acc[ct][2] += o.z; acc[ct][3] += o.w;
                                }
                                *rr = make_float4(acc[ct][0], acc[ct][1], acc[ct][2], acc[ct][3]);
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) gemv_mma::mbar_arrive(&empty[slot]);
                    ++s;
                    if (++slot == ns) {
                        slot = 0;
                        par ^= 1u;
                    }
                }
            }
            gemv_mma::consumer_sync(nct);   // every partial sum of the pass written
            const int B = p.B;
            const int items = nrb * kUnitRows * B;
            if (ks > 1) {
                // this CTA's sums over its K range, per (row block, row, activation row), into the
                // (now idle) record buffer; the cluster then adds its ks ranges in rank order
                float* part = reinterpret_cast<float*>(smem + p.xf_off);
                for (int idx = tid; idx < items; idx += nct) {
                    const int rb = idx / (kUnitRows * B), rem = idx - rb * (kUnitRows * B);
                    const int r16 = rem / B, b = rem - r16 * B;
                    float v = 0.f;
                    for (int w = 0; w < ncw; ++w) v += red[red_index<NT>(rb, w, ncw, r16, b)];
                    part[idx] = v;
                }
                cluster_sync_all();
                const int nout = nrb / NMAT * kUnitRows * B;   // outputs (unit row, activation row)
                const int chunk = (nout + ks - 1) / ks;
                for (int oi = rank * chunk + tid; oi < min(nout, (rank + 1) * chunk); oi += nct) {
                    const int u = oi / (kUnitRows * B), rem = oi - u * (kUnitRows * B);
                    const int r16 = rem / B, b = rem - r16 * B;
                    const int64_t n = static_cast<int64_t>(ub + u) * kUnitRows + r16;
                    if (n >= p.N) continue;
                    const int ig = ((u * NMAT) * kUnitRows + r16) * B + b;
                    float v = 0.f, uv = 0.f;
                    for (int r = 0; r < ks; ++r) v += ld_cluster_f32(part + ig, static_cast<uint32_t>(r));
                    if (NMAT == 2)
                        for (int r = 0; r < ks; ++r)
                            uv += ld_cluster_f32(part + ig + kUnitRows * B, static_cast<uint32_t>(r));
                    const float out = p.rowinfo[b].y;
                    v *= out;
                    if (NMAT == 1) {
                        if (p.residual) v += p.residual[b * p.ldr + n];
                    } else {
                        v = gemv_mma::act_fn(v, p.act) * (uv * out);
                    }
                    p.y[b * p.ldy + n] = v;
                }
                cluster_sync_all();   // the peers have read this CTA's sums
                continue;
            }
            for (int idx = tid; idx < items; idx += nct) {
                const int rb = idx / (kUnitRows * B), rem = idx - rb * (kUnitRows * B);
                const int r16 = rem / B, b = rem - r16 * B;
                if (NMAT == 2 && (rb & 1)) continue;
                const int64_t n = static_cast<int64_t>(ub + rb / NMAT) * kUnitRows + r16;
                if (n >= p.N) continue;
                float v = 0.f;
                for (int w = 0; w < ncw; ++w) v += red[red_index<NT>(rb, w, ncw, r16, b)];
                const float out = p.rowinfo[b].y;
                v *= out;
                if (NMAT == 1) {
                    if (p.residual) v += p.residual[b * p.ldr + n];
                } else {
                    float uv = 0.f;
                    for (int w = 0; w < ncw; ++w) uv += red[red_index<NT>(rb + 1, w, ncw, r16, b)];
                    v = gemv_mma::act_fn(v, p.act) * (uv * out);
                }
                p.y[b * p.ldy + n] = v;
            }
        }
    };
    if (odd) run(std::true_type{});
    else run(std::false_type{});
    if (!ok) atomicOr(&any_failed, 1);
    gemv_mma::consumer_sync(nct);
    if (any_failed && tid == 0) drain_stages(full, ns, max(0, s - ns), s - 1);
}

}  // namespace gemv_bn
}  // namespace gem
