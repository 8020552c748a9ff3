// gem_attn.cu — grouped-query decode attention over a binary16 KV cache.
//
// GELO LLM generation, sections 02/05: at decode one query per head attends the
// n_cache + 1 cached positions; G = n_q / n_kv query heads share each KV head; a sliding
// window keeps the last W positions (here a ring of W slots).  "gem" research record,
// decode-attention notes: attention states over disjoint token ranges compose, and the
// partial results are merged in ascending partition order.
//
// Schedule.  Grid = (split, kv head, sequence).  The attended slots form the prefix
// [0, T) of the cache (T = p + 1, or min(W, p + 1) for a ring), cut into tiles of TP slots
// and split into contiguous tile ranges.  A CTA streams its K tiles and then its V tiles
// through one ring of shared-memory stages with TMA (2-D map over [B*n_kv*cap][d]
// binary16, boxes of TP rows x 64 elements, 128-byte swizzle so ldmatrix is conflict-free).
// When launched inside the layer chain, the tiles are requested before
// griddepcontrol.wait.  That is safe under the library's launch rule (gem_device.cuh): the
// kernel two or more launches back (e.g. the previous step's append of this layer) has
// completed by then, and of the cache only the new token's slot can be written by the
// immediately preceding kernel; that one row is re-read (or, fused, produced) after the wait.
//
// Arithmetic.  Scores S = (scale q) K^T and the value sum P V run on mma.sync m16n8k16
// (binary16 inputs, fp32 accumulate).  K and V are binary16 already (exact operands); q
// and the probabilities are fp32 and enter as hi + lo binary16 pairs in rows h and h + 8
// of the 16-row A operand (G <= 8 heads per KV head), so products keep ~22 bits.  The
// split's softmax is exact (max over the split first, then exponentials); the split
// writes (max, denominator, unnormalised output) and a merge kernel combines splits in
// ascending order.  A split that has the whole range writes the final output directly.
#include <algorithm>
#include <cmath>
#include <map>
#include <mutex>
#include <tuple>

#include "gem_device.cuh"

namespace gem {
namespace {

constexpr int kAttnThreads = 128;
constexpr int kMaxSplitSlots = 1024;   // slots one CTA may own (scores kept in shared memory)

struct AttnParams {
    const float* q;
    int64_t ldq;
    int B, n_q, n_kv, G;
    int64_t cap;
    int window;
    float scale;
    const int32_t* pos;
    float* out;
    int64_t ldo;
    float* part;          // [B][n_q][nsplit_max][D + 2]
    int nsplit_max;
    int tp;               // slots per tile
    int ltile;            // max tiles per split
    int ns;               // ring stages
    int early;            // positions and tiles may be read before griddepcontrol.wait
    const uint16_t* k_cache;
    const uint16_t* v_cache;
    uint32_t tile_bytes, bar_off, qa_off, sc_off, pa_off, st_off;
    int* status;
    // fused QK-norm / RoPE / append (flash kernel only): q rows are the raw projections
    int fuse;
    const float *g_q, *g_k;
    float eps;
    int rope_dim, v_mode;
    uint16_t *k_out, *v_out;
    // flash kernel: one arrival counter per (sequence, KV head) in the workspace, zero between
    // calls (the CTA that merges resets it)
    unsigned* cnt;
    // compact cache (V rows only): rebuilt-K buffers, offset table and tile anchors
    uint32_t kr_off, tb_off, an_off;
};

__host__ __device__ __forceinline__ int tile_slots(int d) { return d <= 64 ? 128 : (d <= 128 ? 64 : 32); }

__device__ __forceinline__ void split_range(int T, int tp, int nsplit_max, int s, int& nsplit, int& t0, int& t1) {
    const int nt = (T + tp - 1) / tp;
    nsplit = min(nsplit_max, nt);
    t0 = static_cast<int>((static_cast<int64_t>(s) * nt) / nsplit);
    t1 = static_cast<int>((static_cast<int64_t>(s + 1) * nt) / nsplit);
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1) gqa_split_kernel(const __grid_constant__ CUtensorMap tmK,
                                                                 const __grid_constant__ CUtensorMap tmV,
                                                                 const AttnParams P) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 128-byte-swizzled TMA tiles need a 1024-byte aligned base (the host adds the slack)
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P.bar_off);
    __half* qa = reinterpret_cast<__half*>(smem + P.qa_off);   // [16][D + 8]
    float* sc = reinterpret_cast<float*>(smem + P.sc_off);     // [G][L]
    __half* pa = reinterpret_cast<__half*>(smem + P.pa_off);   // [16][L + 8]
    float* st = reinterpret_cast<float*>(smem + P.st_off);     // [8][2]: max, denominator
    __shared__ int abort_flag;

    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int TP = P.tp;
    const int L = P.ltile * TP;       // score row length
    const int QA = D + 8, PA = L + 8;  // padded row pitches (elements)

    if (!P.early) pdl_wait_trigger();
    const int p = P.pos[b];
    const bool bad = p < 0 || (P.window == 0 && static_cast<int64_t>(p) >= P.cap);
    if (bad) {  // every CTA waits before leaving, so completion of this grid implies its predecessor's
        if (P.early) pdl_wait_trigger();
        if (t == 0 && split == 0 && g == 0) atomicOr(P.status, GEM_DEVFLAG_POS_RANGE);
        return;
    }
    const int T = P.window ? min(P.window, p + 1) : p + 1;
    int nsplit, t0, t1;
    split_range(T, TP, P.nsplit_max, split, nsplit, t0, t1);
    if (split >= nsplit) {
        if (P.early) pdl_wait_trigger();
        return;
    }
    const int ntile = t1 - t0;
    const int nseq = 2 * ntile;                  // K tiles, then V tiles
    const int slot_p = P.window ? p % P.window : p;
    const int64_t row0 = (static_cast<int64_t>(b) * P.n_kv + g) * P.cap;
    int npre = 0;

    if (t == 0) {
        abort_flag = 0;
        for (int i = 0; i < P.ns; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
    }
    __syncthreads();
    uint64_t policy = 0;
    auto issue = [&](int i) {
        const int tile = t0 + (i < ntile ? i : i - ntile);
        const CUtensorMap* tm = i < ntile ? &tmK : &tmV;
        const int slot = i % P.ns;
        uint8_t* dst = smem + static_cast<size_t>(slot) * P.tile_bytes;
        fence_proxy_async_smem();  // generic writes to this slot (row refresh, zeroing) precede the TMA
        mbar_arrive_expect_tx(&bars[slot], P.tile_bytes);
        for (int j = 0; j < D / 64; ++j)
            tma_load_2d(dst + j * TP * 128, tm, j * 64, static_cast<int32_t>(row0 + static_cast<int64_t>(tile) * TP),
                        &bars[slot], policy);
    };
    if (t == 0) {
        policy = l2_policy_evict_first();
        npre = min(P.ns, nseq);
        for (int i = 0; i < npre; ++i) issue(i);
    }
    __shared__ int s_npre;
    if (t == 0) s_npre = npre;
    if (P.early) pdl_wait_trigger();

    // q of this KV head's G query heads -> A operand rows (hi in rows 0..7, lo in 8..15).
    // All loads of a thread are issued before any is used: one L2 round trip in total.
    {
        constexpr int kMaxF4 = 8 * D / 4 / kAttnThreads;  // float4 slots per thread (G <= 8)
        const int nf4 = P.G * D / 4;
        const float4* qsrc = reinterpret_cast<const float4*>(P.q + b * P.ldq + static_cast<int64_t>(g) * P.G * D);
        float4 qv[kMaxF4];
#pragma unroll
        for (int i = 0; i < kMaxF4; ++i) {
            const int f = t + i * kAttnThreads;
            qv[i] = f < nf4 ? qsrc[f] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < kMaxF4; ++i) {
            const int f = t + i * kAttnThreads;
            if (f < nf4) {
                const int h = (f * 4) / D, col = (f * 4) % D;
                const float v[4] = {qv[i].x * P.scale, qv[i].y * P.scale, qv[i].z * P.scale, qv[i].w * P.scale};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    __half hi, lo;
                    split_hi_lo(v[j], hi, lo);
                    qa[h * QA + col + j] = hi;
                    qa[(h + 8) * QA + col + j] = lo;
                }
            }
        }
        for (int e = P.G * D + t; e < 8 * D; e += kAttnThreads) {  // unused head rows
            qa[(e / D) * QA + e % D] = __float2half_rn(0.f);
            qa[(e / D + 8) * QA + e % D] = __float2half_rn(0.f);
        }
    }
    __syncthreads();
    const int pre = s_npre;

    // refresh the new token's row in a tile that was requested before the wait
    auto patch = [&](int i, uint8_t* tile) {
        const int tl = t0 + (i < ntile ? i : i - ntile);
        const int r = slot_p - tl * TP;
        if (i < pre && r >= 0 && r < TP) {
            const uint16_t* src = (i < ntile ? P.k_cache : P.v_cache) + (row0 + slot_p) * D;
            for (int c = t * 8; c < D; c += kAttnThreads * 8)
                *reinterpret_cast<uint4*>(tile + swz(r, c, TP)) = *reinterpret_cast<const uint4*>(src + c);
        }
    };

    // ---- scores -----------------------------------------------------------------------------
    const int gq = lane >> 2, tq = lane & 3;
    // q's A fragments are the same for every position tile: keep them in registers when small
    constexpr bool kQReg = D <= 256;
    uint32_t qf[kQReg ? D / 16 : 1][4];
    if constexpr (kQReg) {
#pragma unroll
        for (int k16 = 0; k16 < D / 16; ++k16) {
            const int arow = (lane & 7) + ((lane >> 3) & 1) * 8, acol = k16 * 16 + (lane >> 4) * 8;
            ldmatrix_x4(qf[k16][0], qf[k16][1], qf[k16][2], qf[k16][3], smem_u32(qa + arow * QA + acol));
        }
    }
    for (int kt = 0; kt < ntile; ++kt) {
        const int i = kt, slot = i % P.ns;
        uint8_t* tile = smem + static_cast<size_t>(slot) * P.tile_bytes;
        if (!mbar_wait(&bars[slot], static_cast<uint32_t>((i / P.ns) & 1), P.status)) abort_flag = 1;
        patch(i, tile);
        __syncthreads();
        const uint32_t tbase = smem_u32(tile);
        for (int n8 = warp; n8 < TP / 8; n8 += 4) {
            float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k16 = 0; k16 < D / 16; ++k16) {
                uint32_t a0, a1, a2, a3, b0, b1;
                if constexpr (kQReg) {
                    a0 = qf[k16][0]; a1 = qf[k16][1]; a2 = qf[k16][2]; a3 = qf[k16][3];
                } else {
                    const int arow = (lane & 7) + ((lane >> 3) & 1) * 8, acol = k16 * 16 + (lane >> 4) * 8;
                    ldmatrix_x4(a0, a1, a2, a3, smem_u32(qa + arow * QA + acol));
                }
                const int brow = n8 * 8 + (lane & 7), bcol = k16 * 16 + ((lane >> 3) & 1) * 8;
                ldmatrix_x2(b0, b1, tbase + swz(brow, bcol, TP));
                mma_16816(c, a0, a1, a2, a3, b0, b1);
            }
            if (gq < P.G) {
                const int col = kt * TP + n8 * 8 + 2 * tq;
                const int s0 = (t0 + kt) * TP + n8 * 8 + 2 * tq;
                sc[gq * L + col] = s0 < T ? c[0] + c[2] : -INFINITY;
                sc[gq * L + col + 1] = s0 + 1 < T ? c[1] + c[3] : -INFINITY;
            }
        }
        __syncthreads();
        if (abort_flag) {  // a copy never landed: drain what is in flight and leave
            if (t == 0) drain_stages(bars, P.ns, i, min(i + P.ns - 1, nseq - 1));
            return;
        }
        if (t == 0 && i + P.ns < nseq) issue(i + P.ns);
    }

    // ---- softmax over the split (exact: max first) -------------------------------------------
    const int Ls = ntile * TP;
    for (int h = warp; h < 8; h += 4) {
        float m = -INFINITY, l = 0.f;
        if (h < P.G) {
            for (int j = lane; j < Ls; j += 32) m = fmaxf(m, sc[h * L + j]);
            m = warp_max(m);
            for (int j = lane; j < Ls; j += 32) {
                const float e = expf(sc[h * L + j] - m);
                l += e;
                __half hi, lo;
                split_hi_lo(e, hi, lo);
                pa[h * PA + j] = hi;
                pa[(h + 8) * PA + j] = lo;
            }
            l = warp_sum(l);
        } else {
            for (int j = lane; j < Ls; j += 32) {
                pa[h * PA + j] = __float2half_rn(0.f);
                pa[(h + 8) * PA + j] = __float2half_rn(0.f);
            }
        }
        if (lane == 0) {
            st[2 * h] = m;
            st[2 * h + 1] = l;
        }
    }
    __syncthreads();

    // ---- P V ---------------------------------------------------------------------------------
    constexpr int NW = D / 32;  // n8 tiles of output dims per warp
    float acc[NW][4];
#pragma unroll
    for (int n = 0; n < NW; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    for (int vt = 0; vt < ntile; ++vt) {
        const int i = ntile + vt, slot = i % P.ns;
        uint8_t* tile = smem + static_cast<size_t>(slot) * P.tile_bytes;
        if (!mbar_wait(&bars[slot], static_cast<uint32_t>((i / P.ns) & 1), P.status)) abort_flag = 1;
        patch(i, tile);
        const int valid = T - (t0 + vt) * TP;   // rows >= valid hold other slots: zero them
        if (valid < TP)
            for (int e = t * 8; e < (TP - valid) * D; e += kAttnThreads * 8) {
                const int r = valid + e / D, c = e % D;
                *reinterpret_cast<uint4*>(tile + swz(r, c, TP)) = make_uint4(0, 0, 0, 0);
            }
        __syncthreads();
        const uint32_t tbase = smem_u32(tile);
        for (int k16 = 0; k16 < TP / 16; ++k16) {
            uint32_t a0, a1, a2, a3;
            const int arow = (lane & 7) + ((lane >> 3) & 1) * 8, acol = vt * TP + k16 * 16 + (lane >> 4) * 8;
            ldmatrix_x4(a0, a1, a2, a3, smem_u32(pa + arow * PA + acol));
#pragma unroll
            for (int n = 0; n < NW; n += 2) {
                const int d0 = (warp * NW + n) * 8;
                uint32_t b0, b1, b2, b3;
                const int vrow = k16 * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int vcol = d0 + (lane >> 4) * 8;
                ldmatrix_x4_trans(b0, b1, b2, b3, tbase + swz(vrow, vcol, TP));
                mma_16816(acc[n], a0, a1, a2, a3, b0, b1);
                mma_16816(acc[n + 1], a0, a1, a2, a3, b2, b3);
            }
        }
        __syncthreads();
        if (abort_flag) {
            if (t == 0) drain_stages(bars, P.ns, i, min(i + P.ns - 1, nseq - 1));
            return;
        }
        if (t == 0 && i + P.ns < nseq) issue(i + P.ns);
    }

    // ---- output ------------------------------------------------------------------------------
    if (gq < P.G) {
        const int h = g * P.G + gq;
        const float m = st[2 * gq], l = st[2 * gq + 1];
        if (nsplit == 1) {
            float* o = P.out + b * P.ldo + static_cast<int64_t>(h) * D;
            const float inv = 1.f / l;
#pragma unroll
            for (int n = 0; n < NW; ++n) {
                const int dd = (warp * NW + n) * 8 + 2 * tq;
                o[dd] = (acc[n][0] + acc[n][2]) * inv;
                o[dd + 1] = (acc[n][1] + acc[n][3]) * inv;
            }
        } else {
            float* o = P.part + ((static_cast<int64_t>(b) * P.n_q + h) * P.nsplit_max + split) * (D + 2);
#pragma unroll
            for (int n = 0; n < NW; ++n) {
                const int dd = (warp * NW + n) * 8 + 2 * tq;
                o[dd] = acc[n][0] + acc[n][2];
                o[dd + 1] = acc[n][1] + acc[n][3];
            }
            if (warp == 0 && tq == 0) {
                o[D] = m;
                o[D + 1] = l;
            }
        }
    }
}

// ---- per-warp flash variant (d <= 256, G <= 4) -------------------------------------------
// Each of the CTA's W warps owns every W-th 16-slot tile of the split and streams its K and V
// tiles through a private 2-stage TMA ring.  The grid holds about as many CTAs as the SMs can
// keep resident at once, so a split is a few tiles per warp and most of them are in flight
// before the first is consumed (inside the layer chain they are requested before
// griddepcontrol.wait).  Per tile: S^T = K Q^T on mma (positions are the M rows; the N
// columns are (head, hi/lo) pairs of the pre-scaled query), an online softmax per head held
// in registers (head t lives in lane quad position t), P^T through a 384-byte per-warp
// buffer, and O^T += V^T P^T on mma (head t's hi and lo columns land in the same thread and
// are summed at the end).  The W warps' states are merged once per CTA (ascending warp
// order).  A split then writes its (max, denominator, unnormalised output) to the workspace.
// Inside the layer chain it takes a ticket from its (sequence, KV head) arrival counter; the
// CTA that takes the last ticket combines every split in ascending split order (so the result
// does not depend on which CTA arrives last), writes the output and sets the counter back to
// zero.  A stand-alone call has no cleared counters: the ordered merge kernel combines the
// splits in a second launch.
constexpr int kFlashTile = 16;
constexpr int kFlashStages = 2;
constexpr int kPbufPitch = 24;        // halves per P^T row (16 used; padding avoids bank conflicts)
constexpr int kMaxFlashSplits = 64;   // splits of one (sequence, KV head) at most

template <int D, int W>
__global__ void __launch_bounds__(W * 32, 1) gqa_flash_kernel(const __grid_constant__ CUtensorMap tmK,
                                                               const __grid_constant__ CUtensorMap tmV,
                                                               const AttnParams P,
                                                               const __grid_constant__ RopeFreq fr) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    constexpr int kNT = W * 32;
    constexpr int kTileBytes = kFlashTile * D * 2;            // one K or V tile
    constexpr int kStageBytes = 2 * kTileBytes;               // K + V
    constexpr int kWarpRing = kFlashStages * kStageBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + W * kWarpRing);                   // [warp][stage]
    __half* pbuf = reinterpret_cast<__half*>(smem + W * kWarpRing + 128);                 // [warp][8][24]
    float* comb = reinterpret_cast<float*>(smem);             // reuses the ring after the tile loop
    // fused path: rotated query heads [4][D], cos / sin of the rotated pairs, new K / V rows
    float* qs = reinterpret_cast<float*>(smem + W * kWarpRing + 128 + W * 8 * kPbufPitch * 2);
    float* kbuf = qs + 4 * D;
    float* cs = kbuf + D;
    float* sn = cs + D / 2;
    uint16_t* knew = reinterpret_cast<uint16_t*>(sn + D / 2);
    uint16_t* vnew = knew + D;
    __shared__ int last_sh;

    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int t_id = threadIdx.x, lane = t_id & 31, warp = t_id >> 5;
    const int gq = lane >> 2, tq = lane & 3;
    const int G = P.G;

    if (!P.early) pdl_wait_trigger();
    const int p = P.pos[b];
    const bool bad = p < 0 || (P.window == 0 && static_cast<int64_t>(p) >= P.cap);
    if (bad) {
        if (P.early) pdl_wait_trigger();
        if (t_id == 0 && split == 0 && g == 0) atomicOr(P.status, GEM_DEVFLAG_POS_RANGE);
        return;
    }
    const int T = P.window ? min(P.window, p + 1) : p + 1;
    int nsplit, t0, t1;
    split_range(T, kFlashTile, P.nsplit_max, split, nsplit, t0, t1);
    if (split >= nsplit) {   // no tiles in this split (short prefix)
        if (P.early) pdl_wait_trigger();
        return;
    }
    const int ntile = t1 - t0;
    const int nmy = ntile > warp ? (ntile - warp + W - 1) / W : 0;  // my tiles
    const int slot_p = P.window ? p % P.window : p;
    const int64_t row0 = (static_cast<int64_t>(b) * P.n_kv + g) * P.cap;
    uint8_t* ring = smem + warp * kWarpRing;
    uint64_t* wbar = bars + warp * kFlashStages;

    if (lane == 0)
        for (int i = 0; i < kFlashStages; ++i) mbar_init(&wbar[i], 1);
    fence_mbar_init();
    __syncwarp();
    const uint64_t policy = l2_policy_evict_first();
    auto issue = [&](int it) {  // my it-th tile into stage it % kFlashStages (lane 0)
        const int tile = t0 + warp + it * W;
        const int st = it % kFlashStages;
        uint8_t* dst = ring + st * kStageBytes;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&wbar[st], kStageBytes);
        const int32_t r = static_cast<int32_t>(row0 + static_cast<int64_t>(tile) * kFlashTile);
        for (int j = 0; j < D / 64; ++j) {
            tma_load_2d(dst + j * kFlashTile * 128, &tmK, j * 64, r, &wbar[st], policy);
            tma_load_2d(dst + kTileBytes + j * kFlashTile * 128, &tmV, j * 64, r, &wbar[st], policy);
        }
    };
    const int npre = min(kFlashStages, nmy);
    if (lane == 0) {
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
        for (int it = 0; it < npre; ++it) issue(it);
    }
    if (P.early) pdl_wait_trigger();

    const bool owner = slot_p >= t0 * kFlashTile && slot_p < t1 * kFlashTile;
    if (P.fuse) {
        // The raw rows a warp normalises and rotates (a query head for warps < G; the new K row
        // for warp W - 2 and the new V row for warp W - 1 of the CTA holding the new slot) are
        // loaded first, so their L2 round trip overlaps the rotation table.
        const int R = P.rope_dim, half = R / 2;
        const float* qrow0 = P.q + b * P.ldq;
        const float* krow = qrow0 + static_cast<int64_t>(P.n_q + g) * D;
        const float* vsrc = P.v_mode == 1 ? krow : qrow0 + static_cast<int64_t>(P.n_q + P.n_kv + g) * D;
        const bool has_q = warp < G;
        const bool has_k = owner && warp == W - 2, has_v = owner && warp == W - 1;
        float rq[D / 32], rkv[D / 32];
#pragma unroll
        for (int k = 0; k < D / 32; ++k) {
            rq[k] = has_q ? qrow0[static_cast<int64_t>(g * G + warp) * D + lane + 32 * k] : 0.f;
            rkv[k] = has_k ? krow[lane + 32 * k] : (has_v ? vsrc[lane + 32 * k] : 0.f);
        }
        for (int i = t_id; i < half; i += kNT) {   // rotation table of position p
            float c, sv;
            rope_cos_sin(static_cast<double>(p) * fr.w[i], c, sv);
            cs[i] = c;
            sn[i] = sv;
        }
        __syncthreads();   // rotation table complete
        // QK-norm + RoPE of a raw head row held in registers (warp-wide), result in sb[0..D)
        auto rotate = [&](float (&v)[D / 32], const float* gamma, float* sb) {
            float ss = 0.f;
#pragma unroll
            for (int k = 0; k < D / 32; ++k) ss = fmaf(v[k], v[k], ss);
            ss = warp_sum(ss);
            if (gamma) {
                const float r = rsqrtf(ss / static_cast<float>(D) + P.eps);
#pragma unroll
                for (int k = 0; k < D / 32; ++k) v[k] = v[k] * r * gamma[lane + 32 * k];
            }
#pragma unroll
            for (int k = 0; k < D / 32; ++k) sb[lane + 32 * k] = v[k];
            __syncwarp();
#pragma unroll
            for (int k = 0; k < D / 32; ++k) {
                const int e = lane + 32 * k;
                if (e < R) {
                    const int i = e < half ? e : e - half;
                    v[k] = e < half ? fmaf(sb[e], cs[i], -sb[e + half] * sn[i]) : fmaf(sb[e - half], sn[i], sb[e] * cs[i]);
                }
            }
            __syncwarp();
#pragma unroll
            for (int k = 0; k < D / 32; ++k) sb[lane + 32 * k] = v[k];
            __syncwarp();
        };
        if (has_q) rotate(rq, P.g_q, qs + warp * D);
        if (has_k || has_v) {   // the new token's K and V rows: into the cache and into shared memory
            const int64_t crow = (row0 + slot_p) * D;
            if (has_k) {
                rotate(rkv, P.g_k, kbuf);
                for (int e = lane; e < D; e += 32) {
                    const uint16_t h = __half_as_ushort(__float2half_rn(kbuf[e]));
                    knew[e] = h;
                    P.k_out[crow + e] = h;
                }
            } else {
                float r = 1.f;
                if (P.v_mode == 1) {   // V = unweighted RMSNorm of the raw K row
                    float ss = 0.f;
#pragma unroll
                    for (int k = 0; k < D / 32; ++k) ss = fmaf(rkv[k], rkv[k], ss);
                    r = rsqrtf(warp_sum(ss) / static_cast<float>(D) + P.eps);
                }
#pragma unroll
                for (int k = 0; k < D / 32; ++k) {
                    const int e = lane + 32 * k;
                    const uint16_t h = __half_as_ushort(__float2half_rn(P.v_mode == 1 ? rkv[k] * r : rkv[k]));
                    vnew[e] = h;
                    P.v_out[crow + e] = h;
                }
            }
        }
        __syncthreads();   // rotated query heads and the new rows visible to every warp
    }

    // Q^T B fragments: column n = 2h + hl (head h = n / 2, hi or lo), k = dims
    uint32_t qb[D / 16][2];
    {
        const int h = gq >> 1, hl = gq & 1;
        const float* qrow = P.fuse ? qs + h * D : P.q + b * P.ldq + static_cast<int64_t>(g * G + h) * D;
        float2 raw[D / 16][2];
#pragma unroll
        for (int k16 = 0; k16 < D / 16; ++k16) {
            if (h < G) {
                raw[k16][0] = *reinterpret_cast<const float2*>(qrow + k16 * 16 + 2 * tq);
                raw[k16][1] = *reinterpret_cast<const float2*>(qrow + k16 * 16 + 2 * tq + 8);
            } else {
                raw[k16][0] = raw[k16][1] = make_float2(0.f, 0.f);
            }
        }
#pragma unroll
        for (int k16 = 0; k16 < D / 16; ++k16)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                __half h0, l0, h1, l1;
                split_hi_lo(raw[k16][r].x * P.scale, h0, l0);
                split_hi_lo(raw[k16][r].y * P.scale, h1, l1);
                const __half2 v = hl ? __halves2half2(l0, l1) : __halves2half2(h0, h1);
                qb[k16][r] = *reinterpret_cast<const uint32_t*>(&v);
            }
    }

    float o[D / 16][4];
#pragma unroll
    for (int m = 0; m < D / 16; ++m) o[m][0] = o[m][1] = o[m][2] = o[m][3] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;
    const bool head_ok = tq < G;
    __half* pb = pbuf + warp * 8 * kPbufPitch;
    bool ok = true;

    for (int it = 0; it < nmy; ++it) {
        const int st = it % kFlashStages;
        const int tile = t0 + warp + it * W;
        uint8_t* kt = ring + st * kStageBytes;
        uint8_t* vt = kt + kTileBytes;
        if (ok) ok = mbar_wait(&wbar[st], static_cast<uint32_t>((it / kFlashStages) & 1), P.status);
        const int rp = slot_p - tile * kFlashTile;
        if ((P.fuse || it < npre) && rp >= 0 && rp < kFlashTile) {  // the new row: staged before it was written
            const uint16_t* ks = P.fuse ? knew : P.k_cache + (row0 + slot_p) * D;
            const uint16_t* vs = P.fuse ? vnew : P.v_cache + (row0 + slot_p) * D;
            for (int c = lane * 8; c < D; c += 32 * 8) {
                *reinterpret_cast<uint4*>(kt + swz(rp, c, kFlashTile)) = *reinterpret_cast<const uint4*>(ks + c);
                *reinterpret_cast<uint4*>(vt + swz(rp, c, kFlashTile)) = *reinterpret_cast<const uint4*>(vs + c);
            }
        }
        const int valid = T - tile * kFlashTile;  // rows >= valid belong to other slots
        if (valid < kFlashTile)
            for (int e = lane * 8; e < (kFlashTile - valid) * D; e += 32 * 8) {
                const int r = valid + e / D, c = e % D;
                *reinterpret_cast<uint4*>(vt + swz(r, c, kFlashTile)) = make_uint4(0, 0, 0, 0);
            }
        __syncwarp();
        // S^T = K Q^T
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t kb = smem_u32(kt);
#pragma unroll
        for (int k16 = 0; k16 < D / 16; ++k16) {
            uint32_t a0, a1, a2, a3;
            const int arow = (lane & 7) + ((lane >> 3) & 1) * 8, acol = k16 * 16 + (lane >> 4) * 8;
            ldmatrix_x4(a0, a1, a2, a3, kb + swz(arow, acol, kFlashTile));
            mma_16816(c, a0, a1, a2, a3, qb[k16][0], qb[k16][1]);
        }
        // head tq at positions gq and gq + 8
        float s0 = c[0] + c[1], s1 = c[2] + c[3];
        if (gq >= valid) s0 = -INFINITY;
        if (gq + 8 >= valid) s1 = -INFINITY;
        if (!head_ok) s0 = s1 = 0.f;
        float mx = fmaxf(s0, s1);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float m_new = fmaxf(m_run, mx);          // finite: row 0 of a tile is always valid
        const float corr = expf(m_run - m_new);         // 0 on the first tile
        const float p0 = expf(s0 - m_new), p1 = expf(s1 - m_new);
        float ps = p0 + p1;
        ps += __shfl_xor_sync(0xffffffffu, ps, 4);
        ps += __shfl_xor_sync(0xffffffffu, ps, 8);
        ps += __shfl_xor_sync(0xffffffffu, ps, 16);
        l_run = l_run * corr + ps;
        m_run = m_new;
#pragma unroll
        for (int m = 0; m < D / 16; ++m) {
            o[m][0] *= corr; o[m][1] *= corr; o[m][2] *= corr; o[m][3] *= corr;
        }
        // P^T rows: column 2*tq (hi), 2*tq + 1 (lo); positions gq and gq + 8
        {
            __half h0, l0, h1, l1;
            split_hi_lo(p0, h0, l0);
            split_hi_lo(p1, h1, l1);
            pb[(2 * tq) * kPbufPitch + gq] = h0;
            pb[(2 * tq + 1) * kPbufPitch + gq] = l0;
            pb[(2 * tq) * kPbufPitch + gq + 8] = h1;
            pb[(2 * tq + 1) * kPbufPitch + gq + 8] = l1;
        }
        __syncwarp();
        uint32_t pb0, pb1;
        {
            const int n = lane & 7, kk = ((lane >> 3) & 1) * 8;
            ldmatrix_x2(pb0, pb1, smem_u32(pb + n * kPbufPitch + kk));
        }
        // O^T += V^T P^T
        const uint32_t vb = smem_u32(vt);
#pragma unroll
        for (int m = 0; m < D / 16; ++m) {
            uint32_t a0, a1, a2, a3;
            const int vrow = (lane & 7) + (lane >> 4) * 8, vcol = m * 16 + ((lane >> 3) & 1) * 8;
            ldmatrix_x4_trans(a0, a1, a2, a3, vb + swz(vrow, vcol, kFlashTile));
            mma_16816(o[m], a0, a1, a2, a3, pb0, pb1);
        }
        __syncwarp();
        if (lane == 0 && it + kFlashStages < nmy) issue(it + kFlashStages);
    }
    if (!ok && lane == 0) drain_stages(wbar, kFlashStages, max(0, nmy - kFlashStages), nmy - 1);

    // ---- merge the W warps' states (ascending warp order) -----------------------------------
    __syncthreads();  // all rings idle: reuse them for the combine buffers
    float* cm = comb;                        // [warp][4] max
    float* cl = comb + W * 4;                // [warp][4] denominators
    float* co = comb + 2 * W * 4;            // [warp][4][D] outputs
    if (gq == 0 && head_ok) {
        cm[warp * 4 + tq] = nmy ? m_run : -INFINITY;
        cl[warp * 4 + tq] = nmy ? l_run : 0.f;
    }
    if (head_ok) {
#pragma unroll
        for (int m = 0; m < D / 16; ++m) {
            co[(warp * 4 + tq) * D + m * 16 + gq] = o[m][0] + o[m][1];
            co[(warp * 4 + tq) * D + m * 16 + gq + 8] = o[m][2] + o[m][3];
        }
    }
    __syncthreads();
    const int64_t pstride = static_cast<int64_t>(P.nsplit_max) * (D + 2);   // one head's splits
    float* part0 = P.part + (static_cast<int64_t>(b) * P.n_q + g * G) * pstride;
    for (int e = t_id; e < G * D; e += kNT) {
        const int h = e / D, i = e - h * D;
        float M = -INFINITY;
        for (int w = 0; w < W; ++w) M = fmaxf(M, cm[w * 4 + h]);
        float L = 0.f, O = 0.f;
        for (int w = 0; w < W; ++w) {
            const float f = expf(cm[w * 4 + h] - M);   // warps without tiles: e^-inf = 0
            L += f * cl[w * 4 + h];
            O += f * co[(w * 4 + h) * D + i];
        }
        if (nsplit == 1) {
            P.out[b * P.ldo + static_cast<int64_t>(g * G + h) * D + i] = O / L;
        } else {
            float* dst = part0 + h * pstride + static_cast<int64_t>(split) * (D + 2);
            dst[i] = O;
            if (i == 0) {
                dst[D] = M;
                dst[D + 1] = L;
            }
        }
    }
    if (nsplit == 1 || !P.cnt) return;   // no counters: a stand-alone call's merge kernel combines the splits

    // ---- the last split of this (sequence, KV head) to arrive combines all of them ----------
    // The barrier orders every thread's partial-state writes before thread 0's ticket, whose
    // release (cumulative) publishes them device-wide; its acquire orders the merging CTA's
    // reads of the other splits' states after their tickets.
    __syncthreads();
    unsigned* cnt = P.cnt + b * P.n_kv + g;
    if (t_id == 0) {
        unsigned ticket;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(ticket) : "l"(cnt) : "memory");
        last_sh = ticket == static_cast<unsigned>(nsplit - 1);
    }
    __syncthreads();
    if (!last_sh) return;
    // Split weights per head, one warp per head: lane s holds split s (s < nsplit <= 32 per
    // round); the maximum and the weighted denominator are fixed shuffle trees over the lanes,
    // so the result is the same whichever CTA merges.
    float* wsm = comb;                                // [G][kMaxFlashSplits]: e^(m_s - M_h)
    float* lsm = comb + 4 * kMaxFlashSplits;          // [G]: the combined denominators
    if (warp < G) {
        const int h = warp;
        const float* hs = part0 + h * pstride + D;
        float mv[kMaxFlashSplits / 32], lv[kMaxFlashSplits / 32];
        float M = -INFINITY;
#pragma unroll
        for (int r = 0; r < kMaxFlashSplits / 32; ++r) {
            const int sp = lane + 32 * r;
            mv[r] = sp < nsplit ? __ldcg(hs + static_cast<int64_t>(sp) * (D + 2)) : -INFINITY;
            lv[r] = sp < nsplit ? __ldcg(hs + static_cast<int64_t>(sp) * (D + 2) + 1) : 0.f;
            M = fmaxf(M, mv[r]);
        }
        M = warp_max(M);
        float L = 0.f;
#pragma unroll
        for (int r = 0; r < kMaxFlashSplits / 32; ++r) {
            const int sp = lane + 32 * r;
            const float f = sp < nsplit ? expf(mv[r] - M) : 0.f;
            if (sp < nsplit) wsm[h * kMaxFlashSplits + sp] = f;
            L = fmaf(f, lv[r], L);
        }
        L = warp_sum(L);
        if (lane == 0) lsm[h] = L;
    }
    __syncthreads();
    // every split's output element loaded in one round, then summed in ascending split order
    for (int e = t_id; e < G * D; e += kNT) {
        const int h = e / D, i = e - h * D;
        const float* src = part0 + h * pstride + i;
        const float* wh = wsm + h * kMaxFlashSplits;
        float O = 0.f;
        for (int s0 = 0; s0 < nsplit; s0 += 16) {
            float a[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) a[u] = s0 + u < nsplit ? __ldcg(src + static_cast<int64_t>(s0 + u) * (D + 2)) : 0.f;
#pragma unroll
            for (int u = 0; u < 16; ++u)
                if (s0 + u < nsplit) O = fmaf(wh[s0 + u], a[u], O);
        }
        P.out[b * P.ldo + static_cast<int64_t>(g * G + h) * D + i] = O / lsm[h];
    }
    if (t_id == 0) *cnt = 0u;   // ready for the next call (which follows this kernel's completion)
}

// ---- compact full-attention cache (V rows only) --------------------------------------------
// "gem" research record, "Verified model facts": a full-attention layer's cache can keep the
// unweighted normalised V row alone; the historical K row is rebuilt inside the attention as
// V * key_norm, rotated at the row's own position: K_j = RoPE_j(V_j * gamma_k).  Half the
// bytes of the standard layout per cached position.
//
// One CTA of 16 warps per split of the prefix streams the split's V tiles (TP slots x D) through
// a ring of kCompactSlots TMA stages, each V byte read once.  Per tile:
//   1. the rotated dims of K are rebuilt in shared memory as binary16 hi + lo: fp32 rotation by
//      cos / sin of (j0 + t) w_i = tile anchor (fp64-reduced angle of the tile's first position,
//      taken for every tile of the split before the wait) x offset tables of 8 a w_i and b w_i
//      (t = 8 a + b);
//   2. scores on tensor cores: the dims >= R pass through the rotation, so their part is an mma
//      of the V tile itself against (scale * q * gamma_k); the R rotated dims an mma against the
//      rebuilt hi and lo rows; warps take (n8 tile, part) items;
//   3. online softmax, one warp per query head: running max, rescale factor, P as hi + lo;
//   4. each warp rescales its output accumulators and adds P V for its output dims.
// The split's state (unnormalised output, max, denominator) goes to the workspace and the
// ordered merge kernel combines the splits in ascending order (deterministic).
constexpr int kCompactWarps = 16;
constexpr int kCompactThreads = kCompactWarps * 32;
constexpr int kCompactSlots = 4;

template <int D>
__global__ void __launch_bounds__(kCompactThreads, 1) gqa_compact_kernel(const __grid_constant__ CUtensorMap tmV,
                                                                         const AttnParams P,
                                                                         const __grid_constant__ RopeFreq fr) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int TP = P.tp;
    const int R = P.rope_dim, HR = R / 2, KP = R + 8;
    const int NA = TP / 8;   // offset table rows of 8 a w_i
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P.bar_off);    // [kCompactSlots]
    __half* qa = reinterpret_cast<__half*>(smem + P.qa_off);           // [16][D + 8]
    float* sc = reinterpret_cast<float*>(smem + P.sc_off);             // [16 / (TP / 16)][8][TP]: partial scores
    __half* pa = reinterpret_cast<__half*>(smem + P.pa_off);           // [16][TP + 8]
    float* st = reinterpret_cast<float*>(smem + P.st_off);             // [3][8]: max, denominator, rescale
    __half* kr = reinterpret_cast<__half*>(smem + P.kr_off);           // [2][TP][R + 8]
    float2* an = reinterpret_cast<float2*>(smem + P.an_off);           // [ltile][HR]: tile anchors
    float2* tlo = reinterpret_cast<float2*>(smem + P.tb_off);          // [8][HR]: b w_i
    float2* thi = tlo + 8 * HR;                                         // [NA][HR]: 8 a w_i
    float2* toff = thi + NA * HR;                                       // [TP][HR]: t w_i = 8 a w_i + b w_i
    float* gks = reinterpret_cast<float*>(toff + TP * HR);              // [R]: gamma_k of the rotated dims
    __shared__ int abort_flag;

    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int QA = D + 8, PA = TP + 8;

    if (!P.early) pdl_wait_trigger();
    const int p = P.pos[b];
    if (p < 0 || static_cast<int64_t>(p) >= P.cap) {
        if (P.early) pdl_wait_trigger();
        if (t == 0 && split == 0 && g == 0) atomicOr(P.status, GEM_DEVFLAG_POS_RANGE);
        return;
    }
    const int T = p + 1;
    int nsplit, t0, t1;
    split_range(T, TP, P.nsplit_max, split, nsplit, t0, t1);
    if (split >= nsplit) {
        if (P.early) pdl_wait_trigger();
        return;
    }
    const int ntile = t1 - t0;   // <= ltile
    const int64_t row0 = (static_cast<int64_t>(b) * P.n_kv + g) * P.cap;
    uint64_t policy = 0;
    auto issue = [&](int kt) {
        const int slot = kt % kCompactSlots;
        uint8_t* dst = smem + static_cast<size_t>(slot) * P.tile_bytes;
        fence_proxy_async_smem();   // generic writes to this slot (row refresh, zeroing) precede the TMA
        mbar_arrive_expect_tx(&bars[slot], P.tile_bytes);
        for (int j = 0; j < D / 64; ++j)
            tma_load_2d(dst + j * TP * 128, &tmV, j * 64, static_cast<int32_t>(row0 + static_cast<int64_t>(t0 + kt) * TP),
                        &bars[slot], policy);
    };
    if (t == 0) {
        abort_flag = 0;
        for (int i = 0; i < kCompactSlots; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        prefetch_tensormap(&tmV);
        policy = l2_policy_evict_first();
        for (int kt = 0; kt < min(kCompactSlots, ntile); ++kt) issue(kt);
    }
    // rotation tables (positions only: before the wait): offsets b w_i, 8 a w_i and every tile's anchor
    for (int idx = t; idx < (8 + NA) * HR; idx += kCompactThreads) {
        const int r = idx / HR, i = idx - r * HR;
        const double m = r < 8 ? static_cast<double>(r) : 8.0 * (r - 8);
        float c, sv;
        rope_cos_sin(m * fr.w[i], c, sv);
        tlo[idx] = make_float2(c, sv);   // tlo rows 0..7, then thi rows 0..NA-1 (contiguous)
    }
    for (int idx = t; idx < ntile * HR; idx += kCompactThreads) {
        const int kt = idx / HR, i = idx - kt * HR;
        float c, sv;
        rope_cos_sin(static_cast<double>((t0 + kt) * TP) * fr.w[i], c, sv);
        an[idx] = make_float2(c, sv);
    }
    if (P.early) pdl_wait_trigger();

    // query rows (normalised and rotated at p by the preceding launch): A operand rows h (hi) and
    // h + 8 (lo), scale folded in; the pass-through dims also carry gamma_k
    for (int e = t; e < 8 * D; e += kCompactThreads) {
        const int h = e / D, col = e - h * D;
        float v = 0.f;
        if (h < P.G) {
            v = P.q[b * P.ldq + static_cast<int64_t>(g * P.G + h) * D + col] * P.scale;
            if (col >= R) v *= P.g_k[col];
        }
        __half hi, lo;
        split_hi_lo(v, hi, lo);
        qa[h * QA + col] = hi;
        qa[(h + 8) * QA + col] = lo;
    }
    for (int i = t; i < R; i += kCompactThreads) gks[i] = P.g_k[i];
    __syncthreads();   // the offset tables are complete
    for (int idx = t; idx < TP * HR; idx += kCompactThreads) {   // one rotation per row offset t
        const int tt = idx / HR, i = idx - tt * HR;
        const float2 o1 = thi[(tt >> 3) * HR + i], o2 = tlo[(tt & 7) * HR + i];
        toff[idx] = make_float2(o1.x * o2.x - o1.y * o2.y, o1.y * o2.x + o1.x * o2.y);
    }
    for (int e = t; e < 8 * TP; e += kCompactThreads) {   // P rows of absent heads stay zero
        const int h = e / TP, j = e - h * TP;
        if (h >= P.G) {
            pa[h * PA + j] = __float2half_rn(0.f);
            pa[(h + 8) * PA + j] = __float2half_rn(0.f);
        }
    }
    if (t < 8) {
        st[t] = -INFINITY;
        st[8 + t] = 0.f;
        st[16 + t] = 0.f;
    }
    __syncthreads();

    const int gq = lane >> 2, tq = lane & 3;
    constexpr int NPI = (D / 16 + kCompactWarps - 1) / kCompactWarps;   // 16-dim output items per warp
    float acc[NPI][2][4];
#pragma unroll
    for (int i = 0; i < NPI; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h) acc[i][h][0] = acc[i][h][1] = acc[i][h][2] = acc[i][h][3] = 0.f;

    for (int kt = 0; kt < ntile; ++kt) {
        const int slot = kt % kCompactSlots;
        uint8_t* tile = smem + static_cast<size_t>(slot) * P.tile_bytes;
        if (!mbar_wait(&bars[slot], static_cast<uint32_t>((kt / kCompactSlots) & 1), P.status)) abort_flag = 1;
        const int j0 = (t0 + kt) * TP;
        const int r = p - j0;   // the new row: written by the preceding launch
        if (r >= 0 && r < TP)
            for (int c = t * 8; c < D; c += kCompactThreads * 8)
                *reinterpret_cast<uint4*>(tile + swz(r, c, TP)) =
                    __ldcg(reinterpret_cast<const uint4*>(P.v_cache + (row0 + p) * D + c));
        const int valid = T - j0;   // rows >= valid hold other slots: zero them (P V reads them)
        if (valid < TP)
            for (int e = t * 8; e < (TP - valid) * D; e += kCompactThreads * 8) {
                const int rr = valid + e / D, c = e % D;
                *reinterpret_cast<uint4*>(tile + swz(rr, c, TP)) = make_uint4(0, 0, 0, 0);
            }
        __syncthreads();
        if (abort_flag) {
            if (t == 0) drain_stages(bars, kCompactSlots, kt, min(kt + kCompactSlots - 1, ntile - 1));
            return;
        }
        // 1. rebuilt K of the rotated dims (hi + lo): warp rows, two adjacent dims per lane (R is a
        // multiple of 16, so dims i, i + 1 share a 16-byte chunk of the swizzled tile)
        const float2* ak = an + kt * HR;
        for (int tt = warp; tt < TP; tt += kCompactWarps) {
            const float2* ro = toff + tt * HR;
            for (int i = 2 * lane; i < HR; i += 64) {
                const float2 uf = __half22float2(*reinterpret_cast<const __half2*>(tile + swz(tt, i, TP)));
                const float2 wf = __half22float2(*reinterpret_cast<const __half2*>(tile + swz(tt, i + HR, TP)));
                const float2 gu = *reinterpret_cast<const float2*>(gks + i);
                const float2 gw = *reinterpret_cast<const float2*>(gks + i + HR);
                const float4 a01 = *reinterpret_cast<const float4*>(ak + i);   // anchors of dims i, i + 1
                const float4 o01 = *reinterpret_cast<const float4*>(ro + i);   // row offsets of dims i, i + 1
                const float c0 = a01.x * o01.x - a01.y * o01.y, s0 = a01.y * o01.x + a01.x * o01.y;
                const float c1 = a01.z * o01.z - a01.w * o01.w, s1 = a01.w * o01.z + a01.z * o01.w;
                const float u0 = uf.x * gu.x, u1 = uf.y * gu.y, w0 = wf.x * gw.x, w1 = wf.y * gw.y;
                const float ka0 = u0 * c0 - w0 * s0, ka1 = u1 * c1 - w1 * s1;   // dims i, i + 1
                const float kb0 = u0 * s0 + w0 * c0, kb1 = u1 * s1 + w1 * c1;   // dims i + HR, i + HR + 1
                const __half2 ha = __floats2half2_rn(ka0, ka1), hb = __floats2half2_rn(kb0, kb1);
                const float2 fa = __half22float2(ha), fb = __half22float2(hb);
                const __half2 la = __floats2half2_rn(ka0 - fa.x, ka1 - fa.y), lb = __floats2half2_rn(kb0 - fb.x, kb1 - fb.y);
                *reinterpret_cast<__half2*>(kr + tt * KP + i) = ha;
                *reinterpret_cast<__half2*>(kr + tt * KP + i + HR) = hb;
                *reinterpret_cast<__half2*>(kr + (TP + tt) * KP + i) = la;
                *reinterpret_cast<__half2*>(kr + (TP + tt) * KP + i + HR) = lb;
            }
        }
        __syncthreads();
        // 2. scores: item = (16 positions, one of NKS cost-balanced parts of the k16 steps); a
        // rotated step takes two mma (hi and lo), a pass-through step one.  Each q fragment loaded
        // serves two n8 tiles; two accumulator pairs halve the dependent mma chains.
        {
            const uint32_t tbase = smem_u32(tile), kbase = smem_u32(kr);
            const int arow = (lane & 7) + ((lane >> 3) & 1) * 8, acol = (lane >> 4) * 8;
            const int brow = (lane & 7) + ((lane >> 4) << 3), bcol = ((lane >> 3) & 1) * 8;
            const int nrot = R / 16, nk = D / 16, cost = nk + nrot;
            const int NP = TP / 16, NKS = kCompactWarps / NP;   // NP * NKS = kCompactWarps items
            const int item = warp, np = item % NP, ks = item / NP;
            // k16 range of part ks: the first step whose cumulative cost reaches ks * cost / NKS
            auto kstart = [&](int q) {
                const int c = (q * cost + NKS - 1) / NKS;   // cost before the part
                return 2 * nrot >= c ? (c + 1) / 2 : nrot + (c - 2 * nrot);
            };
            const int kb = kstart(ks), ke = ks + 1 == NKS ? nk : kstart(ks + 1);
            float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
            float e0[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f};
            const int r16 = np * 16 + brow;
            for (int k16 = kb; k16 < ke; ++k16) {
                uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
                ldmatrix_x4(a0, a1, a2, a3, smem_u32(qa + arow * QA + k16 * 16 + acol));
                if (k16 < nrot) {
                    uint32_t f0, f1, f2, f3;
                    ldmatrix_x4(b0, b1, b2, b3, kbase + static_cast<uint32_t>((r16 * KP + k16 * 16 + bcol) * 2));
                    ldmatrix_x4(f0, f1, f2, f3, kbase + static_cast<uint32_t>(((TP + r16) * KP + k16 * 16 + bcol) * 2));
                    mma_16816(c0, a0, a1, a2, a3, b0, b1);
                    mma_16816(c1, a0, a1, a2, a3, b2, b3);
                    mma_16816(e0, a0, a1, a2, a3, f0, f1);
                    mma_16816(e1, a0, a1, a2, a3, f2, f3);
                } else {
                    ldmatrix_x4(b0, b1, b2, b3, tbase + swz(r16, k16 * 16 + bcol, TP));
                    if (k16 & 1) {
                        mma_16816(e0, a0, a1, a2, a3, b0, b1);
                        mma_16816(e1, a0, a1, a2, a3, b2, b3);
                    } else {
                        mma_16816(c0, a0, a1, a2, a3, b0, b1);
                        mma_16816(c1, a0, a1, a2, a3, b2, b3);
                    }
                }
            }
            // rows gq (hi) and gq + 8 (lo) of head gq; positions 16 np + 2 tq (+1), and + 8
            float* sp = sc + (ks * 8 + gq) * TP + np * 16 + 2 * tq;
            sp[0] = (c0[0] + c0[2]) + (e0[0] + e0[2]);
            sp[1] = (c0[1] + c0[3]) + (e0[1] + e0[3]);
            sp[8] = (c1[0] + c1[2]) + (e1[0] + e1[2]);
            sp[9] = (c1[1] + c1[3]) + (e1[1] + e1[3]);
        }
        __syncthreads();
        // 3. online softmax, warp h = query head h
        if (warp < P.G) {
            const int h = warp;
            const float m_old = st[h];
            float mt = -INFINITY;
            const int nks = kCompactWarps / (TP / 16);
            for (int j = lane; j < TP; j += 32) {
                float sj = -INFINITY;
                if (j < valid) {
                    sj = 0.f;
                    for (int q = 0; q < nks; ++q) sj += sc[(q * 8 + h) * TP + j];
                }
                sc[h * TP + j] = sj;
                mt = fmaxf(mt, sj);
            }
            mt = warp_max(mt);
            const float m_new = fmaxf(m_old, mt);
            float l = 0.f;
            for (int j = lane; j < TP; j += 32) {
                const float e = expf(sc[h * TP + j] - m_new);   // (-inf rows: 0)
                l += e;
                __half hi, lo;
                split_hi_lo(e, hi, lo);
                pa[h * PA + j] = hi;
                pa[(h + 8) * PA + j] = lo;
            }
            l = warp_sum(l);
            if (lane == 0) {
                const float alpha = m_old == -INFINITY ? 0.f : expf(m_old - m_new);
                st[h] = m_new;
                st[8 + h] = st[8 + h] * alpha + l;
                st[16 + h] = alpha;
            }
        }
        __syncthreads();
        // 4. rescale and accumulate P V for this warp's output dims
        {
            const float alpha = gq < P.G ? st[16 + gq] : 1.f;   // (rows of absent heads stay zero)
            const uint32_t tbase = smem_u32(tile);
            if (!__all_sync(0xffffffffu, alpha == 1.f)) {   // a maximum moved (or the first tile)
#pragma unroll
                for (int pi = 0; pi < NPI; ++pi)
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) acc[pi][h][q4] *= alpha;
            }
            for (int k16 = 0; k16 < TP / 16; ++k16) {
                uint32_t a0, a1, a2, a3;
                const int arow = (lane & 7) + ((lane >> 3) & 1) * 8, acol = k16 * 16 + (lane >> 4) * 8;
                ldmatrix_x4(a0, a1, a2, a3, smem_u32(pa + arow * PA + acol));
#pragma unroll
                for (int pi = 0; pi < NPI; ++pi) {
                    const int item = warp + pi * kCompactWarps;
                    if (item < D / 16) {
                        uint32_t b0, b1, b2, b3;
                        const int vrow = k16 * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                        const int vcol = item * 16 + (lane >> 4) * 8;
                        ldmatrix_x4_trans(b0, b1, b2, b3, tbase + swz(vrow, vcol, TP));
                        mma_16816(acc[pi][0], a0, a1, a2, a3, b0, b1);
                        mma_16816(acc[pi][1], a0, a1, a2, a3, b2, b3);
                    }
                }
            }
        }
        __syncthreads();   // the slot, the scores and P are free
        if (t == 0 && kt + kCompactSlots < ntile) issue(kt + kCompactSlots);
    }

    // ---- output ------------------------------------------------------------------------------
    if (gq < P.G) {
        const int h = g * P.G + gq;
        const float m = st[gq], l = st[8 + gq];
        float* o = nsplit == 1 ? P.out + b * P.ldo + static_cast<int64_t>(h) * D
                               : P.part + ((static_cast<int64_t>(b) * P.n_q + h) * P.nsplit_max + split) * (D + 2);
        const float inv = nsplit == 1 ? 1.f / l : 1.f;
#pragma unroll
        for (int pi = 0; pi < NPI; ++pi) {
            const int item = warp + pi * kCompactWarps;
            if (item < D / 16) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int dd = item * 16 + hh * 8 + 2 * tq;
                    o[dd] = (acc[pi][hh][0] + acc[pi][hh][2]) * inv;
                    o[dd + 1] = (acc[pi][hh][1] + acc[pi][hh][3]) * inv;
                }
            }
        }
        if (nsplit > 1 && warp == 0 && tq == 0) {
            o[D] = m;
            o[D + 1] = l;
        }
    }
}

// Ordered merge of split states:  M = max_s m_s,  out = sum_s e^(m_s - M) acc_s / sum_s e^(m_s - M) l_s
// One CTA per (sequence, query head).  Every global load is issued in one parallel round:
// split maxima and denominators into shared memory, then the split sums of the outputs,
// spread over kMergeGroups thread groups (each summing every kMergeGroups-th split in
// ascending order) and combined in a fixed order, so the result is deterministic.
constexpr int kMergeThreads = 512;
constexpr int kMaxSplits = 1024;

__global__ void __launch_bounds__(kMergeThreads) gqa_merge_kernel(const AttnParams P, int D) {
    __shared__ float wsh[kMaxSplits], lsh[kMaxSplits];
    __shared__ float psum[kMergeThreads];
    __shared__ float red[kMergeThreads / 32];
    pdl_wait_trigger();
    const int bh = blockIdx.x;
    const int b = bh / P.n_q, h = bh - b * P.n_q;
    const int p = P.pos[b];
    if (p < 0 || (P.window == 0 && static_cast<int64_t>(p) >= P.cap)) return;
    const int T = P.window ? min(P.window, p + 1) : p + 1;
    const int nt = (T + P.tp - 1) / P.tp;
    const int nsplit = min(P.nsplit_max, nt);
    if (nsplit <= 1) return;
    const int stride = D + 2;
    const float* base = P.part + (static_cast<int64_t>(b) * P.n_q + h) * P.nsplit_max * stride;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float m = -INFINITY;
    for (int s = tid; s < nsplit; s += kMergeThreads) {
        const float ms = base[s * stride + D];
        wsh[s] = ms;
        lsh[s] = base[s * stride + D + 1];
        m = fmaxf(m, ms);
    }
    m = warp_max(m);
    if (lane == 0) red[warp] = m;
    __syncthreads();
    float M = red[0];
    for (int w = 1; w < kMergeThreads / 32; ++w) M = fmaxf(M, red[w]);
    for (int s = tid; s < nsplit; s += kMergeThreads) wsh[s] = expf(wsh[s] - M);
    __syncthreads();
    // output partial sums: group q handles splits q, q + ngroups, ... for dims i < D
    const int ngroups = kMergeThreads / D;  // D <= 512
    const int q = tid / D, i = tid - q * D;
    float v = 0.f;
    if (q < ngroups) {
        int s = q;
        for (; s + 7 * ngroups < nsplit; s += 8 * ngroups) {
            float a[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) a[u] = base[(s + u * ngroups) * stride + i];
#pragma unroll
            for (int u = 0; u < 8; ++u) v += wsh[s + u * ngroups] * a[u];
        }
        for (; s < nsplit; s += ngroups) v += wsh[s] * base[s * stride + i];
    }
    psum[tid] = v;
    if (warp == 0) {  // denominator in ascending split order
        float den = 0.f;
        for (int s = lane; s < nsplit; s += 32) den += wsh[s] * lsh[s];
        den = warp_sum(den);
        if (lane == 0) red[0] = den;
    }
    __syncthreads();
    if (tid < D) {
        float o = 0.f;
        for (int g2 = 0; g2 < ngroups; ++g2) o += psum[g2 * D + tid];
        P.out[b * P.ldo + static_cast<int64_t>(h) * D + tid] = o / red[0];
    }
}

struct Plan {
    bool flash;
    int W;          // flash: warps per CTA
    int tp, nsplit_max, ltile, ns;
    uint32_t tile_bytes, bar_off, qa_off, sc_off, pa_off, st_off;
    size_t smem, ws, cnt_off;   // cnt_off: byte offset of the flash arrival counters in the workspace
};

bool use_flash(int n_q, int n_kv, int d) { return d <= 256 && n_q / n_kv <= 4; }

size_t flash_smem(int d, int W) {
    const size_t ring = static_cast<size_t>(W) * kFlashStages * 2 * kFlashTile * d * 2;
    // + barriers, P^T buffers, the fused path's query heads, K row, rotation table, new K/V rows
    return align_up(ring + 128 + static_cast<size_t>(W) * 8 * kPbufPitch * 2 + 28ull * d, 1024) + 1024;
}

const void* pick(int d, bool flash, int W);
gem_status ensure_smem_attn(const void* fn, int device, size_t bytes);

// Resident flash CTAs per SM for (d, W) on this device (occupancy query, cached).
int flash_ctas_per_sm(int d, int W, int device) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int>, int> done;
    std::lock_guard<std::mutex> lk(mu);
    auto it = done.find({device, d, W});
    if (it != done.end()) return it->second;
    int n = 1;
    const void* fn = pick(d, true, W);
    const size_t smem = flash_smem(d, W);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) == cudaSuccess &&
        cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared) ==
            cudaSuccess &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, W * 32, smem) == cudaSuccess && n >= 1) {
    } else {
        (void)cudaGetLastError();
        n = 1;
    }
    done[{device, d, W}] = n;
    return n;
}

Plan make_plan(int B, int n_q, int n_kv, int d, int64_t cap, int window, int num_sms, int device) {
    Plan pl{};
    pl.flash = use_flash(n_q, n_kv, d);
    pl.tp = pl.flash ? kFlashTile : tile_slots(d);
    const int64_t tmax = window ? std::min<int64_t>(window, cap) : cap;
    const int64_t nt_max = std::max<int64_t>(1, (tmax + pl.tp - 1) / pl.tp);
    const int64_t pairs = static_cast<int64_t>(B) * n_kv;
    if (pl.flash) {
        // Eight warps per CTA while there are few (sequence, KV head) pairs, else four (smaller
        // CTAs, more of them resident per SM); as many splits as fill the SMs' resident slots.
        pl.W = (d <= 128 && pairs * 8 <= num_sms) ? 8 : 4;
        const int64_t slots = static_cast<int64_t>(flash_ctas_per_sm(d, pl.W, device)) * num_sms;
        int64_t ns = std::max<int64_t>(1, slots / pairs);
        ns = std::min<int64_t>(std::min<int64_t>(ns, nt_max), kMaxFlashSplits);
        pl.nsplit_max = static_cast<int>(ns);
        pl.ltile = static_cast<int>((nt_max + ns - 1) / ns);
        pl.smem = flash_smem(d, pl.W);
        if (ns > 1) {
            const size_t part = static_cast<size_t>(B) * n_q * ns * (d + 2) * sizeof(float);
            pl.cnt_off = align_up(part, 256);
            pl.ws = pl.cnt_off + align_up(static_cast<size_t>(pairs) * sizeof(unsigned), 256);
        }
        return pl;
    }
    const int64_t target = static_cast<int64_t>(num_sms);   // one wave: a CTA per SM
    int64_t ns = std::max<int64_t>(1, (target + pairs - 1) / pairs);
    ns = std::min(ns, nt_max);
    const int max_tiles = kMaxSplitSlots / pl.tp;
    if ((nt_max + ns - 1) / ns > max_tiles) ns = (nt_max + max_tiles - 1) / max_tiles;
    ns = std::min<int64_t>(ns, kMaxSplits);
    pl.nsplit_max = static_cast<int>(ns);
    pl.ltile = static_cast<int>((nt_max + ns - 1) / ns);
    pl.ws = ns > 1 ? static_cast<size_t>(B) * n_q * pl.nsplit_max * (d + 2) * sizeof(float) : 0;
    pl.tile_bytes = static_cast<uint32_t>(pl.tp * d * 2);
    pl.ns = d >= 512 ? 3 : 4;
    pl.ns = static_cast<int>(std::min<int64_t>(pl.ns, 2 * pl.ltile));
    const int G = n_q / n_kv;
    const int L = pl.ltile * pl.tp;
    size_t off = static_cast<size_t>(pl.ns) * pl.tile_bytes;
    pl.bar_off = static_cast<uint32_t>(off);
    off = align_up(off + 8 * 8, 128);
    pl.qa_off = static_cast<uint32_t>(off);
    off = align_up(off + 16 * (d + 8) * 2, 128);
    pl.sc_off = static_cast<uint32_t>(off);
    off = align_up(off + static_cast<size_t>(G) * L * 4, 128);
    pl.pa_off = static_cast<uint32_t>(off);
    off = align_up(off + 16ull * (L + 8) * 2, 128);
    pl.st_off = static_cast<uint32_t>(off);
    off += 16 * 4;
    pl.smem = align_up(off, 1024) + 1024;
    return pl;
}

const void* pick(int d, bool flash, int W) {
    if (flash) {
        switch (d) {
            case 64: return W == 8 ? reinterpret_cast<const void*>(gqa_flash_kernel<64, 8>)
                                   : reinterpret_cast<const void*>(gqa_flash_kernel<64, 4>);
            case 128: return W == 8 ? reinterpret_cast<const void*>(gqa_flash_kernel<128, 8>)
                                    : reinterpret_cast<const void*>(gqa_flash_kernel<128, 4>);
            default: return reinterpret_cast<const void*>(gqa_flash_kernel<256, 4>);
        }
    }
    switch (d) {
        case 64: return reinterpret_cast<const void*>(gqa_split_kernel<64>);
        case 128: return reinterpret_cast<const void*>(gqa_split_kernel<128>);
        case 256: return reinterpret_cast<const void*>(gqa_split_kernel<256>);
        default: return reinterpret_cast<const void*>(gqa_split_kernel<512>);
    }
}

gem_status ensure_smem_attn(const void* fn, int device, size_t bytes) {
    static std::mutex mu;
    static std::map<std::pair<int, const void*>, size_t> done;
    std::lock_guard<std::mutex> lk(mu);
    size_t& have = done[{device, fn}];
    if (have >= bytes) return GEM_OK;
    GEM_CUDA_TRY(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)));
    have = bytes;
    return GEM_OK;
}

// chain: launched right after the library's QKV projection, which clears the flash arrival
// counters; otherwise (stand-alone calls) the split partials go to the merge kernel.
gem_status attn_launch(const AttnOp& op, cudaStream_t stream, bool early, bool fuse, bool chain) {
    gem_status st = attn_check(op);
    if (st != GEM_OK || op.B == 0 || op.n_q == 0) return st;
    DeviceInfo di;
    if ((st = device_info(&di)) != GEM_OK) return st;
    const Plan pl = make_plan(op.B, op.n_q, op.n_kv, op.d, op.cache_cap, op.window, di.num_sms, di.device);
    if (pl.nsplit_max > 1 && (!op.workspace || op.ws_bytes < pl.ws)) return GEM_ERR_WORKSPACE;
    if (pl.smem > di.smem_optin) return GEM_ERR_UNSUPPORTED_SHAPE;
    AttnParams P{};
    P.q = op.q;
    P.ldq = op.ldq;
    P.B = op.B;
    P.n_q = op.n_q;
    P.n_kv = op.n_kv;
    P.G = op.n_q / op.n_kv;
    P.cap = op.cache_cap;
    P.window = op.window;
    P.scale = op.scale;
    P.pos = op.pos;
    P.out = op.out;
    P.ldo = op.ldo;
    P.part = static_cast<float*>(op.workspace);
    P.nsplit_max = pl.nsplit_max;
    P.tp = pl.tp;
    P.ltile = pl.ltile;
    P.ns = pl.ns;
    P.early = early ? 1 : 0;
    P.k_cache = op.k_cache;
    P.v_cache = op.v_cache;
    P.tile_bytes = pl.tile_bytes;
    P.bar_off = pl.bar_off;
    P.qa_off = pl.qa_off;
    P.sc_off = pl.sc_off;
    P.pa_off = pl.pa_off;
    P.st_off = pl.st_off;
    P.status = op.status ? op.status : di.status_word;
    // Inside the layer chain the last-arriving split merges (the QKV projection clears the
    // counters); a stand-alone call leaves its split partials to the ordered merge kernel, so it
    // needs no cleared counters and no memset between launches.
    P.cnt = pl.flash && pl.nsplit_max > 1 && chain
                ? reinterpret_cast<unsigned*>(static_cast<char*>(op.workspace) + pl.cnt_off)
                : nullptr;
    RopeFreq fr{};
    if (fuse) {
        if (!pl.flash) return GEM_ERR_UNSUPPORTED_SHAPE;
        if (op.rope_dim < 2 || op.rope_dim > op.d || (op.rope_dim & 1) || !(op.theta > 0.f) || op.v_mode < 0 ||
            op.v_mode > 1 || !op.k_out || !op.v_out)
            return GEM_ERR_INVALID_ARG;
        if (op.ldq < static_cast<int64_t>(op.n_q + op.n_kv + (op.v_mode ? 0 : op.n_kv)) * op.d)
            return GEM_ERR_INVALID_ARG;
        P.fuse = 1;
        P.g_q = op.gamma_q;
        P.g_k = op.gamma_k;
        P.eps = op.eps;
        P.rope_dim = op.rope_dim;
        P.v_mode = op.v_mode;
        P.k_out = op.k_out;
        P.v_out = op.v_out;
        for (int i = 0; i < op.rope_dim / 2; ++i)
            fr.w[i] = std::pow(static_cast<double>(op.theta), -2.0 * i / op.rope_dim);
    }

    const uint64_t rows = static_cast<uint64_t>(op.B) * op.n_kv * op.cache_cap;
    CUtensorMap tmK, tmV;
    if ((st = make_tensor_map_2d(&tmK, CU_TENSOR_MAP_DATA_TYPE_UINT16, op.k_cache, op.d, rows,
                                 static_cast<uint64_t>(op.d) * 2, 64, pl.tp, CU_TENSOR_MAP_SWIZZLE_128B)) != GEM_OK)
        return st;
    if ((st = make_tensor_map_2d(&tmV, CU_TENSOR_MAP_DATA_TYPE_UINT16, op.v_cache, op.d, rows,
                                 static_cast<uint64_t>(op.d) * 2, 64, pl.tp, CU_TENSOR_MAP_SWIZZLE_128B)) != GEM_OK)
        return st;
    const void* fn = pick(op.d, pl.flash, pl.W);
    if ((st = ensure_smem_attn(fn, di.device, pl.smem)) != GEM_OK) return st;
    dim3 grid(pl.nsplit_max, op.n_kv, op.B);
    void* args[] = {&tmK, &tmV, &P, &fr};   // the split kernel takes the first three
    if ((st = launch_pdl(fn, grid, dim3(pl.flash ? pl.W * 32 : kAttnThreads), pl.smem, stream, args)) != GEM_OK)
        return st;
    if (pl.nsplit_max > 1 && !P.cnt) {
        int D = op.d;
        void* margs[] = {&P, &D};
        st = launch_pdl(reinterpret_cast<const void*>(gqa_merge_kernel), dim3(op.B * op.n_q), dim3(kMergeThreads), 0,
                        stream, margs);
    }
    return st;
}

// ---- compact cache plan and launch -------------------------------------------------------------
struct CompactPlan {
    int tp, ltile, ns;
    uint32_t tile_bytes, bar_off, qa_off, sc_off, pa_off, st_off, kr_off, tb_off, an_off;
    size_t smem, ws;
};

// About one CTA per SM over the (sequence, KV head) pairs, more splits where a split's tile
// anchors would not fit shared memory.  ok = false when no layout fits.
bool compact_plan(int B, int n_q, int n_kv, int d, int64_t cap, int R, int num_sms, size_t smem_optin,
                  CompactPlan& pl) {
    pl = CompactPlan{};
    pl.tp = tile_slots(d);
    pl.tile_bytes = static_cast<uint32_t>(pl.tp * d * 2);
    const int64_t nt_max = std::max<int64_t>(1, (cap + pl.tp - 1) / pl.tp);
    const int HR = R / 2;
    auto layout = [&](int lt, bool commit) -> size_t {
        size_t off = static_cast<size_t>(kCompactSlots) * pl.tile_bytes;
        const size_t bar = off;
        off = align_up(off + kCompactSlots * 8, 128);
        const size_t qa = off;
        off = align_up(off + 16ull * (d + 8) * 2, 128);
        const size_t sc = off;   // kCompactWarps / (tp / 16) partial score blocks of 8 x tp floats
        off = align_up(off + static_cast<size_t>(kCompactWarps) * 16 * 8 * 4, 128);
        const size_t pa = off;
        off = align_up(off + 16ull * (pl.tp + 8) * 2, 128);
        const size_t st = off;
        off = align_up(off + 3 * 8 * 4, 128);
        const size_t kr = off;
        off = align_up(off + 2ull * pl.tp * (R + 8) * 2, 128);
        const size_t tb = off;   // offsets b w_i (8 rows), 8 a w_i (tp / 8 rows), t w_i (tp rows), gamma_k[R]
        off = align_up(off + static_cast<size_t>(8 + pl.tp / 8 + pl.tp) * HR * 8 + static_cast<size_t>(R) * 4, 128);
        const size_t an = off;
        off += static_cast<size_t>(lt) * HR * 8;
        if (commit) {
            pl.bar_off = static_cast<uint32_t>(bar);
            pl.qa_off = static_cast<uint32_t>(qa);
            pl.sc_off = static_cast<uint32_t>(sc);
            pl.pa_off = static_cast<uint32_t>(pa);
            pl.st_off = static_cast<uint32_t>(st);
            pl.kr_off = static_cast<uint32_t>(kr);
            pl.tb_off = static_cast<uint32_t>(tb);
            pl.an_off = static_cast<uint32_t>(an);
        }
        return align_up(off, 1024) + 1024;
    };
    const int64_t pairs = static_cast<int64_t>(B) * n_kv;
    int64_t ns = std::max<int64_t>(1, std::min<int64_t>(nt_max, (num_sms + pairs - 1) / pairs));
    while (ns <= nt_max && layout(static_cast<int>((nt_max + ns - 1) / ns), false) + 2048 > smem_optin) ++ns;
    if (ns > nt_max || ns > kMaxSplits) return false;
    pl.ns = static_cast<int>(ns);
    pl.ltile = static_cast<int>((nt_max + ns - 1) / ns);
    pl.smem = layout(pl.ltile, true);
    pl.ws = ns > 1 ? static_cast<size_t>(B) * n_q * pl.ns * (d + 2) * sizeof(float) : 0;
    return true;
}

const void* pick_compact(int d) {
    switch (d) {
        case 64: return reinterpret_cast<const void*>(gqa_compact_kernel<64>);
        case 128: return reinterpret_cast<const void*>(gqa_compact_kernel<128>);
        case 256: return reinterpret_cast<const void*>(gqa_compact_kernel<256>);
        default: return reinterpret_cast<const void*>(gqa_compact_kernel<512>);
    }
}

}  // namespace

gem_status compact_check(const CompactAttnOp& op) {
    if (op.B < 0 || op.n_q < 0 || op.n_kv <= 0 || op.cache_cap <= 0) return GEM_ERR_INVALID_ARG;
    if (op.d != 64 && op.d != 128 && op.d != 256 && op.d != 512) return GEM_ERR_UNSUPPORTED_SHAPE;
    if (op.n_q % op.n_kv) return GEM_ERR_INVALID_ARG;
    if (op.n_q / op.n_kv > 8) return GEM_ERR_UNSUPPORTED_SHAPE;
    if (op.rope_dim < 0 || op.rope_dim > op.d || (op.rope_dim % 16)) return GEM_ERR_UNSUPPORTED_SHAPE;
    if (!(op.theta > 0.f)) return GEM_ERR_INVALID_ARG;
    if (op.B == 0 || op.n_q == 0) return GEM_OK;
    if (!op.q || !op.v_cache || !op.pos || !op.out || !op.gamma_k) return GEM_ERR_INVALID_ARG;
    if (op.ldq < static_cast<int64_t>(op.n_q) * op.d || op.ldo < static_cast<int64_t>(op.n_q) * op.d)
        return GEM_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(op.v_cache) & 15) return GEM_ERR_MISALIGNED;
    if (static_cast<uint64_t>(op.B) * op.n_kv * op.cache_cap >= (1ull << 31)) return GEM_ERR_UNSUPPORTED_SHAPE;
    return GEM_OK;
}

size_t compact_workspace_bytes(int B, int n_q, int n_kv, int d, int64_t cache_cap, int rope_dim) {
    if (B <= 0 || n_q <= 0 || n_kv <= 0 || cache_cap <= 0 || n_q % n_kv) return 0;
    DeviceInfo di;
    if (device_info(&di) != GEM_OK) return 0;
    CompactPlan pl;
    if (!compact_plan(B, n_q, n_kv, d, cache_cap, rope_dim, di.num_sms, di.smem_optin, pl)) return 0;
    return align_up(pl.ws, 256);
}

gem_status compact_enqueue(const CompactAttnOp& op, cudaStream_t stream, bool early) {
    gem_status st = compact_check(op);
    if (st != GEM_OK || op.B == 0 || op.n_q == 0) return st;
    DeviceInfo di;
    if ((st = device_info(&di)) != GEM_OK) return st;
    CompactPlan pl;
    if (!compact_plan(op.B, op.n_q, op.n_kv, op.d, op.cache_cap, op.rope_dim, di.num_sms, di.smem_optin, pl))
        return GEM_ERR_UNSUPPORTED_SHAPE;
    if (pl.ns > 1 && (!op.workspace || op.ws_bytes < pl.ws)) return GEM_ERR_WORKSPACE;
    AttnParams P{};
    P.q = op.q;
    P.ldq = op.ldq;
    P.B = op.B;
    P.n_q = op.n_q;
    P.n_kv = op.n_kv;
    P.G = op.n_q / op.n_kv;
    P.cap = op.cache_cap;
    P.window = 0;
    P.scale = op.scale;
    P.pos = op.pos;
    P.out = op.out;
    P.ldo = op.ldo;
    P.part = static_cast<float*>(op.workspace);
    P.nsplit_max = pl.ns;
    P.tp = pl.tp;
    P.ltile = pl.ltile;
    P.early = early ? 1 : 0;
    P.v_cache = op.v_cache;
    P.tile_bytes = pl.tile_bytes;
    P.bar_off = pl.bar_off;
    P.qa_off = pl.qa_off;
    P.sc_off = pl.sc_off;
    P.pa_off = pl.pa_off;
    P.st_off = pl.st_off;
    P.kr_off = pl.kr_off;
    P.tb_off = pl.tb_off;
    P.an_off = pl.an_off;
    P.status = op.status ? op.status : di.status_word;
    P.g_k = op.gamma_k;
    P.rope_dim = op.rope_dim;
    RopeFreq fr{};
    for (int i = 0; i < op.rope_dim / 2; ++i)
        fr.w[i] = std::pow(static_cast<double>(op.theta), -2.0 * i / op.rope_dim);
    const uint64_t rows = static_cast<uint64_t>(op.B) * op.n_kv * op.cache_cap;
    CUtensorMap tmV;
    if ((st = make_tensor_map_2d(&tmV, CU_TENSOR_MAP_DATA_TYPE_UINT16, op.v_cache, op.d, rows,
                                 static_cast<uint64_t>(op.d) * 2, 64, pl.tp, CU_TENSOR_MAP_SWIZZLE_128B)) != GEM_OK)
        return st;
    const void* fn = pick_compact(op.d);
    if ((st = ensure_smem_attn(fn, di.device, pl.smem)) != GEM_OK) return st;
    void* args[] = {&tmV, &P, &fr};
    if ((st = launch_pdl(fn, dim3(pl.ns, op.n_kv, op.B), dim3(kCompactThreads), pl.smem, stream, args)) != GEM_OK)
        return st;
    if (pl.ns > 1) {
        int D = op.d;
        void* margs[] = {&P, &D};
        st = launch_pdl(reinterpret_cast<const void*>(gqa_merge_kernel), dim3(op.B * op.n_q), dim3(kMergeThreads), 0,
                        stream, margs);
    }
    return st;
}

size_t attn_workspace_bytes(int B, int n_q, int n_kv, int d, int64_t cache_cap, int window) {
    if (B <= 0 || n_q <= 0 || n_kv <= 0 || cache_cap <= 0) return 0;
    if (d != 64 && d != 128 && d != 256 && d != 512) return 0;
    DeviceInfo di;
    if (device_info(&di) != GEM_OK) return 0;
    const Plan pl = make_plan(B, n_q, n_kv, d, cache_cap, window, di.num_sms, di.device);
    return pl.nsplit_max > 1 ? align_up(pl.ws, 256) : 0;
}

size_t attn_counter_offset(int B, int n_q, int n_kv, int d, int64_t cache_cap, int window, size_t* bytes) {
    *bytes = 0;
    if (B <= 0 || n_q <= 0 || n_kv <= 0 || cache_cap <= 0 || !use_flash(n_q, n_kv, d)) return 0;
    DeviceInfo di;
    if (device_info(&di) != GEM_OK) return 0;
    const Plan pl = make_plan(B, n_q, n_kv, d, cache_cap, window, di.num_sms, di.device);
    if (pl.nsplit_max <= 1) return 0;
    *bytes = static_cast<size_t>(B) * n_kv * sizeof(unsigned);
    return pl.cnt_off;
}

gem_status attn_check(const AttnOp& op) {
    if (op.B < 0 || op.n_q < 0 || op.n_kv <= 0 || op.cache_cap <= 0 || op.window < 0) return GEM_ERR_INVALID_ARG;
    if (op.d != 64 && op.d != 128 && op.d != 256 && op.d != 512) return GEM_ERR_UNSUPPORTED_SHAPE;
    if (op.n_q % op.n_kv) return GEM_ERR_INVALID_ARG;
    if (op.n_q / op.n_kv > 8) return GEM_ERR_UNSUPPORTED_SHAPE;
    if (op.window > op.cache_cap) return GEM_ERR_INVALID_ARG;
    if (op.B == 0 || op.n_q == 0) return GEM_OK;
    if (!op.q || !op.k_cache || !op.v_cache || !op.pos || !op.out) return GEM_ERR_INVALID_ARG;
    if (op.ldq < static_cast<int64_t>(op.n_q) * op.d || op.ldo < static_cast<int64_t>(op.n_q) * op.d)
        return GEM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(op.k_cache) | reinterpret_cast<uintptr_t>(op.v_cache)) & 15)
        return GEM_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(op.q) & 15) || (op.ldq & 3)) return GEM_ERR_MISALIGNED;  // vector loads of q
    if (static_cast<uint64_t>(op.B) * op.n_kv * op.cache_cap >= (1ull << 31)) return GEM_ERR_UNSUPPORTED_SHAPE;
    return GEM_OK;
}

gem_status attn_enqueue(const AttnOp& op, cudaStream_t stream) { return attn_launch(op, stream, false, false, false); }
gem_status attn_enqueue_in_chain(const AttnOp& op, cudaStream_t stream) {
    return attn_launch(op, stream, true, false, false);
}
bool attn_fusable(int n_q, int n_kv, int d) { return n_kv > 0 && n_q % n_kv == 0 && use_flash(n_q, n_kv, d); }
gem_status attn_enqueue_fused(const AttnOp& op, cudaStream_t stream) { return attn_launch(op, stream, true, true, true); }
// The fused form as a stand-alone call: nothing is read before griddepcontrol.wait.
gem_status attn_enqueue_fused_standalone(const AttnOp& op, cudaStream_t stream) {
    return attn_launch(op, stream, false, true, false);
}

// ---- split-partial scratch owned by the library (gem_gqa_decode_attn_noalloc) --------------
// One fixed array per device (a module-scope __device__ variable exists once in every device
// context), shared by all calls on that device.  The split kernels write every partial state
// that the merge kernel then reads, so no part of it has to start at zero.
static __device__ __align__(256) float g_attn_noalloc_scratch[GEM_ATTN_NOALLOC_SCRATCH_BYTES / sizeof(float)];

namespace {
constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kNoallocMaxDevices];
}  // namespace

// Device address of the current device's scratch array, looked up on the first call made
// with that device current (the look-up is the only set-up; it allocates nothing).
gem_status noalloc_scratch(void** out) {
    int dev = 0;
    GEM_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kNoallocMaxDevices) return GEM_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_attn_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e);
        if (!p) return cuda_fail(cudaErrorInvalidSymbol);
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return GEM_OK;
}

}  // namespace gem

extern "C" {

size_t gem_gqa_decode_attn_workspace(int B, int n_q, int n_kv, int d, int64_t cache_cap, int window) {
    return gem::attn_workspace_bytes(B, n_q, n_kv, d, cache_cap, window);
}

gem_status gem_gqa_decode_attn(const float* q, int64_t ldq, const uint16_t* k_cache, const uint16_t* v_cache, int B,
                               int n_q, int n_kv, int d, int64_t cache_cap, const int32_t* pos, int window,
                               float scale, float* out, int64_t ldo, void* workspace, size_t ws_bytes,
                               int32_t* status, void* stream) {
    gem::AttnOp op{};
    op.q = q;
    op.ldq = ldq;
    op.k_cache = k_cache;
    op.v_cache = v_cache;
    op.B = B;
    op.n_q = n_q;
    op.n_kv = n_kv;
    op.d = d;
    op.cache_cap = cache_cap;
    op.pos = pos;
    op.window = window;
    op.scale = scale;
    op.out = out;
    op.ldo = ldo;
    op.workspace = workspace;
    op.ws_bytes = ws_bytes;
    op.status = status;
    return gem::attn_enqueue(op, static_cast<cudaStream_t>(stream));
}

gem_status gem_gqa_decode_attn_fused(const float* qkv, int64_t ldqkv, int B, int n_q, int n_kv, int d,
                                     const float* gamma_q, const float* gamma_k, int v_mode, float eps,
                                     const int32_t* pos, float theta, int rope_dim, uint16_t* k_cache,
                                     uint16_t* v_cache, int64_t cache_cap, int window, float scale, float* out,
                                     int64_t ldo, void* workspace, size_t ws_bytes, int32_t* status,
                                     void* stream_v) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    gem::RopeOp rope{};
    rope.qkv = const_cast<float*>(qkv);
    rope.ldqkv = ldqkv;
    rope.B = B;
    rope.n_q = n_q;
    rope.n_kv = n_kv;
    rope.d = d;
    rope.gamma_q = gamma_q;
    rope.gamma_k = gamma_k;
    rope.v_mode = v_mode;
    rope.eps = eps;
    rope.pos = pos;
    rope.theta = theta;
    rope.rope_dim = rope_dim;
    rope.k_cache = k_cache;
    rope.v_cache = v_cache;
    rope.cache_cap = cache_cap;
    rope.window = window;
    rope.status = status;
    gem::AttnOp op{};
    op.q = qkv;
    op.ldq = ldqkv;
    op.k_cache = k_cache;
    op.v_cache = v_cache;
    op.B = B;
    op.n_q = n_q;
    op.n_kv = n_kv;
    op.d = d;
    op.cache_cap = cache_cap;
    op.pos = pos;
    op.window = window;
    op.scale = scale;
    op.out = out;
    op.ldo = ldo;
    op.workspace = workspace;
    op.ws_bytes = ws_bytes;
    op.status = status;
    gem_status st;
    if ((st = gem::rope_check(rope)) != GEM_OK || (st = gem::attn_check(op)) != GEM_OK) return st;
    if (B == 0 || n_q == 0) return GEM_OK;
    if (gem::attn_fusable(n_q, n_kv, d)) {
        op.gamma_q = gamma_q;
        op.gamma_k = gamma_k;
        op.eps = eps;
        op.theta = theta;
        op.rope_dim = rope_dim;
        op.v_mode = v_mode;
        op.k_out = k_cache;
        op.v_out = v_cache;
        return gem::attn_enqueue_fused_standalone(op, stream);
    }
    // other shapes: the QK-norm / RoPE / append launch, then attention (as the layer chain does)
    if (gem::attn_workspace_bytes(B, n_q, n_kv, d, cache_cap, window) > ws_bytes ||
        (gem::attn_workspace_bytes(B, n_q, n_kv, d, cache_cap, window) && !workspace))
        return GEM_ERR_WORKSPACE;
    if ((st = gem::rope_enqueue(rope, stream)) != GEM_OK) return st;
    return gem::attn_enqueue_in_chain(op, stream);
}

size_t gem_gqa_decode_attn_compact_workspace(int B, int n_q, int n_kv, int d, int64_t cache_cap, int rope_dim) {
    return gem::compact_workspace_bytes(B, n_q, n_kv, d, cache_cap, rope_dim);
}

gem_status gem_gqa_decode_attn_compact(const float* q, int64_t ldq, const uint16_t* v_cache, int B, int n_q,
                                       int n_kv, int d, int64_t cache_cap, const int32_t* pos, float scale,
                                       const float* gamma_k, int rope_dim, float theta, float* out, int64_t ldo,
                                       void* workspace, size_t ws_bytes, int32_t* status, void* stream) {
    gem::CompactAttnOp op{};
    op.q = q;
    op.ldq = ldq;
    op.v_cache = v_cache;
    op.B = B;
    op.n_q = n_q;
    op.n_kv = n_kv;
    op.d = d;
    op.cache_cap = cache_cap;
    op.pos = pos;
    op.scale = scale;
    op.gamma_k = gamma_k;
    op.rope_dim = rope_dim;
    op.theta = theta;
    op.out = out;
    op.ldo = ldo;
    op.workspace = workspace;
    op.ws_bytes = ws_bytes;
    op.status = status;
    return gem::compact_enqueue(op, static_cast<cudaStream_t>(stream), false);
}

gem_status gem_gqa_decode_attn_noalloc(const float* q, int64_t ldq, const uint16_t* k_cache,
                                       const uint16_t* v_cache, int B, int n_q, int n_kv, int d,
                                       int64_t cache_cap, const int32_t* pos, int window, float scale,
                                       float* out, int64_t ldo, int32_t* status, void* stream) {
    gem::AttnOp op{};
    op.q = q;
    op.ldq = ldq;
    op.k_cache = k_cache;
    op.v_cache = v_cache;
    op.B = B;
    op.n_q = n_q;
    op.n_kv = n_kv;
    op.d = d;
    op.cache_cap = cache_cap;
    op.pos = pos;
    op.window = window;
    op.scale = scale;
    op.out = out;
    op.ldo = ldo;
    op.status = status;
    gem_status st = gem::attn_check(op);
    if (st != GEM_OK || B == 0 || n_q == 0) return st;
    void* scratch = nullptr;
    if ((st = gem::noalloc_scratch(&scratch)) != GEM_OK) return st;
    const size_t need = gem::attn_workspace_bytes(B, n_q, n_kv, d, cache_cap, window);
    if (need > GEM_ATTN_NOALLOC_SCRATCH_BYTES) return GEM_ERR_WORKSPACE;
    op.workspace = scratch;
    op.ws_bytes = GEM_ATTN_NOALLOC_SCRATCH_BYTES;
    return gem::attn_enqueue(op, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
