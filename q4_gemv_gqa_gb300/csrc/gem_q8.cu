// gem_q8.cu — the tied Q8_0 embedding / logit projection (dequantise-and-matvec) and the
// device argmax over the logits.
//
// "gem" engine research record, "Verified model facts": the published layout keeps the token
// embedding, tied with the output projection, as Q8_0 (5,376 x 262,144 for the 31B model);
// the research record then measures the Q8 logit matvec for one token and a fixed-eight-row
// form for a verifier, and picks the next token by argmax with ties to the lowest token id.
//
// Q8_0 record (GGML): 34 bytes = binary16 scale d (little endian), then 32 int8 codes q;
// weight j = q[j] * d.
#include <algorithm>
#include <map>
#include <mutex>

#include "gem_device.cuh"

namespace gem {
namespace {

constexpr int kQ8Block = 34;

struct Q8Params {
    const uint8_t* W;
    int64_t N;
    int K;                // weights per row (multiple of 256)
    int64_t rowbytes;     // K / 32 * 34
    const float* x;
    int64_t ldx;
    int B;
    float* y;
    int64_t ldy;
    int nchunk;           // K-chunks per row
    int* status;
};

__device__ __forceinline__ void bar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// ---- the GEMV on tensor cores, 1..8 activation rows ------------------------------------------
// A stage is 128 weight rows (eight m16 tiles) x 8 blocks (272 bytes of each row), one 2-D TMA
// box: one copy per stage, where one bulk copy per row bounded the stream by the producer's
// issue rate.  In shared memory the box rows are 272 bytes apart, so the lanes g = 0..7 of a
// load land on distinct banks.  Consumer warp w takes block w of the stage for all eight m16
// tiles: the activation operand it builds serves 8 x 4 mma, and the activation rows are read
// once per 128 weight rows.  k16 tile j of a block gives lane quad t the four consecutive codes
// 16 j + 4 t .. + 3 (codes 0-1 sit at k = 2t, 2t+1 of the A fragment, codes 2-3 at k = 2t+8,
// 2t+9), and B column n holds activation row n at the same four positions.  Codes become exact
// binary16 values: the byte biased by 128 is placed under the exponent of 1024 by a byte
// permute, then 1152 is subtracted.  Each activation row is scaled by one power of two (its
// largest magnitude to [2^13, 2^14)) and split into binary16 hi + lo, one mma each.  The two mma
// of a k16 tile start from zero and their sum is scaled by the row's d into the tile
// accumulator (short chains); after the last stage of a row tile the warps' sums are added in a
// fixed order through shared memory and the row's power of two is undone.
constexpr int kQ8mWarps = 8;
constexpr int kQ8mTiles = 8;                                    // m16 tiles per stage
constexpr int kQ8mRows = 16 * kQ8mTiles;
constexpr int kQ8mChunk = 8;                                    // blocks per stage row
constexpr int kQ8mBpw = kQ8mChunk / kQ8mWarps;                  // blocks of a chunk per warp
constexpr int kQ8mBoxBlocks = 8;                                // blocks per TMA box row (272 bytes)
constexpr int kQ8mBoxPitch = kQ8mBoxBlocks * kQ8Block;          // 272
constexpr uint32_t kQ8mBoxBytes = kQ8mRows * kQ8mBoxPitch;      // 8,704
constexpr uint32_t kQ8mStage = (kQ8mChunk / kQ8mBoxBlocks) * kQ8mBoxBytes;   // 34,816
constexpr int kQ8mStages = 4;
constexpr uint32_t kQ8mRedFloats = kQ8mWarps * kQ8mTiles * 4 * 32;   // one buffer: [warp][tile * 4 + e][lane]
constexpr size_t kQ8mSmem = kQ8mStages * kQ8mStage + 2 * kQ8mStages * 8 + 2 * kQ8mRedFloats * 4 + 16 * 4;

__device__ __forceinline__ void mma_16816_zero(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// Four int8 codes (the bytes of w, lowest first) as two exact binary16 pairs (c0, c1), (c2, c3).
__device__ __forceinline__ void q8_codes_half2(uint32_t w, uint32_t& h01, uint32_t& h23) {
    const uint32_t u = w ^ 0x80808080u;   // code + 128 as an unsigned byte
    uint32_t p01, p23;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(p01) : "r"(u), "r"(0x64646464u));   // (1024 + u0, 1024 + u1)
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(p23) : "r"(u), "r"(0x64646464u));   // (1024 + u2, 1024 + u3)
    const uint32_t bias = 0x64806480u;                                              // (1152, 1152)
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(h01) : "r"(p01), "r"(bias));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(h23) : "r"(p23), "r"(bias));
}

// Four activations as binary16 hi + lo pairs: hi = (v0, v1), (v2, v3) rounded; lo the remainders.
__device__ __forceinline__ void q8_split4(float4 v, uint32_t (&hi)[2], uint32_t (&lo)[2]) {
    const __half2 h01 = __floats2half2_rn(v.x, v.y), h23 = __floats2half2_rn(v.z, v.w);
    const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
    const __half2 l01 = __floats2half2_rn(v.x - f01.x, v.y - f01.y), l23 = __floats2half2_rn(v.z - f23.x, v.w - f23.y);
    hi[0] = *reinterpret_cast<const uint32_t*>(&h01);
    hi[1] = *reinterpret_cast<const uint32_t*>(&h23);
    lo[0] = *reinterpret_cast<const uint32_t*>(&l01);
    lo[1] = *reinterpret_cast<const uint32_t*>(&l23);
}

__global__ void __launch_bounds__((kQ8mWarps + 1) * 32, 1) q8_0_gemv_mma_kernel(const __grid_constant__ CUtensorMap tm,
                                                                              const Q8Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kQ8mStages * kQ8mStage);
    uint64_t* empty = full + kQ8mStages;
    float* red = reinterpret_cast<float*>(smem + kQ8mStages * kQ8mStage + 2 * kQ8mStages * 8);
    float* rsc = red + 2 * kQ8mRedFloats;   // [8] 2^e of each activation row, [8..16) 2^-e
    __shared__ int any_failed;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int ns = kQ8mStages;
    const int64_t ntiles = (p.N + kQ8mRows - 1) / kQ8mRows;
    const int nblk = p.K / 32;
    if (tid == 0) {
        any_failed = 0;
        for (int i = 0; i < ns; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kQ8mWarps);
        }
        fence_mbar_init();
        prefetch_tensormap(&tm);
    }
    __syncthreads();

    if (warp == kQ8mWarps) {   // producer: (tile, chunk) stages in order
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_first();
            bool ok = true;
            int s = 0, slot = 0;
            uint32_t par = 1;
            for (int64_t tl = blockIdx.x; tl < ntiles && ok; tl += gridDim.x) {
                const int64_t r0 = tl * kQ8mRows;
                for (int c = 0; c < p.nchunk; ++c) {
                    if (s >= ns && !(ok = mbar_wait(&empty[slot], par, p.status))) break;
                    // boxes of 8 blocks (K % 256 == 0: whole boxes); rows past N arrive as zeros
                    // and count toward the bytes like the others
                    const int nbox = min(kQ8mChunk, nblk - c * kQ8mChunk) / kQ8mBoxBlocks;
                    uint8_t* dst = smem + static_cast<size_t>(slot) * kQ8mStage;
                    mbar_arrive_expect_tx(&full[slot], kQ8mBoxBytes * static_cast<uint32_t>(nbox));
                    for (int q = 0; q < nbox; ++q)   // x in 16-bit units (17 per block): a multiple of 8
                        tma_load_2d(dst + q * kQ8mBoxBytes, &tm, (c * kQ8mChunk + q * kQ8mBoxBlocks) * (kQ8Block / 2),
                                    static_cast<int32_t>(r0), &full[slot], policy);
                    ++s;
                    if (++slot == ns) {
                        slot = 0;
                        par ^= 1u;
                    }
                }
            }
            if (!ok) drain_stages(full, ns, max(0, s - ns), s - 1);
        }
        return;   // the producer warp never triggers dependents: the consumers do, after their wait
    }

    pdl_wait_trigger();   // the activations come from the previous kernel
    const int B = p.B;
    // per activation row: the power of two taking its largest magnitude to [2^13, 2^14)
    if (warp < 8) {
        float m = 0.f;
        if (warp < B) {
            const float4* xr = reinterpret_cast<const float4*>(p.x + warp * p.ldx);
            const int n4 = p.K / 4;
            for (int i0 = lane; i0 < n4; i0 += 32 * 6) {
                float4 v[6];
#pragma unroll
                for (int u = 0; u < 6; ++u)
                    v[u] = i0 + 32 * u < n4 ? __ldg(xr + i0 + 32 * u) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int u = 0; u < 6; ++u)
                    m = fmaxf(m, fmaxf(fmaxf(fabsf(v[u].x), fabsf(v[u].y)), fmaxf(fabsf(v[u].z), fabsf(v[u].w))));
            }
            m = warp_max(m);
        }
        int e = 0;
        if (m > 0.f) e = 13 - (((__float_as_int(m) >> 23) & 0xff) - 127);
        e = max(-126, min(126, e));
        if (lane == 0) {
            rsc[warp] = __int_as_float((127 + e) << 23);
            rsc[8 + warp] = __int_as_float((127 - e) << 23);
        }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kQ8mWarps * 32) : "memory");

    const int g = lane >> 2, t = lane & 3;
    const bool xrow = g < B;                  // B column g is a real activation row
    const float sg = rsc[g];
    const float* xg = p.x + (xrow ? g : 0) * p.ldx + 4 * t;
    bool ok = true;
    int s = 0, slot = 0;
    uint32_t par = 0;
    int it = 0;
    for (int64_t tl = blockIdx.x; tl < ntiles; tl += gridDim.x, ++it) {
        const int64_t r0 = tl * kQ8mRows;
        float acc[kQ8mTiles][4];
#pragma unroll
        for (int mt = 0; mt < kQ8mTiles; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
        for (int c = 0; c < p.nchunk; ++c) {
            const int nb = min(kQ8mChunk, nblk - c * kQ8mChunk);   // a multiple of 8: the same count per warp
            // this warp's activations for the chunk, requested before the stage wait
            float4 xv[kQ8mBpw][2];
#pragma unroll
            for (int i = 0; i < kQ8mBpw; ++i) {
                const int blk = warp + kQ8mWarps * i;
                const float* xb = xg + (c * kQ8mChunk + blk) * 32;
                const bool in = xrow && blk < nb;
                xv[i][0] = in ? __ldg(reinterpret_cast<const float4*>(xb)) : make_float4(0.f, 0.f, 0.f, 0.f);
                xv[i][1] = in ? __ldg(reinterpret_cast<const float4*>(xb + 16)) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            if (ok) ok = mbar_wait(&full[slot], par, p.status);
            if (ok) {
                const uint8_t* st = smem + static_cast<size_t>(slot) * kQ8mStage;
#pragma unroll
                for (int i = 0; i < kQ8mBpw; ++i) {
                    const int blk = warp + kQ8mWarps * i;
                    if (blk < nb) {
                        uint32_t bh[2][2], bl[2][2];
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            float4 v = xv[i][j];
                            v.x *= sg; v.y *= sg; v.z *= sg; v.w *= sg;
                            q8_split4(v, bh[j], bl[j]);
                        }
#pragma unroll
                        for (int mt = 0; mt < kQ8mTiles; ++mt) {
                            // rows g and g + 8 of m16 tile mt (plain loads: the stage wait above
                            // orders them after the copy)
                            const uint16_t* ra = reinterpret_cast<const uint16_t*>(
                                st + (blk / kQ8mBoxBlocks) * kQ8mBoxBytes + (mt * 16 + g) * kQ8mBoxPitch +
                                (blk % kQ8mBoxBlocks) * kQ8Block);
                            const uint16_t* rb = ra + 8 * kQ8mBoxPitch / 2;
                            const float dg = half_bits_to_float(ra[0]);
                            const float dg8 = half_bits_to_float(rb[0]);
#pragma unroll
                            for (int j = 0; j < 2; ++j) {
                                const int o = 1 + 8 * j + 2 * t;   // in 16-bit units
                                const uint32_t wg = ra[o] | (static_cast<uint32_t>(ra[o + 1]) << 16);
                                const uint32_t wg8 = rb[o] | (static_cast<uint32_t>(rb[o + 1]) << 16);
                                uint32_t a0, a1, a2, a3;
                                q8_codes_half2(wg, a0, a2);
                                q8_codes_half2(wg8, a1, a3);
                                float cj[4];
                                mma_16816_zero(cj, a0, a1, a2, a3, bh[j][0], bh[j][1]);
                                mma_16816(cj, a0, a1, a2, a3, bl[j][0], bl[j][1]);
                                acc[mt][0] = fmaf(dg, cj[0], acc[mt][0]);
                                acc[mt][1] = fmaf(dg, cj[1], acc[mt][1]);
                                acc[mt][2] = fmaf(dg8, cj[2], acc[mt][2]);
                                acc[mt][3] = fmaf(dg8, cj[3], acc[mt][3]);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) bar_arrive(&empty[slot]);
            ++s;
            if (++slot == ns) {
                slot = 0;
                par ^= 1u;
            }
        }
        // the warps' sums, added in warp order (two buffers: one barrier per tile)
        float* rb = red + (it & 1) * kQ8mRedFloats;
#pragma unroll
        for (int mt = 0; mt < kQ8mTiles; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) rb[(warp * kQ8mTiles * 4 + mt * 4 + e) * 32 + lane] = acc[mt][e];
        asm volatile("bar.sync 1, %0;" ::"r"(kQ8mWarps * 32) : "memory");
        for (int o = tid; o < kQ8mTiles * 4 * 32; o += kQ8mWarps * 32) {
            const int q = o >> 5, ln = o & 31;   // q = tile * 4 + e
            float v = 0.f;
            for (int w = 0; w < kQ8mWarps; ++w) v += rb[(w * kQ8mTiles * 4 + q) * 32 + ln];
            const int e = q & 3;
            const int64_t row = r0 + (q >> 2) * 16 + (ln >> 2) + (e >> 1) * 8;
            const int bcol = 2 * (ln & 3) + (e & 1);
            if (bcol < B && row < p.N) p.y[bcol * p.ldy + row] = v * rsc[8 + bcol];
        }
    }
    // a wait that gave up: the copies of the last stages still get a bounded chance to land
    // before the CTA exits
    if (!ok) atomicOr(&any_failed, 1);
    asm volatile("bar.sync 1, %0;" ::"r"(kQ8mWarps * 32) : "memory");
    if (any_failed && tid == 0) drain_stages(full, ns, max(0, s - ns), s - 1);
}

// ---- argmax ------------------------------------------------------------------------------
// Index of the largest value of each row (lowest index on ties; NaN never chosen; all NaN -> 0).
// CTA (c, b) reduces chunk c of row b and publishes (value, index); the CTA that takes the
// last ticket of row b's arrival counter combines the chunks and resets the counter.
constexpr int kArgThreads = 256;

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    return i >= 0 && (bi < 0 || v > bv || (v == bv && i < bi));
}

__global__ void __launch_bounds__(kArgThreads) argmax_kernel(const float* y, int64_t ldy, int64_t N, int32_t* out,
                                                            float2* part, unsigned* cnt) {
    __shared__ float sv[kArgThreads / 32];
    __shared__ int si[kArgThreads / 32];
    __shared__ int last_sh;
    pdl_wait_trigger();
    const int c = blockIdx.x, b = blockIdx.y, nchunk = gridDim.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float* row = y + b * ldy;
    const int64_t lo = (N * c) / nchunk, hi = (N * (c + 1)) / nchunk;
    float bv = 0.f;
    int bi = -1;
#pragma unroll 8
    for (int64_t i = lo + tid; i < hi; i += kArgThreads) {   // increasing i: ties keep the first
        const float v = __ldg(row + i);
        if (!isnan(v) && (bi < 0 || v > bv)) {
            bv = v;
            bi = static_cast<int>(i);
        }
    }
    auto reduce = [&](float& v, int& i) {   // warp: best (v, i) over the lanes
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, v, o);
            const int oi = __shfl_xor_sync(0xffffffffu, i, o);
            if (better(ov, oi, v, i)) {
                v = ov;
                i = oi;
            }
        }
    };
    reduce(bv, bi);
    if (lane == 0) {
        sv[warp] = bv;
        si[warp] = bi;
    }
    __syncthreads();
    if (warp == 0) {
        float v = lane < kArgThreads / 32 ? sv[lane] : 0.f;
        int i = lane < kArgThreads / 32 ? si[lane] : -1;
        reduce(v, i);
        if (lane == 0) {
            part[static_cast<int64_t>(b) * nchunk + c] = make_float2(v, __int_as_float(i));
            unsigned ticket;
            asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(ticket) : "l"(cnt + b) : "memory");
            last_sh = ticket == static_cast<unsigned>(nchunk - 1);
        }
    }
    __syncthreads();
    if (!last_sh) return;
    float v = 0.f;
    int i = -1;
    for (int k = tid; k < nchunk; k += kArgThreads) {
        const float2 pv = __ldcg(part + static_cast<int64_t>(b) * nchunk + k);
        if (better(pv.x, __float_as_int(pv.y), v, i)) {
            v = pv.x;
            i = __float_as_int(pv.y);
        }
    }
    reduce(v, i);
    __syncthreads();
    if (lane == 0) {
        sv[warp] = v;
        si[warp] = i;
    }
    __syncthreads();
    if (tid == 0) {
        float bv2 = 0.f;
        int bi2 = -1;
        for (int w = 0; w < kArgThreads / 32; ++w)
            if (better(sv[w], si[w], bv2, bi2)) {
                bv2 = sv[w];
                bi2 = si[w];
            }
        out[b] = bi2 < 0 ? 0 : bi2;
        cnt[b] = 0u;   // ready for the next call
    }
}

// chunks of 2048 values (8 per thread): about one CTA per SM at the 262,144-entry vocabulary
// ---- top-k ---------------------------------------------------------------------------------
// The k (<= 64) largest entries of each row, largest first, ties by lowest index, NaN after every
// number (by index).  Each entry becomes one 64-bit key whose order is that order: the high word
// maps the float to an unsigned integer in value order (NaN to 0, below -inf), the low word is the
// inverted index.  A warp selects k keys by k rounds of a warp maximum over the keys its lanes
// hold (the winner's lane clears its key); warp 0 merges the warps' lists the same way; a CTA
// publishes its chunk's list and the CTA taking the last ticket merges the chunks' lists.
constexpr int kTopkMax = 64;
constexpr int kTopkThreads = 256;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkMerge = 2048;   // the chunks' lists together: at most this many keys

__device__ __forceinline__ uint64_t topk_key(float v, int64_t i) {
    uint32_t u = __float_as_uint(v);
    u = isnan(v) ? 0u : ((u & 0x80000000u) ? ~u : (u | 0x80000000u));
    return (static_cast<uint64_t>(u) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(i));
}
__device__ __forceinline__ int topk_index(uint64_t key) { return static_cast<int>(~static_cast<uint32_t>(key)); }

// Each lane sorts its keys in descending order once (a bitonic network over register indices
// known at compile time); then k rounds: the warp maximum of the lanes' first keys is written
// (lane 0) to out[r] and its holder shifts its list by one.  A key of 0 is "nothing" (every real
// key has a nonzero low word).
template <int NPL>
__device__ __forceinline__ void topk_sort_desc(uint64_t (&a)[NPL]) {
#pragma unroll
    for (int k = 2; k <= NPL; k <<= 1)
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1)
#pragma unroll
            for (int i = 0; i < NPL; ++i) {
                const int l = i ^ j;
                if (l > i) {
                    const uint64_t x = a[i], y = a[l];
                    const bool swap = (i & k) == 0 ? x < y : x > y;   // descending runs first
                    a[i] = swap ? y : x;
                    a[l] = swap ? x : y;
                }
            }
}

template <int NPL>
__device__ __forceinline__ void topk_warp_select(uint64_t (&key)[NPL], int k, uint64_t* out, int lane) {
    topk_sort_desc<NPL>(key);
    for (int r = 0; r < k; ++r) {
        uint64_t best = key[0];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const uint64_t other = __shfl_xor_sync(0xffffffffu, best, o);
            best = other > best ? other : best;
        }
        const bool won = key[0] == best;
#pragma unroll
        for (int u = 0; u + 1 < NPL; ++u) key[u] = won ? key[u + 1] : key[u];
        if (won) key[NPL - 1] = 0;
        if (lane == 0) out[r] = best;
    }
}

// the CTA's k largest of the keys its threads hold, into res[0, k) (shared); cand: [warps][64]
template <int NPL>
__device__ __forceinline__ void topk_cta(uint64_t (&key)[NPL], int k, uint64_t* cand, uint64_t* res, int tid) {
    const int lane = tid & 31, warp = tid >> 5;
    topk_warp_select<NPL>(key, k, cand + warp * kTopkMax, lane);
    __syncthreads();
    if (warp == 0) {
        constexpr int M = kTopkWarps * kTopkMax / 32;
        uint64_t mk[M];
#pragma unroll
        for (int u = 0; u < M; ++u) {
            const int e = lane + 32 * u, w = e / kTopkMax, r = e - w * kTopkMax;
            mk[u] = r < k ? cand[w * kTopkMax + r] : 0ull;
        }
        topk_warp_select<M>(mk, k, res, lane);
    }
    __syncthreads();
}

template <int VPT>
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float* y, int64_t ldy, int64_t N, int k,
                                                            uint64_t* part, unsigned* cnt, int32_t* idx, float* val) {
    __shared__ uint64_t cand[kTopkWarps * kTopkMax];
    __shared__ uint64_t res[kTopkMax];
    __shared__ int last_sh;
    pdl_wait_trigger();
    const int c = blockIdx.x, b = blockIdx.y, nchunk = gridDim.x;
    const int tid = threadIdx.x;
    const float* row = y + b * ldy;
    const int64_t lo = (N * c) / nchunk, hi = (N * (c + 1)) / nchunk;
    uint64_t key[VPT];
#pragma unroll
    for (int u = 0; u < VPT; ++u) {   // loads first (independent)
        const int64_t i = lo + tid + static_cast<int64_t>(u) * kTopkThreads;
        key[u] = i < hi ? topk_key(__ldg(row + i), i) : 0ull;
    }
    topk_cta<VPT>(key, k, cand, res, tid);
    uint64_t* mine = part + (static_cast<int64_t>(b) * nchunk + c) * k;
    if (tid < k) mine[tid] = res[tid];
    // the barrier orders every thread's list writes before thread 0's ticket, whose release
    // (cumulative) publishes them; its acquire orders the merging CTA's reads after the tickets
    __syncthreads();
    if (tid == 0) {
        unsigned ticket;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(ticket) : "l"(cnt + b) : "memory");
        last_sh = ticket == static_cast<unsigned>(nchunk - 1);
    }
    __syncthreads();
    if (!last_sh) return;
    constexpr int MPT = kTopkMerge / kTopkThreads;
    uint64_t mk[MPT];
    const int64_t m = static_cast<int64_t>(nchunk) * k;
#pragma unroll
    for (int u = 0; u < MPT; ++u) {
        const int64_t e = tid + static_cast<int64_t>(u) * kTopkThreads;
        mk[u] = e < m ? __ldcg(reinterpret_cast<const unsigned long long*>(part) + static_cast<int64_t>(b) * m + e) : 0ull;
    }
    topk_cta<MPT>(mk, k, cand, res, tid);
    if (tid < k) {
        const int i = topk_index(res[tid]);
        idx[b * k + tid] = i;
        val[b * k + tid] = row[i];
    }
    if (tid == 0) cnt[b] = 0u;   // ready for the next call
}

// values per thread for a row of N and a list of k: the fewest (8, 16, 32) whose chunk lists fit
// the merge (nchunk * k <= 2048); 0 when none does
int topk_vpt(int64_t N, int k) {
    for (int v : {8, 16, 32}) {
        const int64_t nc = (N + 256ll * v - 1) / (256ll * v);
        if (nc * k <= kTopkMerge) return v;
    }
    return 0;
}

int argmax_chunks(int64_t N) { return static_cast<int>(std::min<int64_t>(1024, std::max<int64_t>(1, (N + 2047) / 2048))); }

gem_status ensure_smem_q8(const void* fn, int device, size_t bytes) {
    static std::mutex mu;
    static std::map<std::pair<int, const void*>, size_t> done;
    std::lock_guard<std::mutex> lk(mu);
    size_t& have = done[{device, fn}];
    if (have >= bytes) return GEM_OK;
    GEM_CUDA_TRY(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)));
    have = bytes;
    return GEM_OK;
}

}  // namespace
}  // namespace gem

extern "C" {

gem_status gem_q8_0_gemv(const void* W, int64_t N, int64_t K, const float* x, int64_t ldx, int B, float* y,
                         int64_t ldy, void* stream) {
    using namespace gem;
    if (B < 0 || N < 0 || K < 0) return GEM_ERR_INVALID_ARG;
    if (B > 8 || K % 256 || K > (int64_t(1) << 30)) return GEM_ERR_UNSUPPORTED_SHAPE;
    if (B == 0 || N == 0) return GEM_OK;
    if (!W || !x || !y || K == 0) return GEM_ERR_INVALID_ARG;
    if (ldx < K || ldy < N) return GEM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(W) & 15) || (reinterpret_cast<uintptr_t>(x) & 15) || (ldx & 3) ||
        (reinterpret_cast<uintptr_t>(y) & 3))
        return GEM_ERR_MISALIGNED;
    DeviceInfo di;
    gem_status st;
    if ((st = device_info(&di)) != GEM_OK) return st;
    Q8Params p{};
    p.W = static_cast<const uint8_t*>(W);
    p.N = N;
    p.K = static_cast<int>(K);
    p.rowbytes = K / 32 * kQ8Block;
    p.x = x;
    p.ldx = ldx;
    p.B = B;
    p.y = y;
    p.ldy = ldy;
    p.status = di.status_word;
    p.nchunk = static_cast<int>((K / 32 + kQ8mChunk - 1) / kQ8mChunk);
    if (kQ8mSmem > di.smem_optin) return GEM_ERR_UNSUPPORTED_SHAPE;
    // the matrix as 16-bit elements: rows of K / 32 * 17, boxes of 8 blocks x the tile's rows
    CUtensorMap tm;
    if ((st = make_tensor_map_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT16, W, static_cast<uint64_t>(p.rowbytes / 2),
                                 static_cast<uint64_t>(N), static_cast<uint64_t>(p.rowbytes), kQ8mBoxPitch / 2,
                                 kQ8mRows, CU_TENSOR_MAP_SWIZZLE_NONE)) != GEM_OK)
        return st;
    const void* fn = reinterpret_cast<const void*>(q8_0_gemv_mma_kernel);
    if ((st = ensure_smem_q8(fn, di.device, kQ8mSmem)) != GEM_OK) return st;
    const int64_t ntiles = (N + kQ8mRows - 1) / kQ8mRows;
    const int grid = static_cast<int>(std::min<int64_t>(ntiles, di.num_sms));
    void* args[] = {&tm, &p};
    return launch_pdl(fn, dim3(grid), dim3((kQ8mWarps + 1) * 32), kQ8mSmem, static_cast<cudaStream_t>(stream), args);
}

size_t gem_argmax_workspace(int B, int64_t N) {
    if (B <= 0 || N <= 0) return 0;
    const int nc = gem::argmax_chunks(N);
    return gem::align_up(static_cast<size_t>(B) * nc * sizeof(float2), 256) +
           gem::align_up(static_cast<size_t>(B) * sizeof(unsigned), 256);
}

size_t gem_topk_workspace(int B, int64_t N, int k) {
    if (B <= 0 || N <= 0 || k < 1 || k > gem::kTopkMax || k > N) return 0;
    const int v = gem::topk_vpt(N, k);
    if (!v) return 0;
    const int64_t nc = (N + 256ll * v - 1) / (256ll * v);
    return gem::align_up(static_cast<size_t>(B) * nc * k * sizeof(uint64_t), 256) +
           gem::align_up(static_cast<size_t>(B) * sizeof(unsigned), 256);
}

gem_status gem_topk(const float* y, int64_t ldy, int B, int64_t N, int k, int32_t* idx, float* val, void* workspace,
                    size_t ws_bytes, void* stream_v) {
    using namespace gem;
    if (B < 0 || N < 0 || k < 1 || k > N) return GEM_ERR_INVALID_ARG;
    if (k > kTopkMax || N >= (int64_t(1) << 31)) return GEM_ERR_UNSUPPORTED_SHAPE;
    if (B == 0) return GEM_OK;
    if (!y || !idx || !val || ldy < N) return GEM_ERR_INVALID_ARG;
    const int v = topk_vpt(N, k);
    if (!v) return GEM_ERR_UNSUPPORTED_SHAPE;
    const size_t need = gem_topk_workspace(B, N, k);
    if (!workspace || ws_bytes < need) return GEM_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return GEM_ERR_MISALIGNED;
    const int nc = static_cast<int>((N + 256ll * v - 1) / (256ll * v));
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    uint64_t* part = static_cast<uint64_t*>(workspace);
    unsigned* cnt = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) +
                                                align_up(static_cast<size_t>(B) * nc * k * sizeof(uint64_t), 256));
    GEM_CUDA_TRY(cudaMemsetAsync(cnt, 0, sizeof(unsigned) * B, stream));
    void* args[] = {const_cast<float**>(&y), &ldy, &N, &k, &part, &cnt, &idx, &val};
    const void* fn = v == 8 ? reinterpret_cast<const void*>(topk_kernel<8>)
                     : v == 16 ? reinterpret_cast<const void*>(topk_kernel<16>)
                               : reinterpret_cast<const void*>(topk_kernel<32>);
    return launch_pdl(fn, dim3(nc, B), dim3(kTopkThreads), 0, stream, args);
}

gem_status gem_argmax(const float* y, int64_t ldy, int B, int64_t N, int32_t* idx, void* workspace, size_t ws_bytes,
                      void* stream_v) {
    using namespace gem;
    if (B < 0 || N < 0) return GEM_ERR_INVALID_ARG;
    if (B == 0) return GEM_OK;
    if (!y || !idx || ldy < N || N >= (int64_t(1) << 31)) return N >= (int64_t(1) << 31) ? GEM_ERR_UNSUPPORTED_SHAPE
                                                                                        : GEM_ERR_INVALID_ARG;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    if (N == 0) {
        GEM_CUDA_TRY(cudaMemsetAsync(idx, 0, sizeof(int32_t) * B, stream));
        return GEM_OK;
    }
    const size_t need = gem_argmax_workspace(B, N);
    if (!workspace || ws_bytes < need) return GEM_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return GEM_ERR_MISALIGNED;
    const int nc = argmax_chunks(N);
    float2* part = static_cast<float2*>(workspace);
    unsigned* cnt = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) +
                                                align_up(static_cast<size_t>(B) * nc * sizeof(float2), 256));
    GEM_CUDA_TRY(cudaMemsetAsync(cnt, 0, sizeof(unsigned) * B, stream));
    void* args[] = {const_cast<float**>(&y), &ldy, &N, &idx, &part, &cnt};
    return launch_pdl(reinterpret_cast<const void*>(argmax_kernel), dim3(nc, B), dim3(kArgThreads), 0, stream, args);
}

}  // extern "C"
