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
//
// GEMV schedule.  Rows come in tiles of 4 per consumer warp; the CTAs take tiles round robin.  A producer warp
// bulk-copies (cp.async.bulk, one 1-D copy per row) a tile's rows one K-chunk of 16 blocks at
// a time into a ring of shared-memory stages; the consumer warps (16 for up to two activation
// rows, else 8) each take four rows of a stage.  A warp covers four blocks per step: lane (b, m) takes codes 4m .. 4m + 3 of block b
// for each of its four rows (two 16-bit loads: a block's codes are only 2-byte aligned), with
// the four activations in one float4 shared by the rows, sums the four products and scales
// the sum by the block's d (per activation row: independent accumulators per row).  Each row's
// 32 lane sums are added by a warp reduction (fixed order) after the last chunk.
#include <algorithm>
#include <map>
#include <mutex>

#include "gem_device.cuh"

namespace gem {
namespace {

constexpr int kQ8Block = 34;
// A stage: each consumer warp's rows x one K-chunk.  Up to two activation rows: 2 rows per warp
// and chunks of 32 blocks (1088 contiguous bytes per row: short per-row runs cost HBM
// throughput); more rows: 4 rows per warp and 16-block chunks, so each activation load from L1
// serves more weights.  Either way a stage is 34,816 (16 warps) or 17,408 bytes (8 warps).
__host__ __device__ constexpr int q8_rows_per_warp(int bmax) { return bmax <= 2 ? 2 : 4; }
__host__ __device__ constexpr int q8_chunk_blocks(int bmax) { return bmax <= 2 ? 32 : 16; }
constexpr int kQ8RingBytes = 139264;   // 4 stages of 16 warps' rows, 8 of 8 warps' rows
// consumer warps (four rows of a tile each): 16 for up to two activation rows, else 8
__host__ __device__ constexpr int q8_warps(int bmax) { return bmax <= 2 ? 16 : 8; }

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
    int ns;               // ring stages
    int* status;
};

__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ uint32_t gemv_mma_lds16(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ void bar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// BMAX: the largest activation row count this instance handles (B <= BMAX at run time).
template <int BMAX>
__global__ void __launch_bounds__((q8_warps(BMAX) + 1) * 32, 1) q8_0_gemv_kernel(const Q8Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int kQ8Warps = q8_warps(BMAX);
    constexpr int kQ8RowsPerWarp = q8_rows_per_warp(BMAX);
    constexpr int kQ8ChunkBlocks = q8_chunk_blocks(BMAX);
    constexpr int kQ8TileRows = kQ8Warps * kQ8RowsPerWarp;
    constexpr uint32_t kStageBytes = kQ8TileRows * kQ8ChunkBlocks * kQ8Block;
    constexpr int kQ8MaxStages = kQ8RingBytes / kStageBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kQ8MaxStages * kStageBytes);
    uint64_t* empty = full + kQ8MaxStages;
    // up to two activation rows stay resident in shared memory for the whole call; more rows are
    // read through L1
    constexpr bool kXRes = BMAX <= 2;
    float* xs = reinterpret_cast<float*>(smem + kQ8MaxStages * kStageBytes + 2 * kQ8MaxStages * 8);
    __shared__ int any_failed;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ns = p.ns;
    const int64_t ntiles = (p.N + kQ8TileRows - 1) / kQ8TileRows;
    if (tid == 0) {
        any_failed = 0;
        for (int i = 0; i < ns; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kQ8Warps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kQ8Warps) {   // producer: (tile, chunk) stages in order
        if (lane == 0) {
            bool ok = true;
            int s = 0, slot = 0;
            uint32_t par = 1;
            for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                const int64_t r0 = t * kQ8TileRows;
                const int nr = static_cast<int>(p.N - r0 < kQ8TileRows ? p.N - r0 : kQ8TileRows);
                for (int c = 0; c < p.nchunk; ++c) {
                    if (s >= ns && !(ok = mbar_wait(&empty[slot], par, p.status))) break;
                    const int nb = min(kQ8ChunkBlocks, p.K / 32 - c * kQ8ChunkBlocks);
                    const uint32_t cb = static_cast<uint32_t>(nb * kQ8Block);   // multiple of 16 (K % 256 == 0)
                    uint8_t* dst = smem + static_cast<size_t>(slot) * kStageBytes;
                    mbar_arrive_expect_tx(&full[slot], cb * static_cast<uint32_t>(nr));
                    for (int r = 0; r < nr; ++r)
                        bulk_copy(dst + r * (kQ8ChunkBlocks * kQ8Block),
                                  p.W + (r0 + r) * p.rowbytes + static_cast<int64_t>(c) * kQ8ChunkBlocks * kQ8Block, cb,
                                  &full[slot]);
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
    if constexpr (kXRes) {
        const int n4 = p.K / 4;
        for (int bb = 0; bb < p.B; ++bb)
            for (int i = tid; i < n4; i += kQ8Warps * 32)
                reinterpret_cast<float4*>(xs + bb * p.K)[i] = __ldg(reinterpret_cast<const float4*>(p.x + bb * p.ldx) + i);
        asm volatile("bar.sync 1, %0;" ::"r"(kQ8Warps * 32) : "memory");
    }
    bool ok = true;
    int s = 0, slot = 0;
    uint32_t par = 0;
    const int B = p.B;
    const int bl = lane >> 3, m = lane & 7;   // block of a step, code quad of the block
    constexpr uint32_t kRowChunk = kQ8ChunkBlocks * kQ8Block;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int64_t r0 = t * kQ8TileRows;
        float acc[kQ8RowsPerWarp][BMAX];
#pragma unroll
        for (int rr = 0; rr < kQ8RowsPerWarp; ++rr)
#pragma unroll
            for (int b = 0; b < BMAX; ++b) acc[rr][b] = 0.f;
        for (int c = 0; c < p.nchunk; ++c) {
            const int nb = min(kQ8ChunkBlocks, p.K / 32 - c * kQ8ChunkBlocks);   // a multiple of 8
            if (ok) ok = mbar_wait(&full[slot], par, p.status);
            if (ok) {
                const uint32_t st = smem_u32(smem) + static_cast<uint32_t>(slot) * kStageBytes +
                                    static_cast<uint32_t>(kQ8RowsPerWarp * warp) * kRowChunk;
                const float4* xc = reinterpret_cast<const float4*>(p.x + static_cast<int64_t>(c) * kQ8ChunkBlocks * 32);
                const float4* xr = reinterpret_cast<const float4*>(xs + c * kQ8ChunkBlocks * 32);
                for (int blk = bl; blk < nb; blk += 4) {
                    float4 xv[BMAX];
#pragma unroll
                    for (int bb = 0; bb < BMAX; ++bb) {
                        if (bb < B) {
                            if constexpr (kXRes) xv[bb] = xr[bb * (p.K >> 2) + blk * 8 + m];
                            else xv[bb] = __ldg(xc + bb * (p.ldx >> 2) + blk * 8 + m);
                        }
                    }
#pragma unroll
                    for (int rr = 0; rr < kQ8RowsPerWarp; ++rr) {
                        const uint32_t a = st + rr * kRowChunk + blk * kQ8Block;
                        const float d = half_bits_to_float(gemv_mma_lds16(a));
                        const uint32_t c4 = gemv_mma_lds16(a + 2 + 4 * m) | (gemv_mma_lds16(a + 4 + 4 * m) << 16);
                        // each code sign-extended by moving its byte to the top and shifting back
                        const float q0 = static_cast<float>(static_cast<int>(c4 << 24) >> 24);
                        const float q1 = static_cast<float>(static_cast<int>(c4 << 16) >> 24);
                        const float q2 = static_cast<float>(static_cast<int>(c4 << 8) >> 24);
                        const float q3 = static_cast<float>(static_cast<int>(c4) >> 24);
#pragma unroll
                        for (int bb = 0; bb < BMAX; ++bb) {
                            if (bb < B) {
                                float v = q0 * xv[bb].x;
                                v = fmaf(q1, xv[bb].y, v);
                                v = fmaf(q2, xv[bb].z, v);
                                v = fmaf(q3, xv[bb].w, v);
                                acc[rr][bb] = fmaf(d, v, acc[rr][bb]);
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
#pragma unroll
        for (int rr = 0; rr < kQ8RowsPerWarp; ++rr) {
            const int64_t n = r0 + kQ8RowsPerWarp * warp + rr;
#pragma unroll
            for (int bb = 0; bb < BMAX; ++bb) {
                if (bb < B) {
                    const float v = warp_sum(acc[rr][bb]);
                    if (lane == 0 && n < p.N) p.y[bb * p.ldy + n] = v;
                }
            }
        }
    }
    // a wait that gave up: the copies of the last stages still get a bounded chance to land
    // before the CTA exits
    if (!ok) atomicOr(&any_failed, 1);
    asm volatile("bar.sync 1, %0;" ::"r"(kQ8Warps * 32) : "memory");
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
    const int bmax = B <= 1 ? 1 : (B <= 2 ? 2 : (B <= 4 ? 4 : 8));
    p.nchunk = static_cast<int>((K / 32 + q8_chunk_blocks(bmax) - 1) / q8_chunk_blocks(bmax));
    p.status = di.status_word;
    const int nw = q8_warps(bmax);
    const size_t stage = static_cast<size_t>(nw) * q8_rows_per_warp(bmax) * q8_chunk_blocks(bmax) * kQ8Block;
    p.ns = static_cast<int>(kQ8RingBytes / stage);
    // the ring, its barriers (sized for the most stages any instance has), then x for up to two rows
    const size_t stage8 = static_cast<size_t>(q8_warps(8)) * q8_rows_per_warp(8) * q8_chunk_blocks(8) * kQ8Block;
    const size_t smem = kQ8RingBytes + 2 * (kQ8RingBytes / std::min(stage, stage8)) * 8 +
                        (bmax <= 2 ? static_cast<size_t>(bmax) * K * 4 : 0);
    if (smem > di.smem_optin) return GEM_ERR_UNSUPPORTED_SHAPE;
    const void* fn = bmax == 1 ? reinterpret_cast<const void*>(q8_0_gemv_kernel<1>)
                     : bmax == 2 ? reinterpret_cast<const void*>(q8_0_gemv_kernel<2>)
                     : bmax == 4 ? reinterpret_cast<const void*>(q8_0_gemv_kernel<4>)
                                 : reinterpret_cast<const void*>(q8_0_gemv_kernel<8>);
    if ((st = ensure_smem_q8(fn, di.device, smem)) != GEM_OK) return st;
    const int64_t ntiles = (N + nw * q8_rows_per_warp(bmax) - 1) / (nw * q8_rows_per_warp(bmax));
    const int grid = static_cast<int>(std::min<int64_t>(ntiles, di.num_sms));
    void* args[] = {&p};
    return launch_pdl(fn, dim3(grid), dim3((nw + 1) * 32), smem, static_cast<cudaStream_t>(stream), args);
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
