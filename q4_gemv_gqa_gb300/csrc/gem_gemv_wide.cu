// gem_gemv_wide.cu — Q4_0 GEMV on tensor cores for 2..8 activation rows, one launch, tall tiles.
//
// Q4_0 ("gem" engine research record, "Verified model facts"): 18-byte blocks, binary16 scale d
// then 16 code bytes; byte j holds element j (low nibble) and element j + 16 (high nibble);
// weight = (q - 8) * d.
//
// Schedule.  A tile is 16 MT rows of each of the NMAT matrices; the CTAs take tiles round robin.
// A stage is a tile's rows x 16 blocks (two 144-byte groups), one 2-D TMA box per matrix and
// group, so a copy moves 16 MT rows at once, plus the 16 blocks' activations of the B rows (two
// more boxes, copied once the previous kernel is complete).  Consumer warp w (of 16) takes
// block w of the stage for all the tile's m16 tiles: the activation operand it builds for the
// block serves NMAT x MT x 4 mma.
//
// Fragments.  Lane quad t of a block owns code bytes 4t .. 4t + 3 of a row: their low nibbles
// (elements 4t .. 4t + 3) form k16 tile 0, their high nibbles (elements 16 + 4t ..) k16 tile 1.
// A nibble becomes an exact binary16 value under the exponent of 1024 by one lop3 and then
// q - 8 by one subtraction (or multiply-add for the high nibble); bytes 0 and 2 of the word
// give the pair at k = 2t, 2t + 1, bytes 1 and 3 the pair at k = 2t + 8, 2t + 9, so B column
// n carries activation row n's elements (4t, 4t + 2) and (4t + 1, 4t + 3) in the same slots.
// Each activation row's block of 32 is scaled by its own power of two (its largest magnitude
// to [2^13, 2^14), from the four lanes of the quad) and split into binary16 hi + lo, one mma
// each; the block's four mma start from zero and the sum is scaled by d times the inverse
// power of two of its column into the accumulator.  A fused RMSNorm multiplies the activations
// by gamma and each output by 1 / rms of its row, whose sum of squares the warps gather while
// they build the first tile's operands.  After a tile's last stage the warps' sums meet in
// shared memory in a fixed order (deterministic results).
#include <algorithm>
#include <map>
#include <mutex>

#include "gem_device.cuh"
#include "gem_gemv_mma.cuh"

namespace gem {
namespace gemv_wide {

constexpr int kWarps = 16;                 // consumer warps: one block of each stage apiece
constexpr int kBlk = 18;                   // Q4_0 block bytes
constexpr int kGroup = 8 * kBlk;           // 144: one box row (8 blocks)
constexpr int kStageBlocks = 16;           // blocks per stage row (two boxes per matrix)
constexpr int kMaxStages = 16;
constexpr int kXCols = 256;                // activations per TMA box row (8 blocks)

struct Params {
    int64_t N;
    int K;
    int nblk;                  // K / 32
    int nchunk;                // stages per tile
    int ns;                    // ring stages
    uint32_t stage;            // bytes of a stage: the weight boxes, then two activation boxes
    uint32_t xbox;             // bytes of an activation box: B rows x 256 fp32
    int B;
    const float* x;
    int64_t ldx;
    float* y;
    int64_t ldy;
    const float* residual;     // NMAT == 1, nullable
    int64_t ldr;
    const float* gamma;        // nullable: fused RMSNorm
    float eps;
    int act;                   // NMAT == 2
    int* status;
    unsigned* clear;
    int nclear;
};

template <int NMAT, int MT>
struct Shape {
    static constexpr int kRows = 16 * MT;
    static constexpr uint32_t kBox = static_cast<uint32_t>(kRows) * kGroup;        // one box
    static constexpr uint32_t kWts = NMAT * 2 * kBox;                             // weight boxes of a stage
    static constexpr int kOut = NMAT * MT * 4;                                    // accumulators per lane
    static constexpr uint32_t kRed = kWarps * kOut * 32;                          // floats per buffer
    // fixed part: barriers, the two reduction buffers and the sums of squares
    static constexpr size_t kFixed = 2 * kMaxStages * 8 + 2 * kRed * 4 + kWarps * 8 * 4;
};

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void mma_zero(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// (v.x, v.z) and (v.y, v.w) as binary16 hi pairs and their remainders.
__device__ __forceinline__ void split_pairs(float4 v, uint32_t& h0, uint32_t& h1, uint32_t& l0, uint32_t& l1) {
    const __half2 a = __floats2half2_rn(v.x, v.z), b = __floats2half2_rn(v.y, v.w);
    const float2 fa = __half22float2(a), fb = __half22float2(b);
    const __half2 la = __floats2half2_rn(v.x - fa.x, v.z - fa.y), lb = __floats2half2_rn(v.y - fb.x, v.w - fb.y);
    h0 = *reinterpret_cast<const uint32_t*>(&a);
    h1 = *reinterpret_cast<const uint32_t*>(&b);
    l0 = *reinterpret_cast<const uint32_t*>(&la);
    l1 = *reinterpret_cast<const uint32_t*>(&lb);
}

template <int NMAT, int MT>
__global__ void __launch_bounds__((kWarps + 1) * 32, 1) q4_0_gemv_wide_kernel(const __grid_constant__ CUtensorMap tm0,
                                                                              const __grid_constant__ CUtensorMap tm1,
                                                                              const __grid_constant__ CUtensorMap tmx,
                                                                              const Params p) {
    using S = Shape<NMAT, MT>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int ns = p.ns;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(ns) * p.stage);
    uint64_t* empty = full + kMaxStages;
    float* red = reinterpret_cast<float*>(full + 2 * kMaxStages);
    float* ssw = red + 2 * S::kRed;   // [warp][row]: partial sums of squares of the activation rows
    __shared__ int any_failed;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t ntiles = (p.N + S::kRows - 1) / S::kRows;
    if (tid == 0) {
        any_failed = 0;
        for (int i = 0; i < ns; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kWarps);
        }
        fence_mbar_init();
        prefetch_tensormap(&tm0);
        if (NMAT == 2) prefetch_tensormap(&tm1);
        prefetch_tensormap(&tmx);
    }
    __syncthreads();

    // producer: (tile, chunk) stages in order.  A stage is the tile's weight boxes and the
    // chunk's activation boxes (B rows x 256 values each).  The weights of the first ring's worth
    // of stages are requested before griddepcontrol.wait (nothing running writes them); the
    // activations, which the previous kernel writes, only after it.
    if (warp == kWarps) {
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_first();
            bool ok = true;
            int s = 0, slot = 0;
            uint32_t par = 1;
            const uint64_t keep = l2_policy_evict_last();   // the activations are read by every tile
            auto issue_x = [&](int sl, int c) {
                const int nbox = min(kStageBlocks, p.nblk - c * kStageBlocks) / 8;
                uint8_t* dst = smem + static_cast<size_t>(sl) * p.stage + S::kWts;
                for (int q = 0; q < nbox; ++q)
                    tma_load_2d(dst + q * p.xbox, &tmx, c * kStageBlocks * 32 + q * kXCols, 0, &full[sl], keep);
            };
            int pend[kMaxStages];   // chunk of each stage issued before the wait
            bool waited = false;
            for (int64_t tl = blockIdx.x; tl < ntiles && ok; tl += gridDim.x) {
                const int32_t r0 = static_cast<int32_t>(tl * S::kRows);
                for (int c = 0; c < p.nchunk; ++c) {
                    if (s >= ns && !(ok = mbar_wait(&empty[slot], par, p.status))) break;
                    const int nbox = min(kStageBlocks, p.nblk - c * kStageBlocks) / 8;   // 1 or 2 (K % 256 == 0)
                    uint8_t* dst = smem + static_cast<size_t>(slot) * p.stage;
                    mbar_arrive_expect_tx(&full[slot], (S::kBox * NMAT + p.xbox) * static_cast<uint32_t>(nbox));
                    for (int m = 0; m < NMAT; ++m)
                        for (int q = 0; q < nbox; ++q)   // column coordinate: whole 144-byte groups
                            tma_load_2d(dst + (m * 2 + q) * S::kBox, m ? &tm1 : &tm0, (c * 2 + q) * kGroup, r0,
                                        &full[slot], policy);
                    if (waited) {
                        issue_x(slot, c);
                    } else {
                        pend[slot] = c;
                        if (s + 1 == ns) {   // the ring is full: wait, then the pending activations
                            pdl_wait();
                            waited = true;
                            for (int i = 0; i < ns; ++i) issue_x(i, pend[i]);
                        }
                    }
                    ++s;
                    if (++slot == ns) {
                        slot = 0;
                        par ^= 1u;
                    }
                }
            }
            if (!waited) {   // fewer stages than ring slots (or a wait gave up)
                pdl_wait();
                for (int i = 0; i < min(s, ns); ++i) issue_x(i, pend[i]);
            }
            if (!ok) drain_stages(full, ns, max(0, s - ns), s - 1);
        }
        return;   // the producer warp never triggers dependents: the consumers do, after their wait
    }

    pdl_wait_trigger();   // the activations (and residual) come from the previous kernel
    clear_words(p.clear, p.nclear, tid, kWarps * 32);
    const int B = p.B;
    const int g = lane >> 2, t = lane & 3;
    const float* gg = p.gamma ? p.gamma + 4 * t : nullptr;
    float ss = 0.f;                          // this lane's share of row g's sum of squares
    // this warp's block of the stage in the stage's activation boxes: row g, columns
    // (warp % 8) * 32 + 4t (+ 16) of box warp / 8 (lanes of rows past B read nothing)
    const bool xrow = g < B;
    const uint32_t xoff = S::kWts + (warp / 8) * p.xbox + ((xrow ? g : 0) * kXCols + (warp % 8) * 32 + 4 * t) * 4;
    bool ok = true;
    int s = 0, slot = 0;
    uint32_t par = 0;
    int it = 0;
    for (int64_t tl = blockIdx.x; tl < ntiles; tl += gridDim.x, ++it) {
        const int64_t r0 = tl * S::kRows;
        float acc[NMAT * MT][4];
#pragma unroll
        for (int u = 0; u < NMAT * MT; ++u) acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = 0.f;
        for (int c = 0; c < p.nchunk; ++c) {
            const int nb = min(kStageBlocks, p.nblk - c * kStageBlocks);   // 8 or 16
            // gamma of this warp's block (a weight: requested before the stage wait)
            float4 gv[2];
            {
                const int e0 = (c * kStageBlocks + warp) * 32;
                const bool gin = gg && warp < nb;
                gv[0] = gin ? __ldg(reinterpret_cast<const float4*>(gg + e0)) : make_float4(1.f, 1.f, 1.f, 1.f);
                gv[1] = gin ? __ldg(reinterpret_cast<const float4*>(gg + e0 + 16)) : make_float4(1.f, 1.f, 1.f, 1.f);
            }
            if (ok) ok = mbar_wait(&full[slot], par, p.status);
            if (ok) {
                const uint8_t* st = smem + static_cast<size_t>(slot) * p.stage;
                {
                    const int blk = warp;
                    if (blk < nb) {
                        float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
                        if (xrow) {
                            v0 = *reinterpret_cast<const float4*>(st + xoff);
                            v1 = *reinterpret_cast<const float4*>(st + xoff + 64);
                        }
                        if (it == 0)
                            ss += v0.x * v0.x + v0.y * v0.y + v0.z * v0.z + v0.w * v0.w + v1.x * v1.x +
                                  v1.y * v1.y + v1.z * v1.z + v1.w * v1.w;
                        v0.x *= gv[0].x; v0.y *= gv[0].y; v0.z *= gv[0].z; v0.w *= gv[0].w;
                        v1.x *= gv[1].x; v1.y *= gv[1].y; v1.z *= gv[1].z; v1.w *= gv[1].w;
                        // the block's power of two for row g: the quad's largest magnitude to [2^13, 2^14)
                        float m = fmaxf(fmaxf(fmaxf(fabsf(v0.x), fabsf(v0.y)), fmaxf(fabsf(v0.z), fabsf(v0.w))),
                                        fmaxf(fmaxf(fabsf(v1.x), fabsf(v1.y)), fmaxf(fabsf(v1.z), fabsf(v1.w))));
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
                        int e = 0;
                        if (m > 0.f) e = 13 - (((__float_as_int(m) >> 23) & 0xff) - 127);
                        e = max(-126, min(126, e));
                        const float sc = __int_as_float((127 + e) << 23);
                        const float inv = __int_as_float((127 - e) << 23);
                        const float ic0 = __shfl_sync(0xffffffffu, inv, 8 * t);       // column 2t
                        const float ic1 = __shfl_sync(0xffffffffu, inv, 8 * t + 4);   // column 2t + 1
                        v0.x *= sc; v0.y *= sc; v0.z *= sc; v0.w *= sc;
                        v1.x *= sc; v1.y *= sc; v1.z *= sc; v1.w *= sc;
                        uint32_t bh0[2], bl0[2], bh1[2], bl1[2];
                        split_pairs(v0, bh0[0], bh0[1], bl0[0], bl0[1]);
                        split_pairs(v1, bh1[0], bh1[1], bl1[0], bl1[1]);
#pragma unroll
                        for (int mm = 0; mm < NMAT; ++mm)
#pragma unroll
                            for (int mt = 0; mt < MT; ++mt) {
                                // rows g and g + 8 of m16 tile mt of matrix mm (plain loads: the stage
                                // wait above orders them after the copy)
                                const uint8_t* ra =
                                    st + (mm * 2 + blk / 8) * S::kBox + (mt * 16 + g) * kGroup + (blk % 8) * kBlk;
                                const uint8_t* rb = ra + 8 * kGroup;
                                const float dg = half_bits_to_float(*reinterpret_cast<const uint16_t*>(ra));
                                const float dg8 = half_bits_to_float(*reinterpret_cast<const uint16_t*>(rb));
                                // the lane's code bytes 4t .. 4t + 3 (block offset 2 + 4t): 4-byte
                                // aligned in odd blocks, two aligned words joined in even ones
                                uint32_t wg, wg8;
                                if (blk & 1) {
                                    wg = *reinterpret_cast<const uint32_t*>(ra + 2 + 4 * t);
                                    wg8 = *reinterpret_cast<const uint32_t*>(rb + 2 + 4 * t);
                                } else {
                                    wg = __funnelshift_r(*reinterpret_cast<const uint32_t*>(ra + 4 * t),
                                                         *reinterpret_cast<const uint32_t*>(ra + 4 + 4 * t), 16);
                                    wg8 = __funnelshift_r(*reinterpret_cast<const uint32_t*>(rb + 4 * t),
                                                          *reinterpret_cast<const uint32_t*>(rb + 4 + 4 * t), 16);
                                }
                                uint32_t l02, l13, h02, h13, m02, m13, n02, n13;
                                gemv_mma::dequant_word(wg, l02, l13, h02, h13);
                                gemv_mma::dequant_word(wg8, m02, m13, n02, n13);
                                float cb[4];
                                mma_zero(cb, l02, m02, l13, m13, bh0[0], bh0[1]);
                                mma_16816(cb, l02, m02, l13, m13, bl0[0], bl0[1]);
                                mma_16816(cb, h02, n02, h13, n13, bh1[0], bh1[1]);
                                mma_16816(cb, h02, n02, h13, n13, bl1[0], bl1[1]);
                                float* a = acc[mm * MT + mt];
                                a[0] = fmaf(dg * ic0, cb[0], a[0]);
                                a[1] = fmaf(dg * ic1, cb[1], a[1]);
                                a[2] = fmaf(dg8 * ic0, cb[2], a[2]);
                                a[3] = fmaf(dg8 * ic1, cb[3], a[3]);
                            }
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
        // the warps' sums, added in warp order (two buffers: one barrier per tile); the first
        // tile also publishes each warp's share of the rows' sums of squares
        float* rb = red + (it & 1) * S::kRed;
#pragma unroll
        for (int u = 0; u < NMAT * MT; ++u)
#pragma unroll
            for (int e = 0; e < 4; ++e) rb[(warp * S::kOut + u * 4 + e) * 32 + lane] = acc[u][e];
        if (it == 0) {
            float q = ss + __shfl_xor_sync(0xffffffffu, ss, 1);
            q += __shfl_xor_sync(0xffffffffu, q, 2);
            if (t == 0) ssw[warp * 8 + g] = q;
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kWarps * 32) : "memory");
        for (int o = tid; o < MT * 4 * 32; o += kWarps * 32) {
            const int q = o >> 5, ln = o & 31;   // q = tile * 4 + e
            const int e = q & 3;
            const int64_t row = r0 + (q >> 2) * 16 + (ln >> 2) + (e >> 1) * 8;
            const int bcol = 2 * (ln & 3) + (e & 1);
            if (bcol >= B || row >= p.N) continue;
            float out = 1.f;
            if (p.gamma) {
                float sq = 0.f;
                for (int w = 0; w < kWarps; ++w) sq += ssw[w * 8 + bcol];
                out = rsqrtf(sq / static_cast<float>(p.K) + p.eps);
            }
            float v = 0.f;
            for (int w = 0; w < kWarps; ++w) v += rb[(w * S::kOut + q) * 32 + ln];
            v *= out;
            if (NMAT == 1) {
                if (p.residual) v += p.residual[bcol * p.ldr + row];
            } else {
                float uv = 0.f;
                for (int w = 0; w < kWarps; ++w) uv += rb[(w * S::kOut + MT * 4 + q) * 32 + ln];
                v = gemv_mma::act_fn(v, p.act) * (uv * out);
            }
            p.y[bcol * p.ldy + row] = v;
        }
    }
    // a wait that gave up: the copies of the last stages still get a bounded chance to land
    // before the CTA exits
    if (!ok) atomicOr(&any_failed, 1);
    asm volatile("bar.sync 1, %0;" ::"r"(kWarps * 32) : "memory");
    if (any_failed && tid == 0) drain_stages(full, ns, max(0, s - ns), s - 1);
}

template <int NMAT, int MT>
const void* kernel_ptr() {
    return reinterpret_cast<const void*>(q4_0_gemv_wide_kernel<NMAT, MT>);
}

gem_status ensure_smem_wide(const void* fn, int device, size_t bytes) {
    static std::mutex mu;
    static std::map<std::pair<int, const void*>, size_t> done;
    std::lock_guard<std::mutex> lk(mu);
    size_t& have = done[{device, fn}];
    if (have >= bytes) return GEM_OK;
    GEM_CUDA_TRY(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)));
    have = bytes;
    return GEM_OK;
}

template <int NMAT, int MT>
gem_status launch(const GemvOp& op, cudaStream_t stream, const DeviceInfo& di, Params& p) {
    using S = Shape<NMAT, MT>;
    p.xbox = static_cast<uint32_t>(op.B) * kXCols * 4;
    p.stage = static_cast<uint32_t>(align_up(S::kWts + 2 * p.xbox, 128));
    // as many stages as shared memory holds next to the fixed part, at most kMaxStages
    if (di.smem_optin < S::kFixed + 2 * p.stage) return GEM_ERR_UNSUPPORTED_SHAPE;
    p.ns = static_cast<int>(std::min<size_t>(kMaxStages, (di.smem_optin - S::kFixed) / p.stage));
    const size_t smem = static_cast<size_t>(p.ns) * p.stage + S::kFixed;
    const uint64_t rowbytes = static_cast<uint64_t>(op.K / 32) * kBlk;
    CUtensorMap tm0, tm1;
    gem_status st;
    if ((st = make_tensor_map_2d(&tm0, CU_TENSOR_MAP_DATA_TYPE_UINT8, op.W0, rowbytes, static_cast<uint64_t>(op.N),
                                 rowbytes, kGroup, S::kRows, CU_TENSOR_MAP_SWIZZLE_NONE)) != GEM_OK)
        return st;
    if (NMAT == 2) {
        if ((st = make_tensor_map_2d(&tm1, CU_TENSOR_MAP_DATA_TYPE_UINT8, op.W1, rowbytes, static_cast<uint64_t>(op.N),
                                     rowbytes, kGroup, S::kRows, CU_TENSOR_MAP_SWIZZLE_NONE)) != GEM_OK)
            return st;
    } else {
        tm1 = tm0;
    }
    // the activation rows: K x B fp32 (row stride ldx), boxes of 256 values x B rows
    CUtensorMap tmx;
    if ((st = make_tensor_map_2d(&tmx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, op.x, static_cast<uint64_t>(op.K),
                                 static_cast<uint64_t>(op.B), static_cast<uint64_t>(op.ldx) * 4, kXCols,
                                 static_cast<uint32_t>(op.B), CU_TENSOR_MAP_SWIZZLE_NONE)) != GEM_OK)
        return st;
    const void* fn = kernel_ptr<NMAT, MT>();
    if ((st = ensure_smem_wide(fn, di.device, smem)) != GEM_OK) return st;
    const int64_t ntiles = (op.N + S::kRows - 1) / S::kRows;
    const int grid = static_cast<int>(std::min<int64_t>(ntiles, di.num_sms));
    void* args[] = {&tm0, &tm1, &tmx, &p};
    return launch_pdl(fn, dim3(grid), dim3((kWarps + 1) * 32), smem, stream, args);
}

}  // namespace gemv_wide

// 2..8 rows (callers check the fast-path conditions: K % 256 == 0, aligned operands).  The tile
// height (32 or 64 rows per matrix) is, among those that give every SM a tile, the one
// whose round-robin makespan is shortest, counting a tile's fixed cost as two m16 tiles' work
// (taller on ties); with fewer rows than that, 32-row tiles.
gem_status gemv_enqueue_wide(const GemvOp& op, cudaStream_t stream, const DeviceInfo& di) {
    using namespace gemv_wide;
    const int nmat = op.W1 ? 2 : 1;
    Params p{};
    p.N = op.N;
    p.K = static_cast<int>(op.K);
    p.nblk = static_cast<int>(op.K / 32);
    p.nchunk = (p.nblk + kStageBlocks - 1) / kStageBlocks;
    p.B = op.B;
    p.x = op.x;
    p.ldx = op.ldx;
    p.y = op.y;
    p.ldy = op.ldy;
    p.residual = op.residual;
    p.ldr = op.ldr;
    p.gamma = op.norm_gamma;
    p.eps = op.eps;
    p.act = op.act;
    p.status = di.status_word;
    p.clear = op.clear;
    p.nclear = op.nclear;
    int best = 2;
    int64_t best_cost = -1;
    for (int mt : {4, 2}) {
        if (nmat == 2 && mt == 4) continue;   // the reduction buffers of 2 x 64 rows and 16 warps leave too little ring
        const int64_t ntiles = (op.N + 16 * mt - 1) / (16 * mt);
        if (ntiles < di.num_sms) continue;
        const int64_t cost = (ntiles + di.num_sms - 1) / di.num_sms * (mt + 2);
        if (best_cost < 0 || cost < best_cost) {
            best = mt;
            best_cost = cost;
        }
    }
    if (nmat == 1) {
        if (best == 4) return launch<1, 4>(op, stream, di, p);
        return launch<1, 2>(op, stream, di, p);
    }
    return launch<2, 2>(op, stream, di, p);
}

}  // namespace gem
