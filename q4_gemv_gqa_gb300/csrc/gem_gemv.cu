// gem_gemv.cu — Q4_0 dequantise-and-matvec for decode (B = 1..8 activation rows).
//
// Q4_0 ("gem" engine research record, "Verified model facts"): rows of 18-byte blocks,
// binary16 scale d then 16 bytes of 4-bit codes; weight = (q - 8) * d; byte j carries
// element j (low nibble) and element j + 16 (high nibble).
//
// Data movement.  A matrix row of K weights is K*9/16 bytes; with K % 256 == 0 it is a
// multiple of 144 bytes = 8 blocks = one "group" of 256 weights, and 16-byte aligned.  The
// matrix is viewed as a 2-D byte tensor [N][K*9/16] and streamed by TMA in boxes of
// 16 rows x 144 bytes into a ring of shared-memory stages, completion tracked by mbarriers.
// Each CTA owns a contiguous range of 16-row units (balanced to one unit across CTAs) and
// walks K in stages of `gps` groups, so every thread keeps one running sum per row and the
// activation chunk for a stage is read once per CTA.  Weight boxes for the first stages
// are requested before griddepcontrol.wait, so with programmatic dependent launch the
// weight stream starts while the previous kernel in the stream is still running.
//
// Arithmetic.  Each thread owns one (row, group) task per stage: it loads its 144 bytes
// with nine 16-byte shared loads, and for each block forms the floats 1 + q/16 with one
// byte permute per weight (exponent 0x3F8, code in mantissa bits 19..22); one packed add
// of -1.5 turns them into the exact codes (q - 8)/16.  Products accumulate in fp32 with
// packed f32x2 FMAs in two chains per block; the block sum is scaled by d in fp32 and the
// factor 16 is applied once in the epilogue.  (Folding the -8 into a per-block sum of x
// instead would save the add but cancels about two bits, which unit-scale attention
// downstream of the QKV projection amplifies.)  No tensor cores: at batch 1..8 the op
// streams 0.5625 bytes per weight and the budget is instruction issue, not math.
#include <algorithm>
#include <cstdlib>
#include <map>
#include <mutex>

#include "gem_gemv_kernels.cuh"

GEM_GEMV_DECLARE_BATCH(1)
GEM_GEMV_DECLARE_BATCH(2)
GEM_GEMV_DECLARE_BATCH(3)
GEM_GEMV_DECLARE_BATCH(4)
GEM_GEMV_DECLARE_BATCH(5)
GEM_GEMV_DECLARE_BATCH(6)
GEM_GEMV_DECLARE_BATCH(7)
GEM_GEMV_DECLARE_BATCH(8)

namespace gem {
namespace {

using gemv_detail::GemvParams;
using gemv_detail::kBoxBytes;
using gemv_detail::kGroupBytes;
using gemv_detail::kMaxThreads;
using gemv_detail::kSmemBudget;
using gemv_detail::kUnitRows;

const void* pick_tma(int B, int nmat) {
    switch (B) {
        case 1: return gemv_tma_kernel_b1(nmat);
        case 2: return gemv_tma_kernel_b2(nmat);
        case 3: return gemv_tma_kernel_b3(nmat);
        case 4: return gemv_tma_kernel_b4(nmat);
        case 5: return gemv_tma_kernel_b5(nmat);
        case 6: return gemv_tma_kernel_b6(nmat);
        case 7: return gemv_tma_kernel_b7(nmat);
        default: return gemv_tma_kernel_b8(nmat);
    }
}

const void* pick_gen(int B, int nmat) {
    switch (B) {
        case 1: return gemv_generic_kernel_b1(nmat);
        case 2: return gemv_generic_kernel_b2(nmat);
        case 3: return gemv_generic_kernel_b3(nmat);
        case 4: return gemv_generic_kernel_b4(nmat);
        case 5: return gemv_generic_kernel_b5(nmat);
        case 6: return gemv_generic_kernel_b6(nmat);
        case 7: return gemv_generic_kernel_b7(nmat);
        default: return gemv_generic_kernel_b8(nmat);
    }
}

// dynamic shared memory opt-in, once per (device, kernel, size)
gem_status ensure_smem(const void* fn, int device, size_t bytes) {
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

gem_status gemv_check(const GemvOp& op) {
    if (op.B < 0 || op.N < 0 || op.K < 0) return GEM_ERR_INVALID_ARG;
    if (op.B > 8) return GEM_ERR_UNSUPPORTED_SHAPE;
    if (op.K % 32) return GEM_ERR_UNSUPPORTED_SHAPE;
    if (op.B == 0 || op.N == 0) return GEM_OK;
    if (!op.W0 || !op.y || (op.K > 0 && !op.x)) return GEM_ERR_INVALID_ARG;
    if (op.ldx < op.K || op.ldy < op.N) return GEM_ERR_INVALID_ARG;
    if (op.residual && op.ldr < op.N) return GEM_ERR_INVALID_ARG;
    if (op.act < 0 || op.act > 1) return GEM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(op.x) | reinterpret_cast<uintptr_t>(op.y)) & 3) return GEM_ERR_MISALIGNED;
    return GEM_OK;
}

gem_status gemv_enqueue(const GemvOp& op, cudaStream_t stream) {
    gem_status st = gemv_check(op);
    if (st != GEM_OK || op.B == 0 || op.N == 0) return st;
    DeviceInfo di;
    if ((st = device_info(&di)) != GEM_OK) return st;
    const int nmat = op.W1 ? 2 : 1;

    GemvParams p{};
    p.N = op.N;
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

    const uintptr_t wbits = reinterpret_cast<uintptr_t>(op.W0) | reinterpret_cast<uintptr_t>(op.W1);
    const uintptr_t xbits = reinterpret_cast<uintptr_t>(op.x) | reinterpret_cast<uintptr_t>(op.norm_gamma);
    const bool fast = op.K > 0 && op.K % 256 == 0 && (wbits & 15) == 0 && (xbits & 15) == 0 &&
                      op.ldx % 4 == 0 && op.N < (int64_t(1) << 31) && op.K / 256 < (1 << 20);
    if (!fast) {
        const int rows_per_cta = 8;
        dim3 grid(static_cast<unsigned>((op.N + rows_per_cta - 1) / rows_per_cta));
        const void* fn = pick_gen(op.B, nmat);
        const uint8_t* w0 = static_cast<const uint8_t*>(op.W0);
        const uint8_t* w1 = static_cast<const uint8_t*>(op.W1 ? op.W1 : op.W0);
        int64_t N = op.N, K = op.K;
        void* args[] = {&w0, &w1, &N, &K, &p};
        return launch_pdl(fn, grid, dim3(256), 0, stream, args);
    }

    static const bool cuda_cores = [] {
        const char* e = getenv("GEM_GEMV_CUDA_CORES");
        return e && e[0] == '1';
    }();
    if (!cuda_cores) return gemv_enqueue_mma(op, stream, di);

    const int64_t rowbytes = op.K / 32 * 18;
    const int B = op.B;
    p.G = static_cast<int>(op.K / 256);
    p.U = static_cast<int>((op.N + kUnitRows - 1) / kUnitRows);
    const int C = std::min(di.num_sms, p.U);
    const int umax = (p.U + C - 1) / C;
    constexpr int kParts = gemv_detail::kPartsPerGroup;
    p.up = std::max(1, std::min(umax, kMaxThreads / (kUnitRows * nmat * kParts)));
    const int per_group_tasks = nmat * p.up * kUnitRows * kParts;
    const size_t per_group_bytes = static_cast<size_t>(nmat) * p.up * kBoxBytes;
    // activation staging per group phase: raw ring (3 x (B+1) chunks), transformed x (2 x B),
    // epilogue partials
    auto other_bytes = [&](int g) {
        const size_t chunk = static_cast<size_t>(g) * 256 * 4;
        const size_t red = std::max<size_t>(static_cast<size_t>(per_group_tasks) * g * B * 4,
                                            static_cast<size_t>(kMaxThreads / 32) * B * 4);
        return 3 * (B + 1) * chunk + 2 * B * chunk + red + 8 * 8 + 16 * 4 + 5 * 128;
    };
    // groups per stage: as many as the thread budget allows, but keep a stage to about a
    // third of the budget so at least three stages are in flight
    int gps = std::max(1, std::min(p.G, kMaxThreads / per_group_tasks));
    while (gps > 1 && per_group_bytes * gps * 3 + other_bytes(gps) > kSmemBudget) --gps;
    gps = (p.G + (p.G + gps - 1) / gps - 1) / ((p.G + gps - 1) / gps);  // same stage count, even split
    p.gps = gps;
    p.spp = (p.G + gps - 1) / gps;
    p.tasks = per_group_tasks * gps;
    p.stage_bytes = static_cast<uint32_t>(per_group_bytes * gps);
    const int total_stages = ((umax + p.up - 1) / p.up) * p.spp;
    const size_t other = other_bytes(gps);
    int ns = static_cast<int>((kSmemBudget - std::min(kSmemBudget, other)) / p.stage_bytes);
    ns = std::max(1, std::min(ns, std::min(total_stages, 8)));
    p.ns = ns;
    const size_t chunk_bytes = static_cast<size_t>(gps) * 256 * 4;
    size_t off = static_cast<size_t>(ns) * p.stage_bytes;
    off = align_up(off, 128);
    p.bar_off = static_cast<uint32_t>(off);
    off = align_up(off + 8 * 8, 128);
    p.raw_off = static_cast<uint32_t>(off);
    off = align_up(off + 3 * (B + 1) * chunk_bytes, 128);
    p.xs_off = static_cast<uint32_t>(off);
    off = align_up(off + 2 * B * chunk_bytes, 128);
    p.rstd_off = static_cast<uint32_t>(off);
    off = align_up(off + 16 * 4, 128);
    p.red_off = static_cast<uint32_t>(off);
    off += std::max<size_t>(static_cast<size_t>(p.tasks) * B * 4, static_cast<size_t>(kMaxThreads / 32) * B * 4);
    const size_t smem = align_up(off, 128);
    if (smem > di.smem_optin) return GEM_ERR_UNSUPPORTED_SHAPE;

    CUtensorMap tm0, tm1;
    if ((st = make_tensor_map_2d(&tm0, CU_TENSOR_MAP_DATA_TYPE_UINT8, op.W0, static_cast<uint64_t>(rowbytes),
                                 static_cast<uint64_t>(op.N), static_cast<uint64_t>(rowbytes), kGroupBytes,
                                 kUnitRows, CU_TENSOR_MAP_SWIZZLE_NONE)) != GEM_OK)
        return st;
    if (nmat == 2) {
        if ((st = make_tensor_map_2d(&tm1, CU_TENSOR_MAP_DATA_TYPE_UINT8, op.W1, static_cast<uint64_t>(rowbytes),
                                     static_cast<uint64_t>(op.N), static_cast<uint64_t>(rowbytes), kGroupBytes,
                                     kUnitRows, CU_TENSOR_MAP_SWIZZLE_NONE)) != GEM_OK)
            return st;
    } else {
        tm1 = tm0;
    }
    const void* fn = pick_tma(op.B, nmat);
    if ((st = ensure_smem(fn, di.device, smem)) != GEM_OK) return st;
    const int threads = (p.tasks + 31) / 32 * 32;
    void* args[] = {&tm0, &tm1, &p};
    return launch_pdl(fn, dim3(C), dim3(threads), smem, stream, args);
}

}  // namespace gem

extern "C" gem_status gem_q4_0_gemv(const void* W, int64_t N, int64_t K, const float* x, int64_t ldx, int B,
                                    float* y, int64_t ldy, const float* residual, void* stream) {
    gem::GemvOp op{};
    op.W0 = W;
    op.W1 = nullptr;
    op.N = N;
    op.K = K;
    op.B = B;
    op.x = x;
    op.ldx = ldx;
    op.y = y;
    op.ldy = ldy;
    op.residual = residual;
    op.ldr = ldy;
    op.norm_gamma = nullptr;
    op.eps = 0.f;
    op.act = 0;
    return gem::gemv_enqueue(op, static_cast<cudaStream_t>(stream));
}
