// gem_gemv_mma.cu — host plan and launch of the tensor-core Q4_0 GEMV (gem_gemv_mma.cuh).
#include <algorithm>
#include <map>
#include <mutex>

#include "gem_gemv_mma.cuh"

namespace gem {
namespace {

using namespace gemv_mma;

const void* pick(bool packed, int nmat) {
    if (packed) return nmat == 2 ? reinterpret_cast<const void*>(q4_0_gemv_mma_kernel<true, 2>)
                                 : reinterpret_cast<const void*>(q4_0_gemv_mma_kernel<true, 1>);
    return nmat == 2 ? reinterpret_cast<const void*>(q4_0_gemv_mma_kernel<false, 2>)
                     : reinterpret_cast<const void*>(q4_0_gemv_mma_kernel<false, 1>);
}

gem_status ensure_smem_mma(const void* fn, int device, size_t bytes) {
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

// Plan and launch; the caller has checked the op and that the fast-path conditions hold
// (K % 256 == 0, 16-byte aligned matrices and activation rows).
gem_status gemv_enqueue_mma(const GemvOp& op, cudaStream_t stream, const DeviceInfo& di) {
    // 2..8 rows: the one-launch tall-tile kernel up to 64M weights per call (the matrices of a
    // 4B-class layer, where the records kernel's extra launch costs more than it saves); larger
    // matrices stream faster through the records kernel's deeper per-SM pipeline.
    const int64_t weights = (op.W1 ? 2 : 1) * op.N * op.K;
    if (op.B >= 2 && op.B <= 8 && weights <= (int64_t(64) << 20)) return gemv_enqueue_wide(op, stream, di);
    {
        bool planned = false;
        const gem_status st1 = op.B == 1 ? gemv_enqueue_b1(op, stream, di, &planned)
                                         : gemv_enqueue_bn(op, stream, di, &planned);
        if (planned || st1 != GEM_OK) return st1;
    }
    const int nmat = op.W1 ? 2 : 1;
    const int B = op.B;
    Params p{};
    p.N = op.N;
    p.G = static_cast<int>(op.K / 256);
    p.B = B;
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
    p.U = static_cast<int>((op.N + kUnitRows - 1) / kUnitRows);
    const int C = std::min(di.num_sms, p.U);
    const int umax = (p.U + C - 1) / C;

    // Shared memory for phases of gps groups, `up` units per pass and ns ring slots.
    const size_t ssq_bytes = static_cast<size_t>(B) * 2 * p.G * 4;
    // Activation fragments of every phase stay resident when they are small (4 B * K bytes).
    const bool resident = 4ull * B * p.G * 256 <= kResidentX;
    auto nbuf_of = [&](int gps) { return resident ? (p.G + gps - 1) / gps : 2; };
    auto layout = [&](int gps, int up, int ns, bool commit) -> size_t {
        const size_t stage = static_cast<size_t>(gps) * kBoxBytes;
        const size_t xf = 4ull * B * gps * 256;
        const size_t xsc = static_cast<size_t>(gps) * 2 * B * 4;
        const int nbuf = nbuf_of(gps);
        const size_t red = static_cast<size_t>(nmat) * up * kUnitRows * (2 * gps) * B * 4;
        size_t off = align_up(static_cast<size_t>(ns) * stage, 128);
        const size_t full_off = off;
        off += kMaxSlots * 8;
        const size_t empty_off = off;
        off = align_up(off + kMaxSlots * 8, 128);
        const size_t xf_off = off;
        off = align_up(off + nbuf * xf, 128);
        const size_t xsc_off = off;
        off = align_up(off + nbuf * xsc, 128);
        const size_t ssq_off = off;
        off = align_up(off + ssq_bytes, 128);
        const size_t red_off = off;
        off = align_up(off + red, 128);
        const size_t rstd_off = off;
        off += 8 * 4;
        if (commit) {
            p.stage_bytes = static_cast<uint32_t>(stage);
            p.full_off = static_cast<uint32_t>(full_off);
            p.empty_off = static_cast<uint32_t>(empty_off);
            p.xf_off = static_cast<uint32_t>(xf_off);
            p.xf_bytes = static_cast<uint32_t>(xf);
            p.xsc_off = static_cast<uint32_t>(xsc_off);
            p.ssq_off = static_cast<uint32_t>(ssq_off);
            p.red_off = static_cast<uint32_t>(red_off);
            p.rstd_off = static_cast<uint32_t>(rstd_off);
        }
        return align_up(off, 128);
    };
    // Phase width: up to kMaxConsumerWarps / 2 groups (one consumer warp per half group), as
    // wide as possible for long contiguous runs per row, split evenly over K.  Then all of a
    // CTA's units in one pass if the partial-sum area allows, and as many ring slots as fit
    // (at least min(4, stages)).
    const size_t budget = std::min<size_t>(kSmemBudget, di.smem_optin);
    const int nphase = (p.G + kMaxConsumerWarps / 2 - 1) / (kMaxConsumerWarps / 2);
    int gps = (p.G + nphase - 1) / nphase;
    int up = umax, ns = 0;
    for (;; ) {
        const int stages = std::max(1, nmat * std::min(up, umax) * ((p.G + gps - 1) / gps));
        const int want = std::min(4, stages);
        ns = 0;
        for (int n = std::min(kMaxSlots, stages); n >= want && !ns; --n)
            if (layout(gps, up, n, false) <= budget) ns = n;
        if (ns) break;
        if (up > 1) up = (up + 1) / 2;
        else if (gps > 1) --gps;
        else return GEM_ERR_UNSUPPORTED_SHAPE;
    }
    p.up = up;
    p.gps = gps;
    p.nphase = (p.G + gps - 1) / gps;
    p.ns = ns;
    p.ncw = 2 * gps;
    p.nbuf = nbuf_of(gps);
    const size_t smem = layout(gps, up, ns, true);

    const int64_t rowbytes = op.K / 32 * 18;
    CUtensorMap tm0, tm1;
    gem_status st;
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
    const void* fn = pick(B <= 4, nmat);
    if ((st = ensure_smem_mma(fn, di.device, smem)) != GEM_OK) return st;
    void* args[] = {&tm0, &tm1, &p};
    return launch_pdl(fn, dim3(C), dim3((p.ncw + 1) * 32), smem, stream, args);
}

}  // namespace gem
