// gem_gemv_b1.cu — host plan and launch of the one-row tensor-core Q4_0 GEMV (gem_gemv_b1.cuh).
#include <algorithm>
#include <map>
#include <mutex>

#include "gem_gemv_b1.cuh"

namespace gem {
namespace {

using namespace gemv_b1;

gem_status ensure_smem_b1(const void* fn, int device, size_t bytes) {
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

// B = 1 fast path.  Sets *planned = false (and launches nothing) when the activation records of
// all of K do not fit next to a ring of at least 4 stages; the caller then uses the general
// tensor-core kernel.
gem_status gemv_enqueue_b1(const GemvOp& op, cudaStream_t stream, const DeviceInfo& di, bool* planned) {
    *planned = false;
    const int nmat = op.W1 ? 2 : 1;
    Params p{};
    p.N = op.N;
    p.G = static_cast<int>(op.K / 256);
    p.x = op.x;
    p.y = op.y;
    p.residual = op.residual;
    p.gamma = op.norm_gamma;
    p.eps = op.eps;
    p.act = op.act;
    p.status = di.status_word;
    p.U = static_cast<int>((op.N + kUnitRows - 1) / kUnitRows);
    const int C = std::min(di.num_sms, p.U);
    const int umax = (p.U + C - 1) / C;

    // Phase width: 4..9 groups (2 consumer warps per group); the widest (longest runs per row,
    // most warps) unless a narrower one wastes at least 5 % fewer warp slots over its
    // ceil(G / gps) phases.
    int gps = 1;
    double best = -1.0;
    for (int c = std::min(kMaxConsumerWarps / 2, p.G); c >= std::min(4, p.G); --c) {
        const int nph = (p.G + c - 1) / c;
        const double eff = static_cast<double>(p.G) / (static_cast<double>(nph) * c);
        if (eff > best + 0.05) {
            best = eff;
            gps = c;
        }
    }
    // Stages hold up to three row blocks sharing the activation operand (as many as the CTAs'
    // units allow; three when they come in threes, e.g. nine units per CTA).
    const int rbmax = umax * nmat;
    int rps = rbmax >= kMaxRps && rbmax % kMaxRps == 0 ? kMaxRps : std::min(2, rbmax);
    const size_t budget = std::min<size_t>(gemv_mma::kSmemBudget, di.smem_optin);
    const size_t xf = static_cast<size_t>(2 * p.G) * kRecBytes + kZeroBytes;
    auto layout = [&](int up, int ns, bool commit) -> size_t {
        const size_t stage = static_cast<size_t>(rps * gps) * kBoxBytes;
        const size_t red = static_cast<size_t>(nmat) * up * kUnitRows * (2 * gps) * 4;
        size_t off = align_up(static_cast<size_t>(ns) * stage, 128);
        const size_t full_off = off;
        off += kMaxSlots * 8;
        const size_t empty_off = off;
        off = align_up(off + kMaxSlots * 8, 128);
        const size_t xf_off = off;
        off = align_up(off + xf, 128);
        const size_t red_off = off;
        off = align_up(off + red, 128);
        const size_t misc_off = off;
        off += 128 * 4;
        if (commit) {
            p.stage_bytes = static_cast<uint32_t>(stage);
            p.full_off = static_cast<uint32_t>(full_off);
            p.empty_off = static_cast<uint32_t>(empty_off);
            p.xf_off = static_cast<uint32_t>(xf_off);
            p.red_off = static_cast<uint32_t>(red_off);
            p.misc_off = static_cast<uint32_t>(misc_off);
        }
        return align_up(off, 128);
    };
    const int nphase = (p.G + gps - 1) / gps;
    int up = umax, ns = 0;
    for (;;) {
        const int stages = (nmat * up + rps - 1) / rps * nphase;
        // at least 4 stages in flight (3 when a stage is >= 40 KB)
        const int want = std::min(static_cast<size_t>(rps * gps) * kBoxBytes >= 40 * 1024 ? 3 : 4, stages);
        ns = 0;
        for (int n = std::min(kMaxSlots, stages); n >= want && !ns; --n)
            if (layout(up, n, false) <= budget) ns = n;
        if (ns && (up == umax || rps <= 2)) break;
        if (ns || rps > 2) {   // three row blocks only with every unit in one pass
            rps = std::min(2, rbmax);
            up = umax;
            continue;
        }
        if (up > 1) up = (up + 1) / 2;
        else return GEM_OK;   // not planned: records too large for this K
    }
    p.rps = rps;
    p.up = up;
    p.gps = gps;
    p.nphase = nphase;
    p.ns = ns;
    p.ncw = 2 * gps;
    const size_t smem = layout(up, ns, true);

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
    const void* fn = nmat == 2 ? reinterpret_cast<const void*>(q4_0_gemv_b1_kernel<2>)
                               : reinterpret_cast<const void*>(q4_0_gemv_b1_kernel<1>);
    if ((st = ensure_smem_b1(fn, di.device, smem)) != GEM_OK) return st;
    *planned = true;
    void* args[] = {&tm0, &tm1, &p};
    return launch_pdl(fn, dim3(C), dim3((p.ncw + 1) * 32), smem, stream, args);
}

}  // namespace gem
