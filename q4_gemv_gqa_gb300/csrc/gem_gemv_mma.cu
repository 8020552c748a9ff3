// gem_gemv_mma.cu — host plan and launch of the tensor-core Q4_0 GEMV (gem_gemv_mma.cuh).
#include <algorithm>
#include <map>
#include <mutex>

#include "gem_gemv_mma.cuh"

namespace gem {
namespace {

using namespace gemv_mma;

constexpr size_t kXfMax = 48 * 1024;   // activation fragments of one K-phase

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
    p.U = static_cast<int>((op.N + kUnitRows - 1) / kUnitRows);
    const int C = std::min(di.num_sms, p.U);
    const int umax = (p.U + C - 1) / C;
    p.up = std::max(1, std::min(umax, kMaxConsumerWarps / (2 * nmat)));
    int gps = std::max(1, std::min(p.G, kMaxConsumerWarps / (2 * nmat * p.up)));
    const int stages_for = (p.G + gps - 1) / gps;
    gps = (p.G + stages_for - 1) / stages_for;   // same stage count, even split
    p.gps = gps;
    p.spp = (p.G + gps - 1) / gps;
    p.ncw = 2 * nmat * p.up * gps;
    p.stage_bytes = static_cast<uint32_t>(nmat) * p.up * gps * kBoxBytes;
    const int nct = p.ncw * 32;
    // K-phase: as much of K as the fragment area and the register prefetch hold
    const int step = 256 * gps;
    const int64_t cap_xf = static_cast<int64_t>(kXfMax) / (4 * B);
    const int64_t cap_pf = static_cast<int64_t>(kPrefetchF4) * nct * 4 / B;
    int64_t kp = std::min<int64_t>({cap_xf, cap_pf, static_cast<int64_t>(p.spp) * step});
    kp = std::max<int64_t>(step, kp / step * step);
    p.kp = static_cast<int>(kp);
    p.nphase = static_cast<int>((static_cast<int64_t>(p.spp) * step + kp - 1) / kp);
    const int nph = 2 * gps;
    const int rows_in_pass = nmat * p.up * kUnitRows;
    const size_t xf_bytes = 4ull * B * p.kp;
    const size_t xsc_bytes = static_cast<size_t>(p.kp / 128) * B * 4;
    const size_t ssq_bytes = static_cast<size_t>(B) * 2 * p.G * 4;
    const size_t red_bytes = static_cast<size_t>(rows_in_pass) * nph * B * 4;
    const size_t other = align_up(xf_bytes, 128) + align_up(xsc_bytes, 128) + align_up(ssq_bytes, 128) +
                         align_up(red_bytes, 128) + 128 + 2 * 8 * 8 + 128;
    const int total_stages = ((umax + p.up - 1) / p.up) * p.spp;
    int ns = static_cast<int>((kSmemBudget > other ? kSmemBudget - other : 0) / p.stage_bytes);
    ns = std::max(2, std::min(ns, std::min(total_stages, 8)));
    ns = std::min(ns, total_stages);
    p.ns = std::max(1, ns);
    size_t off = align_up(static_cast<size_t>(p.ns) * p.stage_bytes, 128);
    p.full_off = static_cast<uint32_t>(off);
    off += 8 * 8;
    p.empty_off = static_cast<uint32_t>(off);
    off = align_up(off + 8 * 8, 128);
    p.xf_off = static_cast<uint32_t>(off);
    off = align_up(off + xf_bytes, 128);
    p.xsc_off = static_cast<uint32_t>(off);
    off = align_up(off + xsc_bytes, 128);
    p.ssq_off = static_cast<uint32_t>(off);
    off = align_up(off + ssq_bytes, 128);
    p.red_off = static_cast<uint32_t>(off);
    off = align_up(off + red_bytes, 128);
    p.rstd_off = static_cast<uint32_t>(off);
    off += 8 * 4;
    const size_t smem = align_up(off, 128);
    if (smem > di.smem_optin) return GEM_ERR_UNSUPPORTED_SHAPE;

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
