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
    p.clear = op.clear;
    p.nclear = op.nclear;
    p.U = static_cast<int>((op.N + kUnitRows - 1) / kUnitRows);
    auto kernel_of = [&](int ks) {
        if (ks == 2)
            return nmat == 2 ? reinterpret_cast<const void*>(q4_0_gemv_b1_kernel<2, 2>)
                             : reinterpret_cast<const void*>(q4_0_gemv_b1_kernel<1, 2>);
        return nmat == 2 ? reinterpret_cast<const void*>(q4_0_gemv_b1_kernel<2, 1>)
                         : reinterpret_cast<const void*>(q4_0_gemv_b1_kernel<1, 1>);
    };
    const size_t budget = std::min<size_t>(gemv_mma::kSmemBudget, di.smem_optin);
    int gps = 1, rps = 1, rbmax = 1, umax = 1, up = 1, ns = 0, Gk = p.G;
    auto layout = [&](int u, int n, bool commit) -> size_t {
        const size_t xf = static_cast<size_t>(2 * Gk) * kRecBytes + kZeroBytes;
        const size_t stage = static_cast<size_t>(rps * gps) * kBoxBytes;
        const size_t red = static_cast<size_t>(nmat) * u * kUnitRows * (2 * gps) * 4;
        size_t off = align_up(static_cast<size_t>(n) * stage, 128);
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
        const size_t bsc_off = off;
        off += static_cast<size_t>(Gk) * 8 * 4;   // per block: 2^-e of its operand scale
        if (commit) {
            p.bsc_off = static_cast<uint32_t>(bsc_off);
            p.stage_bytes = static_cast<uint32_t>(stage);
            p.full_off = static_cast<uint32_t>(full_off);
            p.empty_off = static_cast<uint32_t>(empty_off);
            p.xf_off = static_cast<uint32_t>(xf_off);
            p.red_off = static_cast<uint32_t>(red_off);
            p.misc_off = static_cast<uint32_t>(misc_off);
        }
        return align_up(off, 128);
    };
    // Plan for ks-way K splits (each CTA owns ceil(G / ks) groups) and ncl CTA groups over the
    // units.  Phase width: 4..9 groups (2 consumer warps per group); the widest (longest runs per
    // row, most warps) unless a narrower one wastes at least 5 % fewer warp slots over its
    // phases.  Stages hold up to three row blocks sharing the activation operand (three when a
    // CTA's units come in threes and still fit one pass).  A split needs one pass.
    auto plan = [&](int ks, int ncl) -> bool {
        Gk = (p.G + ks - 1) / ks;
        umax = (p.U + ncl - 1) / ncl;
        gps = 1;
        double best = -1.0;
        for (int c = std::min(kMaxConsumerWarps / 2, Gk); c >= std::min(4, Gk); --c) {
            const int nph = (Gk + c - 1) / c;
            const double eff = static_cast<double>(Gk) / (static_cast<double>(nph) * c);
            if (eff > best + 0.05) {
                best = eff;
                gps = c;
            }
        }
        rbmax = umax * nmat;
        rps = rbmax >= kMaxRps && rbmax % kMaxRps == 0 ? kMaxRps : std::min(2, rbmax);
        const int nphase = (Gk + gps - 1) / gps;
        up = umax;
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
            else return false;
        }
        return ks == 1 || up == umax;
    };
    // K split over 2-CTA clusters where the units do not divide evenly over the SMs and the
    // slowest CTA's share shrinks by at least 10 % (e.g. 336 units: 3 per CTA, or 5 per CTA pair
    // at half the groups each).
    int ks = 1, ncl = std::min(di.num_sms, p.U);
    const int um1 = (p.U + ncl - 1) / ncl;
    if (p.U % ncl != 0 && um1 <= 3 && p.G >= 64) {   // long K (K >= 16384: measured faster split)
        int n = std::min(di.num_sms / 2, p.U);
        if (plan(2, n)) {
            cudaLaunchConfig_t cfg{};
            cfg.gridDim = dim3(2 * n);
            cfg.blockDim = dim3((2 * gps + 1) * 32);
            cfg.dynamicSmemBytes = layout(up, ns, false);
            cudaLaunchAttribute a[1];
            a[0].id = cudaLaunchAttributeClusterDimension;
            a[0].val.clusterDim.x = 2;
            a[0].val.clusterDim.y = 1;
            a[0].val.clusterDim.z = 1;
            cfg.attrs = a;
            cfg.numAttrs = 1;
            gem_status st0;
            if ((st0 = ensure_smem_b1(kernel_of(2), di.device, cfg.dynamicSmemBytes)) != GEM_OK) return st0;
            int nmax = 0;
            if (cudaOccupancyMaxActiveClusters(&nmax, kernel_of(2), &cfg) != cudaSuccess || nmax <= 0) {
                (void)cudaGetLastError();
            } else {
                if (nmax < n) n = nmax;
                if (plan(2, n) && 10 * ((p.U + n - 1) / n) < 2 * 9 * um1) {
                    ks = 2;
                    ncl = n;
                }
            }
        }
    }
    if (ks == 1 && !plan(1, ncl)) return GEM_OK;   // not planned: records too large for this K
    const int C = ncl * ks;
    p.ks = ks;
    p.rps = rps;
    p.up = up;
    p.gps = gps;
    p.nphase = (Gk + gps - 1) / gps;
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
    const void* fn = kernel_of(ks);
    if ((st = ensure_smem_b1(fn, di.device, smem)) != GEM_OK) return st;
    *planned = true;
    void* args[] = {&tm0, &tm1, &p};
    return launch_pdl_cluster(fn, dim3(C), dim3((p.ncw + 1) * 32), smem, stream, args, ks);
}

}  // namespace gem
