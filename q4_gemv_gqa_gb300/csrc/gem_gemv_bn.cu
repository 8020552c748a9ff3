// gem_gemv_bn.cu — host plan and launches of the 2..32-row tensor-core Q4_0 GEMV (gem_gemv_bn.cuh):
// the activation prep kernel, then the GEMV.
#include <algorithm>
#include <map>
#include <mutex>

#include "gem_gemv_bn.cuh"

// Library-owned operand records for calls that pass no workspace (gem_q4_0_gemv): one array per
// device, shared by every such call on that device.
static __device__ __align__(256) uint8_t g_gemv_rec_scratch[gem::kGemvRecScratchBytes];

namespace gem {
namespace {

using namespace gemv_bn;

constexpr int kMaxDevices = 64;
std::mutex g_rec_mu;
void* g_rec_addr[kMaxDevices];

gem_status rec_scratch(void** out) {
    int dev = 0;
    GEM_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return GEM_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_rec_mu);
    if (!g_rec_addr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_gemv_rec_scratch);
        if (e != cudaSuccess) return cuda_fail(e);
        if (!p) return cuda_fail(cudaErrorInvalidSymbol);
        g_rec_addr[dev] = p;
    }
    *out = g_rec_addr[dev];
    return GEM_OK;
}

gem_status ensure_smem_bn(const void* fn, int device, size_t bytes) {
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

int gemv_col_tiles(int B) { return B <= 8 ? 1 : (B <= 16 ? 2 : 4); }

size_t gemv_rec_bytes(int B, int64_t K) {
    if (B < 2 || B > kMaxRows || K % 256) return 0;
    return static_cast<size_t>(K / 256) * 2 * kHgBytes * gemv_col_tiles(B) + kMaxRows * sizeof(float2);
}

gem_status gemv_enqueue_bn(const GemvOp& op, cudaStream_t stream, const DeviceInfo& di, bool* planned) {
    *planned = false;
    const int nmat = op.W1 ? 2 : 1;
    const int B = op.B;
    Params p{};
    p.N = op.N;
    p.G = static_cast<int>(op.K / 256);
    p.B = B;
    p.y = op.y;
    p.ldy = op.ldy;
    p.residual = op.residual;
    p.ldr = op.ldr;
    p.act = op.act;
    p.status = di.status_word;
    p.U = static_cast<int>((op.N + kUnitRows - 1) / kUnitRows);
    // operand records: the caller's workspace, else the library's array
    const size_t rec_bytes = gemv_rec_bytes(B, op.K);
    uint8_t* rec = static_cast<uint8_t*>(op.act_ws);
    gem_status st;
    if (!rec || op.act_ws_bytes < rec_bytes) {
        void* s = nullptr;
        if ((st = rec_scratch(&s)) != GEM_OK) return st;
        if (rec_bytes > kGemvRecScratchBytes) return GEM_OK;   // not planned
        rec = static_cast<uint8_t*>(s);
    }
    p.rec = rec;
    p.rowinfo = reinterpret_cast<const float2*>(rec + rec_bytes - kMaxRows * sizeof(float2));
    const int NT = gemv_col_tiles(B);
    const void* fn = nullptr;
    switch (NT * 2 + nmat) {
        case 3: fn = reinterpret_cast<const void*>(q4_0_gemv_bn_kernel<1, 1>); break;
        case 4: fn = reinterpret_cast<const void*>(q4_0_gemv_bn_kernel<2, 1>); break;
        case 5: fn = reinterpret_cast<const void*>(q4_0_gemv_bn_kernel<1, 2>); break;
        case 6: fn = reinterpret_cast<const void*>(q4_0_gemv_bn_kernel<2, 2>); break;
        case 9: fn = reinterpret_cast<const void*>(q4_0_gemv_bn_kernel<1, 4>); break;
        default: fn = reinterpret_cast<const void*>(q4_0_gemv_bn_kernel<2, 4>); break;
    }
    const int ncw_per_group = 2 * NT;   // consumer warps per group of a phase
    const int gps_max = NT == 1 ? 7 : 16 / ncw_per_group;

    const size_t budget = std::min<size_t>(gemv_mma::kSmemBudget, di.smem_optin);
    int rps = 1, umax = 1;
    auto layout = [&](int gp, int u, int n, bool commit) -> size_t {
        const size_t stage = static_cast<size_t>(rps * gp) * kBoxBytes;
        const size_t recbuf = static_cast<size_t>(2 * gp) * kHgBytes * NT;
        const size_t red = static_cast<size_t>(nmat) * u * (ncw_per_group * gp) * NT * 32 * 16;
        size_t off = align_up(static_cast<size_t>(n) * stage, 128);
        const size_t full_off = off;
        off += kMaxSlots * 8;
        const size_t empty_off = off;
        off += kMaxSlots * 8;
        const size_t rfull_off = off;
        off += 8;
        const size_t rempty_off = off;
        off = align_up(off + 8, 128);
        const size_t xf_off = off;
        off = align_up(off + recbuf, 128);
        const size_t red_off = off;
        off += red;
        if (commit) {
            p.stage_bytes = static_cast<uint32_t>(stage);
            p.full_off = static_cast<uint32_t>(full_off);
            p.empty_off = static_cast<uint32_t>(empty_off);
            p.rfull_off = static_cast<uint32_t>(rfull_off);
            p.rempty_off = static_cast<uint32_t>(rempty_off);
            p.xf_off = static_cast<uint32_t>(xf_off);
            p.red_off = static_cast<uint32_t>(red_off);
        }
        return align_up(off, 128);
    };
    // For ks-way K splits (each CTA sees ceil(G / ks) groups) and ncl CTA groups over the units:
    // phase width 1..7 groups (2 consumer warps per group, one record buffer of 2 gps half groups
    // x 4 KB); for each width the most units per pass with a ring of at least 4 stages; then the
    // width with the most busy warps per stage (2 gps x its share of full phases), fewer passes on
    // ties.  A split needs every CTA's units in one pass and its sums to fit the record buffer.
    int gps = 0, up = 0, ns = 0;
    auto plan = [&](int ks, int ncl) -> bool {
        umax = (p.U + ncl - 1) / ncl;
        rps = umax * nmat >= 2 ? 2 : 1;
        const int Gk = (p.G + ks - 1) / ks;
        double best = -1.0;
        gps = 0;
        for (int c = std::min(gps_max, Gk); c >= 1; --c) {
            const int nph = (Gk + c - 1) / c;
            for (int u = umax; u >= 1; u = u > 1 ? (u + 1) / 2 : 0) {
                if (ks > 1 && u < umax) break;
                const int stages = (nmat * u + rps - 1) / rps * nph;
                const int want = std::min(4, stages);
                int n = 0;
                for (int m = std::min(kMaxSlots, stages); m >= want && !n; --m)
                    if (layout(c, u, m, false) <= budget) n = m;
                if (!n) {
                    if (u == 1) break;
                    continue;
                }
                if (ks > 1 && static_cast<size_t>(nmat) * u * kUnitRows * B * 4 > static_cast<size_t>(2 * c) * kHgBytes)
                    break;
                const int passes = (umax + u - 1) / u;
                const double score = 2.0 * Gk / static_cast<double>(nph) - (NT == 1 ? 0.01 : 1.0) * passes;
                if (score > best) {
                    best = score;
                    gps = c;
                    up = u;
                    ns = n;
                }
                break;
            }
        }
        return gps > 0;
    };
    // A K split (clusters of ks CTAs) where each CTA would otherwise hold at most two units: there
    // every CTA would copy all of K's records (4 B x K x B) for a few rows of weights.
    int ks = 1, ncl = std::min(di.num_sms, p.U);
    const int um1 = (p.U + di.num_sms - 1) / di.num_sms;
    for (int k : {4, 2}) {
        if (um1 > 2 || p.G < 32 || NT > 1) continue;   // K >= 8192 (shorter K measured no faster split)
        int n = std::min(di.num_sms / k, p.U);
        if (!plan(k, n)) continue;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(n * k);
        cfg.blockDim = dim3((ncw_per_group * gps + 1) * 32);
        cfg.dynamicSmemBytes = layout(gps, up, ns, false);
        cudaLaunchAttribute a[1];
        a[0].id = cudaLaunchAttributeClusterDimension;
        a[0].val.clusterDim.x = k;
        a[0].val.clusterDim.y = 1;
        a[0].val.clusterDim.z = 1;
        cfg.attrs = a;
        cfg.numAttrs = 1;
        if ((st = ensure_smem_bn(fn, di.device, cfg.dynamicSmemBytes)) != GEM_OK) return st;
        int nmax = 0;
        if (cudaOccupancyMaxActiveClusters(&nmax, fn, &cfg) != cudaSuccess || nmax <= 0) {
            (void)cudaGetLastError();
            continue;
        }
        if (nmax < n) {
            n = nmax;
            if (!plan(k, n)) continue;
        }
        ks = k;
        ncl = n;
        break;
    }
    if (ks == 1 && !plan(1, ncl)) return GEM_OK;   // not planned
    const int C = ncl * ks;
    p.ks = ks;
    p.rps = rps;
    p.up = up;
    p.gps = gps;
    p.nphase = ((p.G + ks - 1) / ks + gps - 1) / gps;
    p.ns = ns;
    p.ncw = ncw_per_group * gps;
    const size_t smem = layout(gps, up, ns, true);

    const int64_t rowbytes = op.K / 32 * 18;
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
    if ((st = ensure_smem_bn(fn, di.device, smem)) != GEM_OK) return st;
    *planned = true;

    PrepParams pp{};
    pp.x = op.x;
    pp.ldx = op.ldx;
    pp.gamma = op.norm_gamma;
    pp.eps = op.eps;
    pp.G = p.G;
    pp.B = B;
    pp.nt = NT;
    pp.nchunk = std::max(1, std::min((32 * p.G + kPrepThreads - 1) / kPrepThreads, std::max(1, 152 / B)));
    pp.rec = rec;
    pp.clear = op.clear;
    pp.nclear = op.nclear;
    pp.rowinfo = reinterpret_cast<float2*>(rec + rec_bytes - kMaxRows * sizeof(float2));
    void* pargs[] = {&pp};
    if ((st = launch_pdl(reinterpret_cast<const void*>(act_prep_kernel), dim3(pp.nchunk, B), dim3(kPrepThreads), 0,
                         stream, pargs)) != GEM_OK)
        return st;
    void* args[] = {&tm0, &tm1, &p};
    return launch_pdl_cluster(fn, dim3(C), dim3((p.ncw + 1) * 32), smem, stream, args, ks);
}

}  // namespace gem
