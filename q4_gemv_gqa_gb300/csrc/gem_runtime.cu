// gem_runtime.cu — host runtime pieces: status strings, CUDA error recording, per-device
// properties and flag word, tensor-map encoding and PDL launches.
#include <cudaTypedefs.h>

#include <mutex>
#include <set>
#include <utility>
#include <vector>

#include "gem_internal.h"

namespace {

thread_local int g_last_cuda_error = 0;

// One flag word per device; kernels OR GEM_DEVFLAG_* bits into it when the caller passes
// no status pointer of its own.
__device__ int g_device_flags;

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
bool g_dev_ready[kMaxDevices];
gem::DeviceInfo g_dev[kMaxDevices];

// Host handles of every translation unit's wait-limit and test-injection device words.
struct ControlSymbols {
    std::mutex mu;
    std::vector<std::pair<const void*, const void*>> syms;
};
ControlSymbols& control_symbols() {
    static ControlSymbols c;   // constructed on first use (static initialisation order)
    return c;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

}  // namespace

namespace gem {

void register_device_controls(const void* wait_limit_symbol, const void* inject_symbol) {
    ControlSymbols& c = control_symbols();
    std::lock_guard<std::mutex> lk(c.mu);
    c.syms.emplace_back(wait_limit_symbol, inject_symbol);
}

gem_status cuda_fail(cudaError_t e) {
    g_last_cuda_error = static_cast<int>(e);
    return GEM_ERR_CUDA;
}

gem_status device_info(DeviceInfo* out) {
    int dev = 0;
    GEM_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return GEM_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_dev_mutex);
    if (!g_dev_ready[dev]) {
        DeviceInfo d{};
        d.device = dev;
        GEM_CUDA_TRY(cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev));
        int optin = 0;
        GEM_CUDA_TRY(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
        d.smem_optin = static_cast<size_t>(optin);
        void* p = nullptr;
        GEM_CUDA_TRY(cudaGetSymbolAddress(&p, g_device_flags));
        d.status_word = static_cast<int*>(p);
        g_dev[dev] = d;
        g_dev_ready[dev] = true;
    }
    *out = g_dev[dev];
    return GEM_OK;
}

gem_status make_tensor_map_2d(CUtensorMap* tm, CUtensorMapDataType dtype, const void* base, uint64_t dim0,
                              uint64_t dim1, uint64_t stride1_bytes, uint32_t box0, uint32_t box1,
                              CUtensorMapSwizzle swizzle) {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                        cudaEnableDefault, &q);
        if (g_encode_err == cudaSuccess && q != cudaDriverEntryPointSuccess)
            g_encode_err = cudaErrorSymbolNotFound;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (g_encode_err != cudaSuccess || !g_encode) return cuda_fail(g_encode_err);
    cuuint64_t dims[2] = {dim0, dim1};
    cuuint64_t strides[1] = {stride1_bytes};
    cuuint32_t box[2] = {box0, box1};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(tm, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
    return GEM_OK;
}

gem_status launch_pdl(const void* kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                      void** args) {
    return launch_pdl_cluster(kernel, grid, block, smem, stream, args, 1);
}

gem_status launch_pdl_cluster(const void* kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              void** args, int cluster_x) {
    // Every kernel of the library asks for the largest shared-memory carveout, so consecutive
    // launches never need the SM's L1/shared split changed (which would keep a dependent launch
    // from starting on an SM until the previous kernel has drained from it).
    {
        static std::mutex mu;
        static std::set<std::pair<int, const void*>> done;
        int dev = 0;
        GEM_CUDA_TRY(cudaGetDevice(&dev));
        std::lock_guard<std::mutex> lk(mu);
        if (done.insert({dev, kernel}).second)
            GEM_CUDA_TRY(cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                              cudaSharedmemCarveoutMaxShared));
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cluster_x > 1) {
        if (grid.x % static_cast<unsigned>(cluster_x)) return GEM_ERR_INVALID_ARG;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = static_cast<unsigned>(cluster_x);
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    GEM_CUDA_TRY(cudaLaunchKernelExC(&cfg, kernel, args));
    return GEM_OK;
}

}  // namespace gem

extern "C" {

const char* gem_status_string(int status) {
    switch (status) {
        case GEM_OK: return "ok";
        case GEM_ERR_INVALID_ARG: return "invalid argument";
        case GEM_ERR_MISALIGNED: return "misaligned pointer or stride";
        case GEM_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case GEM_ERR_CUDA: return "CUDA runtime error";
        case GEM_ERR_DEVICE_FLAG: return "device-side flag set";
        case GEM_ERR_TIMEOUT: return "device-side wait timed out";
        case GEM_ERR_WORKSPACE: return "workspace missing or too small";
        default: return "unknown status";
    }
}

int gem_last_cuda_error(void) { return g_last_cuda_error; }

gem_status gem_status_from_flags(int32_t flags) {
    if (flags & GEM_DEVFLAG_TIMEOUT) return GEM_ERR_TIMEOUT;
    if (flags) return GEM_ERR_DEVICE_FLAG;
    return GEM_OK;
}

gem_status gem_set_wait_limit(uint64_t ns) {
    if (ns == 0) ns = GEM_WAIT_LIMIT_NS;
    if (ns < 1000ull || ns > 60000000000ull) return GEM_ERR_INVALID_ARG;
    const unsigned long long v = ns;
    ControlSymbols& c = control_symbols();
    std::lock_guard<std::mutex> lk(c.mu);
    for (const auto& sym : c.syms) GEM_CUDA_TRY(cudaMemcpyToSymbol(sym.first, &v, sizeof(v)));
    return GEM_OK;
}

gem_status gem_set_test_injection(int mask) {
    if (mask & ~(GEM_INJECT_RING_SHORTFALL | GEM_INJECT_GRID_ARRIVAL)) return GEM_ERR_INVALID_ARG;
    ControlSymbols& c = control_symbols();
    std::lock_guard<std::mutex> lk(c.mu);
    for (const auto& sym : c.syms) GEM_CUDA_TRY(cudaMemcpyToSymbol(sym.second, &mask, sizeof(mask)));
    return GEM_OK;
}

int gem_version(void) { return 100; }

gem_status gem_device_status(int32_t* flags, int reset) {
    if (!flags) return GEM_ERR_INVALID_ARG;
    gem::DeviceInfo di;
    gem_status st = gem::device_info(&di);
    if (st != GEM_OK) return st;
    int v = 0;
    GEM_CUDA_TRY(cudaMemcpy(&v, di.status_word, sizeof(int), cudaMemcpyDeviceToHost));
    if (reset) GEM_CUDA_TRY(cudaMemset(di.status_word, 0, sizeof(int)));
    *flags = v;
    return GEM_OK;
}

}  // extern "C"
