// gem_gemv.cu — Q4_0 dequantise-and-matvec for decode (B = 1..8 activation rows) and the batched
// prefill GEMM (9..32 rows).
//
// Q4_0 ("gem" engine research record, "Verified model facts"): rows of 18-byte blocks,
// binary16 scale d then 16 bytes of 4-bit codes; weight = (q - 8) * d; byte j carries
// element j (low nibble) and element j + 16 (high nibble).
//
// Dispatch.  When K % 256 == 0 (rows are whole 144-byte groups), the matrices and
// activation rows are 16-byte aligned and the sizes fit 32-bit TMA coordinates, the
// tensor-core kernel of gem_gemv_mma.cuh streams the matrix with TMA (the fast path).  Any
// other K % 32 == 0 shape or alignment takes the general kernel of gem_gemv_kernels.cuh:
// one warp per output row, plain byte loads, the same arithmetic definition.
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

}  // namespace

gem_status gemv_check(const GemvOp& op) {
    if (op.B < 0 || op.N < 0 || op.K < 0) return GEM_ERR_INVALID_ARG;
    if (op.B > kMaxGemmRows) return GEM_ERR_UNSUPPORTED_SHAPE;
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
    p.x = op.x;
    p.ldx = op.ldx;
    p.y = op.y;
    p.ldy = op.ldy;
    p.residual = op.residual;
    p.ldr = op.ldr;
    p.gamma = op.norm_gamma;
    p.eps = op.eps;
    p.act = op.act;
    p.clear = op.clear;
    p.nclear = op.nclear;

    const uintptr_t wbits = reinterpret_cast<uintptr_t>(op.W0) | reinterpret_cast<uintptr_t>(op.W1);
    const uintptr_t xbits = reinterpret_cast<uintptr_t>(op.x) | reinterpret_cast<uintptr_t>(op.norm_gamma);
    const bool fast = op.K > 0 && op.K % 256 == 0 && (wbits & 15) == 0 && (xbits & 15) == 0 &&
                      op.ldx % 4 == 0 && op.N < (int64_t(1) << 31) && op.K / 256 < (1 << 20);
    if (op.B > 8) {
        // 9..32 rows: the column-tiled tensor-core kernel streams the weights once for all rows;
        // where it has no layout (or the shape is not on the fast path) chunks of <= 8 rows
        if (fast) {
            bool planned = false;
            st = gemv_enqueue_bn(op, stream, di, &planned);
            if (planned || st != GEM_OK) return st;
        }
        for (int b0 = 0; b0 < op.B; b0 += 8) {
            GemvOp c = op;
            c.B = std::min(8, op.B - b0);
            c.x = op.x + b0 * op.ldx;
            c.y = op.y + b0 * op.ldy;
            if (op.residual) c.residual = op.residual + b0 * op.ldr;
            if (b0) {
                c.clear = nullptr;
                c.nclear = 0;
            }
            if ((st = gemv_enqueue(c, stream)) != GEM_OK) return st;
        }
        return GEM_OK;
    }
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

    return gemv_enqueue_mma(op, stream, di);
}

}  // namespace gem

extern "C" size_t gem_q4_0_gemv_workspace(int B, int64_t K) {
    if (B < 2 || B > 8 || K <= 0) return 0;
    return gem::align_up(gem::gemv_rec_bytes(B, K), 256);
}

extern "C" size_t gem_q4_0_gemm_workspace(int M, int64_t K) {
    if (M < 2 || M > gem::kMaxGemmRows || K <= 0) return 0;
    return gem::align_up(gem::gemv_rec_bytes(M, K), 256);
}

extern "C" gem_status gem_q4_0_gemm(const void* W0, const void* W1, int64_t N, int64_t K, const float* x, int64_t ldx,
                                    int M, const float* gamma, float eps, int act, float* y, int64_t ldy,
                                    const float* residual, void* workspace, size_t ws_bytes, void* stream) {
    gem::GemvOp op{};
    op.W0 = W0;
    op.W1 = W1;
    op.N = N;
    op.K = K;
    op.B = M;
    op.x = x;
    op.ldx = ldx;
    op.y = y;
    op.ldy = ldy;
    op.residual = residual;
    op.ldr = ldy;
    op.norm_gamma = gamma;
    op.eps = eps;
    op.act = act;
    if (W1 && residual) return GEM_ERR_INVALID_ARG;
    if (gamma && !(eps >= 0.f)) return GEM_ERR_INVALID_ARG;
    gem_status st = gem::gemv_check(op);
    if (st != GEM_OK || M == 0 || N == 0) return st;
    const size_t need = gem_q4_0_gemm_workspace(M, K);
    if (need) {
        if (!workspace || ws_bytes < need) return GEM_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(workspace) & 255) return GEM_ERR_MISALIGNED;
        op.act_ws = workspace;
        op.act_ws_bytes = ws_bytes;
    }
    return gem::gemv_enqueue(op, static_cast<cudaStream_t>(stream));
}

extern "C" gem_status gem_q4_0_gemv_ws(const void* W, int64_t N, int64_t K, const float* x, int64_t ldx, int B,
                                       float* y, int64_t ldy, const float* residual, void* workspace,
                                       size_t ws_bytes, void* stream) {
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
    if (B > 8) return GEM_ERR_UNSUPPORTED_SHAPE;   // 9..32 rows: gem_q4_0_gemm
    gem_status st = gem::gemv_check(op);
    if (st != GEM_OK || B == 0 || N == 0) return st;
    const size_t need = gem_q4_0_gemv_workspace(B, K);
    if (need) {
        if (!workspace || ws_bytes < need) return GEM_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(workspace) & 255) return GEM_ERR_MISALIGNED;
        op.act_ws = workspace;
        op.act_ws_bytes = ws_bytes;
    }
    return gem::gemv_enqueue(op, static_cast<cudaStream_t>(stream));
}

extern "C" gem_status gem_q4_0_gemv_fused(const void* W0, const void* W1, int64_t N, int64_t K, const float* x,
                                          int64_t ldx, int B, const float* gamma, float eps, int act, float* y,
                                          int64_t ldy, const float* residual, void* workspace, size_t ws_bytes,
                                          void* stream) {
    gem::GemvOp op{};
    op.W0 = W0;
    op.W1 = W1;
    op.N = N;
    op.K = K;
    op.B = B;
    op.x = x;
    op.ldx = ldx;
    op.y = y;
    op.ldy = ldy;
    op.residual = residual;
    op.ldr = ldy;
    op.norm_gamma = gamma;
    op.eps = eps;
    op.act = act;
    if (W1 && residual) return GEM_ERR_INVALID_ARG;
    if (gamma && !(eps >= 0.f)) return GEM_ERR_INVALID_ARG;
    if (B > 8) return GEM_ERR_UNSUPPORTED_SHAPE;   // 9..32 rows: gem_q4_0_gemm
    gem_status st = gem::gemv_check(op);
    if (st != GEM_OK || B == 0 || N == 0) return st;
    const size_t need = gem_q4_0_gemv_workspace(B, K);
    if (need) {
        if (!workspace || ws_bytes < need) return GEM_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(workspace) & 255) return GEM_ERR_MISALIGNED;
        op.act_ws = workspace;
        op.act_ws_bytes = ws_bytes;
    }
    return gem::gemv_enqueue(op, static_cast<cudaStream_t>(stream));
}

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
    if (B > 8) return GEM_ERR_UNSUPPORTED_SHAPE;   // 9..32 rows: gem_q4_0_gemm
    return gem::gemv_enqueue(op, static_cast<cudaStream_t>(stream));
}
