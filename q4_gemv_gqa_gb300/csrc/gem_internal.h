// gem_internal.h — declarations shared by the library's translation units (host side
// plans and launchers; constants shared with device code).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/gem.h"

// Default wall-time limit of every device-side wait on an asynchronous copy or a grid
// barrier (1 s); gem_set_wait_limit() changes it at run time.
#define GEM_WAIT_LIMIT_NS 1000000000ull

namespace gem {

// Called once per translation unit with kernels (static initialisation): the host handles of
// that unit's wait-limit (unsigned long long) and test-injection (int) device words.
void register_device_controls(const void* wait_limit_symbol, const void* inject_symbol);

// Record a CUDA error for gem_last_cuda_error() and map it to a status.
gem_status cuda_fail(cudaError_t e);
#define GEM_CUDA_TRY(expr)                              \
    do {                                                \
        cudaError_t _e = (expr);                        \
        if (_e != cudaSuccess) return gem::cuda_fail(_e); \
    } while (0)

struct DeviceInfo {
    int device;
    int num_sms;
    size_t smem_optin;   // max dynamic shared memory per block
    int* status_word;    // library-owned device flag word
};
// Properties of the current device (cached per device).
gem_status device_info(DeviceInfo* out);

// 2-D tiled tensor map (no interleave).  Returns GEM_ERR_CUDA if encoding fails.
gem_status make_tensor_map_2d(CUtensorMap* tm, CUtensorMapDataType dtype, const void* base,
                              uint64_t dim0, uint64_t dim1, uint64_t stride1_bytes,
                              uint32_t box0, uint32_t box1, CUtensorMapSwizzle swizzle);

// Launch with programmatic stream serialization enabled.
gem_status launch_pdl(const void* kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                      void** args);
// Same, with thread-block clusters of cluster_x CTAs along x (gridDim.x a multiple of it).
gem_status launch_pdl_cluster(const void* kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              void** args, int cluster_x);

// ---- Q4_0 GEMV ----------------------------------------------------------------------------
struct GemvOp {
    const void* W0;            // matrix (gate in pair mode)
    const void* W1;            // up matrix in pair mode, else nullptr
    int64_t N, K;
    int B;
    const float* x; int64_t ldx;
    float* y; int64_t ldy;
    const float* residual; int64_t ldr;   // nullable
    const float* norm_gamma;              // nullable: RMSNorm x first (gamma over K)
    float eps;
    int act;                              // pair mode: 0 SiLU, 1 GELU-tanh
    void* act_ws;                         // nullable: operand records of a 2..8-row call
    size_t act_ws_bytes;                  //   (gemv_rec_bytes); else the library's own array
    unsigned* clear;                      // nullable: words set to zero after the wait (by CTA 0);
    int nclear;                           //   the layer chain clears the next attention's counters
};
gem_status gemv_check(const GemvOp& op);
gem_status gemv_enqueue(const GemvOp& op, cudaStream_t stream);
// Tensor-core path (mma.sync) for the TMA-eligible shapes; called by gemv_enqueue.
gem_status gemv_enqueue_mma(const GemvOp& op, cudaStream_t stream, const DeviceInfo& di);
// One-row (B = 1) tensor-core kernel; *planned = false when K is too long for its shared-memory
// layout (nothing launched).
gem_status gemv_enqueue_b1(const GemvOp& op, cudaStream_t stream, const DeviceInfo& di, bool* planned);
// 2..8 rows: activation prep kernel + tensor-core kernel over operand records; *planned = false
// when no layout fits (nothing launched).  Records live in op.act_ws when it holds
// gemv_rec_bytes(B, K), else in a library-owned per-device array of kGemvRecScratchBytes (shared
// by every call on the device: calls on concurrently running streams must not both use it).
constexpr size_t kGemvRecScratchBytes = size_t(4) << 20;
constexpr int kMaxGemmRows = 32;   // the batched prefill GEMM's activation rows
size_t gemv_rec_bytes(int B, int64_t K);
gem_status gemv_enqueue_bn(const GemvOp& op, cudaStream_t stream, const DeviceInfo& di, bool* planned);
// 2..8 rows in one launch: tall TMA tiles, activation operands built in the kernel (no records).
gem_status gemv_enqueue_wide(const GemvOp& op, cudaStream_t stream, const DeviceInfo& di);

// ---- norms / RoPE / activation -------------------------------------------------------------
struct RopeOp {
    float* qkv; int64_t ldqkv;
    int B, n_q, n_kv, d;
    const float *gamma_q, *gamma_k;
    int v_mode;
    float eps;
    const int32_t* pos;
    float theta;
    int rope_dim;
    uint16_t *k_cache, *v_cache;
    int64_t cache_cap;
    int window;
    int32_t* status;
};
gem_status rope_check(const RopeOp& op);
gem_status rope_enqueue(const RopeOp& op, cudaStream_t stream);
// Same, inside a layer chain: positions are read before griddepcontrol.wait (the preceding
// kernel does not write them), so the rotation table is built while it still runs.
gem_status rope_enqueue_in_chain(const RopeOp& op, cudaStream_t stream);

gem_status rmsnorm_enqueue(const float* x, int B, int64_t H, const float* gamma, float eps, float* out,
                           cudaStream_t stream);
gem_status swiglu_enqueue(const float* gate, const float* up, int B, int64_t F, int act, float* out,
                          cudaStream_t stream);
// x[b] += RMSNorm(t[b]) * gamma   (Gemma post-attention / post-FFN norm before the residual add)
gem_status postnorm_residual_enqueue(float* x, const float* t, int B, int64_t H, const float* gamma,
                                     float eps, cudaStream_t stream);

// ---- attention -----------------------------------------------------------------------------
struct AttnOp {
    const float* q; int64_t ldq;
    const uint16_t *k_cache, *v_cache;
    int B, n_q, n_kv, d;
    int64_t cache_cap;
    const int32_t* pos;
    int window;
    float scale;
    float* out; int64_t ldo;
    void* workspace; size_t ws_bytes;
    int32_t* status;
    // Fused QK-norm / RoPE / KV append (attn_enqueue_fused): q points at the raw QKV
    // projection row (Q heads, K heads, then V heads unless v_mode == 1).
    const float *gamma_q, *gamma_k;   // nullable
    float eps, theta;
    int rope_dim, v_mode;
    uint16_t *k_out, *v_out;           // the same caches, written at the new slot
};

// Rotation frequencies theta^(-2i/R), i < R/2, computed on the host in fp64.
constexpr int kMaxHeadDim = 512;
struct RopeFreq {
    double w[kMaxHeadDim / 2];
};
size_t attn_workspace_bytes(int B, int n_q, int n_kv, int d, int64_t cache_cap, int window);
// Byte offset (in the attention workspace) and size of the flash kernel's arrival counters;
// *bytes = 0 when the plan has none.  The counters are zero between calls.
size_t attn_counter_offset(int B, int n_q, int n_kv, int d, int64_t cache_cap, int window, size_t* bytes);
gem_status attn_check(const AttnOp& op);
gem_status attn_enqueue(const AttnOp& op, cudaStream_t stream);
// Same, for use right after the RoPE/append kernel of a layer step: positions and the
// cached rows are read before griddepcontrol.wait (the preceding kernel writes neither,
// except the new token's row, which is re-read after the wait).
gem_status attn_enqueue_in_chain(const AttnOp& op, cudaStream_t stream);
// Inside a layer chain, right after the QKV projection: the attention kernel itself applies
// QK-norm and RoPE to its query heads and appends the new K/V row (no separate RoPE launch).
// Only for shapes that attn_fusable() accepts.
bool attn_fusable(int n_q, int n_kv, int d);
gem_status attn_enqueue_fused(const AttnOp& op, cudaStream_t stream);
gem_status attn_enqueue_fused_standalone(const AttnOp& op, cudaStream_t stream);

// Attention over a compact full-attention cache (V rows only; K_j = RoPE_j(V_j * gamma_k)).
struct CompactAttnOp {
    const float* q; int64_t ldq;      // normalised and rotated query heads
    const uint16_t* v_cache;          // [B][n_kv][cap][d] binary16
    int B, n_q, n_kv, d;
    int64_t cache_cap;
    const int32_t* pos;
    float scale;
    const float* gamma_k;             // [d]
    int rope_dim;                     // multiple of 16
    float theta;
    float* out; int64_t ldo;
    void* workspace; size_t ws_bytes;
    int32_t* status;
};
gem_status compact_check(const CompactAttnOp& op);
size_t compact_workspace_bytes(int B, int n_q, int n_kv, int d, int64_t cache_cap, int rope_dim);
// early: positions and the cached rows are requested before griddepcontrol.wait (inside the
// layer chain, after the QK-norm / RoPE / V-append launch, whose new row is re-read after it)
gem_status compact_enqueue(const CompactAttnOp& op, cudaStream_t stream, bool early);

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace gem
