// gem_elem.cu — the small per-token kernels of the decode step: weighted RMSNorm,
// per-head QK-norm + NeoX/partial RoPE + binary16 KV append, the gated FFN activation and
// the post-norm residual add.  All are memory-trivial (a few KB per token); they exist as
// separate launches only where a grid-wide reduction separates them from a matvec.
#include <cmath>

#include "gem_device.cuh"

namespace gem {
namespace {

__device__ __forceinline__ float act_apply(float g, int act) {
    if (act == 0) return g / (1.0f + __expf(-g));
    const float c = 0.7978845608028654f;  // sqrt(2/pi)
    return 0.5f * g * (1.0f + tanhf(c * (g + 0.044715f * g * g * g)));
}

// block-wide sum; `red` holds blockDim/32 floats
__device__ float block_sum(float v, float* red) {
    v = warp_sum(v);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) red[w] = v;
    __syncthreads();
    float s = 0.f;
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) s += red[i];
    return s;
}

// "gem" research record: weighted RMSNorm over one or many heads.
__global__ void __launch_bounds__(512) rmsnorm_kernel(const float* __restrict__ x, int64_t H,
                                                      const float* __restrict__ gamma, float eps,
                                                      float* __restrict__ out) {
    __shared__ float red[32];
    pdl_wait_trigger();
    const float* xr = x + blockIdx.x * H;
    float* orow = out + blockIdx.x * H;
    float ss = 0.f;
    for (int64_t i = threadIdx.x; i < H; i += blockDim.x) ss = fmaf(xr[i], xr[i], ss);
    const float r = rsqrtf(block_sum(ss, red) / static_cast<float>(H) + eps);
    for (int64_t i = threadIdx.x; i < H; i += blockDim.x) orow[i] = xr[i] * r * (gamma ? gamma[i] : 1.f);
}

// x += RMSNorm(t) * gamma  (post-attention / post-FFN norm before the residual add).
__global__ void __launch_bounds__(512) postnorm_residual_kernel(float* __restrict__ x, const float* __restrict__ t,
                                                                int64_t H, const float* __restrict__ gamma,
                                                                float eps) {
    __shared__ float red[32];
    pdl_wait_trigger();
    const float* tr = t + blockIdx.x * H;
    float* xr = x + blockIdx.x * H;
    float ss = 0.f;
    for (int64_t i = threadIdx.x; i < H; i += blockDim.x) ss = fmaf(tr[i], tr[i], ss);
    const float r = rsqrtf(block_sum(ss, red) / static_cast<float>(H) + eps);
    for (int64_t i = threadIdx.x; i < H; i += blockDim.x) xr[i] += tr[i] * r * gamma[i];
}

__global__ void swiglu_kernel(const float* __restrict__ gate, const float* __restrict__ up, int64_t n, int act,
                              float* __restrict__ out) {
    pdl_wait_trigger();
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        out[i] = act_apply(gate[i], act) * up[i];
}

// One warp per head (Q heads first, then K heads, whose warp also writes the V row).
// GELO section 02/05: per-head RMSNorm with a shared (d,) gamma before RoPE; p-RoPE
// rotates the first rope_dim dims.  "gem" research record: NeoX pairing (i, i + R/2); on
// full-attention layers V is the unweighted RMSNorm of the raw K projection.
constexpr int kRopeWarps = 4;
__global__ void __launch_bounds__(kRopeWarps * 32) qknorm_rope_kernel(const RopeOp op, const RopeFreq fr, int early) {
    __shared__ float buf[kRopeWarps][kMaxHeadDim];
    __shared__ float cs_tab[kMaxHeadDim / 2], sn_tab[kMaxHeadDim / 2];
    if (!early) pdl_wait_trigger();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int b = blockIdx.y;
    const int d = op.d;
    const int p = op.pos[b];
    const bool bad = p < 0 || (op.window == 0 && static_cast<int64_t>(p) >= op.cache_cap);
    if (bad) {
        if (early) pdl_wait_trigger();
        if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(op.status, GEM_DEVFLAG_POS_RANGE);
        return;
    }
    const int R = op.rope_dim, half = R / 2;
    for (int i = threadIdx.x; i < half; i += blockDim.x) {
        float c, s;
        rope_cos_sin(static_cast<double>(p) * fr.w[i], c, s);
        cs_tab[i] = c;
        sn_tab[i] = s;
    }
    if (early) pdl_wait_trigger();  // q/k/v rows come from the preceding projection
    __syncthreads();
    const int head = blockIdx.x * kRopeWarps + w;
    const int nheads = op.n_q + op.n_kv;
    if (head >= nheads) return;
    const bool is_q = head < op.n_q;
    const int j = is_q ? head : head - op.n_q;  // KV head index
    float* row = op.qkv + b * op.ldqkv + static_cast<int64_t>(head) * d;
    float* sb = buf[w];
    const int64_t slot = op.window ? (p % op.window) : p;
    const int64_t crow = ((static_cast<int64_t>(b) * op.n_kv + j) * op.cache_cap + slot) * d;

    // raw head into shared memory
    float ss = 0.f;
    for (int e = lane; e < d; e += 32) {
        const float v = row[e];
        sb[e] = v;
        ss = fmaf(v, v, ss);
    }
    ss = warp_sum(ss);
    if (!is_q) {
        if (op.v_mode == 1) {  // V = unweighted RMSNorm of the raw K row
            const float r = rsqrtf(ss / static_cast<float>(d) + op.eps);
            for (int e = lane; e < d; e += 32) op.v_cache[crow + e] = __half_as_ushort(__float2half_rn(sb[e] * r));
        } else {
            const float* vrow = op.qkv + b * op.ldqkv + static_cast<int64_t>(op.n_q + op.n_kv + j) * d;
            for (int e = lane; e < d; e += 32) op.v_cache[crow + e] = __half_as_ushort(__float2half_rn(vrow[e]));
        }
    }
    const float* gamma = is_q ? op.gamma_q : op.gamma_k;
    if (gamma) {
        const float r = rsqrtf(ss / static_cast<float>(d) + op.eps);
        for (int e = lane; e < d; e += 32) sb[e] = sb[e] * r * gamma[e];
    }
    __syncwarp();
    for (int e = lane; e < d; e += 32) {
        float v = sb[e];
        if (e < R) {
            const int i = e < half ? e : e - half;
            const float c = cs_tab[i], s = sn_tab[i];
            v = e < half ? fmaf(sb[e], c, -sb[e + half] * s) : fmaf(sb[e - half], s, sb[e] * c);
        }
        row[e] = v;
        if (!is_q && op.k_cache) op.k_cache[crow + e] = __half_as_ushort(__float2half_rn(v));
    }
}

}  // namespace

gem_status rmsnorm_enqueue(const float* x, int B, int64_t H, const float* gamma, float eps, float* out,
                           cudaStream_t stream) {
    if (B < 0 || H < 0) return GEM_ERR_INVALID_ARG;
    if (B == 0 || H == 0) return GEM_OK;
    if (!x || !out) return GEM_ERR_INVALID_ARG;
    void* args[] = {&x, &H, &gamma, &eps, &out};
    return launch_pdl(reinterpret_cast<const void*>(rmsnorm_kernel), dim3(B), dim3(512), 0, stream, args);
}

gem_status postnorm_residual_enqueue(float* x, const float* t, int B, int64_t H, const float* gamma, float eps,
                                     cudaStream_t stream) {
    if (B == 0 || H == 0) return GEM_OK;
    void* args[] = {&x, &t, &H, &gamma, &eps};
    return launch_pdl(reinterpret_cast<const void*>(postnorm_residual_kernel), dim3(B), dim3(512), 0, stream,
                      args);
}

gem_status swiglu_enqueue(const float* gate, const float* up, int B, int64_t F, int act, float* out,
                          cudaStream_t stream) {
    if (B < 0 || F < 0 || act < 0 || act > 1) return GEM_ERR_INVALID_ARG;
    const int64_t n = static_cast<int64_t>(B) * F;
    if (n == 0) return GEM_OK;
    if (!gate || !up || !out) return GEM_ERR_INVALID_ARG;
    const int64_t blocks = std::min<int64_t>((n + 255) / 256, 4096);
    void* args[] = {&gate, &up, const_cast<int64_t*>(&n), &act, &out};
    return launch_pdl(reinterpret_cast<const void*>(swiglu_kernel), dim3(static_cast<unsigned>(blocks)), dim3(256),
                      0, stream, args);
}

gem_status rope_check(const RopeOp& op) {
    if (op.B < 0 || op.n_q < 0 || op.n_kv < 0 || op.d <= 0) return GEM_ERR_INVALID_ARG;
    if (op.d > kMaxHeadDim) return GEM_ERR_UNSUPPORTED_SHAPE;
    if (op.rope_dim < 0 || op.rope_dim > op.d || (op.rope_dim & 1)) return GEM_ERR_INVALID_ARG;
    if (op.v_mode < 0 || op.v_mode > 1) return GEM_ERR_INVALID_ARG;
    if (op.window < 0 || op.cache_cap <= 0) return GEM_ERR_INVALID_ARG;
    if (op.window > op.cache_cap) return GEM_ERR_INVALID_ARG;
    if (!(op.theta > 0.f)) return GEM_ERR_INVALID_ARG;
    if (op.B == 0 || op.n_q + op.n_kv == 0) return GEM_OK;
    // a compact full-attention cache (v_mode 1) may keep V rows only: k_cache NULL
    if (!op.qkv || !op.pos || (op.n_kv > 0 && (!op.v_cache || (!op.k_cache && op.v_mode != 1))))
        return GEM_ERR_INVALID_ARG;
    const int64_t need = static_cast<int64_t>(op.n_q + op.n_kv + (op.v_mode ? 0 : op.n_kv)) * op.d;
    if (op.ldqkv < need) return GEM_ERR_INVALID_ARG;
    return GEM_OK;
}

namespace {
gem_status rope_launch(const RopeOp& op_in, cudaStream_t stream, int early) {
    gem_status st = rope_check(op_in);
    if (st != GEM_OK || op_in.B == 0 || op_in.n_q + op_in.n_kv == 0) return st;
    RopeOp op = op_in;
    if (!op.status) {
        DeviceInfo di;
        if ((st = device_info(&di)) != GEM_OK) return st;
        op.status = di.status_word;
    }
    RopeFreq fr{};
    for (int i = 0; i < op.rope_dim / 2; ++i)
        fr.w[i] = std::pow(static_cast<double>(op.theta), -2.0 * i / op.rope_dim);
    dim3 grid((op.n_q + op.n_kv + kRopeWarps - 1) / kRopeWarps, op.B);
    void* args[] = {&op, &fr, &early};
    return launch_pdl(reinterpret_cast<const void*>(qknorm_rope_kernel), grid, dim3(kRopeWarps * 32), 0, stream,
                      args);
}
}  // namespace

gem_status rope_enqueue(const RopeOp& op, cudaStream_t stream) { return rope_launch(op, stream, 0); }
gem_status rope_enqueue_in_chain(const RopeOp& op, cudaStream_t stream) { return rope_launch(op, stream, 1); }

}  // namespace gem

extern "C" {

gem_status gem_rmsnorm(const float* x, int B, int64_t H, const float* gamma, float eps, float* out,
                       void* stream) {
    return gem::rmsnorm_enqueue(x, B, H, gamma, eps, out, static_cast<cudaStream_t>(stream));
}

gem_status gem_rmsnorm_qknorm_rope(float* qkv, int64_t ldqkv, int B, int n_q, int n_kv, int d,
                                   const float* gamma_q, const float* gamma_k, int v_mode, float eps,
                                   const int32_t* pos, float theta, int rope_dim, uint16_t* k_cache,
                                   uint16_t* v_cache, int64_t cache_cap, int window, int32_t* status,
                                   void* stream) {
    gem::RopeOp op{};
    op.qkv = qkv;
    op.ldqkv = ldqkv;
    op.B = B;
    op.n_q = n_q;
    op.n_kv = n_kv;
    op.d = d;
    op.gamma_q = gamma_q;
    op.gamma_k = gamma_k;
    op.v_mode = v_mode;
    op.eps = eps;
    op.pos = pos;
    op.theta = theta;
    op.rope_dim = rope_dim;
    op.k_cache = k_cache;
    op.v_cache = v_cache;
    op.cache_cap = cache_cap;
    op.window = window;
    op.status = status;
    return gem::rope_enqueue(op, static_cast<cudaStream_t>(stream));
}

gem_status gem_swiglu(const float* gate, const float* up, int B, int64_t F, int act, float* out, void* stream) {
    return gem::swiglu_enqueue(gate, up, B, F, act, out, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
