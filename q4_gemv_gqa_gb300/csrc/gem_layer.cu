// gem_layer.cu — one decoder layer step as a chain of PDL-linked launches.
//
// GELO LLM generation, section 06 (block topology: pre-norm, merged QKV, QK-norm, RoPE,
// GQA over the cache, O projection + residual, pre-FFN norm, merged gate/up, gated
// activation, down projection + residual).  "gem" research record, "Verified model
// facts": Gemma 4 full-attention layers have no V projection; V is the unweighted RMSNorm
// of the K projection.
//
//   1  QKV GEMV, pre-attention RMSNorm fused into its activation staging
//   2  QK-norm + RoPE + binary16 KV append (head_dim <= 256 and n_q / n_kv <= 4: inside 3)
//   3  split-K GQA attention (+ ordered merge launch when the range is split)
//   4  O GEMV with the residual add fused (post_norms: O GEMV, then norm + residual)
//   5  gate/up GEMV pair, pre-FFN RMSNorm fused in, gated activation in the epilogue
//   6  down GEMV with the residual add fused (post_norms: down GEMV, then norm + residual)
// compact_kv (full-attention layers with V from K): 2 appends the V row only and 3 is the
// compact-cache attention, which rebuilds K_j = RoPE_j(V_j * gamma_k) from the V rows.
// Every kernel requests its weights (or cached K/V rows) before griddepcontrol.wait, so
// each launch's HBM stream starts while its predecessor is still running.
#include <algorithm>

#include "gem_internal.h"

namespace gem {
namespace {

struct LayerWs {
    float *qkv, *attn, *act, *tmp;
    void* attn_ws;
    size_t attn_ws_bytes;
    void* rec;            // GEMV operand records (2..8 rows), shared by the layer's GEMVs in turn
    size_t rec_bytes;
    size_t total;
};

LayerWs layout(const gem_layer_desc* L, int B, int64_t cap, void* base) {
    LayerWs w{};
    const int64_t nqkv = (L->n_q + L->n_kv + (L->v_from_k ? 0 : L->n_kv)) * L->d;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 256);
        return static_cast<char*>(base) + o;
    };
    w.qkv = reinterpret_cast<float*>(take(sizeof(float) * B * nqkv));
    w.attn = reinterpret_cast<float*>(take(sizeof(float) * B * L->n_q * L->d));
    w.act = reinterpret_cast<float*>(take(sizeof(float) * B * L->F));
    w.tmp = reinterpret_cast<float*>(take(sizeof(float) * B * L->H));
    w.attn_ws_bytes = L->compact_kv
                          ? compact_workspace_bytes(B, static_cast<int>(L->n_q), static_cast<int>(L->n_kv),
                                                    static_cast<int>(L->d), cap, L->rope_dim)
                          : attn_workspace_bytes(B, static_cast<int>(L->n_q), static_cast<int>(L->n_kv),
                                                 static_cast<int>(L->d), cap, L->window);
    w.attn_ws = take(w.attn_ws_bytes);
    const int64_t kmax = std::max<int64_t>(std::max<int64_t>(L->H, L->n_q * L->d), L->F);
    w.rec_bytes = gemv_rec_bytes(B, kmax);
    w.rec = w.rec_bytes ? take(w.rec_bytes) : nullptr;
    w.total = off;
    return w;
}

gem_status check_desc(const gem_layer_desc* L, int B) {
    if (!L) return GEM_ERR_INVALID_ARG;
    if (B < 0) return GEM_ERR_INVALID_ARG;
    if (B > 8) return GEM_ERR_UNSUPPORTED_SHAPE;
    if (L->H <= 0 || L->n_q <= 0 || L->n_kv <= 0 || L->d <= 0 || L->F <= 0) return GEM_ERR_INVALID_ARG;
    if (L->n_q % L->n_kv) return GEM_ERR_INVALID_ARG;
    if (!L->w_qkv || !L->w_o || !L->w_gate || !L->w_up || !L->w_down || !L->g_attn || !L->g_ffn)
        return GEM_ERR_INVALID_ARG;
    if (L->qk_norm && (!L->g_q || !L->g_k)) return GEM_ERR_INVALID_ARG;
    if (L->post_norms && (!L->g_post_attn || !L->g_post_ffn)) return GEM_ERR_INVALID_ARG;
    if (L->act < 0 || L->act > 1) return GEM_ERR_INVALID_ARG;
    // the compact cache rebuilds K from V * gamma_k: V from K, QK-norm, full attention
    if (L->compact_kv && (!L->v_from_k || !L->qk_norm || L->window)) return GEM_ERR_INVALID_ARG;
    return GEM_OK;
}

}  // namespace
}  // namespace gem

extern "C" {

size_t gem_decode_layer_workspace(const gem_layer_desc* L, int B, int64_t cache_cap) {
    if (gem::check_desc(L, B) != GEM_OK || B == 0 || cache_cap <= 0) return 0;
    return gem::layout(L, B, cache_cap, nullptr).total;
}

gem_status gem_decode_layer(const gem_layer_desc* L, int B, float* x, uint16_t* k_cache, uint16_t* v_cache,
                            int64_t cache_cap, const int32_t* pos, void* workspace, size_t ws_bytes,
                            int32_t* status, void* stream_v) {
    using namespace gem;
    gem_status st = check_desc(L, B);
    if (st != GEM_OK || B == 0) return st;
    if (!x || (!k_cache && !L->compact_kv) || !v_cache || !pos) return GEM_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return GEM_ERR_MISALIGNED;
    const LayerWs w = layout(L, B, cache_cap, workspace);
    if (!workspace || ws_bytes < w.total) return GEM_ERR_WORKSPACE;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    const int64_t H = L->H, d = L->d, nq = L->n_q, nkv = L->n_kv, F = L->F;
    const int64_t nqkv = (nq + nkv + (L->v_from_k ? 0 : nkv)) * d;

    // validate every stage before enqueueing any of them
    GemvOp qkv{L->w_qkv, nullptr, nqkv, H, B, x, H, w.qkv, nqkv, nullptr, 0, L->g_attn, L->eps, 0};
    GemvOp oproj{L->w_o, nullptr, H, nq * d, B, w.attn, nq * d, L->post_norms ? w.tmp : x, H,
                 L->post_norms ? nullptr : x, H, nullptr, 0.f, 0};
    GemvOp gateup{L->w_gate, L->w_up, F, H, B, x, H, w.act, F, nullptr, 0, L->g_ffn, L->eps, L->act};
    GemvOp down{L->w_down, nullptr, H, F, B, w.act, F, L->post_norms ? w.tmp : x, H,
                L->post_norms ? nullptr : x, H, nullptr, 0.f, 0};
    for (GemvOp* op : {&qkv, &oproj, &gateup, &down}) {
        op->act_ws = w.rec;
        op->act_ws_bytes = w.rec_bytes;
    }
    RopeOp rope{};
    rope.qkv = w.qkv;
    rope.ldqkv = nqkv;
    rope.B = B;
    rope.n_q = static_cast<int>(nq);
    rope.n_kv = static_cast<int>(nkv);
    rope.d = static_cast<int>(d);
    rope.gamma_q = L->qk_norm ? L->g_q : nullptr;
    rope.gamma_k = L->qk_norm ? L->g_k : nullptr;
    rope.v_mode = L->v_from_k ? 1 : 0;
    rope.eps = L->eps;
    rope.pos = pos;
    rope.theta = L->theta;
    rope.rope_dim = L->rope_dim;
    rope.k_cache = L->compact_kv ? nullptr : k_cache;
    rope.v_cache = v_cache;
    rope.cache_cap = cache_cap;
    rope.window = L->window;
    rope.status = status;
    AttnOp attn{};
    attn.q = w.qkv;
    attn.ldq = nqkv;
    attn.k_cache = k_cache;
    attn.v_cache = v_cache;
    attn.B = B;
    attn.n_q = static_cast<int>(nq);
    attn.n_kv = static_cast<int>(nkv);
    attn.d = static_cast<int>(d);
    attn.cache_cap = cache_cap;
    attn.pos = pos;
    attn.window = L->window;
    attn.scale = L->scale;
    attn.out = w.attn;
    attn.ldo = nq * d;
    attn.workspace = w.attn_ws;
    attn.ws_bytes = w.attn_ws_bytes;
    attn.status = status;
    // flash-eligible shapes: QK-norm, RoPE and the KV append run inside the attention kernel
    const bool fused = !L->compact_kv && attn_fusable(static_cast<int>(nq), static_cast<int>(nkv), static_cast<int>(d));
    if (fused) {
        attn.gamma_q = rope.gamma_q;
        attn.gamma_k = rope.gamma_k;
        attn.eps = L->eps;
        attn.theta = L->theta;
        attn.rope_dim = L->rope_dim;
        attn.v_mode = rope.v_mode;
        attn.k_out = k_cache;
        attn.v_out = v_cache;
    }
    if (fused) {   // the QKV projection clears the attention's arrival counters for it
        size_t cbytes = 0;
        const size_t coff = attn_counter_offset(B, static_cast<int>(nq), static_cast<int>(nkv), static_cast<int>(d),
                                                cache_cap, L->window, &cbytes);
        if (cbytes) {
            qkv.clear = reinterpret_cast<unsigned*>(static_cast<char*>(w.attn_ws) + coff);
            qkv.nclear = static_cast<int>(cbytes / sizeof(unsigned));
        }
    }
    if ((st = gemv_check(qkv)) != GEM_OK || (st = gemv_check(oproj)) != GEM_OK ||
        (st = gemv_check(gateup)) != GEM_OK || (st = gemv_check(down)) != GEM_OK ||
        (st = rope_check(rope)) != GEM_OK || (!L->compact_kv && (st = attn_check(attn)) != GEM_OK))
        return st;

    CompactAttnOp cat{};
    if (L->compact_kv) {
        cat.q = w.qkv;
        cat.ldq = nqkv;
        cat.v_cache = v_cache;
        cat.B = B;
        cat.n_q = static_cast<int>(nq);
        cat.n_kv = static_cast<int>(nkv);
        cat.d = static_cast<int>(d);
        cat.cache_cap = cache_cap;
        cat.pos = pos;
        cat.scale = L->scale;
        cat.gamma_k = L->g_k;
        cat.rope_dim = L->rope_dim;
        cat.theta = L->theta;
        cat.out = w.attn;
        cat.ldo = nq * d;
        cat.workspace = w.attn_ws;
        cat.ws_bytes = w.attn_ws_bytes;
        cat.status = status;
        if ((st = compact_check(cat)) != GEM_OK) return st;
    }

    if ((st = gemv_enqueue(qkv, stream)) != GEM_OK) return st;
    if (L->compact_kv) {
        if ((st = rope_enqueue_in_chain(rope, stream)) != GEM_OK) return st;
        if ((st = compact_enqueue(cat, stream, true)) != GEM_OK) return st;
    } else if (fused) {
        if ((st = attn_enqueue_fused(attn, stream)) != GEM_OK) return st;
    } else {
        if ((st = rope_enqueue_in_chain(rope, stream)) != GEM_OK) return st;
        if ((st = attn_enqueue_in_chain(attn, stream)) != GEM_OK) return st;
    }
    if ((st = gemv_enqueue(oproj, stream)) != GEM_OK) return st;
    if (L->post_norms && (st = postnorm_residual_enqueue(x, w.tmp, B, H, L->g_post_attn, L->eps, stream)) != GEM_OK)
        return st;
    if ((st = gemv_enqueue(gateup, stream)) != GEM_OK) return st;
    if ((st = gemv_enqueue(down, stream)) != GEM_OK) return st;
    if (L->post_norms && (st = postnorm_residual_enqueue(x, w.tmp, B, H, L->g_post_ffn, L->eps, stream)) != GEM_OK)
        return st;
    return GEM_OK;
}

}  // extern "C"
