// gem_step.cu — the whole decode step (every layer) as one persistent kernel.
//
// GELO LLM generation, section 06 (block topology); sections 02/05 (QK-norm, RoPE, GQA
// decode over the cache); "gem" research record (Q4_0 blocks, decode-attention notes:
// partial attention states over disjoint ranges compose and are merged in ascending
// order).  The arithmetic of every step is that of the separate kernels (gem_gemv_mma,
// gem_attn, gem_elem); what changes is the schedule.
//
// Why one kernel.  A decode layer at batch 1 moves ~45 MB (Qwen3-1.7B shape), which HBM
// streams in ~7 us, but as a chain of seven launches each boundary costs a few
// microseconds of launch, first-byte latency and tail, and the large GEMV CTAs cannot be
// co-resident with their successor, so the next launch's weight stream cannot start early.
// Here one cooperative launch runs every layer: grid = one CTA per SM, 16 consumer warps
// and one producer warp per CTA.
//
// The producer warp walks the CTA's whole schedule (per layer: QKV weights, the K/V stages
// of its attention items, O, gate/up, down weights) and streams each stage by TMA into a
// ring of kNs slots, waiting only for free slots.  Weights and old cache rows never
// depend on the step's activations, so the stream runs ahead across phase boundaries:
// while the consumers wait at a grid barrier, the next phase's data is already landing.
//
// The consumer warps walk the same schedule.  Phases of a layer, separated by grid
// barriers (bounded waits; a timeout raises a global abort flag that every wait checks):
//   1  QKV GEMV, the pre-attention RMSNorm fused into the activation staging;
//   2  attention items (kv head, sequence, split): QK-norm and RoPE of the item's query
//      heads; the item that holds the new token's slot also normalises and rotates the
//      new K row, rounds K and V to binary16, writes them to the cache and patches its
//      staged copy; split-K flash attention over the item's stages; the last split of a
//      (sequence, kv head) to finish merges all splits in ascending order;
//   3  O GEMV + residual;  4  gate/up GEMV pair, pre-FFN RMSNorm fused, SwiGLU epilogue;
//   5  down GEMV + residual.
// Every consumer warp passes through every ring stage in order (a GEMV stage is shared by
// all warps; an attention stage is computed by one warp and skipped by the others), so
// each slot's full/empty barriers are always waited on in phase order.
//
// Scope: Qwen-style layers (no post-norms, separate V projection), head_dim 64/128/256,
// n_q / n_kv <= 4, batch <= 4, every GEMV with K % 256 == 0.  Other shapes use the
// per-layer chain (gem_decode_layer).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

#include "gem_device.cuh"

struct gem_step_plan;

namespace gem {
namespace step {

constexpr int kNcw = 16;                       // consumer warps
constexpr int kThreads = (kNcw + 1) * 32;
constexpr int kNs = 6;                         // ring slots
constexpr int kGroupBytes = 144;               // 256 Q4_0 weights of one row
constexpr int kUnitRows = 16;
constexpr int kBoxBytes = kGroupBytes * kUnitRows;
constexpr int kSlot = 8 * kBoxBytes;           // 18432: 8 groups x 16 rows, or one K+V stage (16 KB)
constexpr int kKVStage = 16384;
constexpr int kScratch = 96 * 1024;
constexpr int kRingBytes = kNs * kSlot;
constexpr int kBarOff = kRingBytes;
constexpr int kScrOff = kRingBytes + 256;
constexpr int kRopeOff = kScrOff + kScratch;       // [kMaxB][cos 128 | sin 128] of the current layer
constexpr size_t kSmemBytes = 1024 + kRopeOff + 4 * 256 * 4;   // + slack for the 1024-byte alignment
constexpr int kMaxB = 4;

struct GemvPlan {
    int N, K, G, U, gps, nphase;
    int resident;   // all K-phases' activation fragments fit the scratch at once
};

__host__ __device__ constexpr size_t aup(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layer {
    CUtensorMap tm_qkv, tm_o, tm_gate, tm_up, tm_down, tm_k, tm_v;
    const float *g_attn, *g_ffn, *g_q, *g_k;
    uint16_t *k_cache, *v_cache;
    const double* rope_w;     // theta^(-2i/R), i < R/2 (fp64)
    int64_t cap;
    int H, n_q, n_kv, d, F, n_qkv, rope_dim, window, act, qk_norm;
    float eps, scale;
    int nsplit_max;
    GemvPlan qkv, o, gu, down;
};

struct Sync {
    unsigned long long arrived;   // monotonic: barrier k of the kernel's life ends at (k + 1) * CTAs
    int abort;
};

struct Params {
    const Layer* layers;
    int nlayers, B;
    float* x;
    const int32_t* pos;
    float *qkv, *attn, *act, *part;
    unsigned* merge_cnt;     // [B * n_kv] arrival counters, back to 0 after each merge
    Sync* sync;
    int* status;
};

__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"r"(kNcw * 32) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ unsigned long long ld_acquire64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long atom_add_release64(unsigned long long* p, unsigned long long v) {
    unsigned long long old;
    asm volatile("atom.add.release.gpu.global.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
    return old;
}

__device__ __forceinline__ int ld_volatile(const int* p) { return *reinterpret_cast<const volatile int*>(p); }

__device__ __forceinline__ void tma_load_box(void* dst, const CUtensorMap* tm, int c0, int c1, uint64_t* bar,
                                             uint64_t policy) {
    tma_load_2d(dst, tm, c0, c1, bar, policy);
}

// Bounded wait on a ring barrier that also gives up when the step was aborted (by any CTA)
// or this CTA's consumers stopped.  A wait that runs out of time records
// GEM_DEVFLAG_TIMEOUT and aborts the step for every CTA.
__device__ bool ring_wait(uint64_t* bar, uint32_t par, Sync* sync, const volatile int* stop, int* status) {
    if (mbar_try_wait(bar, par)) return true;
    const uint64_t t0 = globaltimer_ns();
    const uint64_t limit = wait_limit_ns();
    for (;;) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, par)) return true;
        if (*stop || ld_volatile(&sync->abort)) return false;
        if (globaltimer_ns() - t0 > limit) {
            atomicOr(status, GEM_DEVFLAG_TIMEOUT);
            atomicExch(&sync->abort, 1);
            return false;
        }
    }
}

struct Ring {
    int slot;
    uint32_t par;
    __device__ __forceinline__ void next() {
        if (++slot == kNs) {
            slot = 0;
            par ^= 1u;
        }
    }
};

__device__ __forceinline__ int split_lo(int n, int parts, int i) {
    return static_cast<int>((static_cast<int64_t>(i) * n) / parts);
}

// The attention item list: item = ((b * n_kv + g) * nsplit_max + split); returns false for
// an item with no work (bad position, or a split beyond the sequence's stage count).
template <int D>
__device__ __forceinline__ bool attn_item(const Layer& L, const int32_t* pos, int item, int& b, int& g, int& split, int& p,
                          int& T, int& nsplit, int& s0, int& s1) {
    constexpr int PS = 4096 / D;
    split = item % L.nsplit_max;
    const int bg = item / L.nsplit_max;
    g = bg % L.n_kv;
    b = bg / L.n_kv;
    p = pos[b];
    if (p < 0 || (L.window == 0 && static_cast<int64_t>(p) >= L.cap)) return false;
    T = L.window ? min(L.window, p + 1) : p + 1;
    const int nst = (T + PS - 1) / PS;
    nsplit = min(L.nsplit_max, nst);
    if (split >= nsplit) return false;
    s0 = split_lo(nst, nsplit, split);
    s1 = split_lo(nst, nsplit, split + 1);
    return true;
}

// ================================ producer =====================================================
template <int D>
__device__ __forceinline__ void producer(const Params& P, uint8_t* smem, uint64_t* full, uint64_t* empty, volatile int* stop) {
    constexpr int PS = 4096 / D;
    const int C = gridDim.x, c = blockIdx.x;
    const uint64_t policy = l2_policy_evict_first();
    int s = 0, slot = 0;
    uint32_t epar = 1;
    bool ok = true;
    auto acquire = [&]() -> uint8_t* {   // next free slot (waits from the second lap on)
        if (s >= kNs && !ring_wait(&empty[slot], epar, P.sync, stop, P.status)) {
            ok = false;
            return nullptr;
        }
        return smem + slot * kSlot;
    };
    auto advance = [&]() {
        ++s;
        if (++slot == kNs) {
            slot = 0;
            epar ^= 1u;
        }
    };
    auto gemv = [&](const GemvPlan& pl, const CUtensorMap* tm0, const CUtensorMap* tm1, int nmat) {
        const int u0 = split_lo(pl.U, C, c), u1 = split_lo(pl.U, C, c + 1);
        for (int ph = 0; ph < pl.nphase && ok; ++ph) {
            const int g0 = ph * pl.gps, ng = min(pl.gps, pl.G - g0);
            for (int u = u0; u < u1 && ok; ++u)
                for (int m = 0; m < nmat && ok; ++m) {
                    uint8_t* dst = acquire();
                    if (!dst) break;
                    mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(ng * kBoxBytes));
                    for (int j = 0; j < ng; ++j)
                        tma_load_box(dst + j * kBoxBytes, m ? tm1 : tm0, (g0 + j) * kGroupBytes, u * kUnitRows,
                                     &full[slot], policy);
                    advance();
                }
        }
    };
    for (int l = 0; l < P.nlayers && ok; ++l) {
        const Layer& L = P.layers[l];
        gemv(L.qkv, &L.tm_qkv, nullptr, 1);
        const int nitems = P.B * L.n_kv * L.nsplit_max;
        for (int it = c; it < nitems && ok; it += C) {
            int b, g, split, p, T, nsplit, s0, s1;
            if (!attn_item<D>(L, P.pos, it, b, g, split, p, T, nsplit, s0, s1)) continue;
            const int row0 = (b * L.n_kv + g) * static_cast<int>(L.cap);
            for (int st = s0; st < s1 && ok; ++st) {
                uint8_t* dst = acquire();
                if (!dst) break;
                mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(kKVStage));
                for (int j = 0; j < D / 64; ++j) {
                    tma_load_box(dst + j * PS * 128, &L.tm_k, j * 64, row0 + st * PS, &full[slot], policy);
                    tma_load_box(dst + kKVStage / 2 + j * PS * 128, &L.tm_v, j * 64, row0 + st * PS, &full[slot],
                                 policy);
                }
                advance();
            }
        }
        gemv(L.o, &L.tm_o, nullptr, 1);
        gemv(L.gu, &L.tm_gate, &L.tm_up, 2);
        gemv(L.down, &L.tm_down, nullptr, 1);
    }
    // copies still in flight land before the CTA exits (bounded)
    for (int i = max(0, s - kNs); i < s; ++i) (void)mbar_wait(&full[i % kNs], static_cast<uint32_t>((i / kNs) & 1), nullptr);
}

// ================================ consumers ====================================================
struct Ctx {
    const Params* P;
    uint8_t* smem;
    uint64_t *full, *empty;
    uint8_t* scr;
    volatile int* stop;
    Ring ring;
    bool ok;
    __device__ bool wait_full() {
        if (!ok) return false;
        ok = ring_wait(&full[ring.slot], ring.par, P->sync, stop, P->status);
        return ok;
    }
    __device__ void release() {
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(&empty[ring.slot]);
        ring.next();
    }
};

// Grid-wide barrier of the consumer warps (the producer warps never join one).  One
// release-add on a monotonic arrival counter per CTA; a CTA leaves when the counter
// reaches the end of its barrier's round (acquire loads), so no reset or second flag is
// needed and the last arrival releases everyone with its own add.
// Test hook (GEM_INJECT_GRID_ARRIVAL): CTA 0 leaves out its arrival at the first barrier of
// the step, so every CTA's wait runs out; the step is aborted (the plan must be recreated).
__device__ __forceinline__ bool grid_sync(Ctx& cx, bool first) {
    __shared__ int ok_sh;
    consumer_sync();
    if (threadIdx.x == 0) {
        Sync* sy = cx.P->sync;
        bool ok = cx.ok;
        const unsigned long long C = gridDim.x;
        const bool skip = first && blockIdx.x == 0 && (test_inject() & GEM_INJECT_GRID_ARRIVAL);
        const unsigned long long old = skip ? ld_acquire64(&sy->arrived) : atom_add_release64(&sy->arrived, 1ull);
        const unsigned long long target = (old / C + 1) * C;
        if (ld_acquire64(&sy->arrived) < target) {
            const uint64_t t0 = globaltimer_ns();
            const uint64_t limit = wait_limit_ns();
            while (ld_acquire64(&sy->arrived) < target) {
                if (ld_volatile(&sy->abort)) {
                    ok = false;
                    break;
                }
                if (globaltimer_ns() - t0 > limit) {
                    atomicOr(cx.P->status, GEM_DEVFLAG_TIMEOUT);
                    atomicExch(&sy->abort, 1);
                    ok = false;
                    break;
                }
            }
        }
        if (ld_volatile(&sy->abort)) ok = false;
        ok_sh = ok;
    }
    consumer_sync();
    cx.ok = ok_sh != 0;
    return cx.ok;
}

__device__ __forceinline__ float act_fn(float g, int act) {
    if (act == 0) return g / (1.0f + __expf(-g));
    const float c = 0.7978845608028654f;  // sqrt(2/pi)
    return 0.5f * g * (1.0f + tanhf(c * (g + 0.044715f * g * g * g)));
}

template <int JPAR>
__device__ __forceinline__ uint32_t code_word(const uint8_t* row, int jj, int t) {
    const int off = 18 * jj + 2 + 4 * t;
    if constexpr (JPAR == 1) return *reinterpret_cast<const uint32_t*>(row + off);
    else return __funnelshift_r(*reinterpret_cast<const uint32_t*>(row + off - 2),
                                *reinterpret_cast<const uint32_t*>(row + off + 2), 16);
}

__device__ __forceinline__ uint32_t lop3_mask_or(uint32_t a, uint32_t mask, uint32_t orv) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(orv));
    return d;
}
__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t hfma2_bits(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// Exact codes q - 8 as binary16 pairs (exponent magic 0x6400 = 1024), as in the GEMV kernel.
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t& t0a, uint32_t& t0b, uint32_t& t1a,
                                             uint32_t& t1b) {
    const uint32_t w8 = w >> 8;
    t0a = hsub2_bits(lop3_mask_or(w, 0x000F000Fu, 0x64006400u), 0x64086408u);
    t0b = hsub2_bits(lop3_mask_or(w8, 0x000F000Fu, 0x64006400u), 0x64086408u);
    t1a = hfma2_bits(lop3_mask_or(w, 0x00F000F0u, 0x64006400u), 0x2C002C00u, 0xD480D480u);
    t1b = hfma2_bits(lop3_mask_or(w8, 0x00F000F0u, 0x64006400u), 0x2C002C00u, 0xD480D480u);
}

// B fragment entry (B <= 4, columns 2b = hi, 2b + 1 = lo): (half group, block, quad t, column)
__device__ __forceinline__ uint32_t xf_entry(int hg, int j, int t, int n, int B) {
    return static_cast<uint32_t>((((hg * 4 + j) * 4 + t) * (2 * B) + n) * 16);
}

// One GEMV phase: y = W(norm(x)) (+ residual) or act(gate) * up for the pair.
// Activations of all K-phases are converted at once when they fit (one round of global
// loads after the grid barrier), else one K-phase at a time.
template <int NMAT>
__device__ __forceinline__ void gemv_phase(Ctx& cx, const GemvPlan& pl, const float* in, int ldx, const float* gamma,
                                           float eps, float* out, int ldy, const float* residual, int act) {
    const Params& P = *cx.P;
    const int B = P.B;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nct = kNcw * 32;
    const int C = gridDim.x, c = blockIdx.x;
    const int u0 = split_lo(pl.U, C, c), u1 = split_lo(pl.U, C, c + 1);
    const int nup = u1 - u0;
    const int kp = pl.gps * 256, nhg = kp / 128, kp4 = kp / 4;
    const bool resident = pl.resident != 0;
    const int nbuf = resident ? pl.nphase : 1;
    // scratch: xf [nbuf][4 B kp] | xsc [nbuf][nhg B] | ssq [B 2G] | red [NMAT nup 16][kNcw][B] | rstd [B]
    uint8_t* xf0 = cx.scr;
    const size_t xf_bytes = 4ull * B * kp;
    float* xsc0 = reinterpret_cast<float*>(xf0 + aup(nbuf * xf_bytes, 128));
    float* ssq = xsc0 + aup(nbuf * nhg * B, 32);
    float* red = ssq + aup(B * 2 * pl.G, 32);
    float* rstd = red + NMAT * nup * kUnitRows * kNcw * B;
    const int g = lane >> 2, t = lane & 3;
    const int jg = warp >> 1, eta = warp & 1, hg = jg * 2 + eta;
    const bool col_ok = g < 2 * B;
    const int nw = 2 * pl.gps;   // warps that own a half group (the others only pass through)

    // K-phases [q0, q0 + nq) -> buffers (q - q0): loads first (up to 4 slots per thread), then
    // the conversions, so the global latency is paid once per round.
    auto convert = [&](int q0, int nq) {
        const int per = B * kp4;
        const int total = nq * per;
        for (int f0 = tid; f0 < total; f0 += 4 * nct) {
            float4 xv[4], gv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int f = f0 + i * nct;
                xv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                gv[i] = make_float4(1.f, 1.f, 1.f, 1.f);
                if (f < total) {
                    const int q = q0 + f / per, r = f % per;
                    const int b = r / kp4, e = (r - b * kp4) * 4;
                    const int k = q * kp + e;
                    if (k < pl.K) {
                        xv[i] = __ldcg(reinterpret_cast<const float4*>(in + static_cast<int64_t>(b) * ldx + k));
                        if (gamma) gv[i] = __ldg(reinterpret_cast<const float4*>(gamma + k));
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int f = f0 + i * nct;
                if (f >= total) continue;   // warp-uniform: total and nct are multiples of 32
                const int q = q0 + f / per, r = f % per;
                const int b = r / kp4, e4 = r - b * kp4;
                float4 v = xv[i];
                if (gamma) {
                    const int hgk = q * nhg + (e4 >> 5);
                    const float ps = warp_sum(v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w);
                    if (lane == 0 && hgk < 2 * pl.G) ssq[b * 2 * pl.G + hgk] = ps;
                    v.x *= gv[i].x; v.y *= gv[i].y; v.z *= gv[i].z; v.w *= gv[i].w;
                }
                float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
                m = warp_max(m);
                int ex = 0;
                if (m > 0.f) ex = ((__float_as_int(m) >> 23) & 0xff) - 127 - 13;
                ex = max(-100, min(100, ex));
                const float sc = __int_as_float((127 - ex) << 23);
                const int hgi = e4 >> 5, ln = e4 & 31;
                const int j = ln >> 3, tile = (ln >> 2) & 1, tt = ln & 3;
                __half h0, l0, h1, l1, h2, l2, h3, l3;
                split_hi_lo(v.x * sc, h0, l0);
                split_hi_lo(v.y * sc, h1, l1);
                split_hi_lo(v.z * sc, h2, l2);
                split_hi_lo(v.w * sc, h3, l3);
                const __half2 hb0 = __halves2half2(h0, h2), hb1 = __halves2half2(h1, h3);
                const __half2 lb0 = __halves2half2(l0, l2), lb1 = __halves2half2(l1, l3);
                uint8_t* xf = xf0 + (q - q0) * xf_bytes;
                *reinterpret_cast<uint2*>(xf + xf_entry(hgi, j, tt, 2 * b, B) + tile * 8) =
                    make_uint2(*reinterpret_cast<const uint32_t*>(&hb0), *reinterpret_cast<const uint32_t*>(&hb1));
                *reinterpret_cast<uint2*>(xf + xf_entry(hgi, j, tt, 2 * b + 1, B) + tile * 8) =
                    make_uint2(*reinterpret_cast<const uint32_t*>(&lb0), *reinterpret_cast<const uint32_t*>(&lb1));
                if (lane == 0) xsc0[(q - q0) * nhg * B + hgi * B + b] = __int_as_float((127 + ex) << 23);
            }
        }
    };

    // residual rows of the epilogue, requested now (slots idx = tid, tid + nct)
    float rres[2] = {0.f, 0.f};
    const int nout = nup * kUnitRows * B;
    if (NMAT == 1 && residual) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int idx = tid + k * nct;
            if (idx < nout) {
                const int ur = idx / B, b = idx - ur * B;
                const int64_t n = static_cast<int64_t>(u0) * kUnitRows + ur;
                if (n < pl.N) rres[k] = __ldcg(residual + b * ldy + n);
            }
        }
    }

    for (int ph = 0; ph < pl.nphase; ++ph) {
        if (!resident || ph == 0) {
            consumer_sync();   // fragments and partial sums of the previous use are no longer read
            convert(ph, resident ? pl.nphase : 1);
            consumer_sync();
        }
        const int buf = resident ? ph : 0;
        const uint8_t* xf = xf0 + buf * xf_bytes;
        const float* xsc = xsc0 + buf * nhg * B;
        const int ng = min(pl.gps, pl.G - ph * pl.gps);
        const bool mine = jg < ng;
        uint4 xh[4];
        float sc0 = 0.f;
        if (mine) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                xh[j] = col_ok ? *reinterpret_cast<const uint4*>(xf + xf_entry(hg, j, t, g, B)) : make_uint4(0, 0, 0, 0);
            sc0 = t < B ? xsc[hg * B + t] : 0.f;
        }
        float* rr = red + (g * kNcw + warp) * B;
        for (int ul = 0; ul < nup; ++ul) {
            for (int m = 0; m < NMAT; ++m, rr += kUnitRows * kNcw * B) {
                const bool have = cx.wait_full();
                float acc0 = 0.f, acc1 = 0.f;
                if (mine && have) {
                    const uint8_t* rg = cx.smem + cx.ring.slot * kSlot + jg * kBoxBytes + g * kGroupBytes;
                    const uint8_t* rg8 = rg + 8 * kGroupBytes;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int jj = eta * 4 + j;
                        uint32_t wg, wg8;
                        if (j & 1) {
                            wg = code_word<1>(rg, jj, t);
                            wg8 = code_word<1>(rg8, jj, t);
                        } else {
                            wg = code_word<0>(rg, jj, t);
                            wg8 = code_word<0>(rg8, jj, t);
                        }
                        const float dg = half_bits_to_float(*reinterpret_cast<const uint16_t*>(rg + 18 * jj));
                        const float dg8 = half_bits_to_float(*reinterpret_cast<const uint16_t*>(rg8 + 18 * jj));
                        uint32_t a0, a2, a4, a6, a1, a3, a5, a7;
                        dequant_word(wg, a0, a2, a4, a6);
                        dequant_word(wg8, a1, a3, a5, a7);
                        float cf[4] = {0.f, 0.f, 0.f, 0.f};
                        mma_16816(cf, a0, a1, a2, a3, xh[j].x, xh[j].y);
                        mma_16816(cf, a4, a5, a6, a7, xh[j].z, xh[j].w);
                        acc0 = fmaf(dg, cf[0] + cf[1], acc0);
                        acc1 = fmaf(dg8, cf[2] + cf[3], acc1);
                    }
                }
                cx.release();
                if (mine && t < B) {
                    float* rr8 = rr + 8 * kNcw * B;
                    rr[t] = (ph ? rr[t] : 0.f) + sc0 * acc0;
                    rr8[t] = (ph ? rr8[t] : 0.f) + sc0 * acc1;
                }
            }
        }
        if (!resident) consumer_sync();   // partial sums of this phase written before the next conversion
    }
    consumer_sync();
    if (gamma && tid < B) {
        float sum = 0.f;
        for (int i = 0; i < 2 * pl.G; ++i) sum += ssq[tid * 2 * pl.G + i];
        rstd[tid] = rsqrtf(sum / static_cast<float>(pl.K) + eps);
    }
    if (gamma) consumer_sync();
    for (int k = 0, idx = tid; idx < nout; ++k, idx += nct) {
        const int ur = idx / B, b = idx - ur * B;
        const int ul = ur / kUnitRows, r16 = ur - ul * kUnitRows;
        const int64_t n = static_cast<int64_t>(u0 + ul) * kUnitRows + r16;
        if (n >= pl.N) continue;
        const int row = (ul * NMAT) * kUnitRows + r16;
        float v = 0.f;
        for (int w = 0; w < nw; ++w) v += red[(row * kNcw + w) * B + b];
        if (gamma) v *= rstd[b];
        if (NMAT == 1) {
            if (residual) v += k < 2 ? rres[k] : __ldcg(residual + b * ldy + n);
        } else {
            float uv = 0.f;
            for (int w = 0; w < nw; ++w) uv += red[((row + kUnitRows) * kNcw + w) * B + b];
            if (gamma) uv *= rstd[b];
            v = act_fn(v, act) * uv;
        }
        __stcg(out + b * ldy + n, v);
    }
}

// One attention phase: every item of this CTA (usually one).
template <int D>
__device__ __forceinline__ void attn_phase(Ctx& cx, const Layer& L) {
    constexpr int PS = 4096 / D;          // positions per stage
    constexpr int KB = kKVStage / 2;      // K bytes of a stage
    constexpr int kPbufPitch = 24;
    const Params& P = *cx.P;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nct = kNcw * 32;
    const int C = gridDim.x, c = blockIdx.x;
    const int G = L.n_q / L.n_kv;
    const int gq = lane >> 2, tq = lane & 3;
    // scratch: qs [4][D] | (unused) [D] | knew [D] | vnew [D] (u16) | pbuf [kNcw][8][24] half
    //          | cm [kNcw][4] | cl [kNcw][4] | co [kNcw][G][D] | flag
    float* qs = reinterpret_cast<float*>(cx.scr);
    const float* rtab = reinterpret_cast<const float*>(cx.smem + kRopeOff);
    uint16_t* knew = reinterpret_cast<uint16_t*>(qs + 5 * D);
    uint16_t* vnew = knew + D;
    __half* pbuf = reinterpret_cast<__half*>(vnew + D);
    float* cm = reinterpret_cast<float*>(pbuf + kNcw * 8 * kPbufPitch);
    float* cl = cm + kNcw * 4;
    float* co = cl + kNcw * 4;
    int* flag = reinterpret_cast<int*>(co + kNcw * G * D);
    const int nitems = P.B * L.n_kv * L.nsplit_max;

    for (int it = c; it < nitems; it += C) {
        int b, g, split, p, T, nsplit, s0, s1;
        if (!attn_item<D>(L, P.pos, it, b, g, split, p, T, nsplit, s0, s1)) {
            if (tid == 0 && split == 0) {
                const int pp = P.pos[b];
                if (pp < 0 || (L.window == 0 && static_cast<int64_t>(pp) >= L.cap))
                    atomicOr(P.status, GEM_DEVFLAG_POS_RANGE);
            }
            continue;
        }
        const int slot_p = L.window ? p % L.window : p;
        const bool owner = slot_p >= s0 * PS && slot_p < s1 * PS;
        const int64_t crow = (static_cast<int64_t>(b) * L.n_kv + g) * L.cap;
        const float* qrow = P.qkv + static_cast<int64_t>(b) * L.n_qkv;
        consumer_sync();   // scratch of the previous item is no longer read
        const int R = L.rope_dim, half = R / 2;
        const float* cs = rtab + b * 256;   // cos / sin at this sequence's position (rope_table)
        const float* sn = cs + 128;
        // warps 0..G-1: query heads; warp 4: the new K row; warp 5: the new V row
        const bool is_q = warp < G, is_k = owner && warp == 4, is_v = owner && warp == 5;
        if (is_q || is_k) {
            const float* src = qrow + (is_q ? (g * G + warp) : (L.n_q + g)) * D;
            const float* gm = is_q ? L.g_q : L.g_k;
            float v[D / 32];
            float ssum = 0.f;
#pragma unroll
            for (int k = 0; k < D / 32; ++k) {
                v[k] = __ldcg(src + lane + 32 * k);
                ssum = fmaf(v[k], v[k], ssum);
            }
            ssum = warp_sum(ssum);
            if (L.qk_norm) {
                const float r = rsqrtf(ssum / static_cast<float>(D) + L.eps);
#pragma unroll
                for (int k = 0; k < D / 32; ++k) v[k] = v[k] * r * __ldg(gm + lane + 32 * k);
            }
            float* sb = is_q ? qs + warp * D : qs + 3 * D;   // the K row borrows the last q row only when G < 4
            if (!is_q && G == 4) sb = co;                     // (co is free until the tiles are done)
#pragma unroll
            for (int k = 0; k < D / 32; ++k) sb[lane + 32 * k] = v[k];
            __syncwarp();
#pragma unroll
            for (int k = 0; k < D / 32; ++k) {
                const int e = lane + 32 * k;
                float r = sb[e];
                if (e < R) {
                    const int i = e < half ? e : e - half;
                    r = e < half ? fmaf(sb[e], cs[i], -sb[e + half] * sn[i]) : fmaf(sb[e - half], sn[i], sb[e] * cs[i]);
                }
                v[k] = r;
            }
            __syncwarp();
            if (is_q) {
#pragma unroll
                for (int k = 0; k < D / 32; ++k) sb[lane + 32 * k] = v[k] * L.scale;
            } else {
#pragma unroll
                for (int k = 0; k < D / 32; ++k) {
                    const uint16_t h = __half_as_ushort(__float2half_rn(v[k]));
                    knew[lane + 32 * k] = h;
                    L.k_cache[(crow + slot_p) * D + lane + 32 * k] = h;
                }
            }
        }
        if (is_v) {
            const float* src = qrow + (L.n_q + L.n_kv + g) * D;
#pragma unroll
            for (int k = 0; k < D / 32; ++k) {
                const uint16_t h = __half_as_ushort(__float2half_rn(__ldcg(src + lane + 32 * k)));
                vnew[lane + 32 * k] = h;
                L.v_cache[(crow + slot_p) * D + lane + 32 * k] = h;
            }
        }
        consumer_sync();
        // Q^T B fragments: column n = 2h + hl (head h = n / 2, hi or lo), k = dims
        uint32_t qb[D / 16][2];
        {
            const int h = gq >> 1, hl = gq & 1;
#pragma unroll
            for (int k16 = 0; k16 < D / 16; ++k16)
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    float2 q2 = make_float2(0.f, 0.f);
                    if (h < G) q2 = *reinterpret_cast<const float2*>(qs + h * D + k16 * 16 + 2 * tq + 8 * r);
                    __half h0, l0, h1, l1;
                    split_hi_lo(q2.x, h0, l0);
                    split_hi_lo(q2.y, h1, l1);
                    const __half2 hv = hl ? __halves2half2(l0, l1) : __halves2half2(h0, h1);
                    qb[k16][r] = *reinterpret_cast<const uint32_t*>(&hv);
                }
        }
        float o[D / 16][4];
#pragma unroll
        for (int m = 0; m < D / 16; ++m) o[m][0] = o[m][1] = o[m][2] = o[m][3] = 0.f;
        float m_run = -INFINITY, l_run = 0.f;
        int nmine = 0;
        const bool head_ok = tq < G;
        __half* pb = pbuf + warp * 8 * kPbufPitch;

        for (int k = 0; k < s1 - s0; ++k) {
            const bool have = cx.wait_full();
            if ((k % kNcw) == warp && have) {
                const int st = s0 + k;
                uint8_t* kt = cx.smem + cx.ring.slot * kSlot;
                uint8_t* vt = kt + KB;
                const int rp = slot_p - st * PS;
                if (rp >= 0 && rp < PS)   // the new row: the cache copy was requested before it was written
                    for (int e = lane * 8; e < D; e += 32 * 8) {
                        *reinterpret_cast<uint4*>(kt + swz(rp, e, PS)) = *reinterpret_cast<const uint4*>(knew + e);
                        *reinterpret_cast<uint4*>(vt + swz(rp, e, PS)) = *reinterpret_cast<const uint4*>(vnew + e);
                    }
                const int valid = T - st * PS;   // rows >= valid belong to other slots
                if (valid < PS)
                    for (int e = lane * 8; e < (PS - valid) * D; e += 32 * 8) {
                        const int r = valid + e / D, cc = e % D;
                        *reinterpret_cast<uint4*>(vt + swz(r, cc, PS)) = make_uint4(0, 0, 0, 0);
                    }
                __syncwarp();
                const uint32_t kb = smem_u32(kt), vb = smem_u32(vt);
                for (int u = 0; u < PS / 16; ++u) {
                    const int tv = valid - u * 16;    // valid rows of this 16-row tile
                    if (tv <= 0) break;
                    float cacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int k16 = 0; k16 < D / 16; ++k16) {
                        uint32_t a0, a1, a2, a3;
                        const int arow = u * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, acol = k16 * 16 + (lane >> 4) * 8;
                        ldmatrix_x4(a0, a1, a2, a3, kb + swz(arow, acol, PS));
                        mma_16816(cacc, a0, a1, a2, a3, qb[k16][0], qb[k16][1]);
                    }
                    float s0v = cacc[0] + cacc[1], s1v = cacc[2] + cacc[3];
                    if (gq >= tv) s0v = -INFINITY;
                    if (gq + 8 >= tv) s1v = -INFINITY;
                    if (!head_ok) s0v = s1v = 0.f;
                    float mx = fmaxf(s0v, s1v);
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                    const float m_new = fmaxf(m_run, mx);
                    const float corr = expf(m_run - m_new);
                    const float p0 = expf(s0v - m_new), p1 = expf(s1v - m_new);
                    float ps = p0 + p1;
                    ps += __shfl_xor_sync(0xffffffffu, ps, 4);
                    ps += __shfl_xor_sync(0xffffffffu, ps, 8);
                    ps += __shfl_xor_sync(0xffffffffu, ps, 16);
                    l_run = l_run * corr + ps;
                    m_run = m_new;
#pragma unroll
                    for (int m = 0; m < D / 16; ++m) {
                        o[m][0] *= corr; o[m][1] *= corr; o[m][2] *= corr; o[m][3] *= corr;
                    }
                    {
                        __half h0, l0, h1, l1;
                        split_hi_lo(p0, h0, l0);
                        split_hi_lo(p1, h1, l1);
                        pb[(2 * tq) * kPbufPitch + gq] = h0;
                        pb[(2 * tq + 1) * kPbufPitch + gq] = l0;
                        pb[(2 * tq) * kPbufPitch + gq + 8] = h1;
                        pb[(2 * tq + 1) * kPbufPitch + gq + 8] = l1;
                    }
                    __syncwarp();
                    uint32_t pb0, pb1;
                    ldmatrix_x2(pb0, pb1, smem_u32(pb + (lane & 7) * kPbufPitch + ((lane >> 3) & 1) * 8));
#pragma unroll
                    for (int m = 0; m < D / 16; ++m) {
                        uint32_t a0, a1, a2, a3;
                        const int vrow = u * 16 + (lane & 7) + (lane >> 4) * 8, vcol = m * 16 + ((lane >> 3) & 1) * 8;
                        ldmatrix_x4_trans(a0, a1, a2, a3, vb + swz(vrow, vcol, PS));
                        mma_16816(o[m], a0, a1, a2, a3, pb0, pb1);
                    }
                    __syncwarp();
                }
                ++nmine;
                fence_proxy_async_smem();   // generic writes above precede the next copy into this slot
            }
            cx.release();
        }
        // ---- combine the warps' states (ascending warp order) ----
        if (gq == 0 && head_ok) {
            cm[warp * 4 + tq] = nmine ? m_run : -INFINITY;
            cl[warp * 4 + tq] = nmine ? l_run : 0.f;
        }
        consumer_sync();   // co may still hold the rotated K row of the prologue (G == 4)
        if (head_ok) {
#pragma unroll
            for (int m = 0; m < D / 16; ++m) {
                co[(warp * G + tq) * D + m * 16 + gq] = o[m][0] + o[m][1];
                co[(warp * G + tq) * D + m * 16 + gq + 8] = o[m][2] + o[m][3];
            }
        }
        consumer_sync();
        for (int e = tid; e < G * D; e += nct) {
            const int h = e / D, i = e - h * D;
            float M = -INFINITY;
            for (int w = 0; w < kNcw; ++w) M = fmaxf(M, cm[w * 4 + h]);
            float Lsum = 0.f, O = 0.f;
            for (int w = 0; w < kNcw; ++w) {
                const float f = expf(cm[w * 4 + h] - M);
                Lsum += f * cl[w * 4 + h];
                O += f * co[(w * G + h) * D + i];
            }
            const int hq = g * G + h;
            if (nsplit == 1) {
                __stcg(P.attn + static_cast<int64_t>(b) * L.n_q * D + hq * D + i, O / Lsum);
            } else {
                float* dst = P.part + ((static_cast<int64_t>(b) * L.n_q + hq) * L.nsplit_max + split) * (D + 2);
                __stcg(dst + i, O);
                if (i == 0) {
                    __stcg(dst + D, M);
                    __stcg(dst + D + 1, Lsum);
                }
            }
        }
        if (nsplit > 1) {
            __threadfence();
            consumer_sync();
            if (tid == 0) {
                const unsigned prev = atomicAdd(&P.merge_cnt[b * L.n_kv + g], 1u);
                *flag = prev == static_cast<unsigned>(nsplit - 1);
            }
            consumer_sync();
            if (*flag) {   // the last split of (b, g) to finish: ordered merge of all splits
                __threadfence();
                // split maxima and denominators in one round of loads, then per-head weights
                float* wm = co;                          // [G][nsplit] maxima, then weights
                float* wl = co + G * L.nsplit_max;       // [G][nsplit] denominators
                const float* base0 = P.part + (static_cast<int64_t>(b) * L.n_q + g * G) * L.nsplit_max * (D + 2);
                for (int e = tid; e < G * nsplit; e += nct) {
                    const int h = e / nsplit, sp = e - h * nsplit;
                    const float* src = base0 + (static_cast<int64_t>(h) * L.nsplit_max + sp) * (D + 2);
                    wm[h * nsplit + sp] = __ldcg(src + D);
                    wl[h * nsplit + sp] = __ldcg(src + D + 1);
                }
                consumer_sync();
                if (tid < G) {
                    float M = -INFINITY;
                    for (int sp = 0; sp < nsplit; ++sp) M = fmaxf(M, wm[tid * nsplit + sp]);
                    float den = 0.f;
                    for (int sp = 0; sp < nsplit; ++sp) {
                        const float w = expf(wm[tid * nsplit + sp] - M);
                        wm[tid * nsplit + sp] = w;
                        den += w * wl[tid * nsplit + sp];
                    }
                    cl[tid] = den;
                }
                consumer_sync();
                for (int e = tid; e < G * D; e += nct) {
                    const int h = e / D, i = e - h * D;
                    const float* src = base0 + static_cast<int64_t>(h) * L.nsplit_max * (D + 2) + i;
                    float num = 0.f;
                    int sp = 0;
                    for (; sp + 8 <= nsplit; sp += 8) {   // eight independent loads per round
                        float a8[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) a8[u] = __ldcg(src + (sp + u) * (D + 2));
#pragma unroll
                        for (int u = 0; u < 8; ++u) num += wm[h * nsplit + sp + u] * a8[u];
                    }
                    for (; sp < nsplit; ++sp) num += wm[h * nsplit + sp] * __ldcg(src + sp * (D + 2));
                    __stcg(P.attn + static_cast<int64_t>(b) * L.n_q * D + (g * G + h) * D + i, num / cl[h]);
                }
                if (tid == 0) P.merge_cnt[b * L.n_kv + g] = 0u;
            }
        }
    }
}

// cos / sin of every rotated pair at each sequence's position for layer L, into the rope
// table (outside the scratch, so it is written before the barrier that precedes attention).
__device__ __forceinline__ void rope_table(Ctx& cx, const Layer& L) {
    float* rtab = reinterpret_cast<float*>(cx.smem + kRopeOff);
    const int half = L.rope_dim / 2;
    for (int e = threadIdx.x; e < cx.P->B * half; e += kNcw * 32) {
        const int b = e / half, i = e - b * half;
        const int p = cx.P->pos[b];
        float cc, ss;
        rope_cos_sin(static_cast<double>(max(p, 0)) * L.rope_w[i], cc, ss);
        rtab[b * 256 + i] = cc;
        rtab[b * 256 + 128 + i] = ss;
    }
}

template <int D>
__device__ __forceinline__ void consumer(const Params& P, uint8_t* smem, uint64_t* full, uint64_t* empty, uint8_t* scr,
                         volatile int* stop) {
    Ctx cx{&P, smem, full, empty, scr, stop, Ring{0, 0u}, true};
    for (int l = 0; l < P.nlayers; ++l) {
        const Layer& L = P.layers[l];
        const int H = L.H, nqd = L.n_q * L.d;
        if (l == 0 || L.rope_w != P.layers[l - 1].rope_w || L.rope_dim != P.layers[l - 1].rope_dim)
            rope_table(cx, L);   // read by attention after the barrier, which also orders it
        gemv_phase<1>(cx, L.qkv, P.x, H, L.g_attn, L.eps, P.qkv, L.n_qkv, nullptr, 0);
        if (!grid_sync(cx, l == 0)) break;
        attn_phase<D>(cx, L);
        if (!grid_sync(cx, false)) break;
        gemv_phase<1>(cx, L.o, P.attn, nqd, nullptr, 0.f, P.x, H, P.x, 0);
        if (!grid_sync(cx, false)) break;
        gemv_phase<2>(cx, L.gu, P.x, H, L.g_ffn, L.eps, P.act, L.F, nullptr, L.act);
        if (!grid_sync(cx, false)) break;
        gemv_phase<1>(cx, L.down, P.act, L.F, nullptr, 0.f, P.x, H, P.x, 0);
        if (l + 1 < P.nlayers && !grid_sync(cx, false)) break;
    }
    if (!cx.ok && threadIdx.x == 0) *stop = 1;   // the producer stops issuing and drains
}

template <int D>
__global__ void __maxnreg__(96) step_kernel(const Params P) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);
    uint64_t* empty = full + kNs;
    __shared__ int stop;
    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) {
        stop = 0;
        for (int i = 0; i < kNs; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kNcw);
        }
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == kNcw) {
        if ((tid & 31) == 0) producer<D>(P, smem, full, empty, &stop);
        return;
    }
    consumer<D>(P, smem, full, empty, smem + kScrOff, &stop);
}

}  // namespace step
}  // namespace gem

// ================================ host ==========================================================
struct gem_step_plan {
    int device, B, nlayers, d, num_sms;
    size_t smem;
    gem::step::Layer* d_layers;
    double* d_rope;
    float *qkv, *attn, *act, *part;
    unsigned* merge_cnt;
    gem::step::Sync* sync;
};

namespace {

using namespace gem;
using namespace gem::step;

gem_status plan_gemv(GemvPlan& pl, int64_t N, int64_t K, int nmat, int B, int C) {
    if (K % 256 || N <= 0) return GEM_ERR_UNSUPPORTED_SHAPE;
    pl.N = static_cast<int>(N);
    pl.K = static_cast<int>(K);
    pl.G = static_cast<int>(K / 256);
    pl.nphase = (pl.G + 7) / 8;
    pl.gps = (pl.G + pl.nphase - 1) / pl.nphase;
    pl.U = static_cast<int>((N + kUnitRows - 1) / kUnitRows);
    const int nu = (pl.U + C - 1) / C;
    const size_t kp = static_cast<size_t>(pl.gps) * 256;
    auto need = [&](int nbuf) {
        return aup(nbuf * 4 * B * kp, 128) + 4 * (aup(nbuf * 2 * pl.gps * B, 32) + aup(B * 2 * pl.G, 32) +
                                                  static_cast<size_t>(nmat) * nu * kUnitRows * kNcw * B + B);
    };
    pl.resident = need(pl.nphase) <= static_cast<size_t>(kScratch) ? 1 : 0;
    return need(pl.resident ? pl.nphase : 1) <= static_cast<size_t>(kScratch) ? GEM_OK : GEM_ERR_UNSUPPORTED_SHAPE;
}

const void* step_fn(int d) {
    switch (d) {
        case 64: return reinterpret_cast<const void*>(step_kernel<64>);
        case 128: return reinterpret_cast<const void*>(step_kernel<128>);
        default: return reinterpret_cast<const void*>(step_kernel<256>);
    }
}

void free_plan(gem_step_plan* p) {
    if (!p) return;
    cudaFree(p->d_layers);
    cudaFree(p->d_rope);
    cudaFree(p->qkv);
    cudaFree(p->attn);
    cudaFree(p->act);
    cudaFree(p->part);
    cudaFree(p->merge_cnt);
    cudaFree(p->sync);
    delete p;
}

}  // namespace

extern "C" {

gem_status gem_step_plan_create(const gem_layer_desc* layers, int nlayers, int B, uint16_t* const* k_caches,
                                uint16_t* const* v_caches, const int64_t* cache_caps, gem_step_plan** out) {
    if (!out) return GEM_ERR_INVALID_ARG;
    *out = nullptr;
    if (!layers || nlayers <= 0 || !k_caches || !v_caches || !cache_caps) return GEM_ERR_INVALID_ARG;
    if (B < 1 || B > kMaxB) return GEM_ERR_UNSUPPORTED_SHAPE;
    DeviceInfo di;
    gem_status st = device_info(&di);
    if (st != GEM_OK) return st;
    const int C = di.num_sms;
    const int d = static_cast<int>(layers[0].d);
    if (d != 64 && d != 128 && d != 256) return GEM_ERR_UNSUPPORTED_SHAPE;
    std::vector<Layer> hl(nlayers);
    std::vector<double> rope;
    std::vector<size_t> rope_off(nlayers);
    size_t qkv_max = 0, attn_max = 0, act_max = 0, part_max = 0, cnt_max = 0;
    for (int l = 0; l < nlayers; ++l) {
        const gem_layer_desc& L = layers[l];
        Layer& D = hl[l];
        std::memset(&D, 0, sizeof(D));
        if (L.d != d || L.n_kv <= 0 || L.n_q % L.n_kv || L.n_q / L.n_kv > 4 || L.post_norms || L.v_from_k)
            return GEM_ERR_UNSUPPORTED_SHAPE;
        if (L.rope_dim < 2 || L.rope_dim > d || (L.rope_dim & 1) || L.window < 0 || L.window > cache_caps[l] ||
            cache_caps[l] <= 0 || !(L.theta > 0.f) || L.act < 0 || L.act > 1)
            return GEM_ERR_INVALID_ARG;
        if (L.qk_norm && (!L.g_q || !L.g_k)) return GEM_ERR_INVALID_ARG;
        if (!L.w_qkv || !L.w_o || !L.w_gate || !L.w_up || !L.w_down || !L.g_attn || !L.g_ffn || !k_caches[l] ||
            !v_caches[l])
            return GEM_ERR_INVALID_ARG;
        const uintptr_t al = reinterpret_cast<uintptr_t>(L.w_qkv) | reinterpret_cast<uintptr_t>(L.w_o) |
                             reinterpret_cast<uintptr_t>(L.w_gate) | reinterpret_cast<uintptr_t>(L.w_up) |
                             reinterpret_cast<uintptr_t>(L.w_down) | reinterpret_cast<uintptr_t>(L.g_attn) |
                             reinterpret_cast<uintptr_t>(L.g_ffn) | reinterpret_cast<uintptr_t>(k_caches[l]) |
                             reinterpret_cast<uintptr_t>(v_caches[l]);
        if (al & 15) return GEM_ERR_MISALIGNED;
        const int G = static_cast<int>(L.n_q / L.n_kv);
        if (static_cast<size_t>(kNcw) * G * d * 4 + 4 * d * 4 + 4 * d + kNcw * 8 * 24 * 2 + kNcw * 8 * 4 + 64 >
            static_cast<size_t>(kScratch))
            return GEM_ERR_UNSUPPORTED_SHAPE;
        if (static_cast<uint64_t>(B) * L.n_kv * cache_caps[l] >= (1ull << 31)) return GEM_ERR_UNSUPPORTED_SHAPE;
        D.H = static_cast<int>(L.H);
        D.n_q = static_cast<int>(L.n_q);
        D.n_kv = static_cast<int>(L.n_kv);
        D.d = d;
        D.F = static_cast<int>(L.F);
        D.n_qkv = static_cast<int>((L.n_q + 2 * L.n_kv) * d);
        D.rope_dim = L.rope_dim;
        D.window = L.window;
        D.act = L.act;
        D.qk_norm = L.qk_norm;
        D.eps = L.eps;
        D.scale = L.scale;
        D.cap = cache_caps[l];
        D.g_attn = L.g_attn;
        D.g_ffn = L.g_ffn;
        D.g_q = L.g_q;
        D.g_k = L.g_k;
        D.k_cache = k_caches[l];
        D.v_cache = v_caches[l];
        if ((st = plan_gemv(D.qkv, D.n_qkv, L.H, 1, B, C)) != GEM_OK ||
            (st = plan_gemv(D.o, L.H, L.n_q * d, 1, B, C)) != GEM_OK ||
            (st = plan_gemv(D.gu, L.F, L.H, 2, B, C)) != GEM_OK ||
            (st = plan_gemv(D.down, L.H, L.F, 1, B, C)) != GEM_OK)
            return st;
        const int PS = 4096 / d;
        const int64_t tmax = L.window ? std::min<int64_t>(L.window, cache_caps[l]) : cache_caps[l];
        const int64_t nst_max = (tmax + PS - 1) / PS;
        int64_t ns = std::max<int64_t>(1, (C + static_cast<int64_t>(B) * L.n_kv - 1) / (static_cast<int64_t>(B) * L.n_kv));
        D.nsplit_max = static_cast<int>(std::min(ns, nst_max));
        auto mk = [&](CUtensorMap* tm, const void* w, int64_t N, int64_t K) {
            const int64_t rb = K / 32 * 18;
            return make_tensor_map_2d(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, static_cast<uint64_t>(rb),
                                      static_cast<uint64_t>(N), static_cast<uint64_t>(rb), kGroupBytes, kUnitRows,
                                      CU_TENSOR_MAP_SWIZZLE_NONE);
        };
        if ((st = mk(&D.tm_qkv, L.w_qkv, D.n_qkv, L.H)) != GEM_OK || (st = mk(&D.tm_o, L.w_o, L.H, L.n_q * d)) != GEM_OK ||
            (st = mk(&D.tm_gate, L.w_gate, L.F, L.H)) != GEM_OK || (st = mk(&D.tm_up, L.w_up, L.F, L.H)) != GEM_OK ||
            (st = mk(&D.tm_down, L.w_down, L.H, L.F)) != GEM_OK)
            return st;
        const uint64_t rows = static_cast<uint64_t>(B) * L.n_kv * cache_caps[l];
        if ((st = make_tensor_map_2d(&D.tm_k, CU_TENSOR_MAP_DATA_TYPE_UINT16, k_caches[l], d, rows,
                                     static_cast<uint64_t>(d) * 2, 64, PS, CU_TENSOR_MAP_SWIZZLE_128B)) != GEM_OK ||
            (st = make_tensor_map_2d(&D.tm_v, CU_TENSOR_MAP_DATA_TYPE_UINT16, v_caches[l], d, rows,
                                     static_cast<uint64_t>(d) * 2, 64, PS, CU_TENSOR_MAP_SWIZZLE_128B)) != GEM_OK)
            return st;
        if (l > 0 && L.theta == layers[l - 1].theta && L.rope_dim == layers[l - 1].rope_dim) {
            rope_off[l] = rope_off[l - 1];   // same table: the kernel keeps it across layers
        } else {
            rope_off[l] = rope.size();
            for (int i = 0; i < L.rope_dim / 2; ++i)
                rope.push_back(std::pow(static_cast<double>(L.theta), -2.0 * i / L.rope_dim));
        }
        qkv_max = std::max<size_t>(qkv_max, static_cast<size_t>(B) * D.n_qkv);
        attn_max = std::max<size_t>(attn_max, static_cast<size_t>(B) * L.n_q * d);
        act_max = std::max<size_t>(act_max, static_cast<size_t>(B) * L.F);
        part_max = std::max<size_t>(part_max, static_cast<size_t>(B) * L.n_q * D.nsplit_max * (d + 2));
        cnt_max = std::max<size_t>(cnt_max, static_cast<size_t>(B) * L.n_kv);
    }
    const void* fn = step_fn(d);
    if (kSmemBytes > di.smem_optin) return GEM_ERR_UNSUPPORTED_SHAPE;
    GEM_CUDA_TRY(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemBytes)));
    int occ = 0;
    GEM_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, kThreads, kSmemBytes));
    if (occ < 1) return GEM_ERR_UNSUPPORTED_SHAPE;

    gem_step_plan* p = new gem_step_plan{};
    p->device = di.device;
    p->B = B;
    p->nlayers = nlayers;
    p->d = d;
    p->num_sms = C;
    p->smem = kSmemBytes;
    auto fail = [&](cudaError_t e) {
        free_plan(p);
        return cuda_fail(e);
    };
    cudaError_t e;
    if ((e = cudaMalloc(&p->d_rope, std::max<size_t>(1, rope.size()) * sizeof(double))) != cudaSuccess) return fail(e);
    for (int l = 0; l < nlayers; ++l) hl[l].rope_w = p->d_rope + rope_off[l];
    if ((e = cudaMalloc(&p->d_layers, sizeof(Layer) * nlayers)) != cudaSuccess) return fail(e);
    if ((e = cudaMalloc(&p->qkv, qkv_max * 4)) != cudaSuccess || (e = cudaMalloc(&p->attn, attn_max * 4)) != cudaSuccess ||
        (e = cudaMalloc(&p->act, act_max * 4)) != cudaSuccess || (e = cudaMalloc(&p->part, std::max<size_t>(1, part_max) * 4)) != cudaSuccess ||
        (e = cudaMalloc(&p->merge_cnt, cnt_max * 4)) != cudaSuccess || (e = cudaMalloc(&p->sync, sizeof(Sync))) != cudaSuccess)
        return fail(e);
    if ((e = cudaMemcpy(p->d_rope, rope.data(), rope.size() * sizeof(double), cudaMemcpyHostToDevice)) != cudaSuccess ||
        (e = cudaMemcpy(p->d_layers, hl.data(), sizeof(Layer) * nlayers, cudaMemcpyHostToDevice)) != cudaSuccess ||
        (e = cudaMemset(p->merge_cnt, 0, cnt_max * 4)) != cudaSuccess || (e = cudaMemset(p->sync, 0, sizeof(Sync))) != cudaSuccess ||
        (e = cudaDeviceSynchronize()) != cudaSuccess)
        return fail(e);
    *out = p;
    return GEM_OK;
}

gem_status gem_decode_step(const gem_step_plan* plan, float* x, const int32_t* pos, int32_t* status, void* stream) {
    if (!plan || !x || !pos) return GEM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x) & 15)) return GEM_ERR_MISALIGNED;
    int dev = 0;
    GEM_CUDA_TRY(cudaGetDevice(&dev));
    if (dev != plan->device) return GEM_ERR_INVALID_ARG;
    DeviceInfo di;
    gem_status st = device_info(&di);
    if (st != GEM_OK) return st;
    Params P{};
    P.layers = plan->d_layers;
    P.nlayers = plan->nlayers;
    P.B = plan->B;
    P.x = x;
    P.pos = pos;
    P.qkv = plan->qkv;
    P.attn = plan->attn;
    P.act = plan->act;
    P.part = plan->part;
    P.merge_cnt = plan->merge_cnt;
    P.sync = plan->sync;
    P.status = status ? status : di.status_word;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(plan->num_sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = plan->smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {&P};
    GEM_CUDA_TRY(cudaLaunchKernelExC(&cfg, step_fn(plan->d), args));
    return GEM_OK;
}

void gem_step_plan_destroy(gem_step_plan* plan) { free_plan(plan); }

}  // extern "C"
