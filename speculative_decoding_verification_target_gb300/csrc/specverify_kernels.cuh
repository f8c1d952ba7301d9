// Verification kernels for sm_103a.
//
// rows_kernel: one persistent grid of thread-block clusters. A cluster of C CTAs works through a list of
// "items": a target row (b, j) together with the rows verified against it (the draft row for standard and
// Cactus verification, the N drafter rows for the counterfactual evaluation, none for the bonus row
// j = K). CTA `rank` owns the vocabulary slice [rank * slice, (rank + 1) * slice) of every row; the slice
// is cut into pieces of PE logits. Inside a CTA:
//   - W consumer warps take the pieces round robin. Each warp streams its own pieces through a private
//     ring of R shared-memory slots: it issues the bulk (TMA) copy of a piece R pieces ahead, waits on the
//     slot's mbarrier, copies the piece into registers and refills the slot at once. No warp waits for
//     another warp's data, and there is no CTA-wide barrier on the hot path;
//   - a reducer warp merges the consumer warps' softmax partials of a row, exchanges them with the other
//     CTAs of the cluster through distributed shared memory (remote stores + remote mbarrier arrivals)
//     and publishes the row scalars (log-normaliser, p(t), the Cactus constants);
//   - a loader warp (resident mode, below) brings each item's target slice into shared memory.
// Every row is processed in two passes. Pass 1 computes the partial (max, sum of exponentials) of each
// piece straight from HBM. Pass 2, which needs the row's final normaliser, re-reads the same piece one
// unit of work later, while it is still in L2 (this GPU re-reads L2 at about three times the HBM rate),
// and evaluates for the piece:
//   - sum_x min(p_target, p_other)              (HedgeSpec gamma partials; gamma = 1 - TV)
//   - the residual mass (h - p_draft)+ of the piece, h = p_target or the Cactus h (verified row)
//   - or the mass of p_target (bonus row)
// The cluster exchange of a unit's normaliser thus runs behind the next unit's pass 1. When an item has
// two or more drafters the target slice instead stays resident in shared memory for the whole item
// (double buffered across items), so the target is read from HBM once and from shared memory by every
// drafter.
// finish_kernel: one warp per sequence turns the per-position records into the accept/reject chain and
// draws the residual (or bonus) token by inverse CDF: a prefix scan over the piece masses of the chosen
// row, then one re-read of that piece. gamma_reduce_kernel sums the gamma partials.
//
// Sources for the arithmetic (web pages, by title and section):
//   "Speculative Decoding 为什么是 Lossless 的 — 详细证明教程": §5.1 (accept r * q(t) < p(t), residual
//   (p - q)+ / Z), §6.3-§6.4 (P(accept) = sum min(p, q), Z = 1 - sum min(p, q)), §8 Q4 (one temperature
//   for both rows), §9.1 (gamma-step chain, K+1 target rows).
//   "Not-a-Bandit: Provably No-Regret Drafter Selection in Speculative Decoding for LLMs", Key design 1
//   (gamma_{j,i} = 1 - TV(p, q_i) for every drafter from one verified trajectory), Key design 3 (loss
//   1 - gamma).
//   "Cactus: Accelerating Auto-Regressive Decoding with Constrained Acceptance Speculative Sampling",
//   Key design 2 (h_n = gamma*, h_i = (1 - gamma*) / (1 - q(n)) q(i)) and 3 (gamma* closed form); that
//   page names the target q and the draft p.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "device_common.cuh"

namespace specv {

constexpr int W = 14;                   // consumer warps per CTA (16 warps in all: 128 registers a thread)
constexpr int NT = (W + 2) * 32;        // plus the reducer (warp W) and the target loader (warp W + 1)
constexpr int CHUNK = 8;                // logits per lane per load (16 B of bf16)
constexpr int PE = 2048;                // logits per piece: one bulk copy, a consumer warp's unit of work, one residual tile
constexpr int PCH = PE / CHUNK / 32;    // chunks per lane per piece
constexpr int MAX_R = 8;                // ring slots per consumer warp
constexpr int SLICE_Q = 128;            // granularity of the per-CTA vocabulary slice
constexpr int REC = 8;                  // 32-bit words per position record
constexpr int MAX_LEAD = 1;             // pass 2 of unit u - 1 runs after pass 1 of unit u. The resident
                                        // target is double buffered, and two one-unit (bonus) items in a row
                                        // need its buffer back within one unit.
constexpr int NXB = 4;                  // exchange buffers in flight
static_assert(NXB > MAX_LEAD + 1, "exchange buffers must outlive the pass-2 lead");
constexpr int XW = 8;                   // floats per exchange entry
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;   // bounded waits: 2 s
constexpr unsigned STATUS_BAD_TOKEN = 1u;
constexpr unsigned STATUS_TIMEOUT = 2u;

// record words (per target row b, j)
constexpr int R_HT = 0;      // h(t): p_target(t), or gamma* for Cactus
constexpr int R_PD = 1;      // p_draft(t) of the verified drafter
constexpr int R_BT = 2;      // log2 h(x) = x c + R_BT away from t (Cactus-scaled)
constexpr int R_BO = 3;      // log2 p_draft(x) = x c + R_BO
constexpr int R_BTP = 4;     // log2 p_target(x) = x c + R_BTP (plain)

struct KParams {
    const unsigned char* target;   // [B, K+1, V]
    const unsigned char* others;   // [N, B, K, V]
    const int32_t* tokens;         // [B, K] (null: gamma only)
    const uint64_t* seeds;         // [B] (with tokens)
    int all_residuals;             // 1: residual masses for every position (diag wants Z everywhere)
    int B, K, V, N;
    int selected;                  // drafter whose chain is verified (processed last); -1: none
    int BK;                        // B * K: items below BK are (b, j < K), the rest are bonus rows
    int num_items;                 // B * K, plus B bonus rows when a chain is verified
    float c;                       // log2(e) / temperature
    float delta;                   // Cactus divergence budget
    int cactus;
    int slice_elems;               // per-CTA slice, multiple of SLICE_Q
    int pcap;                      // pieces per full slice (ceil(slice_elems / PE))
    int tma;                       // 1: every piece is 16-byte aligned -> bulk copies
    int resident;                  // 1: the target slice stays in shared memory for the whole item
    int R;                         // ring slots per consumer warp
    int lead;                      // pass 2 of unit u - lead follows pass 1 of unit u (1 .. MAX_LEAD)
    float* rec;                    // [B, K+1, REC] or null
    float* tiles;                  // [B, K+1, C, pcap] or null
    float* gpart;                  // [N, B, K, C, W] or null
    unsigned* status;
};

// ------------------------------------------------------------------------------------------------
// element formats: a chunk is 8 consecutive logits of one row (16 B of bf16 or 32 B of fp32)
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

struct Bf16 {
    using Raw = uint4;
    using Max = uint32_t;            // running max as a packed bf16 pair
    static constexpr int BYTES = 2;
    __device__ static Raw ninf() { return make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u); }
    __device__ static Raw lds(const unsigned char* slot, int k) { return reinterpret_cast<const uint4*>(slot)[k]; }
    // elements 2w and 2w+1 of the chunk
    __device__ static float2 pair(const Raw& r, int w) {
        const uint32_t v = w == 0 ? r.x : (w == 1 ? r.y : (w == 2 ? r.z : r.w));
        return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
    }
    __device__ static Max max_init() { return 0xFF80FF80u; }
    __device__ static Max max_acc(Max m, const Raw& r) {
        return bf16x2_max(bf16x2_max(m, r.x), bf16x2_max(bf16x2_max(r.y, r.z), r.w));
    }
    __device__ static float max_fin(Max m) { return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u)); }
    __device__ static float at(const unsigned char* slot, int e) {
        return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(slot)[e]) << 16);
    }
    // element-wise staging for rows that are not 16-byte aligned (pads the last chunk with -inf)
    __device__ static void copy_slice(unsigned char* slot, const unsigned char* src, int n_el, int lane) {
        const uint16_t* s = reinterpret_cast<const uint16_t*>(src);
        uint16_t* d = reinterpret_cast<uint16_t*>(slot);
        const int padded = (n_el + CHUNK - 1) / CHUNK * CHUNK;
        for (int e = lane; e < padded; e += 32) d[e] = e < n_el ? __ldg(s + e) : static_cast<uint16_t>(0xFF80u);
    }
    // the same, by one thread
    __device__ static void copy_slice_thread(unsigned char* slot, const unsigned char* src, int n_el) {
        const uint16_t* s = reinterpret_cast<const uint16_t*>(src);
        uint16_t* d = reinterpret_cast<uint16_t*>(slot);
        const int padded = (n_el + CHUNK - 1) / CHUNK * CHUNK;
        for (int e = 0; e < padded; ++e) d[e] = e < n_el ? __ldg(s + e) : static_cast<uint16_t>(0xFF80u);
    }
    // One chunk of a row in global memory, -inf from element n_el on. AL: the row is 16-byte aligned and n_el
    // a multiple of CHUNK, so a chunk is in range whole or not at all: one predicated 16-byte load into
    // registers preset to -inf, with no branch and no register merge after it, so that all the loads of a
    // piece stay in flight together. Otherwise element by element (rows of any alignment).
    template <bool AL>
    __device__ static Raw gload(const unsigned char* row, int e0, int n_el) {
        if constexpr (AL) {
            uint4 v = ninf();
            const uint4* ptr = reinterpret_cast<const uint4*>(row) + e0 / CHUNK;
            asm volatile(
                "{\n\t.reg .pred q;\n\tsetp.lt.s32 q, %4, %5;\n\t"
                "@q ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%6];\n\t}"
                : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)
                : "r"(e0), "r"(n_el), "l"(ptr));
            return v;
        } else {
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int e = e0 + 2 * q;
                const uint32_t lo = e < n_el ? __ldg(reinterpret_cast<const uint16_t*>(row) + e) : 0xFF80u;
                const uint32_t hi = e + 1 < n_el ? __ldg(reinterpret_cast<const uint16_t*>(row) + e + 1) : 0xFF80u;
                w[q] = lo | (hi << 16);
            }
            return make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
};

struct F32 {
    struct Raw {
        float4 a, b;
    };
    using Max = float;
    static constexpr int BYTES = 4;
    __device__ static Raw ninf() {
        const float n = __uint_as_float(0xFF800000u);
        return {make_float4(n, n, n, n), make_float4(n, n, n, n)};
    }
    __device__ static Raw lds(const unsigned char* slot, int k) {
        const float4* p = reinterpret_cast<const float4*>(slot) + 2 * k;
        return {p[0], p[1]};
    }
    __device__ static float2 pair(const Raw& r, int w) {
        return w == 0 ? make_float2(r.a.x, r.a.y)
                      : (w == 1 ? make_float2(r.a.z, r.a.w) : (w == 2 ? make_float2(r.b.x, r.b.y) : make_float2(r.b.z, r.b.w)));
    }
    __device__ static Max max_init() { return __uint_as_float(0xFF800000u); }
    __device__ static Max max_acc(Max m, const Raw& r) {
        return fmaxf(fmaxf(fmaxf(m, fmaxf(r.a.x, r.a.y)), fmaxf(r.a.z, r.a.w)),
                     fmaxf(fmaxf(r.b.x, r.b.y), fmaxf(r.b.z, r.b.w)));
    }
    __device__ static float max_fin(Max m) { return m; }
    __device__ static float at(const unsigned char* slot, int e) { return reinterpret_cast<const float*>(slot)[e]; }
    __device__ static void copy_slice(unsigned char* slot, const unsigned char* src, int n_el, int lane) {
        const uint32_t* s = reinterpret_cast<const uint32_t*>(src);
        uint32_t* d = reinterpret_cast<uint32_t*>(slot);
        const int padded = (n_el + CHUNK - 1) / CHUNK * CHUNK;
        for (int e = lane; e < padded; e += 32) d[e] = e < n_el ? __ldg(s + e) : 0xFF800000u;
    }
    __device__ static void copy_slice_thread(unsigned char* slot, const unsigned char* src, int n_el) {
        const uint32_t* s = reinterpret_cast<const uint32_t*>(src);
        uint32_t* d = reinterpret_cast<uint32_t*>(slot);
        const int padded = (n_el + CHUNK - 1) / CHUNK * CHUNK;
        for (int e = 0; e < padded; ++e) d[e] = e < n_el ? __ldg(s + e) : 0xFF800000u;
    }
    template <bool AL>
    __device__ static Raw gload(const unsigned char* row, int e0, int n_el) {
        const float* f = reinterpret_cast<const float*>(row);
        if constexpr (AL) {
            Raw v = ninf();
            const float* ptr = f + e0;
            asm volatile(
                "{\n\t.reg .pred q;\n\tsetp.lt.s32 q, %8, %9;\n\t"
                "@q ld.global.cs.v4.f32 {%0, %1, %2, %3}, [%10];\n\t"
                "@q ld.global.cs.v4.f32 {%4, %5, %6, %7}, [%10+16];\n\t}"
                : "+f"(v.a.x), "+f"(v.a.y), "+f"(v.a.z), "+f"(v.a.w), "+f"(v.b.x), "+f"(v.b.y), "+f"(v.b.z),
                  "+f"(v.b.w)
                : "r"(e0), "r"(n_el), "l"(ptr));
            return v;
        } else {
            float v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] = e0 + q < n_el ? __ldg(f + e0 + q) : __uint_as_float(0xFF800000u);
            return {make_float4(v[0], v[1], v[2], v[3]), make_float4(v[4], v[5], v[6], v[7])};
        }
    }
};

__device__ __forceinline__ float2 ex2x2(float2 t) { return make_float2(ex2(t.x), ex2(t.y)); }

// ------------------------------------------------------------------------------------------------
// per-thread building blocks
// ------------------------------------------------------------------------------------------------
// Overlap only: adds 2^min(log2 h, log2 p_other) of the chunk's 8 elements to acc.
template <class E>
__device__ __forceinline__ float2 chunk_overlap(const typename E::Raw& rt, const typename E::Raw& ro, float2 cc,
                                                float2 bt, float2 bo, float2 acc) {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const float2 a = __ffma2_rn(E::pair(rt, w), cc, bt);
        const float2 d = __ffma2_rn(E::pair(ro, w), cc, bo);
        acc = __fadd2_rn(acc, ex2x2(make_float2(fminf(a.x, d.x), fminf(a.y, d.y))));
    }
    return acc;
}

// Per-element masses of one chunk. mode 1: residual (h - p_other)+ (overlap min(h, p_other) added to
// ovl); mode 2: h itself. h(x) = 2^(x c + bt) except element `et` (>= 0), which is `hpatch`. Each element
// goes through the same operations as in chunk_mass, so the values agree bit for bit.
template <class E>
__device__ __forceinline__ void chunk_values(int mode, const typename E::Raw& rt, const typename E::Raw& ro, float c,
                                             float bt, float bo, int et, float hpatch, float (&v)[8], float& ovl) {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const float2 xt = E::pair(rt, w);
        const float2 xo = E::pair(ro, w);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int e = 2 * w + h;
            float ph = ex2(fmaf(h ? xt.y : xt.x, c, bt));
            if (e == et) ph = hpatch;
            if (mode == 1) {
                const float po = ex2(fmaf(h ? xo.y : xo.x, c, bo));
                const float mn = fminf(ph, po);
                ovl += mn;
                v[e] = ph - mn;
            } else {
                v[e] = ph;
            }
        }
    }
}

// Chunk mass (sum of the residual, mode 1, or of h, mode 2) with the overlap added to ovl2.
template <class E>
__device__ __forceinline__ float chunk_mass(int mode, const typename E::Raw& rt, const typename E::Raw& ro, float2 cc,
                                            float2 bt, float2 bo, float2& ovl2) {
    float2 m2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const float2 ph = ex2x2(__ffma2_rn(E::pair(rt, w), cc, bt));
        if (mode == 1) {
            const float2 po = ex2x2(__ffma2_rn(E::pair(ro, w), cc, bo));
            const float2 mn = make_float2(fminf(ph.x, po.x), fminf(ph.y, po.y));
            ovl2 = __fadd2_rn(ovl2, mn);
            m2 = __fadd2_rn(m2, __ffma2_rn(mn, make_float2(-1.f, -1.f), ph));   // ph - mn, one rounding
        } else {
            m2 = __fadd2_rn(m2, ph);
        }
    }
    return m2.x + m2.y;
}

// Chunk mass with the optional patch at element et: the single definition used by the row pass and by
// the draw, so both see the same numbers.
template <class E>
__device__ __forceinline__ float chunk_mass_patched(int mode, const typename E::Raw& rt, const typename E::Raw& ro,
                                                    float c, float bt, float bo, int et, float hpatch, float2& ovl2) {
    if (et < 0)
        return chunk_mass<E>(mode, rt, ro, make_float2(c, c), make_float2(bt, bt), make_float2(bo, bo), ovl2);
    float v[8], ovl = 0.f;
    chunk_values<E>(mode, rt, ro, c, bt, bo, et, hpatch, v, ovl);
    ovl2.x += ovl;
    const float2 a = make_float2(v[0] + v[2] + v[4] + v[6], v[1] + v[3] + v[5] + v[7]);
    return a.x + a.y;
}
// (chunk_mass_patch_only below computes the patched case with exactly these operations)

// The patched chunk (the one holding the draft token) as a separate, non-inlined routine: only one thread
// of one CTA per row takes this branch, and keeping it out of line stops the compiler from evaluating it
// alongside the fast path in every thread.
template <class E>
__device__ __noinline__ float chunk_mass_patch_only(int mode, typename E::Raw rt, typename E::Raw ro, float c, float bt,
                                                    float bo, int et, float hpatch, float& ovl) {
    float v[8];
    chunk_values<E>(mode, rt, ro, c, bt, bo, et, hpatch, v, ovl);
    const float2 a = make_float2(v[0] + v[2] + v[4] + v[6], v[1] + v[3] + v[5] + v[7]);
    return a.x + a.y;
}

// Inclusive scan across the warp (Hillis-Steele, fixed association order).
__device__ __forceinline__ float warp_incl_scan(float v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
    }
    return v;
}

// log2 p(x) = x c + beta with beta = -(M c + log2 S).
__device__ __forceinline__ float beta_of(MaxSum g, float c) { return -fmaf(g.m, c, lg2(g.s)); }

// p(x) for one logit with the row's global (M, S): 2^((x - M) c - log2 S).
__device__ __forceinline__ float prob_of(float x, MaxSum g, float c) {
    if (!(x > __uint_as_float(0xFF800000u)) || !(g.s > 0.f)) return 0.f;
    return ex2(fmaf(x - g.m, c, -lg2(g.s)));
}

// Cactus closed form on q = p_target(t): gamma* = min(q + sqrt(2 delta q (1 - q)), 1) and the log2 of the
// scale (1 - gamma*) / (1 - q) applied to every other token (-inf when q = 1).
__device__ __forceinline__ void cactus_scalars(float q, float delta, float& gstar, float& log2s) {
    float gs = q + sqrtf(2.f * delta * q * (1.f - q));
    gs = fminf(gs, 1.f);
    const float s = q < 1.f ? __fdiv_rn(1.f - gs, 1.f - q) : 0.f;
    gstar = gs;
    log2s = log2f(s);
}


__device__ __forceinline__ int drafter_at(int i, int N, int selected) {
    if (selected < 0) return i;
    return i == N - 1 ? selected : (i < selected ? i : i + 1);
}

// ------------------------------------------------------------------------------------------------
// the work list of a cluster
// ------------------------------------------------------------------------------------------------
// Items are numbered with the B * K verified positions first (item w = b * K + j) and the B bonus rows
// last (item B * K + b), and cluster `cid` takes items cid, cid + ncl, cid + 2 ncl, ... Every cluster
// thus gets the same number of positions up to one, and the bonus rows (one row each instead of 1 + N)
// land first on the clusters that got one position fewer.
// A unit is one row verified against the item's target (other index i in processing order, the verified
// drafter last), or, for a bonus row, the target alone.
struct Unit {
    int k;         // item index in the cluster's list
    int b, j, n;   // sequence, position, other rows of the item (0: bonus row)
    int i;         // other row index in processing order
    int d;         // drafter index of row i (-1 for a bonus row)
    int tok;       // draft token of the position (-1: none)
};

// Draft tokens of the cluster's items, 32 items per warp-wide load, the next block prefetched while the
// current one is used. Warp-collective.
struct TokenCache {
    int cur = -1, nxt = -1, block = -2;   // -2: nothing loaded yet (block + 1 must not match block 0)
    __device__ __forceinline__ int load(const KParams& p, int cid, int ncl, int my_items, int blk, int lane) const {
        const int k = blk * 32 + lane;
        if (!p.tokens || k >= my_items) return -1;
        const int w = cid + k * ncl;
        return w < p.BK ? __ldg(p.tokens + w) : -1;   // item w < B * K is position (w / K, w % K)
    }
    __device__ __forceinline__ int get(const KParams& p, int cid, int ncl, int my_items, int k, int lane) {
        const int blk = k >> 5;
        if (blk != block) {
            cur = blk == block + 1 ? nxt : load(p, cid, ncl, my_items, blk, lane);
            nxt = load(p, cid, ncl, my_items, blk + 1, lane);
            block = blk;
        }
        return __shfl_sync(0xffffffffu, cur, k & 31);
    }
};

// Unit 0 of item k. `tc` null: the token is not looked up (tok = -1).
__device__ __forceinline__ Unit item_unit(const KParams& p, int cid, int ncl, int my_items, int k, TokenCache* tc,
                                          int lane) {
    Unit u;
    u.k = k;
    u.i = 0;
    const int w = cid + k * ncl;
    if (w < p.BK) {
        u.b = w / p.K;
        u.j = w - u.b * p.K;
        u.n = p.N;
    } else {
        u.b = w - p.BK;
        u.j = p.K;
        u.n = 0;
    }
    u.d = u.n > 0 ? drafter_at(0, p.N, p.selected) : -1;
    u.tok = (tc && k < my_items) ? tc->get(p, cid, ncl, my_items, k, lane) : -1;
    return u;
}

__device__ __forceinline__ Unit next_unit(const KParams& p, int cid, int ncl, int my_items, const Unit& u,
                                          TokenCache* tc, int lane) {
    if (u.n > 0 && u.i + 1 < u.n) {
        Unit v = u;
        v.i += 1;
        v.d = drafter_at(v.i, p.N, p.selected);
        return v;
    }
    return item_unit(p, cid, ncl, my_items, u.k + 1, tc, lane);
}

__device__ __forceinline__ bool unit_verified(const KParams& p, const Unit& u) {
    return p.selected >= 0 && u.n > 0 && u.i == u.n - 1;
}
__device__ __forceinline__ bool unit_last(const Unit& u) { return u.n == 0 || u.i == u.n - 1; }

// ------------------------------------------------------------------------------------------------
// per-piece building blocks (one warp, one piece of up to PE logits held in registers; lane l owns
// chunks l + 32 q, q < PCH; chunks past the end of the slice are -inf and contribute exact zeros)
// ------------------------------------------------------------------------------------------------
template <class E>
__device__ __forceinline__ void piece_load(const unsigned char* src, int nchunks, int lane, typename E::Raw (&r)[PCH]) {
    if (nchunks == PCH * 32) {   // a whole piece (all but the last of a slice)
#pragma unroll
        for (int q = 0; q < PCH; ++q) r[q] = E::lds(src, lane + 32 * q);
        return;
    }
#pragma unroll
    for (int q = 0; q < PCH; ++q) {
        const int k = lane + 32 * q;
        r[q] = k < nchunks ? E::lds(src, k) : E::ninf();
    }
}

// Pass 1: folds the piece into the lane's running (max m, sum s of 2^((x - m) c)).
template <class E>
__device__ __forceinline__ void piece_stats(const typename E::Raw (&r)[PCH], float c, float& m, float& s) {
    const float NINF = __uint_as_float(0xFF800000u);
    typename E::Max mm = E::max_init();
#pragma unroll
    for (int q = 0; q < PCH; ++q) mm = E::max_acc(mm, r[q]);
    const float pm = E::max_fin(mm);
    if (pm > NINF) {
        if (pm > m) {
            s = s > 0.f ? s * ex2((m - pm) * c) : 0.f;
            m = pm;
        }
        const float2 cc = make_float2(c, c);
        const float nb = -m * c;
        const float2 nb2 = make_float2(nb, nb);
        float2 s2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int q = 0; q < PCH; ++q)
#pragma unroll
            for (int w = 0; w < 4; ++w) s2[w] = __fadd2_rn(s2[w], ex2x2(__ffma2_rn(E::pair(r[q], w), cc, nb2)));
        const float2 t = __fadd2_rn(__fadd2_rn(s2[0], s2[1]), __fadd2_rn(s2[2], s2[3]));   // independent chains
        s += t.x + t.y;
    }
}

// Pass 2, overlap only: adds sum 2^min(log2 h, log2 p_other) over the piece to acc.
template <class E>
__device__ __forceinline__ void piece_overlap(const typename E::Raw (&rt)[PCH], const typename E::Raw (&ro)[PCH], float c,
                                              float bt, float bo, float2& acc) {
    const float2 cc = make_float2(c, c), bt2 = make_float2(bt, bt), bo2 = make_float2(bo, bo);
    float2 a4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
    for (int q = 0; q < PCH; ++q) a4[q & 3] = chunk_overlap<E>(rt[q], ro[q], cc, bt2, bo2, a4[q & 3]);
    acc = __fadd2_rn(acc, __fadd2_rn(__fadd2_rn(a4[0], a4[1]), __fadd2_rn(a4[2], a4[3])));
}

// Pass 2 with masses: mode 1, residual (h - p_other)+ of the verified row (overlap added to acc); mode 2,
// mass of h (bonus row). Element et of the piece (-1: none) holds the draft token, whose h is patched to
// hpatch. Returns the piece mass, the same value in every lane.
template <class E>
__device__ __forceinline__ float piece_mass(int mode, const typename E::Raw (&rt)[PCH], const typename E::Raw (&ro)[PCH],
                                            int lane, float c, float bt, float bo, int et, float hpatch, float2& acc) {
    const float2 cc = make_float2(c, c), bt2 = make_float2(bt, bt), bo2 = make_float2(bo, bo);
    const int etc = et >= 0 ? et / CHUNK : -1;
    float lm = 0.f;
#pragma unroll
    for (int q = 0; q < PCH; ++q) {
        if (lane + 32 * q != etc) {
            lm += chunk_mass<E>(mode, rt[q], ro[q], cc, bt2, bo2, acc);
        } else {
            float ovl = 0.f;
            lm += chunk_mass_patch_only<E>(mode, rt[q], ro[q], c, bt, bo, et % CHUNK, hpatch, ovl);
            acc.x += ovl;
        }
    }
    return warp_sum(lm);
}

// ------------------------------------------------------------------------------------------------
// the persistent row kernel
// ------------------------------------------------------------------------------------------------
// Shared memory of one CTA:
//   [2][tb_bytes]         resident target slices (only when prm.resident)
//   [W][R][PE * E::BYTES] each consumer warp's private ring of R piece slots
//   full[W * R], tfull[2], tempty[2], lbar[NXB], cbar[NXB], sbar[NXB]   mbarriers
//   lx[NXB][W][XW]        consumer-warp partials of a unit  (max_t, sum_t, max_o, sum_o, x_t, x_o)
//   cx[NXB][C][XW]        the CTAs' partials of a unit, written by every CTA of the cluster
//   sc[NXB][XW]           row scalars of a unit             (bt, bo, btp, h(t), residual needed)
//   abort flag
struct Ctx {
    unsigned char* tbuf;
    unsigned char* ring;
    uint64_t *full, *tfull, *tempty, *lbar, *cbar, *sbar;
    float *lx, *cx, *sc;
    volatile int* abort_flag;
    uint32_t C, rank;
    int cid, ncl;
    int slice_start, n_el, np, my_items;   // np pieces per row slice
    int tb_bytes, slot_bytes;
    size_t row_bytes;
};

// Bounded wait. After any wait of this CTA has timed out, every later wait returns at once, so that a
// failure ends the kernel within a few wait limits instead of one limit per wait.
template <bool CLUSTER = false>
__device__ __forceinline__ bool ctx_wait(const Ctx& x, const KParams& p, uint64_t* bar, uint32_t parity) {
    if (*x.abort_flag) return false;
    if (mbar_wait_bounded<CLUSTER>(bar, parity, p.status, STATUS_TIMEOUT, WAIT_LIMIT_NS)) return true;
    *x.abort_flag = 1;
    return false;
}

__device__ __forceinline__ int piece_len(const Ctx& x, int pc) { return min(PE, x.n_el - pc * PE); }
__device__ __forceinline__ int piece_chunks(const Ctx& x, int pc) { return (piece_len(x, pc) + CHUNK - 1) / CHUNK; }
// first piece of a job owned by consumer warp w, when the job's pieces start at global piece gm (mod W)
__device__ __forceinline__ int first_mine(int gm, int w) { return (w - gm + W) % W; }

// ---------------------------------------- the row-piece walker ----------------------------------------
// The sequence of row pieces a consumer warp reads through its ring, in the order it reads them. Per unit
// u: the warp's pieces of pass 1 of u's other row (O1), of u's target row on an item's first unit (T1,
// streamed mode only), then of pass 2 of unit u - lead (target and other row in streamed mode, the other
// row alone in resident mode; the target alone for a bonus row in streamed mode). Pieces of a job go to
// the warps round robin, continuing the count across jobs; a job with no rows to stream (resident T1,
// resident bonus pass 2) still takes its turn in the count. The row pointers of a job are computed once,
// when the walker enters it.

// sequence b, position j, other rows n and drafter index d of unit (item k, other index i)
__device__ __forceinline__ void unit_geom(const KParams& p, int cid, int ncl, int k, int i, int& b, int& j, int& n,
                                          int& d) {
    const int w = cid + k * ncl;
    if (w < p.BK) {
        b = w / p.K;
        j = w - b * p.K;
        n = p.N;
    } else {
        b = w - p.BK;
        j = p.K;
        n = 0;
    }
    d = n > 0 ? drafter_at(i, p.N, p.selected) : -1;
}

struct Walker {
    int ck = 0, ci = 0;   // the unit whose pass 1 runs this round (item, other index); ck >= my_items: none
    int pk[MAX_LEAD] = {-1}, pi[MAX_LEAD] = {0};   // the last units; pk[lead - 1]: pass 2 this round
    int phase = 0;        // 0: O1 of the pass-1 unit, 1: its T1, 2: pass 2 of unit pk[lead - 1]
    int pc = -1;          // next piece of this warp in the current job (-1: not inside a job)
    int r = 0, per = 0, lr = 0;
    int gm = 0;           // global piece counter mod W at the start of the current job
    const unsigned char* r0 = nullptr;
    const unsigned char* r1 = nullptr;
};

// Advances to this warp's next row piece. Returns false at the end of the sequence.
template <class E>
__device__ bool walker_next(Walker& k, const KParams& p, const Ctx& x, int w, const unsigned char*& src, int& len,
                            int& last_read) {
    const bool res = p.resident != 0;
    const int eb = E::BYTES;
    const size_t slice_off = static_cast<size_t>(x.slice_start) * eb;
    for (;;) {
        if (k.pc >= 0) {
            if (k.pc < x.np) {
                src = (k.r == 0 ? k.r0 : k.r1) + static_cast<size_t>(k.pc) * PE * eb;
                len = piece_len(x, k.pc);
                last_read = k.lr;
                if (++k.r == k.per) {
                    k.r = 0;
                    k.pc += W;
                }
                return true;
            }
            k.gm = (k.gm + x.np) % W;
            k.pc = -1;
        } else {
            const int lead = p.lead;
            const bool have_c = k.ck < x.my_items;
            const int pk = lead == 1 ? k.pk[0] : k.pk[MAX_LEAD - 1];
            const int pi = lead == 1 ? k.pi[0] : k.pi[MAX_LEAD - 1];
            const bool have_p = pk >= 0;
            bool any = have_c || have_p;
#pragma unroll
            for (int q = 0; q < MAX_LEAD; ++q) any = any || k.pk[q] >= 0;
            if (!any) return false;
            int b, j, n, d;
            bool exists = false;
            k.per = 0;
            if (k.phase < 2 && have_c) {
                unit_geom(p, x.cid, x.ncl, k.ck, k.ci, b, j, n, d);
                if (k.phase == 0 && n > 0) {
                    exists = true;
                    k.per = 1;
                    k.r0 = p.others + ((static_cast<size_t>(d) * p.B + b) * p.K + j) * x.row_bytes + slice_off;
                } else if (k.phase == 1 && k.ci == 0) {
                    exists = true;
                    k.per = res ? 0 : 1;
                    k.r0 = p.target + (static_cast<size_t>(b) * (p.K + 1) + j) * x.row_bytes + slice_off;
                }
                k.lr = 0;
            } else if (k.phase == 2 && have_p) {
                unit_geom(p, x.cid, x.ncl, pk, pi, b, j, n, d);
                exists = true;
                const unsigned char* t = p.target + (static_cast<size_t>(b) * (p.K + 1) + j) * x.row_bytes + slice_off;
                if (n > 0) {
                    const unsigned char* o =
                        p.others + ((static_cast<size_t>(d) * p.B + b) * p.K + j) * x.row_bytes + slice_off;
                    k.per = res ? 1 : 2;
                    k.r0 = res ? o : t;
                    k.r1 = o;
                } else {
                    k.per = res ? 0 : 1;
                    k.r0 = t;
                }
                k.lr = 1;
            }
            if (exists) {
                if (k.per > 0) {
                    k.pc = first_mine(k.gm, w);
                    k.r = 0;
                    continue;
                }
                k.gm = (k.gm + x.np) % W;   // a job without streamed rows still takes its turn
            }
        }
        // next phase; after pass 2, the pass-1 unit becomes the pass-2 unit and the next unit follows
        if (++k.phase == 3) {
            k.phase = 0;
#pragma unroll
            for (int q = MAX_LEAD - 1; q > 0; --q) {
                k.pk[q] = k.pk[q - 1];
                k.pi[q] = k.pi[q - 1];
            }
            if (k.ck < x.my_items) {
                k.pk[0] = k.ck;
                k.pi[0] = k.ci;
                int b, j, n, d;
                unit_geom(p, x.cid, x.ncl, k.ck, k.ci, b, j, n, d);
                if (n > 0 && k.ci + 1 < n) {
                    k.ci += 1;
                } else {
                    k.ck += 1;
                    k.ci = 0;
                }
            } else {
                k.pk[0] = -1;
            }
        }
    }
}

// ---------------------------------------- consumer warps ----------------------------------------
// Walks the cluster's units. For unit u: pass 1 of its other row (O1) and, on an item's first unit, of
// the target (T1), then the warp's partials go to the reducer; then pass 2 of unit u - lead (O2, or T2 for
// a bonus row), with the scalars the reducer published for it. Every row piece the warp reads comes through
// its private ring: the warp issues the bulk copy of a piece R pieces before it needs it (a walker runs
// ahead through the same sequence), copies the landed piece into registers and refills the slot at once.
// Only the warp itself waits on its slots, one use after the other, so the parity waits are unambiguous.
template <class E>
__device__ __forceinline__ void consumer_warp(const Ctx& x, const KParams& p, int w, int lane) {
    using Raw = typename E::Raw;
    const float NINF = __uint_as_float(0xFF800000u);
    const float c = p.c;
    const bool res = p.resident != 0;
    const int R = p.R, np = x.np, K = p.K;
    const int eb = E::BYTES;
    unsigned char* const ring = x.ring + static_cast<size_t>(w) * R * x.slot_bytes;
    uint64_t* const full = x.full + w * R;
    const uint64_t pol_keep = policy_evict_normal();   // pass 1: the piece is read again shortly
    const uint64_t pol_last = policy_evict_first();    // pass 2: last read

    Walker iss;   // runs R row pieces ahead of consumption
    int issued = 0, consumed = 0;
    int islot = 0, cslot = 0;   // issued % R and consumed % R, kept as wrapping counters
    uint32_t cpar = 0;          // (consumed / R) & 1
    auto issue_one = [&]() {
        const unsigned char* src;
        int len, last_read;
        if (!walker_next<E>(iss, p, x, w, src, len, last_read)) return;
        const int slot = islot;
        if (++islot == R) islot = 0;
        unsigned char* dst = ring + static_cast<size_t>(slot) * x.slot_bytes;
        if (p.tma) {
            if (lane == 0) {
                // the warp's earlier reads of this slot (generic proxy) come before the copy that refills it
                fence_proxy_async_shared();
                const uint32_t bytes = static_cast<uint32_t>(len) * eb;
                mbar_arrive_expect_tx(&full[slot], bytes);
                bulk_load(dst, src, bytes, &full[slot], last_read ? pol_last : pol_keep);
            }
        } else {
            E::copy_slice(dst, src, len, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[slot]);
        }
        ++issued;
    };
    // Next row piece into registers (the piece's chunks pc); `tl`, if inside the piece, is read as `xv`.
    auto take = [&](int pc, Raw (&r)[PCH], int tl, float& xv) {
        const int slot = cslot;
        const unsigned char* src = ring + static_cast<size_t>(slot) * x.slot_bytes;
        ctx_wait(x, p, &full[slot], cpar);
        if (++cslot == R) {
            cslot = 0;
            cpar ^= 1u;
        }
        piece_load<E>(src, piece_chunks(x, pc), lane, r);
        if (tl >= 0 && tl / PE == pc && lane == ((tl % PE) / CHUNK) % 32) xv = E::at(src, tl % PE);
        __syncwarp();
        ++consumed;
        issue_one();
    };
    for (int i = 0; i < R; ++i) issue_one();

    int gm = 0;   // global piece counter mod W
    TokenCache tc;
    Unit cur{};
    Unit pend[MAX_LEAD];   // the last units, pend[lead - 1] the one whose pass 2 runs this round
    bool have[MAX_LEAD] = {};
    const int lead = p.lead;
    bool have_cur = x.my_items > 0;
    if (have_cur) cur = item_unit(p, x.cid, x.ncl, x.my_items, 0, &tc, lane);
    auto local_tok = [&](int tok) {
        return (tok >= 0 && tok < p.V && tok >= x.slice_start && tok < x.slice_start + x.n_el) ? tok - x.slice_start : -1;
    };
    auto any_left = [&]() {
        bool a = have_cur;
#pragma unroll
        for (int q = 0; q < MAX_LEAD; ++q) a = a || have[q];
        return a;
    };
    for (int u = 0; any_left(); ++u) {
        if (have_cur) {
            const bool ver = unit_verified(p, cur);
            const int tl = local_tok(cur.tok);
            float mt = NINF, st = 0.f, mo = NINF, so = 0.f, xt = NINF, xo = NINF;
            if (cur.n > 0) {   // O1: pass 1 of the other row, from HBM
                for (int pc = first_mine(gm, w); pc < np; pc += W) {
                    Raw r[PCH];
                    take(pc, r, ver ? tl : -1, xo);
                    piece_stats<E>(r, c, mo, so);
                }
                gm = (gm + np) % W;
            }
            if (cur.i == 0) {   // T1: pass 1 of the target row
                const unsigned char* tb = x.tbuf + static_cast<size_t>(cur.k & 1) * x.tb_bytes;
                bool waited = false;
                for (int pc = first_mine(gm, w); pc < np; pc += W) {
                    Raw r[PCH];
                    if (res) {
                        if (!waited) ctx_wait(x, p, &x.tfull[cur.k & 1], static_cast<uint32_t>((cur.k >> 1) & 1));
                        waited = true;
                        const unsigned char* src = tb + static_cast<size_t>(pc) * PE * eb;
                        piece_load<E>(src, piece_chunks(x, pc), lane, r);
                        if (tl >= 0 && tl / PE == pc && lane == ((tl % PE) / CHUNK) % 32) xt = E::at(src, tl % PE);
                    } else {
                        take(pc, r, tl, xt);
                    }
                    piece_stats<E>(r, c, mt, st);
                }
                gm = (gm + np) % W;
            }
            // the warp's partials of unit u to the reducer
            const MaxSum a = warp_ms(MaxSum{mt, st}, c);
            const MaxSum o = warp_ms(MaxSum{mo, so}, c);
            const float xtm = warp_max(xt), xom = warp_max(xo);
            if (lane == 0) {
                float* e = x.lx + (static_cast<size_t>(u % NXB) * W + w) * XW;
                e[0] = a.m;
                e[1] = a.s;
                e[2] = o.m;
                e[3] = o.s;
                e[4] = xtm;
                e[5] = xom;
                mbar_arrive(&x.lbar[u % NXB]);
            }
        }
        if (lead == 1 ? have[0] : have[MAX_LEAD - 1]) {   // pass 2 of unit u - lead, re-read from L2
            const Unit& prev = lead == 1 ? pend[0] : pend[MAX_LEAD - 1];
            const int pu = u - lead;
            const bool ver = unit_verified(p, prev);
            const int f0 = first_mine(gm, w);
            // Every warp waits for the scalars, also one without a piece in this pass: the wait keeps all
            // warps within lead + 1 units of the reducer, which the reuse of the exchange buffers and
            // barriers (NXB > lead + 1 units deep) relies on.
            ctx_wait(x, p, &x.sbar[pu % NXB], static_cast<uint32_t>((pu / NXB) & 1));
            const float* sp = x.sc + (pu % NXB) * XW;
            const float bt = sp[0], bo = sp[1], btp = sp[2], ht = sp[3];
            const bool need_res = sp[4] != 0.f;   // verified row that rejects (or every row when diag is wanted)
            if (res && f0 < np) ctx_wait(x, p, &x.tfull[prev.k & 1], static_cast<uint32_t>((prev.k >> 1) & 1));
            const size_t row = static_cast<size_t>(prev.b) * (K + 1) + prev.j;
            const unsigned char* tb = x.tbuf + static_cast<size_t>(prev.k & 1) * x.tb_bytes;
            float* const tiles = p.tiles ? p.tiles + (row * x.C + x.rank) * p.pcap : nullptr;
            float2 acc = make_float2(0.f, 0.f);
            float unused = NINF;
            if (prev.n > 0) {   // O2
                const int tl = ver ? local_tok(prev.tok) : -1;
                for (int pc = f0; pc < np; pc += W) {
                    Raw rt[PCH], ro[PCH];
                    if (res) piece_load<E>(tb + static_cast<size_t>(pc) * PE * eb, piece_chunks(x, pc), lane, rt);
                    else take(pc, rt, -1, unused);
                    take(pc, ro, -1, unused);
                    if (ver && need_res) {
                        const int et = (tl >= 0 && tl / PE == pc) ? tl % PE : -1;
                        const float m = piece_mass<E>(1, rt, ro, lane, c, bt, bo, et, ht, acc);
                        if (lane == 0 && tiles) tiles[pc] = m;
                    } else if (!ver || p.gpart) {
                        piece_overlap<E>(rt, ro, c, bt, bo, acc);
                    }
                }
                if (p.gpart) {
                    const float sum = warp_sum(acc.x + acc.y);
                    if (lane == 0)
                        p.gpart[(((static_cast<size_t>(prev.d) * p.B + prev.b) * K + prev.j) * x.C + x.rank) * W + w] = sum;
                }
            } else {   // T2: bonus row, mass of p_target per piece
                for (int pc = f0; pc < np; pc += W) {
                    Raw rt[PCH];
                    if (res) piece_load<E>(tb + static_cast<size_t>(pc) * PE * eb, piece_chunks(x, pc), lane, rt);
                    else take(pc, rt, -1, unused);
                    const float m = piece_mass<E>(2, rt, rt, lane, c, btp, 0.f, -1, 0.f, acc);
                    if (lane == 0 && tiles) tiles[pc] = m;
                }
            }
            gm = (gm + np) % W;
            if (res && unit_last(prev)) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&x.tempty[prev.k & 1]);
            }
        }
#pragma unroll
        for (int q = MAX_LEAD - 1; q > 0; --q) {
            pend[q] = pend[q - 1];
            have[q] = have[q - 1];
        }
        pend[0] = cur;
        have[0] = have_cur;
        if (have_cur) {
            cur = next_unit(p, x.cid, x.ncl, x.my_items, cur, &tc, lane);
            have_cur = cur.k < x.my_items;
        }
    }
    // Copies issued but not consumed (only after a failure): they must land before the CTA may exit.
    if (p.tma && lane == 0)
        for (int k = consumed; k < issued; ++k)
            mbar_wait_bounded(&full[k % R], static_cast<uint32_t>((k / R) & 1), p.status, STATUS_TIMEOUT, WAIT_LIMIT_NS);
    __syncwarp();
}

// ---------------------------------------- reducer warp ----------------------------------------
// Per unit: merges the W consumer partials, sends the CTA's partial to every CTA of the cluster, merges
// the C partials it receives (the same C entries in the same order in every CTA, so every CTA derives
// bit-identical scalars), publishes the row scalars to the consumers and, in CTA 0, writes the record.
template <class E>
__device__ __forceinline__ void reducer_warp(const Ctx& x, const KParams& p, int lane) {
    const float NINF = __uint_as_float(0xFF800000u);
    const float c = p.c;
    const int K = p.K;
    TokenCache tc;
    float bt = 0.f, btp = 0.f, ht = 0.f;   // the current item's target scalars
    Unit cur{};
    if (x.my_items > 0) cur = item_unit(p, x.cid, x.ncl, x.my_items, 0, &tc, lane);
    for (int u = 0; cur.k < x.my_items; ++u) {
        const int xb = u % NXB;
        const uint32_t par = static_cast<uint32_t>((u / NXB) & 1);
        ctx_wait(x, p, &x.lbar[xb], par);
        MaxSum a{NINF, 0.f}, o{NINF, 0.f};
        float xt = NINF, xo = NINF;
        if (lane < W) {
            const float* e = x.lx + (static_cast<size_t>(xb) * W + lane) * XW;
            a = {e[0], e[1]};
            o = {e[2], e[3]};
            xt = e[4];
            xo = e[5];
        }
        a = warp_ms(a, c);
        o = warp_ms(o, c);
        xt = warp_max(xt);
        xo = warp_max(xo);
        if (lane < static_cast<int>(x.C)) {
            const uint32_t local = smem_addr(x.cx + (static_cast<size_t>(xb) * x.C + x.rank) * XW);
            const uint32_t remote = map_to_rank(local, static_cast<uint32_t>(lane));
            st_cluster_f32x4(remote, a.m, a.s, o.m, o.s);
            st_cluster_f32x4(remote + 16, xt, xo, 0.f, 0.f);
            mbar_arrive_remote(map_to_rank(smem_addr(&x.cbar[xb]), static_cast<uint32_t>(lane)));
        }
        ctx_wait<true>(x, p, &x.cbar[xb], par);
        MaxSum ga{NINF, 0.f}, go{NINF, 0.f};
        float gxt = NINF, gxo = NINF;
        if (lane < static_cast<int>(x.C)) {
            const float* e = x.cx + (static_cast<size_t>(xb) * x.C + lane) * XW;
            ga = {e[0], e[1]};
            go = {e[2], e[3]};
            gxt = e[4];
            gxo = e[5];
        }
        ga = warp_ms(ga, c);
        go = warp_ms(go, c);
        gxt = warp_max(gxt);
        gxo = warp_max(gxo);
        const bool ver = unit_verified(p, cur);
        if (cur.i == 0) {
            btp = beta_of(ga, c);
            bt = btp;
            ht = prob_of(gxt, ga, c);   // 0 when no CTA holds the token (none, or outside [0, V))
            if (p.cactus && cur.j < K) {
                float log2s;
                cactus_scalars(ht, p.delta, ht, log2s);
                bt = btp + log2s;
            }
        }
        const float bo = cur.n > 0 ? beta_of(go, c) : 0.f;
        const float pd = ver ? prob_of(gxo, go, c) : 0.f;
        // The residual of a verified position is drawn from only if the position rejects. The decision is
        // the finish kernel's own comparison on the same floats (h(t) and p_draft(t) go to the record
        // unchanged), so an accepted position can skip its residual masses.
        float need_residual = 1.f;
        if (ver && !p.all_residuals && p.seeds) {
            const float r = philox_uniform(__ldg(p.seeds + cur.b), static_cast<uint32_t>(cur.b),
                                           static_cast<uint32_t>(cur.j), 0u);
            need_residual = r * pd < ht ? 0.f : 1.f;
        }
        if (lane == 0) {
            float* s = x.sc + xb * XW;
            s[0] = bt;
            s[1] = bo;
            s[2] = btp;
            s[3] = ht;
            s[4] = need_residual;
            mbar_arrive(&x.sbar[xb]);
            if (x.rank == 0) {
                if (cur.i == 0 && cur.j < K && p.tokens && !(cur.tok >= 0 && cur.tok < p.V))
                    atomicOr(p.status, STATUS_BAD_TOKEN);
                if (p.rec) {
                    float* rp = p.rec + (static_cast<size_t>(cur.b) * (K + 1) + cur.j) * REC;
                    if (cur.i == 0) {
                        rp[R_HT] = ht;
                        rp[R_BT] = bt;
                        rp[R_BTP] = btp;
                        if (cur.n == 0) {
                            rp[R_PD] = 0.f;
                            rp[R_BO] = 0.f;
                        }
                    }
                    if (ver) {
                        rp[R_PD] = pd;
                        rp[R_BO] = bo;
                    }
                }
            }
        }
        cur = next_unit(p, x.cid, x.ncl, x.my_items, cur, &tc, lane);
    }
}

// ---------------------------------------- target loader warp ----------------------------------------
// Resident mode only: loads each item's target slice into buffer k % 2 as soon as the consumer warps have
// released the item that used the buffer before (two items earlier).
template <class E>
__device__ __forceinline__ void loader_warp(const Ctx& x, const KParams& p, int lane) {
    if (!p.resident) return;
    const int K = p.K;
    const int eb = E::BYTES;
    const uint64_t pol_last = policy_evict_first();
    const size_t slice_off = static_cast<size_t>(x.slice_start) * eb;
    const uint32_t bytes = static_cast<uint32_t>(x.n_el) * eb;
    int kt = 0;
    for (; kt < x.my_items; ++kt) {
        if (kt >= 2) {
            bool ok = !*x.abort_flag;
            if (ok && lane == 0)
                ok = mbar_wait_bounded(&x.tempty[kt & 1], static_cast<uint32_t>(((kt >> 1) - 1) & 1), p.status,
                                       STATUS_TIMEOUT, WAIT_LIMIT_NS);
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
                *x.abort_flag = 1;
                break;
            }
        }
        const int w = x.cid + kt * x.ncl;
        const int b = w < p.BK ? w / K : w - p.BK;
        const int j = w < p.BK ? w - b * K : K;
        const unsigned char* src = p.target + (static_cast<size_t>(b) * (K + 1) + j) * x.row_bytes + slice_off;
        unsigned char* dst = x.tbuf + static_cast<size_t>(kt & 1) * x.tb_bytes;
        uint64_t* bar = &x.tfull[kt & 1];
        if (p.tma) {
            if (lane == 0) {
                mbar_arrive_expect_tx(bar, bytes);
                for (uint32_t off = 0; off < bytes; off += 32768u)
                    bulk_load(dst + off, src + off, min(32768u, bytes - off), bar, pol_last);
            }
        } else {
            E::copy_slice(dst, src, x.n_el, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar);
        }
    }
    // every copy issued must have landed before the CTA may exit
    if (p.tma && lane == 0) {
        for (int q = 0; q < min(kt, 2); ++q) {
            const int last = q + ((kt - 1 - q) / 2) * 2;
            mbar_wait_bounded(&x.tfull[q], static_cast<uint32_t>((last >> 1) & 1), p.status, STATUS_TIMEOUT, WAIT_LIMIT_NS);
        }
    }
    __syncwarp();
}

template <class E>
__global__ void __launch_bounds__(NT, 1) rows_kernel(const __grid_constant__ KParams prm) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int R = prm.R;
    Ctx x;
    x.C = cluster_nctarank();
    x.rank = cluster_ctarank();
    x.cid = static_cast<int>(cluster_id_x());
    x.ncl = static_cast<int>(ncluster_x());
    x.slot_bytes = PE * E::BYTES;
    x.tb_bytes = prm.resident ? (prm.slice_elems * E::BYTES + 127) / 128 * 128 : 0;
    x.tbuf = smem;
    x.ring = smem + 2 * static_cast<size_t>(x.tb_bytes);
    x.full = reinterpret_cast<uint64_t*>(x.ring + static_cast<size_t>(W) * R * x.slot_bytes);
    x.tfull = x.full + W * R;
    x.tempty = x.tfull + 2;
    x.lbar = x.tempty + 2;
    x.cbar = x.lbar + NXB;
    x.sbar = x.cbar + NXB;
    x.lx = reinterpret_cast<float*>(x.sbar + NXB);
    x.cx = x.lx + NXB * W * XW;
    x.sc = x.cx + NXB * x.C * XW;
    x.abort_flag = reinterpret_cast<volatile int*>(x.sc + NXB * XW);
    x.slice_start = static_cast<int>(x.rank) * prm.slice_elems;
    x.n_el = max(0, min(prm.slice_elems, prm.V - x.slice_start));
    x.np = (x.n_el + PE - 1) / PE;
    x.my_items = x.cid < prm.num_items ? (prm.num_items - 1 - x.cid) / x.ncl + 1 : 0;
    x.row_bytes = static_cast<size_t>(prm.V) * E::BYTES;

    if (tid == 0) {
        for (int s = 0; s < W * R; ++s) mbar_init(&x.full[s], 1);
        for (int q = 0; q < 2; ++q) {
            mbar_init(&x.tfull[q], 1);
            mbar_init(&x.tempty[q], W);
        }
        for (int q = 0; q < NXB; ++q) {
            mbar_init(&x.lbar[q], W);
            mbar_init(&x.cbar[q], x.C);
            mbar_init(&x.sbar[q], 1);
        }
        *x.abort_flag = 0;
        fence_mbarrier_init_cluster();
    }
    __syncthreads();
    cluster_sync_all();   // barriers initialised and every CTA running before any remote access

    if (warp < W) consumer_warp<E>(x, prm, warp, lane);
    else if (warp == W) reducer_warp<E>(x, prm, lane);
    else loader_warp<E>(x, prm, lane);

    // no CTA may leave while a peer can still write into its shared memory
    cluster_sync_all();
}

// ------------------------------------------------------------------------------------------------
// gamma partial reduction: one warp per (drafter, sequence, level), C * W partials in a fixed order
// ------------------------------------------------------------------------------------------------
struct GParams {
    const float* gpart;   // [N*B*K, C, W]
    int n_out, C;
    float* gamma;
    float* loss;
};

__global__ void __launch_bounds__(256) gamma_reduce_kernel(const GParams g) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int o = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (o >= g.n_out) return;
    const int n = g.C * W;
    const float* p = g.gpart + static_cast<size_t>(o) * n;
    float s = 0.f;
    for (int i = lane; i < n; i += 32) s += p[i];
    s = warp_sum(s);
    if (lane == 0) {
        g.gamma[o] = s;
        if (g.loss) g.loss[o] = 1.f - s;
    }
}

// ------------------------------------------------------------------------------------------------
// chain finish and draw: one warp per sequence (lossless tutorial §9.1: verify left to right, stop at
// the first reject and emit its residual draw; all accepted: emit the bonus draw)
// ------------------------------------------------------------------------------------------------
struct FParams {
    const float* rec;            // [B, K+1, REC]
    const float* tiles;          // [B, K+1, C, pcap]: mass of each piece of each CTA slice
    const unsigned char* target; // [B, K+1, V]
    const unsigned char* other;  // verified drafter rows: row (b, j) starts at element (b * K + j) * V
    const int32_t* tokens;       // [B, K]
    const uint64_t* seeds;       // [B]
    int B, K, V, C, slice_elems, pcap;
    float c;
    int32_t* accept_len;         // [B]
    int32_t* out_tokens;         // [B, K+1]
    float* diag;                 // [B, K, 4] or null
    float* gamma_star;           // [B, K] or null (Cactus)
};

__device__ __forceinline__ int fp_slice_len(const FParams& f, int r) {
    return max(0, min(f.slice_elems, f.V - r * f.slice_elems));
}
__device__ __forceinline__ int fp_slice_pieces(const FParams& f, int r) { return (fp_slice_len(f, r) + PE - 1) / PE; }

// piece `flat` of the row in vocabulary order (slice-major); sets its first element and length
__device__ __forceinline__ float fp_piece(const FParams& f, size_t row, int flat, int* e_begin = nullptr,
                                          int* len = nullptr) {
    int r = 0;
    while (r < f.C - 1 && flat >= fp_slice_pieces(f, r)) {
        flat -= fp_slice_pieces(f, r);
        ++r;
    }
    if (e_begin) *e_begin = r * f.slice_elems + flat * PE;
    if (len) *len = min(PE, fp_slice_len(f, r) - flat * PE);
    return f.tiles[(row * f.C + r) * f.pcap + flat];
}

// Scans the logits [e_begin, e_end) of the rows (pointers to logit 0) in ascending order, 256 per step,
// and returns the first element whose running mass (starting at `before`) exceeds tp; when none does,
// the last element with positive mass (-1 if there is none). mode 1: residual (h - p_other)+, mode 2: h.
// Logit `tok` of h is patched to ht. The values are computed exactly as in the row pass.
template <class E, bool AL>
__device__ int scan_pick(float c, const unsigned char* trow, const unsigned char* orow, int mode, int e_begin,
                         int e_end, float bt, float bo, int tok, float ht, float tp, float before, int lane) {
    using Raw = typename E::Raw;
    int last_pos = -1;
    for (int base = e_begin; base < e_end; base += 32 * CHUNK) {
        const int e0 = base + lane * CHUNK;
        float v[8];
        float m = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = 0.f;
        if (e0 < e_end) {
            const Raw rt = E::template gload<AL>(trow, e0, e_end);
            const Raw ro = mode == 1 ? E::template gload<AL>(orow, e0, e_end) : rt;
            const int et = (tok >= e0 && tok < e0 + CHUNK) ? tok - e0 : -1;
            float ovl = 0.f;
            chunk_values<E>(mode, rt, ro, c, bt, bo, et, ht, v, ovl);
#pragma unroll
            for (int q = 0; q < 8; ++q) m += v[q];
        }
        const float incl = warp_incl_scan(m, lane);
        const unsigned over = __ballot_sync(0xffffffffu, m > 0.f && before + incl > tp);
        const unsigned posm = __ballot_sync(0xffffffffu, m > 0.f);
        if (over) {
            const int ln = __ffs(over) - 1;
            int pick = -1;
            if (lane == ln) {
                float a = before + incl - m;
                int lp = -1;
                for (int q = 0; q < 8; ++q) {
                    a += v[q];
                    if (v[q] > 0.f) {
                        lp = q;
                        if (pick < 0 && a > tp) pick = q;
                    }
                }
                pick = e0 + (pick >= 0 ? pick : lp);
            }
            return __shfl_sync(0xffffffffu, pick, ln);
        }
        if (posm) {
            const int ln = 31 - __clz(posm);
            int lp = -1;
            for (int q = 0; q < 8; ++q)
                if (v[q] > 0.f) lp = q;
            last_pos = __shfl_sync(0xffffffffu, e0 + lp, ln);
        }
        before = __shfl_sync(0xffffffffu, before + incl, 31);
    }
    return last_pos;
}

// The same scan over one piece of at most PE logits, with every load issued before the scan (one memory
// latency instead of one per 256 logits). Lane l holds logits e_begin + 256 r + 8 l .. + 7 of round r.
template <class E, bool AL>
__device__ int scan_pick_piece(float c, const unsigned char* trow, const unsigned char* orow, int mode, int e_begin,
                               int e_end, float bt, float bo, int tok, float ht, float tp, float before, int lane) {
    using Raw = typename E::Raw;
    Raw rt[PCH], ro[PCH];
#pragma unroll
    for (int r = 0; r < PCH; ++r) {
        const int e0 = e_begin + r * 32 * CHUNK + lane * CHUNK;
        rt[r] = E::template gload<AL>(trow, e0, e_end);
        ro[r] = mode == 1 ? E::template gload<AL>(orow, e0, e_end) : rt[r];
    }
    int last_pos = -1;
#pragma unroll 1
    for (int r = 0; r < PCH; ++r) {
        const int base = e_begin + r * 32 * CHUNK;
        if (base >= e_end) break;
        const int e0 = base + lane * CHUNK;
        float v[8];
        float m = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = 0.f;
        Raw a = rt[0], b = ro[0];
#pragma unroll
        for (int q = 1; q < PCH; ++q)
            if (q == r) {
                a = rt[q];
                b = ro[q];
            }
        if (e0 < e_end) {
            const int et = (tok >= e0 && tok < e0 + CHUNK) ? tok - e0 : -1;
            float ovl = 0.f;
            chunk_values<E>(mode, a, b, c, bt, bo, et, ht, v, ovl);
#pragma unroll
            for (int q = 0; q < 8; ++q) m += v[q];
        }
        const float incl = warp_incl_scan(m, lane);
        const unsigned over = __ballot_sync(0xffffffffu, m > 0.f && before + incl > tp);
        const unsigned posm = __ballot_sync(0xffffffffu, m > 0.f);
        if (over) {
            const int ln = __ffs(over) - 1;
            int pick = -1;
            if (lane == ln) {
                float acc = before + incl - m;
                int lp = -1;
                for (int q = 0; q < 8; ++q) {
                    acc += v[q];
                    if (v[q] > 0.f) {
                        lp = q;
                        if (pick < 0 && acc > tp) pick = q;
                    }
                }
                pick = e0 + (pick >= 0 ? pick : lp);
            }
            return __shfl_sync(0xffffffffu, pick, ln);
        }
        if (posm) {
            const int ln = 31 - __clz(posm);
            int lp = -1;
            for (int q = 0; q < 8; ++q)
                if (v[q] > 0.f) lp = q;
            last_pos = __shfl_sync(0xffffffffu, e0 + lp, ln);
        }
        before = __shfl_sync(0xffffffffu, before + incl, 31);
    }
    return last_pos;
}

template <class E, bool AL>
__global__ void __launch_bounds__(256) finish_kernel(const FParams f) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (b >= f.B) return;
    const int K = f.K;
    const uint64_t seed = f.seeds[b];
    const size_t row_bytes = static_cast<size_t>(f.V) * E::BYTES;
    int total = 0;
    for (int r = 0; r < f.C; ++r) total += fp_slice_pieces(f, r);

    // ---- accept chain ----
    int L = K;
    for (int base = 0; base < K; base += 32) {
        const int j = base + lane;
        bool acc = true;
        if (j < K) {
            const float* rp = f.rec + (static_cast<size_t>(b) * (K + 1) + j) * REC;
            const float r = philox_uniform(seed, static_cast<uint32_t>(b), static_cast<uint32_t>(j), 0u);
            acc = r * rp[R_PD] < rp[R_HT];
            if (f.gamma_star) f.gamma_star[static_cast<size_t>(b) * K + j] = rp[R_HT];
        }
        const unsigned rej = __ballot_sync(0xffffffffu, !acc);
        if (L == K && rej) L = base + __ffs(rej) - 1;
    }

    // ---- draw from row L: residual (L < K) or the bonus target row (L = K) ----
    const size_t row = static_cast<size_t>(b) * (K + 1) + L;
    const float* rp = f.rec + row * REC;
    const int mode = L < K ? 1 : 2;
    const int tok = L < K ? f.tokens[static_cast<size_t>(b) * K + L] : -1;
    const float bt = mode == 1 ? rp[R_BT] : rp[R_BTP];
    const float bo = rp[R_BO];
    const float ht = rp[R_HT];
    const float u = philox_uniform(seed, static_cast<uint32_t>(b), static_cast<uint32_t>(L), 1u);
    const unsigned char* trow = f.target + row * row_bytes;
    const unsigned char* orow = mode == 1 ? f.other + (static_cast<size_t>(b) * K + L) * row_bytes : trow;
    // inclusive prefix of the piece masses in vocabulary order; every lane owns a contiguous run
    const int seg = (total + 31) / 32;
    const int lo = lane * seg, hi = min(total, lo + seg);
    float local = 0.f;
    for (int t = lo; t < hi; ++t) local += fp_piece(f, row, t);
    const float incl = warp_incl_scan(local, lane);
    float excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl = 0.f;
    const float Z = __shfl_sync(0xffffffffu, incl, 31);
    int emitted;
    if (mode == 1 && !(Z > 0.f)) {
        // the residual rounded to zero mass: draw from h over the whole row instead (the reading for a
        // reject whose computed Z is not positive)
        float all = 0.f;
        for (int e0 = lane * CHUNK; e0 < f.V; e0 += 32 * CHUNK) {
            const typename E::Raw rt = E::template gload<AL>(trow, e0, f.V);
            float2 unused = make_float2(0.f, 0.f);
            const int et = (tok >= e0 && tok < e0 + CHUNK) ? tok - e0 : -1;
            all += chunk_mass_patched<E>(2, rt, rt, f.c, bt, 0.f, et, ht, unused);
        }
        const float tp = u * warp_sum(all);
        emitted = scan_pick<E, AL>(f.c, trow, trow, 2, 0, f.V, bt, 0.f, tok, ht, tp, 0.f, lane);
    } else {
        const float tp = u * Z;
        // first piece whose prefix exceeds tp (else the last piece with mass)
        int found = -1, lastp = -1;
        float before_found = 0.f, before_last = 0.f;
        float run = excl;
        for (int t = lo; t < hi; ++t) {
            const float m = fp_piece(f, row, t);
            const float pre = run + m;
            if (m > 0.f) {
                lastp = t;
                before_last = run;
                if (found < 0 && pre > tp) {
                    found = t;
                    before_found = run;
                }
            }
            run = pre;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, found >= 0);
        int ft;
        float before_piece;
        if (hit) {
            const int ln = __ffs(hit) - 1;
            ft = __shfl_sync(0xffffffffu, found, ln);
            before_piece = __shfl_sync(0xffffffffu, before_found, ln);
        } else {
            const unsigned any = __ballot_sync(0xffffffffu, lastp >= 0);
            const int ln = any ? 31 - __clz(any) : 0;
            ft = __shfl_sync(0xffffffffu, lastp, ln);
            before_piece = __shfl_sync(0xffffffffu, before_last, ln);
        }
        emitted = -1;
        if (ft >= 0) {
            int e_begin = 0, len = 0;
            fp_piece(f, row, ft, &e_begin, &len);
            emitted = scan_pick_piece<E, AL>(f.c, trow, orow, mode, e_begin, e_begin + len, bt, bo, tok, ht, tp,
                                             before_piece, lane);
        }
    }

    // ---- outputs ----
    for (int j = lane; j <= K; j += 32) {
        int v;
        if (j < L) v = f.tokens[static_cast<size_t>(b) * K + j];
        else if (j == L) v = emitted;
        else v = -1;
        f.out_tokens[static_cast<size_t>(b) * (K + 1) + j] = v;
    }
    if (lane == 0) f.accept_len[b] = L;
    if (f.diag) {
        for (int j = 0; j < K; ++j) {
            const size_t rj = static_cast<size_t>(b) * (K + 1) + j;
            float zs = 0.f;
            for (int t = lane; t < total; t += 32) zs += fp_piece(f, rj, t);
            zs = warp_sum(zs);
            if (lane == 0) {
                const float* q = f.rec + rj * REC;
                float* d = f.diag + (static_cast<size_t>(b) * K + j) * 4;
                d[0] = q[R_HT];
                d[1] = q[R_PD];
                d[2] = zs;
                d[3] = philox_uniform(seed, static_cast<uint32_t>(b), static_cast<uint32_t>(j), 0u);
            }
        }
    }
}

}  // namespace specv
