// Verification kernels for sm_103a.
//
// rows_kernel: one persistent grid of thread-block clusters. A cluster of C CTAs works on one "item" at a
// time: the target row (b, j) plus the other rows verified against it (the draft row for standard and
// Cactus verification, all N drafter rows for the counterfactual evaluation, none for the bonus row
// j = K). CTA `rank` owns the vocabulary slice [rank * slice, (rank + 1) * slice) of every row. In each CTA
// one producer warp streams the row slices into shared memory with bulk (TMA) copies through full/empty
// mbarriers, and 15 consumer warps compute. Every logit is read from HBM once. Each row's softmax
// normaliser (global max and sum of exponentials) is combined across the cluster through distributed
// shared memory, signalled by remote mbarrier arrivals (no cluster-wide barrier per row). With the
// normalisers known, each CTA evaluates for its slice:
//   - sum_x min(p_target, p_other) per warp        (HedgeSpec gamma partials; gamma = 1 - TV)
//   - the residual mass (h - p_draft)+ per 256-token tile, h = p_target or the Cactus h (verified row)
//   - or the mass of p_target per tile (bonus row)
// and writes them, with one record per position (h(t), p_draft(t) and the rows' log-offsets), to the
// workspace.
// finish_kernel: one warp per sequence turns the records into the accept/reject chain and draws the
// residual (or bonus) token by inverse CDF: a prefix scan over the tile masses of the chosen row, then one
// re-read of that 256-token tile. gamma_reduce_kernel sums the gamma partials.
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

constexpr int NWC = 15;                 // consumer warps per CTA
constexpr int NTC = NWC * 32;           // consumer threads
constexpr int NT = NTC + 32;            // plus one producer warp
constexpr int CHUNK = 8;                // elements per consumer thread per pass (16 B of bf16)
constexpr int TILE = CHUNK * 32;        // elements per warp per pass: one residual tile
constexpr int SLICE_Q = 128;            // granularity of the per-CTA vocabulary slice
constexpr int REC = 8;                  // 32-bit words per position record
constexpr int MAX_SLOTS = 4;
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
    int B, K, V, N;
    int selected;                  // drafter whose chain is verified (processed last); -1: none
    int J;                         // items per sequence (K, or K + 1 with the bonus row)
    int num_items;                 // B * J
    float c;                       // log2(e) / temperature
    float delta;                   // Cactus divergence budget
    int cactus;
    int slice_elems;               // per-CTA slice, multiple of SLICE_Q
    int tma;                       // 1: every row slice is 16-byte aligned -> bulk copies
    int ts, r;                     // target slots, ring slots for the other rows
    int slot_bytes;
    int tiles_cap;                 // tiles per slice in the workspace layout
    float* rec;                    // [B, K+1, REC] or null
    float* tiles;                  // [B, K+1, C, tiles_cap] or null
    float* gpart;                  // [N, B, K, C, NWC] or null
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
    // one chunk of a row in global memory, -inf beyond n_el (rows of any alignment)
    __device__ static Raw gchunk(const unsigned char* row, int e0, int n_el, bool aligned) {
        if (aligned && e0 + CHUNK <= n_el) return __ldcs(reinterpret_cast<const uint4*>(row) + e0 / CHUNK);
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
    __device__ static Raw gchunk(const unsigned char* row, int e0, int n_el, bool aligned) {
        const float* f = reinterpret_cast<const float*>(row);
        if (aligned && e0 + CHUNK <= n_el) {
            const float4* p = reinterpret_cast<const float4*>(f + e0);
            return {__ldcs(p), __ldcs(p + 1)};
        }
        float v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = e0 + q < n_el ? __ldg(f + e0 + q) : __uint_as_float(0xFF800000u);
        return {make_float4(v[0], v[1], v[2], v[3]), make_float4(v[4], v[5], v[6], v[7])};
    }
};

__device__ __forceinline__ float2 ex2x2(float2 t) { return make_float2(ex2(t.x), ex2(t.y)); }

// ------------------------------------------------------------------------------------------------
// per-thread building blocks
// ------------------------------------------------------------------------------------------------
template <class E, int P>
__device__ __forceinline__ void load_raw(const unsigned char* slot, int ctid, int nchunks, typename E::Raw (&raw)[P]) {
#pragma unroll
    for (int p = 0; p < P; ++p) {
        const int k = p * NTC + ctid;
        raw[p] = k < nchunks ? E::lds(slot, k) : E::ninf();
    }
}

// Thread-local (max m, sum of 2^((x - m) c)) over the thread's chunks.
template <class E, int P>
__device__ __forceinline__ MaxSum local_stats(const typename E::Raw (&raw)[P], float c) {
    typename E::Max mm = E::max_init();
#pragma unroll
    for (int p = 0; p < P; ++p) mm = E::max_acc(mm, raw[p]);
    const float m = E::max_fin(mm);
    if (!(m > __uint_as_float(0xFF800000u))) return {m, 0.f};
    const float2 cc = make_float2(c, c);
    const float2 nb = make_float2(-m * c, -m * c);
    float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int p = 0; p < P; ++p)
#pragma unroll
        for (int w = 0; w < 4; ++w) s2 = __fadd2_rn(s2, ex2x2(__ffma2_rn(E::pair(raw[p], w), cc, nb)));
    return {m, s2.x + s2.y};
}

// Same statistics streamed from a shared-memory slot (no register copy of the row is kept).
template <class E, int P>
__device__ __forceinline__ MaxSum local_stats_smem(const unsigned char* slot, int ctid, int nchunks, float c) {
    typename E::Max mm = E::max_init();
#pragma unroll
    for (int p = 0; p < P; ++p) {
        const int k = p * NTC + ctid;
        if (k < nchunks) mm = E::max_acc(mm, E::lds(slot, k));
    }
    const float m = E::max_fin(mm);
    if (!(m > __uint_as_float(0xFF800000u))) return {m, 0.f};
    const float2 cc = make_float2(c, c);
    const float2 nb = make_float2(-m * c, -m * c);
    float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int p = 0; p < P; ++p) {
        const int k = p * NTC + ctid;
        if (k < nchunks) {
            const typename E::Raw r = E::lds(slot, k);
#pragma unroll
            for (int w = 0; w < 4; ++w) s2 = __fadd2_rn(s2, ex2x2(__ffma2_rn(E::pair(r, w), cc, nb)));
        }
    }
    return {m, s2.x + s2.y};
}

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

// Merge of word pair (wm, ws) over the cluster's records; every lane of the calling warp gets the result.
__device__ __forceinline__ MaxSum merge_ranks(const float* rec8, uint32_t C, int lane, int wm, int ws, float c) {
    MaxSum v{__uint_as_float(0xFF800000u), 0.f};
    if (lane < static_cast<int>(C)) v = {rec8[lane * 8 + wm], rec8[lane * 8 + ws]};
    return warp_ms(v, c);
}

__device__ __forceinline__ float max_ranks(const float* rec8, uint32_t C, int lane, int word) {
    return warp_max(lane < static_cast<int>(C) ? rec8[lane * 8 + word] : __uint_as_float(0xFF800000u));
}

__device__ __forceinline__ int drafter_at(int i, int N, int selected) {
    if (selected < 0) return i;
    return i == N - 1 ? selected : (i < selected ? i : i + 1);
}

// ------------------------------------------------------------------------------------------------
// the persistent row kernel
// ------------------------------------------------------------------------------------------------
template <class E, int P>
__global__ void __launch_bounds__(NT, 2) rows_kernel(const KParams prm) {
    using Raw = typename E::Raw;
    extern __shared__ __align__(128) unsigned char smem[];
    const float NINF = __uint_as_float(0xFF800000u);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t C = cluster_nctarank(), rank = cluster_ctarank();
    const int cid = static_cast<int>(cluster_id_x()), ncl = static_cast<int>(ncluster_x());
    const int nslots = prm.ts + prm.r;
    unsigned char* const slots = smem;
    uint64_t* const full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(nslots) * prm.slot_bytes);
    uint64_t* const empty = full + MAX_SLOTS;
    uint64_t* const xbar = empty + MAX_SLOTS;                           // [2]
    float* const xchg = reinterpret_cast<float*>(xbar + 2);             // [2][C][8]
    float* const scr = xchg + 2 * C * 8;                                // [NWC][4]

    const int slice_start = static_cast<int>(rank) * prm.slice_elems;
    const int n_el = max(0, min(prm.slice_elems, prm.V - slice_start));
    const int nchunks = (n_el + CHUNK - 1) / CHUNK;
    const int ntiles = (nchunks + 31) / 32;
    const float c = prm.c;
    const int K = prm.K, J = prm.J;
    const size_t row_bytes = static_cast<size_t>(prm.V) * E::BYTES;
    const int my_items = cid < prm.num_items ? (prm.num_items - 1 - cid) / ncl + 1 : 0;

    if (tid == 0) {
        for (int s = 0; s < nslots; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NWC);
        }
        mbar_init(&xbar[0], C);
        mbar_init(&xbar[1], C);
        fence_mbarrier_init_cluster();
    }
    __syncthreads();
    cluster_sync_all();   // barriers initialised and every CTA running before any remote access

    if (warp == NWC) {
        // ================================ producer warp ================================
        const uint32_t slice_bytes = static_cast<uint32_t>(n_el) * E::BYTES;
        const size_t off = static_cast<size_t>(slice_start) * E::BYTES;
        const uint64_t policy = prm.tma ? policy_evict_first() : 0ull;
        int g = 0;
        for (int k = 0; k < my_items; ++k) {
            const int w = cid + k * ncl;
            const int b = w / J, j = w % J;
            const int nothers = j < K ? prm.N : 0;
            for (int i = -1; i < nothers; ++i) {
                int s, u;
                const unsigned char* src;
                if (i < 0) {
                    s = k % prm.ts;
                    u = k / prm.ts;
                    src = prm.target + (static_cast<size_t>(b) * (K + 1) + j) * row_bytes + off;
                } else {
                    const int d = drafter_at(i, prm.N, prm.selected);
                    s = prm.ts + g % prm.r;
                    u = g / prm.r;
                    src = prm.others + ((static_cast<size_t>(d) * prm.B + b) * K + j) * row_bytes + off;
                    ++g;
                }
                if (u > 0)
                    mbar_wait_bounded(&empty[s], static_cast<uint32_t>((u - 1) & 1), prm.status, STATUS_TIMEOUT, WAIT_LIMIT_NS);
                unsigned char* dst = slots + static_cast<size_t>(s) * prm.slot_bytes;
                if (prm.tma) {
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&full[s], slice_bytes);
                        if (slice_bytes) bulk_load(dst, src, slice_bytes, &full[s], policy);
                    }
                } else {
                    E::copy_slice(dst, src, n_el, lane);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&full[s]);
                }
            }
        }
    } else {
        // ================================ consumer warps ================================
        const int ctid = tid;   // 0 .. NTC-1
        int g = 0;              // other rows consumed so far
        int e = 0;              // exchanges so far
        // the draft token of an item is loaded one item ahead so that its latency stays hidden
        auto token_of = [&](int kk) {
            if (kk >= my_items || !prm.tokens) return -1;
            const int ww = cid + kk * ncl;
            const int jj = ww % J;
            return jj < K ? __ldg(prm.tokens + static_cast<size_t>(ww / J) * K + jj) : -1;
        };
        int tok_next = token_of(0);
        MaxSum st_t_next{NINF, 0.f};
        for (int k = 0; k < my_items; ++k) {
            const int w = cid + k * ncl;
            const int b = w / J, j = w % J;
            const int nothers = j < K ? prm.N : 0;
            const size_t row = static_cast<size_t>(b) * (K + 1) + j;
            const int ts_slot = k % prm.ts;
            const unsigned char* tslot = slots + static_cast<size_t>(ts_slot) * prm.slot_bytes;
            const int tok = tok_next;
            tok_next = token_of(k + 1);
            int tl = -1;   // the draft token's index within my slice, -1 if elsewhere (or no token)
            if (j < K && prm.tokens) {
                const bool ok = tok >= 0 && tok < prm.V;
                if (!ok && ctid == 0 && rank == 0) atomicOr(prm.status, STATUS_BAD_TOKEN);
                if (ok && tok >= slice_start && tok < slice_start + n_el) tl = tok - slice_start;
            }

            // ---- target row: local statistics (already computed during the previous item's exchange
            // when two target slots let the next target arrive early) ----
            MaxSum st_t;
            if (k > 0 && prm.ts >= 2) {
                st_t = st_t_next;
            } else {
                mbar_wait_bounded(&full[ts_slot], static_cast<uint32_t>((k / prm.ts) & 1), prm.status, STATUS_TIMEOUT,
                                  WAIT_LIMIT_NS);
                st_t = local_stats_smem<E, P>(tslot, ctid, nchunks, c);
            }
            float bt = 0.f, btp = 0.f, ht = 0.f;   // row scalars, identical in every consumer thread
            Raw ro[P];
            for (int i = 0; i < (nothers > 0 ? nothers : 1); ++i) {
                const bool verified = nothers > 0 && prm.selected >= 0 && i == nothers - 1;
                MaxSum st_o{NINF, 0.f};
                float xo = NINF;
                if (nothers > 0) {
                    const int s = prm.ts + g % prm.r;
                    const unsigned char* oslot = slots + static_cast<size_t>(s) * prm.slot_bytes;
                    mbar_wait_bounded(&full[s], static_cast<uint32_t>((g / prm.r) & 1), prm.status, STATUS_TIMEOUT, WAIT_LIMIT_NS);
                    load_raw<E, P>(oslot, ctid, nchunks, ro);
                    if (verified && tl >= 0 && ctid == 0) xo = E::at(oslot, tl);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s]);   // this warp is done with the slot
                    st_o = local_stats<E, P>(ro, c);
                    ++g;
                }
                // CTA-level merge, then one record to every CTA of the cluster
                {
                    const MaxSum a = warp_ms(i == 0 ? st_t : MaxSum{NINF, 0.f}, c);
                    const MaxSum o = warp_ms(st_o, c);
                    if (lane == 0) {
                        scr[warp * 4 + 0] = a.m;
                        scr[warp * 4 + 1] = a.s;
                        scr[warp * 4 + 2] = o.m;
                        scr[warp * 4 + 3] = o.s;
                    }
                }
                named_sync(1, NTC);
                const int xp = e & 1;
                if (warp == 0) {
                    MaxSum a{NINF, 0.f}, o{NINF, 0.f};
                    if (lane < NWC) {
                        a = {scr[lane * 4 + 0], scr[lane * 4 + 1]};
                        o = {scr[lane * 4 + 2], scr[lane * 4 + 3]};
                    }
                    a = warp_ms(a, c);
                    o = warp_ms(o, c);
                    const float xt = (i == 0 && tl >= 0) ? E::at(tslot, tl) : NINF;
                    const float xo0 = __shfl_sync(0xffffffffu, xo, 0);
                    if (lane < static_cast<int>(C)) {
                        const uint32_t local = smem_addr(xchg + (xp * C + rank) * 8);
                        const uint32_t remote = map_to_rank(local, static_cast<uint32_t>(lane));
                        st_cluster_f32x4(remote, a.m, a.s, o.m, o.s);
                        st_cluster_f32x4(remote + 16, xt, xo0, 0.f, 0.f);
                        mbar_arrive_remote(map_to_rank(smem_addr(&xbar[xp]), static_cast<uint32_t>(lane)));
                    }
                }
                // while the records travel: statistics of the next item's target, if its slot is separate
                if (i == 0 && prm.ts >= 2 && k + 1 < my_items) {
                    const int ns = (k + 1) % prm.ts;
                    mbar_wait_bounded(&full[ns], static_cast<uint32_t>(((k + 1) / prm.ts) & 1), prm.status,
                                      STATUS_TIMEOUT, WAIT_LIMIT_NS);
                    st_t_next = local_stats_smem<E, P>(slots + static_cast<size_t>(ns) * prm.slot_bytes, ctid, nchunks, c);
                }
                // only warp 0 polls for the cluster's records; the others park in the named barrier
                if (warp == 0)
                    mbar_wait_bounded<true>(&xbar[xp], static_cast<uint32_t>((e >> 1) & 1), prm.status, STATUS_TIMEOUT,
                                            WAIT_LIMIT_NS);
                named_sync(2, NTC);
                ++e;
                // every warp merges the cluster's records itself (no broadcast round trip)
                const float* r8 = xchg + xp * C * 8;
                const MaxSum go = merge_ranks(r8, C, lane, 2, 3, c);
                const float bo = beta_of(go, c);
                if (i == 0) {
                    const MaxSum gt = merge_ranks(r8, C, lane, 0, 1, c);
                    const float xt = max_ranks(r8, C, lane, 4);
                    btp = beta_of(gt, c);
                    bt = btp;
                    ht = prob_of(xt, gt, c);
                    if (prm.cactus && j < K) {
                        float log2s;
                        cactus_scalars(ht, prm.delta, ht, log2s);
                        bt = btp + log2s;
                    }
                }
                const float pd = verified ? prob_of(max_ranks(r8, C, lane, 5), go, c) : 0.f;
                if (rank == 0 && ctid == 0 && prm.rec) {
                    float* rp = prm.rec + row * REC;
                    if (i == 0) {
                        rp[R_HT] = ht;
                        rp[R_BT] = bt;
                        rp[R_BTP] = btp;
                        if (nothers == 0) {
                            rp[R_PD] = 0.f;
                            rp[R_BO] = 0.f;
                        }
                    }
                    if (verified) {
                        rp[R_PD] = pd;
                        rp[R_BO] = bo;
                    }
                }
                if (nothers == 0) break;

                // ---- phase B: overlap with the target; residual tiles of the verified drafter ----
                const float2 cc = make_float2(c, c), bt2 = make_float2(bt, bt), bo2 = make_float2(bo, bo);
                float2 ovl2 = make_float2(0.f, 0.f);
                if (!verified) {
#pragma unroll
                    for (int p = 0; p < P; ++p) {
                        const int kc = p * NTC + ctid;
                        if (kc < nchunks) ovl2 = chunk_overlap<E>(E::lds(tslot, kc), ro[p], cc, bt2, bo2, ovl2);
                    }
                } else {
                    const int etc = tl >= 0 ? tl / CHUNK : -1;
#pragma unroll
                    for (int p = 0; p < P; ++p) {
                        const int kc = p * NTC + ctid;
                        float mass = 0.f;
                        if (kc < nchunks) {
                            const Raw rt = E::lds(tslot, kc);
                            mass = (kc == etc) ? chunk_mass_patched<E>(1, rt, ro[p], c, bt, bo, tl % CHUNK, ht, ovl2)
                                               : chunk_mass<E>(1, rt, ro[p], cc, bt2, bo2, ovl2);
                        }
                        const float incl = warp_incl_scan(mass, lane);
                        const int tau = p * NWC + warp;
                        if (lane == 31 && tau < ntiles && prm.tiles)
                            prm.tiles[(row * C + rank) * prm.tiles_cap + tau] = incl;
                    }
                }
                if (prm.gpart) {
                    const float s = warp_sum(ovl2.x + ovl2.y);
                    const int d = drafter_at(i, prm.N, prm.selected);
                    if (lane == 0)
                        prm.gpart[((((static_cast<size_t>(d) * prm.B + b) * K + j) * C) + rank) * NWC + warp] = s;
                }
            }
            if (nothers == 0) {
                // ---- bonus row: target mass per tile ----
                const float2 cc = make_float2(c, c), bt2 = make_float2(btp, btp);
                float2 unused = make_float2(0.f, 0.f);
#pragma unroll
                for (int p = 0; p < P; ++p) {
                    const int kc = p * NTC + ctid;
                    float mass = 0.f;
                    if (kc < nchunks) {
                        const Raw rt = E::lds(tslot, kc);
                        mass = chunk_mass<E>(2, rt, rt, cc, bt2, bt2, unused);
                    }
                    const float incl = warp_incl_scan(mass, lane);
                    const int tau = p * NWC + warp;
                    if (lane == 31 && tau < ntiles && prm.tiles) prm.tiles[(row * C + rank) * prm.tiles_cap + tau] = incl;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[ts_slot]);   // this warp is done with the target slot
        }
    }
    // no CTA may leave while a peer can still write into its shared memory
    cluster_sync_all();
}

// ------------------------------------------------------------------------------------------------
// gamma partial reduction: one warp per (drafter, sequence, level)
// ------------------------------------------------------------------------------------------------
struct GParams {
    const float* gpart;   // [N*B*K, C, NWC]
    int n_out, C;
    float* gamma;
    float* loss;
};

__global__ void __launch_bounds__(256) gamma_reduce_kernel(const GParams g) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int o = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (o >= g.n_out) return;
    const int n = g.C * NWC;
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
    const float* tiles;          // [B, K+1, C, tiles_cap]
    const unsigned char* target; // [B, K+1, V]
    const unsigned char* other;  // verified drafter rows: row (b, j) starts at element (b * K + j) * V
    const int32_t* tokens;       // [B, K]
    const uint64_t* seeds;       // [B]
    int B, K, V, C, slice_elems, tiles_cap, aligned;
    float c;
    int32_t* accept_len;         // [B]
    int32_t* out_tokens;         // [B, K+1]
    float* diag;                 // [B, K, 4] or null
    float* gamma_star;           // [B, K] or null (Cactus)
};

__device__ __forceinline__ int fp_slice_tiles(const FParams& f, int r) {
    const int n = max(0, min(f.slice_elems, f.V - r * f.slice_elems));
    return ((n + CHUNK - 1) / CHUNK + 31) / 32;
}

// tile `flat` of the row in vocabulary order (slice-major)
__device__ __forceinline__ float fp_tile(const FParams& f, size_t row, int flat) {
    int r = 0;
    while (flat >= fp_slice_tiles(f, r)) {
        flat -= fp_slice_tiles(f, r);
        ++r;
    }
    return f.tiles[(row * f.C + r) * f.tiles_cap + flat];
}

// Draw from h over a whole target row in vocabulary order (slow path; only after a reject whose residual
// mass rounded to zero). Returns the token.
template <class E>
__device__ int draw_whole_row(const FParams& f, const unsigned char* trow, float bt, int tok, float ht, float u, int lane) {
    using Raw = typename E::Raw;
    float all = 0.f;
    for (int e0 = lane * CHUNK; e0 < f.V; e0 += 32 * CHUNK) {
        const Raw rt = E::gchunk(trow, e0, f.V, f.aligned);
        float2 unused = make_float2(0.f, 0.f);
        const int et = (tok >= e0 && tok < e0 + CHUNK) ? tok - e0 : -1;
        all += chunk_mass_patched<E>(2, rt, rt, f.c, bt, 0.f, et, ht, unused);
    }
    const float tp = u * warp_sum(all);
    float before = 0.f;
    int last_pos = -1;
    for (int base = 0; base < f.V; base += 32 * CHUNK) {
        const int e0 = base + lane * CHUNK;
        const Raw rt = E::gchunk(trow, e0, f.V, f.aligned);
        const int et = (tok >= e0 && tok < e0 + CHUNK) ? tok - e0 : -1;
        float v[8], ovl = 0.f;
        chunk_values<E>(2, rt, rt, f.c, bt, 0.f, et, ht, v, ovl);
        float m = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) m += v[q];
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

template <class E>
__global__ void __launch_bounds__(256) finish_kernel(const FParams f) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    using Raw = typename E::Raw;
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (b >= f.B) return;
    const int K = f.K;
    const uint64_t seed = f.seeds[b];
    const size_t row_bytes = static_cast<size_t>(f.V) * E::BYTES;
    int total_tiles = 0;
    for (int r = 0; r < f.C; ++r) total_tiles += fp_slice_tiles(f, r);

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
    // inclusive prefix of the tile masses in vocabulary order; every lane owns a contiguous run
    const int seg = (total_tiles + 31) / 32;
    const int lo = lane * seg, hi = min(total_tiles, lo + seg);
    float local = 0.f;
    for (int t = lo; t < hi; ++t) local += fp_tile(f, row, t);
    const float incl = warp_incl_scan(local, lane);
    float excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl = 0.f;
    const int last_lane = total_tiles > 0 ? (total_tiles - 1) / seg : 0;
    const float Z = __shfl_sync(0xffffffffu, excl + local, last_lane);
    int emitted;
    if (mode == 1 && !(Z > 0.f)) {
        emitted = draw_whole_row<E>(f, f.target + row * row_bytes, bt, tok, ht, u, lane);
    } else {
        const float tp = u * Z;
        // first tile whose prefix exceeds tp (else the last tile with mass)
        int found = -1, lastp = -1;
        float before_found = 0.f, before_last = 0.f;
        float run = excl;
        for (int t = lo; t < hi; ++t) {
            const float m = fp_tile(f, row, t);
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
        float before_tile;
        if (hit) {
            const int ln = __ffs(hit) - 1;
            ft = __shfl_sync(0xffffffffu, found, ln);
            before_tile = __shfl_sync(0xffffffffu, before_found, ln);
        } else {
            const unsigned any = __ballot_sync(0xffffffffu, lastp >= 0);
            const int ln = any ? 31 - __clz(any) : 0;
            ft = __shfl_sync(0xffffffffu, lastp, ln);
            before_tile = __shfl_sync(0xffffffffu, before_last, ln);
        }
        // slice and tile within it; the tile's warp layout in the row pass: pass ft / NWC, warp ft % NWC
        int r = 0, tloc = ft < 0 ? 0 : ft;
        while (tloc >= fp_slice_tiles(f, r) && r < f.C - 1) {
            tloc -= fp_slice_tiles(f, r);
            ++r;
        }
        const int slice_start = r * f.slice_elems;
        const int n_el = max(0, min(f.slice_elems, f.V - slice_start));
        const int nchunks = (n_el + CHUNK - 1) / CHUNK;
        const int kc = (tloc / NWC) * NTC + (tloc % NWC) * 32 + lane;
        const int e0 = kc * CHUNK;
        const unsigned char* trow = f.target + row * row_bytes + static_cast<size_t>(slice_start) * E::BYTES;
        const unsigned char* orow = mode == 1 ? f.other + (static_cast<size_t>(b) * K + L) * row_bytes +
                                                    static_cast<size_t>(slice_start) * E::BYTES
                                              : trow;
        float v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = 0.f;
        float mass = 0.f;
        if (ft >= 0 && kc < nchunks) {
            const Raw rt = E::gchunk(trow, e0, n_el, f.aligned);
            const Raw ro = E::gchunk(orow, e0, n_el, f.aligned);
            const int et = (mode == 1 && tok >= slice_start + e0 && tok < slice_start + e0 + CHUNK)
                               ? tok - slice_start - e0 : -1;
            float2 o2 = make_float2(0.f, 0.f);
            mass = chunk_mass_patched<E>(mode, rt, ro, f.c, bt, bo, et, ht, o2);
            float ovl = 0.f;
            chunk_values<E>(mode, rt, ro, f.c, bt, bo, et, ht, v, ovl);
        }
        const float in2 = warp_incl_scan(mass, lane);
        float ex2v = __shfl_up_sync(0xffffffffu, in2, 1);
        if (lane == 0) ex2v = 0.f;
        const unsigned over = __ballot_sync(0xffffffffu, mass > 0.f && before_tile + in2 > tp);
        const unsigned posm = __ballot_sync(0xffffffffu, mass > 0.f);
        const int ln = over ? __ffs(over) - 1 : (posm ? 31 - __clz(posm) : -1);
        int pick = -1;
        if (lane == ln) {
            float a = before_tile + ex2v;
            int lp = -1;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                a += v[q];
                if (v[q] > 0.f) {
                    lp = q;
                    if (pick < 0 && a > tp) pick = q;
                }
            }
            pick = slice_start + e0 + (pick >= 0 ? pick : lp);
        }
        emitted = ln >= 0 ? __shfl_sync(0xffffffffu, pick, ln) : -1;
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
            for (int t = lane; t < total_tiles; t += 32) zs += fp_tile(f, rj, t);
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
