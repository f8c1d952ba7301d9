// Verification kernels for sm_103a.
//
// One persistent grid of thread-block clusters. Each cluster of C CTAs works on one "item" at a time:
// the target row (b, j) plus the other rows verified against it (the draft row for standard and
// Cactus verification; all N drafter rows for the counterfactual evaluation; none for the bonus row
// j = K). CTA `rank` owns the vocabulary slice [rank * slice, (rank + 1) * slice) of every row of the
// item. Rows are staged into shared memory by bulk (TMA) copies; the logits are read from HBM exactly
// once. The softmax normalisers of every row are combined across the cluster through distributed shared
// memory, so every CTA knows each row's global (max, sum) and evaluates, for its own slice:
//   - sum_x min(p_target, p_other)                 (acceptance probability = 1 - TV, HedgeSpec gamma)
//   - sum_x (h - p_draft)+ per 256-token tile       (residual mass, h = p_target or the Cactus h)
//   - or sum_x p_target per tile                    (bonus row)
// and the slice that holds the inverse-CDF point of the residual (or bonus) draw finds the token from
// its shared-memory copy. The per-position records (h(t), p_draft(t), Z, overlap, token) go to the
// workspace; a small second kernel turns them into the accept/reject chain.
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

constexpr int NT = 512;                 // threads per CTA
constexpr int NWARPS = NT / 32;
constexpr int CHUNK = 8;                // elements per thread per pass (16 B of bf16)
constexpr int TILE = CHUNK * 32;        // elements per warp per pass: the residual tile
constexpr int SLICE_Q = 128;            // granularity of the per-CTA vocabulary slice
constexpr int REC = 8;                  // 32-bit words per position record
constexpr int MAX_SLOTS = 4;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;   // bounded wait for a bulk copy
constexpr unsigned STATUS_BAD_TOKEN = 1u;
constexpr unsigned STATUS_TIMEOUT = 2u;

// record words
constexpr int R_HT = 0;      // h(t): p_target(t), or gamma* for Cactus
constexpr int R_PD = 1;      // p_draft(t)
constexpr int R_Z = 2;       // residual mass Z
constexpr int R_OVL = 3;     // sum min(p_target, p_draft)
constexpr int R_TOK = 4;     // resample token (j < K) or bonus token (j = K), int bits

struct KParams {
    const unsigned char* target;   // [B, K+1, V]
    const unsigned char* others;   // [N, B, K, V]
    const int32_t* tokens;         // [B, K] (null: gamma only)
    const uint64_t* seeds;         // [B]    (null: gamma only)
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
    int tiles_cap;                 // >= ceil(slice_elems / TILE), multiple of 4
    float* gamma;                  // [N, B, K] or null
    float* loss;                   // [N, B, K] or null
    float* rec;                    // [B, K+1, REC] or null
    unsigned* status;
};

// ------------------------------------------------------------------------------------------------
// element formats
// ------------------------------------------------------------------------------------------------
struct Bf16 {
    using Raw = uint4;                                   // 8 packed bf16
    static constexpr int BYTES = 2;
    __device__ static Raw ninf() { return make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u); }
    __device__ static Raw lds(const unsigned char* slot, int k) {
        return reinterpret_cast<const uint4*>(slot)[k];
    }
    __device__ static void cvt(const Raw& r, float (&x)[8]) {
        x[0] = __uint_as_float(r.x << 16);
        x[1] = __uint_as_float(r.x & 0xFFFF0000u);
        x[2] = __uint_as_float(r.y << 16);
        x[3] = __uint_as_float(r.y & 0xFFFF0000u);
        x[4] = __uint_as_float(r.z << 16);
        x[5] = __uint_as_float(r.z & 0xFFFF0000u);
        x[6] = __uint_as_float(r.w << 16);
        x[7] = __uint_as_float(r.w & 0xFFFF0000u);
    }
    __device__ static float at(const unsigned char* slot, int e) {
        return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(slot)[e]) << 16);
    }
    // element-wise copy for rows that are not 16-byte aligned (pads the last chunk with -inf)
    __device__ static void copy_slice(unsigned char* slot, const unsigned char* src, int n_el, int tid) {
        const uint16_t* s = reinterpret_cast<const uint16_t*>(src);
        uint16_t* d = reinterpret_cast<uint16_t*>(slot);
        const int padded = (n_el + CHUNK - 1) / CHUNK * CHUNK;
        for (int e = tid; e < padded; e += NT) d[e] = e < n_el ? __ldg(s + e) : static_cast<uint16_t>(0xFF80u);
    }
};

struct F32 {
    struct Raw {
        float4 a, b;
    };
    static constexpr int BYTES = 4;
    __device__ static Raw ninf() {
        const float n = __uint_as_float(0xFF800000u);
        return {make_float4(n, n, n, n), make_float4(n, n, n, n)};
    }
    __device__ static Raw lds(const unsigned char* slot, int k) {
        const float4* p = reinterpret_cast<const float4*>(slot) + 2 * k;
        return {p[0], p[1]};
    }
    __device__ static void cvt(const Raw& r, float (&x)[8]) {
        x[0] = r.a.x; x[1] = r.a.y; x[2] = r.a.z; x[3] = r.a.w;
        x[4] = r.b.x; x[5] = r.b.y; x[6] = r.b.z; x[7] = r.b.w;
    }
    __device__ static float at(const unsigned char* slot, int e) { return reinterpret_cast<const float*>(slot)[e]; }
    __device__ static void copy_slice(unsigned char* slot, const unsigned char* src, int n_el, int tid) {
        const uint32_t* s = reinterpret_cast<const uint32_t*>(src);
        uint32_t* d = reinterpret_cast<uint32_t*>(slot);
        const int padded = (n_el + CHUNK - 1) / CHUNK * CHUNK;
        for (int e = tid; e < padded; e += NT) d[e] = e < n_el ? __ldg(s + e) : 0xFF800000u;
    }
};

// ------------------------------------------------------------------------------------------------
// per-CTA state shared by the helpers
// ------------------------------------------------------------------------------------------------
struct Cta {
    int tid, lane, warp;
    uint32_t C, rank;
    int slice_start, n_el, nchunks, ntiles;
    unsigned char* slots;
    uint64_t* bars;
    float* xchg;     // [2][C][8]
    float* tiles;    // [tiles_cap]
    float* scr;      // [NWARPS * 4]
    int* bci;        // [8]
    float* bcf;      // [8]
};

// Thread-local (max, sum 2^((x - max) c)) over this thread's chunks of a slice held in registers.
template <class E, int P>
__device__ __forceinline__ MaxSum local_stats(const typename E::Raw (&raw)[P], float c) {
    float m = __uint_as_float(0xFF800000u);
#pragma unroll
    for (int p = 0; p < P; ++p) {
        float x[8];
        E::cvt(raw[p], x);
#pragma unroll
        for (int e = 0; e < 8; ++e) m = fmaxf(m, x[e]);
    }
    float s = 0.f;
    if (m != __uint_as_float(0xFF800000u)) {
        const float mc = m * c;
#pragma unroll
        for (int p = 0; p < P; ++p) {
            float x[8];
            E::cvt(raw[p], x);
#pragma unroll
            for (int e = 0; e < 8; ++e) s += ex2(fmaf(x[e], c, -mc));
        }
    }
    return {m, s};
}

template <class E, int P>
__device__ __forceinline__ void load_raw(const Cta& t, const unsigned char* slot, typename E::Raw (&raw)[P]) {
#pragma unroll
    for (int p = 0; p < P; ++p) {
        const int k = p * NT + t.tid;
        raw[p] = k < t.nchunks ? E::lds(slot, k) : E::ninf();
    }
}

// Values of one chunk in phase B, with h(x) = 2^(x_t c + bt) and p_other(x) = 2^(x_o c + bo).
// mode 0: overlap only, sum 2^min(log2 h, log2 p_other); mode 1: residual (h - p_other)+ and overlap
// sum min(h, p_other); mode 2: mass of h itself. `et` >= 0 patches element et of h to `hpatch`
// (Cactus h_n = gamma*). If vals != nullptr the per-element masses are stored (for the draw).
template <class E>
__device__ __forceinline__ void chunk_eval(int mode, const typename E::Raw& rt, const typename E::Raw& ro,
                                           float c, float bt, float bo, int et, float hpatch, float& ovl,
                                           float& mass, float* vals) {
    float xt[8], xo[8];
    E::cvt(rt, xt);
    ovl = 0.f;
    mass = 0.f;
    if (mode == 0) {
        E::cvt(ro, xo);
#pragma unroll
        for (int e = 0; e < 8; ++e) ovl += ex2(fminf(fmaf(xt[e], c, bt), fmaf(xo[e], c, bo)));
    } else if (mode == 1) {
        E::cvt(ro, xo);
        if (et < 0) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float ph = ex2(fmaf(xt[e], c, bt));
                const float po = ex2(fmaf(xo[e], c, bo));
                const float mn = fminf(ph, po);
                const float res = ph - mn;
                ovl += mn;
                mass += res;
                if (vals) vals[e] = res;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float ph = ex2(fmaf(xt[e], c, bt));
                if (e == et) ph = hpatch;
                const float po = ex2(fmaf(xo[e], c, bo));
                const float mn = fminf(ph, po);
                const float res = ph - mn;
                ovl += mn;
                mass += res;
                if (vals) vals[e] = res;
            }
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float ph = ex2(fmaf(xt[e], c, bt));
            if (e == et) ph = hpatch;
            mass += ph;
            if (vals) vals[e] = ph;
        }
    }
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

// Sum over the CTA; the result is valid in every lane of warp 0. Uses scr[0..NWARPS); ends with the
// CTA synchronised so scr may be reused after the next __syncthreads.
__device__ __forceinline__ float cta_sum_warp0(const Cta& t, float v) {
    v = warp_sum(v);
    if (t.lane == 0) t.scr[t.warp] = v;
    __syncthreads();
    float r = 0.f;
    if (t.warp == 0) {
        r = t.lane < NWARPS ? t.scr[t.lane] : 0.f;
        r = warp_sum(r);
    }
    return r;
}

// Turns tiles[0..ntiles) (per-tile masses) into inclusive prefix sums; warp 0 only. Returns the slice
// total (the last prefix) in all lanes of warp 0.
__device__ __forceinline__ float tiles_to_prefix(const Cta& t) {
    const int nt = t.ntiles;
    const int seg = (nt + 31) / 32;
    const int lo = t.lane * seg, hi = min(nt, lo + seg);
    float local = 0.f;
    for (int i = lo; i < hi; ++i) {
        local += t.tiles[i];
        t.tiles[i] = local;
    }
    const float incl = warp_incl_scan(local, t.lane);
    float excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (t.lane == 0) excl = 0.f;
    for (int i = lo; i < hi; ++i) t.tiles[i] = excl + t.tiles[i];
    __syncwarp();
    return nt > 0 ? t.tiles[nt - 1] : 0.f;
}

// Pushes this CTA's 8-float record to slot [par][rank] of every CTA in the cluster (lanes 0..C-1 of
// warp 0 each serve one destination), then synchronises the whole cluster.
__device__ __forceinline__ void exchange(const Cta& t, int par, const float (&v)[8]) {
    if (t.warp == 0 && t.lane < static_cast<int>(t.C)) {
        const uint32_t local = smem_addr(t.xchg + (par * t.C + t.rank) * 8);
        const uint32_t remote = map_to_rank(local, static_cast<uint32_t>(t.lane));
        st_cluster_f32x4(remote, v[0], v[1], v[2], v[3]);
        st_cluster_f32x4(remote + 16, v[4], v[5], v[6], v[7]);
    }
    cluster_sync_all();
}

__device__ __forceinline__ float xget(const Cta& t, int par, int r, int w) { return t.xchg[(par * t.C + r) * 8 + w]; }

// Global (max, sum) of word pair (wm, ws) over the cluster, merged in rank order.
__device__ __forceinline__ MaxSum xmerge(const Cta& t, int par, int wm, int ws, float c) {
    MaxSum acc{__uint_as_float(0xFF800000u), 0.f};
    for (uint32_t r = 0; r < t.C; ++r) acc = ms_merge(acc, MaxSum{xget(t, par, r, wm), xget(t, par, r, ws)}, c);
    return acc;
}

// log2 p(x) = x c + beta with beta = -(M c + log2 S).
__device__ __forceinline__ float beta_of(MaxSum g, float c) { return -fmaf(g.m, c, log2f(g.s)); }

// p(x) for one logit with the row's global (M, S): 2^((x - M) c - log2 S).
__device__ __forceinline__ float prob_of(float x, MaxSum g, float c) {
    if (!(x > __uint_as_float(0xFF800000u))) return 0.f;
    return ex2(fmaf(x - g.m, c, -log2f(g.s)));
}

// ------------------------------------------------------------------------------------------------
// the persistent verification kernel
// ------------------------------------------------------------------------------------------------
// Writes tiles[p * NWARPS + warp] = mass of the warp's 256-token tile of pass p (Hillis-Steele scan
// over the 32 chunk masses; the draw repeats the same scan, so the numbers agree bit for bit).
template <class E, int P>
__device__ __forceinline__ float phase_b(const Cta& t, int mode, const unsigned char* tslot,
                                         const typename E::Raw (&ro)[P], float c, float bt, float bo,
                                         int et_chunk, int et_elem, float hpatch) {
    float ovl_acc = 0.f;
#pragma unroll
    for (int p = 0; p < P; ++p) {
        const int kc = p * NT + t.tid;
        float ovl = 0.f, mass = 0.f;
        if (kc < t.nchunks) {
            const typename E::Raw rt = E::lds(tslot, kc);
            chunk_eval<E>(mode, rt, ro[p], c, bt, bo, kc == et_chunk ? et_elem : -1, hpatch, ovl, mass, nullptr);
        }
        ovl_acc += ovl;
        if (mode != 0) {
            const float incl = warp_incl_scan(mass, t.lane);
            if (t.lane == 31 && p * NWARPS + t.warp < t.ntiles) t.tiles[p * NWARPS + t.warp] = incl;
        }
    }
    return ovl_acc;
}

template <class E, int P>
__global__ void __launch_bounds__(NT, 2) rows_kernel(const KParams prm) {
    using Raw = typename E::Raw;
    extern __shared__ __align__(128) unsigned char smem[];
    const float NINF = __uint_as_float(0xFF800000u);
    Cta t;
    t.tid = threadIdx.x;
    t.lane = t.tid & 31;
    t.warp = t.tid >> 5;
    t.C = cluster_nctarank();
    t.rank = cluster_ctarank();
    const uint32_t cid = cluster_id_x(), ncl = ncluster_x();
    const int nslots = prm.ts + prm.r;
    t.slots = smem;
    t.bars = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(nslots) * prm.slot_bytes);
    t.xchg = reinterpret_cast<float*>(t.bars + MAX_SLOTS);
    t.tiles = t.xchg + 2 * t.C * 8;
    t.scr = t.tiles + prm.tiles_cap;
    t.bci = reinterpret_cast<int*>(t.scr + NWARPS * 4);
    t.bcf = reinterpret_cast<float*>(t.bci + 8);
    t.slice_start = static_cast<int>(t.rank) * prm.slice_elems;
    t.n_el = max(0, min(prm.slice_elems, prm.V - t.slice_start));
    t.nchunks = (t.n_el + CHUNK - 1) / CHUNK;
    t.ntiles = (t.nchunks + 31) / 32;
    const uint32_t slice_bytes = static_cast<uint32_t>(t.n_el) * E::BYTES;
    const size_t row_bytes = static_cast<size_t>(prm.V) * E::BYTES;
    const float c = prm.c;
    const int K = prm.K, J = prm.J;
    const int my_items = cid < static_cast<uint32_t>(prm.num_items)
                             ? (prm.num_items - 1 - static_cast<int>(cid)) / static_cast<int>(ncl) + 1
                             : 0;
    uint64_t policy = 0;
    if (prm.tma) policy = policy_evict_first();

    if (t.tid == 0)
        for (int s = 0; s < nslots; ++s) mbar_init(&t.bars[s], 1);
    __syncthreads();
    cluster_sync_all();   // every CTA of the cluster is running before any remote store

    auto slot_ptr = [&](int s) { return t.slots + static_cast<size_t>(s) * prm.slot_bytes; };
    auto item_of = [&](int k) { return static_cast<int>(cid) + k * static_cast<int>(ncl); };
    auto others_of = [&](int w) { return (w % J) < K ? prm.N : 0; };
    // drafter index of the i-th other row of an item: the verified (selected) drafter goes last
    auto drafter_of = [&](int i) {
        if (prm.selected < 0) return i;
        if (i == prm.N - 1) return prm.selected;
        return i < prm.selected ? i : i + 1;
    };
    auto target_src = [&](int w) {
        const int b = w / J, j = w % J;
        return prm.target + (static_cast<size_t>(b) * (K + 1) + j) * row_bytes +
               static_cast<size_t>(t.slice_start) * E::BYTES;
    };
    auto other_src = [&](int w, int i) {
        const int b = w / J, j = w % J;
        const int d = drafter_of(i);
        return prm.others + ((static_cast<size_t>(d) * prm.B + b) * K + j) * row_bytes +
               static_cast<size_t>(t.slice_start) * E::BYTES;
    };

    // ---------------- producer: thread 0 issues bulk copies as slots free up ----------------
    int tgt_issued = 0, oth_issued = 0, oth_item = 0, oth_idx = 0;
    auto issue = [&](int items_done, int oth_released) {
        if (!prm.tma || t.tid != 0) return;
        while (tgt_issued < my_items && tgt_issued < items_done + prm.ts) {
            const int s = tgt_issued % prm.ts;
            mbar_arrive_expect_tx(&t.bars[s], slice_bytes);
            if (slice_bytes) bulk_load(slot_ptr(s), target_src(item_of(tgt_issued)), slice_bytes, &t.bars[s], policy);
            ++tgt_issued;
        }
        while (oth_issued < oth_released + prm.r) {
            while (oth_item < my_items && oth_idx >= others_of(item_of(oth_item))) {
                ++oth_item;
                oth_idx = 0;
            }
            if (oth_item >= my_items) break;
            const int s = prm.ts + oth_issued % prm.r;
            mbar_arrive_expect_tx(&t.bars[s], slice_bytes);
            if (slice_bytes)
                bulk_load(slot_ptr(s), other_src(item_of(oth_item), oth_idx), slice_bytes, &t.bars[s], policy);
            ++oth_idx;
            ++oth_issued;
        }
    };
    // consumer side: wait for a slot's bulk copy, or copy synchronously when rows are unaligned
    auto acquire = [&](int s, int use, const unsigned char* src) {
        if (prm.tma) {
            mbar_wait_bounded(&t.bars[s], static_cast<uint32_t>(use & 1), prm.status, STATUS_TIMEOUT, WAIT_LIMIT_NS);
        } else {
            E::copy_slice(slot_ptr(s), src, t.n_el, t.tid);
            __syncthreads();
        }
    };

    issue(0, 0);
    int oth_released = 0;   // other rows whose ring slot has been handed back to the producer
    int xpar = 0;           // parity of the next exchange buffer

    for (int k = 0; k < my_items; ++k) {
        const int w = item_of(k);
        const int b = w / J, j = w % J;
        const int nothers = others_of(w);
        const int ts_slot = k % prm.ts;
        const unsigned char* tslot = slot_ptr(ts_slot);
        int tok = -1;
        bool tok_ok = false;
        if (j < K && prm.tokens) {
            tok = prm.tokens[static_cast<size_t>(b) * K + j];
            tok_ok = tok >= 0 && tok < prm.V;
            if (!tok_ok && t.tid == 0 && t.rank == 0) atomicOr(prm.status, STATUS_BAD_TOKEN);
        }
        const int tl = tok_ok ? tok - t.slice_start : -1;   // the draft token's index in my slice
        const bool own_tok = tok_ok && tl >= 0 && tl < t.n_el;

        // ---- phase A: local (max, sum) of the target row and of the first other row ----
        acquire(ts_slot, k / prm.ts, target_src(w));
        MaxSum st_t;
        {
            Raw rt[P];
            load_raw<E, P>(t, tslot, rt);
            st_t = local_stats<E, P>(rt, c);
        }
        Raw ro[P];
        MaxSum st_o{NINF, 0.f};
        float xo_tok = NINF;   // thread 0: logit of the verified drafter at the token, if in my slice
        const int g0 = oth_released;
        auto take_other = [&](int i) {
            const int g = g0 + i;
            const int s = prm.ts + g % prm.r;
            acquire(s, g / prm.r, other_src(w, i));
            load_raw<E, P>(t, slot_ptr(s), ro);
            st_o = local_stats<E, P>(ro, c);
        };
        // after the CTA barrier that follows phase A of other row i: read the token logit (thread 0),
        // then hand the slot back and let the producer refill it
        auto release_other = [&](int i) {
            const int g = g0 + i;
            if (t.tid == 0 && own_tok && i == nothers - 1 && prm.selected >= 0)
                xo_tok = E::at(slot_ptr(prm.ts + g % prm.r), tl);
            ++oth_released;
            issue(k, oth_released);
        };
        if (nothers > 0) take_other(0);
        {
            const MaxSum a = warp_ms(st_t, c), o = warp_ms(st_o, c);
            if (t.lane == 0) {
                t.scr[t.warp * 4 + 0] = a.m;
                t.scr[t.warp * 4 + 1] = a.s;
                t.scr[t.warp * 4 + 2] = o.m;
                t.scr[t.warp * 4 + 3] = o.s;
            }
        }
        __syncthreads();
        if (nothers > 0) release_other(0);
        float v[8];
        if (t.warp == 0) {
            MaxSum a2{NINF, 0.f}, o2{NINF, 0.f};
            if (t.lane < NWARPS) {
                a2 = {t.scr[t.lane * 4 + 0], t.scr[t.lane * 4 + 1]};
                o2 = {t.scr[t.lane * 4 + 2], t.scr[t.lane * 4 + 3]};
            }
            a2 = warp_ms(a2, c);
            o2 = warp_ms(o2, c);
            const float xt_tok = own_tok ? E::at(tslot, tl) : NINF;
            v[0] = a2.m; v[1] = a2.s; v[2] = o2.m; v[3] = o2.s;
            v[4] = xt_tok;
            v[5] = __shfl_sync(0xffffffffu, xo_tok, 0);
            v[6] = 0.f; v[7] = 0.f;
        }
        exchange(t, xpar, v);
        const MaxSum gt = xmerge(t, xpar, 0, 1, c);
        MaxSum go = xmerge(t, xpar, 2, 3, c);
        float x_t_tok = NINF, x_o_tok = NINF;
        for (uint32_t r = 0; r < t.C; ++r) {
            x_t_tok = fmaxf(x_t_tok, xget(t, xpar, r, 4));
            x_o_tok = fmaxf(x_o_tok, xget(t, xpar, r, 5));
        }
        xpar ^= 1;
        const float bt_plain = beta_of(gt, c);
        float bt = bt_plain;            // log2 h(x) = x c + bt for x != t
        const float pt_tok = prob_of(x_t_tok, gt, c);
        float h_tok = pt_tok;           // h(t): p_target(t), or gamma* (Cactus)
        // h(t) enters the residual as the same float in both variants (p_target(t) for standard
        // verification, gamma* for Cactus), so delta = 0 reproduces standard verification bit for bit.
        int et_chunk = -1, et_elem = -1;
        if (own_tok) {
            et_chunk = tl / CHUNK;
            et_elem = tl % CHUNK;
        }
        if (prm.cactus && j < K) {
            // Cactus: gamma* = min(q + sqrt(2 delta q (1 - q)), 1) with q = p_target(t);
            // h(t) = gamma*, h(x) = (1 - gamma*) / (1 - q) p_target(x) elsewhere.
            float gs = pt_tok + sqrtf(2.f * prm.delta * pt_tok * (1.f - pt_tok));
            gs = fminf(gs, 1.f);
            const float s = pt_tok < 1.f ? __fdiv_rn(1.f - gs, 1.f - pt_tok) : 0.f;
            bt = bt_plain + log2f(s);
            h_tok = gs;
        }

        // ---- phase B over the other rows; exchange i carries stats(i) and the overlap of row i-1 ----
        float pend_ovl = 0.f;   // warp 0: CTA overlap of the previous other row, sent with the next exchange
        int pend_d = -1;
        float slice_total = 0.f;    // warp 0: this slice's mass for the draw
        auto write_gamma = [&](int par, int d) {
            if (t.tid == 0 && t.rank == 0 && prm.gamma) {
                float tot = 0.f;
                for (uint32_t r = 0; r < t.C; ++r) tot += xget(t, par, r, 6);
                const size_t o_idx = (static_cast<size_t>(d) * prm.B + b) * K + j;
                prm.gamma[o_idx] = tot;
                if (prm.loss) prm.loss[o_idx] = 1.f - tot;
            }
        };
        for (int i = 0; i < nothers; ++i) {
            if (i > 0) {
                take_other(i);
                {
                    const MaxSum o = warp_ms(st_o, c);
                    if (t.lane == 0) {
                        t.scr[t.warp * 4 + 2] = o.m;
                        t.scr[t.warp * 4 + 3] = o.s;
                    }
                }
                __syncthreads();
                release_other(i);
                if (t.warp == 0) {
                    MaxSum o2{NINF, 0.f};
                    if (t.lane < NWARPS) o2 = {t.scr[t.lane * 4 + 2], t.scr[t.lane * 4 + 3]};
                    o2 = warp_ms(o2, c);
                    v[0] = 0.f; v[1] = 0.f; v[2] = o2.m; v[3] = o2.s;
                    v[4] = NINF;
                    v[5] = __shfl_sync(0xffffffffu, xo_tok, 0);
                    v[6] = pend_ovl; v[7] = 0.f;
                }
                exchange(t, xpar, v);
                write_gamma(xpar, pend_d);
                go = xmerge(t, xpar, 2, 3, c);
                x_o_tok = NINF;
                for (uint32_t r = 0; r < t.C; ++r) x_o_tok = fmaxf(x_o_tok, xget(t, xpar, r, 5));
                xpar ^= 1;
            }
            const float bo = beta_of(go, c);
            const bool resample_row = prm.selected >= 0 && i == nothers - 1;
            const float ovl_acc = phase_b<E, P>(t, resample_row ? 1 : 0, tslot, ro, c, bt, bo,
                                                resample_row ? et_chunk : -1, et_elem, h_tok);
            const float cta_ovl = cta_sum_warp0(t, ovl_acc);   // its barrier also publishes the tiles
            if (resample_row && t.warp == 0) slice_total = tiles_to_prefix(t);
            pend_ovl = cta_ovl;
            pend_d = drafter_of(i);
            __syncthreads();
        }
        if (nothers == 0) {
            // bonus row: mass of the target row per tile
            phase_b<E, P>(t, 2, tslot, ro, c, bt_plain, 0.f, -1, -1, 0.f);
            __syncthreads();
            if (t.warp == 0) slice_total = tiles_to_prefix(t);
        }

        // ---- closing exchange: overlap of the last other row and this slice's mass for the draw ----
        if (t.warp == 0) {
            v[0] = v[1] = v[2] = v[3] = v[4] = v[5] = 0.f;
            v[6] = pend_ovl;
            v[7] = slice_total;
        }
        exchange(t, xpar, v);
        int par_tot = xpar;
        xpar ^= 1;
        if (nothers > 0) write_gamma(par_tot, pend_d);
        const bool draw = nothers == 0 || prm.selected >= 0;
        if (draw) {
            int mode = nothers == 0 ? 2 : 1;
            float Z = 0.f, ovl_tot = 0.f;
            for (uint32_t r = 0; r < t.C; ++r) {
                Z += xget(t, par_tot, r, 7);
                ovl_tot += xget(t, par_tot, r, 6);
            }
            const float z_resid = Z;
            int et_c = mode == 1 ? et_chunk : -1;
            if (mode == 1 && !(Z > 0.f)) {
                // A reject with no residual mass can only come from rounding: draw from h itself.
                mode = 2;
                phase_b<E, P>(t, 2, tslot, ro, c, bt, 0.f, et_chunk, et_elem, h_tok);
                __syncthreads();
                if (t.warp == 0) {
                    v[0] = v[1] = v[2] = v[3] = v[4] = v[5] = v[6] = 0.f;
                    v[7] = tiles_to_prefix(t);
                }
                exchange(t, xpar, v);
                par_tot = xpar;
                xpar ^= 1;
                Z = 0.f;
                for (uint32_t r = 0; r < t.C; ++r) Z += xget(t, par_tot, r, 7);
            }
            const float u = philox_uniform(prm.seeds[b], static_cast<uint32_t>(b), static_cast<uint32_t>(j), 1u);
            const float tp = u * Z;
            // owner slice: the first rank whose running total exceeds tp (else the last rank with mass)
            int owner = -1, last_pos = -1;
            float before = 0.f, before_last = 0.f, cum = 0.f;
            for (uint32_t r = 0; r < t.C; ++r) {
                const float tr = xget(t, par_tot, r, 7);
                const float prev = cum;
                cum += tr;
                if (tr > 0.f) {
                    last_pos = static_cast<int>(r);
                    before_last = prev;
                    if (owner < 0 && cum > tp) {
                        owner = static_cast<int>(r);
                        before = prev;
                    }
                }
            }
            if (owner < 0) {
                owner = last_pos;
                before = before_last;
            }
            if (owner == static_cast<int>(t.rank)) {
                if (t.warp == 0) {
                    // tile: the first prefix exceeding tp (else the last tile with mass)
                    int found = -1, lastp = -1;
                    for (int base = 0; base < t.ntiles; base += 32) {
                        const int ti = base + t.lane;
                        const bool in = ti < t.ntiles;
                        const float pre = in ? t.tiles[ti] : 0.f;
                        const float prv = (in && ti > 0) ? t.tiles[ti - 1] : 0.f;
                        const bool pos = in && pre > prv;
                        const unsigned over = __ballot_sync(0xffffffffu, pos && before + pre > tp);
                        const unsigned posm = __ballot_sync(0xffffffffu, pos);
                        if (found < 0 && over) found = base + __ffs(over) - 1;
                        if (posm) lastp = base + 31 - __clz(posm);
                    }
                    if (found < 0) found = lastp;
                    if (t.lane == 0) {
                        t.bci[0] = found;
                        t.bcf[0] = before + (found > 0 ? t.tiles[found - 1] : 0.f);
                    }
                }
                __syncthreads();
                const int tau = t.bci[0];
                const float before_tile = t.bcf[0];
                if (tau >= 0 && t.warp == tau % NWARPS) {
                    // the tile's warp recomputes its chunk masses exactly as in phase B
                    const int pp = tau / NWARPS;
                    const int kc = pp * NT + t.tid;
                    float vals[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) vals[e] = 0.f;
                    float ovl = 0.f, mass = 0.f;
                    if (kc < t.nchunks) {
                        const Raw rt = E::lds(tslot, kc);
                        Raw rsel = rt;
#pragma unroll
                        for (int p = 0; p < P; ++p)
                            if (p == pp) rsel = ro[p];
                        chunk_eval<E>(mode, rt, rsel, c, mode == 2 && nothers == 0 ? bt_plain : bt, beta_of(go, c),
                                      kc == (nothers == 0 ? -1 : et_chunk) ? et_elem : -1, h_tok, ovl, mass, vals);
                    }
                    const float incl = warp_incl_scan(mass, t.lane);
                    float excl = __shfl_up_sync(0xffffffffu, incl, 1);
                    if (t.lane == 0) excl = 0.f;
                    const unsigned over = __ballot_sync(0xffffffffu, mass > 0.f && before_tile + incl > tp);
                    const unsigned posm = __ballot_sync(0xffffffffu, mass > 0.f);
                    const int ln = over ? __ffs(over) - 1 : (posm ? 31 - __clz(posm) : -1);
                    if (t.lane == ln) {
                        float acc = before_tile + excl;
                        int pick = -1, lastpos = -1;
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            acc += vals[e];
                            if (vals[e] > 0.f) {
                                lastpos = e;
                                if (pick < 0 && acc > tp) pick = e;
                            }
                        }
                        if (pick < 0) pick = lastpos;
                        if (prm.rec)
                            reinterpret_cast<int*>(prm.rec)[(static_cast<size_t>(b) * (K + 1) + j) * REC + R_TOK] =
                                t.slice_start + kc * CHUNK + pick;
                    }
                }
            }
            (void)et_c;
            if (t.tid == 0 && t.rank == 0 && prm.rec && j < K) {
                float* rp = prm.rec + (static_cast<size_t>(b) * (K + 1) + j) * REC;
                rp[R_HT] = h_tok;
                rp[R_PD] = prob_of(x_o_tok, go, c);
                rp[R_Z] = z_resid;
                rp[R_OVL] = ovl_tot;
            }
        }
        __syncthreads();   // every thread is done with the target slot and the tile sums
        issue(k + 1, oth_released);
    }
    // no CTA may leave while a peer can still write into its shared memory
    cluster_sync_all();
}

// ------------------------------------------------------------------------------------------------
// chain finish: one warp per sequence turns the per-position records into the accept/reject chain
// (tutorial §9.1: verify left to right, stop at the first reject, emit its residual draw; all accepted:
// emit the bonus draw).
// ------------------------------------------------------------------------------------------------
struct FParams {
    const float* rec;            // [B, K+1, REC]
    const int32_t* tokens;       // [B, K]
    const uint64_t* seeds;       // [B]
    int B, K;
    int32_t* accept_len;         // [B]
    int32_t* out_tokens;         // [B, K+1]
    float* diag;                 // [B, K, 4] or null
    float* gamma_star;           // [B, K] or null (Cactus)
};

__global__ void __launch_bounds__(256) finish_kernel(const FParams f) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (b >= f.B) return;
    const int K = f.K;
    const uint64_t seed = f.seeds[b];
    int L = K;
    for (int base = 0; base < K; base += 32) {
        const int j = base + lane;
        bool acc = true;
        if (j < K) {
            const float* rp = f.rec + (static_cast<size_t>(b) * (K + 1) + j) * REC;
            const float ht = rp[R_HT], pd = rp[R_PD], z = rp[R_Z];
            const float r = philox_uniform(seed, static_cast<uint32_t>(b), static_cast<uint32_t>(j), 0u);
            acc = r * pd < ht;
            if (f.diag) {
                float* d = f.diag + (static_cast<size_t>(b) * K + j) * 4;
                d[0] = ht;
                d[1] = pd;
                d[2] = z;
                d[3] = r;
            }
            if (f.gamma_star) f.gamma_star[static_cast<size_t>(b) * K + j] = ht;
        }
        const unsigned rej = __ballot_sync(0xffffffffu, !acc);
        if (L == K && rej) L = base + __ffs(rej) - 1;
    }
    const int emitted = reinterpret_cast<const int*>(f.rec)[(static_cast<size_t>(b) * (K + 1) + L) * REC + R_TOK];
    for (int j = lane; j <= K; j += 32) {
        int v;
        if (j < L) v = f.tokens[static_cast<size_t>(b) * K + j];
        else if (j == L) v = emitted;
        else v = -1;
        f.out_tokens[static_cast<size_t>(b) * (K + 1) + j] = v;
    }
    if (lane == 0) f.accept_len[b] = L;
}

}  // namespace specv
