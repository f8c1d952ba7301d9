// Chain verification in two kernels (standard and Cactus speculative sampling of one drafter).
//
// Which rows need what:
//   - every target row (b, j) and draft row (b, j) needs its softmax normaliser, so that p(t) of the
//     draft token can be evaluated: one pass over every row;
//   - the accept chain (r * q(t) < p(t) from left to right) then fixes the first reject L of each
//     sequence; only row L needs the residual (p - q)+ and its draw, and only when every position accepts
//     does the bonus row K need its own draw. (Lossless tutorial §5.1 and §9.1: the chain stops at the
//     first reject; the positions after it are never sampled from.)
// So the rows are streamed once, in one balanced pass (stats_kernel), and a second kernel (draw_kernel)
// re-reads only the one row pair per sequence that a draw needs (the distribution diag, which reports
// Z for every position, re-reads every pair).
//
// stats_kernel: all rows of the call (the target rows, then the draft rows) are cut into pieces of PE
// logits, numbered row-major, and the piece range is split into G equal contiguous runs, one per warp of
// the grid. A warp streams its run through a private ring of R shared-memory slots (one bulk copy per
// piece, issued R pieces ahead), folds each piece into its lanes' running (max, sum of exponentials) and,
// where its run leaves a row (or ends), merges the lanes and stores the (max, sum) of that segment.
// Segment (warp g, row r) goes to entry g + r of the partials array: walking the segments in piece order,
// g or r (or both) grows at every step, so the entries are distinct, and there are at most
// min(G, pieces) + rows - 1 of them. There is no barrier and no exchange between warps.
//
// draw_kernel: one cluster of CTAs per sequence. Its warps merge the segments of the sequence's 2K + 1 rows
// (in ascending warp order), evaluate p(t) and q(t) at the draft tokens, run the chain (with the Cactus h
// when asked), then compute the residual (or bonus) mass of every piece of row L in parallel across the
// cluster, prefix-sum those masses in CTA 0, and find the drawn token with one scan of the chosen piece. The per-element arithmetic is the
// one of the inverse-CDF scan (chunk_mass / chunk_values / scan_pick), so every probability of the draw is
// computed the same way wherever it is needed.
#pragma once
#include "specverify_kernels.cuh"

namespace specv {

constexpr int SW = 16;                  // warps per CTA of the statistics kernel
constexpr int SNT = SW * 32;
constexpr int S_MAX_R = 4;              // ring slots per warp
constexpr int S_MAX_CTAS = 1024;        // grid cap (partials are sized for S_MAX_CTAS * SW warps)
constexpr int DW = 16;                  // warps per CTA of the draw kernel
constexpr int DNT = DW * 32;
constexpr int D_MAX_K = 64;             // positions per sequence
constexpr int D_LIST_CAP = 2 * DNT;     // kept logits of a listed row (standardised sampling): two a thread
constexpr int D_MAX_PIECES = 128;       // pieces per row (V <= 262144)

// The equal split of P pieces over G warps: warp g takes base + (g < rem) pieces from g * base + min(g, rem).
struct Split {
    long long base, rem;
    __host__ __device__ Split(long long P, long long G) : base(P / G), rem(P % G) {}
    __host__ __device__ long long start(long long g) const { return g * base + (g < rem ? g : rem); }
    __host__ __device__ long long count(long long g) const { return base + (g < rem ? 1 : 0); }
    // the warp whose run holds piece x (x < P)
    __host__ __device__ long long warp_of(long long x) const {
        const long long big = rem * (base + 1);
        return x < big ? x / (base + 1) : rem + (x - big) / base;
    }
};

struct SParams {
    const unsigned char* rows_a;   // the first rows_a_n rows: target rows [B, K+1, V]
    const unsigned char* rows_b;   // the next rows: draft rows [B, K, V]
    long long rows_a_n, rows_n;    // rows in the first block, rows in all
    int V, np;                     // logits per row, pieces per row
    long long P;                   // rows_n * np
    int G;                         // warps in the grid
    float c;                       // log2(e) / temperature
    int tma;                       // 1: rows 16-byte aligned and V a multiple of CHUNK -> bulk copies
    int R;                         // ring slots per warp
    int K;                         // draft positions per sequence
    int keep_j, keep_b;            // rows (b, j) with j < keep_j and b < keep_b are kept in L2 (evict-last)
                                   // for the draw kernel, which re-reads the row pair of the first reject
    float2* part;                  // (max, sum) of segment (g, r) at entry g + r
    unsigned* status;
};

template <class E>
__device__ __forceinline__ const unsigned char* s_row(const SParams& p, long long r, size_t row_bytes) {
    return r < p.rows_a_n ? p.rows_a + static_cast<size_t>(r) * row_bytes
                          : p.rows_b + static_cast<size_t>(r - p.rows_a_n) * row_bytes;
}

// Greedy mode of the statistics pass: folds a piece into the lane's running (largest logit m, its index).
// The lane's elements come in increasing index order (chunk lane + 32 q, q ascending, inside a piece;
// pieces ascending along the warp's run), so a strictly larger value is the only reason to move the
// index: the lane keeps the first occurrence. The piece is rescanned only when its bf16x2 maximum beats m.
template <class E>
__device__ __forceinline__ void piece_argmax(const typename E::Raw (&r)[PCH], int e_piece, int lane, float& m,
                                             int& idx) {
    typename E::Max mm = E::max_init();
#pragma unroll
    for (int q = 0; q < PCH; ++q) mm = E::max_acc(mm, r[q]);
    const float pm = E::max_fin(mm);
    if (pm > m) {
        int found = -1;
#pragma unroll
        for (int q = 0; q < PCH; ++q)
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float2 v = E::pair(r[q], w);
                const int e = e_piece + (lane + 32 * q) * CHUNK + 2 * w;
                if (found < 0 && v.x == pm) found = e;
                if (found < 0 && v.y == pm) found = e + 1;
            }
        m = pm;
        idx = found;
    }
}

// Warp merge of the lanes' (m, idx): the largest value, and the smallest index among the lanes holding it.
__device__ __forceinline__ void warp_argmax(float& m, int& idx) {
    const float M = warp_max(m);
    unsigned cand = (m == M && idx >= 0) ? static_cast<unsigned>(idx) : 0xFFFFFFFFu;
    unsigned r;
    asm volatile("redux.sync.min.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(cand));
    m = M;
    idx = r == 0xFFFFFFFFu ? -1 : static_cast<int>(r);
}

template <class E, bool ARGMAX = false>
__global__ void __launch_bounds__(SNT, 1) stats_kernel(const __grid_constant__ SParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    using Raw = typename E::Raw;
    const float NINF = __uint_as_float(0xFF800000u);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int R = p.R;
    const int eb = E::BYTES;
    const size_t row_bytes = static_cast<size_t>(p.V) * eb;
    const int slot_bytes = PE * eb;
    const float c = p.c;
    const Split sp(p.P, p.G);
    // the draw kernel may be scheduled now: its CTAs take the SMs this grid frees and read their inputs
    // before they wait for this grid to finish
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const long long g = static_cast<long long>(blockIdx.x) * SW + warp;
    const long long cnt = sp.count(g);
    if (cnt == 0) return;   // no CTA-wide barrier below
    const long long start = sp.start(g);
    long long row = start / p.np;
    int pc = static_cast<int>(start - row * p.np);
    float m = NINF, s = 0.f;
    int amax = -1;   // greedy mode: index of m in the row (-1: none yet)

    auto fold = [&](Raw (&r)[PCH], long long t) {
        if constexpr (ARGMAX) piece_argmax<E>(r, pc * PE, lane, m, amax);
        else piece_stats<E>(r, c, m, s);
        if (pc == p.np - 1 || t == cnt - 1) {   // the run leaves row `row` here: store the segment
            if constexpr (ARGMAX) {
                warp_argmax(m, amax);
                if (lane == 0) p.part[g + row] = make_float2(m, __int_as_float(amax));
                amax = -1;
            } else {
                const MaxSum a = warp_ms(MaxSum{m, s}, c);
                if (lane == 0) p.part[g + row] = make_float2(a.m, a.s);
            }
            m = NINF;
            s = 0.f;
        }
        if (++pc == p.np) {
            pc = 0;
            ++row;
        }
    };

    if (!p.tma) {   // rows of any alignment: element-wise loads straight into registers
        for (long long t = 0; t < cnt; ++t) {
            const unsigned char* src = s_row<E>(p, row, row_bytes);
            Raw r[PCH];
#pragma unroll
            for (int q = 0; q < PCH; ++q) {
                const int e0 = pc * PE + (lane + 32 * q) * CHUNK;
                r[q] = E::template gload<false>(src, e0, p.V);
            }
            fold(r, t);
        }
        return;
    }

    unsigned char* const ring = smem + static_cast<size_t>(warp) * R * slot_bytes;
    uint64_t* const full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(SW) * R * slot_bytes) + warp * R;
    if (lane == 0) {
        for (int q = 0; q < R; ++q) mbar_init(&full[q], 1);
        fence_mbarrier_init_cluster();
    }
    __syncwarp();
    // Every logit is read once here (evict-first), except the rows of the first draft positions: the draw
    // kernel re-reads the row pair at the sequence's first reject, most often position 0, right after this
    // grid, and finds them in L2 (evict-last; its own read demotes them).
    const uint64_t pol_first = policy_evict_first(), pol_last = policy_evict_last();
    auto row_policy = [&](long long r) -> uint64_t {
        const long long kp = r < p.rows_a_n ? p.K + 1 : p.K;
        const long long rr = r < p.rows_a_n ? r : r - p.rows_a_n;
        const long long b = rr / kp, j = rr - b * kp;
        return (j < p.keep_j && b < p.keep_b) ? pol_last : pol_first;
    };
    uint64_t ipol = 0;

    // the issue walker runs R pieces ahead of consumption
    long long irow = row;
    int ipc = pc;
    ipol = row_policy(irow);
    int islot = 0;
    long long issued = 0;   // pieces the walker has passed
    long long copies = 0;   // lane 0: bulk copies actually started (slot k % R for copy k)
    bool issuing = true;    // lane 0: false after a failed wait (no new copies into an unconfirmed slot)
    auto issue = [&]() {
        const int len = min(PE, p.V - ipc * PE);
        if (lane == 0 && issuing) {
            // the warp's reads of this slot (generic proxy) come before the copy that refills it
            fence_proxy_async_shared();
            const uint32_t bytes = static_cast<uint32_t>(len) * eb;
            mbar_arrive_expect_tx(&full[islot], bytes);
            bulk_load(ring + static_cast<size_t>(islot) * slot_bytes,
                      s_row<E>(p, irow, row_bytes) + static_cast<size_t>(ipc) * PE * eb, bytes, &full[islot], ipol);
            ++copies;
        }
        ++issued;
        if (++islot == R) islot = 0;
        if (++ipc == p.np) {
            ipc = 0;
            ++irow;
            ipol = row_policy(irow);
        }
    };
    for (int q = 0; q < R && issued < cnt; ++q) issue();

    int cslot = 0;
    uint32_t cpar = 0;
    bool ok = true;
    for (long long t = 0; t < cnt; ++t) {
        if (ok) ok = mbar_wait_bounded(&full[cslot], cpar, p.status, STATUS_TIMEOUT, WAIT_LIMIT_NS);
        if (lane == 0 && !ok) issuing = false;
        Raw r[PCH];
        piece_load<E>(ring + static_cast<size_t>(cslot) * slot_bytes, (min(PE, p.V - pc * PE) + CHUNK - 1) / CHUNK,
                      lane, r);
        __syncwarp();
        if (++cslot == R) {
            cslot = 0;
            cpar ^= 1u;
        }
        if (issued < cnt) issue();
        fold(r, t);
    }
    // after a failed wait, copies may still be in flight: they must land before the CTA may exit
    if (lane == 0 && !issuing) {
        // the last copy of each slot (a completed phase reads as complete again: no other copy followed)
        for (long long k = copies - R > 0 ? copies - R : 0; k < copies; ++k)
            mbar_wait_bounded(&full[k % R], static_cast<uint32_t>((k / R) & 1), p.status, STATUS_TIMEOUT, WAIT_LIMIT_NS);
    }
    __syncwarp();
}


// ------------------------------------------------------------------------------------------------
// draw kernel
// ------------------------------------------------------------------------------------------------
constexpr int D_MAX_CPS = 8;            // CTAs per sequence (one cluster)
constexpr float D_TAU = 1.f / 1024.f;   // fast chunk mass (residual plus overlap) above which a chunk is recomputed
                                        // at float-float precision
constexpr int D_QCH = 32;               // chunks of a warp's queue of such chunks
constexpr int D_CPP = PE / CHUNK;       // chunks per piece

struct DParams {
    const unsigned char* target;   // [B, K+1, V]
    const unsigned char* draft;    // [B, K, V]
    const float2* part;            // stats_kernel's segment partials (when row_ms is null)
    const float2* row_ms;          // or the (max, sum) of every statistics row, written by the gamma kernel
    long long P;                   // pieces of the statistics pass
    int G;                         // its warps
    int np;                        // pieces per row
    long long rows_a_n;            // B * (K + 1): draft row (b, j) is statistics row rows_a_n + b K + j
    const int32_t* tokens;         // [B, K]
    const uint64_t* seeds;         // [B]
    int B, K, V;
    int cps;                       // CTAs per sequence, the cluster size (piece pc belongs to CTA pc % cps)
    int tma;                       // 1: pieces come through a per-warp shared-memory slot by bulk copies
    float c, delta;
    int cactus;                    // 0: standard, 1: Cactus (Taylor gamma*), 2: Cactus (root of the KL constraint)
    FFc k;                         // constants of the float-float arithmetic of the draw
    int32_t* accept_len;           // [B]
    int32_t* out_tokens;           // [B, K+1]
    float* diag;                   // [B, K, 4] or null
    float* gamma_star;             // [B, K] or null (Cactus)
    const float* thr;              // FILT: per statistics row, the logits below it count as -inf
    const int* list_n;             // FILT: per target row, its kept logits listed (-1: none, read the row)
    const int* list_idx;           // FILT: [B (K+1), list_cap] their element indices, ascending
    const float* list_x;           // FILT: [B (K+1), list_cap] their values
    int list_cap;
    unsigned* status;
};

// (max, sum) of statistics row r: its segments merged in ascending warp order (warp-collective), or the
// row's entry of row_ms when the gamma kernel computed the rows whole.
__device__ __forceinline__ MaxSum d_row_stats(const DParams& p, const Split& sp, long long r, float c, int lane) {
    if (p.row_ms) {
        const float2 v = p.row_ms[r];
        return MaxSum{v.x, v.y};
    }
    const long long g0 = sp.warp_of(r * p.np), g1 = sp.warp_of(r * p.np + p.np - 1);
    MaxSum a{__uint_as_float(0xFF800000u), 0.f};
    for (long long g = g0 + lane; g <= g1; g += 32) {
        const float2 v = p.part[g + r];
        a = ms_merge(a, MaxSum{v.x, v.y}, c);
    }
    return warp_ms(a, c);
}

// A float pair stored into the shared memory of CTA 0 of this cluster from CTA `self`.
__device__ __forceinline__ void st_cta0_f32x2(float2* local, uint32_t self, float a, float b) {
    if (self == 0) *local = make_float2(a, b);
    else st_cluster_f32x2(map_to_rank(smem_addr(local), 0), a, b);
}

// What warp 0 of CTA 0 hands to the CTA for the pick inside the chosen piece.
struct PickPlan {
    int ft;          // chosen piece (-1: none, -2: already drawn)
    FF before, tp;   // mass before the piece; the target u * Z
};

// The fast mass of one chunk (element et, if >= 0, is the Cactus token with h = hpatch) and its overlap.
template <class E>
__device__ __forceinline__ float fast_chunk(int mode, const typename E::Raw& rt, const typename E::Raw& ro, float c,
                                            PairOff o, int et, float hpatch, float& ovl) {
    float2 o2 = make_float2(0.f, 0.f);
    if (et < 0) {
        const float m = chunk_mass<E>(mode, rt, ro, c, o, o2);
        ovl = o2.x + o2.y;
        return m;
    }
    ovl = 0.f;
    return chunk_mass_patch_only<E>(mode, rt, ro, c, o, et, hpatch, ovl);
}

// Cactus at one position, from the token's logit x and its row's offsets: the float-float p_T(n), gamma* and
// the scale s = (1 - gamma*) / (1 - p_T(n)) of the other tokens (out of line: once per position).
__device__ __noinline__ void cactus_precise(float x, float nm, float l, float l_lo, float delta, bool kl, const FFc& k,
                                            const float2* tab, FF& g, FF& sc) {
    const FF dt = ff_two_sum(x, nm);
    const FF q1 = ff_exp2(ff_exponent(dt.hi, k, l, l_lo, dt.lo), k, tab);
    g = cactus_gamma_ff(q1, delta, kl, k);
    const FF one = {1.f, 0.f};
    sc = q1.hi < 1.f ? ff_div(ff_sub(one, g), ff_sub(one, q1)) : FF{0.f, 0.f};
}

// A warp's queue of large chunks (n of them, n <= D_QCH: raw logits of both rows, the fast mass, the Cactus
// token's index in the chunk or -1) evaluated at float-float precision, eight lanes to a chunk and four chunks
// at a time (warp-collective). Returns this lane's share of the corrections (float-float mass minus fast mass).
template <class E>
__device__ __noinline__ FF flush_chunks(int mode, const typename E::Raw* qrt, const typename E::Raw* qro, const float* qcm,
                                        const int* qet, int n, const PairOffX po, const FFc& k, const float2* tab, FF g,
                                        int lane) {
    __syncwarp();
    FF acc = {0.f, 0.f};
    const int e = lane & 7;
    for (int base = 0; base < n; base += 4) {
        const int i = base + (lane >> 3);
        FF r = {0.f, 0.f};
        if (i < n) {
            const float2 xt2 = E::pair(qrt[i], e >> 1), xd2 = E::pair(qro[i], e >> 1);
            r = elem_exact(mode, (e & 1) ? xt2.y : xt2.x, (e & 1) ? xd2.y : xd2.x, po, k, tab, e == qet[i], g);
        }
        const FF sum = group8_sum(r);
        if (i < n && e == 0) acc = ff_add(acc, ff_addf(sum, -qcm[i]));
    }
    __syncwarp();
    return acc;
}

// A chunk as the filter leaves it (FILT: logits below t are -inf), else as loaded.
template <class E, bool FILT>
__device__ __forceinline__ typename E::Raw filt(const typename E::Raw& r, float t) {
    if constexpr (FILT) return E::mask(r, t);
    else return r;
}

// Every large chunk of piece pc (more than a queue holds), read again from memory: its float-float mass minus
// the fast one, eight lanes to a chunk (warp-collective; returns this lane's share). FILT: logits below tt
// (target row) and to (the other row) count as -inf.
template <class E, bool AL, bool FILT>
__device__ __noinline__ FF piece_exact(int mode, const unsigned char* trow, const unsigned char* orow, int pc, int V,
                                       float c, const PairOff po, const PairOffX px, const FFc& k, const float2* tab,
                                       int tok, float hpatch, FF g, int lane, float tt, float to) {
    FF acc = {0.f, 0.f};
    const int e = lane & 7;
    for (int base = 0; base < PE / CHUNK; base += 4) {
        const int e0 = pc * PE + (base + (lane >> 3)) * CHUNK;
        FF r = {0.f, 0.f};
        float cm = 0.f;
        bool big = false;
        if (e0 < V) {
            const typename E::Raw rt = filt<E, FILT>(E::template gload<AL>(trow, e0, V), tt);
            const typename E::Raw ro = mode == 1 ? filt<E, FILT>(E::template gload<AL>(orow, e0, V), to) : rt;
            const int et = (tok >= e0 && tok < e0 + CHUNK) ? tok - e0 : -1;
            float ovl;
            cm = fast_chunk<E>(mode, rt, ro, c, po, et, hpatch, ovl);
            big = cm + ovl > k.tau || et >= 0;
            if (big) {
                const float2 xt2 = E::pair(rt, e >> 1), xd2 = E::pair(ro, e >> 1);
                r = elem_exact(mode, (e & 1) ? xt2.y : xt2.x, (e & 1) ? xd2.y : xd2.x, px, k, tab, e == et, g);
            }
        }
        const FF sum = group8_sum(r);
        if (big && e == 0) acc = ff_add(acc, ff_addf(sum, -cm));
    }
    return acc;
}

// The draw's shared-memory state (one CTA; a draw kernel CTA holds it statically, the one-launch
// counterfactual kernel inside its dynamic shared memory once the gamma phase is over).
template <class E>
struct DrawShared {
    using Raw = typename E::Raw;
    float s_ht[D_MAX_K + 1], s_pd[D_MAX_K];
    // row offsets: target rows (nm, l as a float pair), the fast h rows of the chain (l with the Cactus
    // scale), draft rows
    float s_nmt[D_MAX_K + 1], s_ltp[D_MAX_K + 1], s_ltp_lo[D_MAX_K + 1], s_lt[D_MAX_K];
    float s_nmo[D_MAX_K], s_lo[D_MAX_K], s_lo_lo[D_MAX_K];
    float s_xt[D_MAX_K], s_xd[D_MAX_K];
    int s_tok[D_MAX_K];
    float2 s_sc[D_MAX_K], s_g[D_MAX_K];   // Cactus, per position: precise scale s and gamma*
    float2 s_tiles[D_MAX_PIECES];          // per piece: residual mass (float-float), gathered in CTA 0
    float2 s_tab[33];                      // the float-float exp2 table
    Raw s_qrt[DW][D_QCH], s_qro[DW][D_QCH];   // per warp: queue of large chunks (logits of both rows,
    float s_qcm[DW][D_QCH];                   // fast mass, Cactus token index)
    int s_qet[DW][D_QCH];
    int s_pl[D_CPP], s_pn;                 // the pick: large chunks of the chosen piece,
    float2 s_pm[D_CPP];                    // their float-float masses (by chunk)
    float2 s_pr[D_CPP][8];                 // and element residuals (by list position)
    float2 s_wscan[DW];                    // the pick's per-warp chunk totals
    int s_wfirst[DW], s_wlast[DW];
    PickPlan s_plan;
    int s_L, s_emit;
};

// One position's pass from its target row's kept logits alone (standardised sampling, when the threshold
// kernel listed them): h is 0 off that list, and so is the residual. The masses of the ln entries in
// vocabulary order at float-float precision (the draft logit at each entry's index read and masked), Z, and
// at the drawn position the pick by the full-row pass's rule: the first element of positive mass whose
// running mass exceeds u Z, else the last element of positive mass. All DNT threads of the cluster's CTA 0;
// thread t takes entries 2t and 2t + 1. Returns the drawn token (-1 off the drawn position).
template <class E>
__device__ __noinline__ int list_pass(const DParams& p, DrawShared<E>& S, int mode, int j, int L, int b, int ln,
                                      const unsigned char* orow, const PairOffX px, float to, uint64_t seed) {
    static_assert(2 * DNT >= D_LIST_CAP, "two entries a thread");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t base = (static_cast<size_t>(b) * (p.K + 1) + j) * static_cast<size_t>(p.list_cap);
    const int* const idx = p.list_idx + base;
    const float* const xs = p.list_x + base;
    const FF zero = {0.f, 0.f};
    // entry e's residual (m = 1) or target probability (m = 2)
    auto value = [&](int e, int m) -> FF {
        if (e >= ln) return zero;
        const float xt = xs[e];
        const float xd = m == 1 ? mask1(E::at(orow, idx[e]), to) : xt;
        return elem_exact(m, xt, xd, px, p.k, S.s_tab, false, zero);
    };
    // the mass before this thread's entries and the total, in entry order (fixed association)
    auto scan = [&](FF r0, FF r1, FF& before, FF& total) {
        const FF incl = warp_incl_scan_ff(ff_add(r0, r1), lane);
        if (lane == 31) S.s_wscan[warp] = make_float2(incl.hi, incl.lo);
        __syncthreads();
        FF start = zero;
        total = zero;
        for (int w = 0; w < DW; ++w) {
            const FF t = FF{S.s_wscan[w].x, S.s_wscan[w].y};
            if (w < warp) start = ff_add(start, t);
            total = ff_add(total, t);
        }
        FF excl = ff_shfl_up(incl, 1);
        if (lane == 0) excl = zero;
        before = ff_add(start, excl);
        __syncthreads();   // s_wscan may be written again
    };
    FF r0 = value(2 * tid, mode), r1 = value(2 * tid + 1, mode);
    FF before, Z;
    scan(r0, r1, before, Z);
    if (p.diag && j < p.K && tid == 0) p.diag[(static_cast<size_t>(b) * p.K + j) * 4 + 2] = Z.hi + Z.lo;
    if (j != L) return -1;
    const float u = philox_uniform(seed, static_cast<uint32_t>(b), static_cast<uint32_t>(L), 1u);
    if (mode == 1 && !(Z.hi > 0.f)) {   // the residual rounded to zero mass: draw from h over the row instead
        r0 = value(2 * tid, 2);
        r1 = value(2 * tid + 1, 2);
        scan(r0, r1, before, Z);
    }
    const FF tp = ff_mulf(Z, u);
    int first = 0x7fffffff, last = -1;
    FF a = ff_add(before, r0);
    if (r0.hi > 0.f) {
        last = 2 * tid;
        if (ff_gt(a, tp)) first = 2 * tid;
    }
    a = ff_add(a, r1);
    if (r1.hi > 0.f) {
        last = 2 * tid + 1;
        if (first == 0x7fffffff && ff_gt(a, tp)) first = 2 * tid + 1;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        first = min(first, __shfl_xor_sync(0xffffffffu, first, o));
        last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
    }
    if (lane == 0) {
        S.s_wfirst[warp] = first;
        S.s_wlast[warp] = last;
    }
    __syncthreads();
    int f = 0x7fffffff, l = -1;
    for (int w = 0; w < DW; ++w) {
        f = min(f, S.s_wfirst[w]);
        l = max(l, S.s_wlast[w]);
    }
    __syncthreads();
    const int chosen = f != 0x7fffffff ? f : l;
    return chosen >= 0 ? idx[chosen] : -1;
}

// One cluster of cps CTAs per sequence. Every CTA derives the row scalars
// and the chain itself (the same arithmetic on the same data, so the same L); the pieces of the drawn row
// are dealt to the CTAs round robin, each piece's residual mass (its large chunks recomputed at float-float
// precision) goes to CTA 0, and CTA 0 finds the piece holding u * Z and re-reads that one piece to find the
// token (fast_chunk, chunk_values and elem_exact give the same values in both places).
// draw_body runs it for one sequence on all DNT threads of one CTA: sequence blockIdx.x / cps and rank
// cluster_ctarank() in a draw kernel launch (LAUNCHED), else sequence b_arg as the only CTA of its cluster
// (cps = 1). d_smem: the bulk-copy slots and their mbarriers (bulk-copy mode). FILT: the logits of each row
// below its threshold p.thr[row] count as -inf (standardised sampling), wherever the draw reads them; a
// position whose target row's kept logits the threshold kernels listed (p.list_n >= 0) is drawn from that
// list by list_pass, and no CTA reads its rows.
template <class E, bool AL, bool LAUNCHED, bool FILT = false>
__device__ __forceinline__ void draw_body(const DParams& p, DrawShared<E>& S, unsigned char* const d_smem,
                                          const int b_arg) {
    using Raw = typename E::Raw;
    auto& s_ht = S.s_ht;
    auto& s_pd = S.s_pd;
    auto& s_nmt = S.s_nmt;
    auto& s_ltp = S.s_ltp;
    auto& s_ltp_lo = S.s_ltp_lo;
    auto& s_lt = S.s_lt;
    auto& s_nmo = S.s_nmo;
    auto& s_lo = S.s_lo;
    auto& s_lo_lo = S.s_lo_lo;
    auto& s_xt = S.s_xt;
    auto& s_xd = S.s_xd;
    auto& s_tok = S.s_tok;
    auto& s_sc = S.s_sc;
    auto& s_g = S.s_g;
    auto& s_tiles = S.s_tiles;
    auto& s_tab = S.s_tab;
    auto& s_qrt = S.s_qrt;
    auto& s_qro = S.s_qro;
    auto& s_qcm = S.s_qcm;
    auto& s_qet = S.s_qet;
    auto& s_pl = S.s_pl;
    auto& s_pn = S.s_pn;
    auto& s_pm = S.s_pm;
    auto& s_pr = S.s_pr;
    auto& s_wscan = S.s_wscan;
    auto& s_wfirst = S.s_wfirst;
    auto& s_wlast = S.s_wlast;
    auto& s_plan = S.s_plan;
    auto& s_L = S.s_L;
    auto& s_emit = S.s_emit;
    const float NINF = __uint_as_float(0xFF800000u);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int cps = LAUNCHED ? p.cps : 1;
    const uint32_t rank = LAUNCHED ? cluster_ctarank() : 0u;
    const int b = LAUNCHED ? static_cast<int>(blockIdx.x) / cps : b_arg;
    const int K = p.K, V = p.V, np = p.np;
    const float c = p.c;
    const size_t row_bytes = static_cast<size_t>(V) * E::BYTES;
    const Split sp(p.P, p.G);
    const bool use_tma = AL && p.tma;
    constexpr int PIECE_BYTES = PE * E::BYTES;
    unsigned char* const slot = d_smem + static_cast<size_t>(warp) * 2 * PIECE_BYTES;
    uint64_t* const fullb = reinterpret_cast<uint64_t*>(d_smem + static_cast<size_t>(DW) * 2 * PIECE_BYTES) + warp;
    if (use_tma && lane == 0) {
        mbar_init(fullb, 1);
        fence_mbarrier_init_cluster();
    }
    for (int i = threadIdx.x; i < 33; i += DNT) s_tab[i] = p.k.tab[i];
    __syncwarp();
    uint32_t uses = 0;       // completed phases of this warp's mbarrier
    int n_issued = 0;        // lane 0: bulk-copy groups started
    bool ok_all = true;      // every wait so far succeeded (warp-uniform)

    // ---- inputs only (nothing the statistics pass writes): read before the wait on that grid, while its
    // last CTAs still run. Draft tokens and their target and draft logits. ----
    const uint64_t seed = __ldg(p.seeds + b);
    for (int j = threadIdx.x; j < K; j += DNT) {
        int tok = __ldg(p.tokens + static_cast<size_t>(b) * K + j);
        float xt = NINF, xd = NINF;
        if (tok >= 0 && tok < V) {
            xt = E::at(p.target + (static_cast<size_t>(b) * (K + 1) + j) * row_bytes, tok);
            xd = E::at(p.draft + (static_cast<size_t>(b) * K + j) * row_bytes, tok);
        } else {
            tok = -1;
            if (rank == 0) atomicOr(p.status, STATUS_BAD_TOKEN);
        }
        s_tok[j] = tok;
        s_xt[j] = xt;
        s_xd[j] = xd;
    }
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // ---- normalisers of the 2K + 1 rows and the probabilities of the draft tokens (one warp a row) ----
    for (int q = warp; q < 2 * K + 1; q += DW) {
        const bool tgt = q <= K;
        const int j = tgt ? q : q - K - 1;
        const long long r = tgt ? static_cast<long long>(b) * (K + 1) + j : p.rows_a_n + static_cast<long long>(b) * K + j;
        float x = j < K ? (tgt ? s_xt[j] : s_xd[j]) : NINF;
        if constexpr (FILT) x = mask1(x, p.thr[r]);   // thresholds come from the grid before: read after its wait
        const MaxSum ms = d_row_stats(p, sp, r, c, lane);
        if (lane == 0) {
            const RowOff o = row_off(ms);
            const float pt = prob_at(x, o, c);   // 0 without a (valid) token
            // the row offset -log2 S also as a float pair, for the exact recomputations
            float ll = 0.f;
            if (ms.s > 0.f) {
                const FF l2 = ff_log2(FF{ms.s, 0.f}, p.k);
                ll = __fsub_rn(__fsub_rn(-l2.hi, o.l), l2.lo);
            }
            if constexpr (FILT) {
                if (j < K) (tgt ? s_xt[j] : s_xd[j]) = x;
            }
            if (tgt) {
                s_nmt[j] = o.nm;
                s_ltp[j] = o.l;
                s_ltp_lo[j] = ll;
                s_ht[j] = pt;
            } else {
                s_nmo[j] = o.nm;
                s_lo[j] = o.l;
                s_lo_lo[j] = ll;
                s_pd[j] = pt;
            }
        }
    }
    __syncthreads();

    // ---- the chain: accept r * q(t) < h(t) from the left (h = p_target, or the Cactus h) ----
    if (warp == 0) {
        int L = K;
        for (int base = 0; base < K; base += 32) {
            const int j = base + lane;
            bool acc = true;
            if (j < K) {
                float ht = s_ht[j], lt = s_ltp[j];
                if (p.cactus) {
                    float log2s, sf;
                    if (p.cactus == 2) cactus_scalars_kl(s_ht[j], p.delta, ht, log2s, sf);
                    else cactus_scalars(s_ht[j], p.delta, ht, log2s, sf);
                    lt = s_ltp[j] + log2s;
                }
                s_ht[j] = ht;
                s_lt[j] = lt;
                const float r = philox_uniform(seed, static_cast<uint32_t>(b), static_cast<uint32_t>(j), 0u);
                acc = r * s_pd[j] < ht;
                if (rank == 0) {
                    if (p.gamma_star) p.gamma_star[static_cast<size_t>(b) * K + j] = ht;
                    if (p.diag) {
                        float* d = p.diag + (static_cast<size_t>(b) * K + j) * 4;
                        d[0] = ht;
                        d[1] = s_pd[j];
                        d[3] = r;
                    }
                }
            }
            const unsigned rej = __ballot_sync(0xffffffffu, !acc);
            if (L == K && rej) L = base + __ffs(rej) - 1;
        }
        if (lane == 0) s_L = L;
    }
    __syncthreads();
    const int L = s_L;
    // Cactus, at the positions whose residual is drawn (or reported): gamma* and the scale s of the other
    // tokens from the float-float p_T(n). The fast masses use them too (h(n) = gamma*, log2 s in the offset).
    if (p.cactus && warp == 0) {
        for (int j = lane; j < K; j += 32) {
            if (s_tok[j] < 0 || !(p.diag || j == L)) continue;
            FF g1, sc;
            cactus_precise(s_xt[j], s_nmt[j], s_ltp[j], s_ltp_lo[j], p.delta, p.cactus == 2, p.k, s_tab, g1, sc);
            s_sc[j] = make_float2(sc.hi, sc.lo);
            s_g[j] = make_float2(g1.hi, g1.lo);
            s_lt[j] = s_ltp[j] + log2f(sc.hi);
        }
    }
    __syncthreads();

    // ---- masses of row L (of every position's row pair, too, when diag asks for Z) ----
    // The number of passes, and so of cluster barriers, depends on the call alone, never on L: with diag,
    // pass K (the bonus row) runs empty unless L = K.
    const int n_pass = p.diag ? K + 1 : 1;
    int emitted = -1;
    for (int it = 0; it < n_pass; ++it) {
        const int j = p.diag ? it : L;
        const bool idle = j == K && L != K;
        const int mode = j < K ? 1 : 2;   // 1: residual (h - q)+ against the draft row, 2: the bonus p_target
        const bool cact = mode == 1 && p.cactus && s_tok[j] >= 0;
        const unsigned char* trow = p.target + (static_cast<size_t>(b) * (K + 1) + j) * row_bytes;
        const unsigned char* orow = mode == 1 ? p.draft + (static_cast<size_t>(b) * K + j) * row_bytes : trow;
        // fast offsets (h row with the Cactus scale folded in) and the exact ones
        const PairOff po = mode == 1 ? PairOff{s_nmt[j], s_lt[j], s_nmo[j], s_lo[j]} : PairOff{s_nmt[K], s_ltp[K], 0.f, 0.f};
        const PairOffX px = mode == 1 ? PairOffX{s_nmt[j], s_ltp[j], s_ltp_lo[j], cact ? s_sc[j].x : 1.f, s_nmo[j], s_lo[j], s_lo_lo[j]}
                                      : PairOffX{s_nmt[K], s_ltp[K], s_ltp_lo[K], 1.f, 0.f, 0.f, 0.f};
        const int tok = cact ? s_tok[j] : -1;
        const FF gx = cact ? FF{s_g[j].x, s_g[j].y} : FF{0.f, 0.f};
        const float hpatch = gx.hi;
        float tt = 0.f, to = 0.f;   // the rows' filter thresholds
        if constexpr (FILT) {
            tt = p.thr[static_cast<size_t>(b) * (K + 1) + j];
            to = mode == 1 ? p.thr[p.rows_a_n + static_cast<long long>(b) * K + j] : tt;
        }
        if constexpr (FILT) {
            // a listed target row: CTA 0 works from the list, and no CTA reads the rows
            const int ln = p.list_n[static_cast<size_t>(b) * (K + 1) + j];
            if (ln >= 0) {
                if (rank == 0 && !idle) {
                    const int e = list_pass<E>(p, S, mode, j, L, b, ln, orow, px, to, seed);
                    if (j == L) emitted = e;
                }
                if (it + 1 < n_pass) cluster_sync_all();
                continue;
            }
        }
        // bulk copy of piece pc of both rows (the target alone for a bonus row) into this warp's slot
        auto issue = [&](int pc) {
            if (lane == 0 && ok_all) {
                const uint32_t bytes = static_cast<uint32_t>(min(PE, V - pc * PE)) * E::BYTES;
                fence_proxy_async_shared();   // the warp's reads of the slot come before the copy refilling it
                mbar_arrive_expect_tx(fullb, mode == 1 ? 2 * bytes : bytes);
                const uint64_t pol = policy_evict_first();
                bulk_load(slot, trow + static_cast<size_t>(pc) * PIECE_BYTES, bytes, fullb, pol);
                if (mode == 1) bulk_load(slot + PIECE_BYTES, orow + static_cast<size_t>(pc) * PIECE_BYTES, bytes, fullb, pol);
                ++n_issued;
            }
        };
        if (use_tma && !idle && static_cast<int>(rank) + cps * warp < np) issue(static_cast<int>(rank) + cps * warp);
        for (int i = warp; !idle; i += DW) {   // this CTA's pieces pc = rank + cps i
            const int pc = static_cast<int>(rank) + cps * i;
            if (pc >= np) break;
            Raw rt[PCH], ro[PCH];
            if (use_tma) {
                bool okw = ok_all ? mbar_wait_bounded(fullb, uses & 1u, p.status, STATUS_TIMEOUT, WAIT_LIMIT_NS) : false;
                okw = __shfl_sync(0xffffffffu, okw ? 1 : 0, 0) != 0;
                ok_all = ok_all && okw;
                ++uses;
                const int nch = (min(PE, V - pc * PE) + CHUNK - 1) / CHUNK;
                piece_load<E>(slot, nch, lane, rt);
                if (mode == 1) piece_load<E>(slot + PIECE_BYTES, nch, lane, ro);
                if constexpr (FILT) {
#pragma unroll
                    for (int q = 0; q < PCH; ++q) rt[q] = E::mask(rt[q], tt);
                    if (mode == 1) {
#pragma unroll
                        for (int q = 0; q < PCH; ++q) ro[q] = E::mask(ro[q], to);
                    }
                }
                if (mode != 1) {
#pragma unroll
                    for (int q = 0; q < PCH; ++q) ro[q] = rt[q];
                }
                __syncwarp();
                const int pc2 = static_cast<int>(rank) + cps * (i + DW);
                if (pc2 < np) issue(pc2);
            } else {
#pragma unroll
                for (int q = 0; q < PCH; ++q) {
                    const int e0 = pc * PE + (lane + 32 * q) * CHUNK;
                    rt[q] = filt<E, FILT>(E::template gload<AL>(trow, e0, V), tt);
                    ro[q] = mode == 1 ? filt<E, FILT>(E::template gload<AL>(orow, e0, V), to) : rt[q];
                }
            }
            FF loc = {0.f, 0.f};
            int nq = 0;   // large chunks of this piece in the warp's queue (more than D_QCH: all redone below)
#pragma unroll
            for (int q = 0; q < PCH; ++q) {
                const int e0 = pc * PE + (lane + 32 * q) * CHUNK;
                const int et = (tok >= e0 && tok < e0 + CHUNK) ? tok - e0 : -1;
                float ovl, cm;
                // filtered rows: where every target logit is -inf, h and so the residual and the overlap are 0
                // (most chunks of a top-k row): the warp skips the arithmetic when all its chunks are such
                if (!FILT || __any_sync(0xffffffffu, E::any_kept(rt[q]) || et >= 0)) {
                    cm = fast_chunk<E>(mode, rt[q], ro[q], c, po, et, hpatch, ovl);
                } else {
                    cm = 0.f;
                    ovl = 0.f;
                }
                loc = ff_addf(loc, cm);
                // a large chunk (or the Cactus token's) joins the queue: its float-float mass will replace cm
                const bool big = cm + ovl > p.k.tau || et >= 0;
                const unsigned bm = __ballot_sync(0xffffffffu, big);
                if (bm) {
                    const int at = nq + __popc(bm & ((1u << lane) - 1u));
                    if (big && at < D_QCH) {
                        s_qrt[warp][at] = rt[q];
                        s_qro[warp][at] = ro[q];
                        s_qcm[warp][at] = cm;
                        s_qet[warp][at] = et;
                    }
                    nq += __popc(bm);
                }
            }
            if (nq > D_QCH)   // a flat row: every large chunk of the piece again, from memory
                loc = ff_add(loc, piece_exact<E, AL, FILT>(mode, trow, orow, pc, V, c, po, px, p.k, s_tab, tok, hpatch,
                                                                 gx, lane, tt, to));
            else if (nq)
                loc = ff_add(loc, flush_chunks<E>(mode, s_qrt[warp], s_qro[warp], s_qcm[warp], s_qet[warp], nq, px, p.k,
                                                  s_tab, gx, lane));
            const FF m = warp_sum(loc);
            // the piece mass goes straight to CTA 0, which makes the draw
            if (lane == 0) st_cta0_f32x2(&s_tiles[pc], rank, m.hi, m.lo);
        }
        cluster_sync_all();   // every CTA's masses are in place and visible to the cluster
        if (rank == 0) {
            if (warp == 0 && !idle) {
                // piece masses in vocabulary order (np <= 4 * 32: lane l owns pieces seg l .. seg l + seg - 1)
                const int seg = (np + 31) / 32;
                const int lo = min(np, lane * seg), hi = min(np, lo + seg);
                FF tv[4];
                FF local = {0.f, 0.f};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int t = lo + k;
                    tv[k] = t < hi ? FF{s_tiles[t].x, s_tiles[t].y} : FF{0.f, 0.f};
                    local = ff_add(local, tv[k]);
                }
                const FF incl = warp_incl_scan_ff(local, lane);
                FF excl = ff_shfl_up(incl, 1);
                if (lane == 0) excl = FF{0.f, 0.f};
                const FF Z = ff_shfl(incl, 31);
                if (p.diag && j < K && lane == 0) p.diag[(static_cast<size_t>(b) * K + j) * 4 + 2] = Z.hi + Z.lo;
                if (j == L) {
                    const float u = philox_uniform(seed, static_cast<uint32_t>(b), static_cast<uint32_t>(L), 1u);
                    PickPlan plan = {};
                    plan.ft = -1;
                    if (mode == 1 && !(Z.hi > 0.f)) {
                        // the residual rounded to zero mass: draw from h over the whole row instead
                        const float ht = s_ht[j];
                        const int tk = s_tok[j];
                        double all = 0.0;
                        for (int e0 = lane * CHUNK; e0 < V; e0 += 32 * CHUNK) {
                            const Raw rt = filt<E, FILT>(E::template gload<AL>(trow, e0, V), tt);
                            float2 unused = make_float2(0.f, 0.f);
                            const int et = (tk >= e0 && tk < e0 + CHUNK) ? tk - e0 : -1;
                            all += static_cast<double>(chunk_mass_patched<E>(2, rt, rt, c, po, et, ht, unused));
                        }
                        const double tpd = static_cast<double>(u) * warp_sum(all);
                        emitted = scan_pick<E, AL, FILT>(c, trow, trow, 2, 0, V, po, tk, ht, tpd, 0.0, lane, tt, tt);
                        plan.ft = -2;
                    } else {
                        const FF tp = ff_mulf(Z, u);
                        // first piece whose prefix exceeds tp (else the last piece with mass)
                        int found = -1, lastp = -1;
                        FF before_found = {0.f, 0.f}, before_last = {0.f, 0.f};
                        FF run = excl;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int t = lo + k;
                            if (t < hi) {
                                const FF mm = tv[k];
                                const FF pre = ff_add(run, mm);
                                if (mm.hi > 0.f) {
                                    lastp = t;
                                    before_last = run;
                                    if (found < 0 && ff_gt(pre, tp)) {
                                        found = t;
                                        before_found = run;
                                    }
                                }
                                run = pre;
                            }
                        }
                        const unsigned hit = __ballot_sync(0xffffffffu, found >= 0);
                        if (hit) {
                            const int ln = __ffs(hit) - 1;
                            plan.ft = __shfl_sync(0xffffffffu, found, ln);
                            plan.before = ff_shfl(before_found, ln);
                        } else {
                            const unsigned any = __ballot_sync(0xffffffffu, lastp >= 0);
                            const int ln = any ? 31 - __clz(any) : 0;
                            plan.ft = __shfl_sync(0xffffffffu, lastp, ln);
                            plan.before = ff_shfl(before_last, ln);
                        }
                        plan.tp = tp;
                    }
                    if (lane == 0) {
                        s_plan = plan;
                        s_emit = emitted;
                    }
                }
            }
            __syncthreads();   // CTA 0: the plan is in place
            if (j == L && !idle && s_plan.ft >= 0) {
                // ---- the pick inside piece ft: one thread a chunk, the chunks' masses scanned across the CTA in
                // vocabulary order, then the elements of the chunk holding u * Z ----
                const PickPlan plan = s_plan;
                const int ft = plan.ft;
                const int nch = (min(PE, V - ft * PE) + CHUNK - 1) / CHUNK;
                const int ch = threadIdx.x;   // chunk of the piece (D_CPP = 256 <= DNT)
                const int e0 = ft * PE + ch * CHUNK;
                const int et = (tok >= e0 && tok < e0 + CHUNK) ? tok - e0 : -1;
                float v[8];   // the chunk's fast residual per element
                if constexpr (FILT) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) v[q] = 0.f;
                }
                FF m = {0.f, 0.f};
                bool big = false;
                Raw rt = E::ninf(), ro = E::ninf();
                if (threadIdx.x == 0) s_pn = 0;
                __syncthreads();
                if (ch < nch) {
                    rt = filt<E, FILT>(E::template gload<AL>(trow, e0, V), tt);
                    ro = mode == 1 ? filt<E, FILT>(E::template gload<AL>(orow, e0, V), to) : rt;
                    if (!FILT || E::any_kept(rt) || et >= 0) {   // (else the chunk's residual is 0: v stays 0)
                        float ovl, unused = 0.f;
                        const float cm = fast_chunk<E>(mode, rt, ro, c, po, et, hpatch, ovl);
                        chunk_values<E>(mode, rt, ro, c, po, et, hpatch, v, unused);
                        m = FF{cm, 0.f};
                        big = cm + ovl > p.k.tau || et >= 0;
                        if (big) s_pl[atomicAdd(&s_pn, 1)] = ch;
                    }
                }
                __syncthreads();
                // the piece's large chunks at float-float precision, eight threads to a chunk
                {
                    const int npl = s_pn;
                    for (int base = 0; base < npl; base += DNT / 8) {
                        const int li = base + threadIdx.x / 8, e = threadIdx.x & 7;
                        FF r = {0.f, 0.f};
                        if (li < npl) {
                            const int cj = s_pl[li];
                            const int c0 = ft * PE + cj * CHUNK;
                            const Raw xt = filt<E, FILT>(E::template gload<AL>(trow, c0, V), tt);
                            const Raw xd = mode == 1 ? filt<E, FILT>(E::template gload<AL>(orow, c0, V), to) : xt;
                            const float2 xt2 = E::pair(xt, e >> 1), xd2 = E::pair(xd, e >> 1);
                            const int cet = (tok >= c0 && tok < c0 + CHUNK) ? tok - c0 : -1;
                            r = elem_exact(mode, (e & 1) ? xt2.y : xt2.x, (e & 1) ? xd2.y : xd2.x, px, p.k, s_tab, e == cet, gx);
                            s_pr[li][e] = make_float2(r.hi, r.lo);
                        }
                        const FF sum = group8_sum(r);
                        if (li < npl && e == 0) s_pm[s_pl[li]] = make_float2(sum.hi, sum.lo);
                    }
                }
                __syncthreads();
                if (big) m = FF{s_pm[ch].x, s_pm[ch].y};
                // CTA-wide scan of the chunk masses (warps in order)
                const FF incl = warp_incl_scan_ff(m, lane);
                if (lane == 31) s_wscan[warp] = make_float2(incl.hi, incl.lo);
                __syncthreads();
                FF start = plan.before;
                for (int w = 0; w < warp; ++w) start = ff_add(start, FF{s_wscan[w].x, s_wscan[w].y});
                FF excl = ff_shfl_up(incl, 1);
                if (lane == 0) excl = FF{0.f, 0.f};
                start = ff_add(start, excl);
                const FF end = ff_add(start, m);
                const bool pos = ch < nch && m.hi > 0.f;
                const unsigned over = __ballot_sync(0xffffffffu, pos && ff_gt(end, plan.tp));
                const unsigned posm = __ballot_sync(0xffffffffu, pos);
                if (lane == 0) {
                    s_wfirst[warp] = over ? warp * 32 + __ffs(over) - 1 : 0x7fffffff;
                    s_wlast[warp] = posm ? warp * 32 + 31 - __clz(posm) : -1;
                }
                __syncthreads();
                int first = 0x7fffffff, last = -1;
                for (int w = 0; w < DW; ++w) {
                    first = min(first, s_wfirst[w]);
                    last = max(last, s_wlast[w]);
                }
                const int chosen = first != 0x7fffffff ? first : last;
                if (ch == chosen) {
                    int li = -1;   // the chunk's place in the list of large chunks
                    if (big)
                        for (int t = 0; t < s_pn; ++t)
                            if (s_pl[t] == ch) li = t;
                    FF a = start;
                    int pick = -1, lp = -1;
                    for (int e = 0; e < 8; ++e) {
                        const FF r = li >= 0 ? FF{s_pr[li][e].x, s_pr[li][e].y} : FF{v[e], 0.f};
                        a = ff_add(a, r);
                        if (r.hi > 0.f) {
                            lp = e;
                            if (pick < 0 && ff_gt(a, plan.tp)) pick = e;
                        }
                    }
                    s_emit = pick >= 0 ? e0 + pick : (lp >= 0 ? e0 + lp : -1);
                }
                __syncthreads();
            }
            if (j == L && !idle) emitted = s_emit;
        }
        // CTA 0 has read the other CTAs' masses before a next pass rewrites them; after the last pass no CTA
        // touches another's shared memory, so each may finish on its own
        if (it + 1 < n_pass) cluster_sync_all();
    }

    // after a failed wait a copy may still be in flight: it must land before the CTA may exit
    if (use_tma && lane == 0 && !ok_all && n_issued > 0)
        mbar_wait_bounded(fullb, static_cast<uint32_t>((n_issued - 1) & 1), p.status, STATUS_TIMEOUT, WAIT_LIMIT_NS);
    if (use_tma && lane == 0) mbar_inval(fullb);   // the slot's memory may be reused (a next draw_body call)
    __syncwarp();

    // ---- outputs ----
    if (rank == 0 && warp == 0) {
        for (int j = lane; j <= K; j += 32) {
            int v;
            if (j < L) v = __ldg(p.tokens + static_cast<size_t>(b) * K + j);
            else if (j == L) v = emitted;
            else v = -1;
            p.out_tokens[static_cast<size_t>(b) * (K + 1) + j] = v;
        }
        if (lane == 0) p.accept_len[b] = L;
    }
}

// One cluster of cps CTAs per sequence (CTA rank = blockIdx.x % cps).
template <class E, bool AL, bool FILT = false>
__global__ void __launch_bounds__(DNT, 1) draw_kernel(const __grid_constant__ DParams p) {
    // dynamic shared memory (bulk-copy mode): one slot per warp holding a target piece and a draft piece,
    // then one mbarrier per warp
    extern __shared__ __align__(128) unsigned char d_smem[];
    __shared__ DrawShared<E> S;
    draw_body<E, AL, true, FILT>(p, S, d_smem, 0);
}

// ------------------------------------------------------------------------------------------------
// greedy chain
// ------------------------------------------------------------------------------------------------
struct GrParams {
    const float2* part;            // the greedy statistics pass's segments: (largest logit, its index)
    long long P;                   // pieces of that pass
    int G;                         // its warps
    int np;                        // pieces per row
    const int32_t* tokens;         // [B, K]
    int B, K, V;
    int32_t* accept_len;           // [B]
    int32_t* out_tokens;           // [B, K+1]
    unsigned* status;
};

// One warp per sequence: the argmax of target rows (b, 0..K) from their segments (in piece order, so the
// first segment holding the largest value holds its first index), then the chain: accept draft j iff it
// is row j's argmax; emit the argmax of the first rejecting row, or of row K.
__global__ void __launch_bounds__(256) greedy_chain_kernel(const __grid_constant__ GrParams p) {
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int K = p.K;
    // draft tokens are inputs, read before waiting for the statistics grid: position lane in tokv0,
    // position lane + 32 in tokv1 (K <= 64)
    const int tokv0 = (b < p.B && lane < K) ? __ldg(p.tokens + static_cast<size_t>(b) * K + lane) : 0;
    const int tokv1 = (b < p.B && lane + 32 < K) ? __ldg(p.tokens + static_cast<size_t>(b) * K + lane + 32) : 0;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (b >= p.B) return;
    const Split sp(p.P, p.G);
    int L = K, emit = -1;
    for (int j = 0; j <= K; ++j) {
        const long long r = static_cast<long long>(b) * (K + 1) + j;
        const long long g0 = sp.warp_of(r * p.np), g1 = sp.warp_of(r * p.np + p.np - 1);
        // segments in index order: lane-strided walk keeping (largest, first index), then the warp merge
        float m = __uint_as_float(0xFF800000u);
        int idx = -1;
        for (long long gg = g0 + lane; gg <= g1; gg += 32) {
            const float2 v = p.part[gg + r];
            const int vi = __float_as_int(v.y);
            if (v.x > m || (v.x == m && vi >= 0 && (idx < 0 || vi < idx))) {
                m = v.x;
                idx = vi;
            }
        }
        warp_argmax(m, idx);
        const int am = idx >= 0 ? idx : 0;   // a row with every logit -inf: index 0
        int t = __shfl_sync(0xffffffffu, j < 32 ? tokv0 : tokv1, j & 31);
        if (j < K && (t < 0 || t >= p.V)) {
            if (lane == 0) atomicOr(p.status, STATUS_BAD_TOKEN);
            t = -1;
        }
        if (j == K || t != am) {
            L = j;
            emit = am;
            break;
        }
    }
    for (int j = lane; j <= K; j += 32) {
        int v;
        if (j < L) v = __ldg(p.tokens + static_cast<size_t>(b) * K + j);
        else if (j == L) v = emit;
        else v = -1;
        p.out_tokens[static_cast<size_t>(b) * (K + 1) + j] = v;
    }
    if (lane == 0) p.accept_len[b] = L;
}

}  // namespace specv
