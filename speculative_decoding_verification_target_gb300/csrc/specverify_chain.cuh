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
    int32_t* accept_len;           // [B]
    int32_t* out_tokens;           // [B, K+1]
    float* diag;                   // [B, K, 4] or null
    float* gamma_star;             // [B, K] or null (Cactus)
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

// Masses of the chunks lane l holds of a piece (chunks l + 32 q): mode 1 the residual (h - q)+, mode 2 h
// itself, element `et` of the piece (if >= 0) being h = hpatch. Element for element the values of
// chunk_mass and chunk_values.
template <class E>
__device__ __forceinline__ void piece_chunk_masses(int mode, const typename E::Raw (&rt)[PCH],
                                                   const typename E::Raw (&ro)[PCH], int lane, float c, PairOff o,
                                                   int et, float hpatch, float (&cm)[PCH]) {
    const int etc = et >= 0 ? et / CHUNK : -1;
    float2 unused = make_float2(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < PCH; ++q) {
        if (lane + 32 * q != etc) {
            cm[q] = chunk_mass<E>(mode, rt[q], ro[q], c, o, unused);
        } else {
            float ovl = 0.f;
            cm[q] = chunk_mass_patch_only<E>(mode, rt[q], ro[q], c, o, et % CHUNK, hpatch, ovl);
        }
    }
}

// A float (float-float) of the shared memory of CTA `owner` of this cluster (this CTA's own when owner == self).
__device__ __forceinline__ float cluster_f32(const float* local, uint32_t owner, uint32_t self) {
    return owner == self ? *local : ld_cluster_f32(map_to_rank(smem_addr(local), owner));
}
__device__ __forceinline__ FF cluster_ff(const float2* local, uint32_t owner, uint32_t self) {
    const float2 v = owner == self ? *local : ld_cluster_f32x2(map_to_rank(smem_addr(local), owner));
    return {v.x, v.y};
}

// Inverse CDF inside piece ft of the row (warp-collective): the chunk whose running mass (from `before`,
// accumulated in float-float like every sum above the chunk) first exceeds tp, from the chunk masses its CTA kept (chunks 8 l .. 8 l + 7 to lane l), then the element
// inside that chunk from its recomputed values. When rounding leaves no chunk above tp, the last chunk with
// positive mass; inside the chunk, the last positive element likewise. -1 if the piece has no mass.
template <class E, bool AL>
__device__ int pick_in_piece(const float* cm_slot, uint32_t owner, uint32_t self, const unsigned char* trow,
                             const unsigned char* orow, int mode, int e_begin, int V, float c, PairOff o,
                             int tok, float ht, FF tp, FF before, int lane) {
    const int nch = (min(PE, V - e_begin) + CHUNK - 1) / CHUNK;
    float cv[8];
    FF loc = {0.f, 0.f};
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int k = 8 * lane + q;
        cv[q] = k < nch ? cluster_f32(cm_slot + k, owner, self) : 0.f;
        loc = ff_addf(loc, cv[q]);
    }
    const FF incl = warp_incl_scan_ff(loc, lane);
    const FF end = ff_add(before, incl);
    const unsigned over = __ballot_sync(0xffffffffu, loc.hi > 0.f && ff_gt(end, tp));
    const unsigned posm = __ballot_sync(0xffffffffu, loc.hi > 0.f);
    if (!posm) return -1;
    const int ln = over ? __ffs(over) - 1 : 31 - __clz(posm);
    int chunk = -1;
    FF bchunk = {0.f, 0.f};
    if (lane == ln) {
        FF a = ff_sub(end, loc);
        int pk = -1, lp = -1;
        FF bpk = {0.f, 0.f}, blp = {0.f, 0.f};
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const FF a2 = ff_addf(a, cv[q]);
            if (cv[q] > 0.f) {
                lp = q;
                blp = a;
                if (pk < 0 && ff_gt(a2, tp)) {
                    pk = q;
                    bpk = a;
                }
            }
            a = a2;
        }
        chunk = 8 * ln + (pk >= 0 ? pk : lp);
        bchunk = pk >= 0 ? bpk : blp;
    }
    chunk = __shfl_sync(0xffffffffu, chunk, ln);
    bchunk = ff_shfl(bchunk, ln);
    const int e0 = e_begin + chunk * CHUNK;
    const typename E::Raw rt = E::template gload<AL>(trow, e0, V);
    const typename E::Raw ro = mode == 1 ? E::template gload<AL>(orow, e0, V) : rt;
    const int et = (tok >= e0 && tok < e0 + CHUNK) ? tok - e0 : -1;
    float v[8], ovl = 0.f;
    chunk_values<E>(mode, rt, ro, c, o, et, ht, v, ovl);
    FF a = bchunk;
    int pick = -1, lp = -1;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        a = ff_addf(a, v[q]);
        if (v[q] > 0.f) {
            lp = q;
            if (pick < 0 && ff_gt(a, tp)) pick = q;
        }
    }
    return pick >= 0 ? e0 + pick : (lp >= 0 ? e0 + lp : -1);
}

// One cluster of cps CTAs per sequence b (CTA rank = blockIdx.x % cps). Every CTA derives the row scalars
// and the chain itself (the same arithmetic on the same data, so the same L); the pieces of the drawn row
// are dealt to the CTAs round robin, and CTA 0 makes the draw from the masses the CTAs keep in shared
// memory, read across the cluster.
template <class E, bool AL>
__global__ void __launch_bounds__(DNT, 1) draw_kernel(const __grid_constant__ DParams p) {
    using Raw = typename E::Raw;
    // dynamic shared memory: [ceil(np / cps)][D_CPP] chunk masses of this CTA's pieces, then (bulk-copy
    // mode) one slot per warp holding a target piece and a draft piece, then one mbarrier per warp
    extern __shared__ __align__(128) float d_cm[];
    __shared__ float s_ht[D_MAX_K + 1], s_pd[D_MAX_K];
    // row offsets: target rows (nm, plain l), the h rows of the chain (l with the Cactus scale), draft rows
    __shared__ float s_nmt[D_MAX_K + 1], s_ltp[D_MAX_K + 1], s_lt[D_MAX_K], s_nmo[D_MAX_K], s_lo[D_MAX_K];
    __shared__ float s_xt[D_MAX_K], s_xd[D_MAX_K];
    __shared__ int s_tok[D_MAX_K];
    __shared__ float2 s_tiles[D_MAX_PIECES];  // piece masses (float-float sums of chunk masses), gathered in CTA 0
    __shared__ int s_L;
    const float NINF = __uint_as_float(0xFF800000u);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int cps = p.cps;
    const uint32_t rank = cluster_ctarank();
    const int b = blockIdx.x / cps;
    const int K = p.K, V = p.V, np = p.np;
    const float c = p.c;
    const size_t row_bytes = static_cast<size_t>(V) * E::BYTES;
    const Split sp(p.P, p.G);
    const bool use_tma = AL && p.tma;
    constexpr int PIECE_BYTES = PE * E::BYTES;
    unsigned char* const ring = reinterpret_cast<unsigned char*>(d_cm) +
                                static_cast<size_t>((np + cps - 1) / cps) * D_CPP * sizeof(float);
    unsigned char* const slot = ring + static_cast<size_t>(warp) * 2 * PIECE_BYTES;
    uint64_t* const fullb = reinterpret_cast<uint64_t*>(ring + static_cast<size_t>(DW) * 2 * PIECE_BYTES) + warp;
    if (use_tma && lane == 0) {
        mbar_init(fullb, 1);
        fence_mbarrier_init_cluster();
    }
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
        const float x = j < K ? (tgt ? s_xt[j] : s_xd[j]) : NINF;
        const MaxSum ms = d_row_stats(p, sp, r, c, lane);
        if (lane == 0) {
            const RowOff o = row_off(ms);
            const float pt = prob_at(x, o, c);   // 0 without a (valid) token
            if (tgt) {
                s_nmt[j] = o.nm;
                s_ltp[j] = o.l;
                s_ht[j] = pt;
            } else {
                s_nmo[j] = o.nm;
                s_lo[j] = o.l;
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
                    float log2s;
                    if (p.cactus == 2) cactus_scalars_kl(s_ht[j], p.delta, ht, log2s);
                    else cactus_scalars(s_ht[j], p.delta, ht, log2s);
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

    // ---- chunk and piece masses of row L (of every position's row pair, too, when diag asks for Z) ----
    // The number of passes, and so of cluster barriers, depends on the call alone, never on L: with diag,
    // pass K (the bonus row) runs empty unless L = K.
    const int n_pass = p.diag ? K + 1 : 1;
    int emitted = -1;
    for (int it = 0; it < n_pass; ++it) {
        const int j = p.diag ? it : L;
        const bool idle = j == K && L != K;
        const int mode = j < K ? 1 : 2;   // 1: residual (h - q)+ against the draft row, 2: the bonus p_target
        const unsigned char* trow = p.target + (static_cast<size_t>(b) * (K + 1) + j) * row_bytes;
        const unsigned char* orow = mode == 1 ? p.draft + (static_cast<size_t>(b) * K + j) * row_bytes : trow;
        const PairOff po = mode == 1 ? PairOff{s_nmt[j], s_lt[j], s_nmo[j], s_lo[j]} : PairOff{s_nmt[K], s_ltp[K], 0.f, 0.f};
        const float ht = mode == 1 ? s_ht[j] : 0.f;
        const int tok = mode == 1 ? s_tok[j] : -1;
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
                else {
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
                    rt[q] = E::template gload<AL>(trow, e0, V);
                    ro[q] = mode == 1 ? E::template gload<AL>(orow, e0, V) : rt[q];
                }
            }
            const int et = (tok >= pc * PE && tok < pc * PE + PE) ? tok - pc * PE : -1;
            float cm[PCH];
            piece_chunk_masses<E>(mode, rt, ro, lane, c, po, et, ht, cm);
            FF loc = {0.f, 0.f};
#pragma unroll
            for (int q = 0; q < PCH; ++q) {
                d_cm[i * D_CPP + lane + 32 * q] = cm[q];
                loc = ff_addf(loc, cm[q]);
            }
            const FF m = warp_sum(loc);
            // the piece mass goes straight to CTA 0, which makes the draw
            if (lane == 0) {
                if (rank == 0) s_tiles[pc] = make_float2(m.hi, m.lo);
                else st_cluster_f32x2(map_to_rank(smem_addr(&s_tiles[pc]), 0), m.hi, m.lo);
            }
        }
        cluster_sync_all();   // every CTA's masses are in place and visible to the cluster
        if (rank == 0 && warp == 0 && !idle) {
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
                if (mode == 1 && !(Z.hi > 0.f)) {
                    // the residual rounded to zero mass: draw from h over the whole row instead
                    double all = 0.0;
                    for (int e0 = lane * CHUNK; e0 < V; e0 += 32 * CHUNK) {
                        const Raw rt = E::template gload<AL>(trow, e0, V);
                        float2 unused = make_float2(0.f, 0.f);
                        const int et = (tok >= e0 && tok < e0 + CHUNK) ? tok - e0 : -1;
                        all += static_cast<double>(chunk_mass_patched<E>(2, rt, rt, c, po, et, ht, unused));
                    }
                    const double tp = static_cast<double>(u) * warp_sum(all);
                    emitted = scan_pick<E, AL>(c, trow, trow, 2, 0, V, po, tok, ht, tp, 0.0, lane);
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
                            const FF m = tv[k];
                            const FF pre = ff_add(run, m);
                            if (m.hi > 0.f) {
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
                    int ft;
                    FF before_piece;
                    if (hit) {
                        const int ln = __ffs(hit) - 1;
                        ft = __shfl_sync(0xffffffffu, found, ln);
                        before_piece = ff_shfl(before_found, ln);
                    } else {
                        const unsigned any = __ballot_sync(0xffffffffu, lastp >= 0);
                        const int ln = any ? 31 - __clz(any) : 0;
                        ft = __shfl_sync(0xffffffffu, lastp, ln);
                        before_piece = ff_shfl(before_last, ln);
                    }
                    if (ft >= 0)
                        emitted = pick_in_piece<E, AL>(d_cm + (ft / cps) * D_CPP, static_cast<uint32_t>(ft % cps), rank,
                                                       trow, orow, mode, ft * PE, V, c, po, tok, ht, tp,
                                                       before_piece, lane);
                }
            }
        }
        cluster_sync_all();   // CTA 0 has read the other CTAs' masses; the buffers may be rewritten or released
    }

    // after a failed wait a copy may still be in flight: it must land before the CTA may exit
    if (use_tma && lane == 0 && !ok_all && n_issued > 0)
        mbar_wait_bounded(fullb, static_cast<uint32_t>((n_issued - 1) & 1), p.status, STATUS_TIMEOUT, WAIT_LIMIT_NS);
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
