// Counterfactual acceptance for N drafters, gamma[i, b, j] = sum_x min(p_target(x), q_i(x)), with the loss
// 1 - gamma ("Not-a-Bandit: Provably No-Regret Drafter Selection in Speculative Decoding for LLMs", Key
// design 1 and 3; the identity sum min(p, q) = 1 - TV(p, q) is the lossless tutorial's §6.3-§6.4).
//
// Every term needs both rows' normalisers, so each drafter row is visited twice: once for its (max, sum
// of exponentials) and once for the sum of minima. gamma_kernel reads every logit from HBM once and keeps
// the second visit on chip:
//   - a CTA owns a contiguous run of "units" in the order T(b, j), D_0(b, j), ..., D_{N-1}(b, j) for every
//     position, then the bonus target rows T(b, K) when a chain is verified as well. A T unit computes the
//     target row's normaliser; a D unit computes the drafter row's normaliser and then its gamma. A CTA
//     whose run starts inside a position first computes that position's T unit itself;
//   - a whole row is split over the CTA's 16 warps (warp w takes pieces w, w + 16, ...), so the normaliser
//     of a row is complete once every warp has passed one CTA barrier: no exchange between CTAs;
//   - pass 1 streams the pieces of unit s from HBM through a private ring of bulk-copy slots per warp.
//     Each warp parks the raw logits of its first four drafter pieces in tensor memory (its 32 lanes x
//     128 columns of the CTA's 512-column allocation: 16 KB, so a row of up to 64 x 4 KB is held whole);
//   - pass 2 of unit s - 1 runs in the same step, piece by piece ahead of pass 1 of unit s: it reads the
//     parked drafter piece back from tensor memory (the columns are then free for unit s), reads the target
//     piece from L2 (the CTA keeps one target row hot while it walks that position's drafters) and adds
//     sum 2^min(log2 p_target, log2 q_i). Pieces past the tensor-memory share are re-read from L2.
// One CTA barrier per step merges the 16 warps' (max, sum) pairs of unit s and their gamma partials of
// unit s - 1, each in a fixed order, so the result does not depend on timing.
#pragma once
#include "specverify_chain.cuh"

namespace specv {

constexpr int GW = 16;                       // warps per CTA
constexpr int GNT = GW * 32;
constexpr int G_PIECE_BYTES = 4096;          // one bulk copy: 2048 bf16 or 1024 fp32 logits
constexpr int G_R = 3;                       // ring slots per warp
constexpr int G_CAP = 4;                     // pieces a warp parks in tensor memory (32 columns each)
constexpr int G_TMEM_COLS = 512;
constexpr size_t G_SMEM = static_cast<size_t>(GW) * G_R * G_PIECE_BYTES + static_cast<size_t>(GW) * G_R * 8;

struct CgParams {
    const unsigned char* target;     // [B, K+1, V]
    const unsigned char* drafters;   // [N, B, K, V]
    int B, K, V, N;
    int np;                          // pieces per row
    long long U;                     // units in all
    int G;                           // CTAs
    float c;                         // log2(e) / temperature
    int tma;                         // 1: rows 16-byte aligned and V a multiple of 8 -> bulk copies
    int selected;                    // drafter whose rows' (max, sum) go to row_ms (-1: none)
    float* gamma;                    // [N, B, K]
    float* loss;                     // [N, B, K] or null
    float2* row_ms;                  // (max, sum) per statistics row, or null (see below)
    unsigned* status;
};
// row_ms layout (the one draw_kernel reads): target row (b, j) at b (K + 1) + j for j <= K, then the rows
// of drafter `selected` at B (K + 1) + b K + j.

struct GUnit {
    const unsigned char* row;   // the row pass 1 reads
    const unsigned char* trow;  // the target row of the position (pass 2 of a D unit)
    int kind;                   // 0: T unit of (b, j); 1: D unit of drafter i at (b, j); 2: bonus row (b, K)
    int b, j, i;
};

__device__ __forceinline__ GUnit g_unit(const CgParams& p, long long u, size_t row_bytes) {
    GUnit r;
    const long long nd = static_cast<long long>(p.B) * p.K * (p.N + 1);
    if (u < nd) {
        const long long item = u / (p.N + 1);
        const int k = static_cast<int>(u - item * (p.N + 1));
        r.b = static_cast<int>(item / p.K);
        r.j = static_cast<int>(item - static_cast<long long>(r.b) * p.K);
        r.trow = p.target + (static_cast<size_t>(r.b) * (p.K + 1) + r.j) * row_bytes;
        if (k == 0) {
            r.kind = 0;
            r.i = -1;
            r.row = r.trow;
        } else {
            r.kind = 1;
            r.i = k - 1;
            r.row = p.drafters + ((static_cast<size_t>(r.i) * p.B + r.b) * p.K + r.j) * row_bytes;
        }
    } else {
        r.kind = 2;
        r.b = static_cast<int>(u - nd);
        r.j = p.K;
        r.i = -1;
        r.trow = p.target + (static_cast<size_t>(r.b) * (p.K + 1) + p.K) * row_bytes;
        r.row = r.trow;
    }
    return r;
}

// ---------------------------------------- tensor memory ----------------------------------------
// A warp may address only the 32 lanes of its quarter (warp index mod 4). Each thread stores / loads 32
// consecutive 32-bit columns of its own lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
        "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
        "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
          "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
          "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
          "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// A piece held by one lane as 32 words: bf16, 8 chunks of 16 B; fp32, 4 chunks of 32 B.
template <class E>
struct GPiece;
template <>
struct GPiece<Bf16> {
    static constexpr int NCH = 8;
    __device__ static void to_words(const Bf16::Raw (&r)[NCH], uint32_t (&w)[32]) {
#pragma unroll
        for (int q = 0; q < NCH; ++q) {
            w[4 * q] = r[q].x;
            w[4 * q + 1] = r[q].y;
            w[4 * q + 2] = r[q].z;
            w[4 * q + 3] = r[q].w;
        }
    }
    __device__ static void from_words(const uint32_t (&w)[32], Bf16::Raw (&r)[NCH]) {
#pragma unroll
        for (int q = 0; q < NCH; ++q) r[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    }
    // one chunk from global memory through the read-only path without L1 allocation, normal L2 policy
    // (target rows are read again by the position's next drafters). Chunks at or past n_el are -inf.
    __device__ static Bf16::Raw ld_keep(const unsigned char* row, int e0, int n_el) {
        uint4 v = Bf16::ninf();
        const uint4* ptr = reinterpret_cast<const uint4*>(row) + e0 / CHUNK;
        asm volatile(
            "{\n\t.reg .pred q;\n\tsetp.lt.s32 q, %4, %5;\n\t"
            "@q ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%6];\n\t}"
            : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)
            : "r"(e0), "r"(n_el), "l"(ptr));
        return v;
    }
};
template <>
struct GPiece<F32> {
    static constexpr int NCH = 4;
    __device__ static void to_words(const F32::Raw (&r)[NCH], uint32_t (&w)[32]) {
#pragma unroll
        for (int q = 0; q < NCH; ++q) {
            w[8 * q] = __float_as_uint(r[q].a.x);
            w[8 * q + 1] = __float_as_uint(r[q].a.y);
            w[8 * q + 2] = __float_as_uint(r[q].a.z);
            w[8 * q + 3] = __float_as_uint(r[q].a.w);
            w[8 * q + 4] = __float_as_uint(r[q].b.x);
            w[8 * q + 5] = __float_as_uint(r[q].b.y);
            w[8 * q + 6] = __float_as_uint(r[q].b.z);
            w[8 * q + 7] = __float_as_uint(r[q].b.w);
        }
    }
    __device__ static void from_words(const uint32_t (&w)[32], F32::Raw (&r)[NCH]) {
#pragma unroll
        for (int q = 0; q < NCH; ++q) {
            r[q].a = make_float4(__uint_as_float(w[8 * q]), __uint_as_float(w[8 * q + 1]), __uint_as_float(w[8 * q + 2]),
                                 __uint_as_float(w[8 * q + 3]));
            r[q].b = make_float4(__uint_as_float(w[8 * q + 4]), __uint_as_float(w[8 * q + 5]),
                                 __uint_as_float(w[8 * q + 6]), __uint_as_float(w[8 * q + 7]));
        }
    }
    __device__ static F32::Raw ld_keep(const unsigned char* row, int e0, int n_el) {
        F32::Raw v = F32::ninf();
        const float* ptr = reinterpret_cast<const float*>(row) + e0;
        asm volatile(
            "{\n\t.reg .pred q;\n\tsetp.lt.s32 q, %8, %9;\n\t"
            "@q ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%10];\n\t"
            "@q ld.global.nc.L1::no_allocate.v4.f32 {%4, %5, %6, %7}, [%10+16];\n\t}"
            : "+f"(v.a.x), "+f"(v.a.y), "+f"(v.a.z), "+f"(v.a.w), "+f"(v.b.x), "+f"(v.b.y), "+f"(v.b.z), "+f"(v.b.w)
            : "r"(e0), "r"(n_el), "l"(ptr));
        return v;
    }
};

// ---------------------------------------- per-piece arithmetic ----------------------------------------
// Pass 1: folds the piece into the lane's running (max m, sum s of 2^((x - m) c)).
template <class E>
__device__ __forceinline__ void g_stats(const typename E::Raw (&r)[GPiece<E>::NCH], float c, float& m, float& s) {
    chunks_stats<E, GPiece<E>::NCH>(r, c, m, s);
}

// Pass 2: adds sum_x 2^min(x_t c + bt, x_d c + bd) over the piece (bt, bd: the rows' log2 offsets).
template <class E>
__device__ __forceinline__ void g_overlap(const typename E::Raw (&rt)[GPiece<E>::NCH],
                                          const typename E::Raw (&rd)[GPiece<E>::NCH], float c, float bt, float bd,
                                          float2& acc) {
    constexpr int NCH = GPiece<E>::NCH;
    const float2 cc = make_float2(c, c), bt2 = make_float2(bt, bt), bd2 = make_float2(bd, bd);
    float2 a4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
    for (int q = 0; q < NCH; ++q) a4[q & 3] = chunk_overlap<E>(rt[q], rd[q], cc, bt2, bd2, a4[q & 3]);
    acc = __fadd2_rn(acc, __fadd2_rn(__fadd2_rn(a4[0], a4[1]), __fadd2_rn(a4[2], a4[3])));
}

// ---------------------------------------- the kernel ----------------------------------------
template <class E>
__global__ void __launch_bounds__(GNT, 1) gamma_kernel(const __grid_constant__ CgParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint32_t s_tmem;
    __shared__ float2 s_ms[2][GW];   // per step parity: the warps' (max, sum) of unit s
    __shared__ float s_g[2][GW];     // per step parity: the warps' gamma partials of unit s - 1
    using Raw = typename E::Raw;
    constexpr int NCH = GPiece<E>::NCH;
    constexpr int PEG = G_PIECE_BYTES / E::BYTES;   // logits per piece
    const float NINF = __uint_as_float(0xFF800000u);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int V = p.V, np = p.np;
    const size_t row_bytes = static_cast<size_t>(V) * E::BYTES;
    const float c = p.c;
    // a chained draw kernel may be scheduled now; it waits for this grid before it reads row_ms
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // all 512 tensor-memory columns (the dynamic shared memory admits one CTA per SM)
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&s_tmem)),
                     "r"(G_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    unsigned char* const ring = smem + static_cast<size_t>(warp) * G_R * G_PIECE_BYTES;
    uint64_t* const full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(GW) * G_R * G_PIECE_BYTES) + warp * G_R;
    if (p.tma && lane == 0) {
        for (int q = 0; q < G_R; ++q) mbar_init(&full[q], 1);
        fence_mbarrier_init_cluster();
    }
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    const uint32_t tbase = s_tmem;
    // this warp's columns: lanes 32 (warp mod 4) .. + 31, columns 128 (warp / 4) .. + 127
    const uint32_t twarp = tbase + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + static_cast<uint32_t>((warp >> 2) * G_CAP * 32);

    // this CTA's run of units
    const long long u0 = static_cast<long long>(blockIdx.x) * p.U / p.G;
    const long long u1 = static_cast<long long>(blockIdx.x + 1) * p.U / p.G;
    const long long nd = static_cast<long long>(p.B) * p.K * (p.N + 1);
    const bool pre = u0 < nd && (u0 % (p.N + 1)) != 0;
    const long long S = (u1 - u0) + (pre ? 1 : 0);
    auto unit_of = [&](long long t) -> GUnit {
        const long long u = pre ? (t == 0 ? u0 - u0 % (p.N + 1) : u0 + t - 1) : u0 + t;
        return g_unit(p, u, row_bytes);
    };
    const int nmine = warp < np ? (np - 1 - warp) / GW + 1 : 0;   // pieces warp, warp + 16, ... of a row

    // ---- ring of pass-1 pieces (bulk copies), the issue walker runs G_R pieces ahead ----
    const uint64_t pol_first = policy_evict_first(), pol_normal = policy_evict_normal();
    long long it_t = 0;
    int it_k = 0;
    GUnit it_u = unit_of(0);
    const long long total = S * nmine;
    long long issued = 0, copies = 0;
    int islot = 0;
    bool issuing = true;
    auto issue = [&]() {
        const int pc = warp + GW * it_k;
        const int len = min(PEG, V - pc * PEG);
        if (lane == 0 && issuing) {
            fence_proxy_async_shared();   // the warp's reads of this slot come before the copy refilling it
            const uint32_t bytes = static_cast<uint32_t>(len) * E::BYTES;
            mbar_arrive_expect_tx(&full[islot], bytes);
            // evict-first where this is the logits' last read; target rows and re-read drafter pieces stay
            const bool last = it_u.kind == 2 || (it_u.kind == 1 && it_k < G_CAP);
            bulk_load(ring + static_cast<size_t>(islot) * G_PIECE_BYTES, it_u.row + static_cast<size_t>(pc) * G_PIECE_BYTES,
                      bytes, &full[islot], last ? pol_first : pol_normal);
            ++copies;
        }
        ++issued;
        if (++islot == G_R) islot = 0;
        if (++it_k == nmine) {
            it_k = 0;
            if (++it_t < S) it_u = unit_of(it_t);
        }
    };
    if (p.tma)
        for (int q = 0; q < G_R && issued < total; ++q) issue();
    int cslot = 0;
    uint32_t cpar = 0;
    bool ok = true;

    GUnit prev = it_u;   // unit s - 1 (valid from step 1 on)
    float pend_bt = 0.f, pend_bd = 0.f;   // log2 offsets of unit s - 1 when it is a D unit
    float bt_item = 0.f;                  // log2 offset of the latest T unit's row
    for (long long s = 0; s <= S; ++s) {
        const bool has1 = s < S;
        const GUnit cur = has1 ? unit_of(s) : prev;
        const bool has2 = s >= 1 && prev.kind == 1;
        float m = NINF, sm = 0.f;
        float2 acc = make_float2(0.f, 0.f);
        for (int k = 0; k < nmine; ++k) {
            const int pc = warp + GW * k;
            const int len = min(PEG, V - pc * PEG);
            const size_t poff = static_cast<size_t>(pc) * G_PIECE_BYTES;
            if (has2) {   // pass 2 of unit s - 1: the target piece from L2, the drafter piece from tensor memory
                Raw rt[NCH], rd[NCH];
                if (p.tma) {
#pragma unroll
                    for (int q = 0; q < NCH; ++q) rt[q] = GPiece<E>::ld_keep(prev.trow + poff, (lane + 32 * q) * CHUNK, len);
                } else {
#pragma unroll
                    for (int q = 0; q < NCH; ++q) rt[q] = E::template gload<false>(prev.trow + poff, (lane + 32 * q) * CHUNK, len);
                }
                if (k < G_CAP) {
                    uint32_t w[32];
                    tmem_ld32(twarp + 32 * k, w);
                    GPiece<E>::from_words(w, rd);
                } else if (p.tma) {
#pragma unroll
                    for (int q = 0; q < NCH; ++q) rd[q] = E::template gload<true>(prev.row + poff, (lane + 32 * q) * CHUNK, len);
                } else {
#pragma unroll
                    for (int q = 0; q < NCH; ++q) rd[q] = E::template gload<false>(prev.row + poff, (lane + 32 * q) * CHUNK, len);
                }
                g_overlap<E>(rt, rd, c, pend_bt, pend_bd, acc);
            }
            if (has1) {   // pass 1 of unit s
                Raw r1[NCH];
                if (p.tma) {
                    if (ok) ok = mbar_wait_bounded(&full[cslot], cpar, p.status, STATUS_TIMEOUT, WAIT_LIMIT_NS);
                    if (lane == 0 && !ok) issuing = false;
                    const int nch = (len + CHUNK - 1) / CHUNK;
                    const unsigned char* slot = ring + static_cast<size_t>(cslot) * G_PIECE_BYTES;
#pragma unroll
                    for (int q = 0; q < NCH; ++q) {
                        const int kk = lane + 32 * q;
                        r1[q] = kk < nch ? E::lds(slot, kk) : E::ninf();
                    }
                    __syncwarp();
                    if (++cslot == G_R) {
                        cslot = 0;
                        cpar ^= 1u;
                    }
                    if (issued < total) issue();
                } else {
#pragma unroll
                    for (int q = 0; q < NCH; ++q) r1[q] = E::template gload<false>(cur.row + poff, (lane + 32 * q) * CHUNK, len);
                }
                if (cur.kind == 1 && k < G_CAP) {   // park the drafter piece (its columns were read above)
                    uint32_t w[32];
                    GPiece<E>::to_words(r1, w);
                    tmem_st32(twarp + 32 * k, w);
                }
                g_stats<E>(r1, c, m, sm);
            }
        }
        if (has1) {
            const MaxSum w = warp_ms(MaxSum{m, sm}, c);
            if (lane == 0) s_ms[s & 1][warp] = make_float2(w.m, w.s);
            if (cur.kind == 1) tmem_wait_st();
        }
        if (has2) {
            const float g = warp_sum(acc.x + acc.y);
            if (lane == 0) s_g[s & 1][warp] = g;
        }
        __syncthreads();
        if (has2 && warp == GW - 1) {   // gamma of unit s - 1: the 16 partials in warp order
            const float g = warp_sum(lane < GW ? s_g[s & 1][lane] : 0.f);
            if (lane == 0) {
                const size_t o = (static_cast<size_t>(prev.i) * p.B + prev.b) * p.K + prev.j;
                p.gamma[o] = g;
                if (p.loss) p.loss[o] = 1.f - g;
            }
        }
        if (has1) {   // the row's (max, sum): the 16 warp pairs merged in warp order, the same in every warp
            const float2 v = lane < GW ? s_ms[s & 1][lane] : make_float2(NINF, 0.f);
            const MaxSum r = warp_ms(MaxSum{v.x, v.y}, c);
            const float beta = beta_of(r, c);
            if (cur.kind == 1) {
                pend_bt = bt_item;
                pend_bd = beta;
            } else if (cur.kind == 0) {
                bt_item = beta;
            }
            if (p.row_ms && warp == 0 && lane == 0) {
                long long ri = -1;
                if (cur.kind != 1) ri = static_cast<long long>(cur.b) * (p.K + 1) + cur.j;
                else if (cur.i == p.selected)
                    ri = static_cast<long long>(p.B) * (p.K + 1) + static_cast<long long>(cur.b) * p.K + cur.j;
                if (ri >= 0) p.row_ms[ri] = make_float2(r.m, r.s);
            }
        }
        prev = cur;
    }

    // after a failed wait, copies may still be in flight: they must land before the CTA may exit
    if (p.tma && lane == 0 && !issuing) {
        for (long long q = copies - G_R > 0 ? copies - G_R : 0; q < copies; ++q)
            mbar_wait_bounded(&full[q % G_R], static_cast<uint32_t>((q / G_R) & 1), p.status, STATUS_TIMEOUT, WAIT_LIMIT_NS);
    }
    __syncwarp();
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(G_TMEM_COLS) : "memory");
}

}  // namespace specv
