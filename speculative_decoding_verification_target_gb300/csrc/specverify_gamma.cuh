// Counterfactual acceptance for N drafters, gamma[i, b, j] = sum_x min(p_target(x), q_i(x)), with the loss
// 1 - gamma ("Not-a-Bandit: Provably No-Regret Drafter Selection in Speculative Decoding for LLMs", Key
// design 1 and 3; the identity sum min(p, q) = 1 - TV(p, q) is the lossless tutorial's §6.3-§6.4).
//
// Every term needs both rows' normalisers, so each drafter row is visited twice: once for its (max, sum
// of exponentials) and once for the sum of minima. gamma_kernel reads every logit from HBM once and keeps
// the second visit on chip:
//   - a CTA owns a contiguous run of "units" in the order T(b, j), D_0(b, j), ..., D_{N-1}(b, j) for every
//     position, then the bonus target rows T(b, K) when a chain is verified as well. A T unit computes the
//     target row's normaliser; a D unit computes the drafter row's normaliser and then its gamma. The runs
//     hold equal numbers of units. A CTA whose run starts inside a position first computes that position's
//     T unit itself;
//   - a whole row is split over the CTA's 16 warps (warp w takes pieces w, w + 16, ...), so the normaliser
//     of a row is complete once every warp has published its pair: no exchange between CTAs;
//   - pass 1 streams the pieces of unit s from HBM through a private ring of bulk-copy slots per warp.
//     Each warp parks the raw logits of its first two drafter pieces in tensor memory, in one of two halves
//     of its 32 lanes x 128 columns (unit s uses half s mod 2);
//   - pass 2 of unit s - 1 runs in the same step, after pass 1 of unit s: it reads the parked drafter
//     pieces back from tensor memory, reads the target piece from L2 (the CTA keeps one target row hot
//     while it walks that position's drafters) and adds sum 2^min(log2 p_target, log2 q_i). Pieces past the
//     tensor-memory share are re-read from L2.
// The warps publish their (max, sum) of a unit and their gamma partials of a unit with mbarrier arrivals,
// and wait for the other warps' a whole pass later; each merge runs in warp order, so the result does not
// depend on timing.
#pragma once
#include "specverify_chain.cuh"

namespace specv {

constexpr int GW = 16;                       // warps per CTA
constexpr int GNT = GW * 32;
constexpr int G_PIECE_BYTES = 4096;          // one bulk copy: 2048 bf16 or 1024 fp32 logits
constexpr int G_R = 3;                       // ring slots per warp
constexpr int G_CAP = 4;                     // pieces of a warp's tensor-memory share (32 columns each)
constexpr int G_HALF = G_CAP / 2;            // pieces of one unit parked (the share is double buffered)
constexpr int G_TMEM_COLS = 512;
constexpr size_t G_SMEM = static_cast<size_t>(GW) * G_R * G_PIECE_BYTES + static_cast<size_t>(GW) * G_R * 8;

struct CgParams {
    const unsigned char* target;     // [B, K+1, V]
    const unsigned char* drafters;   // [N, B, K, V]
    int B, K, V, N;
    int np;                          // pieces per row
    long long U;                     // units in all (< 2^31)
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

// A CTA's run of units, walked in order with no division per step. Unit u < B K (N + 1) is position
// (b, j) = divmod(u / (N + 1), K) with k = u mod (N + 1): k = 0 the T unit, else the D unit of drafter k - 1;
// unit u >= B K (N + 1) is the bonus row of sequence u - B K (N + 1). A run that starts inside a position
// (k > 0) is preceded by that position's T unit.
struct UnitSeq {
    int b, j, k;       // position and unit within it (k = N + 1 marks the bonus row of sequence b)
    int t;             // index in the run

    __device__ void set(const CgParams& p, int u) {
        const int nd = p.B * p.K * (p.N + 1);
        if (u < nd) {
            const int item = u / (p.N + 1);
            k = u - item * (p.N + 1);
            b = item / p.K;
            j = item - b * p.K;
        } else {
            b = u - nd;
            j = p.K;
            k = p.N + 1;
        }
    }
    // the run starting at unit u0; true when it starts inside a position (its T unit is inserted first)
    __device__ bool start(const CgParams& p, int u0) {
        t = 0;
        set(p, u0);
        const bool pre = k > 0 && k <= p.N;
        if (pre) k = 0;
        return pre;
    }
    __device__ void next(const CgParams& p, bool pre, int u0) {
        ++t;
        if (t == 1 && pre) {
            set(p, u0);
            return;
        }
        if (k == p.N + 1) {   // bonus rows follow one another
            ++b;
            return;
        }
        if (++k == p.N + 1) {
            k = 0;
            if (++j == p.K) {
                j = 0;
                if (++b == p.B) {   // past the last position: the bonus rows
                    b = 0;
                    j = p.K;
                    k = p.N + 1;
                }
            }
        }
    }
    __device__ int kind(const CgParams& p) const { return k == 0 ? 0 : (k == p.N + 1 ? 2 : 1); }
    __device__ int drafter() const { return k - 1; }
    __device__ const unsigned char* trow(const CgParams& p, size_t row_bytes) const {
        return p.target + (static_cast<size_t>(b) * (p.K + 1) + j) * row_bytes;
    }
    // the row pass 1 reads
    __device__ const unsigned char* row(const CgParams& p, size_t row_bytes) const {
        if (k == 0 || k == p.N + 1) return trow(p, row_bytes);
        return p.drafters + ((static_cast<size_t>(k - 1) * p.B + b) * p.K + j) * row_bytes;
    }
};

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
    // one chunk from global memory through the read-only path, no L1 allocation, L2 eviction policy `pol`;
    // chunks at or past n_el are -inf (ld_full: the chunk is known to be in range)
    __device__ static Bf16::Raw ld_keep(const unsigned char* row, int e0, int n_el, uint64_t pol) {
        uint4 v = Bf16::ninf();
        const uint4* ptr = reinterpret_cast<const uint4*>(row) + e0 / CHUNK;
        asm volatile(
            "{\n\t.reg .pred q;\n\tsetp.lt.s32 q, %4, %5;\n\t"
            "@q ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%6], %7;\n\t}"
            : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)
            : "r"(e0), "r"(n_el), "l"(ptr), "l"(pol));
        return v;
    }
    __device__ static Bf16::Raw ld_full(const unsigned char* row, int e0, uint64_t pol) {
        uint4 v;
        const uint4* ptr = reinterpret_cast<const uint4*>(row) + e0 / CHUNK;
        asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "l"(ptr), "l"(pol));
        return v;
    }
    // the piece's 32 words to / from this thread's lane, columns [taddr, taddr + 32)
    __device__ static void tmem_st(uint32_t taddr, const Bf16::Raw (&r)[NCH]) {
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
            "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
            "r"(r[0].x), "r"(r[0].y), "r"(r[0].z), "r"(r[0].w), "r"(r[1].x), "r"(r[1].y), "r"(r[1].z), "r"(r[1].w),
            "r"(r[2].x), "r"(r[2].y), "r"(r[2].z), "r"(r[2].w), "r"(r[3].x), "r"(r[3].y), "r"(r[3].z), "r"(r[3].w),
            "r"(r[4].x), "r"(r[4].y), "r"(r[4].z), "r"(r[4].w), "r"(r[5].x), "r"(r[5].y), "r"(r[5].z), "r"(r[5].w),
            "r"(r[6].x), "r"(r[6].y), "r"(r[6].z), "r"(r[6].w), "r"(r[7].x), "r"(r[7].y), "r"(r[7].z), "r"(r[7].w)
            : "memory");
    }
    __device__ static void tmem_ld(uint32_t taddr, Bf16::Raw (&r)[NCH]) {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
            "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
            "tcgen05.wait::ld.sync.aligned;"
            : "=r"(r[0].x), "=r"(r[0].y), "=r"(r[0].z), "=r"(r[0].w), "=r"(r[1].x), "=r"(r[1].y), "=r"(r[1].z),
              "=r"(r[1].w), "=r"(r[2].x), "=r"(r[2].y), "=r"(r[2].z), "=r"(r[2].w), "=r"(r[3].x), "=r"(r[3].y),
              "=r"(r[3].z), "=r"(r[3].w), "=r"(r[4].x), "=r"(r[4].y), "=r"(r[4].z), "=r"(r[4].w), "=r"(r[5].x),
              "=r"(r[5].y), "=r"(r[5].z), "=r"(r[5].w), "=r"(r[6].x), "=r"(r[6].y), "=r"(r[6].z), "=r"(r[6].w),
              "=r"(r[7].x), "=r"(r[7].y), "=r"(r[7].z), "=r"(r[7].w)
            : "r"(taddr)
            : "memory");
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
    __device__ static void tmem_st(uint32_t taddr, const F32::Raw (&r)[NCH]) {
        uint32_t w[32];
        to_words(r, w);
        tmem_st32(taddr, w);
    }
    __device__ static void tmem_ld(uint32_t taddr, F32::Raw (&r)[NCH]) {
        uint32_t w[32];
        tmem_ld32(taddr, w);
        from_words(w, r);
    }
    __device__ static F32::Raw ld_keep(const unsigned char* row, int e0, int n_el, uint64_t pol) {
        F32::Raw v = F32::ninf();
        const float* ptr = reinterpret_cast<const float*>(row) + e0;
        asm volatile(
            "{\n\t.reg .pred q;\n\tsetp.lt.s32 q, %8, %9;\n\t"
            "@q ld.global.nc.L1::no_allocate.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%10], %11;\n\t"
            "@q ld.global.nc.L1::no_allocate.L2::cache_hint.v4.f32 {%4, %5, %6, %7}, [%10+16], %11;\n\t}"
            : "+f"(v.a.x), "+f"(v.a.y), "+f"(v.a.z), "+f"(v.a.w), "+f"(v.b.x), "+f"(v.b.y), "+f"(v.b.z), "+f"(v.b.w)
            : "r"(e0), "r"(n_el), "l"(ptr), "l"(pol));
        return v;
    }
    __device__ static F32::Raw ld_full(const unsigned char* row, int e0, uint64_t pol) {
        F32::Raw v;
        const float* ptr = reinterpret_cast<const float*>(row) + e0;
        asm volatile(
            "ld.global.nc.L1::no_allocate.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%8], %9;\n\t"
            "ld.global.nc.L1::no_allocate.L2::cache_hint.v4.f32 {%4, %5, %6, %7}, [%8+16], %9;"
            : "=f"(v.a.x), "=f"(v.a.y), "=f"(v.a.z), "=f"(v.a.w), "=f"(v.b.x), "=f"(v.b.y), "=f"(v.b.z), "=f"(v.b.w)
            : "l"(ptr), "l"(pol));
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
// The gamma kernel's work on one CTA (all GNT threads): its run of units, then the release of its tensor
// memory.
template <class E>
__device__ __forceinline__ void gamma_body(const CgParams& p) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint32_t s_tmem;
    __shared__ float2 s_ms[4][GW];   // per unit u (mod 4): the warps' (max, sum) of its row
    __shared__ float s_g[4][GW];     // per unit u (mod 4): the warps' gamma partials
    __shared__ uint64_t s_bar_a[2];  // per unit parity: every warp has stored its (max, sum) of unit u
    __shared__ uint64_t s_bar_g[2];  // per unit parity: every warp has stored its gamma partial of unit u
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
    if (threadIdx.x == 0) {
        for (int q = 0; q < 2; ++q) {
            mbar_init(&s_bar_a[q], GW);
            mbar_init(&s_bar_g[q], GW);
        }
        fence_mbarrier_init_cluster();
    }
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    const uint32_t tbase = s_tmem;
    // this warp's columns: lanes 32 (warp mod 4) .. + 31, columns 128 (warp / 4) .. + 127, as two halves of
    // G_HALF pieces: unit u parks its first G_HALF pieces in half u mod 2
    const uint32_t twarp = tbase + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + static_cast<uint32_t>((warp >> 2) * G_CAP * 32);
    auto tcol = [&](int u, int k) -> uint32_t { return twarp + static_cast<uint32_t>(((u & 1) * G_HALF + k) * 32); };

    // this CTA's run of units (the host checks that U fits in 31 bits)
    const int u0 = static_cast<int>(static_cast<long long>(blockIdx.x) * p.U / p.G);
    const int u1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * p.U / p.G);
    UnitSeq first;
    const bool pre = first.start(p, u0);
    const int S = (u1 - u0) + (pre ? 1 : 0);
    const int nmine = warp < np ? (np - 1 - warp) / GW + 1 : 0;   // pieces warp, warp + 16, ... of a row

    // ---- ring of pass-1 pieces: the issue walker runs G_R bulk copies ahead of use. Pass 2 reads the target
    // piece (and a drafter piece past the tensor-memory share) straight from L2 into registers. ----
    const uint64_t pol_first = policy_evict_first(), pol_normal = policy_evict_normal(), pol_last = policy_evict_last();
    UnitSeq iu = first;   // the walker's unit
    int it_k = 0;
    const unsigned char* it_row = iu.row(p, row_bytes);
    int it_kind = iu.kind(p);
    const long long total = p.tma ? static_cast<long long>(S) * nmine : 0;
    long long issued = 0, copies = 0;
    int islot = 0;
    bool issuing = true;
    auto issue = [&]() {
        if (issued >= total) return;
        const int pc = warp + GW * it_k;
        const int len = min(PEG, V - pc * PEG);
        if (lane == 0 && issuing) {
            fence_proxy_async_shared();   // the warp's reads of this slot come before the copy refilling it
            const uint32_t bytes = static_cast<uint32_t>(len) * E::BYTES;
            mbar_arrive_expect_tx(&full[islot], bytes);
            // evict-first where this is the logits' last read (bonus rows, drafter pieces parked in tensor
            // memory); evict-last for a position's target row, which its drafters' pass 2 reads again, and for
            // the drafter pieces pass 2 re-reads from L2
            const uint64_t pol = it_kind == 0 ? pol_last : ((it_kind == 2 || it_k < G_HALF) ? pol_first : pol_last);
            bulk_load(ring + static_cast<size_t>(islot) * G_PIECE_BYTES, it_row + static_cast<size_t>(pc) * G_PIECE_BYTES,
                      bytes, &full[islot], pol);
            ++copies;
        }
        ++issued;
        if (++islot == G_R) islot = 0;
        if (++it_k == nmine) {
            it_k = 0;
            iu.next(p, pre, u0);
            if (iu.t < S) {
                it_row = iu.row(p, row_bytes);
                it_kind = iu.kind(p);
            }
        }
    };
    for (int q = 0; q < G_R; ++q) issue();
    int cslot = 0;
    uint32_t cpar = 0;
    bool ok = true;
    // the next piece of the ring into registers (chunks past len are -inf), then its slot is refilled
    auto take = [&](Raw (&r)[NCH], int len) {
        if (ok) ok = mbar_wait_bounded(&full[cslot], cpar, p.status, STATUS_TIMEOUT, WAIT_LIMIT_NS);
        if (lane == 0 && !ok) issuing = false;
        const unsigned char* slot = ring + static_cast<size_t>(cslot) * G_PIECE_BYTES;
        if (len == PEG) {
#pragma unroll
            for (int q = 0; q < NCH; ++q) r[q] = E::lds(slot, lane + 32 * q);
        } else {
            const int nch = (len + CHUNK - 1) / CHUNK;
#pragma unroll
            for (int q = 0; q < NCH; ++q) {
                const int kk = lane + 32 * q;
                r[q] = kk < nch ? E::lds(slot, kk) : E::ninf();
            }
        }
        __syncwarp();
        if (++cslot == G_R) {
            cslot = 0;
            cpar ^= 1u;
        }
        issue();
    };
    // element-wise loads of a piece (rows of any alignment; the unit geometry is recomputed here, off the
    // bulk-copy path)
    auto gather = [&](Raw (&r)[NCH], const unsigned char* row, size_t poff, int len) {
        const unsigned char* piece = row + poff;
#pragma unroll
        for (int q = 0; q < NCH; ++q) r[q] = E::template gload<false>(piece, (lane + 32 * q) * CHUNK, len);
    };

    // Step t: pass 1 of unit t, whose (max, sum) pairs are published with an arrival on s_bar_a; then the
    // wait for every warp's pass 1 of unit t - 1, its row statistics, and (a D unit) its pass 2, published on
    // s_bar_g; the last warp sums unit t - 2's gamma partials. A warp waits for the others only a whole pass
    // after it published, so the warps need not run in step. Every unit arrives on both barriers, so a
    // barrier's phase parity is the unit index / 2 mod 2; a warp can reach unit u + 2's arrival only after
    // unit u's phase completed, and the shared slots (unit mod 4) are rewritten only after every warp read them.
    float pend_bt = 0.f, pend_bd = 0.f;   // log2 offsets of the D unit whose pass 2 runs in this step
    float bt_item = 0.f;                  // log2 offset of the latest T unit's row
    size_t gidx1 = 0, gidx2 = 0;          // gamma index of units t - 1 and t - 2 (D units)
    int kind1 = -1, kind2 = -1;           // kinds of units t - 1 and t - 2
    const unsigned char* prev_trow = nullptr;   // rows of unit t - 1
    const unsigned char* prev_row = nullptr;
    bool prev_last = false;
    bool okb = true;                      // every barrier wait so far succeeded
    UnitSeq cu = first;                   // unit t
    UnitSeq pu = first;                   // unit t - 1
    auto sum_gamma = [&](int u, size_t gidx) {   // the last warp: unit u's 16 partials in warp order
        if (okb) okb = mbar_wait_bounded(&s_bar_g[u & 1], static_cast<uint32_t>((u >> 1) & 1), p.status, STATUS_TIMEOUT, WAIT_LIMIT_NS);
        const float g = warp_sum(lane < GW ? s_g[u & 3][lane] : 0.f);
        if (lane == 0) {
            p.gamma[gidx] = g;
            if (p.loss) p.loss[gidx] = 1.f - g;
        }
    };
    for (int t = 0; t <= S; ++t) {
        const int kind0 = t < S ? cu.kind(p) : -1;
        // ---- pass 1 of unit t ----
        if (t < S) {
            const unsigned char* cur_row = p.tma ? nullptr : cu.row(p, row_bytes);
            float m = NINF, sm = 0.f;
            for (int k = 0; k < nmine; ++k) {
                const int pc = warp + GW * k;
                const int len = min(PEG, V - pc * PEG);
                Raw r1[NCH];
                if (p.tma) take(r1, len);
                else gather(r1, cur_row, static_cast<size_t>(pc) * G_PIECE_BYTES, len);
                if (kind0 == 1 && k < G_HALF) GPiece<E>::tmem_st(tcol(t, k), r1);
                g_stats<E>(r1, c, m, sm);
            }
            const MaxSum w = warp_ms(MaxSum{m, sm}, c);
            if (lane == 0) s_ms[t & 3][warp] = make_float2(w.m, w.s);
            if (kind0 == 1) tmem_wait_st();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_bar_a[t & 1]);
        }
        // ---- unit t - 1: its row statistics, then its pass 2 ----
        if (t >= 1) {
            const int u = t - 1;
            if (okb) okb = mbar_wait_bounded(&s_bar_a[u & 1], static_cast<uint32_t>((u >> 1) & 1), p.status, STATUS_TIMEOUT, WAIT_LIMIT_NS);
            // the row's (max, sum): the 16 warp pairs merged in warp order, the same in every warp
            const float2 v = lane < GW ? s_ms[u & 3][lane] : make_float2(NINF, 0.f);
            const MaxSum r = warp_ms(MaxSum{v.x, v.y}, c);
            const float beta = beta_of(r, c);
            if (kind1 == 0) {
                bt_item = beta;
            } else if (kind1 == 1) {
                pend_bt = bt_item;
                pend_bd = beta;
            }
            if (p.row_ms && warp == 0 && lane == 0) {
                long long ri = -1;
                if (kind1 != 1) ri = static_cast<long long>(pu.b) * (p.K + 1) + pu.j;
                else if (pu.drafter() == p.selected)
                    ri = static_cast<long long>(p.B) * (p.K + 1) + static_cast<long long>(pu.b) * p.K + pu.j;
                if (ri >= 0) p.row_ms[ri] = make_float2(r.m, r.s);
            }
            float2 acc = make_float2(0.f, 0.f);
            if (kind1 == 1) {   // pass 2: the target piece from L2, the drafter piece from tensor memory or L2
                for (int k = 0; k < nmine; ++k) {
                    const int pc = warp + GW * k;
                    const int len = min(PEG, V - pc * PEG);
                    const size_t poff = static_cast<size_t>(pc) * G_PIECE_BYTES;
                    Raw rt[NCH], rd[NCH];
                    if (p.tma) {
                        // the target row stays in L2 for the position's next drafter; the last one lets it go
                        const uint64_t tpol = prev_last ? pol_first : pol_last;
                        const unsigned char* tp = prev_trow + poff;
                        if (len == PEG) {
#pragma unroll
                            for (int q = 0; q < NCH; ++q) rt[q] = GPiece<E>::ld_full(tp, (lane + 32 * q) * CHUNK, tpol);
                        } else {
#pragma unroll
                            for (int q = 0; q < NCH; ++q)
                                rt[q] = GPiece<E>::ld_keep(tp, (lane + 32 * q) * CHUNK, len, tpol);
                        }
                    } else {
                        gather(rt, prev_trow, poff, len);
                    }
                    if (k < G_HALF) {
                        GPiece<E>::tmem_ld(tcol(u, k), rd);
                    } else if (p.tma) {
#pragma unroll
                        for (int q = 0; q < NCH; ++q)
                            rd[q] = E::template gload<true>(prev_row + poff, (lane + 32 * q) * CHUNK, len);
                    } else {
                        gather(rd, prev_row, poff, len);
                    }
                    g_overlap<E>(rt, rd, c, pend_bt, pend_bd, acc);
                }
                const float g = warp_sum(acc.x + acc.y);
                if (lane == 0) s_g[u & 3][warp] = g;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_bar_g[u & 1]);
        }
        // ---- unit t - 2's gamma (its partials were published one step ago) ----
        if (warp == GW - 1 && t >= 2 && kind2 == 1) sum_gamma(t - 2, gidx2);
        // ---- move the unit window ----
        kind2 = kind1;
        gidx2 = gidx1;
        if (t < S) {
            kind1 = kind0;
            pu = cu;
            if (kind0 == 1) {
                const int i = cu.drafter();
                gidx1 = (static_cast<size_t>(i) * p.B + cu.b) * p.K + cu.j;
                prev_trow = cu.trow(p, row_bytes);
                prev_row = cu.row(p, row_bytes);
                prev_last = i == p.N - 1;
            }
            cu.next(p, pre, u0);
        }
    }
    // unit S - 1's gamma (published in the last step)
    if (warp == GW - 1 && kind2 == 1 && S >= 1) sum_gamma(S - 1, gidx2);

    // after a failed wait, copies may still be in flight: they must land before the CTA may exit
    if (p.tma && lane == 0 && !issuing) {
        for (long long q = copies - G_R > 0 ? copies - G_R : 0; q < copies; ++q)
            mbar_wait_bounded(&full[q % G_R], static_cast<uint32_t>((q / G_R) & 1), p.status, STATUS_TIMEOUT, WAIT_LIMIT_NS);
    }
    if (p.tma && lane == 0)   // the ring's memory may be reused after this (the one-launch kernel's draw)
        for (int q = 0; q < G_R; ++q) mbar_inval(&full[q]);
    __syncwarp();
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(G_TMEM_COLS) : "memory");
}

template <class E>
__global__ void __launch_bounds__(GNT, 1) gamma_kernel(const __grid_constant__ CgParams p) {
    gamma_body<E>(p);
}

// ---------------------------------------- one launch: gamma, then the chain ----------------------------------------
// The counterfactual call with a selected drafter as a single cooperative launch: every CTA runs its gamma
// units, a grid barrier makes every row's (max, sum) visible, and then CTA g draws sequences g, g + G, ...
// with the draw kernel's arithmetic (one CTA per sequence), its state placed in the dynamic shared memory
// that the gamma phase no longer uses.
struct FuseParams {
    CgParams g;
    DParams d;
    unsigned* bar;   // [0] arrivals (0 between uses), [1] generation: the grid barrier's words
};

// The DrawShared block sits at the top of the gamma kernel's dynamic shared memory, above the draw's
// bulk-copy slots (bf16 rows) at its bottom.
template <class E>
__host__ __device__ constexpr size_t fused_draw_shared_off() {
    return (G_SMEM - sizeof(DrawShared<E>)) / 128 * 128;
}
constexpr size_t FUSED_DRAW_RING = static_cast<size_t>(DW) * (2 * static_cast<size_t>(PE) * 2 + sizeof(uint64_t));
static_assert(GNT == DNT, "the draw phase runs on the gamma kernel's threads");
static_assert(FUSED_DRAW_RING <= fused_draw_shared_off<Bf16>(), "bf16 draw slots and DrawShared overlap");
static_assert(sizeof(DrawShared<F32>) <= G_SMEM, "DrawShared does not fit the gamma kernel's shared memory");

// A barrier across every CTA of a cooperative launch: thread 0 of each CTA arrives on bar[0]; the last to
// arrive resets it and advances the generation bar[1], which the others wait for (sleeping between polls).
// Writes before it are visible to reads after it. A wait that outlasts WAIT_LIMIT_NS sets STATUS_TIMEOUT and
// gives up (the results are then invalid).
__device__ __forceinline__ void grid_barrier(unsigned* bar, unsigned n, unsigned* status) {
    __syncthreads();
    if (threadIdx.x == 0) {
        volatile unsigned* gen = bar + 1;
        const unsigned g0 = *gen;
        __threadfence();
        if (atomicAdd(bar, 1u) == n - 1) {
            atomicExch(bar, 0u);
            __threadfence();
            atomicAdd(bar + 1, 1u);
        } else {
            const uint64_t t0 = global_timer_ns();
            for (int it = 0; *gen == g0; ++it) {
                __nanosleep(128);
                if ((it & 63) == 63 && global_timer_ns() - t0 > WAIT_LIMIT_NS) {
                    atomicOr(status, STATUS_TIMEOUT);
                    break;
                }
            }
        }
        __threadfence();
    }
    __syncthreads();
}

// The draw phase out of line, so that its registers do not crowd the gamma phase's allocation.
template <class E>
__device__ __noinline__ void fused_draws(const DParams& d, DrawShared<E>& S, unsigned char* smem) {
    for (int b = static_cast<int>(blockIdx.x); b < d.B; b += static_cast<int>(gridDim.x)) {
        draw_body<E, true, false>(d, S, smem, b);
        __syncthreads();   // the next sequence's draw reuses the slots and the DrawShared block
    }
}

template <class E>
__global__ void __launch_bounds__(GNT, 1) gamma_chain_kernel(const __grid_constant__ FuseParams f) {
    gamma_body<E>(f.g);
    grid_barrier(f.bar, gridDim.x, f.g.status);
    extern __shared__ __align__(128) unsigned char smem[];
    fused_draws<E>(f.d, *reinterpret_cast<DrawShared<E>*>(smem + fused_draw_shared_off<E>()), smem);
}

// ------------------------------------------------------------------------------------------------
// accept-length estimate
// ------------------------------------------------------------------------------------------------
// HedgeSpec's accept-length estimate from the counterfactual gamma ("Not-a-Bandit ...", Key design 2 and
// 3; the page's displays are missing, reading: est = 1 + sum_{k=1..K} prod_{j<=k} gamma_j, loss =
// K + 1 - est): one thread per (drafter, sequence), gamma [N, B, K] read in order.
__global__ void __launch_bounds__(256) accept_length_kernel(const float* __restrict__ gamma, long long rows, int K,
                                                            float* __restrict__ est, float* __restrict__ loss) {
    const long long r = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (r >= rows) return;
    const float* g = gamma + r * K;
    float run = 1.f, total = 1.f;
    for (int k = 0; k < K; ++k) {
        run *= __ldg(g + k);
        total += run;
    }
    est[r] = total;
    if (loss) loss[r] = static_cast<float>(K + 1) - total;
}

// ------------------------------------------------------------------------------------------------
// NormalHedge
// ------------------------------------------------------------------------------------------------
// One NormalHedge round (Chaudhuri, Freund, Hsu, "A parameter-free hedging algorithm", NIPS 2009), the
// learner the HedgeSpec notes name for drafter selection ("Not-a-Bandit ...", Key design 3); the pages
// state no update rule. The learner played weights p over N <= 64 experts and saw losses l: the regret to
// expert i grows by (p . l) - l_i, and the new weights are p_i proportional to ([R_i]+ / c)
// exp([R_i]+^2 / (2 c)), where c solves (1/N) sum_i exp([R_i]+^2 / (2 c)) = e (uniform weights when no
// regret is positive). One warp; lane l holds experts l and l + 32. c lies in [m^2 / (2 ln(N e)), m^2 / 2]
// for the largest positive regret m (all exponents below 1 above that bracket, the largest alone above
// e N below it), found by bisection on log c with the mean taken as a log-sum-exp.
__device__ __forceinline__ float nh_log_mean(float a0, float a1, bool v0, bool v1, int N) {
    const float NINF = __uint_as_float(0xFF800000u);
    const float mx = warp_max(fmaxf(v0 ? a0 : NINF, v1 ? a1 : NINF));
    const float s = warp_sum((v0 ? expf(a0 - mx) : 0.f) + (v1 ? expf(a1 - mx) : 0.f));
    return mx + logf(s / static_cast<float>(N));
}

// One NormalHedge round on the registers of one warp: lane l holds experts l (valid v0) and l + 32 (v1), their
// regrets r0, r1 and weights p0, p1; l0, l1 are this round's losses. Every lane ends with the new state.
__device__ __forceinline__ void nh_round(int N, bool v0, bool v1, float l0, float l1, float& r0, float& r1,
                                         float& p0, float& p1) {
    const float lp = warp_sum((v0 ? p0 * l0 : 0.f) + (v1 ? p1 * l1 : 0.f));
    r0 = v0 ? r0 + (lp - l0) : 0.f;
    r1 = v1 ? r1 + (lp - l1) : 0.f;
    const float q0 = fmaxf(r0, 0.f), q1 = fmaxf(r1, 0.f);
    const float m = warp_max(fmaxf(q0, q1));
    if (!(m > 0.f)) {
        const float u = 1.f / static_cast<float>(N);
        p0 = v0 ? u : 0.f;
        p1 = v1 ? u : 0.f;
        return;
    }
    const float lm2 = 2.f * logf(m);
    float lo = lm2 - logf(2.f * (logf(static_cast<float>(N)) + 1.f)), hi = lm2 - logf(2.f);
    for (int it = 0; it < 48; ++it) {
        const float mid = 0.5f * (lo + hi);
        const float c = expf(mid);
        if (nh_log_mean(q0 * q0 / (2.f * c), q1 * q1 / (2.f * c), v0, v1, N) > 1.f) lo = mid;
        else hi = mid;
    }
    const float c = expf(0.5f * (lo + hi));
    const float NINF = __uint_as_float(0xFF800000u);
    const float w0 = (v0 && q0 > 0.f) ? logf(q0 / c) + q0 * q0 / (2.f * c) : NINF;
    const float w1 = (v1 && q1 > 0.f) ? logf(q1 / c) + q1 * q1 / (2.f * c) : NINF;
    const float mx = warp_max(fmaxf(w0, w1));
    const float e0 = w0 > NINF ? expf(w0 - mx) : 0.f, e1 = w1 > NINF ? expf(w1 - mx) : 0.f;
    const float sum = warp_sum(e0 + e1);
    p0 = e0 / sum;
    p1 = e1 / sum;
}

__global__ void __launch_bounds__(32) normalhedge_kernel(float* __restrict__ regret, const float* __restrict__ loss,
                                                         float* __restrict__ weights, int N) {
    const int lane = threadIdx.x;
    const bool v0 = lane < N, v1 = lane + 32 < N;
    float p0 = v0 ? weights[lane] : 0.f, p1 = v1 ? weights[lane + 32] : 0.f;
    const float l0 = v0 ? loss[lane] : 0.f, l1 = v1 ? loss[lane + 32] : 0.f;
    float r0 = v0 ? regret[lane] : 0.f, r1 = v1 ? regret[lane + 32] : 0.f;
    nh_round(N, v0, v1, l0, l1, r0, r1, p0, p1);
    if (v0) {
        regret[lane] = r0;
        weights[lane] = p0;
    }
    if (v1) {
        regret[lane + 32] = r1;
        weights[lane + 32] = p1;
    }
}

// ------------------------------------------------------------------------------------------------
// NormalHedge under delayed, censored feedback
// ------------------------------------------------------------------------------------------------
// "Not-a-Bandit ...", Key design 3: the accepted tokens of a round are revealed as one block when it ends,
// the counterfactual feedback is censored unless the selected drafter fills the chunk, the loss is 1 - gamma or
// the accept length still available up to K + 1, the delay is at most 2K, and the learner keeps a queue of
// feedback and keeps applying the next available one (the stochastic-setting reduction of Joulani, Gyorgy,
// Szepesvari, ICML 2013). Reading (one learner per sequence): round t reveals levels j < min(L_t + 1, K) of its
// gamma [N, K], in level order, as the sequence's next feedback items; the later levels are censored and
// skipped. Objective 0: item n's loss 1 - gamma is available at once. Objective 1: item n's loss is K + 1 minus
// the accept-length estimate over items n .. n + K - 1, available once item n + K - 1 has arrived. Each push
// applies every newly available loss, oldest first, as one NormalHedge round.
//
// State of one sequence (HF_HEAD bytes of header, then regrets and weights of up to 64 drafters, then a ring of
// 2K items of N floats): at most 2K - 1 items wait at once (K - 1 left after a push, K new ones).
constexpr int HF_HEAD = 32;
constexpr unsigned HF_STATUS_BAD_LEN = 1u;   // an accepted length outside [0, K]: that round was skipped
struct HfHead {
    int count, head, applied, objective;
    unsigned status;
    int pad[3];
};
__host__ __device__ constexpr size_t hf_seq_bytes(int N, int K) {
    return (static_cast<size_t>(HF_HEAD) + 2 * 64 * sizeof(float) + static_cast<size_t>(2 * K) * N * sizeof(float) + 15) /
           16 * 16;
}

struct HfParams {
    unsigned char* state;          // B sequences of hf_seq_bytes(N, K)
    const float* gamma;            // [N, B, K] (push)
    const int32_t* accept_len;     // [B] (push)
    int N, B, K, objective;        // objective: init only
    float* weights;                // [B, N] or null: the distribution for the next round
    int32_t* applied;              // [B] or null: NormalHedge rounds applied so far
};

// One warp per sequence: regrets 0, uniform weights, empty queue.
__global__ void __launch_bounds__(256) hedge_feedback_init_kernel(const HfParams p) {
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (b >= p.B) return;
    unsigned char* st = p.state + static_cast<size_t>(b) * hf_seq_bytes(p.N, p.K);
    HfHead* h = reinterpret_cast<HfHead*>(st);
    float* R = reinterpret_cast<float*>(st + HF_HEAD);
    float* W = R + 64;
    R[lane] = 0.f;
    R[lane + 32] = 0.f;
    W[lane] = lane < p.N ? 1.f / static_cast<float>(p.N) : 0.f;
    W[lane + 32] = lane + 32 < p.N ? 1.f / static_cast<float>(p.N) : 0.f;
    if (lane == 0) {
        h->count = 0;
        h->head = 0;
        h->applied = 0;
        h->objective = p.objective;
        h->status = 0u;
    }
}

// One warp per sequence: append the revealed levels of this round's gamma, then apply every available loss.
__global__ void __launch_bounds__(256) hedge_feedback_push_kernel(const HfParams p) {
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (b >= p.B) return;
    const int N = p.N, K = p.K, cap = 2 * K;
    unsigned char* st = p.state + static_cast<size_t>(b) * hf_seq_bytes(N, K);
    HfHead* h = reinterpret_cast<HfHead*>(st);
    float* R = reinterpret_cast<float*>(st + HF_HEAD);
    float* W = R + 64;
    float* ring = W + 64;
    const bool v0 = lane < N, v1 = lane + 32 < N;
    int count = h->count, head = h->head, applied = h->applied;
    const int objective = h->objective;
    const int L = __ldg(p.accept_len + b);
    if (L < 0 || L > K) {
        if (lane == 0) h->status |= HF_STATUS_BAD_LEN;
    } else {
        const int valid = min(L + 1, K);
        for (int j = 0; j < valid; ++j) {
            float* item = ring + static_cast<size_t>((head + count) % cap) * N;
            if (v0) item[lane] = __ldg(p.gamma + (static_cast<size_t>(lane) * p.B + b) * K + j);
            if (v1) item[lane + 32] = __ldg(p.gamma + (static_cast<size_t>(lane + 32) * p.B + b) * K + j);
            ++count;
        }
        __syncwarp();
    }
    float r0 = v0 ? R[lane] : 0.f, r1 = v1 ? R[lane + 32] : 0.f;
    float p0 = v0 ? W[lane] : 0.f, p1 = v1 ? W[lane + 32] : 0.f;
    while (objective == 0 ? count >= 1 : count >= K) {
        float l0, l1;
        if (objective == 0) {
            const float* item = ring + static_cast<size_t>(head) * N;
            l0 = v0 ? 1.f - item[lane] : 0.f;
            l1 = v1 ? 1.f - item[lane + 32] : 0.f;
        } else {   // K + 1 minus the accept-length estimate 1 + sum_k prod_{j<=k} gamma_j over the window
            float run0 = 1.f, tot0 = 1.f, run1 = 1.f, tot1 = 1.f;
            for (int k = 0; k < K; ++k) {
                const float* item = ring + static_cast<size_t>((head + k) % cap) * N;
                if (v0) {
                    run0 *= item[lane];
                    tot0 += run0;
                }
                if (v1) {
                    run1 *= item[lane + 32];
                    tot1 += run1;
                }
            }
            l0 = v0 ? static_cast<float>(K + 1) - tot0 : 0.f;
            l1 = v1 ? static_cast<float>(K + 1) - tot1 : 0.f;
        }
        nh_round(N, v0, v1, l0, l1, r0, r1, p0, p1);
        head = (head + 1) % cap;
        --count;
        ++applied;
    }
    if (v0) {
        R[lane] = r0;
        W[lane] = p0;
        if (p.weights) p.weights[static_cast<size_t>(b) * N + lane] = p0;
    }
    if (v1) {
        R[lane + 32] = r1;
        W[lane + 32] = p1;
        if (p.weights) p.weights[static_cast<size_t>(b) * N + lane + 32] = p1;
    }
    if (lane == 0) {
        h->count = count;
        h->head = head;
        h->applied = applied;
        if (p.applied) p.applied[b] = applied;
    }
}

// Test hook: the draw's float-float exponent and exp2 on n inputs (d = x - M, row offset l as a pair).
__global__ void __launch_bounds__(256) ff_exp2_probe_kernel(const float* __restrict__ d, const float* __restrict__ l_hi,
                                                            const float* __restrict__ l_lo, float* __restrict__ out,
                                                            int n, const FFc k) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const FF e = ff_exponent(d[i], k, l_hi[i], l_lo[i]);
    const FF y = ff_exp2(e, k, k.tab);
    out[2 * i] = y.hi;
    out[2 * i + 1] = y.lo;
}

}  // namespace specv
