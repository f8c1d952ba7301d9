// Shared device building blocks of the verification kernels for sm_103a: the element formats (bf16 and
// fp32 logits, 8 to a chunk), the per-chunk arithmetic of pass 1 (softmax statistics), of the residual
// masses and of the overlap sum min(p, q), and the inverse-CDF scan.
//
// Precision. A probability is evaluated as p(x) = 2^((x - M) c + L) with c = log2(e) / T, M the row's
// maximum logit and L = -log2(S), S = sum_y 2^((y - M) c). The difference x - M of two bf16 logits is exact
// in fp32 and the offsets stay small (|L| <= log2 V), so the exponent carries one rounding of its own
// size, not of the size of M c. The residual (p - q)+ subtracts two such values; an error common to a
// whole row (a rounded offset of size M c) would not cancel there and would move the inverse CDF.
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

constexpr int CHUNK = 8;                // logits per lane per load (16 B of bf16)
constexpr int PE = 2048;                // logits per piece: one bulk copy, one residual tile
constexpr int PCH = PE / CHUNK / 32;    // chunks per lane per piece
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;   // bounded waits: 2 s
constexpr unsigned STATUS_BAD_TOKEN = 1u;
constexpr unsigned STATUS_TIMEOUT = 2u;

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
    // whether a chunk holds a logit other than -inf
    __device__ static bool any_kept(const Raw& r) {
        const uint32_t ni = 0xFF80FF80u;
        return (r.x != ni) | (r.y != ni) | (r.z != ni) | (r.w != ni);
    }
    // a chunk with every logit below t replaced by -inf (standardised sampling's filter)
    __device__ static Raw mask(const Raw& r, float t) {
        auto m = [t](uint32_t w) -> uint32_t {
            const uint32_t lo = __uint_as_float(w << 16) >= t ? (w & 0xFFFFu) : 0xFF80u;
            const uint32_t hi = __uint_as_float(w & 0xFFFF0000u) >= t ? (w & 0xFFFF0000u) : 0xFF800000u;
            return lo | hi;
        };
        return make_uint4(m(r.x), m(r.y), m(r.z), m(r.w));
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
    __device__ static bool any_kept(const Raw& r) {
        const float ni = __uint_as_float(0xFF800000u);
        return (r.a.x != ni) | (r.a.y != ni) | (r.a.z != ni) | (r.a.w != ni) | (r.b.x != ni) | (r.b.y != ni) |
               (r.b.z != ni) | (r.b.w != ni);
    }
    // a chunk with every logit below t replaced by -inf (standardised sampling's filter)
    __device__ static Raw mask(const Raw& r, float t) {
        auto m = [t](float x) { return x >= t ? x : __uint_as_float(0xFF800000u); };
        Raw o;
        o.a = make_float4(m(r.a.x), m(r.a.y), m(r.a.z), m(r.a.w));
        o.b = make_float4(m(r.b.x), m(r.b.y), m(r.b.z), m(r.b.w));
        return o;
    }
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
// row offsets
// ------------------------------------------------------------------------------------------------
// A row's (max M, sum S) as the two numbers of p(x) = 2^((x + nm) c + l): nm = -M, l = -log2 S (libm
// log2f, correctly rounded to about one ulp). An empty row (every logit -inf, S = 0) gives p = 0.
struct RowOff {
    float nm, l;
};
__device__ __forceinline__ RowOff row_off(MaxSum g) {
    if (!(g.s > 0.f)) return {0.f, __uint_as_float(0xFF800000u)};
    return {-g.m, -log2f(g.s)};
}

// p(x) for one logit.
__device__ __forceinline__ float prob_at(float x, RowOff o, float c) {
    if (!(x > __uint_as_float(0xFF800000u))) return 0.f;
    return ex2(fmaf(x + o.nm, c, o.l));
}

// log2 p(x) = x c + beta with beta = -(M c + log2 S): one fused multiply-add a logit, used where the
// tolerance allows it (the overlap sums of gamma).
__device__ __forceinline__ float beta_of(MaxSum g, float c) { return -fmaf(g.m, c, lg2(g.s)); }

// Cactus closed form on q = p_target(t): gamma* = min(q + sqrt(2 delta q (1 - q)), 1) and the log2 of the
// scale (1 - gamma*) / (1 - q) applied to every other token (-inf when q = 1).
__device__ __forceinline__ void cactus_scalars(float q, float delta, float& gstar, float& log2s, float& scale) {
    float gs = q + sqrtf(2.f * delta * q * (1.f - q));
    gs = fminf(gs, 1.f);
    const float s = q < 1.f ? __fdiv_rn(1.f - gs, 1.f - q) : 0.f;
    gstar = gs;
    log2s = log2f(s);
    scale = s;
}

// The same scalars with gamma* the root of the divergence constraint instead of its Taylor closed form
// ([Cactus] Key design 2 with the KL divergence of Key design 3): with h_n = g and the other tokens scaled
// by (1 - g) / (1 - q), KL(h || p_target) = g ln(g / q) + (1 - g) ln((1 - g) / (1 - q)) =: F(g). F(q) = 0,
// F increases and is convex on [q, 1], so Newton's method inside the bracket [q, 1] (a bisection step
// whenever Newton leaves it) finds the root of F(g) = delta. No root below 1 (ln(1/q) <= delta) gives
// gamma* = 1; delta = 0 or q = 0 gives gamma* = q exactly.
__device__ __forceinline__ float cactus_kl_f(float q, float g) {
    const float a = g > 0.f ? g * logf(g / q) : 0.f;
    const float b = g < 1.f ? (1.f - g) * logf((1.f - g) / (1.f - q)) : 0.f;
    return a + b;
}
__device__ __forceinline__ float cactus_root_kl(float q, float delta) {
    float gs;
    if (!(delta > 0.f) || !(q > 0.f)) {
        gs = q;
    } else if (!(q < 1.f) || cactus_kl_f(q, 1.f) <= delta) {
        gs = 1.f;
    } else {
        float lo = q, hi = 1.f;
        float g = fminf(q + sqrtf(2.f * delta * q * (1.f - q)), 0.5f * (q + 1.f));   // the Taylor start
        for (int it = 0; it < 64; ++it) {
            const float f = cactus_kl_f(q, g) - delta;
            if (f > 0.f) hi = g;
            else lo = g;
            const float d = logf(g / q) - logf((1.f - g) / (1.f - q));   // F'(g) > 0 inside (q, 1)
            float gn = g - f / d;
            if (!(gn > lo && gn < hi)) gn = 0.5f * (lo + hi);
            if (fabsf(gn - g) <= 1e-7f * g || hi - lo <= 1e-7f * hi) {
                g = gn;
                break;
            }
            g = gn;
        }
        gs = g;
    }
    return gs;
}
__device__ __noinline__ void cactus_scalars_kl(float q, float delta, float& gstar, float& log2s, float& scale) {
    const float gs = cactus_root_kl(q, delta);
    const float s = q < 1.f ? __fdiv_rn(1.f - gs, 1.f - q) : 0.f;
    gstar = gs;
    log2s = log2f(s);
    scale = s;
}

// A logit kept by the filter (t = -inf keeps every finite or infinite logit), else -inf.
__device__ __forceinline__ float mask1(float x, float t) { return x >= t ? x : __uint_as_float(0xFF800000u); }

// ------------------------------------------------------------------------------------------------
// per-chunk arithmetic
// ------------------------------------------------------------------------------------------------
// Overlap only: adds 2^min(x_t c + bt, x_o c + bo) of the chunk's 8 elements to acc.
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

// The row offsets of the two rows a mass is made of: h (the target, or the Cactus h) and the other row
// (the draft; unused in mode 2).
struct PairOff {
    float nmt, lt, nmo, lo;
};

// Per-element masses of one chunk. mode 1: residual (h - p_other)+ (overlap min(h, p_other) added to
// ovl); mode 2: h itself. h(x) = 2^((x + nmt) c + lt) except element `et` (>= 0), which is `hpatch`. Each
// element goes through the same operations as in chunk_mass, so the values agree bit for bit.
template <class E>
__device__ __forceinline__ void chunk_values(int mode, const typename E::Raw& rt, const typename E::Raw& ro, float c,
                                             PairOff o, int et, float hpatch, float (&v)[8], float& ovl) {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const float2 xt = E::pair(rt, w);
        const float2 xo = E::pair(ro, w);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int e = 2 * w + h;
            float ph = ex2(fmaf((h ? xt.y : xt.x) + o.nmt, c, o.lt));
            if (e == et) ph = hpatch;
            if (mode == 1) {
                const float po = ex2(fmaf((h ? xo.y : xo.x) + o.nmo, c, o.lo));
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
__device__ __forceinline__ float chunk_mass(int mode, const typename E::Raw& rt, const typename E::Raw& ro, float c,
                                            PairOff o, float2& ovl2) {
    const float2 cc = make_float2(c, c);
    const float2 nmt = make_float2(o.nmt, o.nmt), lt = make_float2(o.lt, o.lt);
    const float2 nmo = make_float2(o.nmo, o.nmo), lo = make_float2(o.lo, o.lo);
    float2 m2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const float2 ph = ex2x2(__ffma2_rn(__fadd2_rn(E::pair(rt, w), nmt), cc, lt));
        if (mode == 1) {
            const float2 po = ex2x2(__ffma2_rn(__fadd2_rn(E::pair(ro, w), nmo), cc, lo));
            const float2 mn = make_float2(fminf(ph.x, po.x), fminf(ph.y, po.y));
            ovl2 = __fadd2_rn(ovl2, mn);
            m2 = __fadd2_rn(m2, __ffma2_rn(mn, make_float2(-1.f, -1.f), ph));   // ph - mn, one rounding
        } else {
            m2 = __fadd2_rn(m2, ph);
        }
    }
    return m2.x + m2.y;
}

// The chunk holding the draft token (element et patched to hpatch), out of line: one thread of one CTA per
// row takes this branch. Its sum pairs the elements exactly as chunk_mass does.
template <class E>
__device__ __noinline__ float chunk_mass_patch_only(int mode, typename E::Raw rt, typename E::Raw ro, float c, PairOff o,
                                                    int et, float hpatch, float& ovl) {
    float v[8];
    chunk_values<E>(mode, rt, ro, c, o, et, hpatch, v, ovl);
    const float2 a = make_float2(v[0] + v[2] + v[4] + v[6], v[1] + v[3] + v[5] + v[7]);
    return a.x + a.y;
}

// Chunk mass with the optional patch at element et.
template <class E>
__device__ __forceinline__ float chunk_mass_patched(int mode, const typename E::Raw& rt, const typename E::Raw& ro,
                                                    float c, PairOff o, int et, float hpatch, float2& ovl2) {
    if (et < 0) return chunk_mass<E>(mode, rt, ro, c, o, ovl2);
    float ovl = 0.f;
    const float m = chunk_mass_patch_only<E>(mode, rt, ro, c, o, et, hpatch, ovl);
    ovl2.x += ovl;
    return m;
}

// ------------------------------------------------------------------------------------------------
// the residual draw at float-float precision
// ------------------------------------------------------------------------------------------------
// The draw compares a running sum of residual masses with u * Z, so every error it makes moves a CDF
// boundary. The fast per-element arithmetic above rounds the exponent (x - M) c + L (a few 1e-7 of the element
// for exponents of 8 to 32) and its SFU exp2 adds about 1e-7. Summed over a row these errors are a few 1e-9
// of mass, and most of it comes from the few largest elements (an emulation of that arithmetic on rows of the
// Llama-3 workload: a median error of 3.9e-9 at the drawn boundary, 1.6e-9 once the elements above 1e-2 are
// exact). So the draw recomputes, at float-float precision (about 44 bits: the exponent as a float-float
// with c = log2(e) / T and L as float pairs, and a float-float exp2), every chunk whose fast mass (residual
// plus overlap) exceeds a threshold, and corrects its piece's mass by the difference. The large chunks of a
// warp wait in a queue and are evaluated eight lanes to a chunk (one lane alone would run each element's long
// chain of dependent float-float steps one after another). Cactus: gamma* and the scale s of the other tokens
// come from the float-float p_T(n) (the Taylor form in float-float, the divergence root refined by one
// float-float Newton step); the token's chunk always takes the exact path.
// Host-computed constants of the float-float arithmetic (double precision, split into float pairs).
struct FFc {
    float2 tab[33];          // 2^(k / 32), k = -16 .. 16
    float ln2_hi, ln2_lo;    // ln 2
    float c_hi, c_lo;        // log2(e) / T, c_hi rounded towards zero (c_lo > 0)
    float tau;               // a chunk whose fast mass (residual plus overlap) exceeds this is recomputed exactly
};

// (x - M) c + L as a float-float, with d = x - M given as the float-float d_hi + d_lo (d_lo = 0 for bf16 logits,
// whose difference is exact in float): the product's rounding error by a fused multiply-add, the sum's by
// TwoSum.
__device__ __forceinline__ FF ff_exponent(float d, const FFc& k, float l_hi, float l_lo, float d_lo = 0.f) {
    const float p1 = __fmul_rn(d, k.c_hi);
    const float e1 = __fmaf_rn(d, k.c_hi, -p1);
    const FF s = ff_two_sum(p1, l_hi);
    const float small = __fmaf_rn(d_lo, k.c_hi, __fmaf_rn(d, k.c_lo, l_lo));
    return ff_fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(e1, small)));
}

// 2^e for a float-float e (0 below 2^-125; tab = k.tab, or a copy of it in shared memory, where lanes that look
// up different entries do not serialise): e.hi = n + j/32 + g with n and j integers and
// |g| <= 1/64 (all exact in float), 2^(j/32) from the table, 2^(g + e.lo) = exp(q) with q = (g + e.lo) ln 2
// as a float-float and the Taylor series of exp to q^5 / 5! (|q| < 0.011: the next term is below 3e-15).
__device__ __forceinline__ FF ff_exp2(FF e, const FFc& k, const float2* tab) {
    if (!(e.hi > -125.f)) return {0.f, 0.f};
    const float n = rintf(e.hi);
    const float f = __fsub_rn(e.hi, n);
    const float jf = rintf(__fmul_rn(f, 32.f));
    const float g = __fmaf_rn(jf, -0.03125f, f);
    const float qh = __fmul_rn(g, k.ln2_hi);
    const float ql = __fadd_rn(__fmaf_rn(g, k.ln2_hi, -qh), __fmaf_rn(g, k.ln2_lo, __fmul_rn(e.lo, k.ln2_hi)));
    // exp(qh) = 1 + qh + qh^2 / 2 + qh^2 t with t = qh / 6 + qh^2 / 24 + qh^3 / 120; qh^2 exactly as a pair
    float t = __fmaf_rn(qh, 1.f / 120.f, 1.f / 24.f);
    t = __fmul_rn(qh, __fmaf_rn(qh, t, 1.f / 6.f));
    const FF q2 = ff_two_prod(qh, qh);
    const float tail_r = __fmaf_rn(q2.hi, t, __fmul_rn(0.5f, q2.lo));
    FF one_q = ff_fast_two_sum(1.f, qh);
    const FF with_sq = ff_fast_two_sum(one_q.hi, __fmul_rn(0.5f, q2.hi));
    // exp(qh + ql) = exp(qh) (1 + ql), to first order in ql
    const float lo = __fadd_rn(__fadd_rn(one_q.lo, with_sq.lo), __fmaf_rn(ql, with_sq.hi, tail_r));
    one_q.hi = with_sq.hi;
    const float2 T = tab[static_cast<int>(jf) + 16];
    const float ph = __fmul_rn(one_q.hi, T.x);
    const float pl = __fadd_rn(__fmaf_rn(one_q.hi, T.x, -ph), __fmaf_rn(one_q.hi, T.y, __fmaf_rn(lo, T.x, __fmul_rn(lo, T.y))));
    const FF r = ff_fast_two_sum(ph, pl);
    const float sc = __int_as_float((static_cast<int>(n) + 127) << 23);   // 2^n, exact for n >= -125
    return {__fmul_rn(r.hi, sc), __fmul_rn(r.lo, sc)};
}

// log2 of a float-float x > 0: the float log2 and one Newton step on 2^y = x, y = y0 + (x 2^-y0 - 1) / ln 2
// (the residual x 2^-y0 - 1 is about 1e-7, so the step leaves an error of order 1e-14).
__device__ __noinline__ FF ff_log2(FF x, const FFc& k) {
    const float y0 = log2f(x.hi);
    const FF r = ff_sub(ff_mul(x, ff_exp2(FF{-y0, 0.f}, k, k.tab)), FF{1.f, 0.f});
    // (r.hi + r.lo) / ln 2 with 1 / ln 2 = log2(e) = c_hi * T for T = 1 is not available here: divide by ln 2
    const float inv_ln2 = __fdiv_rn(1.f, k.ln2_hi);
    return ff_fast_two_sum(y0, __fmul_rn(__fadd_rn(r.hi, r.lo), inv_ln2));
}
// natural log of a float-float x > 0 (log2 x times ln 2)
__device__ __forceinline__ FF ff_log(FF x, const FFc& k) { return ff_mul(ff_log2(x, k), FF{k.ln2_hi, k.ln2_lo}); }

// gamma* at float-float precision from a float-float q = p_target(n): the Taylor closed form min(q +
// sqrt(2 delta q (1 - q)), 1) in float-float, or (kl) the float root of the divergence constraint refined by
// one Newton step in float-float (the float root is within about 1e-7 of the root, so one step leaves an error
// of order 1e-14).
__device__ __noinline__ FF cactus_gamma_ff(FF q, float delta, bool kl, const FFc& k) {
    if (!(delta > 0.f) || !(q.hi > 0.f)) return q;
    const FF one = {1.f, 0.f};
    if (!kl) {
        const FF root = ff_sqrt(ff_mulf(ff_mul(q, ff_sub(one, q)), 2.f * delta));
        const FF g = ff_add(q, root);
        return ff_gt(g, one) ? one : g;
    }
    if (!(q.hi < 1.f)) return one;
    const float g0 = cactus_root_kl(q.hi, delta);
    if (!(g0 < 1.f) || !(g0 > q.hi)) return FF{g0, 0.f};
    const FF g = {g0, 0.f};
    const FF a = ff_log(ff_div(g, q), k);                          // ln(g / q)
    const FF b = ff_log(ff_div(ff_sub(one, g), ff_sub(one, q)), k);  // ln((1 - g) / (1 - q))
    const FF f = ff_sub(ff_add(ff_mul(g, a), ff_mul(ff_sub(one, g), b)), FF{delta, 0.f});
    const FF d = ff_sub(a, b);
    if (!(d.hi > 0.f)) return g;
    const FF gn = ff_sub(g, ff_div(f, d));
    return (gn.hi > q.hi && gn.hi < 1.f) ? gn : g;
}

// Offsets of the row pair a draw is exactly recomputed from: target row (nmt = -M_T, L_T = -log2 S_T as
// lt + lt_lo, and the Cactus scale s of h = s p^_T; 1 otherwise), draft row (nmo = -M_D, lo + lo_lo).
struct PairOffX {
    float nmt, lt, lt_lo, s, nmo, lo, lo_lo;
};

// One element of a row pair at float-float precision. mode 1: the residual r = (h - p_D)+ with h = s p^_T, or
// h = g for the Cactus token (tok); mode 2: the bonus row, r = p^_T. xt, xd: the element's logits. The exponent
// (x - M) c + L is a float-float (c = c_hi + c_lo, L = lt + lt_lo; x - M as a float-float, exact for bf16
// logits) and so is its exp2. The draw evaluates this for every element of its few large chunks, eight lanes
// to a chunk, and replaces the chunk's fast mass by their sum.
__device__ __noinline__ FF elem_exact(int mode, float xt, float xd, const PairOffX& po, const FFc& k,
                                         const float2* tab, bool tok, FF g) {
    const float NINF = __uint_as_float(0xFF800000u);
    FF h;
    if (tok) {
        h = g;
    } else {
        FF pt = {0.f, 0.f};
        if (xt > NINF) {
            const FF dt = ff_two_sum(xt, po.nmt);
            pt = ff_exp2(ff_exponent(dt.hi, k, po.lt, po.lt_lo, dt.lo), k, tab);
        }
        h = ff_mulf(pt, po.s);
    }
    if (mode != 1) return h;
    FF q = {0.f, 0.f};
    if (xd > NINF) {
        const FF dd = ff_two_sum(xd, po.nmo);
        q = ff_exp2(ff_exponent(dd.hi, k, po.lo, po.lo_lo, dd.lo), k, tab);
    }
    return ff_gt(h, q) ? ff_sub(h, q) : FF{0.f, 0.f};
}

// Sum of a float-float over aligned groups of 8 lanes (fixed association: every lane of a group gets the
// same value).
__device__ __forceinline__ FF group8_sum(FF v) {
#pragma unroll
    for (int o = 1; o < 8; o <<= 1)
        v = ff_add(v, FF{__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)});
    return v;
}

// Inclusive scan across the warp (Hillis-Steele, fixed association order).
template <class T>
__device__ __forceinline__ T warp_incl_scan(T v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const T y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
    }
    return v;
}

// ------------------------------------------------------------------------------------------------
// per-piece building blocks (one warp, one piece of up to PE logits held in registers; lane l owns
// chunks l + 32 q, q < PCH; chunks past the end of the row are -inf and contribute exact zeros)
// ------------------------------------------------------------------------------------------------
template <class E>
__device__ __forceinline__ void piece_load(const unsigned char* src, int nchunks, int lane, typename E::Raw (&r)[PCH]) {
    if (nchunks == PCH * 32) {
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

// Pass 1: folds NCH chunks into the lane's running (max m, sum s of 2^((x - m) c)). Each term is
// 2^((x - m) c) with x - m exact, so the sum carries no error common to the lane's terms.
template <class E, int NCH>
__device__ __forceinline__ void chunks_stats(const typename E::Raw (&r)[NCH], float c, float& m, float& s) {
    typename E::Max mm = E::max_init();
#pragma unroll
    for (int q = 0; q < NCH; ++q) mm = E::max_acc(mm, r[q]);
    const float pm = E::max_fin(mm);
    if (pm > __uint_as_float(0xFF800000u)) {
        if (pm > m) {
            s = s > 0.f ? s * ex2((m - pm) * c) : 0.f;
            m = pm;
        }
        const float2 cc = make_float2(c, c);
        const float2 nm2 = make_float2(-m, -m);
        float2 s2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int q = 0; q < NCH; ++q)
#pragma unroll
            for (int w = 0; w < 4; ++w)
                s2[w] = __fadd2_rn(s2[w], ex2x2(__fmul2_rn(__fadd2_rn(E::pair(r[q], w), nm2), cc)));
        const float2 t = __fadd2_rn(__fadd2_rn(s2[0], s2[1]), __fadd2_rn(s2[2], s2[3]));
        s += t.x + t.y;
    }
}

template <class E>
__device__ __forceinline__ void piece_stats(const typename E::Raw (&r)[PCH], float c, float& m, float& s) {
    chunks_stats<E, PCH>(r, c, m, s);
}

// ------------------------------------------------------------------------------------------------
// inverse CDF
// ------------------------------------------------------------------------------------------------
// FILT: logits of the target row below tt, and of the other row below to, count as -inf.
template <class E, bool AL, bool FILT = false>
__device__ __noinline__ int scan_pick(float c, const unsigned char* trow, const unsigned char* orow, int mode, int e_begin,
                         int e_end, PairOff o, int tok, float ht, double tp, double before, int lane, float tt = 0.f,
                         float to = 0.f) {
    using Raw = typename E::Raw;
    int last_pos = -1;
    for (int base = e_begin; base < e_end; base += 32 * CHUNK) {
        const int e0 = base + lane * CHUNK;
        float v[8];
        double m = 0.0;
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = 0.f;
        if (e0 < e_end) {
            Raw rt = E::template gload<AL>(trow, e0, e_end);
            Raw ro = mode == 1 ? E::template gload<AL>(orow, e0, e_end) : rt;
            if constexpr (FILT) {
                rt = E::mask(rt, tt);
                ro = E::mask(ro, mode == 1 ? to : tt);
            }
            const int et = (tok >= e0 && tok < e0 + CHUNK) ? tok - e0 : -1;
            float ovl = 0.f;
            chunk_values<E>(mode, rt, ro, c, o, et, ht, v, ovl);
#pragma unroll
            for (int q = 0; q < 8; ++q) m += static_cast<double>(v[q]);
        }
        const double incl = warp_incl_scan(m, lane);
        const unsigned over = __ballot_sync(0xffffffffu, m > 0.0 && before + incl > tp);
        const unsigned posm = __ballot_sync(0xffffffffu, m > 0.0);
        if (over) {
            const int ln = __ffs(over) - 1;
            int pick = -1;
            if (lane == ln) {
                double a = before + incl - m;
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


}  // namespace specv
