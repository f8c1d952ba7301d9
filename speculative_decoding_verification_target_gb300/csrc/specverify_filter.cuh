// Standardised sampling ("Speculative Decoding 为什么是 Lossless 的 — 详细证明教程", §8 Q4: temperature,
// top-k and top-p are folded into p and q, the same transforms for the target and the draft row, before the
// ratio is taken). Every such filter keeps the logits at or above a per-row threshold, so the filtered
// verification is the ordinary one on rows whose other logits are -inf. Two kernels write each row's
// threshold and the kept logits' (max, sum of 2^((x - max) c)), which the draw takes as its row normalisers:
//   - bound_kernel (top-k up to FB_MAX_K on rows of whole 16-byte words): a bound from the row's line maxima,
//     the candidates at or above it, sorted (its own comment below);
//   - threshold_kernel (every other filter, and the rows bound_kernel leaves): radix selection on
//     order-preserving integer keys of the logits, 4 bits a pass from the top (4 passes for bf16, 8 for
//     fp32). Top-k (0 < k < V) descends by counts to the k-th largest value; top-p (0 < top_p < 1), on what
//     top-k kept, descends by the mass sum_x 2^((x - M) c) to the value at which the mass from the largest
//     logit down first reaches top_p of the kept total. Once the elements still in play fit in shared memory
//     (at most F_CAP keys), one more pass over the row copies them there and the remaining passes read only
//     them.
// Ties at a threshold are all kept (the kept set depends on values only). The draw kernel then reads the
// caller's rows as they are and replaces every logit below its row's threshold by -inf as it arrives in
// registers (its FILT form): no filtered copy is made and no statistics pass runs.
// The masses are integer sums, so they do not depend on the order of the additions: masses in 64-bit fixed
// point (2^-44 units; a mass 2^((x - M) c) is at most 1 and a row holds at most 2^18 logits, so a sum cannot
// overflow). In threshold_kernel each thread adds into its own column of the shared-memory histograms (no
// atomics, no contention however the keys cluster) and the columns are summed after the pass.
#pragma once
#include "specverify_kernels.cuh"

namespace specv {

constexpr int FT_NT = 256;               // threads of a threshold CTA
constexpr int FT_W = FT_NT / 32;
constexpr int F_DIGIT = 4;               // bits of a radix digit
constexpr int F_BINS = 1 << F_DIGIT;
constexpr int F_CAP = 4096;              // keys a CTA's candidate list holds
constexpr size_t F_SMEM = static_cast<size_t>(F_BINS) * FT_NT * (sizeof(unsigned long long) + sizeof(unsigned)) +
                          static_cast<size_t>(F_CAP) * sizeof(uint32_t);

// order-preserving keys: a larger logit has a larger unsigned key (negative values reversed)
template <class E>
struct FKey;
template <>
struct FKey<Bf16> {
    using K = uint32_t;
    static constexpr int BITS = 16;
    __device__ static K of_bits(uint32_t b) { return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u); }
    __device__ static K key(const unsigned char* row, int e) {
        return of_bits(reinterpret_cast<const uint16_t*>(row)[e]);
    }
    __device__ static float value_of(K k) {
        const uint32_t b = (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu);
        return __uint_as_float(b << 16);
    }
};
template <>
struct FKey<F32> {
    using K = uint32_t;
    static constexpr int BITS = 32;
    __device__ static K of_bits(uint32_t b) { return (b & 0x80000000u) ? ~b : (b | 0x80000000u); }
    __device__ static K key(const unsigned char* row, int e) {
        return of_bits(reinterpret_cast<const uint32_t*>(row)[e]);
    }
    __device__ static float value_of(K k) {
        const uint32_t b = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
        return __uint_as_float(b);
    }
};

struct FParams {
    const unsigned char* rows_a;   // target rows [B, K+1, V]
    const unsigned char* rows_b;   // draft rows [B, K, V]
    long long rows_a_n, rows_n;
    int V;
    float c;                       // log2(e) / temperature
    int top_k;                     // 0 or V: none
    float top_p;                   // >= 1: none
    float* thr;                    // [rows_n] threshold value (-inf: nothing filtered; NaN: left to threshold_kernel)
    float2* row_ms;                // [rows_n] (max, sum of 2^((x - max) c)) over the logits the filter keeps
    int flagged_only;              // threshold_kernel: only the rows whose threshold is NaN (else every row)
    int* list_n;                   // [rows_a_n] kept logits of a target row listed for the draw (-1: none)
    int* list_idx;                 // [rows_a_n, list_cap] their element indices, ascending
    float* list_x;                 // [rows_a_n, list_cap] their values
    int list_cap;
    int vec;                       // every row starts on 16 bytes and holds whole 16-byte words
};

__device__ __forceinline__ const unsigned char* f_row(const FParams& p, long long r, size_t row_bytes) {
    return r < p.rows_a_n ? p.rows_a + static_cast<size_t>(r) * row_bytes
                          : p.rows_b + static_cast<size_t>(r - p.rows_a_n) * row_bytes;
}

constexpr float F_FIX = 17592186044416.f;    // 2^44: the fixed-point unit of the mass histograms

// The key of a value that is one of the row's elements, taking -0 for a zero (keys order -0 below +0, float
// comparison does not): never above the element's own key.
template <class E>
__device__ __forceinline__ typename FKey<E>::K key_at_most(float v) {
    if (v == 0.f) v = -0.f;
    if constexpr (E::BYTES == 2) return FKey<E>::of_bits(__float_as_uint(v) >> 16);
    else return FKey<E>::of_bits(__float_as_uint(v));
}

// One 16-byte word of a row through the read-only path with an L2 eviction policy.
__device__ __forceinline__ uint4 ld_word(const uint4* ptr, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(ptr), "l"(pol));
    return v;
}

// This thread's largest value of the row (the CTA's threads striding over 16-byte words, vec rows only): a
// packed bf16 max per word pair for bf16 rows, -inf when the thread holds no element. The row is read
// evict-last: the compaction that follows reads it again.
template <class E>
__device__ __forceinline__ float thread_max_words(const unsigned char* row, int V) {
    const uint4* w4 = reinterpret_cast<const uint4*>(row);
    const int n4 = static_cast<int>(static_cast<size_t>(V) * E::BYTES / 16);
    const uint64_t pol = policy_evict_last();
    if constexpr (E::BYTES == 2) {
        uint32_t m2 = 0xFF80FF80u;
#pragma unroll 8
        for (int i = threadIdx.x; i < n4; i += FT_NT) {
            const uint4 w = ld_word(w4 + i, pol);
            m2 = bf16x2_max(m2, bf16x2_max(bf16x2_max(w.x, w.y), bf16x2_max(w.z, w.w)));
        }
        return fmaxf(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xFFFF0000u));
    } else {
        float m = __uint_as_float(0xFF800000u);
#pragma unroll 8
        for (int i = threadIdx.x; i < n4; i += FT_NT) {
            const uint4 w = ld_word(w4 + i, pol);
            m = fmaxf(m, fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)),
                               fmaxf(__uint_as_float(w.z), __uint_as_float(w.w))));
        }
        return m;
    }
}

// Calls f(key, valid) for every logit of a row, a CTA's threads striding over it: 16-byte words when the row
// allows them (vec), else single elements. Every thread of a warp makes the same number of calls (valid is
// false past the end), so f may use warp votes.
template <class E, class F>
__device__ __forceinline__ void for_row_keys(const unsigned char* row, int V, bool vec, F&& f) {
    using KT = typename FKey<E>::K;
    if (vec) {
        const uint4* w4 = reinterpret_cast<const uint4*>(row);
        const int n4 = static_cast<int>(static_cast<size_t>(V) * E::BYTES / 16);
#pragma unroll 2
        for (int i0 = 0; i0 < n4; i0 += FT_NT) {
            const int i = i0 + static_cast<int>(threadIdx.x);
            const bool ok = i < n4;
            const uint4 w = ok ? __ldg(w4 + i) : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if constexpr (E::BYTES == 2) {
                    f(static_cast<KT>(FKey<E>::of_bits(u[j] & 0xFFFFu)), ok);
                    f(static_cast<KT>(FKey<E>::of_bits(u[j] >> 16)), ok);
                } else {
                    f(static_cast<KT>(FKey<E>::of_bits(u[j])), ok);
                }
            }
        }
    } else {
        for (int e0 = 0; e0 < V; e0 += FT_NT) {
            const int e = e0 + static_cast<int>(threadIdx.x);
            const bool ok = e < V;
            f(ok ? FKey<E>::key(row, e) : KT(0), ok);
        }
    }
}

// Sum of one float per thread in a fixed order (warp trees, then the warps in order): the same bits on every
// run. Every thread of the CTA calls it; thread 0 gets the sum.
template <int NT>
__device__ __forceinline__ float cta_sum_fixed(float v, float* s_red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
    if (lane == 0) s_red[warp] = v;
    __syncthreads();
    float t = 0.f;
    if (threadIdx.x == 0)
        for (int w = 0; w < NT / 32; ++w) t += s_red[w];
    __syncthreads();
    return t;
}

// The threshold and the kept logits' (max, sum) of row r (all FT_NT threads of the CTA).
template <class E>
__device__ __forceinline__ void threshold_row(const FParams& p, const long long r) {
    using KT = typename FKey<E>::K;
    constexpr int BITS = FKey<E>::BITS;
    extern __shared__ __align__(16) unsigned char f_smem[];
    unsigned long long* hm = reinterpret_cast<unsigned long long*>(f_smem);   // masses [F_BINS][FT_NT]
    unsigned* hc = reinterpret_cast<unsigned*>(hm + F_BINS * FT_NT);          // counts [F_BINS][FT_NT]
    KT* cand = reinterpret_cast<KT*>(hc + F_BINS * FT_NT);                     // candidate keys [F_CAP]
    __shared__ unsigned s_cnt[F_BINS];
    __shared__ unsigned long long s_mass[F_BINS];
    __shared__ unsigned s_sel, s_n;
    __shared__ unsigned long long s_above;
    __shared__ KT s_kmax[FT_W];
    __shared__ KT s_tmax[FT_NT];                 // top-k by bound: every thread's largest key
    __shared__ KT s_bound, s_rowmax;
    __shared__ float s_red[FT_W];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int V = p.V;
    const bool vec = p.vec != 0;
    const size_t row_bytes = static_cast<size_t>(V) * E::BYTES;
    const unsigned char* row = f_row(p, r, row_bytes);
    const float NINF = __uint_as_float(0xFF800000u);
    for (int b = 0; b < F_BINS; ++b) {
        hc[b * FT_NT + tid] = 0u;
        hm[b * FT_NT + tid] = 0ull;
    }

    // is key k in the set: k >= lo and its digits from bit `from` up equal `prefix` (from >= BITS: any digits)
    auto in_set = [&](KT k, KT prefix, int from, KT lo) {
        return k >= lo && (from >= BITS || (k >> from) == prefix);
    };
    // the largest key of the row (all threads get it); kmax holds this thread's share
    auto cta_kmax = [&](KT kmax) -> KT {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) kmax = max(kmax, static_cast<KT>(__shfl_xor_sync(0xffffffffu, kmax, o)));
        if (lane == 0) s_kmax[warp] = kmax;
        __syncthreads();
        KT m = 0;
        for (int w2 = 0; w2 < FT_W; ++w2) m = max(m, s_kmax[w2]);
        return m;
    };
    // one radix pass over the set (the row, or the n_c candidates when n_c >= 0): its histogram by the digit
    // at `shift`, counts and (mass) masses 2^((x - M) c) in fixed point; leaves the bins in s_cnt / s_mass.
    // *kmax (when given) receives the largest key the pass read.
    auto pass = [&](int n_c, KT prefix, int shift, KT lo, bool mass, float M, KT* kmax) {
        KT km = 0;
        auto add = [&](KT k, bool ok) {
            km = max(km, ok ? k : KT(0));
            if (ok && in_set(k, prefix, shift + F_DIGIT, lo)) {
                const int bin = static_cast<int>((k >> shift) & (F_BINS - 1));
                hc[bin * FT_NT + tid] += 1u;
                // the mass times 2^44, truncated (exact above 2^-21; the truncation is below one unit)
                if (mass) hm[bin * FT_NT + tid] += __float2ull_rz(ex2((FKey<E>::value_of(k) - M) * p.c) * F_FIX);
            }
        };
        if (n_c < 0) for_row_keys<E>(row, V, vec, add);
        else
            for (int i = tid; i < n_c; i += FT_NT) add(cand[i], true);
        __syncthreads();
        {   // FT_NT / F_BINS threads (contiguous lanes) sum the columns of one bin
            constexpr int PER = FT_NT / F_BINS;
            const int b = tid / PER, part = tid % PER;
            unsigned cs = 0u;
            unsigned long long ms = 0ull;
            for (int j = part; j < FT_NT; j += PER) {
                cs += hc[b * FT_NT + j];
                ms += hm[b * FT_NT + j];
            }
#pragma unroll
            for (int o = PER / 2; o > 0; o >>= 1) {
                cs += __shfl_xor_sync(0xffffffffu, cs, o);
                ms += __shfl_xor_sync(0xffffffffu, ms, o);
            }
            if (part == 0) {
                s_cnt[b] = cs;
                s_mass[b] = ms;
            }
        }
        __syncthreads();
        for (int b = 0; b < F_BINS; ++b) {   // this thread's columns, cleared for the next pass
            hc[b * FT_NT + tid] = 0u;
            hm[b * FT_NT + tid] = 0ull;
        }
        if (kmax) *kmax = cta_kmax(km);
    };
    // the bin, from the top, where the running total first reaches `need`; returns the total above it
    auto choose = [&](unsigned long long need, bool mass) -> unsigned long long {
        if (tid == 0) {
            unsigned long long above = 0ull;
            int b = 0;
            for (b = F_BINS - 1; b > 0; --b) {
                const unsigned long long h = mass ? s_mass[b] : static_cast<unsigned long long>(s_cnt[b]);
                if (above + h >= need) break;
                above += h;
            }
            s_sel = static_cast<unsigned>(b);
            s_above = above;
        }
        __syncthreads();
        return s_above;
    };
    // copies into the candidate list (any order: what follows only sums integers) the keys >= lo whose digits
    // from bit `from` up equal prefix, or (ge) are at least prefix; returns how many there are (the list holds
    // the first F_CAP)
    auto compact = [&](KT prefix, int from, KT lo, bool ge) -> int {
        if (tid == 0) s_n = 0u;
        __syncthreads();
        for_row_keys<E>(row, V, vec, [&](KT k, bool ok) {
            const bool in = ok && k >= lo && (from >= BITS || (ge ? (k >> from) >= prefix : (k >> from) == prefix));
            const unsigned bal = __ballot_sync(0xffffffffu, in);
            if (bal) {
                unsigned base = 0u;
                if (lane == 0) base = atomicAdd(&s_n, static_cast<unsigned>(__popc(bal)));
                base = __shfl_sync(0xffffffffu, base, 0);
                if (in) {
                    const unsigned at = base + static_cast<unsigned>(__popc(bal & ((1u << lane) - 1u)));
                    if (at < static_cast<unsigned>(F_CAP)) cand[at] = k;
                }
            }
        });
        __syncthreads();
        const int n = static_cast<int>(s_n);
        __syncthreads();
        return n;
    };

    // compact(0, BITS, b, false) for vec rows, a word at a time: the values of a 16-byte word are compared
    // with b's value as floats (every key >= b passes: key order refines float order), and only a word with a
    // passing value takes the exact key test and the list append
    auto compact_bound = [&](KT b) -> int {
        if (tid == 0) s_n = 0u;
        __syncthreads();
        const float bv = FKey<E>::value_of(b);
        const uint4* w4 = reinterpret_cast<const uint4*>(row);
        const int n4 = static_cast<int>(row_bytes / 16);
        const uint64_t pol = policy_evict_first();   // the row's last read
        constexpr int BATCH = 4;                       // words a thread loads before testing them
        for (int i0 = 0; i0 < n4; i0 += BATCH * FT_NT) {
            uint4 ws[BATCH];
#pragma unroll
            for (int r = 0; r < BATCH; ++r) {
                const int i = i0 + r * FT_NT + tid;
                ws[r] = i < n4 ? ld_word(w4 + i, pol) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int r = 0; r < BATCH; ++r) {
            const int i = i0 + r * FT_NT + tid;
            const bool ok = i < n4;
            const uint4 w = ws[r];
            const uint32_t u[4] = {w.x, w.y, w.z, w.w};
            bool any = false;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if constexpr (E::BYTES == 2)
                    any |= (__uint_as_float(u[j] << 16) >= bv) | (__uint_as_float(u[j] & 0xFFFF0000u) >= bv);
                else
                    any |= __uint_as_float(u[j]) >= bv;
            }
            if (!__any_sync(0xffffffffu, ok && any)) continue;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
#pragma unroll
                for (int h = 0; h < (E::BYTES == 2 ? 2 : 1); ++h) {
                    const KT k = E::BYTES == 2 ? FKey<E>::of_bits(h ? (u[j] >> 16) : (u[j] & 0xFFFFu))
                                               : FKey<E>::of_bits(u[j]);
                    const bool in = ok && k >= b;
                    const unsigned bal = __ballot_sync(0xffffffffu, in);
                    if (bal) {
                        unsigned base = 0u;
                        if (lane == 0) base = atomicAdd(&s_n, static_cast<unsigned>(__popc(bal)));
                        base = __shfl_sync(0xffffffffu, base, 0);
                        if (in) {
                            const unsigned at = base + static_cast<unsigned>(__popc(bal & ((1u << lane) - 1u)));
                            if (at < static_cast<unsigned>(F_CAP)) cand[at] = k;
                        }
                    }
                }
            }
            }
        }
        __syncthreads();
        const int n = static_cast<int>(s_n);
        __syncthreads();
        return n;
    };

    KT lo = 0;                             // keep keys >= lo
    KT kmax = 0;                           // the row's largest key (once a pass has read the row)
    bool have_max = false, filtered = false;
    int n_c = -1;                          // keys in the candidate list (-1: passes read the row)
    if (p.top_k > 0 && p.top_k < V) {
        if (p.top_k <= FT_NT) {
            // The threads' own largest keys are FT_NT distinct elements of the row, so the k-th largest of them
            // is at most the row's k-th largest: every key top-k keeps is at or above it. Those keys go to the
            // candidate list when they fit, and the descent below reads only them.
            KT km = 0;
            if (vec) km = key_at_most<E>(thread_max_words<E>(row, V));
            else for_row_keys<E>(row, V, vec, [&](KT k, bool ok) { km = max(km, ok ? k : KT(0)); });
            s_tmax[tid] = km;
            __syncthreads();
            int rank = 0;   // larger keys, and equal keys of lower threads
            for (int t = 0; t < FT_NT; ++t) {
                const KT o = s_tmax[t];
                rank += (o > km || (o == km && t < tid)) ? 1 : 0;
            }
            if (rank == p.top_k - 1) s_bound = km;
            if (rank == 0) s_rowmax = km;
            __syncthreads();
            kmax = s_rowmax;
            have_max = true;
            const int n = vec ? compact_bound(s_bound) : compact(0, BITS, s_bound, false);
            if (n <= F_CAP) n_c = n;
        }
        KT prefix = 0;
        unsigned long long need = static_cast<unsigned long long>(p.top_k);
        for (int shift = BITS - F_DIGIT; shift >= 0; shift -= F_DIGIT) {
            pass(n_c, prefix, shift, 0, false, 0.f, have_max ? nullptr : &kmax);
            have_max = true;
            const unsigned long long above = choose(need, false);
            const unsigned sel = s_sel, cnt = s_cnt[sel];
            need -= above;
            prefix = (prefix << F_DIGIT) | static_cast<KT>(sel);
            __syncthreads();
            // every key from this prefix up: what top-k still sorts and everything it keeps
            const unsigned long long n_ge = static_cast<unsigned long long>(p.top_k) - need + cnt;
            if (n_c < 0 && shift > 0 && n_ge <= static_cast<unsigned long long>(F_CAP))
                n_c = min(compact(prefix, shift, 0, true), F_CAP);
        }
        lo = prefix;
        filtered = true;
    }
    if (p.top_p > 0.f && p.top_p < 1.f) {
        if (!have_max) {
            KT km = 0;
            for_row_keys<E>(row, V, vec, [&](KT k, bool ok) { km = max(km, ok ? k : KT(0)); });
            kmax = cta_kmax(km);
        }
        const float M = FKey<E>::value_of(kmax);
        KT prefix = 0;
        unsigned long long need = 0ull;
        for (int shift = BITS - F_DIGIT; shift >= 0; shift -= F_DIGIT) {
            pass(n_c, prefix, shift, lo, true, M, nullptr);
            if (shift == BITS - F_DIGIT) {   // the first pass sees every kept element: its bins sum to the total
                unsigned long long t = 0ull;
                for (int b = 0; b < F_BINS; ++b) t += s_mass[b];
                // top_p of the total, rounded up: the smallest fixed-point mass that reaches it
                need = static_cast<unsigned long long>(ceil(static_cast<double>(p.top_p) * static_cast<double>(t)));
            }
            const unsigned long long above = choose(need, true);
            const unsigned sel = s_sel, cnt = s_cnt[sel];
            need -= above;
            prefix = (prefix << F_DIGIT) | static_cast<KT>(sel);
            __syncthreads();
            if (n_c < 0 && shift > 0 && cnt <= static_cast<unsigned>(F_CAP)) n_c = min(compact(prefix, shift, lo, false), F_CAP);
        }
        if (!filtered || prefix > lo) lo = prefix;
        filtered = true;
    }
    if (!have_max) {
        KT km = 0;
        for_row_keys<E>(row, V, vec, [&](KT k, bool ok) { km = max(km, ok ? k : KT(0)); });
        kmax = cta_kmax(km);
    }
    // the kept logits (every value at or above the threshold, the row's largest among them): their (max, sum)
    // for the draw, which masks by the same float comparison
    const float th = filtered ? FKey<E>::value_of(lo) : NINF;
    const float M = FKey<E>::value_of(kmax);
    float sacc = 0.f;
    for_row_keys<E>(row, V, vec, [&](KT k, bool ok) {
        const float x = FKey<E>::value_of(k);
        if (ok && x >= th) sacc += ex2((x - M) * p.c);
    });
    const float ssum = cta_sum_fixed<FT_NT>(sacc, s_red);
    if (tid == 0) {
        p.thr[r] = th;
        p.row_ms[r] = make_float2(M, ssum);
        if (r < p.rows_a_n) p.list_n[r] = -1;   // the draw reads this row whole
    }
}

// One CTA per row (flagged_only: the CTAs stride over the rows and take those left with a NaN threshold).
template <class E>
__global__ void __launch_bounds__(FT_NT) threshold_kernel(const __grid_constant__ FParams p) {
    for (long long r = blockIdx.x; r < p.rows_n; r += gridDim.x) {
        if (p.flagged_only && !isnan(p.thr[r])) continue;
        threshold_row<E>(p, r);
        __syncthreads();
    }
}

// ------------------------------------------------------------------------------------------------
// top-k through line maxima (rows of whole 16-byte words, 0 < top_k <= FB_MAX_K < V)
// ------------------------------------------------------------------------------------------------
// A line is 8 words (128 bytes) of a row. The lines' maxima are maxima of disjoint sets, so the k-th
// largest of them is at most the row's k-th largest logit: every logit top-k keeps lies in a line whose
// maximum reaches it. One CTA per row:
//   1. reads the row once (evict-last), keeping each line's maximum as a 16-bit key in shared memory (the
//      upper half of the key for fp32, which rounds it down and keeps the bound valid);
//   2. selects the k-th largest line key by two 8-bit radix passes over shared memory (the bound);
//   3. re-reads only the lines whose maximum reaches the bound (mostly from L2) and lists their logits at or
//      above it: at least k of them, all that top-k can keep;
//   4. sorts the list (descending keys; by rank up to 512 keys, else bitonic): the k-th key is the top-k
//      threshold; top-p scans the kept
//      keys' fixed-point masses from the top (the same masses and the same rule as threshold_kernel, so the
//      same threshold);
//   5. writes the threshold and the kept logits' (max, sum).
// A row whose list would pass F_CAP keys gets a NaN threshold and is left to threshold_kernel.
constexpr int FB_NT = 256;
constexpr int FB_W = FB_NT / 32;
constexpr int FB_MAX_K = F_CAP / 4;
constexpr int FB_MAX_V = 262144;                 // the library's largest vocabulary
constexpr int FB_LINE_WORDS = 8;
constexpr int FB_U = 8;                          // words a thread has in flight in the first read

// a 16-byte word of -inf logits, and the largest value of a word
template <class E>
__device__ __forceinline__ uint4 f_ninf_word() {
    const uint32_t x = E::BYTES == 2 ? 0xFF80FF80u : 0xFF800000u;
    return make_uint4(x, x, x, x);
}
template <class E>
__device__ __forceinline__ float f_word_max(const uint4& w) {
    if constexpr (E::BYTES == 2) {
        const uint32_t m2 = bf16x2_max(bf16x2_max(w.x, w.y), bf16x2_max(w.z, w.w));
        return fmaxf(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xFFFF0000u));
    } else {
        return fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)), fmaxf(__uint_as_float(w.z), __uint_as_float(w.w)));
    }
}

// a line's maximum value as a 16-bit key that is never above the key of the logit it came from
template <class E>
__device__ __forceinline__ uint32_t line_key16(float v) {
    const uint32_t k = key_at_most<E>(v);
    return E::BYTES == 2 ? k : (k >> 16);
}

template <class E>
__global__ void __launch_bounds__(FB_NT, 5) bound_kernel(const __grid_constant__ FParams p) {
    using KT = typename FKey<E>::K;
    static_assert(FB_MAX_V * E::BYTES / (16 * FB_LINE_WORDS) * 2 <= F_CAP * 8, "line keys fit the list's space");
    static_assert(F_CAP * 2 <= FB_W * 256 * 4, "line list fits the histograms' space");
    __shared__ __align__(16) unsigned long long s_a[F_CAP];   // line keys (uint16), then the candidates:
                                                              // key << 32 | element index
    __shared__ __align__(16) uint32_t s_b[FB_W * 256];    // per-warp 8-bit histograms, then the line list (uint16)
    __shared__ unsigned s_wt[FB_W];
    __shared__ unsigned long long s_wm[FB_W];
    __shared__ float s_red[FB_W];
    __shared__ unsigned s_n, s_sel, s_above, s_nk, s_first;
    uint16_t* const lkey = reinterpret_cast<uint16_t*>(s_a);
    uint16_t* const lines = reinterpret_cast<uint16_t*>(s_b);
    unsigned long long* const cand = s_a;
    auto key_of = [&](int i) -> KT { return static_cast<KT>(cand[i] >> 32); };
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long r = blockIdx.x;
    const int V = p.V, k = p.top_k;
    const size_t row_bytes = static_cast<size_t>(V) * E::BYTES;
    const uint4* const w4 = reinterpret_cast<const uint4*>(f_row(p, r, row_bytes));
    const int n4 = static_cast<int>(row_bytes / 16);
    const int n_lines = (n4 + FB_LINE_WORDS - 1) / FB_LINE_WORDS;

    // ---- 1. line maxima: the eight lanes of a line each take one word ----
    {
        const uint64_t pol = policy_evict_last();
        const int n_it = (n4 + FB_NT - 1) / FB_NT;
        for (int it0 = 0; it0 < n_it; it0 += FB_U) {
            uint4 w[FB_U];
#pragma unroll
            for (int u = 0; u < FB_U; ++u) {
                const int i = (it0 + u) * FB_NT + tid;
                w[u] = i < n4 ? ld_word(w4 + i, pol) : f_ninf_word<E>();
            }
#pragma unroll
            for (int u = 0; u < FB_U; ++u) {
                if (it0 + u >= n_it) break;
                float m = f_word_max<E>(w[u]);
#pragma unroll
                for (int o = 1; o < FB_LINE_WORDS; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                const int line = (it0 + u) * (FB_NT / FB_LINE_WORDS) + tid / FB_LINE_WORDS;
                if ((lane & (FB_LINE_WORDS - 1)) == 0 && line < n_lines) lkey[line] = static_cast<uint16_t>(line_key16<E>(m));
            }
        }
    }
    __syncthreads();

    // ---- 2. the k-th largest line key (every key when there are fewer than k lines) ----
    // one 8-bit digit: among the keys whose high byte is `hi` (hi < 0: all), the bin where the count from the
    // top first reaches need; leaves the bin and the count above it in s_sel / s_above
    auto select_byte = [&](int shift, int hi, unsigned need) {
        for (int i = tid; i < FB_W * 256; i += FB_NT) s_b[i] = 0u;
        __syncthreads();
        uint32_t* const h = s_b + warp * 256;
        for (int l = tid; l < n_lines; l += FB_NT) {
            const uint32_t key = lkey[l];
            if (hi < 0 || static_cast<int>(key >> 8) == hi) atomicAdd(&h[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        const int bin = 255 - tid;   // thread t holds bin 255 - t: the scan runs from the top bin down
        unsigned c = 0u;
#pragma unroll
        for (int w2 = 0; w2 < FB_W; ++w2) c += s_b[w2 * 256 + bin];
        unsigned incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) s_wt[warp] = incl;
        __syncthreads();
        for (int w2 = 0; w2 < warp; ++w2) incl += s_wt[w2];
        if (incl >= need && incl - c < need) {
            s_sel = static_cast<unsigned>(bin);
            s_above = incl - c;
        }
        __syncthreads();
    };
    uint32_t bound16 = 0u;
    if (n_lines >= k) {
        select_byte(8, -1, static_cast<unsigned>(k));
        const unsigned hi = s_sel, above = s_above;
        select_byte(0, static_cast<int>(hi), static_cast<unsigned>(k) - above);
        bound16 = (hi << 8) | s_sel;
    }
    // as a key of the row's type; a bound whose value is zero becomes the key of -0, so that every logit the
    // draw's float comparison keeps (-0 >= +0) is listed
    const KT bound = key_at_most<E>(FKey<E>::value_of(E::BYTES == 2 ? static_cast<KT>(bound16) : static_cast<KT>(bound16 << 16)));
    const uint32_t bound_line = E::BYTES == 2 ? bound : (bound >> 16);   // a line holding such a logit reaches it

    // ---- 3. the lines that reach the bound, then their logits at or above it ----
    if (tid == 0) s_n = 0u;
    __syncthreads();
    for (int l0 = 0; l0 < n_lines; l0 += FB_NT) {
        const int l = l0 + tid;
        const bool in = l < n_lines && lkey[l] >= bound_line;
        const unsigned bal = __ballot_sync(0xffffffffu, in);
        if (bal) {
            unsigned base = 0u;
            if (lane == 0) base = atomicAdd(&s_n, static_cast<unsigned>(__popc(bal)));
            base = __shfl_sync(0xffffffffu, base, 0);
            const unsigned at = base + static_cast<unsigned>(__popc(bal & ((1u << lane) - 1u)));
            if (in && at < static_cast<unsigned>(F_CAP)) lines[at] = static_cast<uint16_t>(l);
        }
    }
    __syncthreads();
    const unsigned nl = s_n;   // each listed line holds a logit at or above the bound
    __syncthreads();
    if (nl <= static_cast<unsigned>(F_CAP)) {
        if (tid == 0) s_n = 0u;
        __syncthreads();
        const uint64_t pol = policy_evict_first();   // the row's last read
        const int g = tid / FB_LINE_WORDS, sub = tid % FB_LINE_WORDS;
        constexpr int GPB = FB_NT / FB_LINE_WORDS;   // lines a CTA reads per step
        constexpr int UG = 4;
        for (int base = 0; base < static_cast<int>(nl); base += GPB * UG) {
            uint4 w[UG];
            bool ok[UG];
#pragma unroll
            for (int u = 0; u < UG; ++u) {
                const int li = base + u * GPB + g;
                const int wi = li < static_cast<int>(nl) ? static_cast<int>(lines[li]) * FB_LINE_WORDS + sub : n4;
                ok[u] = wi < n4;
                w[u] = ok[u] ? ld_word(w4 + wi, pol) : make_uint4(0u, 0u, 0u, 0u);
            }
            const float bv = bound == 0u ? __uint_as_float(0xFF800000u) : FKey<E>::value_of(bound);   // 0: all
#pragma unroll
            for (int u = 0; u < UG; ++u) {
                const uint32_t uu[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
                // a word whose values all lie below the bound's (as floats: key order refines float order)
                // holds no key at or above it
                bool any = false;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if constexpr (E::BYTES == 2)
                        any |= (__uint_as_float(uu[j] << 16) >= bv) | (__uint_as_float(uu[j] & 0xFFFF0000u) >= bv);
                    else
                        any |= __uint_as_float(uu[j]) >= bv;
                }
                if (!(ok[u] && any)) continue;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
#pragma unroll
                    for (int h = 0; h < (E::BYTES == 2 ? 2 : 1); ++h) {
                        const KT key = E::BYTES == 2 ? FKey<E>::of_bits(h ? (uu[j] >> 16) : (uu[j] & 0xFFFFu))
                                                     : FKey<E>::of_bits(uu[j]);
                        if (key >= bound) {
                            const unsigned at = atomicAdd(&s_n, 1u);
                            const int wi = static_cast<int>(lines[base + u * GPB + g]) * FB_LINE_WORDS + sub;
                            const unsigned e = static_cast<unsigned>(wi * (16 / E::BYTES) + j * (E::BYTES == 2 ? 2 : 1) + h);
                            if (at < static_cast<unsigned>(F_CAP))
                                cand[at] = (static_cast<unsigned long long>(key) << 32) | e;
                        }
                    }
                }
            }
        }
        __syncthreads();
    }
    const unsigned n = nl <= static_cast<unsigned>(F_CAP) ? s_n : 0xFFFFFFFFu;
    if (n > static_cast<unsigned>(F_CAP) || n < static_cast<unsigned>(k)) {   // too many: threshold_kernel takes the row
        if (tid == 0) {
            p.thr[r] = __uint_as_float(0x7FC00000u);
            if (r < p.rows_a_n) p.list_n[r] = -1;
        }
        return;
    }

    // ---- 4. sort the list, descending keys (then descending element index: the entries are distinct) ----
    if (n <= static_cast<unsigned>(2 * FB_NT)) {
        // by rank (the larger entries): two entries a thread
        unsigned long long mine[2];
        int rank[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int i = tid + q * FB_NT;
            mine[q] = i < static_cast<int>(n) ? cand[i] : 0ull;
            rank[q] = 0;
        }
        for (int jj = 0; jj < static_cast<int>(n); ++jj) {
            const unsigned long long o = cand[jj];
#pragma unroll
            for (int q = 0; q < 2; ++q) rank[q] += o > mine[q] ? 1 : 0;
        }
        __syncthreads();
#pragma unroll
        for (int q = 0; q < 2; ++q)
            if (tid + q * FB_NT < static_cast<int>(n)) cand[rank[q]] = mine[q];
        __syncthreads();
    } else {
        // bitonic over the next power of two, padded with key 0
        int P = 1;
        while (P < static_cast<int>(n)) P <<= 1;
        for (int i = static_cast<int>(n) + tid; i < P; i += FB_NT) cand[i] = 0ull;
        __syncthreads();
        for (int size = 2; size <= P; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                for (int q = tid; q < P / 2; q += FB_NT) {
                    const int i = 2 * q - (q & (stride - 1));
                    const unsigned long long a = cand[i], b = cand[i + stride];
                    if ((i & size) == 0 ? a < b : a > b) {
                        cand[i] = b;
                        cand[i + stride] = a;
                    }
                }
                __syncthreads();
            }
        }
    }
    // keys at or above cand[t - 1] (ties with it included): nk of them
    auto count_ge = [&](KT t) -> unsigned {
        if (tid == 0) s_nk = 0u;
        __syncthreads();
        for (int i = tid; i < static_cast<int>(n); i += FB_NT)
            if (key_of(i) >= t && (i + 1 == static_cast<int>(n) || key_of(i + 1) < t)) s_nk = static_cast<unsigned>(i + 1);
        __syncthreads();
        return s_nk;
    };
    KT lo = key_of(k - 1);
    const float M = FKey<E>::value_of(key_of(0));
    if (p.top_p > 0.f && p.top_p < 1.f) {
        const unsigned nk = count_ge(lo);
        // each thread a run of the sorted keys: its fixed-point masses, then an exclusive scan across the CTA
        const int per = (static_cast<int>(nk) + FB_NT - 1) / FB_NT;
        const int i0 = min(static_cast<int>(nk), tid * per), i1 = min(static_cast<int>(nk), i0 + per);
        auto mass = [&](int i) -> unsigned long long {
            return __float2ull_rz(ex2((FKey<E>::value_of(key_of(i)) - M) * p.c) * F_FIX);
        };
        unsigned long long loc = 0ull;
        for (int i = i0; i < i1; ++i) loc += mass(i);
        unsigned long long incl = loc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) s_wm[warp] = incl;
        if (tid == 0) s_first = 0xFFFFFFFFu;
        __syncthreads();
        unsigned long long before = 0ull, total = 0ull;
        for (int w2 = 0; w2 < FB_W; ++w2) {
            if (w2 < warp) before += s_wm[w2];
            total += s_wm[w2];
        }
        // top_p of the total, rounded up: the smallest fixed-point mass that reaches it
        const unsigned long long need =
            static_cast<unsigned long long>(ceil(static_cast<double>(p.top_p) * static_cast<double>(total)));
        unsigned long long run = before + incl - loc;
        for (int i = i0; i < i1; ++i) {
            run += mass(i);
            if (run >= need) {
                atomicMin(&s_first, static_cast<unsigned>(i));
                break;
            }
        }
        __syncthreads();
        lo = key_of(s_first);
    }

    // ---- 5. threshold, and the kept logits' (max, sum) by the draw's float comparison ----
    const float th = FKey<E>::value_of(lo);
    float sacc = 0.f;
    if (tid == 0) s_nk = 0u;
    __syncthreads();
    for (int i = tid; i < static_cast<int>(n); i += FB_NT) {
        const float x = FKey<E>::value_of(key_of(i));
        if (x >= th) {
            sacc += ex2((x - M) * p.c);
            // the values fall along the list, so the kept logits are its first nkeep entries
            if (i + 1 == static_cast<int>(n) || FKey<E>::value_of(key_of(i + 1)) < th) s_nk = static_cast<unsigned>(i + 1);
        }
    }
    const float ssum = cta_sum_fixed<FB_NT>(sacc, s_red);   // (its barriers also publish s_nk)
    const int nkeep = static_cast<int>(s_nk);
    if (tid == 0) {
        p.thr[r] = th;
        p.row_ms[r] = make_float2(M, ssum);
    }
    // ---- 6. a target row's kept logits for the draw, in vocabulary order (each entry's rank among the kept
    // element indices, which are distinct) ----
    if (r < p.rows_a_n) {
        if (nkeep <= p.list_cap) {
            const size_t base = static_cast<size_t>(r) * p.list_cap;
            for (int i = tid; i < nkeep; i += FB_NT) {
                const unsigned e = static_cast<unsigned>(cand[i]);
                int at = 0;
                for (int jj = 0; jj < nkeep; ++jj) at += static_cast<unsigned>(cand[jj]) < e ? 1 : 0;
                p.list_idx[base + at] = static_cast<int>(e);
                p.list_x[base + at] = FKey<E>::value_of(key_of(i));
            }
        }
        if (tid == 0) p.list_n[r] = nkeep <= p.list_cap ? nkeep : -1;
    }
}

}  // namespace specv
