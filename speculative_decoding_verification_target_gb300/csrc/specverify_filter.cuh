// Standardised sampling ("Speculative Decoding 为什么是 Lossless 的 — 详细证明教程", §8 Q4: temperature,
// top-k and top-p are folded into p and q, the same transforms for the target and the draft row, before the
// ratio is taken). Every such filter keeps the logits at or above a per-row threshold, so the filtered
// verification is the ordinary one on rows whose other logits are -inf:
//   - threshold_kernel: one CTA per row finds the threshold by radix selection on order-preserving integer
//     keys of the logits, 4 bits a pass from the top (4 passes for bf16, 8 for fp32). Top-k (0 < k < V)
//     descends by counts to the k-th largest value; top-p (0 < top_p < 1), on what top-k kept, descends by
//     the mass sum_x 2^((x - M) c) to the value at which the mass from the largest logit down first reaches
//     top_p of the kept total. Ties at a threshold are all kept (the kept set depends on values only). Once
//     the elements still in play fit in shared memory (at most F_CAP keys), one more pass over the row copies
//     them there and the remaining passes read only them;
//   - mask_kernel: writes the filtered rows (kept logits unchanged, the others -inf) into the caller's
//     workspace, and the chain kernels run on them.
// The histograms of a pass are integer sums, so they do not depend on the order of the additions: counts, and
// masses in 64-bit fixed point (2^-44 units; a mass 2^((x - M) c) is at most 1 and a row holds at most 2^18
// logits, so a bin cannot overflow). Each thread adds into its own column of the shared-memory histograms (no
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
    float* thr;                    // [rows_n] threshold value (-inf: nothing filtered)
    unsigned char* out_a;          // filtered copies, same layout as rows_a / rows_b
    unsigned char* out_b;
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

template <class E>
__global__ void __launch_bounds__(FT_NT) threshold_kernel(const __grid_constant__ FParams p) {
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
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long r = blockIdx.x;
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
    if (tid == 0) p.thr[r] = filtered ? FKey<E>::value_of(lo) : NINF;
}

// The filtered copies, one CTA per row: logits at or above the row's threshold, -inf elsewhere (16-byte words
// when every row allows them).
template <class E>
__global__ void __launch_bounds__(256) mask_kernel(const __grid_constant__ FParams p) {
    const long long r = blockIdx.x;
    const size_t V = static_cast<size_t>(p.V);
    const size_t row_bytes = V * E::BYTES;
    const float t = p.thr[r];
    const unsigned char* src = f_row(p, r, row_bytes);
    unsigned char* dst = r < p.rows_a_n ? p.out_a + static_cast<size_t>(r) * row_bytes
                                        : p.out_b + static_cast<size_t>(r - p.rows_a_n) * row_bytes;
    auto keep16 = [&](uint32_t b) -> uint32_t {   // a bf16 in the low half of b
        return __uint_as_float(b << 16) >= t ? b : 0xFF80u;
    };
    auto keep32 = [&](uint32_t b) -> uint32_t { return __uint_as_float(b) >= t ? b : 0xFF800000u; };
    if (p.vec) {
        const uint4* s4 = reinterpret_cast<const uint4*>(src);
        uint4* d4 = reinterpret_cast<uint4*>(dst);
        const size_t n4 = row_bytes / 16;
#pragma unroll 4
        for (size_t i = threadIdx.x; i < n4; i += blockDim.x) {
            uint4 w = __ldg(s4 + i);
            if constexpr (E::BYTES == 2) {
                w.x = keep16(w.x & 0xFFFFu) | (keep16(w.x >> 16) << 16);
                w.y = keep16(w.y & 0xFFFFu) | (keep16(w.y >> 16) << 16);
                w.z = keep16(w.z & 0xFFFFu) | (keep16(w.z >> 16) << 16);
                w.w = keep16(w.w & 0xFFFFu) | (keep16(w.w >> 16) << 16);
            } else {
                w.x = keep32(w.x);
                w.y = keep32(w.y);
                w.z = keep32(w.z);
                w.w = keep32(w.w);
            }
            d4[i] = w;
        }
        return;
    }
    for (size_t e = threadIdx.x; e < V; e += blockDim.x) {
        if constexpr (E::BYTES == 2) {
            const uint16_t b = reinterpret_cast<const uint16_t*>(src)[e];
            reinterpret_cast<uint16_t*>(dst)[e] = static_cast<uint16_t>(keep16(b));
        } else {
            reinterpret_cast<uint32_t*>(dst)[e] = keep32(reinterpret_cast<const uint32_t*>(src)[e]);
        }
    }
}

}  // namespace specv
