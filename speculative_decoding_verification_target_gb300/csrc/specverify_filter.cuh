// Standardised sampling ("Speculative Decoding 为什么是 Lossless 的 — 详细证明教程", §8 Q4: temperature,
// top-k and top-p are folded into p and q, the same transforms for the target and the draft row, before the
// ratio is taken). Every such filter keeps the logits at or above a per-row threshold, so the filtered
// verification is the ordinary one on rows whose other logits are -inf:
//   - threshold_kernel: one CTA per row finds the threshold by radix selection on order-preserving integer
//     keys of the logits, 8 bits a pass from the top (2 passes for bf16, 4 for fp32). Top-k (0 < k < V)
//     descends by counts to the k-th largest value; top-p (0 < top_p < 1), on what top-k kept, descends by
//     the mass sum_x 2^((x - M) c) to the value at which the mass from the largest logit down first reaches
//     top_p of the kept total. Ties at a threshold are all kept (the kept set depends on values only);
//   - mask_kernel: writes the filtered rows (kept logits unchanged, the others -inf) into the caller's
//     workspace, and the chain kernels run on them.
// The masses of a pass are summed in a fixed order (one lane per warp adds its warp's values in lane order;
// warps are merged in warp order), so the threshold does not depend on timing.
#pragma once
#include "specverify_kernels.cuh"

namespace specv {

constexpr int FT_W = 16;                // warps per CTA of the threshold kernel
constexpr int FT_NT = FT_W * 32;

// order-preserving keys: a larger logit has a larger unsigned key (negative values reversed)
template <class E>
struct FKey;
template <>
struct FKey<Bf16> {
    using K = uint32_t;
    static constexpr int BITS = 16;
    __device__ static K key(const unsigned char* row, int e) {
        const uint32_t b = reinterpret_cast<const uint16_t*>(row)[e];
        return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
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
    __device__ static K key(const unsigned char* row, int e) {
        const uint32_t b = reinterpret_cast<const uint32_t*>(row)[e];
        return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
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
};

__device__ __forceinline__ const unsigned char* f_row(const FParams& p, long long r, size_t row_bytes) {
    return r < p.rows_a_n ? p.rows_a + static_cast<size_t>(r) * row_bytes
                          : p.rows_b + static_cast<size_t>(r - p.rows_a_n) * row_bytes;
}

template <class E>
__global__ void __launch_bounds__(FT_NT) threshold_kernel(const __grid_constant__ FParams p) {
    using KT = typename FKey<E>::K;
    constexpr int BITS = FKey<E>::BITS;
    __shared__ float s_hist[FT_W][256];   // per-warp histogram of this pass (counts or masses)
    __shared__ float s_tot[256];
    __shared__ unsigned s_sel[2];          // chosen bin, and the bins above it (as float bits: mass)
    __shared__ float s_red[FT_W];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long r = blockIdx.x;
    const int V = p.V;
    const size_t row_bytes = static_cast<size_t>(V) * E::BYTES;
    const unsigned char* row = f_row(p, r, row_bytes);
    const float NINF = __uint_as_float(0xFF800000u);

    // one radix pass: histogram (by 8-bit digit at `shift`) of the elements whose key is >= lo and whose
    // higher digits equal `prefix`; weight 1 (counts) or the element's mass 2^((x - M) c)
    auto pass = [&](KT prefix, int shift, KT lo, bool mass, float M) {
        for (int q = threadIdx.x; q < FT_W * 256; q += FT_NT) (&s_hist[0][0])[q] = 0.f;
        __syncthreads();
        const int nsteps = (V + FT_NT - 1) / FT_NT;
        for (int it = 0; it < nsteps; ++it) {
            const int e = it * FT_NT + threadIdx.x;
            int bin = -1;
            float w = 0.f;
            if (e < V) {
                const KT k = FKey<E>::key(row, e);
                const bool in = k >= lo && (shift + 8 >= BITS || (k >> (shift + 8)) == prefix);
                if (in) {
                    bin = static_cast<int>((k >> shift) & 0xFFu);
                    w = mass ? ex2((FKey<E>::value_of(k) - M) * p.c) : 1.f;
                }
            }
            // lane 0 adds the warp's 32 contributions in lane order (a fixed summation order)
            for (int src = 0; src < 32; ++src) {
                const int b = __shfl_sync(0xffffffffu, bin, src);
                const float v = __shfl_sync(0xffffffffu, w, src);
                if (lane == 0 && b >= 0) s_hist[warp][b] += v;
            }
        }
        __syncthreads();
        if (threadIdx.x < 256) {
            float t = 0.f;
            for (int w2 = 0; w2 < FT_W; ++w2) t += s_hist[w2][threadIdx.x];
            s_tot[threadIdx.x] = t;
        }
        __syncthreads();
    };
    // the bin, from the top, where the running total first reaches `need`; returns the total above it
    auto choose = [&](float need) -> float {
        if (threadIdx.x == 0) {
            float above = 0.f;
            int b = 0;
            for (b = 255; b > 0; --b) {
                if (above + s_tot[b] >= need) break;
                above += s_tot[b];
            }
            s_sel[0] = static_cast<unsigned>(b);
            s_sel[1] = __float_as_uint(above);
        }
        __syncthreads();
        const float above = __uint_as_float(s_sel[1]);
        return above;
    };

    KT lo = 0;                             // keep keys >= lo
    bool filtered = false;
    if (p.top_k > 0 && p.top_k < V) {
        KT prefix = 0;
        float need = static_cast<float>(p.top_k);
        for (int shift = BITS - 8; shift >= 0; shift -= 8) {
            pass(prefix, shift, 0, false, 0.f);
            need -= choose(need);
            prefix = (prefix << 8) | static_cast<KT>(s_sel[0]);
            __syncthreads();
        }
        lo = prefix;
        filtered = true;
    }
    if (p.top_p > 0.f && p.top_p < 1.f) {
        // the row's largest logit, then the kept total
        float m = NINF;
        for (int e = threadIdx.x; e < V; e += FT_NT) m = fmaxf(m, FKey<E>::value_of(FKey<E>::key(row, e)));
        m = warp_max(m);
        if (lane == 0) s_red[warp] = m;
        __syncthreads();
        float M = NINF;
        for (int w2 = 0; w2 < FT_W; ++w2) M = fmaxf(M, s_red[w2]);
        __syncthreads();
        KT prefix = 0;
        float need = 0.f;
        for (int shift = BITS - 8; shift >= 0; shift -= 8) {
            pass(prefix, shift, lo, true, M);
            if (shift == BITS - 8) {   // the first pass sees every kept element: its bins sum to the total
                if (threadIdx.x == 0) {
                    float t = 0.f;
                    for (int b = 255; b >= 0; --b) t += s_tot[b];
                    s_red[0] = t;
                }
                __syncthreads();
                need = p.top_p * s_red[0];
                __syncthreads();
            }
            need -= choose(need);
            prefix = (prefix << 8) | static_cast<KT>(s_sel[0]);
            __syncthreads();
        }
        if (!filtered || prefix > lo) lo = prefix;
        filtered = true;
    }
    if (threadIdx.x == 0) p.thr[r] = filtered ? FKey<E>::value_of(lo) : NINF;
}

// the filtered copies: logits at or above the row's threshold, -inf elsewhere
template <class E>
__global__ void __launch_bounds__(256) mask_kernel(const __grid_constant__ FParams p) {
    const size_t V = static_cast<size_t>(p.V);
    const size_t total = static_cast<size_t>(p.rows_n) * V;
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const long long r = static_cast<long long>(i / V);
        const size_t e = i - static_cast<size_t>(r) * V;
        const float t = p.thr[r];
        const unsigned char* src = r < p.rows_a_n ? p.rows_a + (static_cast<size_t>(r) * V + e) * E::BYTES
                                                  : p.rows_b + (static_cast<size_t>(r - p.rows_a_n) * V + e) * E::BYTES;
        unsigned char* dst = r < p.rows_a_n ? p.out_a + (static_cast<size_t>(r) * V + e) * E::BYTES
                                            : p.out_b + (static_cast<size_t>(r - p.rows_a_n) * V + e) * E::BYTES;
        if constexpr (E::BYTES == 2) {
            const uint16_t b = *reinterpret_cast<const uint16_t*>(src);
            const float x = __uint_as_float(static_cast<uint32_t>(b) << 16);
            *reinterpret_cast<uint16_t*>(dst) = x >= t ? b : static_cast<uint16_t>(0xFF80u);
        } else {
            const float x = *reinterpret_cast<const float*>(src);
            *reinterpret_cast<float*>(dst) = x >= t ? x : __uint_as_float(0xFF800000u);
        }
    }
}

}  // namespace specv
