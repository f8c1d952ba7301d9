// Device helpers for sm_103a: bulk copies with mbarriers, cluster shared memory, Philox4x32-10,
// fast exp2 and warp reductions. Nothing here is shared with the CPU oracle.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace specv {

// ------------------------------------------------------------------------------------------------
// addresses, timers
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------------------------------------
// mbarrier + bulk (TMA, non-tensor) copies
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// try_wait that lets the thread sleep (up to `hint_ns`) until the phase completes: no hot polling.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Same, with acquire ordering at cluster scope (arrivals come from other CTAs of the cluster).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Waits for phase `parity` of `bar` to complete, giving up after `limit_ns` of wall time. Returns false
// (and ORs `flag` into *status) when it gave up. Between polls the warp sleeps (exponential backoff up to
// 256 ns) so that waiting warps do not take issue slots from the warps that compute. The wait cannot hang
// the GPU.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, unsigned* status,
                                                  unsigned flag, uint64_t limit_ns) {
    constexpr uint32_t HINT = 1000;   // ns
    if (CLUSTER ? mbar_try_wait_cluster(bar, parity, HINT) : mbar_try_wait_sleep(bar, parity, HINT)) return true;
    const uint64_t t0 = global_timer_ns();
    uint32_t backoff = 16;
    for (int it = 0;; ++it) {
        __nanosleep(backoff);
        if (backoff < 256) backoff <<= 1;
        if (CLUSTER ? mbar_try_wait_cluster(bar, parity, HINT) : mbar_try_wait_sleep(bar, parity, HINT)) return true;
        if ((it & 63) == 63 && global_timer_ns() - t0 > limit_ns) {
            atomicOr(status, flag);
            return false;
        }
    }
}

// Invalidates an mbarrier whose phases are all complete, so that its memory may be reused or initialised again.
__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Local arrive (release at CTA scope).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Orders this thread's earlier generic-proxy accesses to shared memory before its later async-proxy
// (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_mbarrier_init_cluster() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Bulk copy global -> this CTA's shared memory; completion is signalled as transaction bytes on `bar`.
// dst and src must be 16-byte aligned, bytes a multiple of 16. `policy` is an L2 cache policy from
// createpolicy (evict-first for data read for the last time).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ------------------------------------------------------------------------------------------------
// thread-block cluster
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
// Address of the same shared-memory variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local_smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_smem_addr), "r"(rank));
    return r;
}
// Load of a float from the shared memory of a CTA of the cluster (address from map_to_rank).
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
// Full cluster barrier; release/acquire orders the shared::cluster stores issued before it.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ------------------------------------------------------------------------------------------------
// math
// ------------------------------------------------------------------------------------------------
// 2^x via the SFU (ex2.approx, flush-to-zero): relative error ~2^-22; 2^-inf = 0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// log2(x) via the SFU (lg2.approx): absolute error ~2^-22 for x near 1.
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Float-float numbers: an unevaluated sum hi + lo of two floats with |lo| <= ulp(hi) / 2, about 44
// significant bits, built on the error-free sum of two floats (Knuth's TwoSum; Dekker's FastTwoSum when the
// first operand is the larger). The intrinsics keep the compiler from contracting or reordering the steps.
struct FF {
    float hi, lo;
};
__device__ __forceinline__ FF ff_two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return {s, e};
}
__device__ __forceinline__ FF ff_fast_two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ FF ff_add(FF a, FF b) {
    const FF s = ff_two_sum(a.hi, b.hi);
    return ff_fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}
__device__ __forceinline__ FF ff_addf(FF a, float b) {
    const FF s = ff_two_sum(a.hi, b);
    return ff_fast_two_sum(s.hi, __fadd_rn(s.lo, a.lo));
}
__device__ __forceinline__ FF ff_sub(FF a, FF b) { return ff_add(a, FF{-b.hi, -b.lo}); }
// a * u for a float u (the product's rounding error recovered with one fused multiply-add)
__device__ __forceinline__ FF ff_mulf(FF a, float u) {
    const float p = __fmul_rn(a.hi, u);
    const float e = __fmaf_rn(a.lo, u, __fmaf_rn(a.hi, u, -p));
    return ff_fast_two_sum(p, e);
}
__device__ __forceinline__ bool ff_gt(FF a, FF b) { return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo); }
__device__ __forceinline__ FF ff_shfl(FF v, int src) {
    return {__shfl_sync(0xffffffffu, v.hi, src), __shfl_sync(0xffffffffu, v.lo, src)};
}
__device__ __forceinline__ FF ff_shfl_up(FF v, int d) {
    return {__shfl_up_sync(0xffffffffu, v.hi, d), __shfl_up_sync(0xffffffffu, v.lo, d)};
}
__device__ __forceinline__ FF warp_sum(FF v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = ff_add(v, FF{__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)});
    return v;
}
// Inclusive scan across the warp (Hillis-Steele, fixed association order).
__device__ __forceinline__ FF warp_incl_scan_ff(FF v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const FF y = ff_shfl_up(v, o);
        if (lane >= o) v = ff_add(v, y);
    }
    return v;
}
// a * b for floats a, b as a float-float (the product's rounding error recovered with one fused multiply-add)
__device__ __forceinline__ FF ff_two_prod(float a, float b) {
    const float p = __fmul_rn(a, b);
    return {p, __fmaf_rn(a, b, -p)};
}
// a * b for float-floats (the lo * lo term, below the result's precision, is dropped)
__device__ __forceinline__ FF ff_mul(FF a, FF b) {
    const FF p = ff_two_prod(a.hi, b.hi);
    return ff_fast_two_sum(p.hi, __fadd_rn(p.lo, __fmaf_rn(a.hi, b.lo, __fmul_rn(a.lo, b.hi))));
}
// Square root of a float-float x >= 0: the float root y0 and one Newton step on the exact residual
// x - y0^2, y = y0 + (x - y0^2) / (2 y0).
__device__ __forceinline__ FF ff_sqrt(FF x) {
    if (!(x.hi > 0.f)) return {0.f, 0.f};
    const float y0 = __fsqrt_rn(x.hi);
    const FF sq = ff_two_prod(y0, y0);
    const float r = __fadd_rn(__fadd_rn(__fsub_rn(x.hi, sq.hi), -sq.lo), x.lo);   // x - y0^2 (x.hi - sq.hi exact)
    return ff_fast_two_sum(y0, __fdiv_rn(r, __fmul_rn(2.f, y0)));
}
// a / b for float-floats, b > 0: the float quotient and one correction with the exact residual.
__device__ __forceinline__ FF ff_div(FF a, FF b) {
    const float q0 = __fdiv_rn(a.hi, b.hi);
    const FF r = ff_sub(a, ff_mul(b, FF{q0, 0.f}));
    return ff_fast_two_sum(q0, __fdiv_rn(__fadd_rn(r.hi, r.lo), b.hi));
}
__device__ __forceinline__ void st_cluster_f32x2(uint32_t addr, float a, float b) {
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}
__device__ __forceinline__ float2 ld_cluster_f32x2(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
    return v;
}

// Online (max, sum of 2^((x - max) c)) pair; s == 0 marks an empty set (every logit -inf).
struct MaxSum {
    float m, s;
};
__device__ __forceinline__ MaxSum ms_merge(MaxSum a, MaxSum b, float c) {
    if (a.s == 0.f) return b;
    if (b.s == 0.f) return a;
    const float m = fmaxf(a.m, b.m);
    return {m, a.s * ex2((a.m - m) * c) + b.s * ex2((b.m - m) * c)};
}
// Warp-wide max of a float (one redux instruction on sm_100-family GPUs).
__device__ __forceinline__ float warp_max(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

// Warp-wide merge of (max, sum) pairs: M = max of the lanes' maxima, S = sum of s * 2^((m - M) c).
// One redux, one exp2 per lane and a butterfly sum: every lane returns the same pair.
__device__ __forceinline__ MaxSum warp_ms(MaxSum v, float c) {
    const bool has = v.s > 0.f;
    const float M = warp_max(has ? v.m : __uint_as_float(0xFF800000u));
    const float s = has ? v.s * ex2((v.m - M) * c) : 0.f;
    return {M, warp_sum(s)};
}

// ------------------------------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11):
// ten rounds of the 4x32 multiply-xor S-box, key bumped by the Weyl constants between rounds.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t philox_word0(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                 uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
        const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    return c0;
}

// Uniform for (seed, sequence b, position j, stream): counter (j, b, stream, 0), key (seed lo, seed hi),
// word 0 mapped to (k + 1/2) 2^-23 with k = w >> 9 (exact in fp32).
__device__ __forceinline__ float philox_uniform(uint64_t seed, uint32_t b, uint32_t j, uint32_t stream) {
    const uint32_t w = philox_word0(j, b, stream, 0u, static_cast<uint32_t>(seed),
                                    static_cast<uint32_t>(seed >> 32));
    return (static_cast<float>(w >> 9) + 0.5f) * (1.0f / 8388608.0f);
}

}  // namespace specv
