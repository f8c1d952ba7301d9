// Host side of the C ABI declared in include/specverify.h: argument validation, launch configuration
// (statistics grid, ring depth, draw clusters) and the launches.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <mutex>

#include "specverify.h"
#include "specverify_internal.h"
#include "specverify_filter.cuh"
#include "specverify_gamma.cuh"

namespace specv {
namespace {

thread_local char g_err[512] = "";

spec_status fail(spec_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return s;
}

constexpr int MAX_K = 64;
constexpr int MAX_V = 262144;
static_assert(MAX_V == FB_MAX_V, "the bound kernel sizes its line keys for the largest vocabulary");
constexpr int MAX_N = 64;
constexpr size_t WS_HEADER = 256;          // status word + padding
constexpr int SMEM_MAX_PER_CTA = 232448;   // opt-in maximum per CTA

int g_stats_grid_override = 0;   // CTAs of the statistics kernel (0 = automatic)
int g_gamma_one_launch = 0;      // 1: a counterfactual call with a selected drafter runs as one launch
float g_draw_tau = 0.f;          // chunk mass above which the draw takes its float-float path (0 = default)
thread_local int g_last_plan[5] = {0, 0, 0, 0, 0};   // see spec_debug_last_plan

// Workspace layout: [status header][row partials]. The row partials are the statistics pass's segment
// (max, sum) pairs (segment (warp g, row r) at entry g + r: fewer than min(G, pieces) + rows entries, sized
// for the largest grid) or, for the gamma kernel, one (max, sum) pair per statistics row (B (2K + 1)).
struct WsLayout {
    size_t part_off, total;
};

WsLayout ws_layout(int B, int K, int V, int N) {
    (void)N;
    WsLayout w;
    w.part_off = WS_HEADER;
    const long long srows = static_cast<long long>(B) * (2 * K + 1);
    const long long pieces = srows * ((V + PE - 1) / PE);
    const long long gmax = static_cast<long long>(S_MAX_CTAS) * SW;
    w.total = w.part_off + static_cast<size_t>(std::min(pieces, gmax) + srows) * sizeof(float2);
    w.total = (w.total + 15) / 16 * 16;
    return w;
}

// Workspace of spec_verify_filtered: [the verify workspace][row thresholds][filtered target rows][filtered
// draft rows], each region 256-byte aligned.
// spec_verify's workspace, then per row a threshold and the kept logits' (max, sum), then per target row the
// count, element indices and values of its kept logits when they are few (D_LIST_CAP at most).
struct FilterLayout {
    size_t thr_off, ms_off, ln_off, li_off, lx_off, total;
};
FilterLayout filter_layout(int B, int K, int V) {
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    FilterLayout f;
    const size_t rows = static_cast<size_t>(B) * (2 * K + 1), rows_a = static_cast<size_t>(B) * (K + 1);
    f.thr_off = up(ws_layout(B, K, V, 1).total);
    f.ms_off = up(f.thr_off + rows * sizeof(float));
    f.ln_off = up(f.ms_off + rows * sizeof(float2));
    f.li_off = up(f.ln_off + rows_a * sizeof(int));
    f.lx_off = up(f.li_off + rows_a * D_LIST_CAP * sizeof(int));
    f.total = up(f.lx_off + rows_a * D_LIST_CAP * sizeof(float));
    return f;
}

struct Call {
    const void* target;
    const void* others;
    spec_dtype dtype;
    const int32_t* tokens;
    const uint64_t* seeds;
    int B, K, V, N, selected;
    float temperature, delta;
    int cactus;
    float* gamma;
    float* loss;
    int32_t* accept_len;
    int32_t* out_tokens;
    float* diag;
    float* gamma_star;
    const float* thr;   // standardised sampling: per statistics row, the logits below it count as -inf (or null)
    const int* list_n;  // standardised sampling: the target rows' kept logits listed for the draw
    const int* list_idx;
    const float* list_x;
    void* workspace;
    size_t workspace_bytes;
    cudaStream_t stream;
};

// CTAs of the statistics kernel resident at once (occupancy x SMs, cached per device and shared memory).
using StatsFn = void (*)(const SParams);
std::mutex g_socc_mu;
struct SOccEntry {
    StatsFn fn;
    size_t smem;
    int device, ctas;
};
SOccEntry g_socc[16];
int g_socc_n = 0;

cudaError_t stats_ctas(StatsFn fn, size_t smem, int& out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lk(g_socc_mu);
        for (int i = 0; i < g_socc_n; ++i)
            if (g_socc[i].fn == fn && g_socc[i].smem == smem && g_socc[i].device == dev) {
                out = g_socc[i].ctas;
                return cudaSuccess;
            }
    }
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX_PER_CTA);
    if (e != cudaSuccess) return e;
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, SNT, smem);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (per_sm < 1 || sms < 1) return cudaErrorInvalidConfiguration;
    out = std::min(per_sm * sms, S_MAX_CTAS);
    std::lock_guard<std::mutex> lk(g_socc_mu);
    if (g_socc_n < 16) g_socc[g_socc_n++] = {fn, smem, dev, out};
    return cudaSuccess;
}

// Raises the dynamic shared-memory ceiling of a draw or gamma kernel once per device (the draw's bulk-copy
// slots take 128 KB for bf16 rows, the gamma kernel's ring 197 KB).
std::mutex g_dsm_mu;
struct DsmEntry {
    const void* fn;
    int device;
    int cap;
};
DsmEntry g_dsm[32];
int g_dsm_n = 0;

// Raises a kernel's dynamic shared-memory limit to all that its static shared memory leaves of the per-CTA
// maximum (once per kernel and device) and returns that limit in *cap.
template <class Fn>
cudaError_t dyn_smem_ceiling(Fn fn, int dev, int* cap) {
    std::lock_guard<std::mutex> lk(g_dsm_mu);
    for (int i = 0; i < g_dsm_n; ++i)
        if (g_dsm[i].fn == reinterpret_cast<const void*>(fn) && g_dsm[i].device == dev) {
            *cap = g_dsm[i].cap;
            return cudaSuccess;
        }
    cudaFuncAttributes at = {};
    cudaError_t e = cudaFuncGetAttributes(&at, fn);
    if (e != cudaSuccess) return e;
    const int c = SMEM_MAX_PER_CTA - static_cast<int>(at.sharedSizeBytes);
    if (c <= 0) return cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, c);
    if (e != cudaSuccess) return e;
    if (g_dsm_n < 32) g_dsm[g_dsm_n++] = {reinterpret_cast<const void*>(fn), dev, c};
    *cap = c;
    return cudaSuccess;
}

// Constants of the draw's float-float arithmetic, from double precision: 2^(k/32) for k = -16..16, ln 2 and
// c = log2(e) / T, each split into a float pair; and the chunk mass above which a chunk takes the exact path.
FFc ff_constants(float temperature) {
    FFc k = {};
    auto split = [](double v) { const float h = static_cast<float>(v); return make_float2(h, static_cast<float>(v - h)); };
    for (int j = -16; j <= 16; ++j) k.tab[j + 16] = split(std::exp2(j / 32.0));
    const double ln2 = std::log(2.0);
    const float2 l = split(ln2);
    k.ln2_hi = l.x;
    k.ln2_lo = l.y;
    // c_hi rounded towards zero, so that c_lo > 0: a -inf logit then gives -inf * c_lo + l = -inf and an
    // exponent of -inf (a negative c_lo would make it -inf + inf = NaN)
    const double cd = 1.0 / (ln2 * static_cast<double>(temperature));
    float ch = static_cast<float>(cd);
    if (static_cast<double>(ch) >= cd) ch = std::nextafter(ch, 0.f);
    k.c_hi = ch;
    k.c_lo = static_cast<float>(cd - static_cast<double>(ch));
    k.tau = g_draw_tau > 0.f ? g_draw_tau : D_TAU;
    return k;
}

// The chain and its draw for one drafter (one cluster per sequence), launched with programmatic stream
// serialisation behind the kernel that computed the row statistics: either the segment partials of
// stats_kernel (part, P pieces over G warps) or whole-row pairs (row_ms, from gamma_kernel).
// The draw's parameters for one drafter (everything but the cluster size and the bulk-copy mode).
DParams draw_params(const Call& a, const unsigned char* draft, const float2* part, const float2* row_ms,
                    long long P, int G, unsigned* status) {
    DParams d = {};
    d.target = static_cast<const unsigned char*>(a.target);
    d.draft = draft;
    d.part = part;
    d.row_ms = row_ms;
    d.P = P;
    d.G = G;
    d.np = (a.V + PE - 1) / PE;
    d.rows_a_n = static_cast<long long>(a.B) * (a.K + 1);
    d.tokens = a.tokens;
    d.seeds = a.seeds;
    d.B = a.B;
    d.K = a.K;
    d.V = a.V;
    d.c = static_cast<float>(1.4426950408889634 / static_cast<double>(a.temperature));
    d.delta = a.delta;
    // delta = 0 makes gamma* = p_target(n) and the scale 1 exactly: the standard draw
    d.cactus = a.delta > 0.f ? a.cactus : 0;
    d.k = ff_constants(a.temperature);
    d.accept_len = a.accept_len;
    d.out_tokens = a.out_tokens;
    d.diag = a.diag;
    d.gamma_star = a.gamma_star;
    d.thr = a.thr;
    d.list_n = a.list_n;
    d.list_idx = a.list_idx;
    d.list_x = a.list_x;
    d.list_cap = D_LIST_CAP;
    d.status = status;
    return d;
}

spec_status launch_draw(const Call& a, bool aligned, const unsigned char* draft, const float2* part,
                        const float2* row_ms, long long P, int G, unsigned* status) {
    const int eb = a.dtype == SPEC_BF16 ? 2 : 4;
    DParams d = draw_params(a, draft, part, row_ms, P, G, status);
    // CTAs per sequence: the largest power of two up to D_MAX_CPS that keeps the grid within one CTA per SM
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "device query failed: %s", cudaGetErrorString(e));
    int cps = 1;
    while (cps < D_MAX_CPS && static_cast<long long>(a.B) * cps * 2 <= sms) cps *= 2;
    d.cps = cps;
    // (bulk-copy mode) a two-piece slot and an mbarrier per warp, when they fit
    const size_t ring_bytes = static_cast<size_t>(DW) * (2 * static_cast<size_t>(PE) * eb + sizeof(uint64_t));
    using DrawFn = void (*)(const DParams);
    DrawFn dfn;
    if (a.thr) dfn = a.dtype == SPEC_BF16 ? (aligned ? draw_kernel<Bf16, true, true> : draw_kernel<Bf16, false, true>)
                                          : (aligned ? draw_kernel<F32, true, true> : draw_kernel<F32, false, true>);
    else dfn = a.dtype == SPEC_BF16 ? (aligned ? draw_kernel<Bf16, true> : draw_kernel<Bf16, false>)
                                    : (aligned ? draw_kernel<F32, true> : draw_kernel<F32, false>);
    int dsmem_cap = 0;
    e = dyn_smem_ceiling(dfn, dev, &dsmem_cap);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "draw kernel attribute failed: %s", cudaGetErrorString(e));
    d.tma = aligned && ring_bytes <= static_cast<size_t>(dsmem_cap) ? 1 : 0;
    const size_t dsmem = d.tma ? ring_bytes : 0;
    // its CTAs start as the grid before it frees SMs and wait for it (griddepcontrol.wait) after reading
    // their inputs
    cudaLaunchAttribute da[2];
    da[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    da[0].val.programmaticStreamSerializationAllowed = 1;
    da[1].id = cudaLaunchAttributeClusterDimension;
    da[1].val.clusterDim.x = static_cast<unsigned>(cps);
    da[1].val.clusterDim.y = 1;
    da[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t dc = {};
    dc.gridDim = dim3(static_cast<unsigned>(a.B * cps), 1, 1);
    dc.blockDim = dim3(DNT, 1, 1);
    dc.dynamicSmemBytes = dsmem;
    dc.stream = a.stream;
    dc.attrs = da;
    dc.numAttrs = 2;
    e = cudaLaunchKernelEx(&dc, dfn, d);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "draw kernel launch failed: %s", cudaGetErrorString(e));
    return SPEC_OK;
}

// Chain verification of one drafter (standard and Cactus): statistics pass over every row, then one cluster
// per sequence for the chain and its draw (specverify_chain.cuh).
spec_status run_chain(const Call& a, bool aligned) {
    const int eb = a.dtype == SPEC_BF16 ? 2 : 4;
    const WsLayout wl = ws_layout(a.B, a.K, a.V, a.N);
    unsigned char* ws = static_cast<unsigned char*>(a.workspace);
    SParams s = {};
    s.rows_a = static_cast<const unsigned char*>(a.target);
    s.rows_b = static_cast<const unsigned char*>(a.others);
    s.rows_a_n = static_cast<long long>(a.B) * (a.K + 1);
    s.rows_n = s.rows_a_n + static_cast<long long>(a.B) * a.K;
    s.V = a.V;
    s.np = (a.V + PE - 1) / PE;
    s.P = s.rows_n * s.np;
    s.c = static_cast<float>(1.4426950408889634 / static_cast<double>(a.temperature));
    s.tma = aligned ? 1 : 0;
    const size_t slot_bytes = static_cast<size_t>(PE) * eb;
    int R = S_MAX_R;
    while (R > 1 && static_cast<size_t>(SW) * R * (slot_bytes + 8) > static_cast<size_t>(SMEM_MAX_PER_CTA)) --R;
    s.R = R;
    const size_t smem = s.tma ? static_cast<size_t>(SW) * R * (slot_bytes + 8) : 0;
    StatsFn sfn = a.dtype == SPEC_BF16 ? stats_kernel<Bf16> : stats_kernel<F32>;
    int ctas = 0;
    cudaError_t e = stats_ctas(sfn, smem, ctas);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "occupancy query failed: %s", cudaGetErrorString(e));
    if (g_stats_grid_override > 0) ctas = g_stats_grid_override;
    const long long need = (s.P + SW - 1) / SW;   // no more warps than pieces
    if (ctas > need) ctas = static_cast<int>(need);
    s.G = ctas * SW;
    s.part = reinterpret_cast<float2*>(ws + wl.part_off);
    // L2 kept for the draw: the rows of the first positions, up to 64 MB (whole positions while they fit,
    // else position 0 of the first sequences)
    {
        const size_t budget = size_t(64) << 20;
        const size_t pair = 2 * static_cast<size_t>(a.V) * eb;
        s.K = a.K;
        const size_t per_position = pair * static_cast<size_t>(a.B);
        s.keep_j = static_cast<int>(std::min<size_t>(a.K, budget / per_position));
        s.keep_b = a.B;
        if (s.keep_j == 0) {
            s.keep_j = 1;
            s.keep_b = static_cast<int>(budget / pair);
        }
    }
    s.status = reinterpret_cast<unsigned*>(ws);
    g_last_plan[0] = 0;
    g_last_plan[1] = R;
    g_last_plan[2] = ctas;
    g_last_plan[3] = 0;
    g_last_plan[4] = s.np;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
    cfg.blockDim = dim3(SNT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = a.stream;
    e = cudaLaunchKernelEx(&cfg, sfn, s);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "statistics kernel launch failed: %s", cudaGetErrorString(e));

    return launch_draw(a, aligned, static_cast<const unsigned char*>(a.others), s.part, nullptr, s.P, s.G, s.status);
}

// Greedy verification: the statistics pass in its argmax mode over the target rows, then one warp per
// sequence for the chain.
spec_status run_greedy(const void* target, spec_dtype dtype, const int32_t* tokens, int B, int K, int V,
                       int32_t* accept_len, int32_t* out_tokens, void* workspace, cudaStream_t stream) {
    const int eb = dtype == SPEC_BF16 ? 2 : 4;
    const bool aligned = (reinterpret_cast<uintptr_t>(target) & 15) == 0 && (static_cast<size_t>(V) * eb) % 16 == 0 &&
                         V % CHUNK == 0;
    const WsLayout wl = ws_layout(B, K, V, 1);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    SParams s = {};
    s.rows_a = static_cast<const unsigned char*>(target);
    s.rows_b = nullptr;
    s.rows_a_n = static_cast<long long>(B) * (K + 1);
    s.rows_n = s.rows_a_n;
    s.V = V;
    s.np = (V + PE - 1) / PE;
    s.P = s.rows_n * s.np;
    s.c = 1.f;
    s.tma = aligned ? 1 : 0;
    s.K = K;
    s.keep_j = 0;   // every logit is read once
    s.keep_b = 0;
    const size_t slot_bytes = static_cast<size_t>(PE) * eb;
    int R = S_MAX_R;
    while (R > 1 && static_cast<size_t>(SW) * R * (slot_bytes + 8) > static_cast<size_t>(SMEM_MAX_PER_CTA)) --R;
    s.R = R;
    const size_t smem = s.tma ? static_cast<size_t>(SW) * R * (slot_bytes + 8) : 0;
    StatsFn sfn = dtype == SPEC_BF16 ? stats_kernel<Bf16, true> : stats_kernel<F32, true>;
    int ctas = 0;
    cudaError_t e = stats_ctas(sfn, smem, ctas);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "occupancy query failed: %s", cudaGetErrorString(e));
    if (g_stats_grid_override > 0) ctas = g_stats_grid_override;
    const long long need = (s.P + SW - 1) / SW;
    if (ctas > need) ctas = static_cast<int>(need);
    s.G = ctas * SW;
    s.part = reinterpret_cast<float2*>(ws + wl.part_off);
    s.status = reinterpret_cast<unsigned*>(ws);
    g_last_plan[0] = 0;
    g_last_plan[1] = R;
    g_last_plan[2] = ctas;
    g_last_plan[3] = 3;
    g_last_plan[4] = s.np;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
    cfg.blockDim = dim3(SNT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    e = cudaLaunchKernelEx(&cfg, sfn, s);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "statistics kernel launch failed: %s", cudaGetErrorString(e));
    GrParams gp = {};
    gp.part = s.part;
    gp.P = s.P;
    gp.G = s.G;
    gp.np = s.np;
    gp.tokens = tokens;
    gp.B = B;
    gp.K = K;
    gp.V = V;
    gp.accept_len = accept_len;
    gp.out_tokens = out_tokens;
    gp.status = s.status;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t gc = {};
    gc.gridDim = dim3(static_cast<unsigned>((B + 7) / 8), 1, 1);
    gc.blockDim = dim3(256, 1, 1);
    gc.stream = stream;
    gc.attrs = at;
    gc.numAttrs = 1;
    e = cudaLaunchKernelEx(&gc, greedy_chain_kernel, gp);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "greedy chain kernel launch failed: %s", cudaGetErrorString(e));
    return SPEC_OK;
}

// Counterfactual gamma for N drafters (gamma_kernel, one CTA per SM, rows whole per CTA), followed by the
// chain and draw of drafter `selected` when one is given.
spec_status run_gamma(const Call& a, bool aligned) {
    const int eb = a.dtype == SPEC_BF16 ? 2 : 4;
    const WsLayout wl = ws_layout(a.B, a.K, a.V, a.N);
    unsigned char* ws = static_cast<unsigned char*>(a.workspace);
    const bool chain = a.selected >= 0;
    CgParams g = {};
    g.target = static_cast<const unsigned char*>(a.target);
    g.drafters = static_cast<const unsigned char*>(a.others);
    g.B = a.B;
    g.K = a.K;
    g.V = a.V;
    g.N = a.N;
    const int pe = G_PIECE_BYTES / eb;
    g.np = (a.V + pe - 1) / pe;
    g.U = static_cast<long long>(a.B) * a.K * (a.N + 1) + (chain ? a.B : 0);
    if (g.U >= (1LL << 31))
        return fail(SPEC_ERR_UNSUPPORTED, "B (K (N + 1) + 1) = %lld rows exceed the gamma kernel's 2^31 row index", g.U);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess || sms < 1) return fail(SPEC_ERR_CUDA, "device query failed: %s", cudaGetErrorString(e));
    g.G = static_cast<int>(std::min<long long>(sms, g.U));
    g.c = static_cast<float>(1.4426950408889634 / static_cast<double>(a.temperature));
    g.tma = aligned ? 1 : 0;
    g.selected = chain ? a.selected : -1;
    g.gamma = a.gamma;
    g.loss = a.loss;
    g.row_ms = chain ? reinterpret_cast<float2*>(ws + wl.part_off) : nullptr;
    g.status = reinterpret_cast<unsigned*>(ws);
    using GammaFn = void (*)(const CgParams);
    GammaFn gfn = a.dtype == SPEC_BF16 ? gamma_kernel<Bf16> : gamma_kernel<F32>;
    int gcap = 0;
    e = dyn_smem_ceiling(gfn, dev, &gcap);
    if (e == cudaSuccess && G_SMEM > static_cast<size_t>(gcap)) e = cudaErrorInvalidValue;
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "gamma kernel attribute failed: %s", cudaGetErrorString(e));
    g_last_plan[0] = 0;
    g_last_plan[1] = G_R;
    g_last_plan[2] = g.G;
    g_last_plan[3] = 2;
    g_last_plan[4] = g.np;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(g.G), 1, 1);
    cfg.blockDim = dim3(GNT, 1, 1);
    cfg.dynamicSmemBytes = G_SMEM;   // also in the unaligned mode: keeps one CTA per SM for the TMEM allocation
    cfg.stream = a.stream;
    if (chain && aligned && g_gamma_one_launch) {
        // gamma and the chain in one cooperative launch (every CTA resident: one per SM)
        FuseParams f = {};
        f.g = g;
        const unsigned char* draft =
            g.drafters + static_cast<size_t>(a.selected) * a.B * a.K * static_cast<size_t>(a.V) * eb;
        f.d = draw_params(a, draft, nullptr, g.row_ms, 0, 0, g.status);
        f.d.cps = 1;
        f.d.tma = a.dtype == SPEC_BF16 ? 1 : 0;   // bf16 slots fit below the DrawShared block
        f.bar = reinterpret_cast<unsigned*>(ws) + 1;
        using FusedFn = void (*)(const FuseParams);
        FusedFn ffn = a.dtype == SPEC_BF16 ? gamma_chain_kernel<Bf16> : gamma_chain_kernel<F32>;
        int fcap = 0;
        e = dyn_smem_ceiling(ffn, dev, &fcap);
        if (e == cudaSuccess && G_SMEM > static_cast<size_t>(fcap)) e = cudaErrorInvalidValue;
        if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "one-launch kernel attribute failed: %s", cudaGetErrorString(e));
        cudaLaunchAttribute ca[1];
        ca[0].id = cudaLaunchAttributeCooperative;
        ca[0].val.cooperative = 1;
        cfg.attrs = ca;
        cfg.numAttrs = 1;
        g_last_plan[3] = 5;
        e = cudaLaunchKernelEx(&cfg, ffn, f);
        if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "one-launch kernel launch failed: %s", cudaGetErrorString(e));
        return SPEC_OK;
    }
    e = cudaLaunchKernelEx(&cfg, gfn, g);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "gamma kernel launch failed: %s", cudaGetErrorString(e));
    if (!chain) return SPEC_OK;
    const unsigned char* draft = g.drafters + static_cast<size_t>(a.selected) * a.B * a.K * static_cast<size_t>(a.V) * eb;
    return launch_draw(a, aligned, draft, nullptr, g.row_ms, 0, 0, g.status);
}

// Standardised sampling: the per-row thresholds and the kept logits' (max, sum), then the draw kernel in its
// filtering form (a logit below its row's threshold is -inf as it is read). Top-k up to FB_MAX_K on rows of
// whole 16-byte words goes through bound_kernel, which leaves the rows it cannot settle to threshold_kernel
// and lists each settled target row's kept logits (up to D_LIST_CAP) for the draw; every other filter goes
// through threshold_kernel alone, and the draw reads those rows whole. No filter at all is spec_verify itself.
spec_status run_filtered(const Call& a, int top_k, float top_p) {
    const int eb = a.dtype == SPEC_BF16 ? 2 : 4;
    const bool rows16 = ((reinterpret_cast<uintptr_t>(a.target) | reinterpret_cast<uintptr_t>(a.others)) & 15) == 0 &&
                        (static_cast<size_t>(a.V) * eb) % 16 == 0;
    const bool aligned = rows16 && a.V % CHUNK == 0;
    const bool by_k = top_k > 0 && top_k < a.V, by_p = top_p < 1.f;
    if (!by_k && !by_p) return run_chain(a, aligned);
    const FilterLayout fl = filter_layout(a.B, a.K, a.V);
    unsigned char* ws = static_cast<unsigned char*>(a.workspace);
    FParams f = {};
    f.rows_a = static_cast<const unsigned char*>(a.target);
    f.rows_b = static_cast<const unsigned char*>(a.others);
    f.rows_a_n = static_cast<long long>(a.B) * (a.K + 1);
    f.rows_n = f.rows_a_n + static_cast<long long>(a.B) * a.K;
    f.V = a.V;
    f.c = static_cast<float>(1.4426950408889634 / static_cast<double>(a.temperature));
    f.top_k = by_k ? top_k : 0;
    f.top_p = top_p;
    f.thr = reinterpret_cast<float*>(ws + fl.thr_off);
    f.row_ms = reinterpret_cast<float2*>(ws + fl.ms_off);
    f.list_n = reinterpret_cast<int*>(ws + fl.ln_off);
    f.list_idx = reinterpret_cast<int*>(ws + fl.li_off);
    f.list_x = reinterpret_cast<float*>(ws + fl.lx_off);
    f.list_cap = D_LIST_CAP;
    f.vec = rows16 ? 1 : 0;
    using ThrFn = void (*)(const FParams);
    ThrFn tfn = a.dtype == SPEC_BF16 ? threshold_kernel<Bf16> : threshold_kernel<F32>;
    int dev = 0, tcap = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = dyn_smem_ceiling(tfn, dev, &tcap);
    if (e == cudaSuccess && F_SMEM > static_cast<size_t>(tcap)) e = cudaErrorInvalidValue;
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "threshold kernel attribute failed: %s", cudaGetErrorString(e));
    const bool bound = by_k && top_k <= FB_MAX_K && rows16;
    unsigned grid = static_cast<unsigned>(f.rows_n);
    if (bound) {
        if (a.dtype == SPEC_BF16) bound_kernel<Bf16><<<static_cast<unsigned>(f.rows_n), FB_NT, 0, a.stream>>>(f);
        else bound_kernel<F32><<<static_cast<unsigned>(f.rows_n), FB_NT, 0, a.stream>>>(f);
        e = cudaGetLastError();
        if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "bound kernel launch failed: %s", cudaGetErrorString(e));
        // the rows it left: CTAs striding over the rows, one wave of them
        f.flagged_only = 1;
        grid = static_cast<unsigned>(std::min<long long>(f.rows_n, 2LL * sms));
    }
    tfn<<<grid, FT_NT, F_SMEM, a.stream>>>(f);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "threshold kernel launch failed: %s", cudaGetErrorString(e));
    g_last_plan[0] = 0;
    g_last_plan[1] = 0;
    g_last_plan[2] = static_cast<int>(grid);
    g_last_plan[3] = bound ? 6 : 7;
    g_last_plan[4] = (a.V + PE - 1) / PE;
    Call c = a;
    c.thr = f.thr;
    c.list_n = f.list_n;
    c.list_idx = f.list_idx;
    c.list_x = f.list_x;
    return launch_draw(c, aligned, static_cast<const unsigned char*>(a.others), nullptr, f.row_ms, 0, 0,
                       reinterpret_cast<unsigned*>(ws));
}

spec_status run(const Call& a) {
    if (a.B == 0) return SPEC_OK;
    const int eb = a.dtype == SPEC_BF16 ? 2 : 4;
    const bool chain = a.selected >= 0;
    const uintptr_t align_mask = 15;
    // bulk copies need 16-byte aligned pieces of whole 8-logit chunks
    const bool aligned = ((reinterpret_cast<uintptr_t>(a.target) | reinterpret_cast<uintptr_t>(a.others)) & align_mask) == 0 &&
                         (static_cast<size_t>(a.V) * eb) % 16 == 0 && a.V % CHUNK == 0;
    if (a.gamma) return run_gamma(a, aligned);
    if (chain && a.N == 1) return run_chain(a, aligned);
    return fail(SPEC_ERR_INVALID, "nothing to compute: no gamma and no chain");
}

spec_status check_common(const void* target, const void* others, spec_dtype dtype, int B, int K, int V, int N,
                         float temperature, void* workspace, size_t workspace_bytes) {
    if (dtype != SPEC_BF16 && dtype != SPEC_FP32) return fail(SPEC_ERR_INVALID, "unknown dtype %d", static_cast<int>(dtype));
    if (B < 0) return fail(SPEC_ERR_INVALID, "B must be >= 0 (got %d)", B);
    if (K < 1 || K > MAX_K) return fail(SPEC_ERR_INVALID, "K must be in [1, %d] (got %d)", MAX_K, K);
    if (V < 1 || V > MAX_V) return fail(SPEC_ERR_INVALID, "V must be in [1, %d] (got %d)", MAX_V, V);
    if (N < 1 || N > MAX_N) return fail(SPEC_ERR_INVALID, "N must be in [1, %d] (got %d)", MAX_N, N);
    if (std::isnan(temperature) || std::isinf(temperature) || temperature < 0.f)
        return fail(SPEC_ERR_INVALID, "temperature must be finite and > 0 (got %g)", static_cast<double>(temperature));
    if (temperature == 0.f) return fail(SPEC_ERR_UNSUPPORTED, "temperature 0 (greedy) is not supported");
    if (B == 0) return SPEC_OK;
    if (!target || !others) return fail(SPEC_ERR_INVALID, "logits pointers must not be NULL");
    if (!workspace) return fail(SPEC_ERR_INVALID, "workspace must not be NULL");
    if (reinterpret_cast<uintptr_t>(workspace) % 16) return fail(SPEC_ERR_INVALID, "workspace must be 16-byte aligned");
    const size_t need = spec_workspace_size(B, K, V, N);
    if (workspace_bytes < need)
        return fail(SPEC_ERR_INVALID, "workspace too small: %zu bytes, need %zu", workspace_bytes, need);
    return SPEC_OK;
}

// Scratch for spec_verify_static: one fixed region per device, part of the library image (static storage,
// so it starts zeroed). Its address is looked up once per device.
constexpr size_t STATIC_SCRATCH_BYTES = size_t(32) << 20;
__device__ __align__(256) unsigned char g_static_scratch[STATIC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
std::mutex g_static_mu;
void* g_static_ptr[MAX_DEVICES] = {};

spec_status static_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "cudaGetDevice failed: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= MAX_DEVICES) return fail(SPEC_ERR_UNSUPPORTED, "device index %d beyond %d", dev, MAX_DEVICES);
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (!g_static_ptr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (e != cudaSuccess || !ptr)
            return fail(SPEC_ERR_CUDA, "looking up the static scratch region failed: %s", cudaGetErrorString(e));
        g_static_ptr[dev] = ptr;
    }
    *out = g_static_ptr[dev];
    return SPEC_OK;
}

}  // namespace
}  // namespace specv

using namespace specv;

extern "C" {

size_t spec_workspace_size(int B, int K, int V, int N) {
    if (B < 0 || K < 0 || V < 1 || N < 1) return 0;
    return ws_layout(B, K, V, N).total;
}

spec_status spec_verify(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                        const int32_t* draft_tokens, const uint64_t* seeds, int B, int K, int V,
                        float temperature, int32_t* accept_len, int32_t* out_tokens, float* diag,
                        void* workspace, size_t workspace_bytes, void* stream) {
    spec_status s = check_common(target_logits, draft_logits, dtype, B, K, V, 1, temperature, workspace, workspace_bytes);
    if (s != SPEC_OK || B == 0) return s;
    if (!draft_tokens || !seeds || !accept_len || !out_tokens)
        return fail(SPEC_ERR_INVALID, "draft_tokens, seeds, accept_len and out_tokens must not be NULL");
    Call a = {};
    a.target = target_logits;
    a.others = draft_logits;
    a.dtype = dtype;
    a.tokens = draft_tokens;
    a.seeds = seeds;
    a.B = B;
    a.K = K;
    a.V = V;
    a.N = 1;
    a.selected = 0;
    a.temperature = temperature;
    a.accept_len = accept_len;
    a.out_tokens = out_tokens;
    a.diag = diag;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.stream = static_cast<cudaStream_t>(stream);
    return run(a);
}

spec_status spec_counterfactual_gamma(const void* target_logits, const void* drafter_logits, spec_dtype dtype,
                                      int N, int B, int K, int V, float temperature, float* gamma, float* loss,
                                      int selected, const int32_t* draft_tokens, const uint64_t* seeds,
                                      int32_t* accept_len, int32_t* out_tokens, float* diag, void* workspace,
                                      size_t workspace_bytes, void* stream) {
    spec_status s = check_common(target_logits, drafter_logits, dtype, B, K, V, N, temperature, workspace, workspace_bytes);
    if (s != SPEC_OK || B == 0) return s;
    if (!gamma) return fail(SPEC_ERR_INVALID, "gamma must not be NULL");
    if (selected < -1 || selected >= N) return fail(SPEC_ERR_INVALID, "selected must be -1 or in [0, N) (got %d)", selected);
    if (selected >= 0 && (!draft_tokens || !seeds || !accept_len || !out_tokens))
        return fail(SPEC_ERR_INVALID, "with selected >= 0, draft_tokens, seeds, accept_len and out_tokens must not be NULL");
    Call a = {};
    a.target = target_logits;
    a.others = drafter_logits;
    a.dtype = dtype;
    a.tokens = draft_tokens;
    a.seeds = seeds;
    a.B = B;
    a.K = K;
    a.V = V;
    a.N = N;
    a.selected = selected;
    a.temperature = temperature;
    a.gamma = gamma;
    a.loss = loss;
    a.accept_len = accept_len;
    a.out_tokens = out_tokens;
    a.diag = diag;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.stream = static_cast<cudaStream_t>(stream);
    return run(a);
}

static spec_status cactus_call(int mode, const void* target_logits, const void* draft_logits, spec_dtype dtype,
                               const int32_t* draft_tokens, const uint64_t* seeds, int B, int K, int V,
                               float temperature, float delta, int32_t* accept_len, int32_t* out_tokens, float* diag,
                               float* gamma_star, void* workspace, size_t workspace_bytes, void* stream) {
    spec_status s = check_common(target_logits, draft_logits, dtype, B, K, V, 1, temperature, workspace, workspace_bytes);
    if (s != SPEC_OK) return s;
    if (std::isnan(delta) || std::isinf(delta) || delta < 0.f)
        return fail(SPEC_ERR_INVALID, "delta must be finite and >= 0 (got %g)", static_cast<double>(delta));
    if (B == 0) return SPEC_OK;
    if (!draft_tokens || !seeds || !accept_len || !out_tokens)
        return fail(SPEC_ERR_INVALID, "draft_tokens, seeds, accept_len and out_tokens must not be NULL");
    Call a = {};
    a.target = target_logits;
    a.others = draft_logits;
    a.dtype = dtype;
    a.tokens = draft_tokens;
    a.seeds = seeds;
    a.B = B;
    a.K = K;
    a.V = V;
    a.N = 1;
    a.selected = 0;
    a.temperature = temperature;
    a.delta = delta;
    a.cactus = mode;
    a.accept_len = accept_len;
    a.out_tokens = out_tokens;
    a.diag = diag;
    a.gamma_star = gamma_star;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.stream = static_cast<cudaStream_t>(stream);
    return run(a);
}

spec_status spec_cactus_verify(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                               const int32_t* draft_tokens, const uint64_t* seeds, int B, int K, int V,
                               float temperature, float delta, int32_t* accept_len, int32_t* out_tokens, float* diag,
                               float* gamma_star, void* workspace, size_t workspace_bytes, void* stream) {
    return cactus_call(1, target_logits, draft_logits, dtype, draft_tokens, seeds, B, K, V, temperature, delta,
                       accept_len, out_tokens, diag, gamma_star, workspace, workspace_bytes, stream);
}

spec_status spec_cactus_kl_verify(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                                  const int32_t* draft_tokens, const uint64_t* seeds, int B, int K, int V,
                                  float temperature, float delta, int32_t* accept_len, int32_t* out_tokens,
                                  float* diag, float* gamma_star, void* workspace, size_t workspace_bytes,
                                  void* stream) {
    return cactus_call(2, target_logits, draft_logits, dtype, draft_tokens, seeds, B, K, V, temperature, delta,
                       accept_len, out_tokens, diag, gamma_star, workspace, workspace_bytes, stream);
}

spec_status spec_greedy_verify(const void* target_logits, spec_dtype dtype, const int32_t* draft_tokens, int B,
                               int K, int V, int32_t* accept_len, int32_t* out_tokens, void* workspace,
                               size_t workspace_bytes, void* stream) {
    if (dtype != SPEC_BF16 && dtype != SPEC_FP32) return fail(SPEC_ERR_INVALID, "unknown dtype %d", static_cast<int>(dtype));
    if (B < 0) return fail(SPEC_ERR_INVALID, "B must be >= 0 (got %d)", B);
    if (K < 1 || K > MAX_K) return fail(SPEC_ERR_INVALID, "K must be in [1, %d] (got %d)", MAX_K, K);
    if (V < 1 || V > MAX_V) return fail(SPEC_ERR_INVALID, "V must be in [1, %d] (got %d)", MAX_V, V);
    if (B == 0) return SPEC_OK;
    if (!target_logits) return fail(SPEC_ERR_INVALID, "target_logits must not be NULL");
    if (!draft_tokens || !accept_len || !out_tokens)
        return fail(SPEC_ERR_INVALID, "draft_tokens, accept_len and out_tokens must not be NULL");
    if (!workspace) return fail(SPEC_ERR_INVALID, "workspace must not be NULL");
    if (reinterpret_cast<uintptr_t>(workspace) % 16) return fail(SPEC_ERR_INVALID, "workspace must be 16-byte aligned");
    const size_t need = spec_workspace_size(B, K, V, 1);
    if (workspace_bytes < need)
        return fail(SPEC_ERR_INVALID, "workspace too small: %zu bytes, need %zu", workspace_bytes, need);
    return run_greedy(target_logits, dtype, draft_tokens, B, K, V, accept_len, out_tokens, workspace,
                      static_cast<cudaStream_t>(stream));
}

spec_status spec_accept_length_estimate(const float* gamma, int N, int B, int K, float* est, float* loss,
                                        void* stream) {
    if (N < 1 || N > MAX_N) return fail(SPEC_ERR_INVALID, "N must be in [1, %d] (got %d)", MAX_N, N);
    if (B < 0) return fail(SPEC_ERR_INVALID, "B must be >= 0 (got %d)", B);
    if (K < 1 || K > MAX_K) return fail(SPEC_ERR_INVALID, "K must be in [1, %d] (got %d)", MAX_K, K);
    if (B == 0) return SPEC_OK;
    if (!gamma || !est) return fail(SPEC_ERR_INVALID, "gamma and est must not be NULL");
    const long long rows = static_cast<long long>(N) * B;
    accept_length_kernel<<<static_cast<unsigned>((rows + 255) / 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        gamma, rows, K, est, loss);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "accept-length kernel launch failed: %s", cudaGetErrorString(e));
    return SPEC_OK;
}

spec_status spec_normalhedge_update(float* regret, const float* loss, float* weights, int N, void* stream) {
    if (N < 1 || N > MAX_N) return fail(SPEC_ERR_INVALID, "N must be in [1, %d] (got %d)", MAX_N, N);
    if (!regret || !loss || !weights) return fail(SPEC_ERR_INVALID, "regret, loss and weights must not be NULL");
    normalhedge_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(regret, loss, weights, N);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "NormalHedge kernel launch failed: %s", cudaGetErrorString(e));
    return SPEC_OK;
}

size_t spec_hedge_feedback_state_size(int N, int B, int K) {
    if (N < 1 || N > MAX_N || B < 0 || K < 1 || K > MAX_K) return 0;
    return hf_seq_bytes(N, K) * static_cast<size_t>(B);
}

spec_status spec_hedge_feedback_init(void* state, int N, int B, int K, int objective, void* stream) {
    if (N < 1 || N > MAX_N) return fail(SPEC_ERR_INVALID, "N must be in [1, %d] (got %d)", MAX_N, N);
    if (B < 0) return fail(SPEC_ERR_INVALID, "B must be >= 0 (got %d)", B);
    if (K < 1 || K > MAX_K) return fail(SPEC_ERR_INVALID, "K must be in [1, %d] (got %d)", MAX_K, K);
    if (objective != 0 && objective != 1) return fail(SPEC_ERR_INVALID, "objective must be 0 or 1 (got %d)", objective);
    if (B == 0) return SPEC_OK;
    if (!state) return fail(SPEC_ERR_INVALID, "state must not be NULL");
    if (reinterpret_cast<uintptr_t>(state) % 16) return fail(SPEC_ERR_INVALID, "state must be 16-byte aligned");
    HfParams h = {};
    h.state = static_cast<unsigned char*>(state);
    h.N = N;
    h.B = B;
    h.K = K;
    h.objective = objective;
    hedge_feedback_init_kernel<<<static_cast<unsigned>((B + 7) / 8), 256, 0, static_cast<cudaStream_t>(stream)>>>(h);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "hedge feedback init launch failed: %s", cudaGetErrorString(e));
    return SPEC_OK;
}

spec_status spec_hedge_feedback_push(void* state, const float* gamma, const int32_t* accept_len, int N, int B, int K,
                                     float* weights, int32_t* applied, void* stream) {
    if (N < 1 || N > MAX_N) return fail(SPEC_ERR_INVALID, "N must be in [1, %d] (got %d)", MAX_N, N);
    if (B < 0) return fail(SPEC_ERR_INVALID, "B must be >= 0 (got %d)", B);
    if (K < 1 || K > MAX_K) return fail(SPEC_ERR_INVALID, "K must be in [1, %d] (got %d)", MAX_K, K);
    if (B == 0) return SPEC_OK;
    if (!state || !gamma || !accept_len) return fail(SPEC_ERR_INVALID, "state, gamma and accept_len must not be NULL");
    if (reinterpret_cast<uintptr_t>(state) % 16) return fail(SPEC_ERR_INVALID, "state must be 16-byte aligned");
    HfParams h = {};
    h.state = static_cast<unsigned char*>(state);
    h.gamma = gamma;
    h.accept_len = accept_len;
    h.N = N;
    h.B = B;
    h.K = K;
    h.weights = weights;
    h.applied = applied;
    hedge_feedback_push_kernel<<<static_cast<unsigned>((B + 7) / 8), 256, 0, static_cast<cudaStream_t>(stream)>>>(h);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "hedge feedback push launch failed: %s", cudaGetErrorString(e));
    return SPEC_OK;
}

size_t spec_filter_workspace_size(int B, int K, int V, spec_dtype dtype) {
    if (B < 0 || K < 0 || V < 1 || (dtype != SPEC_BF16 && dtype != SPEC_FP32)) return 0;
    return filter_layout(B, K, V).total;
}

spec_status spec_verify_filtered(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                                 const int32_t* draft_tokens, const uint64_t* seeds, int B, int K, int V,
                                 float temperature, int top_k, float top_p, int32_t* accept_len, int32_t* out_tokens,
                                 float* diag, void* workspace, size_t workspace_bytes, void* stream) {
    spec_status s = check_common(target_logits, draft_logits, dtype, B, K, V, 1, temperature, workspace, workspace_bytes);
    if (s != SPEC_OK || B == 0) return s;
    if (top_k < 0) return fail(SPEC_ERR_INVALID, "top_k must be >= 0 (got %d)", top_k);
    if (std::isnan(top_p) || !(top_p > 0.f) || top_p > 1.f)
        return fail(SPEC_ERR_INVALID, "top_p must be in (0, 1] (got %g)", static_cast<double>(top_p));
    if (!draft_tokens || !seeds || !accept_len || !out_tokens)
        return fail(SPEC_ERR_INVALID, "draft_tokens, seeds, accept_len and out_tokens must not be NULL");
    const size_t need = spec_filter_workspace_size(B, K, V, dtype);
    if (workspace_bytes < need)
        return fail(SPEC_ERR_INVALID, "workspace too small for the filtered rows: %zu bytes, need %zu", workspace_bytes, need);
    Call a = {};
    a.target = target_logits;
    a.others = draft_logits;
    a.dtype = dtype;
    a.tokens = draft_tokens;
    a.seeds = seeds;
    a.B = B;
    a.K = K;
    a.V = V;
    a.N = 1;
    a.selected = 0;
    a.temperature = temperature;
    a.accept_len = accept_len;
    a.out_tokens = out_tokens;
    a.diag = diag;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.stream = static_cast<cudaStream_t>(stream);
    return run_filtered(a, top_k, top_p);
}

spec_status spec_verify_static(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                               const int32_t* draft_tokens, const uint64_t* seeds, int B, int K, int V,
                               float temperature, int32_t* accept_len, int32_t* out_tokens, float* diag,
                               uint32_t* status_out, void* stream) {
    // sizes first: an oversized call is refused before any CUDA call
    if (B >= 0 && K >= 1 && K <= MAX_K && V >= 1 && V <= MAX_V) {
        const size_t need = spec_workspace_size(B, K, V, 1);
        if (need > STATIC_SCRATCH_BYTES)
            return fail(SPEC_ERR_UNSUPPORTED,
                        "B=%d K=%d V=%d needs %zu bytes of scratch; the static region holds %zu (use spec_verify with "
                        "a caller workspace)", B, K, V, need, STATIC_SCRATCH_BYTES);
    }
    if (dtype != SPEC_BF16 && dtype != SPEC_FP32) return fail(SPEC_ERR_INVALID, "unknown dtype %d", static_cast<int>(dtype));
    if (B < 0) return fail(SPEC_ERR_INVALID, "B must be >= 0 (got %d)", B);
    if (K < 1 || K > MAX_K) return fail(SPEC_ERR_INVALID, "K must be in [1, %d] (got %d)", MAX_K, K);
    if (V < 1 || V > MAX_V) return fail(SPEC_ERR_INVALID, "V must be in [1, %d] (got %d)", MAX_V, V);
    if (std::isnan(temperature) || std::isinf(temperature) || temperature < 0.f)
        return fail(SPEC_ERR_INVALID, "temperature must be finite and > 0 (got %g)", static_cast<double>(temperature));
    if (temperature == 0.f) return fail(SPEC_ERR_UNSUPPORTED, "temperature 0 (greedy) is not supported");
    if (B == 0) return SPEC_OK;
    if (!target_logits || !draft_logits) return fail(SPEC_ERR_INVALID, "logits pointers must not be NULL");
    spec_status s = SPEC_OK;
    if (!draft_tokens || !seeds || !accept_len || !out_tokens)
        return fail(SPEC_ERR_INVALID, "draft_tokens, seeds, accept_len and out_tokens must not be NULL");
    void* scratch = nullptr;
    s = static_scratch(&scratch);
    if (s != SPEC_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the status word is the only part of the scratch that must start at zero
    cudaError_t e = cudaMemsetAsync(scratch, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "status clear failed: %s", cudaGetErrorString(e));
    Call a = {};
    a.target = target_logits;
    a.others = draft_logits;
    a.dtype = dtype;
    a.tokens = draft_tokens;
    a.seeds = seeds;
    a.B = B;
    a.K = K;
    a.V = V;
    a.N = 1;
    a.selected = 0;
    a.temperature = temperature;
    a.accept_len = accept_len;
    a.out_tokens = out_tokens;
    a.diag = diag;
    a.workspace = scratch;
    a.workspace_bytes = STATIC_SCRATCH_BYTES;
    a.stream = st;
    s = run(a);
    if (s != SPEC_OK || !status_out) return s;
    e = cudaMemcpyAsync(status_out, scratch, sizeof(uint32_t), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "status read failed: %s", cudaGetErrorString(e));
    return SPEC_OK;
}

spec_status spec_read_status(const void* workspace, uint32_t* status_out, void* stream) {
    if (!workspace || !status_out) return fail(SPEC_ERR_INVALID, "workspace and status_out must not be NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(status_out, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "status read failed: %s", cudaGetErrorString(e));
    return SPEC_OK;
}

spec_status spec_clear_status(void* workspace, void* stream) {
    if (!workspace) return fail(SPEC_ERR_INVALID, "workspace must not be NULL");
    cudaError_t e = cudaMemsetAsync(workspace, 0, 4 * sizeof(uint32_t), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "status clear failed: %s", cudaGetErrorString(e));
    return SPEC_OK;
}

const char* spec_last_error(void) { return g_err; }

int spec_debug_last_plan(int* out5) {
    if (!out5) return -1;
    for (int i = 0; i < 5; ++i) out5[i] = g_last_plan[i];
    return 0;
}

int spec_debug_exp2ff(const float* d, const float* l_hi, const float* l_lo, float* out, int n, float temperature,
                      void* stream) {
    if (n < 0 || !(temperature > 0.f) || (n > 0 && (!d || !l_hi || !l_lo || !out))) return -1;
    if (n == 0) return 0;
    ff_exp2_probe_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        d, l_hi, l_lo, out, n, ff_constants(temperature));
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int spec_debug_set_gamma_one_launch(int on) {
    if (on != 0 && on != 1) return -1;
    g_gamma_one_launch = on;
    return 0;
}

int spec_debug_set_draw_tau(float tau) {
    if (!(tau >= 0.f)) return -1;
    g_draw_tau = tau;
    return 0;
}

int spec_debug_set_stats_grid(int ctas) {
    if (ctas < 0 || ctas > S_MAX_CTAS) return -1;
    g_stats_grid_override = ctas;
    return 0;
}

}  // extern "C"
