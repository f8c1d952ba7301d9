// Host side of the C ABI declared in include/specverify.h: argument validation, launch planning
// (cluster size, vocabulary slice, shared-memory slots, persistent grid size) and the launches.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <mutex>

#include "specverify.h"
#include "specverify_chain.cuh"

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
constexpr int MAX_N = 64;
constexpr size_t WS_HEADER = 256;          // status word + padding
constexpr int SMEM_MAX_PER_CTA = 232448;   // opt-in maximum per CTA

int g_cluster_override = 0;   // test / tuning hook (0 = automatic)
int g_stats_grid_override = 0;   // CTAs of the statistics kernel (0 = automatic)
thread_local int g_last_plan[5] = {0, 0, 0, 0, 0};   // C, S, clusters launched, resident, pieces per slice

struct Plan {
    int C = 1, slice_elems = 0, pcap = 0, R = 0, resident = 0, tma = 0, ncl = 0;
    size_t smem = 0;
};

int slice_for(int V, int C) { return ((V + SLICE_Q - 1) / SLICE_Q + C - 1) / C * SLICE_Q; }
int pcap_for(int slice_elems) { return (slice_elems + PE - 1) / PE; }

// barriers, exchange entries, scalars and the abort flag (see the layout note above rows_kernel)
size_t fixed_smem(int R, int C) {
    return static_cast<size_t>(W * R + 4 + 3 * NXB) * 8 + static_cast<size_t>(NXB * W * XW + NXB * C * XW + NXB * XW) * 4 + 16;
}

using KernelFn = void (*)(const KParams);

struct OccKey {
    KernelFn fn;
    int C;
    size_t smem;
    int device;
};
std::mutex g_occ_mu;
OccKey g_occ_keys[64];
int g_occ_vals[64];
int g_occ_n = 0;

// Number of clusters of C CTAs with `smem` bytes each that fit on the GPU at once (cached per device).
cudaError_t max_clusters(KernelFn fn, int C, size_t smem, int& out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lk(g_occ_mu);
        for (int i = 0; i < g_occ_n; ++i)
            if (g_occ_keys[i].fn == fn && g_occ_keys[i].C == C && g_occ_keys[i].smem == smem &&
                g_occ_keys[i].device == dev) {
                out = g_occ_vals[i];
                return cudaSuccess;
            }
    }
    // The attribute is a per-function ceiling shared by every plan: always the opt-in maximum, so that a
    // later plan with less shared memory never lowers it under an earlier, cached one.
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX_PER_CTA);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    cfg.gridDim = dim3(static_cast<unsigned>(C), 1, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = static_cast<unsigned>(C);
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    std::lock_guard<std::mutex> lk(g_occ_mu);
    if (g_occ_n < 64) {
        g_occ_keys[g_occ_n] = {fn, C, smem, dev};
        g_occ_vals[g_occ_n] = n;
        ++g_occ_n;
    }
    out = n;
    return cudaSuccess;
}

// Rows handled by the busiest of ncl clusters: items are dealt round robin, the B*K verified positions
// (1 + N rows each) first and the B bonus rows (1 row each) last.
long long busiest_rows(int BK, int B_bonus, int N, int ncl) {
    long long worst = 0;
    for (int c = 0; c < ncl; ++c) {
        const long long pos = BK / ncl + (c < BK % ncl ? 1 : 0);
        // bonus items are numbers BK .. BK + B_bonus - 1; count those congruent to c mod ncl
        const int first = ((c - BK % ncl) % ncl + ncl) % ncl;   // offset of the first bonus item of c
        const long long bon = B_bonus > first ? (B_bonus - 1 - first) / ncl + 1 : 0;
        worst = std::max(worst, pos * (1 + N) + bon);
    }
    return worst;
}

// Chooses the cluster size C and the ring depth R. Each CTA holds, per consumer warp, R slots of one piece
// and, when items have two or more drafters (resident mode), two copies of its target slice. Among the
// cluster sizes whose shared memory fits, the plan minimises an estimate of the busiest CTA's time:
// (rows of its cluster) x (slice length + a fixed per-row cost of the cluster-wide statistics exchange,
// worth about UNIT_COST_EL logits of streaming), using the number of clusters the GPU places at once.
// In streamed mode a slice is re-read from L2 about two rows after its first read; when (CTAs) x (two rows
// of a slice) exceeds half of L2 the estimate grows with the excess. Ties go to the smaller cluster.
constexpr double UNIT_COST_EL = 40000.0;

spec_status make_plan(KernelFn fn, int V, int eb, int N, int BK, int B_bonus, bool aligned, Plan& out) {
    static const int auto_cands[] = {1, 2, 4, 8, 16};
    const int* cands = auto_cands;
    int ncand = 5;
    int forced[1];
    if (g_cluster_override > 0) {
        forced[0] = g_cluster_override;
        cands = forced;
        ncand = 1;
    }
    const int resident = N >= 2 ? 1 : 0;
    const size_t slot_bytes = static_cast<size_t>(PE) * eb;
    int dev = 0;
    cudaGetDevice(&dev);
    int l2 = 0;
    cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
    bool found = false;
    double best = 0.0;
    for (int ci = 0; ci < ncand; ++ci) {
        Plan p;
        p.C = cands[ci];
        p.slice_elems = slice_for(V, p.C);
        p.pcap = pcap_for(p.slice_elems);
        p.resident = resident;
        p.tma = aligned ? 1 : 0;
        const size_t tb = resident ? (static_cast<size_t>(p.slice_elems) * eb + 127) / 128 * 128 : 0;
        int R = MAX_R;
        while (R >= 1 && 2 * tb + W * R * slot_bytes + fixed_smem(R, p.C) > static_cast<size_t>(SMEM_MAX_PER_CTA)) --R;
        if (R < 1) continue;
        p.R = R;
        p.smem = 2 * tb + W * R * slot_bytes + fixed_smem(R, p.C);
        int ncl = 0;
        const cudaError_t e = max_clusters(fn, p.C, p.smem, ncl);
        if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "occupancy query failed: %s", cudaGetErrorString(e));
        p.ncl = ncl;
        double cost = static_cast<double>(busiest_rows(BK, B_bonus, N, ncl)) * (p.slice_elems + UNIT_COST_EL);
        const double footprint = static_cast<double>(ncl) * p.C * 2.0 * p.slice_elems * eb;
        if (!resident && l2 > 0 && footprint > l2 / 2.0) cost *= 1.0 + (footprint - l2 / 2.0) / l2;
        if (!found || cost < best * 0.999) {
            best = cost;
            out = p;
            found = true;
        }
    }
    if (!found) return fail(SPEC_ERR_UNSUPPORTED, "no launch plan fits V=%d (cluster override %d)", V, g_cluster_override);
    return SPEC_OK;
}

// Workspace layout: [status header][records B*(K+1)*REC][piece masses B*(K+1)*pieces_row][gamma partials
// N*B*K*16*W][segment partials of the statistics pass]. The per-row regions are sized for the largest
// cluster split so that any plan fits; the segment region for the largest statistics grid.
struct WsLayout {
    size_t rec_off, tiles_off, gpart_off, part_off, total;
    int tiles_row;   // floats per row in the piece-mass region (>= C * pcap for every plan)
    int gpart_row;   // floats per (drafter, b, j) in the gamma region (>= C * W)
};

WsLayout ws_layout(int B, int K, int V, int N) {
    WsLayout w;
    int tiles_row = 0;
    for (int C = 1; C <= 16; ++C) tiles_row = std::max(tiles_row, C * pcap_for(slice_for(V, C)));
    w.tiles_row = tiles_row;
    w.gpart_row = 16 * W;
    const size_t rows = static_cast<size_t>(B) * static_cast<size_t>(K + 1);
    w.rec_off = WS_HEADER;
    w.tiles_off = w.rec_off + rows * REC * sizeof(float);
    w.gpart_off = w.tiles_off + rows * static_cast<size_t>(tiles_row) * sizeof(float);
    w.part_off = w.gpart_off + static_cast<size_t>(N) * B * K * static_cast<size_t>(w.gpart_row) * sizeof(float);
    w.part_off = (w.part_off + 15) / 16 * 16;   // float2 entries
    // segment (warp g, row r) of the statistics pass at entry g + r: fewer than min(G, pieces) + rows entries
    const long long srows = static_cast<long long>(B) * (2 * K + 1);
    const long long pieces = srows * ((V + PE - 1) / PE);
    const long long gmax = static_cast<long long>(S_MAX_CTAS) * SW;
    w.total = w.part_off + static_cast<size_t>(std::min(pieces, gmax) + srows) * sizeof(float2);
    w.total = (w.total + 15) / 16 * 16;
    return w;
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

// Raises the dynamic shared-memory ceiling of a draw kernel once per device (its chunk masses need up to
// 128 KB).
std::mutex g_dsm_mu;
struct DsmEntry {
    const void* fn;
    int device;
};
DsmEntry g_dsm[32];
int g_dsm_n = 0;

template <class Fn>
cudaError_t draw_smem_ceiling(Fn fn, int dev) {
    std::lock_guard<std::mutex> lk(g_dsm_mu);
    for (int i = 0; i < g_dsm_n; ++i)
        if (g_dsm[i].fn == reinterpret_cast<const void*>(fn) && g_dsm[i].device == dev) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX_PER_CTA - 8192);
    if (e == cudaSuccess && g_dsm_n < 32) g_dsm[g_dsm_n++] = {reinterpret_cast<const void*>(fn), dev};
    return e;
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

    DParams d = {};
    d.target = s.rows_a;
    d.draft = s.rows_b;
    d.part = s.part;
    d.P = s.P;
    d.G = s.G;
    d.np = s.np;
    d.rows_a_n = s.rows_a_n;
    d.tokens = a.tokens;
    d.seeds = a.seeds;
    d.B = a.B;
    d.K = a.K;
    d.V = a.V;
    d.c = s.c;
    d.delta = a.delta;
    d.cactus = a.cactus;
    d.accept_len = a.accept_len;
    d.out_tokens = a.out_tokens;
    d.diag = a.diag;
    d.gamma_star = a.gamma_star;
    d.status = s.status;
    // CTAs per sequence: the largest power of two up to D_MAX_CPS that keeps the grid within one CTA per SM
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int cps = 1;
    while (cps < D_MAX_CPS && static_cast<long long>(a.B) * cps * 2 <= sms) cps *= 2;
    d.cps = cps;
    // chunk masses, plus (bulk-copy mode) a two-piece slot and an mbarrier per warp when they fit
    const size_t cm_bytes = static_cast<size_t>((s.np + cps - 1) / cps) * D_CPP * sizeof(float);
    const size_t ring_bytes = static_cast<size_t>(DW) * (2 * static_cast<size_t>(PE) * eb + sizeof(uint64_t));
    const size_t dsmem_cap = SMEM_MAX_PER_CTA - 8192;   // the ceiling draw_smem_ceiling sets
    d.tma = aligned && cm_bytes + ring_bytes <= dsmem_cap ? 1 : 0;
    const size_t dsmem = cm_bytes + (d.tma ? ring_bytes : 0);
    using DrawFn = void (*)(const DParams);
    DrawFn dfn = a.dtype == SPEC_BF16 ? (aligned ? draw_kernel<Bf16, true> : draw_kernel<Bf16, false>)
                                      : (aligned ? draw_kernel<F32, true> : draw_kernel<F32, false>);
    e = draw_smem_ceiling(dfn, dev);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "draw kernel attribute failed: %s", cudaGetErrorString(e));
    // launched with programmatic stream serialisation: its CTAs start as the grid above frees SMs and wait
    // for it (griddepcontrol.wait) after reading their inputs
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

spec_status run(const Call& a) {
    if (a.B == 0) return SPEC_OK;
    const int eb = a.dtype == SPEC_BF16 ? 2 : 4;
    const bool chain = a.selected >= 0;
    const uintptr_t align_mask = 15;
    // bulk copies need 16-byte aligned pieces of whole 8-logit chunks
    const bool aligned = ((reinterpret_cast<uintptr_t>(a.target) | reinterpret_cast<uintptr_t>(a.others)) & align_mask) == 0 &&
                         (static_cast<size_t>(a.V) * eb) % 16 == 0 && a.V % CHUNK == 0;
    if (chain && a.N == 1 && !a.gamma) return run_chain(a, aligned);
    KernelFn fn = a.dtype == SPEC_BF16 ? rows_kernel<Bf16> : rows_kernel<F32>;
    const int BK = a.B * a.K;
    const int B_bonus = chain ? a.B : 0;
    Plan pl;
    spec_status st = make_plan(fn, a.V, eb, a.N, BK, B_bonus, aligned, pl);
    if (st != SPEC_OK) return st;

    const WsLayout wl = ws_layout(a.B, a.K, a.V, a.N);
    unsigned char* ws = static_cast<unsigned char*>(a.workspace);
    KParams k = {};
    k.target = static_cast<const unsigned char*>(a.target);
    k.others = static_cast<const unsigned char*>(a.others);
    k.tokens = chain ? a.tokens : nullptr;
    k.seeds = chain ? a.seeds : nullptr;
    k.all_residuals = a.diag ? 1 : 0;
    k.B = a.B;
    k.K = a.K;
    k.V = a.V;
    k.N = a.N;
    k.selected = a.selected;
    k.BK = BK;
    k.num_items = BK + B_bonus;
    k.c = static_cast<float>(1.4426950408889634 / static_cast<double>(a.temperature));
    k.delta = a.delta;
    k.cactus = a.cactus;
    k.slice_elems = pl.slice_elems;
    // the kernels index the piece-mass region as (row * C + rank) * pcap + piece: rows are C * pcap <=
    // wl.tiles_row floats apart, so the region sized with wl.tiles_row holds every plan
    k.pcap = pl.pcap;
    k.tma = pl.tma;
    k.resident = pl.resident;
    k.R = pl.R;
    k.lead = 1;
    k.status = reinterpret_cast<unsigned*>(ws);
    k.rec = chain ? reinterpret_cast<float*>(ws + wl.rec_off) : nullptr;
    k.tiles = chain ? reinterpret_cast<float*>(ws + wl.tiles_off) : nullptr;
    k.gpart = a.gamma ? reinterpret_cast<float*>(ws + wl.gpart_off) : nullptr;

    const int grid_clusters = pl.ncl < k.num_items ? pl.ncl : k.num_items;
    g_last_plan[0] = pl.C;
    g_last_plan[1] = pl.R;
    g_last_plan[2] = grid_clusters;
    g_last_plan[3] = pl.resident;
    g_last_plan[4] = pl.pcap;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    cfg.gridDim = dim3(static_cast<unsigned>(grid_clusters * pl.C), 1, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = a.stream;
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = static_cast<unsigned>(pl.C);
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, fn, k);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "verification kernel launch failed: %s", cudaGetErrorString(e));

    // follow-up kernels: launched with programmatic stream serialisation, they wait on the grid above
    // (griddepcontrol.wait) while their launch overlaps its tail
    cudaLaunchAttribute pa[1];
    pa[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pa[0].val.programmaticStreamSerializationAllowed = 1;
    const int per_block = 8;   // warps per block
    if (a.gamma) {
        GParams g = {};
        g.gpart = k.gpart;
        g.n_out = a.N * a.B * a.K;
        g.C = pl.C;
        g.gamma = a.gamma;
        g.loss = a.loss;
        cudaLaunchConfig_t gc = {};
        gc.gridDim = dim3(static_cast<unsigned>((g.n_out + per_block - 1) / per_block), 1, 1);
        gc.blockDim = dim3(per_block * 32, 1, 1);
        gc.stream = a.stream;
        gc.attrs = pa;
        gc.numAttrs = 1;
        e = cudaLaunchKernelEx(&gc, gamma_reduce_kernel, g);
        if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "gamma reduction launch failed: %s", cudaGetErrorString(e));
    }
    if (chain) {
        FParams f = {};
        f.rec = k.rec;
        f.tiles = k.tiles;
        f.target = k.target;
        f.other = k.others + static_cast<size_t>(a.selected) * a.B * a.K * static_cast<size_t>(a.V) * eb;
        f.tokens = a.tokens;
        f.seeds = a.seeds;
        f.B = a.B;
        f.K = a.K;
        f.V = a.V;
        f.C = pl.C;
        f.slice_elems = pl.slice_elems;
        f.pcap = pl.pcap;
        f.c = k.c;
        f.accept_len = a.accept_len;
        f.out_tokens = a.out_tokens;
        f.diag = a.diag;
        f.gamma_star = a.gamma_star;
        cudaLaunchConfig_t fc = {};
        fc.gridDim = dim3(static_cast<unsigned>((a.B + per_block - 1) / per_block), 1, 1);
        fc.blockDim = dim3(per_block * 32, 1, 1);
        fc.stream = a.stream;
        fc.attrs = pa;
        fc.numAttrs = 1;
        if (a.dtype == SPEC_BF16)
            e = aligned ? cudaLaunchKernelEx(&fc, finish_kernel<Bf16, true>, f) : cudaLaunchKernelEx(&fc, finish_kernel<Bf16, false>, f);
        else
            e = aligned ? cudaLaunchKernelEx(&fc, finish_kernel<F32, true>, f) : cudaLaunchKernelEx(&fc, finish_kernel<F32, false>, f);
        if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "chain kernel launch failed: %s", cudaGetErrorString(e));
    }
    return SPEC_OK;
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

spec_status spec_cactus_verify(const void* target_logits, const void* draft_logits, spec_dtype dtype,
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
    a.cactus = 1;
    a.accept_len = accept_len;
    a.out_tokens = out_tokens;
    a.diag = diag;
    a.gamma_star = gamma_star;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.stream = static_cast<cudaStream_t>(stream);
    return run(a);
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
    cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(uint32_t), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "status clear failed: %s", cudaGetErrorString(e));
    return SPEC_OK;
}

const char* spec_last_error(void) { return g_err; }

int spec_debug_last_plan(int* out5) {
    if (!out5) return -1;
    for (int i = 0; i < 5; ++i) out5[i] = g_last_plan[i];
    return 0;
}

int spec_debug_set_cluster_size(int C) {
    if (C < 0 || C > 16) return -1;
    g_cluster_override = C;
    return 0;
}

int spec_debug_set_stats_grid(int ctas) {
    if (ctas < 0 || ctas > S_MAX_CTAS) return -1;
    g_stats_grid_override = ctas;
    return 0;
}

}  // extern "C"
