// C ABI of the library (declared in include/rmsnorm_gb300.h): argument
// checks, engine selection, and the launch sequence of each call on the
// caller's stream and current device.
//
// Backward launch sequences (the pages count the fp32 zero and the cast to
// the parameter dtype inside the call -- FlyDSL PR #854 "Benchmark
// contract"):
//   scratch mode: row pass (partials -> workspace) -> finalize (sum + cast)
//   atomic mode:  zero dweight_f32 -> row pass (fp32 atomics) -> [cast]
// Kernels after the first are launched as programmatic dependents, so their
// launch overlaps the tail of the kernel they wait for.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <string>
#include <unordered_map>

#include "../../include/rmsnorm_gb300.h"
#include "common.cuh"
#include "launch.h"

namespace rn {

static thread_local char g_err[512] = "";
static thread_local char g_plan[256] = "";
static int g_opts[RN_OPT_COUNT] = {0};
static cudaEvent_t g_ev_begin = nullptr, g_ev_end = nullptr;

static rn_status fail(rn_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return st;
}

void set_last_error(const char *msg) { snprintf(g_err, sizeof(g_err), "%s", msg); }

static rn_status cuda_fail(cudaError_t e, const char *what) {
    return fail(RN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

struct DeviceInfo {
    int num_sms = 0;
    size_t smem_optin = 0;
};

static std::mutex g_mu;
static std::unordered_map<int, DeviceInfo> g_devs;
static std::unordered_map<long long, size_t> g_smem_set;  // (device, func) -> bytes set

static cudaError_t device_info(DeviceInfo *out, int *dev_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev_out) *dev_out = dev;
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_devs.find(dev);
    if (it != g_devs.end()) {
        *out = it->second;
        return cudaSuccess;
    }
    DeviceInfo d;
    int v = 0;
    e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    d.num_sms = v;
    e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    d.smem_optin = (size_t)v;
    g_devs[dev] = d;
    *out = d;
    return cudaSuccess;
}

cudaError_t ensure_smem_attr(const void *func, size_t bytes) {
    if (bytes == 0) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const long long key = ((long long)dev << 48) ^ (long long)(uintptr_t)func;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_smem_set.find(key);
        if (it != g_smem_set.end() && it->second >= bytes) return cudaSuccess;
    }
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, func);
    if (e != cudaSuccess) return e;
    // Without the opt-in a launch may use 48 KB of shared memory, the kernel's static shared
    // memory and the dynamic bytes together.
    const size_t base_cap = 48 * 1024 > fa.sharedSizeBytes ? 48 * 1024 - fa.sharedSizeBytes : 0;
    if (bytes <= base_cap) {
        std::lock_guard<std::mutex> lk(g_mu);
        size_t &known = g_smem_set[key];
        if (known < base_cap) known = base_cap;
        return cudaSuccess;
    }
    // Set the kernel's cap to the most dynamic shared memory it can have:
    // the device's opt-in limit minus the kernel's own static shared memory.
    DeviceInfo d;
    e = device_info(&d, nullptr);
    if (e != cudaSuccess) return e;
    const size_t cap = d.smem_optin - fa.sharedSizeBytes;
    if (bytes > cap) return cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cap);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_mu);
    g_smem_set[key] = cap;
    return cudaSuccess;
}

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Workspace partial rows the backward may use on a device.
static int max_partial_rows(const DeviceInfo &d) { return 2 * d.num_sms; }

static size_t ws_bytes_for(const DeviceInfo &d, int64_t N) {
    return kWsHeaderBytes + (size_t)max_partial_rows(d) * (size_t)N * 4;
}

// ------------------------------------------------------------- planning
// Tile of the persistent row engine for rows of `nchunks` 16-byte chunks and
// `nt` streamed tensors; `red_bytes` of shared memory precede the ring and
// `max_cpt` caps the default chunks per thread.
// Extra tile rules of the RMSNorm backward (measured there only).
struct RowTuning {
    size_t ring_cap_3;    // ring cap while at least 3 teams remain
    size_t ring_cap_5;    // ring cap while at least 5 teams remain
    int min_rows_per_team;  // on problems of at least 16 rows per SM
};

static bool plan_row_tile(int64_t M, int nchunks, int nt, size_t red_bytes, int max_cpt,
                          int (*max_threads)(int cpt), const DeviceInfo &d, RowPlan *plan,
                          bool use_options = true, const RowTuning *tune = nullptr) {
    if (nchunks > kRowMaxChunks) return false;
    // RN_OPT_* shape the backward only
    auto opt = [&](int o) { return use_options ? g_opts[o] : 0; };

    // Tile (measured on GB300): 4 chunks per thread for rows of 512+ chunks
    // (bf16 N >= 4096), else 2, else 1 for very short rows.
    int cpt = opt(RN_OPT_CHUNKS_PER_THREAD);
    const bool cpt_forced = cpt == 1 || cpt == 2 || cpt == 4;
    if (!cpt_forced) {
        cpt = nchunks >= 512 ? 4 : (nchunks >= 64 ? 2 : 1);
        while (cpt > max_cpt) cpt /= 2;
        // more chunks per thread when the row does not fit the capped tile
        while (cpt < 4 && ((nchunks + cpt - 1) / cpt + 31) / 32 * 32 > max_threads(cpt)) cpt *= 2;
    }
    auto team_of = [&](int c) { return ((nchunks + c - 1) / c + 31) / 32 * 32; };
    int team = team_of(cpt);
    if (team > max_threads(cpt)) return false;

    const size_t budget = (d.smem_optin < 200 * 1024 ? d.smem_optin : 200 * 1024);
    auto smem_for = [&](int teams_, int stages_) {
        return red_bytes + (size_t)teams_ * stages_ * nt * (size_t)(cpt * team) * 16;
    };
    int teams = opt(RN_OPT_TEAMS_PER_CTA);
    if (teams <= 0) {
        teams = max_threads(cpt) / team;
        if (teams > 15) teams = 15;
        // room for at least 2 slots per team
        while (teams > 1 && smem_for(teams, 2) > budget) --teams;
        if (tune) {
            // softer caps on the ring while enough teams remain
            while (teams > 4 && smem_for(teams, 2) > tune->ring_cap_5) --teams;
            while (teams > 3 && smem_for(teams, 2) > tune->ring_cap_3) --teams;
        }
        // no more teams than rows per SM
        int64_t rows_per_sm = (M + d.num_sms - 1) / d.num_sms;
        if (rows_per_sm < 1) rows_per_sm = 1;
        if (teams > rows_per_sm) teams = (int)rows_per_sm;
        // with enough rows, each team gets a few: fewer teams, and then fewer chunks per
        // thread (more threads on a row) while the CTA still fits
        if (tune && rows_per_sm >= 16 && teams > rows_per_sm / tune->min_rows_per_team) {
            teams = (int)(rows_per_sm / tune->min_rows_per_team);
            while (!cpt_forced && cpt > 1 && team_of(cpt / 2) * teams <= max_threads(cpt / 2)) {
                cpt /= 2;
                team = team_of(cpt);
            }
        }
    }
    const int tc = cpt * team;  // 16-byte chunks per tensor row in a team's slot
    const size_t stage = (size_t)nt * tc * 16;
    if (teams < 1 || teams > 15 || teams * team > max_threads(cpt)) return false;

    // one CTA per SM unless the grid option asks for another count
    int64_t cap = opt(RN_OPT_GRID) > 0 ? opt(RN_OPT_GRID) : d.num_sms;
    if (cap > max_partial_rows(d)) cap = max_partial_rows(d);
    int64_t grid = (M + teams - 1) / teams;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;

    // A shallow ring (one row in flight per thread) measured best: the
    // first rows arrive sooner and more teams fit; a team that is alone on
    // its SM gets one row more. The same holds for the forwards (bf16
    // RMSNorm forward, 2 slots vs ~64 KB in flight per CTA: 15.9 vs 16.2 us
    // at 4096^2, 83.8 vs 86.9 us at 16384 x 8192).
    int stages = opt(RN_OPT_STAGES);
    if (stages <= 0) {
        stages = (int)((budget - red_bytes) / (stage * teams));
        const int want = teams >= 2 ? 2 : 3;
        if (stages > want) stages = want;
        const int64_t rows_per_team = (M + grid * teams - 1) / (grid * teams);
        if (stages > rows_per_team) stages = (int)(rows_per_team < 1 ? 1 : rows_per_team);
    }
    if (stages < 1 || stages > 8) return false;
    const size_t smem = smem_for(teams, stages);
    if (smem > d.smem_optin) return false;

    plan->cpt = cpt;
    plan->team_threads = team;
    plan->teams = teams;
    plan->stages = stages;
    plan->grid = (int)grid;
    plan->smem = smem;
    plan->atomic = false;
    return true;
}

static bool plan_row(const BwdProblem &p, const DeviceInfo &d, RowPlan *plan) {
    const int row_bytes = p.N * elem_bytes(p.dtype);
    if (row_bytes % 16) return false;
    if (!aligned16(p.x) || !aligned16(p.dy) || !aligned16(p.gamma) || !aligned16(p.dx) ||
        (p.dres && !aligned16(p.dres)))
        return false;
    const int nt = p.dres ? 3 : 2;
    // Measured on GB300 (L2 flushed, us per call):
    //  * a ring above ~150 KB costs more than a fourth team gains (bf16 fused-add with
    //    dresidual_out, 4096-wide rows; 3 teams and 147 KB vs 4 and 196 KB): 25.5 vs 26.1 at
    //    M = 4096, 40.0 vs 42.9 at 8192, 79.5 vs 83.2 at 16384, 18.9 vs 19.3 at 2048. With
    //    fewer teams left the larger ring stays (16384 x 8192: 2 teams 159.5, 1 team 173.3);
    //  * with five or more teams, above ~125 KB (fused with dres; 5 teams and 123 KB vs 6 and
    //    147 KB): bf16 4096 x 2048 18.8 vs 21.4, 16384 x 2048 39.9 vs 41.0, f32 16384 x 1024
    //    39.3 vs 40.6;
    //  * at least 4 rows a team once there are 16 rows per SM, with the spare threads put on
    //    each row: bf16 4096 x 1024 (1 chunk x 128 threads, 6 teams vs 2 x 64, 12 teams) 13.3
    //    vs 15.2, fused 14.4 vs 16.3.
    static const RowTuning kTune = {160 * 1024, 125 * 1024, 4};
    // the kernel's reduction slots precede its ring: row_smem_bytes with no ring
    return plan_row_tile(p.M, row_bytes / 16, nt, row_smem_bytes(0, 0, nt, 0), 4,
                         row_max_threads, d, plan, true, &kTune);
}

// Cluster engine: the row split over `csize` CTAs of up to 2048 chunks each.
// Cluster occupancy answers are cached per launch shape.
static std::unordered_map<std::string, int> g_cluster_occ;

// Cluster size, slice, tile and ring depth for rows of `nchunks` chunks and
// `nt` streamed tensors (the occupancy-dependent cluster count is left out).
static bool cluster_tile(int nchunks, int nt, bool forced, const DeviceInfo &d,
                         size_t (*smem_bytes)(int stages, int nt, int cpt, int threads),
                         ClusterPlan *plan) {
    if (nchunks <= kRowMaxChunks && !forced) return false;  // the row engine's range
    int csize = g_opts[RN_OPT_CLUSTER_SIZE];
    if (csize == 0) {
        csize = 2;
        while (csize < 16 && (nchunks + csize - 1) / csize > kRowMaxChunks) csize *= 2;
    }
    if (csize != 2 && csize != 4 && csize != 8 && csize != 16) return false;
    const int slice = (nchunks + csize - 1) / csize;
    if (slice > kRowMaxChunks) return false;
    int cpt = g_opts[RN_OPT_CHUNKS_PER_THREAD];
    if (cpt != 1 && cpt != 2 && cpt != 4) cpt = slice > 1024 ? 4 : (slice > 512 ? 2 : 1);
    const int threads = ((slice + cpt - 1) / cpt + 31) / 32 * 32;
    if (threads > 512) return false;
    const size_t budget = d.smem_optin < 200 * 1024 ? d.smem_optin : 200 * 1024;
    int stages = g_opts[RN_OPT_STAGES];
    if (stages <= 0) {
        stages = 4;
        while (stages > 2 && smem_bytes(stages, nt, cpt, threads) > budget) --stages;
    }
    if (stages < 1 || stages > 8) return false;
    const size_t smem = smem_bytes(stages, nt, cpt, threads);
    if (smem > d.smem_optin) return false;
    plan->csize = csize;
    plan->slice = slice;
    plan->cpt = cpt;
    plan->threads = threads;
    plan->stages = stages;
    plan->smem = smem;
    return true;
}

// The persistent cluster count: what fits at once (queried once per launch
// shape and cached), at most one cluster per row and the workspace's rows.
static bool cluster_count(const char *kind, int64_t M, int dtype, bool dres, const DeviceInfo &d,
                          ClusterPlan *plan, cudaError_t (*query)(const void *ctx,
                                                                 const ClusterPlan &, int *),
                          const void *ctx) {
    char key[128];
    snprintf(key, sizeof(key), "%s/%d/%d/%d/%d/%d/%d/%zu/%d", kind, d.num_sms, dtype, plan->cpt,
             (int)dres, (int)plan->atomic, plan->csize, plan->smem, plan->threads);
    int occ = 0;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_cluster_occ.find(key);
        if (it != g_cluster_occ.end()) occ = it->second;
    }
    if (occ == 0) {
        if (query(ctx, *plan, &occ) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        std::lock_guard<std::mutex> lk(g_mu);
        g_cluster_occ[key] = occ;
    }
    int64_t clusters = occ;
    if (clusters > M) clusters = M;
    if (clusters > max_partial_rows(d)) clusters = max_partial_rows(d);
    if (g_opts[RN_OPT_GRID] > 0 && clusters * plan->csize > g_opts[RN_OPT_GRID])
        clusters = g_opts[RN_OPT_GRID] / plan->csize;
    if (clusters < 1) return false;
    plan->clusters = (int)clusters;
    return true;
}

static size_t rms_cluster_smem(int stages, int nt, int cpt, int threads) {
    return cluster_smem_bytes(stages, nt, cpt, threads);
}

static cudaError_t rms_cluster_query(const void *ctx, const ClusterPlan &plan, int *n) {
    return cluster_max_active(*static_cast<const BwdProblem *>(ctx), plan, n);
}

static bool plan_cluster(const BwdProblem &p, const DeviceInfo &d, bool atomic, bool forced,
                         ClusterPlan *plan) {
    const int row_bytes = p.N * elem_bytes(p.dtype);
    if (row_bytes % 16) return false;
    if (!aligned16(p.x) || !aligned16(p.dy) || !aligned16(p.gamma) || !aligned16(p.dx) ||
        (p.dres && !aligned16(p.dres)))
        return false;
    if (!cluster_tile(row_bytes / 16, p.dres ? 3 : 2, forced, d, rms_cluster_smem, plan))
        return false;
    plan->atomic = atomic;
    return cluster_count("rms", p.M, p.dtype, p.dres != nullptr, d, plan, rms_cluster_query, &p);
}

// The generic engine's vector variant needs every row tensor at the same
// alignment phase (base addresses equal modulo 16, element-aligned) and the
// weight-gradient partial in shared memory.
static bool generic_vec_ok(const BwdProblem &p, const DeviceInfo &d) {
    const uintptr_t S = (uintptr_t)elem_bytes(p.dtype);
    const uintptr_t ph = (uintptr_t)p.x & 15u;
    for (const void *q : {p.x, p.dy, static_cast<const void *>(p.dx), p.dres}) {
        if (q == nullptr) continue;
        if (((uintptr_t)q & 15u) != ph || ((uintptr_t)q % S) != 0) return false;
    }
    const size_t budget = d.smem_optin < 200 * 1024 ? d.smem_optin : 200 * 1024;
    return generic_vec_smem_bytes(p.N) <= budget;
}

// The realigning engine: the vector variant's conditions, and a row of 1024
// to 4 x 512 column blocks of 16 bytes (16 KB to 32 KB: bf16 N 8,185 to
// 16,384) whose buffers fit the shared-memory budget. Measured on GB300 (L2
// flushed, us per call, vector variant -> realigning engine): bf16 16384 x
// 8190 292 -> 233 (fused 321 -> 275), f32 4096 x 4095 68 -> 58 (fused
// 77 -> 67); below 1024 blocks the vector variant was faster (bf16 4096 x
// 4100 48 vs 56, 4096 x 4095 51 vs 53). Taken only when asked for
// (RN_OPT_GENERIC_KERNEL = 3): the phase-class kernel with four chunks a thread
// is faster at every width of its range (kernel us, realigning -> phase-class:
// bf16 4096 x 12290 126.7 -> 87.1, fused 182.1 -> 132.8, 16384 x 12290
// 424.4 -> 331.3, 16384 x 8201 365.4 -> 287.7, 4096 x 16383 138.4 -> 104.1,
// f16 8192 x 10001 207.8 -> 157.2, f32 4096 x 6001 77.8 -> 66.3).
static bool plan_realign(const BwdProblem &p, const DeviceInfo &d, GenericPlan *plan) {
    if (!generic_vec_ok(p, d)) return false;
    const int nb = (int)(((int64_t)p.N * elem_bytes(p.dtype) + 15) / 16);
    if (nb < 1024) return false;
    int cpb = 2;
    while (cpb < 4 && (nb + cpb - 1) / cpb > 512) cpb *= 2;
    if ((nb + cpb - 1) / cpb > 512) return false;
    const int rows = 1;  // rows per CTA iteration (the kernel's R)
    const size_t budget = d.smem_optin < 200 * 1024 ? d.smem_optin : 200 * 1024;
    const size_t smem = realign_smem_bytes(p.N, p.dtype, rows, p.dres != nullptr);
    if (smem > budget) return false;
    plan->cpb = cpb;
    plan->rows = rows;
    plan->threads = ((nb + cpb - 1) / cpb + 31) / 32 * 32;
    plan->smem_dw = false;
    plan->smem = smem;
    // two CTAs per SM when a CTA has at most 256 threads, else one
    int64_t grid = (p.M + rows - 1) / rows;
    const int64_t cap = plan->threads <= 256 ? max_partial_rows(d) : d.num_sms;
    if (grid > cap) grid = cap;
    if (g_opts[RN_OPT_GRID] > 0 && grid > g_opts[RN_OPT_GRID]) grid = g_opts[RN_OPT_GRID];
    if (grid < 1) grid = 1;
    plan->grid = (int)grid;
    plan->atomic = false;
    return true;
}

// The phase-class kernel: the vector variant's conditions (one alignment
// phase) and at most 2048 whole 16-byte chunks per row (bf16 N ~16K, f32 N
// ~8K); 1 chunk per thread up to 256 chunks, 2 up to 1024, else 4. Its grid is the
// kernel's resident CTAs on every SM, at most 2: scratch mode's partial rows
// fill the workspace there, and in atomic mode every CTA adds N values at the
// end. Measured on GB300 (L2 flushed, us per call, 2 CTAs per SM -> all
// resident): f16 16384 x 1001 77.5 -> 101.8 (9 per SM), bf16 4096 x 2047
// 38.0 -> 49.4 (4 per SM). The grid is a multiple of the phase period P when
// it is below M, so that every residue class gets the same number of CTAs,
// and never below min(P, M), so that every class has one.
static int phase_grid(int64_t M, int P, int per_sm, const DeviceInfo &d) {
    if (per_sm < 1) per_sm = 1;
    if (per_sm > 2) per_sm = 2;
    int64_t grid = (int64_t)per_sm * d.num_sms;
    if (g_opts[RN_OPT_GRID] > 0 && grid > g_opts[RN_OPT_GRID]) grid = g_opts[RN_OPT_GRID];
    // every residue class needs a CTA: at least min(P, M), whatever the grid option says
    if (grid >= M) grid = M;
    else if (grid >= P) grid = grid / P * P;
    if (grid < P) grid = M < P ? M : P;
    if (grid < 1) grid = 1;
    return (int)grid;
}

// CTA size and chunks per thread of a phase-class kernel for a row of N
// elements of s bytes: 1 chunk per thread up to 256 whole 16-byte chunks, 2
// up to 1024, else 4, up to max_chunks. False past that.
static bool phase_shape(int N, int dtype, int max_chunks, int *cpt, int *threads) {
    const int64_t nvmax = (int64_t)N * elem_bytes(dtype) / 16;
    if (nvmax > max_chunks) return false;
    *cpt = nvmax > 1024 ? 4 : (nvmax > 256 ? 2 : 1);
    int t = (int)((nvmax + *cpt - 1) / *cpt + 31) / 32 * 32;
    *threads = t < 32 ? 32 : t;
    return true;
}

static bool plan_phase(const BwdProblem &p, const DeviceInfo &d, bool atomic, GenericPlan *plan) {
    if (!generic_vec_ok(p, d)) return false;
    int cpt, threads;
    if (!phase_shape(p.N, p.dtype, 2048, &cpt, &threads)) return false;
    // rows per CTA iteration: RN_OPT_TEAMS_PER_CTA = 1 or 2 forces it; one with four chunks a
    // thread
    int rows = g_opts[RN_OPT_TEAMS_PER_CTA];
    if (rows != 1 && rows != 2) rows = 2;
    if (cpt == 4) rows = 1;
    const int per_sm = phase_blocks_per_sm(p.dtype, p.dres != nullptr, atomic, cpt, rows, threads);
    plan->phase = cpt;
    plan->phase_rows = rows;
    plan->grid = phase_grid(p.M, phase_period(p.N, p.dtype), per_sm, d);
    // L2 prefetch of the rows two iterations ahead. Measured on GB300 (us per call, without ->
    // with): 1 chunk a thread f16 16384 x 1001 59.4 -> 52.0, bf16 4096 x 2047 23.4 -> 23.3;
    // 4 chunks bf16 4096 x 12290 88.9 -> 80.6; 2 chunks it helps with many rows per CTA or wide
    // rows of three tensors (bf16 16384 x 4095 85.5 -> 82.0, fused 4096 x 8190 +dres 72.2 ->
    // 67.4) and hurts otherwise (bf16 4096 x 4095 29.1 -> 29.5, fused +dres 37.5 -> 38.2, f32
    // 4096 x 4095 34.7 -> 37.4).
    {
        const int nt = p.dres ? 3 : 2;
        const int64_t rows_per_cta = (p.M + plan->grid - 1) / plan->grid;
        plan->prefetch = cpt != 2 || rows_per_cta >= 40 ||
                         (int64_t)nt * p.N * elem_bytes(p.dtype) >= 40 * 1024;
    }
    plan->cpb = 0;
    plan->rows = 0;
    plan->threads = threads;
    plan->smem_dw = atomic;
    // the atomic mode's staged partial; with four 16-bit chunks a thread, first the gamma chunks
    size_t smem = atomic ? (size_t)p.N * 4 : 0;
    if (cpt == 4 && p.dtype != kF32 && smem < (size_t)threads * 4 * 16) smem = (size_t)threads * 4 * 16;
    plan->smem = smem;
    plan->atomic = atomic;
    return true;
}

// The staged phase-class kernel: the phase-class kernel's conditions (one
// alignment phase, at most 2048 whole 16-byte chunks per row); 4 chunks a
// thread (RN_OPT_CHUNKS_PER_THREAD forces 1 or 2), teams of the fewest whole
// warps that cover a row, 2 shared-memory slots a team (RN_OPT_STAGES forces
// 2..4), as many teams as fit 512 threads, 15 named barriers and 200 KB of
// ring (RN_OPT_TEAMS_PER_CTA forces 1..15), and the phase-class kernel's grid
// rule at the resident CTAs per SM. The automatic choice takes it from 2048
// rows: with fewer, a CTA has too few rows to fill its pipeline and the
// phase-class kernel is as fast or faster. Measured on GB300 (L2 flushed, us
// per call, phase-class -> staged): bf16 4096 x 4095 29.2 -> 27.6, fused +dres
// 37.7 -> 31.4, 16384 x 4095 81.7 -> 71.4, 4096 x 12290 80.8 -> 66.8, 16384 x
// 2047 63.0 -> 40.8, 32768 x 1001 94.3 -> 42.5, 4096 x 255 20.5 -> 13.9, f32
// 4096 x 4095 34.9 -> 31.9, f16 2048 x 3001 19.3 -> 17.9; with fewer rows
// 1024 x 4095 15.6 -> 15.9, 1000 x 4095 15.5 -> 15.9, 128 x 2047 10.4 ->
// 12.6, 64 x 4095 12.1 -> 12.6.
constexpr int64_t kStageMinRows = 2048;

// A staged tile of two teams of 192-256 threads runs as one team a CTA at two CTAs an SM
// (unless RN_OPT_TEAMS_PER_CTA asks for a count). Measured on GB300 (L2 flushed, us per
// call, two teams -> one team at two CTAs an SM): RMSNorm backward bf16 4096 x 8190 38.3 ->
// 37.8, fused +dres 44.0 -> 42.5, 16384 x 8190 129.0 -> 127.9, f32 8192 x 2999 49.0 -> 48.7;
// forwards bf16 4096 x 8190 27.6 -> 26.5 (fused 44.3 -> 43.1, LayerNorm 36.8 -> 36.1), f32 4096
// x 4095 24.4 -> 22.3 (LayerNorm 26.9 -> 25.8), bf16 16384 x 8190 LayerNorm 117.6 -> 113.0;
// LayerNorm backward bf16 4096 x 4095 35.8 -> 33.5 (the phase-class kernel: 35.7), 8192 x 2999
// 50.7 -> 49.7. Smaller teams lose that way (128 threads, bf16 4096 x 4095: 25.6 -> 31.8).
static int stage_teams_split(int teams, int team_threads) {
    const int want = g_opts[RN_OPT_TEAMS_PER_CTA];
    return (want == 0 && teams == 2 && team_threads >= 192) ? 1 : teams;
}

static bool plan_stage(const BwdProblem &p, const DeviceInfo &d, bool atomic, bool forced,
                       StagePlan *plan) {
    if (!forced && p.M < kStageMinRows) return false;
    if (!generic_vec_ok(p, d)) return false;
    const int64_t maxnv = (int64_t)p.N * elem_bytes(p.dtype) / 16;
    if (maxnv > kRowMaxChunks) return false;
    int cpt = g_opts[RN_OPT_CHUNKS_PER_THREAD];
    if (cpt != 1 && cpt != 2) cpt = 4;
    int tthr = (int)((maxnv + cpt - 1) / cpt + 31) / 32 * 32;
    if (tthr < 32) tthr = 32;
    if (tthr > 512) return false;
    int slots = g_opts[RN_OPT_STAGES];
    if (slots < 2 || slots > 4) slots = 2;
    const bool dres = p.dres != nullptr;
    const size_t budget = d.smem_optin < 200 * 1024 ? d.smem_optin : 200 * 1024;
    int teams = 512 / tthr;
    if (teams > 15) teams = 15;
    const int want_teams = g_opts[RN_OPT_TEAMS_PER_CTA];
    if (want_teams >= 1 && want_teams <= 15 && want_teams * tthr <= 512) teams = want_teams;
    size_t smem = stage_smem_bytes(p.N, p.dtype, dres, teams, slots, cpt, tthr, nullptr, nullptr);
    while (teams > 1 && smem > budget) {
        --teams;
        smem = stage_smem_bytes(p.N, p.dtype, dres, teams, slots, cpt, tthr, nullptr, nullptr);
    }
    if (smem > d.smem_optin) return false;
    teams = stage_teams_split(teams, tthr);
    smem = stage_smem_bytes(p.N, p.dtype, dres, teams, slots, cpt, tthr, nullptr, nullptr);
    plan->cpt = cpt;
    plan->team_threads = tthr;
    plan->teams = teams;
    plan->slots = slots;
    plan->smem = smem;
    plan->atomic = atomic;
    const int per_sm = stage_blocks_per_sm(p.dtype, dres, atomic, cpt, teams * tthr, smem);
    plan->grid = phase_grid(p.M, phase_period(p.N, p.dtype), per_sm, d);
    plan->skip_row = g_opts[RN_OPT_TEST_WAIT_TIMEOUT] > 0 ? g_opts[RN_OPT_TEST_WAIT_TIMEOUT] - 1 : -1;
    return true;
}

static void plan_generic(const BwdProblem &p, const DeviceInfo &d, bool atomic, GenericPlan *plan) {
    plan->cpb = 0;
    plan->phase = 0;
    // RN_OPT_GENERIC_KERNEL: 1 phase-class, 2 vector, 3 realigning, 4 element-wise (5, the
    // staged phase-class kernel, is planned before this)
    const int pick = g_opts[RN_OPT_GENERIC_KERNEL];
    if ((pick <= 1 || pick == 5) && plan_phase(p, d, atomic, plan)) return;
    if (pick == 3 && plan_realign(p, d, plan)) return;
    plan->threads = p.N >= 4096 ? 512 : 256;
    const size_t budget = d.smem_optin < 200 * 1024 ? d.smem_optin : 200 * 1024;
    plan->smem_dw = generic_smem_bytes(p.N, true) <= budget;
    plan->smem = generic_smem_bytes(p.N, plan->smem_dw);
    plan->rows = 0;
    if (pick != 4 && generic_vec_ok(p, d)) {
        // rows in flight per CTA iteration: 4 when a row's chunks leave most
        // threads idle, else 2
        const int chunks = (int)((int64_t)p.N * elem_bytes(p.dtype) / 16);
        plan->threads = chunks >= 256 ? 512 : 256;
        plan->rows = chunks * 2 < plan->threads ? 4 : 2;
        plan->smem_dw = true;
        plan->smem = generic_vec_smem_bytes(p.N);
    }
    int64_t grid = plan->rows ? (p.M + plan->rows - 1) / plan->rows : p.M;
    if (grid > max_partial_rows(d)) grid = max_partial_rows(d);
    if (g_opts[RN_OPT_GRID] > 0 && grid > g_opts[RN_OPT_GRID]) grid = g_opts[RN_OPT_GRID];
    if (grid < 1) grid = 1;
    plan->grid = (int)grid;
    plan->atomic = false;
}

// Weight-gradient mode. Measured on GB300 (L2 flushed, us per call, atomic
// vs scratch): fp32 vector atomics (zeroing and cast overlapped by
// programmatic dependent launch) win from a few MB up: bf16 4096 x 4096
// 22.7 vs 23.3, fused +dres 27.1 vs 27.7, f32 512 x 3000 12.5 vs 12.6. On
// the smallest problems the scratch mode's two launches (row pass, then a
// finalize that sums the partial rows and casts) beat the atomic mode's
// three: f16 128 x 4096 11.9 vs 10.4, bf16 512 x 2048 11.7 vs 10.7, f32
// 128 x 1024 8.6 vs 8.4. So the automatic choice is scratch when a row
// tensor holds at most 2 MiB, else atomics where dweight_f32 is 16-byte
// aligned. RN_OPT_DWEIGHT_MODE = 1 / 2 forces scratch (deterministic,
// bitwise repeatable) / atomics.
constexpr int64_t kSmallProblemBytes = 2 << 20;

static bool want_atomic(const BwdProblem &p) {
    if (p.dw_f32 == nullptr) return false;  // no fp32 buffer to accumulate into
    const int m = g_opts[RN_OPT_DWEIGHT_MODE];
    if (m == 1) return false;
    if (m == 0 && p.M * (int64_t)p.N * elem_bytes(p.dtype) <= kSmallProblemBytes) return false;
    return aligned16(p.dw_f32);
}

// Outputs of the weight-gradient reduction: one or two length-N fp32 results
// (LayerNorm: dgamma, dbeta) with optional casts, and where the scratch
// mode's partial rows are (G rows of ld floats).
struct DwOutputs {
    float *f32_1;
    void *cast_1;
    float *f32_2;
    void *cast_2;
    int N;
    int dtype;
    const float *partials;
    int G;
    int ld;
};

// The kernels of one backward call around its pass: in atomic mode, zero the
// fp32 outputs, run the pass (`pass(true)`: a programmatic dependent of the
// zeroing kernel) and cast; in scratch mode, run the pass and the finalize
// that sums the partial rows and casts. Profile events bracket the pass when
// set.
template <typename Pass>
static rn_status run_sequence(bool atomic, const DwOutputs &o, cudaStream_t s, Pass pass) {
    cudaError_t e;
    if (atomic) {
        e = launch_zero_f32(o.f32_1, o.N, s, o.f32_2);
        if (e != cudaSuccess) return cuda_fail(e, "zero launch");
    }
    const bool prof = g_ev_begin && g_ev_end;
    if (prof) {
        e = cudaEventRecord(g_ev_begin, s);
        if (e != cudaSuccess) return cuda_fail(e, "profile event");
    }
    e = pass(atomic);
    if (e != cudaSuccess) return cuda_fail(e, "backward pass launch");
    if (prof) {
        e = cudaEventRecord(g_ev_end, s);
        if (e != cudaSuccess) return cuda_fail(e, "profile event");
    }
    if (atomic) {
        if (!o.cast_1 && !o.cast_2) return RN_OK;
        // (the atomic mode runs only with the fp32 buffers of every requested output)
        e = launch_cast(o.f32_1, o.cast_1, o.N, o.dtype, s, !prof, o.f32_2, o.cast_2);
        return e == cudaSuccess ? RN_OK : cuda_fail(e, "cast launch");
    }
    if (!o.f32_1 && !o.cast_1 && !o.f32_2 && !o.cast_2) return RN_OK;  // no weight gradient asked
    e = launch_finalize2(o.partials, o.G, o.ld, o.N, o.f32_1, o.cast_1, o.f32_2, o.cast_2, o.dtype,
                         s, !prof);
    return e == cudaSuccess ? RN_OK : cuda_fail(e, "finalize launch");
}

static void plan_string_cluster(const ClusterPlan &cp, const char *engine, bool atomic) {
    snprintf(g_plan, sizeof(g_plan),
             "engine=%s csize=%d slice=%d cpt=%d threads=%d stages=%d clusters=%d smem=%zu dw=%s",
             engine, cp.csize, cp.slice, cp.cpt, cp.threads, cp.stages, cp.clusters, cp.smem,
             atomic ? "atomic" : "scratch");
}

static void plan_string_row(const RowPlan &rp, const char *engine, bool atomic) {
    snprintf(g_plan, sizeof(g_plan),
             "engine=%s cpt=%d team_threads=%d teams=%d stages=%d grid=%d smem=%zu dw=%s",
             engine, rp.cpt, rp.team_threads, rp.teams, rp.stages, rp.grid, rp.smem,
             atomic ? "atomic" : "scratch");
}

static void plan_string_stage(const StagePlan &sp, const char *engine, bool atomic) {
    snprintf(g_plan, sizeof(g_plan),
             "engine=%s staged cpt=%d team_threads=%d teams=%d slots=%d grid=%d smem=%zu dw=%s",
             engine, sp.cpt, sp.team_threads, sp.teams, sp.slots, sp.grid, sp.smem,
             atomic ? "atomic" : "scratch");
}

static void plan_string_generic(const GenericPlan &gp, const char *engine, bool atomic) {
    if (gp.phase)
        snprintf(g_plan, sizeof(g_plan),
                 "engine=%s phase cpt=%d rows=%d threads=%d grid=%d prefetch=%d dw=%s", engine,
                 gp.phase, gp.phase_rows, gp.threads, gp.grid, (int)gp.prefetch,
                 atomic ? "atomic" : "scratch");
    else if (gp.cpb)
        snprintf(g_plan, sizeof(g_plan), "engine=%s realign cpb=%d rows=%d threads=%d grid=%d dw=%s",
                 engine, gp.cpb, gp.rows, gp.threads, gp.grid, atomic ? "atomic" : "scratch");
    else if (gp.rows)
        snprintf(g_plan, sizeof(g_plan), "engine=%s vec rows=%d threads=%d grid=%d dw=%s", engine,
                 gp.rows, gp.threads, gp.grid, atomic ? "atomic" : "scratch");
    else
        snprintf(g_plan, sizeof(g_plan), "engine=%s threads=%d grid=%d smem_dw=%d dw=%s", engine,
                 gp.threads, gp.grid, (int)gp.smem_dw, atomic ? "atomic" : "scratch");
}

// The phase-class forward's launch shape: 1 chunk a thread up to 256 whole
// 16-byte chunks, else 2; the backward phase-class kernel's grid rule (two
// CTAs per SM, a multiple of the period, never below min(P, M)).
struct FwdPhasePlan {
    int cpt, threads, grid;
};

static FwdPhasePlan plan_fwd_phase(const FwdRowProblem &q, const DeviceInfo &d);

// The forward staged phase-class kernel: row tensors at one alignment phase, at most 2048
// whole 16-byte chunks per row; 4 chunks a thread (RN_OPT_CHUNKS_PER_THREAD forces 1 or 2),
// teams of the fewest whole warps that cover a row, 2 shared-memory slots a team
// (RN_OPT_STAGES forces 2..4), as many teams as fit 512 threads, 15 named barriers and 200 KB
// of ring (RN_OPT_TEAMS_PER_CTA forces 1..15), and the phase-class grid rule at the resident
// CTAs per SM. RN_OPT_GENERIC_KERNEL = 5 forces it; any other non-zero pick leaves the rows to
// the vector or phase-class forward.
// The automatic choice, measured on GB300 (L2 flushed, us per call, vector or phase-class ->
// staged), takes it from 2048 rows:
//  * LayerNorm, always: bf16 4096 x 4095 24.6 -> 22.5, 16384 x 8190 177.7 -> 117.3, 4096 x
//    16383 87.9 -> 63.4, 16384 x 2047 71.6 -> 36.4, 32768 x 509 108.0 -> 34.6, f32 4096 x 4095
//    32.8 -> 26.6, f16 2048 x 1001 14.2 -> 10.6; 2048 x 4095 16.4 -> 16.3. Below 2048 rows the
//    16-bit phase-class forward is faster (1024 x 4095 11.9 vs 13.0, 64 x 4095 8.3 vs 10.1, 512
//    x 1001 8.3 vs 10.1), but the vector kernel is not, from 256 rows: f32 300 x 2999 9.7 ->
//    8.4, 512 x 4095 11.3 -> 10.1, 1024 x 6001 17.8 -> 16.2, bf16 256 x 12290 13.0 -> 12.1,
//    1024 x 12290 23.3 -> 20.7, 1024 x 16383 29.0 -> 23.8.
//  * RMSNorm, with at least 6 rows a team or rows of at most 256 chunks (where the vector
//    kernel's CTA per row leaves most threads idle): bf16 4096 x 4095 19.5 -> 18.2, 16384 x
//    8190 98.8 -> 89.1, 32768 x 4095 115.6 -> 86.5, 16384 x 2047 44.8 -> 26.4, f16 16384 x 1001
//    45.2 -> 19.9, f32 4096 x 4095 28.4 -> 24.3; fewer rows a team lose (2048 x 4095 13.1 ->
//    14.1, 3072 x 4095 16.1 -> 16.3), and so do the one-team rows of bf16 12290 (4096 rows 39.1
//    -> 41.3, 16384 rows 142.1 -> 147.1), which keep it for simplicity.
//  * Fused-add, with one team a CTA or rows of at most 256 chunks: bf16 8192 x 16383 176.4 ->
//    169.6, 4096 x 12290 65.7 -> 64.4, f32 16384 x 6001 249.7 -> 241.1, bf16 16384 x 2047 50.6
//    -> 44.2, f16 16384 x 1001 51.2 -> 24.4. With two or more teams the vector kernel's
//    four streams keep the copy engines busier (bf16 16384 x 8190 162.3 vs 171.6, 32768 x 4095
//    165.0 vs 171.2, 16384 x 4095 83.9 vs 86.3, f32 8192 x 4095 82.9 vs 84.2).
constexpr int64_t kFwdStageMinRows = 2048;

static bool plan_fwd_stage(const FwdRowProblem &q, const DeviceInfo &d, StagePlan *plan) {
    const int pick = g_opts[RN_OPT_GENERIC_KERNEL];
    if (pick != 0 && pick != 5) return false;
    if (pick == 0 && q.M < kFwdStageMinRows) {
        // below 2048 rows: only the LayerNorm forward from 256 rows, and only where the vector
        // kernel would take the rows (fp32, or rows past the phase-class kernel's 1024 chunks)
        const bool ln_phase = fwd_phase_ok(q) && (q.dtype != kF32 || !fwd_generic_vec_ok(q));
        if (q.mode != kFwdLn || ln_phase || q.M < 256) return false;
    }
    if (!fwd_stage_ok(q)) return false;
    const int64_t maxnv = (int64_t)q.N * elem_bytes(q.dtype) / 16;
    int cpt = g_opts[RN_OPT_CHUNKS_PER_THREAD];
    if (cpt != 1 && cpt != 2) cpt = 4;
    int tthr = (int)((maxnv + cpt - 1) / cpt + 31) / 32 * 32;
    if (tthr < 32) tthr = 32;
    if (tthr > 512) return false;
    int slots = g_opts[RN_OPT_STAGES];
    if (slots < 2 || slots > 4) slots = 2;
    const size_t budget = d.smem_optin < 200 * 1024 ? d.smem_optin : 200 * 1024;
    int teams = 512 / tthr;
    if (teams > 15) teams = 15;
    const int want_teams = g_opts[RN_OPT_TEAMS_PER_CTA];
    if (want_teams >= 1 && want_teams <= 15 && want_teams * tthr <= 512) teams = want_teams;
    size_t smem = fwd_stage_smem_bytes(q.N, q.dtype, q.mode, teams, slots);
    while (teams > 1 && smem > budget) {
        --teams;
        smem = fwd_stage_smem_bytes(q.N, q.dtype, q.mode, teams, slots);
    }
    if (smem > d.smem_optin) return false;
    plan->cpt = cpt;
    plan->team_threads = tthr;
    plan->teams = teams;
    plan->slots = slots;
    plan->smem = smem;
    plan->atomic = false;
    const int per_sm = fwd_stage_blocks_per_sm(q.dtype, q.mode, cpt, teams * tthr, smem);
    plan->grid = phase_grid(q.M, phase_period(q.N, q.dtype), per_sm, d);
    plan->skip_row = g_opts[RN_OPT_TEST_WAIT_TIMEOUT] > 0 ? g_opts[RN_OPT_TEST_WAIT_TIMEOUT] - 1 : -1;
    if (pick == 0 && maxnv > 256) {
        if (q.mode == kFwdRms && q.M < 6 * (int64_t)plan->grid * teams) return false;
        if (q.mode == kFwdFused && teams > 1) return false;
    }
    const int split = stage_teams_split(teams, tthr);
    if (split != teams) {
        plan->teams = split;
        plan->smem = fwd_stage_smem_bytes(q.N, q.dtype, q.mode, split, slots);
        const int per = fwd_stage_blocks_per_sm(q.dtype, q.mode, cpt, split * tthr, plan->smem);
        plan->grid = phase_grid(q.M, phase_period(q.N, q.dtype), per, d);
    }
    return true;
}

static void plan_string_fwd_stage(const char *op, const StagePlan &sp) {
    snprintf(g_plan, sizeof(g_plan),
             "%s engine=generic staged cpt=%d team_threads=%d teams=%d slots=%d grid=%d smem=%zu", op,
             sp.cpt, sp.team_threads, sp.teams, sp.slots, sp.grid, sp.smem);
}

static void plan_string_fwd(const char *op, bool vec, bool row, bool gvec, const RowPlan &rp,
                            const FwdPhasePlan *fp = nullptr) {
    if (fp) {
        snprintf(g_plan, sizeof(g_plan), "%s engine=generic phase cpt=%d threads=%d grid=%d", op,
                 fp->cpt, fp->threads, fp->grid);
        return;
    }
    if (vec && row)
        snprintf(g_plan, sizeof(g_plan), "%s engine=row cpt=%d team_threads=%d teams=%d stages=%d "
                 "grid=%d", op, rp.cpt, rp.team_threads, rp.teams, rp.stages, rp.grid);
    else
        snprintf(g_plan, sizeof(g_plan), "%s engine=%s", op,
                 vec ? "long" : (gvec ? "generic vec" : "generic"));
}

static rn_status run_bwd(const BwdProblem &p, size_t ws_bytes, cudaStream_t s) {
    DeviceInfo d;
    int dev = 0;
    cudaError_t e = device_info(&d, &dev);
    if (e != cudaSuccess) return cuda_fail(e, "device query");
    if (p.ws == nullptr) return fail(RN_ERR_WORKSPACE, "workspace is NULL");
    if (((uintptr_t)p.ws & 255u) != 0) return fail(RN_ERR_WORKSPACE, "workspace not 256-byte aligned");
    const size_t need = ws_bytes_for(d, p.N);
    if (ws_bytes < need)
        return fail(RN_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", ws_bytes, need);

    if (p.M == 0) {
        snprintf(g_plan, sizeof(g_plan), "empty batch: finalize only");
        if (!p.dw_f32 && !p.dw_cast) return RN_OK;
        e = launch_finalize(nullptr, 0, p.N, p.dw_f32, p.dw_cast, p.dtype, s, false);
        return e == cudaSuccess ? RN_OK : cuda_fail(e, "finalize launch");
    }

    const int engine = g_opts[RN_OPT_BWD_ENGINE];
    RowPlan rp;
    GenericPlan gp;
    ClusterPlan cp;
    bool use_row = false, use_cluster = false;
    bool atomic = want_atomic(p);
    if (engine == 0 || engine == 1) {
        use_row = plan_row(p, d, &rp);
        if (!use_row && engine == 1)
            return fail(RN_ERR_UNSUPPORTED, "row engine cannot take N=%d dtype=%d here", p.N,
                        p.dtype);
    }
    if (!use_row && (engine == 0 || engine == 3)) {
        use_cluster = plan_cluster(p, d, atomic, engine == 3, &cp);
        if (!use_cluster && engine == 3)
            return fail(RN_ERR_UNSUPPORTED, "cluster engine cannot take N=%d dtype=%d here",
                        p.N, p.dtype);
    }
    const float *partials = reinterpret_cast<const float *>(p.ws + kWsHeaderBytes);
    if (use_cluster) {
        plan_string_cluster(cp, "cluster", atomic);
        const DwOutputs o = {p.dw_f32, p.dw_cast, nullptr, nullptr, p.N, p.dtype,
                             partials, cp.clusters, p.N};
        return run_sequence(atomic, o, s, [&](bool pdl) { return launch_bwd_cluster(p, cp, s, pdl); });
    }
    // the staged phase-class kernel first (RN_OPT_GENERIC_KERNEL automatic or 5)
    StagePlan sp;
    const int gpick = g_opts[RN_OPT_GENERIC_KERNEL];
    if (!use_row && (gpick == 0 || gpick == 5) && plan_stage(p, d, atomic, gpick == 5, &sp)) {
        plan_string_stage(sp, "generic", atomic);
        const DwOutputs o = {p.dw_f32, p.dw_cast, nullptr, nullptr, p.N, p.dtype,
                             partials, sp.grid, p.N};
        return run_sequence(atomic, o, s, [&](bool pdl) { return launch_bwd_stage(p, sp, s, pdl); });
    }
    if (!use_row) plan_generic(p, d, atomic, &gp);
    if (!use_row && atomic && !gp.rows && !gp.cpb && !gp.phase &&
        generic_smem_bytes(p.N, true) > d.smem_optin) {
        // the generic engine keeps its atomic-mode partial in shared memory
        if (g_opts[RN_OPT_DWEIGHT_MODE] == 2)
            return fail(RN_ERR_UNSUPPORTED, "atomic mode needs N*4 bytes of shared memory");
        atomic = false;
    }
    rp.atomic = gp.atomic = atomic;
    if (!use_row && atomic && !gp.rows && !gp.cpb && !gp.phase) {
        gp.smem_dw = true;
        gp.smem = generic_smem_bytes(p.N, true);
    }
    if (use_row) plan_string_row(rp, "row", atomic);
    else plan_string_generic(gp, "generic", atomic);
    const DwOutputs o = {p.dw_f32, p.dw_cast, nullptr, nullptr, p.N, p.dtype,
                         partials, use_row ? rp.grid : gp.grid, p.N};
    return run_sequence(atomic, o, s, [&](bool pdl) {
        if (use_row) return launch_bwd_row(p, rp, s, pdl);
        if (gp.phase) return launch_bwd_phase(p, gp, s, pdl);
        return gp.cpb ? launch_bwd_realign(p, gp, s, pdl) : launch_bwd_generic(p, gp, s, pdl);
    });
}

// ------------------------------------------------------------- LayerNorm
static size_t ln_ws_bytes_for(const DeviceInfo &d, int64_t N) {
    return kWsHeaderBytes + (size_t)max_partial_rows(d) * (size_t)N * 8;
}

static bool plan_ln_row(const LnBwdProblem &p, const DeviceInfo &d, RowPlan *plan) {
    const int row_bytes = p.N * elem_bytes(p.dtype);
    if (row_bytes % 16) return false;
    if (!aligned16(p.x) || !aligned16(p.dy) || !aligned16(p.gamma) || !aligned16(p.dx))
        return false;
    const int nchunks = row_bytes / 16;
    const size_t red = ln_row_smem_bytes(0, 0, 0);
    if (!plan_row_tile(p.M, nchunks, 2, red, kLnMaxCpt, ln_row_max_threads, d, plan)) return false;
    const bool forced = g_opts[RN_OPT_CHUNKS_PER_THREAD] || g_opts[RN_OPT_TEAMS_PER_CTA];
    // Measured on GB300 (bf16): when 2 chunks per thread leave one team per
    // SM, 4 chunks per thread and two teams are faster (N = 8192: 131.9 vs
    // 147.5 us at M = 16384, 42.1 vs 47.7 us at M = 4096).
    if (plan->teams == 1 && plan->cpt == 2 && !forced) {
        RowPlan wide;
        if (plan_row_tile(p.M, nchunks, 2, red, 4, ln_row_max_threads, d, &wide) && wide.teams >= 2)
            *plan = wide;
    }
    // A team alone on its SM: a 2-slot ring (N = 16384: 136.4 vs 140.1 us for 3 slots).
    if (plan->teams == 1 && plan->stages > 2 && g_opts[RN_OPT_STAGES] == 0) {
        plan->stages = 2;
        plan->smem = ln_row_smem_bytes(plan->teams, 2, plan->cpt * plan->team_threads);
    }
    return true;
}

static size_t ln_cluster_smem(int stages, int, int cpt, int threads) {
    return ln_cluster_smem_bytes(stages, cpt, threads);
}

static cudaError_t ln_cluster_query(const void *ctx, const ClusterPlan &plan, int *n) {
    return ln_cluster_max_active(*static_cast<const LnBwdProblem *>(ctx), plan, n);
}

static bool plan_ln_cluster(const LnBwdProblem &p, const DeviceInfo &d, bool atomic, bool forced,
                            ClusterPlan *plan) {
    const int row_bytes = p.N * elem_bytes(p.dtype);
    if (row_bytes % 16) return false;
    if (!aligned16(p.x) || !aligned16(p.dy) || !aligned16(p.gamma) || !aligned16(p.dx))
        return false;
    if (!cluster_tile(row_bytes / 16, 2, forced, d, ln_cluster_smem, plan)) return false;
    plan->atomic = atomic;
    return cluster_count("ln", p.M, p.dtype, false, d, plan, ln_cluster_query, &p);
}

// The LayerNorm phase-class kernel: x, dy and dx at one alignment phase and
// the RMSNorm kernel's row-size range and grid rule.
static bool plan_ln_phase(const LnBwdProblem &p, const DeviceInfo &d, bool atomic,
                          GenericPlan *plan) {
    const uintptr_t S = (uintptr_t)elem_bytes(p.dtype), ph = (uintptr_t)p.x & 15u;
    for (const void *q : {p.x, p.dy, static_cast<const void *>(p.dx)})
        if (((uintptr_t)q & 15u) != ph || ((uintptr_t)q % S) != 0) return false;
    int cpt, threads;
    if (!phase_shape(p.N, p.dtype, 1024, &cpt, &threads)) return false;
    const size_t smem = ln_phase_smem_bytes(p.N, atomic);
    if (smem > (size_t)d.smem_optin) return false;
    const int per_sm = ln_phase_blocks_per_sm(p.dtype, atomic, cpt, threads, smem);
    plan->phase = cpt;
    plan->cpb = 0;
    plan->rows = 0;
    plan->threads = threads;
    plan->grid = phase_grid(p.M, phase_period(p.N, p.dtype), per_sm, d);
    // L2 prefetch of the row after the next one, by the RMSNorm phase-class kernel's rule
    {
        const int64_t rows_per_cta = (p.M + plan->grid - 1) / plan->grid;
        plan->prefetch = cpt != 2 || rows_per_cta >= 40 ||
                         (int64_t)2 * p.N * elem_bytes(p.dtype) >= 40 * 1024;
    }
    plan->smem_dw = atomic;
    plan->smem = smem;
    plan->atomic = atomic;
    return true;
}

// The LayerNorm staged phase-class kernel: x, dy and dx at one alignment
// phase, at most 2048 whole 16-byte chunks a row; 2 chunks a thread up to 512
// chunks a row, else 4 (RN_OPT_CHUNKS_PER_THREAD forces 1, 2 or 4; at 4 the two
// fp32 partials a column fill the register budget and ptxas spills 40 bytes, which
// the measurements below include), teams of the fewest whole warps that cover a row, 2 slots
// a team (RN_OPT_STAGES 2..4), as many teams as fit 512 threads, 15 named
// barriers and 200 KB (RN_OPT_TEAMS_PER_CTA forces 1..15), the phase-class
// grid rule. Taken automatically from 2048 rows, as the RMSNorm staged kernel.
// Measured on GB300 (L2 flushed, us per call, phase-class -> staged): f16 16384
// x 1001 62.1 -> 34.3 (8 teams), bf16 16384 x 509 54.5 -> 25.7 (15), 4096 x 2047
// 27.5 -> 23.6 (4), 4096 x 8190 64.7 -> 58.4 (1), 16384 x 8190 211.2 -> 193.1
// (1), f32 4096 x 4095 54.7 -> 43.9 (1), f32 8192 x 2999 80.7 -> 67.0 (1); a tile
// of two 256-thread teams split into one team at two CTAs an SM
// (stage_teams_split): bf16 4096 x 4095 35.7 -> 33.5, 4096 x 4100 35.5 -> 34.8,
// 8192 x 2999 51.1 -> 50.2, but 16384 x 4095 97.7 -> 99.5, where the phase-class
// kernel has 40+ rows a CTA and prefetches, so it keeps those (as two teams in
// one CTA: 35.8, 35.8, 50.5, 102.5; 3 or 4 slots a team no better); below 2048
// rows 1024 x 4095 18.3 -> 19.5, 512 x 4095 15.1 -> 16.8. Four chunks a thread
// against two (us per call): bf16 4096 x 8190 58.3 -> 57.5, 16384 x 8190 193.1 ->
// 184.1, f32 4096 x 4095 44.0 -> 37.9; rows of 1025-2048 chunks, which only 4
// chunks a thread can take, against the vector kernel: bf16 4096 x 12290 216.2 ->
// 91.0, 4096 x 16383 295.4 -> 103.4; shorter rows lose with 4 (4096 x 4095 34.7 ->
// 36.9, 4096 x 2047 23.5 -> 26.0). Rows past 1024 chunks take it at any row count
// (the vector kernel is the alternative there): bf16 1 x 12290 20.0 -> 15.6, 64 x
// 12290 26.4 -> 15.7, 1024 x 12290 74.7 -> 34.8, 1024 x 16383 95.4 -> 39.6, f32
// 512 x 6001 26.1 -> 18.0.
static bool plan_ln_stage(const LnBwdProblem &p, const DeviceInfo &d, bool atomic, bool forced,
                          StagePlan *plan) {
    const int64_t maxnv = (int64_t)p.N * elem_bytes(p.dtype) / 16;
    // below 2048 rows the phase-class kernel, where it can take the rows (up to 1024 chunks)
    if (!forced && p.M < kStageMinRows && maxnv <= 1024) return false;
    const uintptr_t S = (uintptr_t)elem_bytes(p.dtype), ph = (uintptr_t)p.x & 15u;
    for (const void *q : {p.x, p.dy, static_cast<const void *>(p.dx)})
        if (((uintptr_t)q & 15u) != ph || ((uintptr_t)q % S) != 0) return false;
    const int copt = g_opts[RN_OPT_CHUNKS_PER_THREAD];
    const int cpt = (copt == 1 || copt == 2 || copt == 4) ? copt : (maxnv <= 512 ? 2 : 4);
    if (maxnv > 512 * (int64_t)cpt) return false;
    int tthr = (int)((maxnv + cpt - 1) / cpt + 31) / 32 * 32;
    if (tthr < 32) tthr = 32;
    if (tthr > 512) return false;
    int slots = g_opts[RN_OPT_STAGES];
    if (slots < 2 || slots > 4) slots = 2;
    const size_t budget = d.smem_optin < 200 * 1024 ? d.smem_optin : 200 * 1024;
    int teams = 512 / tthr;
    if (teams > 15) teams = 15;
    const int want_teams = g_opts[RN_OPT_TEAMS_PER_CTA];
    if (want_teams >= 1 && want_teams <= 15 && want_teams * tthr <= 512) teams = want_teams;
    size_t smem = ln_stage_smem_bytes(p.N, p.dtype, teams, slots, nullptr, nullptr);
    while (teams > 1 && smem > budget) {
        --teams;
        smem = ln_stage_smem_bytes(p.N, p.dtype, teams, slots, nullptr, nullptr);
    }
    if (smem > d.smem_optin) return false;
    if (!forced && cpt == 2 && stage_teams_split(teams, tthr) != teams) {
        // with 40 or more rows a CTA the phase-class kernel's L2 prefetch pays and it is the
        // faster one there (bf16 16384 x 4095: 97.7 vs 99.5)
        const int64_t g2 = 2 * (int64_t)d.num_sms;
        if ((p.M + g2 - 1) / g2 >= 40) return false;
    }
    teams = stage_teams_split(teams, tthr);
    smem = ln_stage_smem_bytes(p.N, p.dtype, teams, slots, nullptr, nullptr);
    plan->cpt = cpt;
    plan->team_threads = tthr;
    plan->teams = teams;
    plan->slots = slots;
    plan->smem = smem;
    plan->atomic = atomic;
    const int per_sm = ln_stage_blocks_per_sm(p.dtype, atomic, cpt, teams * tthr, smem);
    plan->grid = phase_grid(p.M, phase_period(p.N, p.dtype), per_sm, d);
    plan->skip_row = g_opts[RN_OPT_TEST_WAIT_TIMEOUT] > 0 ? g_opts[RN_OPT_TEST_WAIT_TIMEOUT] - 1 : -1;
    return true;
}

static void plan_ln_generic(const LnBwdProblem &p, const DeviceInfo &d, bool atomic,
                            GenericPlan *plan) {
    plan->phase = 0;
    // RN_OPT_GENERIC_KERNEL: 1 phase-class, 2 (or 3) vector, 4 element-wise
    const int pick = g_opts[RN_OPT_GENERIC_KERNEL];  // 5 (staged, planned before this) as 0
    if ((pick <= 1 || pick == 5) && plan_ln_phase(p, d, atomic, plan)) return;
    plan->threads = p.N >= 4096 ? 512 : 256;
    const size_t budget = d.smem_optin < 200 * 1024 ? d.smem_optin : 200 * 1024;
    plan->smem_dw = ln_generic_smem_bytes(p.N, true) <= budget;
    plan->smem = ln_generic_smem_bytes(p.N, plan->smem_dw);
    plan->rows = 0;
    plan->cpb = 0;
    // vector variant: x, dy and dx at one alignment phase (element-aligned)
    const uintptr_t S = (uintptr_t)elem_bytes(p.dtype), ph = (uintptr_t)p.x & 15u;
    bool vec = pick != 4 && ln_generic_vec_smem_bytes(p.N) <= budget;
    for (const void *q : {p.x, p.dy, static_cast<const void *>(p.dx)})
        vec = vec && ((uintptr_t)q & 15u) == ph && ((uintptr_t)q % S) == 0;
    if (vec) {
        const int chunks = (int)((int64_t)p.N * elem_bytes(p.dtype) / 16);
        plan->threads = chunks >= 256 ? 512 : 256;
        plan->rows = chunks * 2 < plan->threads ? 4 : 2;
        plan->smem_dw = true;
        plan->smem = ln_generic_vec_smem_bytes(p.N);
    }
    int64_t grid = plan->rows ? (p.M + plan->rows - 1) / plan->rows : p.M;
    if (grid > max_partial_rows(d)) grid = max_partial_rows(d);
    if (g_opts[RN_OPT_GRID] > 0 && grid > g_opts[RN_OPT_GRID]) grid = g_opts[RN_OPT_GRID];
    if (grid < 1) grid = 1;
    plan->grid = (int)grid;
    plan->atomic = false;
}

static rn_status run_ln_bwd(const LnBwdProblem &p, size_t ws_bytes, cudaStream_t s) {
    DeviceInfo d;
    int dev = 0;
    cudaError_t e = device_info(&d, &dev);
    if (e != cudaSuccess) return cuda_fail(e, "device query");
    if (p.ws == nullptr) return fail(RN_ERR_WORKSPACE, "workspace is NULL");
    if (((uintptr_t)p.ws & 255u) != 0) return fail(RN_ERR_WORKSPACE, "workspace not 256-byte aligned");
    const size_t need = ln_ws_bytes_for(d, p.N);
    if (ws_bytes < need)
        return fail(RN_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", ws_bytes, need);
    const float *partials = reinterpret_cast<const float *>(p.ws + kWsHeaderBytes);

    if (p.M == 0) {
        snprintf(g_plan, sizeof(g_plan), "empty batch: finalize only");
        if (!p.dg_f32 && !p.dg_cast && !p.db_f32 && !p.db_cast) return RN_OK;
        e = launch_finalize2(nullptr, 0, 2 * p.N, p.N, p.dg_f32, p.dg_cast, p.db_f32, p.db_cast,
                             p.dtype, s, false);
        return e == cudaSuccess ? RN_OK : cuda_fail(e, "finalize launch");
    }

    const int engine = g_opts[RN_OPT_BWD_ENGINE];
    RowPlan rp;
    GenericPlan gp;
    ClusterPlan cp;
    bool use_row = false, use_cluster = false;
    // atomics need the fp32 buffer of every requested output
    bool atomic = g_opts[RN_OPT_DWEIGHT_MODE] != 1 && p.dg_f32 != nullptr &&
                  aligned16(p.dg_f32) && (p.db_cast == nullptr || p.db_f32 != nullptr) &&
                  (p.db_f32 == nullptr || aligned16(p.db_f32));
    if (engine == 0 || engine == 1) {
        use_row = plan_ln_row(p, d, &rp);
        if (!use_row && engine == 1)
            return fail(RN_ERR_UNSUPPORTED, "row engine cannot take N=%d dtype=%d here", p.N,
                        p.dtype);
    }
    if (!use_row && (engine == 0 || engine == 3)) {
        use_cluster = plan_ln_cluster(p, d, atomic, engine == 3, &cp);
        if (!use_cluster && engine == 3)
            return fail(RN_ERR_UNSUPPORTED, "cluster engine cannot take N=%d dtype=%d here",
                        p.N, p.dtype);
    }
    if (use_cluster) {
        plan_string_cluster(cp, "ln_cluster", atomic);
        const DwOutputs o = {p.dg_f32, p.dg_cast, p.db_f32, p.db_cast, p.N, p.dtype,
                             partials, cp.clusters, 2 * p.N};
        return run_sequence(atomic, o, s,
                            [&](bool pdl) { return launch_ln_bwd_cluster(p, cp, s, pdl); });
    }
    // the staged phase-class kernel first (RN_OPT_GENERIC_KERNEL automatic or 5)
    StagePlan sp;
    const int gpick = g_opts[RN_OPT_GENERIC_KERNEL];
    if (!use_row && (gpick == 0 || gpick == 5) && plan_ln_stage(p, d, atomic, gpick == 5, &sp)) {
        plan_string_stage(sp, "ln_generic", atomic);
        const DwOutputs o = {p.dg_f32, p.dg_cast, p.db_f32, p.db_cast, p.N, p.dtype,
                             partials, sp.grid, 2 * p.N};
        return run_sequence(atomic, o, s,
                            [&](bool pdl) { return launch_ln_bwd_stage(p, sp, s, pdl); });
    }
    if (!use_row) plan_ln_generic(p, d, atomic, &gp);
    if (!use_row && atomic && !gp.rows && !gp.phase &&
        ln_generic_smem_bytes(p.N, true) > d.smem_optin) {
        // the generic engine keeps its atomic-mode partials in shared memory
        if (g_opts[RN_OPT_DWEIGHT_MODE] == 2)
            return fail(RN_ERR_UNSUPPORTED, "atomic mode needs N*8 bytes of shared memory");
        atomic = false;
    }
    rp.atomic = gp.atomic = atomic;
    if (!use_row && atomic && !gp.rows && !gp.phase) {
        gp.smem_dw = true;
        gp.smem = ln_generic_smem_bytes(p.N, true);
    }
    if (use_row) plan_string_row(rp, "ln_row", atomic);
    else plan_string_generic(gp, "ln_generic", atomic);
    const DwOutputs o = {p.dg_f32, p.dg_cast, p.db_f32, p.db_cast, p.N, p.dtype,
                         partials, use_row ? rp.grid : gp.grid, 2 * p.N};
    return run_sequence(atomic, o, s, [&](bool pdl) {
        if (use_row) return launch_ln_bwd_row(p, rp, s, pdl);
        return gp.phase ? launch_ln_bwd_phase(p, gp, s, pdl) : launch_ln_bwd_generic(p, gp, s, pdl);
    });
}

static rn_status check_common(int64_t M, int64_t N, int dtype) {
    if (dtype < RN_F32 || dtype > RN_BF16) return fail(RN_ERR_INVALID_ARG, "bad dtype code %d", dtype);
    if (M < 0) return fail(RN_ERR_INVALID_ARG, "M must be >= 0 (got %lld)", (long long)M);
    if (N < 1) return fail(RN_ERR_INVALID_ARG, "N must be >= 1 (got %lld)", (long long)N);
    if (N > (int64_t)1 << 28) return fail(RN_ERR_UNSUPPORTED, "N too large (%lld)", (long long)N);
    if (M > ((int64_t)1 << 62) / N) return fail(RN_ERR_INVALID_ARG, "M*N overflows");
    return RN_OK;
}

// Every buffer must start at a multiple of its element size (the dtype's for
// row tensors, gamma, beta and the casts; 4 bytes for rstd, mean and the fp32
// outputs): the kernels load and store whole elements, and a misaligned one
// would fault on the GPU instead of failing here.
struct Buf {
    const void *p;
    int bytes;
    const char *name;
};

static rn_status check_alignment(std::initializer_list<Buf> bufs) {
    for (const Buf &b : bufs)
        if (b.p && ((uintptr_t)b.p % (uintptr_t)b.bytes) != 0)
            return fail(RN_ERR_INVALID_ARG, "%s is not aligned to its element size (%d bytes)",
                        b.name, b.bytes);
    return RN_OK;
}

static rn_status bwd_entry(const void *x, const void *gamma, const void *dy, const float *rstd,
                           const void *dres, void *dx, float *dw_f32, void *dw_cast, void *ws,
                           size_t ws_bytes, int64_t M, int64_t N, int dtype, void *stream) {
    g_err[0] = 0;
    g_plan[0] = 0;
    rn_status st = check_common(M, N, dtype);
    if (st != RN_OK) return st;
    if (!gamma) return fail(RN_ERR_INVALID_ARG, "gamma is required");
    if (M > 0 && (!x || !dy || !rstd || !dx))
        return fail(RN_ERR_INVALID_ARG, "x, dy, rstd and dx are required when M > 0");
    if (M > 0 && (dx == x || dx == dy || (void *)dx == (void *)rstd))
        return fail(RN_ERR_INVALID_ARG, "dx must not alias x, dy or rstd");
    {
        const int S = elem_bytes(dtype);
        st = check_alignment({{x, S, "x"}, {gamma, S, "gamma"}, {dy, S, "dy"}, {dres, S, "dresidual_out"},
                              {dx, S, "dx"}, {dw_cast, S, "dweight"}, {rstd, 4, "rstd"},
                              {dw_f32, 4, "dweight_f32"}});
        if (st != RN_OK) return st;
    }
    BwdProblem p;
    p.x = x;
    p.gamma = gamma;
    p.dy = dy;
    p.rstd = rstd;
    p.dres = dres;
    p.dx = dx;
    p.dw_f32 = dw_f32;
    p.dw_cast = dw_cast;
    p.ws = static_cast<uint8_t *>(ws);
    p.M = M;
    p.N = (int)N;
    p.dtype = dtype;
    return run_bwd(p, ws_bytes, static_cast<cudaStream_t>(stream));
}

static rn_status fwd_entry(const void *x, const void *residual, const void *gamma, float eps,
                           void *y, void *residual_out, float *rstd, int64_t M, int64_t N,
                           int dtype, void *stream, bool fused) {
    g_err[0] = 0;
    g_plan[0] = 0;
    rn_status st = check_common(M, N, dtype);
    if (st != RN_OK) return st;
    if (!(eps >= 0.f)) return fail(RN_ERR_INVALID_ARG, "eps must be >= 0");
    if (!gamma) return fail(RN_ERR_INVALID_ARG, "gamma is required");
    if (M > 0 && (!x || !y)) return fail(RN_ERR_INVALID_ARG, "input and output are required");
    if (fused && M > 0 && (!residual || !residual_out))
        return fail(RN_ERR_INVALID_ARG, "residual and residual_out are required");
    {
        const int S = elem_bytes(dtype);
        st = check_alignment({{x, S, "x"}, {residual, S, "residual"}, {gamma, S, "gamma"},
                              {y, S, "output"}, {residual_out, S, "residual_out"},
                              {rstd, 4, "rstd"}});
        if (st != RN_OK) return st;
    }
    if (M == 0) return RN_OK;
    DeviceInfo d;
    cudaError_t e = device_info(&d, nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "device query");
    FwdProblem p;
    p.x = x;
    p.residual = fused ? residual : nullptr;
    p.gamma = gamma;
    p.y = y;
    p.residual_out = fused ? residual_out : nullptr;
    p.rstd = rstd;
    p.eps = eps;
    p.M = M;
    p.N = (int)N;
    p.dtype = dtype;
    const int eb = elem_bytes(dtype);
    const bool vec = ((N * eb) % 16 == 0) && aligned16(x) && aligned16(gamma) && aligned16(y) &&
                     (!fused || (aligned16(residual) && aligned16(residual_out)));
    RowPlan rp;
    const int nt = fused ? 2 : 1;
    const bool row = vec && plan_row_tile(M, (int)(N * eb / 16), nt, fwd_row_smem_bytes(0, 0, nt, 0),
                                          4, row_max_threads, d, &rp, false);
    FwdRowProblem q;
    q.mode = fused ? kFwdFused : kFwdRms;
    q.x = x;
    q.residual = fused ? residual : nullptr;
    q.gamma = gamma;
    q.beta = nullptr;
    q.y = y;
    q.residual_out = fused ? residual_out : nullptr;
    q.mean = nullptr;
    q.rstd = rstd;
    q.eps = eps;
    q.M = M;
    q.N = (int)N;
    q.dtype = dtype;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const char *op = fused ? "fused_add_fwd" : "rmsnorm_fwd";
    StagePlan sp;
    if (!vec && plan_fwd_stage(q, d, &sp)) {
        plan_string_fwd_stage(op, sp);
        e = launch_fwd_stage(q, sp, cs);
        return e == cudaSuccess ? RN_OK : cuda_fail(e, "forward launch");
    }
    // The RMSNorm forwards keep the vector kernel where it can run (see plan_fwd_phase); the
    // phase-class kernel takes gamma at any alignment.
    if (!vec && !fwd_generic_vec_ok(q) && fwd_phase_ok(q)) {
        const FwdPhasePlan fp = plan_fwd_phase(q, d);
        plan_string_fwd(op, vec, row, false, rp, &fp);
        e = launch_fwd_phase(q, fp.cpt, fp.grid, fp.threads, cs);
        return e == cudaSuccess ? RN_OK : cuda_fail(e, "forward launch");
    }
    const bool gvec = !vec && fwd_generic_vec_ok(q);
    plan_string_fwd(op, vec, row, gvec, rp);
    if (vec)
        e = row ? launch_fwd_row(q, rp, cs) : launch_fwd_long(q, d.num_sms, cs);
    else
        e = gvec ? launch_fwd_generic_vec(q, d.num_sms, cs) : launch_fwd(p, d.num_sms, cs);
    return e == cudaSuccess ? RN_OK : cuda_fail(e, "forward launch");
}

// Measured on GB300 (L2 flushed, us per call; vector kernel -> phase-class kernel): the
// LayerNorm forward in 16-bit types gains (bf16 4096 x 4095 32.5 -> 24.5, 4096 x 4100 30.8 ->
// 24.6, 16384 x 8190 186.6 -> 175.4, f16 16384 x 1001 62.8 -> 61.3), its rows staying in
// registers through the mean and variance passes. The RMSNorm forwards lose (bf16 4096 x 4095
// 19.2 -> 20.5, fused 23.1 -> 24.6, 16384 x 8190 98.5 -> 149.4) and so does the f32 LayerNorm
// (4096 x 4095 32.8 -> 43.0): the vector kernel's eight CTAs per SM keep more rows in flight.
// So the phase-class forward runs for the 16-bit LayerNorm, and for the others only where the
// vector kernel cannot (gamma or beta off a 16-byte boundary).
static FwdPhasePlan plan_fwd_phase(const FwdRowProblem &q, const DeviceInfo &d) {
    FwdPhasePlan fp;
    const int64_t nvmax = (int64_t)q.N * elem_bytes(q.dtype) / 16;
    fp.cpt = nvmax > 256 ? 2 : 1;
    const int t = (int)((nvmax + fp.cpt - 1) / fp.cpt + 31) / 32 * 32;
    fp.threads = t < 32 ? 32 : t;
    fp.grid = phase_grid(q.M, phase_period(q.N, q.dtype), 2, d);
    return fp;
}

static rn_status ln_fwd_entry(const void *x, const void *gamma, const void *beta, float eps,
                              void *y, float *mean, float *rstd, int64_t M, int64_t N, int dtype,
                              void *stream) {
    g_err[0] = 0;
    g_plan[0] = 0;
    rn_status st = check_common(M, N, dtype);
    if (st != RN_OK) return st;
    if (!(eps >= 0.f)) return fail(RN_ERR_INVALID_ARG, "eps must be >= 0");
    if (!gamma) return fail(RN_ERR_INVALID_ARG, "gamma is required");
    if (M > 0 && (!x || !y)) return fail(RN_ERR_INVALID_ARG, "input and output are required");
    {
        const int S = elem_bytes(dtype);
        st = check_alignment({{x, S, "x"}, {gamma, S, "gamma"}, {beta, S, "beta"}, {y, S, "y"},
                              {mean, 4, "mean"}, {rstd, 4, "rstd"}});
        if (st != RN_OK) return st;
    }
    if (M == 0) return RN_OK;
    DeviceInfo d;
    cudaError_t e = device_info(&d, nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "device query");
    LnFwdProblem p;
    p.x = x;
    p.gamma = gamma;
    p.beta = beta;
    p.y = y;
    p.mean = mean;
    p.rstd = rstd;
    p.eps = eps;
    p.M = M;
    p.N = (int)N;
    p.dtype = dtype;
    const int eb = elem_bytes(dtype);
    const bool vec = ((N * eb) % 16 == 0) && aligned16(x) && aligned16(gamma) && aligned16(y) &&
                     (!beta || aligned16(beta));
    RowPlan rp;
    const bool row = vec && plan_row_tile(M, (int)(N * eb / 16), 1, fwd_row_smem_bytes(0, 0, 1, 0),
                                          4, row_max_threads, d, &rp, false);
    FwdRowProblem q;
    q.mode = kFwdLn;
    q.x = x;
    q.residual = nullptr;
    q.gamma = gamma;
    q.beta = beta;
    q.y = y;
    q.residual_out = nullptr;
    q.mean = mean;
    q.rstd = rstd;
    q.eps = eps;
    q.M = M;
    q.N = (int)N;
    q.dtype = dtype;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    StagePlan sp;
    if (!vec && plan_fwd_stage(q, d, &sp)) {
        plan_string_fwd_stage("layernorm_fwd", sp);
        e = launch_fwd_stage(q, sp, cs);
        return e == cudaSuccess ? RN_OK : cuda_fail(e, "forward launch");
    }
    if (!vec && fwd_phase_ok(q) && (dtype != kF32 || !fwd_generic_vec_ok(q))) {
        const FwdPhasePlan fp = plan_fwd_phase(q, d);
        plan_string_fwd("layernorm_fwd", vec, row, false, rp, &fp);
        e = launch_fwd_phase(q, fp.cpt, fp.grid, fp.threads, cs);
        return e == cudaSuccess ? RN_OK : cuda_fail(e, "forward launch");
    }
    const bool gvec = !vec && fwd_generic_vec_ok(q);
    plan_string_fwd("layernorm_fwd", vec, row, gvec, rp);
    if (vec)
        e = row ? launch_fwd_row(q, rp, cs) : launch_fwd_long(q, d.num_sms, cs);
    else
        e = gvec ? launch_fwd_generic_vec(q, d.num_sms, cs) : launch_ln_fwd(p, d.num_sms, cs);
    return e == cudaSuccess ? RN_OK : cuda_fail(e, "forward launch");
}

static rn_status ln_bwd_entry(const void *x, const void *gamma, const void *dy, const float *mean,
                              const float *rstd, void *dx, float *dg_f32, float *db_f32,
                              void *dg_cast, void *db_cast, void *ws, size_t ws_bytes, int64_t M,
                              int64_t N, int dtype, void *stream) {
    g_err[0] = 0;
    g_plan[0] = 0;
    rn_status st = check_common(M, N, dtype);
    if (st != RN_OK) return st;
    if (!gamma) return fail(RN_ERR_INVALID_ARG, "gamma is required");
    if (db_f32 && db_f32 == dg_f32)
        return fail(RN_ERR_INVALID_ARG, "dbeta_f32 must not alias dgamma_f32");
    if (M > 0 && (!x || !dy || !mean || !rstd || !dx))
        return fail(RN_ERR_INVALID_ARG, "x, dy, mean, rstd and dx are required when M > 0");
    if (M > 0 && (dx == x || dx == dy || (void *)dx == (void *)mean || (void *)dx == (void *)rstd))
        return fail(RN_ERR_INVALID_ARG, "dx must not alias x, dy, mean or rstd");
    {
        const int S = elem_bytes(dtype);
        st = check_alignment({{x, S, "x"}, {gamma, S, "gamma"}, {dy, S, "dy"}, {dx, S, "dx"},
                              {dg_cast, S, "dgamma"}, {db_cast, S, "dbeta"}, {mean, 4, "mean"},
                              {rstd, 4, "rstd"}, {dg_f32, 4, "dgamma_f32"},
                              {db_f32, 4, "dbeta_f32"}});
        if (st != RN_OK) return st;
    }
    LnBwdProblem p;
    p.x = x;
    p.gamma = gamma;
    p.dy = dy;
    p.mean = mean;
    p.rstd = rstd;
    p.dx = dx;
    p.dg_f32 = dg_f32;
    p.db_f32 = db_f32;
    p.dg_cast = dg_cast;
    p.db_cast = db_cast;
    p.ws = static_cast<uint8_t *>(ws);
    p.M = M;
    p.N = (int)N;
    p.dtype = dtype;
    return run_ln_bwd(p, ws_bytes, static_cast<cudaStream_t>(stream));
}

}  // namespace rn

using namespace rn;

extern "C" {

int rn_abi_version(void) { return 1; }

const char *rn_status_string(int s) {
    switch (s) {
    case RN_OK: return "ok";
    case RN_ERR_INVALID_ARG: return "invalid argument";
    case RN_ERR_UNSUPPORTED: return "unsupported shape or alignment";
    case RN_ERR_CUDA: return "CUDA error";
    case RN_ERR_WORKSPACE: return "bad workspace";
    default: return "unknown status";
    }
}

const char *rn_last_error(void) { return g_err; }

const char *rn_last_plan(void) { return g_plan; }

rn_status rn_set_option(int option, int value) {
    if (option < 0 || option >= RN_OPT_COUNT) return fail(RN_ERR_INVALID_ARG, "bad option %d", option);
    if (value < 0) return fail(RN_ERR_INVALID_ARG, "option values are >= 0");
    g_opts[option] = value;
    return RN_OK;
}

int rn_get_option(int option) {
    if (option < 0 || option >= RN_OPT_COUNT) return -1;
    return g_opts[option];
}

rn_status rn_take_device_status(unsigned int *status) {
    g_err[0] = 0;
    if (!status) return fail(RN_ERR_INVALID_ARG, "status is NULL");
    cudaError_t e = take_device_status(status);
    return e == cudaSuccess ? RN_OK : cuda_fail(e, "device status");
}

rn_status rn_set_profile_events(void *ev_begin, void *ev_end) {
    g_ev_begin = static_cast<cudaEvent_t>(ev_begin);
    g_ev_end = static_cast<cudaEvent_t>(ev_end);
    return RN_OK;
}

rn_status rn_rmsnorm_fwd(const void *x, const void *gamma, float eps, void *y, float *rstd,
                         int64_t M, int64_t N, int dtype, void *stream) {
    return fwd_entry(x, nullptr, gamma, eps, y, nullptr, rstd, M, N, dtype, stream, false);
}

rn_status rn_fused_add_rmsnorm_fwd(const void *x, const void *residual, const void *gamma,
                                   float eps, void *out, void *residual_out, float *rstd,
                                   int64_t M, int64_t N, int dtype, void *stream) {
    return fwd_entry(x, residual, gamma, eps, out, residual_out, rstd, M, N, dtype, stream, true);
}

rn_status rn_bwd_workspace_bytes(int64_t M, int64_t N, int dtype, size_t *bytes) {
    g_err[0] = 0;
    rn_status st = check_common(M, N, dtype);
    if (st != RN_OK) return st;
    if (!bytes) return fail(RN_ERR_INVALID_ARG, "bytes is NULL");
    DeviceInfo d;
    cudaError_t e = device_info(&d, nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "device query");
    *bytes = ws_bytes_for(d, N);
    return RN_OK;
}

rn_status rn_rmsnorm_bwd(const void *x, const void *gamma, const void *dy, const float *rstd,
                         void *dx, float *dweight_f32, void *dweight, void *workspace,
                         size_t workspace_bytes, int64_t M, int64_t N, int dtype, void *stream) {
    return bwd_entry(x, gamma, dy, rstd, nullptr, dx, dweight_f32, dweight, workspace,
                     workspace_bytes, M, N, dtype, stream);
}

rn_status rn_fused_add_rmsnorm_bwd(const void *added, const void *gamma, const void *dy,
                                   const float *rstd, const void *dresidual_out, void *dx,
                                   float *dweight_f32, void *dweight, void *workspace,
                                   size_t workspace_bytes, int64_t M, int64_t N, int dtype,
                                   void *stream) {
    return bwd_entry(added, gamma, dy, rstd, dresidual_out, dx, dweight_f32, dweight, workspace,
                     workspace_bytes, M, N, dtype, stream);
}

rn_status rn_layernorm_fwd(const void *x, const void *gamma, const void *beta, float eps, void *y,
                           float *mean, float *rstd, int64_t M, int64_t N, int dtype,
                           void *stream) {
    return ln_fwd_entry(x, gamma, beta, eps, y, mean, rstd, M, N, dtype, stream);
}

rn_status rn_layernorm_bwd_workspace_bytes(int64_t M, int64_t N, int dtype, size_t *bytes) {
    g_err[0] = 0;
    rn_status st = check_common(M, N, dtype);
    if (st != RN_OK) return st;
    if (!bytes) return fail(RN_ERR_INVALID_ARG, "bytes is NULL");
    DeviceInfo d;
    cudaError_t e = device_info(&d, nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "device query");
    *bytes = ln_ws_bytes_for(d, N);
    return RN_OK;
}

rn_status rn_layernorm_bwd(const void *x, const void *gamma, const void *dy, const float *mean,
                           const float *rstd, void *dx, float *dgamma_f32, float *dbeta_f32,
                           void *dgamma, void *dbeta, void *workspace, size_t workspace_bytes,
                           int64_t M, int64_t N, int dtype, void *stream) {
    return ln_bwd_entry(x, gamma, dy, mean, rstd, dx, dgamma_f32, dbeta_f32, dgamma, dbeta,
                        workspace, workspace_bytes, M, N, dtype, stream);
}

}  // extern "C"
