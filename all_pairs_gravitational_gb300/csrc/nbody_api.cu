// nbody_api.cu -- the C ABI: argument checks, the launch planner, per-device
// state, workspace handling and dispatch.  See include/nbody.h for the
// contract of each call.
#include <cfloat>
#include <climits>
#include <cmath>
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "nbody.h"
#include "nbody_internal.h"

namespace {

thread_local int g_last_cuda_error = 0;

nbody_status cuda_fail(cudaError_t e) {
    g_last_cuda_error = static_cast<int>(e);
    return NBODY_ERR_CUDA;
}

// ---------------------------------------------------------------- host checks

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// [a, a + a_bytes) and [b, b + b_bytes) share a byte.
bool overlap2(const void *a, int64_t a_bytes, const void *b, int64_t b_bytes) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a);
    const uintptr_t y = reinterpret_cast<uintptr_t>(b);
    return x < y + static_cast<uintptr_t>(b_bytes) && y < x + static_cast<uintptr_t>(a_bytes);
}

bool overlap(const void *a, const void *b, int64_t bytes) { return overlap2(a, bytes, b, bytes); }

nbody_status check_n(int64_t n) {
    return (n < 0 || n > INT32_MAX) ? NBODY_ERR_INVALID_ARG : NBODY_OK;
}

bool eps2_ok(float eps2) { return std::isfinite(eps2) && eps2 >= NBODY_MIN_EPS2; }

nbody_status check_forces(const float *pm, int64_t n, float eps2, const float *acc) {
    if (check_n(n) != NBODY_OK) return NBODY_ERR_INVALID_ARG;
    if (n == 0) return NBODY_OK;
    if (pm == nullptr || acc == nullptr) return NBODY_ERR_INVALID_ARG;
    if (!eps2_ok(eps2)) return NBODY_ERR_INVALID_ARG;
    if (!aligned16(pm) || !aligned16(acc)) return NBODY_ERR_MISALIGNED;
    if (overlap(pm, acc, 16 * n)) return NBODY_ERR_ALIAS;
    return NBODY_OK;
}

// A caller's workspace: 16-byte aligned, overlapping none of the arrays.
nbody_status check_workspace(const void *ws, size_t bytes,
                             std::initializer_list<std::pair<const void *, int64_t>> arrays) {
    if (bytes == 0 || ws == nullptr) return NBODY_OK;
    if (bytes > static_cast<size_t>(INT64_MAX)) return NBODY_ERR_INVALID_ARG;
    if (!aligned16(ws)) return NBODY_ERR_MISALIGNED;
    for (const auto &a : arrays)
        if (a.first != nullptr && a.second > 0 &&
            overlap2(ws, static_cast<int64_t>(bytes), a.first, a.second))
            return NBODY_ERR_ALIAS;
    return NBODY_OK;
}

// ---------------------------------------------------------------- per-device state

constexpr int kMaxDevices = 64;
constexpr int kMaxVariants = 32;

struct Occupancy {
    const int *tiled;
    const int *cluster;
    const int *sym;
};

struct PlanKey {
    int64_t nt, ns, budget;
    int32_t all_pairs, sm;
    nbody_forces_opts opts;
    bool operator==(const PlanKey &o) const {
        return nt == o.nt && ns == o.ns && budget == o.budget && all_pairs == o.all_pairs &&
               sm == o.sm && std::memcmp(&opts, &o.opts, sizeof(opts)) == 0;
    }
};

constexpr int kPlanCache = 16;

struct DeviceState {
    bool ready = false;
    int sm_count = 0;
    int tiled_occ[kMaxVariants] = {0};
    int cluster_occ[kMaxVariants] = {0};
    int sym_occ[kMaxVariants] = {0};
    cudaMemPool_t pool = nullptr;     // stream-ordered workspace of the pool-based calls
    // recently made plans (planning a large n searches thousands of shapes)
    PlanKey plan_key[kPlanCache];
    nbody_plan plan_val[kPlanCache];
    int plan_count = 0;
    int plan_next = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

nbody_status current_device(int *dev) {
    const cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (*dev < 0 || *dev >= kMaxDevices) return NBODY_ERR_DEVICE;
    return NBODY_OK;
}

nbody_status device_state(DeviceState **out) {
    int dev = 0;
    nbody_status st = current_device(&dev);
    if (st != NBODY_OK) return st;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &d = g_dev[dev];
    if (!d.ready) {
        cudaError_t e;
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e);
        if (major != 10 || minor != 3) return NBODY_ERR_DEVICE;   // built for sm_103a only
        for (int v = 0; v < nbody::tiled_variant_count() && v < kMaxVariants; ++v) {
            const nbody::TiledVariant &tv = nbody::tiled_variant(v);
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.tiled_occ[v], tv.fn_pot,
                                                              tv.threads, 0);
            if (e != cudaSuccess) return cuda_fail(e);
        }
        for (int v = 0; v < nbody::cluster_variant_count() && v < kMaxVariants; ++v) {
            const nbody::ClusterVariant &cv = nbody::cluster_variant(v);
            if (cv.whole) {
                for (const void *fn : {cv.fn_pot, cv.fn_acc})
                    if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  static_cast<int>(nbody::kWholeSmemMax))) != cudaSuccess)
                        return cuda_fail(e);
            }
            // register-limited residency (whole-range launches are further
            // limited by their shared memory, see plan_cluster_variant)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.cluster_occ[v], cv.fn_pot,
                                                              cv.warps * 32, 0);
            if (e != cudaSuccess) return cuda_fail(e);
        }
        for (int v = 0; v < nbody::sym_variant_count() && v < kMaxVariants; ++v) {
            const nbody::SymVariant &sv = nbody::sym_variant(v);
            for (const void *fn : {sv.fn_pot, sv.fn_acc})
                if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(sv.smem))) != cudaSuccess)
                    return cuda_fail(e);
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.sym_occ[v], sv.fn_pot,
                                                              sv.warps * 32, sv.smem);
            if (e != cudaSuccess) return cuda_fail(e);
        }
        for (int v = 0; v < nbody::rows_variant_count(); ++v) {
            const nbody::RowsVariant &rv = nbody::rows_variant(v);
            for (const void *fn : {rv.fn_pot, rv.fn_acc, rv.fn_pot_euler, rv.fn_acc_euler})
                if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(nbody::kRowsSmemMax))) != cudaSuccess)
                    return cuda_fail(e);
        }
        d.ready = true;
    }
    *out = &d;
    return NBODY_OK;
}

// The device's workspace pool, created on first use.  Freed blocks above
// NBODY_POOL_KEEP_BYTES go back to the system at each synchronisation.
nbody_status device_pool(DeviceState *d, cudaMemPool_t *pool) {
    int dev = 0;
    nbody_status st = current_device(&dev);
    if (st != NBODY_OK) return st;
    std::lock_guard<std::mutex> lock(g_mu);
    if (d->pool == nullptr) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t p = nullptr;
        cudaError_t e = cudaMemPoolCreate(&p, &props);
        if (e != cudaSuccess) return cuda_fail(e);
        uint64_t keep = static_cast<uint64_t>(NBODY_POOL_KEEP_BYTES);
        if ((e = cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess) {
            cudaMemPoolDestroy(p);
            return cuda_fail(e);
        }
        d->pool = p;
    }
    *pool = d->pool;
    return NBODY_OK;
}

// ---------------------------------------------------------------- planner
//
// A plan has two layers.  The decomposition -- the path, the kernel shape,
// the pieces of each source range and (symmetric path) the groups of
// distances -- depends only on n, the device and the options, and fixes
// every partial sum and the order they are added in.  The execution -- how
// many groups each force launch takes -- follows from the workspace: one
// pass when all partials fit, otherwise passes of as many groups as fit,
// with the running compensated total carried between passes exactly.  A
// workspace too small for one group of the decomposition falls back to a
// decomposition without partials.

constexpr int kDefaultTiledVariant = 0;
constexpr int kCompensatedTiledVariant = 7;
constexpr int kMaxSplits = 1024;
constexpr int64_t kDesignBudget = NBODY_DEFAULT_WORKSPACE_BYTES;
// Relative cost model (only ratios matter): pair rate of one SM, the fixed
// cost of a work item in source-body equivalents, one launch, scratch traffic.
constexpr double kPairsPerSmSecond = 1.4e10;
constexpr int kItemOverheadBodies = 96;
constexpr double kLaunchSeconds = 2.5e-6;
constexpr double kScratchBytesPerSecond = 5.0e12;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Workspace of the pool-based calls: the default budget, or where n is so
// large that one group of symmetric partials exceeds it (n above about 20
// million), the least workspace any symmetric plan needs (3 partial arrays).
int64_t pool_budget(int64_t n) { return std::max<int64_t>(kDesignBudget, 48 * n); }

// Groups per pass for `groups` groups of `per_group` bytes each within
// `budget`: all in one pass, or passes plus one carry slot of `carry` bytes.
// Returns 0 if not even one group fits.
int64_t groups_per_pass(int64_t groups, int64_t per_group, int64_t carry, int64_t budget) {
    if (groups * per_group <= budget) return groups;
    const int64_t g = (budget - carry) / per_group;
    return g < 1 ? 0 : std::min(g, groups);
}

int64_t pass_bytes(int64_t groups, int64_t gpp, int64_t per_group, int64_t carry) {
    return gpp >= groups ? groups * per_group : gpp * per_group + carry;
}

bool plan_tiled(int64_t nt, int64_t ns, int sm, int occ, int variant, int splits_req,
                int64_t budget, nbody_plan *p) {
    const nbody::TiledVariant &v = nbody::tiled_variant(variant);
    const int64_t bi = static_cast<int64_t>(v.threads) * v.i_per_thread;
    const int64_t num_ib = ceil_div(nt, bi);
    const int64_t ntiles = ceil_div(ns, v.tile);
    const int64_t slots = static_cast<int64_t>(sm > 0 ? sm : 1) * (occ > 0 ? occ : 1);
    const double slot_rate = kPairsPerSmSecond / (occ > 0 ? occ : 1);
    const int64_t rec = 16 * nt;   // one partial array

    // decomposition: pieces S within the design budget
    int64_t s_lo = 1, s_hi = std::min<int64_t>(ntiles, kMaxSplits);
    s_hi = std::max<int64_t>(1, std::min<int64_t>(s_hi, kDesignBudget / rec));
    if (splits_req > 0) s_lo = s_hi = std::min<int64_t>(splits_req, ntiles);
    double best_t = INFINITY;
    int64_t best_s = 1, best_tps = ntiles;
    for (int64_t s = s_lo; s <= s_hi; ++s) {
        const int64_t tps = ceil_div(ntiles, s);
        const int64_t used = ceil_div(ntiles, tps);
        if (used != s && splits_req <= 0) continue;   // same as a smaller S
        const int64_t waves = ceil_div(num_ib * used, slots);
        double t = static_cast<double>(waves) *
                   static_cast<double>(tps * v.tile + kItemOverheadBodies) * bi / slot_rate;
        if (used > 1) t += kLaunchSeconds + 32.0 * used * nt / kScratchBytesPerSecond;
        if (t < best_t * (1.0 - 1e-3)) {
            best_t = t;
            best_s = used;
            best_tps = tps;
        }
    }
    // execution within the workspace
    int64_t gpp = 1;
    if (best_s > 1) {
        gpp = groups_per_pass(best_s, rec, rec, budget);
        if (gpp == 0) {   // not even one piece and the carry: no partials
            best_s = 1;
            best_tps = ntiles;
            gpp = 1;
        }
    }
    const int64_t passes = ceil_div(best_s, gpp);
    const int64_t waves = ceil_div(num_ib * gpp, slots);
    p->path = NBODY_PATH_TILED;
    p->variant = variant;
    p->i_per_thread = v.i_per_thread;
    p->threads = v.threads;
    p->tile = v.tile;
    p->num_iblocks = static_cast<int32_t>(num_ib);
    p->splits = static_cast<int32_t>(best_s);
    p->tiles_per_split = static_cast<int32_t>(best_tps);
    p->cluster = 1;
    p->warps_j = 1;
    p->dists = 0;
    p->groups = static_cast<int32_t>(best_s);
    p->groups_per_pass = static_cast<int32_t>(gpp);
    p->passes = static_cast<int32_t>(passes);
    p->grid = num_ib * gpp;
    p->scratch_bytes = best_s > 1 ? pass_bytes(best_s, gpp, rec, rec) : 0;
    p->scratch_min_bytes = best_s > 1 ? std::min<int64_t>(best_s, 2) * rec : 0;
    p->fill = static_cast<double>(num_ib * gpp) / static_cast<double>(waves * slots);
    return true;
}

// Small-N path: a cluster of C CTAs (C in 1, 2, 4, 8) shares 32 K targets;
// each CTA has W warps.  Cost model: the busiest SM holds ceil(CTAs / SMs)
// CTAs (waves beyond the occupancy limit are counted), and an SM reaches its
// full pair rate with kWarpsToSaturate resident warps.
constexpr int kWarpsToSaturate = 16;
// Cost of one CTA-wide barrier of the tiled cluster kernel, in source bodies.
constexpr int kTileBarrierBodies = 32;
// Shared memory of one SM available to resident CTAs (sm_103: 228 KB, 1 KB
// reserved per CTA).
constexpr int64_t kSmemPerSm = 228 * 1024;
void plan_cluster_variant(int64_t nt, int64_t ns, int sm, int occ, int variant, nbody_plan *p,
                          double *t_out) {
    const nbody::ClusterVariant &v = nbody::cluster_variant(variant);
    const int64_t bi = 32LL * v.i_per_thread;
    const int64_t num_ib = ceil_div(nt, bi);
    const int64_t ntiles = ceil_div(ns, v.tile);
    double best_t = INFINITY;
    int64_t best_c = 1, best_tpc = ntiles;
    double best_fill = 0.0;
    for (int64_t c = 1; c <= 8; c *= 2) {
        if (c > ntiles) break;
        const int64_t tpc = ceil_div(ntiles, c);
        int64_t occ_c = occ > 0 ? occ : 1;
        if (v.whole) {
            const int64_t smem = static_cast<int64_t>(
                nbody::whole_smem_bytes(v.i_per_thread, v.warps, static_cast<int>(tpc)));
            if (smem > static_cast<int64_t>(nbody::kWholeSmemMax)) continue;
            occ_c = std::min<int64_t>(occ_c, kSmemPerSm / (smem + 1024));
            if (occ_c < 1) continue;
        }
        const int64_t ctas = num_ib * c;
        const int64_t per_sm = ceil_div(ctas, sm);
        const int64_t resident = std::min<int64_t>(per_sm, occ_c);
        const int64_t waves = ceil_div(per_sm, resident);
        const double rate = kPairsPerSmSecond *
                            std::min(1.0, static_cast<double>(resident * v.warps) / kWarpsToSaturate);
        const int64_t barrier_bodies = v.whole ? kTileBarrierBodies : tpc * kTileBarrierBodies;
        const double cta_pairs =
            static_cast<double>(tpc * v.tile + kItemOverheadBodies + barrier_bodies) * bi;
        const double t = waves * resident * cta_pairs / rate + 0.2e-6 * (c > 1);
        if (t < best_t * (1.0 - 1e-3)) {
            best_t = t;
            best_c = c;
            best_tpc = tpc;
            best_fill = static_cast<double>(ctas) / static_cast<double>(waves * resident * sm);
        }
    }
    if (!std::isfinite(best_t)) {   // no cluster size fits this variant's shared memory
        *t_out = INFINITY;
        return;
    }
    p->path = NBODY_PATH_CLUSTER;
    p->variant = variant;
    p->i_per_thread = v.i_per_thread;
    p->threads = v.warps * 32;
    p->tile = v.tile;
    p->num_iblocks = static_cast<int32_t>(num_ib);
    p->splits = static_cast<int32_t>(best_c * v.warps);
    p->tiles_per_split = static_cast<int32_t>(best_tpc);
    p->cluster = static_cast<int32_t>(best_c);
    p->warps_j = v.warps;
    p->dists = 0;
    p->groups = 1;
    p->groups_per_pass = 1;
    p->passes = 1;
    p->grid = num_ib * best_c;
    p->scratch_bytes = 0;
    p->scratch_min_bytes = 0;
    p->fill = best_fill > 1.0 ? 1.0 : best_fill;
    *t_out = best_t;
}

// The cluster variant a forced cluster-path call takes by size (the
// automatic choice sends small calls to the row-split path instead).
// Measured on GB300 inside CUDA graphs (force call, microseconds) over
// variants 0 (K = 2, 4 warps, 128-body tiles), 6 (K = 2, 8 warps, whole
// range staged) and 7 (K = 4, 8 warps, whole range); the times jump with
// the integer counts of target blocks, cluster sizes and waves, so the
// choice is a table of the measured best:
//   n:      2048  2560  3072  3584  4096  4352  4608  4864  5120  5376  5632  6144
//   v0:     4.81  8.20  8.33 12.66 12.74 15.26 15.25 26.52 25.64 31.27 31.02 31.63
//   v6:     5.01  8.98 10.40 12.80 12.97 14.36 14.36 27.56 27.61 30.27 30.28 25.71
//   v7:     6.87  9.47  9.48 11.67 11.66 14.05 16.53 20.04 25.29 27.64 27.72 29.91
// (1024 bodies: variant 0, 3.2 us.)
int auto_cluster_variant(int64_t n) {
    if (n <= 3072) return 0;
    if (n <= 4352) return 7;
    if (n <= 4608) return 6;
    return 7;
}

// Row-split path (few sources): CTA b takes targets [b tb, (b + 1) tb) with
// tb = ceil(nt / SMs), so every SM gets the same share of the pairs; its
// warp items are K targets against one of S pieces of the sources, a piece
// holding at most kRowsPieceMax sources.  Cost model, in units of one
// target's 32-column step at the FMA pipe's rate: item `it` runs on warp
// it mod W, whose scheduler is it mod 4 (W is a multiple of 4), so the
// busiest scheduler runs ceil(items / 4) items of K x (steps + the row
// sums' shuffle tree, about kRowsTreeSteps steps) each; and a warp runs
// ceil(items / W) items one after another, each step at least one
// dependency chain long (kRowsStepLatency units), which sets the time when
// few items share a scheduler.  S is the cheapest count by that model, the
// fewest on a tie.
constexpr int64_t kRowsPieceMax = 2048;
// The automatic choice takes the row-split path when both the targets and
// the sources number fewer than this (from 10240 all-pairs bodies the
// symmetric path is as fast: 50.7 against 50.5 us at 10240, 69.7 against
// 70.6 us at 12288).  Against the tiled and cluster paths, measured inside
// CUDA graphs on GB300 (force call, us):
//   n:         1024  2048  3072  4096  4864  6144  8192
//   row-split: 2.54  3.99  6.80  9.35 13.29 19.36 31.42
//   before:    3.19  4.85  8.28 11.66 20.08 24.17 38.65   (cluster to 4864, then tiled)
constexpr int64_t kRowsMaxAutoN = 10240;
// Target/source calls (separate arrays) with fewer than kRowsMaxAutoN sources
// take the row-split path up to this many targets, if its piece sums fit in
// shared memory: measured against the tiled path (us), 20000 x 1000 sources:
// 12.7 against 21.5; 100000 x 2000: 90.7 / 101.3; 131072 x 2000: 117.4 /
// 133.2; 150000 x 4000: 263.1 / 262.2; 1000000 x 1000: 465.0 / 423.8.
constexpr int64_t kRowsMaxAutoTargets = 131072;
constexpr double kRowsTreeSteps = 2.5;
constexpr double kRowsStepLatency = 2.3;
constexpr int64_t kRowsMaxPieces = 64;

bool plan_rows(int64_t nt, int64_t ns, int sm, int variant, int forced_pieces, nbody_plan *p,
               double *t_out = nullptr) {
    const nbody::RowsVariant &v = nbody::rows_variant(variant);
    const int64_t K = v.i_per_warp;
    const int64_t tb = ceil_div(nt, sm);
    const int64_t grid = ceil_div(nt, tb);
    const int64_t groups = ceil_div(tb, K);
    const int64_t s_lo = forced_pieces > 0 ? forced_pieces
                                           : std::max<int64_t>(1, ceil_div(ns, kRowsPieceMax));
    const int64_t s_hi = forced_pieces > 0 ? forced_pieces : std::max(s_lo, kRowsMaxPieces);
    double best_t = INFINITY;
    int64_t best_s = 0, best_cols = 0;
    for (int64_t s = s_lo; s <= s_hi; ++s) {
        const int64_t cols = ceil_div(ns, 64 * s) * 32;
        const int64_t ns_pad = 2 * s * cols;
        if (ns_pad > INT32_MAX || groups * K * s > INT32_MAX ||
            nbody::rows_smem_bytes(static_cast<int>(ns_pad), static_cast<int>(s),
                                   static_cast<int>(groups * K)) > nbody::kRowsSmemMax)
            continue;
        const double steps = static_cast<double>(cols / 32);
        const double t =
            static_cast<double>(ceil_div(groups * s, 4)) * static_cast<double>(K) *
                (steps + kRowsTreeSteps) +
            static_cast<double>(ceil_div(groups * s, v.warps)) * steps * kRowsStepLatency;
        if (t < best_t * (1.0 - 1e-9)) {
            best_t = t;
            best_s = s;
            best_cols = cols;
        }
    }
    if (best_s == 0) return false;   // the sources (or the piece sums) exceed shared memory
    if (t_out != nullptr) *t_out = best_t;
    const int64_t items = groups * best_s;
    p->path = NBODY_PATH_ROWS;
    p->variant = variant;
    p->i_per_thread = static_cast<int32_t>(K);
    p->threads = v.warps * 32;
    p->tile = static_cast<int32_t>(2 * best_cols);
    p->num_iblocks = static_cast<int32_t>(grid);
    p->splits = static_cast<int32_t>(best_s);
    p->tiles_per_split = static_cast<int32_t>(tb);
    p->cluster = 1;
    p->warps_j = v.warps;
    p->dists = 0;
    p->groups = 1;
    p->groups_per_pass = 1;
    p->passes = 1;
    p->grid = grid;
    p->scratch_bytes = 0;
    p->scratch_min_bytes = 0;
    // useful pairs over the pair slots of the busiest schedulers
    p->fill = static_cast<double>(nt) * static_cast<double>(ns) /
              (static_cast<double>(sm) * 4.0 * static_cast<double>(ceil_div(items, 4)) *
               static_cast<double>(K) * static_cast<double>(2 * best_cols));
    return true;
}

// The automatic row-split plan: the variant (K targets per item: 7, 6, or 4
// with 12 warps) with the cheapest modelled time, the first on a tie.
// Measured on GB300 inside CUDA graphs (force call, us), the model picks
// the fastest of the three at every size measured:
//   n:       1024  2048  3072  4096  4864  6144  8192 10239
//   K = 7:   2.59  4.11  6.98  9.51 14.46 19.60 32.42 51.37
//   K = 6:   2.95  5.26  7.24 11.58 15.12 21.36 33.92 54.38
//   K = 4:   2.79  4.92  7.11 10.91 12.99 20.77 33.41 51.42
bool plan_rows_auto(int64_t nt, int64_t ns, int sm, int forced_pieces, nbody_plan *p) {
    double best_t = INFINITY;
    bool found = false;
    for (int v : {0, 1, 2}) {
        nbody_plan q = {};
        double t = INFINITY;
        if (plan_rows(nt, ns, sm, v, forced_pieces, &q, &t) && t < best_t * (1.0 - 1e-9)) {
            best_t = t;
            *p = q;
            found = true;
        }
    }
    return found;
}

// The kernel-side decomposition of a row-split plan.
nbody::RowsLaunch rows_launch(const nbody_plan &plan) {
    nbody::RowsLaunch rl;
    rl.tb = plan.tiles_per_split;
    rl.groups = (plan.tiles_per_split + plan.i_per_thread - 1) / plan.i_per_thread;
    rl.tb_pad = rl.groups * plan.i_per_thread;
    rl.pieces = plan.splits;
    rl.cols = plan.tile / 2;
    rl.ns_pad = plan.splits * plan.tile;
    return rl;
}

// Symmetric path (each unordered pair once).  Smallest n the automatic choice
// sends to it, and the variant it takes by size, measured on GB300 inside
// CUDA graphs: from 10240 bodies every shape below beats the tiled path
// (54.5 against 57.6 us at 10240; 221 against 264 us at 24576), 512-body
// blocks win up to about 45K bodies (better filled waves), 1024-body blocks
// (with the finer pieces below) up to about 330K, and 2048-body blocks above
// (fewer partial slots): 1024 against 2048, ms: 163840 bodies 8.21 / 8.39,
// 262144 20.85 / 21.09, 393216 46.96 / 47.10, 524288 83.83 / 83.68, 2^20
// 335.8 / 334.3.  Each choice is within 4.5 % of the fastest shape at every
// size measured.
constexpr int64_t kSymMinN = 10240;
constexpr int64_t kSymMidN = 45056;     // from here 1024-body blocks
constexpr int64_t kSymLargeN = 327680;  // from here 2048-body blocks
constexpr int64_t kSymFinerMinN = 16384; // finer pieces for the smaller blocks from here
constexpr int kSymSmallVariant = 2;     // K = 8, 2 warps: 512-body blocks
constexpr int kSymMidVariant = 1;       // K = 8, 4 warps: 1024-body blocks
constexpr int kDefaultSymVariant = 0;   // K = 8, 8 warps: 2048-body blocks
// Relative cost model of the symmetric path: evaluations (two interactions
// each) per SM-second, the fixed cost of a CTA in evaluations.
constexpr double kSymEvalsPerSmSecond = 1.1e10;
constexpr double kSymItemOverheadEvals = 64.0 * 1024.0;

struct SymGeometry {
    int64_t block, nb, ndist, spb;
};

SymGeometry sym_geometry(const nbody::SymVariant &v, int64_t n) {
    SymGeometry g;
    g.block = 32LL * v.warps * v.i_per_thread;
    g.nb = ceil_div(n, g.block);
    g.ndist = nbody::sym_ndist(static_cast<int>(g.nb));
    g.spb = g.block / v.sub;
    return g;
}

// Modelled time of the symmetric decomposition (P pieces, D distances per
// group) run in passes of gpp groups.
double sym_time(const SymGeometry &g, int64_t n, const nbody::SymVariant &v, int64_t slots,
                double slot_rate, int64_t P, int64_t D, int64_t js, int64_t gpp) {
    const int64_t groups = ceil_div(g.ndist, D);
    const bool reduce = !(g.nb == 1 && P == 1);
    const int64_t passes = ceil_div(groups, gpp);
    const double unit_evals = static_cast<double>(g.block) * v.sub;
    auto pass_time = [&](int64_t gp, int64_t dists_last, bool carry_in, bool carry_out) {
        const int64_t waves = ceil_div(g.nb * P * gp, slots);
        // the largest piece: D distances (dists_last in a pass of the last group alone)
        const int64_t d_big = gp > 1 ? D : dists_last;
        const int64_t upp = ceil_div(d_big * g.spb, P);
        double t = static_cast<double>(waves) * (upp * unit_evals + kSymItemOverheadEvals) / slot_rate +
                   kLaunchSeconds;
        if (reduce) {
            const double recs = static_cast<double>(gp * (P + js)) + 1.0 + (carry_in ? 2.0 : 0.0) +
                                (carry_out ? 1.0 : 0.0);
            t += kLaunchSeconds + 16.0 * recs * n / kScratchBytesPerSecond;
        }
        return t;
    };
    const int64_t last_groups = groups - (passes - 1) * gpp;
    const int64_t dists_last = g.ndist - (groups - 1) * D;
    double t = 0.0;
    if (passes > 1) {
        t += pass_time(gpp, D, false, true);                       // first
        if (passes > 2) t += (passes - 2) * pass_time(gpp, D, true, true);
        t += pass_time(last_groups, last_groups > 1 ? D : dists_last, true, false);
    } else {
        t = pass_time(groups, groups > 1 ? D : dists_last, false, false);
    }
    return t;
}

// Returns false if the decomposition cannot run within `budget` (a workspace
// smaller than one group and its carry slot).
bool plan_sym(int64_t n, int sm, int occ, int variant, int splits_req, int dists_req,
              int64_t budget, nbody_plan *p) {
    const nbody::SymVariant &v = nbody::sym_variant(variant);
    const SymGeometry g = sym_geometry(v, n);
    const int64_t slots = static_cast<int64_t>(sm > 0 ? sm : 1) * (occ > 0 ? occ : 1);
    const double slot_rate = kSymEvalsPerSmSecond / (occ > 0 ? occ : 1);
    const int64_t rec = 16 * n;
    // the decomposition is chosen within the design budget (or the least
    // workspace any decomposition needs, for very large n)
    const int64_t design = pool_budget(n);
    const int64_t grid_cap = INT32_MAX;

    // distances per group: those giving distinct group counts
    int64_t dcand[4096];
    int nd = 0;
    if (dists_req > 0) {
        dcand[nd++] = std::min<int64_t>(dists_req, g.ndist);
    } else {
        int64_t last = -1;
        for (int64_t k = 1; k <= g.ndist && nd < 4096; ++k) {
            const int64_t D = ceil_div(g.ndist, k);
            if (D != last) dcand[nd++] = D;
            last = D;
            if (D == 1) break;
        }
    }
    double best_t = INFINITY;
    int64_t best_p = 0, best_d = 0;
    int64_t p_hi_req = splits_req > 0 ? splits_req : 0;
    for (;;) {
        for (int c = 0; c < nd; ++c) {
            const int64_t D = dcand[c];
            const int64_t groups = ceil_div(g.ndist, D);
            const int64_t js = nbody::sym_group_jslots(static_cast<int>(g.nb), static_cast<int>(D));
            const int64_t p_max = std::max<int64_t>(1, std::min<int64_t>(kMaxSplits, D * g.spb));
            const int64_t lo = p_hi_req > 0 ? std::min(p_hi_req, p_max) : 1;
            const int64_t hi = p_hi_req > 0 ? lo : p_max;
            for (int64_t P = lo; P <= hi; ++P) {
                const bool reduce = !(g.nb == 1 && P == 1);
                const int64_t per_group = (P + js) * rec;
                const int64_t gpp = reduce ? groups_per_pass(groups, per_group, rec, design) : groups;
                if (gpp == 0 || g.nb * P * gpp > grid_cap) continue;
                const double t = sym_time(g, n, v, slots, slot_rate, P, D, js, gpp);
                if (t < best_t * (1.0 - 1e-4)) {
                    best_t = t;
                    best_p = P;
                    best_d = D;
                }
            }
        }
        if (best_p > 0 || p_hi_req <= 1) break;
        p_hi_req = p_hi_req / 2;   // a forced piece count too large for the design budget
    }
    if (best_p == 0) return false;

    // Finer pieces for the 512- and 1024-body blocks from kSymFinerMinN
    // bodies, in one pass: the wave model above counts whole waves, but
    // several waves of smaller CTAs balance better across the SMs.
    // Measured on GB300 (force call, us, model P -> 2P -> 3P):
    //   16384: 115.4 / 112.1 / 125.9 (3P leaves pieces of 1 and 2 units)
    //   20000: 168.3 / 160.4 / 157.2      45056: 750.9 / 715.8 / 697.5
    //   65536: 1398 / 1365 / 1357        100000: 3469 / 3328 / 3268
    //  163839: 8310 / 8232 / 8212   (2048-body blocks: +-0.5 %)
    // so 3P where the pieces stay within 10 % of equal, else 2P.
    if (splits_req <= 0 && variant != kDefaultSymVariant && n >= kSymFinerMinN) {
        const int64_t groups0 = ceil_div(g.ndist, best_d);
        const int64_t js0 = nbody::sym_group_jslots(static_cast<int>(g.nb), static_cast<int>(best_d));
        const int64_t units = std::min<int64_t>(best_d, g.ndist) * g.spb;   // of the largest group
        for (int64_t k : {3, 2}) {
            const int64_t P2 = k * best_p;
            if (P2 > std::min<int64_t>(kMaxSplits, units)) continue;
            if (static_cast<double>(ceil_div(units, P2) * P2) > 1.1 * static_cast<double>(units))
                continue;
            if (groups0 * (P2 + js0) * rec > design || g.nb * P2 * groups0 > grid_cap) continue;
            best_p = P2;
            break;
        }
    }

    // execution within the workspace
    const int64_t P = best_p, D = best_d;
    const int64_t groups = ceil_div(g.ndist, D);
    const int64_t js = nbody::sym_group_jslots(static_cast<int>(g.nb), static_cast<int>(D));
    const bool reduce = !(g.nb == 1 && P == 1);
    const int64_t per_group = (P + js) * rec;
    int64_t gpp = groups;
    if (reduce) {
        gpp = groups_per_pass(groups, per_group, rec, budget);
        if (gpp == 0) return false;
        while (g.nb * P * gpp > grid_cap) --gpp;
    }
    const int64_t passes = ceil_div(groups, gpp);
    const int64_t waves = ceil_div(g.nb * P * gpp, slots);
    p->path = NBODY_PATH_SYMMETRIC;
    p->variant = variant;
    p->i_per_thread = v.i_per_thread;
    p->threads = v.warps * 32;
    p->tile = v.sub;
    p->num_iblocks = static_cast<int32_t>(g.nb);
    p->splits = static_cast<int32_t>(P);
    p->tiles_per_split = static_cast<int32_t>(ceil_div(std::min<int64_t>(D, g.ndist) * g.spb, P));
    p->cluster = 1;
    p->warps_j = 1;
    p->dists = static_cast<int32_t>(D);
    p->groups = static_cast<int32_t>(groups);
    p->groups_per_pass = static_cast<int32_t>(gpp);
    p->passes = static_cast<int32_t>(passes);
    p->grid = g.nb * P * gpp;
    p->scratch_bytes = reduce ? pass_bytes(groups, gpp, per_group, rec) : 0;
    p->scratch_min_bytes = reduce ? std::min<int64_t>(groups * per_group, per_group + rec) : 0;
    p->fill = static_cast<double>(g.nb * P * gpp) / static_cast<double>(waves * slots);
    return true;
}

// Tiled variant for all-pairs calls below the symmetric path, measured on
// GB300 inside CUDA graphs (force call, microseconds): variant 0 (K = 4, 256
// threads: 1024-target blocks) against variant 6 (K = 2, 256 threads,
// two sources per step: 512-target blocks),
//   n:     5120  6144  7168  8192  9216 10239 12288
//   v0:    23.2  24.2  38.0  38.6  53.8  55.2  70.3
//   v6:    19.9  25.2  31.9  40.5  44.7  58.4  74.5
// The smaller blocks win when the count of 1024-target blocks is odd (the
// pieces then fill the waves worse), so that is the rule.
constexpr int kSmallTiledVariant = 6;

int auto_tiled_variant(int64_t nt, int64_t ns, bool all_pairs) {
    if (all_pairs && nt == ns && nt < kSymMinN && (ceil_div(nt, 1024) & 1))
        return kSmallTiledVariant;
    return kDefaultTiledVariant;
}

int auto_sym_variant(int64_t n) {
    return n < kSymMidN ? kSymSmallVariant : (n < kSymLargeN ? kSymMidVariant : kDefaultSymVariant);
}

nbody_status make_plan_uncached(int64_t nt, int64_t ns, bool all_pairs, int sm,
                                const Occupancy &occ, const nbody_forces_opts &o_in,
                                int64_t budget, nbody_plan *p) {
    nbody_forces_opts o = o_in;
    if (o.precision == NBODY_PRECISION_COMPENSATED) {   // the tiled path's compensated kernel
        if (o.path == NBODY_PATH_CLUSTER || o.path == NBODY_PATH_SYMMETRIC ||
            o.path == NBODY_PATH_ROWS ||
            (o.variant >= 0 && o.variant != kCompensatedTiledVariant))
            return NBODY_ERR_INVALID_ARG;
        o.path = NBODY_PATH_TILED;
        o.variant = kCompensatedTiledVariant;
    }
    all_pairs = all_pairs && nt == ns;
    if (o.path == NBODY_PATH_SYMMETRIC && !all_pairs) return NBODY_ERR_INVALID_ARG;
    if (o.dists != 0 && o.path != NBODY_PATH_SYMMETRIC && o.path != NBODY_PATH_AUTO)
        return NBODY_ERR_INVALID_ARG;
    int path = o.path;
    bool auto_rows = false;
    if (path == NBODY_PATH_AUTO) {
        if (ns < kRowsMaxAutoN &&
            (nt < kRowsMaxAutoN || (!all_pairs && nt <= kRowsMaxAutoTargets))) {
            path = NBODY_PATH_ROWS;   // a forced variant is the row-split path's
            auto_rows = true;
        } else if (all_pairs && nt >= kSymMinN &&
                   plan_sym(nt, sm, occ.sym[auto_sym_variant(nt)], auto_sym_variant(nt), o.splits,
                            o.dists, budget, p)) {
            return NBODY_OK;
        } else {
            path = NBODY_PATH_TILED;
        }
    }
    if (path == NBODY_PATH_SYMMETRIC) {
        const int variant = o.variant < 0 ? auto_sym_variant(nt) : o.variant;
        if (variant >= nbody::sym_variant_count() || variant >= kMaxVariants)
            return NBODY_ERR_INVALID_ARG;
        return plan_sym(nt, sm, occ.sym[variant], variant, o.splits, o.dists, budget, p)
                   ? NBODY_OK
                   : NBODY_ERR_WORKSPACE;
    }
    if (path == NBODY_PATH_ROWS) {
        if (o.variant >= nbody::rows_variant_count()) return NBODY_ERR_INVALID_ARG;
        const bool ok = o.variant < 0 ? plan_rows_auto(nt, ns, sm, o.splits, p)
                                      : plan_rows(nt, ns, sm, o.variant, o.splits, p);
        if (ok) return NBODY_OK;
        // the sources or the piece sums do not fit shared memory: a forced
        // path is an error, the automatic choice takes the tiled path
        if (!auto_rows || o.variant >= 0 || o.splits != 0) return NBODY_ERR_INVALID_ARG;
        path = NBODY_PATH_TILED;
    }
    if (path == NBODY_PATH_TILED) {
        const int variant = o.variant < 0 ? auto_tiled_variant(nt, ns, all_pairs) : o.variant;
        if (variant >= nbody::tiled_variant_count() || variant >= kMaxVariants)
            return NBODY_ERR_INVALID_ARG;
        plan_tiled(nt, ns, sm, occ.tiled[variant], variant, o.splits, budget, p);
        return NBODY_OK;
    }
    if (o.splits != 0) return NBODY_ERR_INVALID_ARG;   // the cluster path plans its own split
    if (o.variant >= nbody::cluster_variant_count()) return NBODY_ERR_INVALID_ARG;
    // The cost model picks the cluster size well but ranks the kernel
    // variants poorly, so automatic planning takes the variant from the
    // measured table above; a forced variant is honoured.
    const int only = o.variant >= 0 ? o.variant : auto_cluster_variant(std::max(nt, ns));
    double t = INFINITY;
    plan_cluster_variant(nt, ns, sm, occ.cluster[only], only, p, &t);
    // a forced whole-range variant whose range cannot fit shared memory
    return std::isfinite(t) ? NBODY_OK : NBODY_ERR_INVALID_ARG;
}

// all_pairs: the targets are the sources (same array, nt == ns), the case the
// symmetric path needs.  `budget`: workspace bytes the plan may use.
nbody_status make_plan(int64_t nt, int64_t ns, bool all_pairs, int sm, const Occupancy &occ,
                       const nbody_forces_opts *opts, int64_t budget, nbody_plan *p,
                       DeviceState *cache = nullptr) {
    if (nt <= 0 || nt > INT32_MAX || ns <= 0 || ns > INT32_MAX || sm <= 0 || p == nullptr ||
        budget < 0)
        return NBODY_ERR_INVALID_ARG;
    nbody_forces_opts o = {NBODY_PATH_AUTO, -1, 0, NBODY_PRECISION_DEFAULT,
                           NBODY_QUANTITIES_ACC_POT, 0};
    if (opts != nullptr) o = *opts;
    if (o.path < NBODY_PATH_AUTO || o.path > NBODY_PATH_ROWS || o.splits < 0 || o.dists < 0)
        return NBODY_ERR_INVALID_ARG;
    if (o.precision < 0 || o.precision > 1) return NBODY_ERR_INVALID_ARG;
    if (o.quantities < 0 || o.quantities > 1) return NBODY_ERR_INVALID_ARG;
    const PlanKey key = {nt, ns, budget, all_pairs ? 1 : 0, sm, o};
    if (cache != nullptr) {
        std::lock_guard<std::mutex> lock(g_mu);
        for (int k = 0; k < cache->plan_count; ++k)
            if (cache->plan_key[k] == key) {
                *p = cache->plan_val[k];
                return NBODY_OK;
            }
    }
    nbody_plan plan = {};
    const nbody_status st = make_plan_uncached(nt, ns, all_pairs, sm, occ, o, budget, &plan);
    if (st != NBODY_OK) return st;
    *p = plan;
    if (cache != nullptr) {
        std::lock_guard<std::mutex> lock(g_mu);
        cache->plan_key[cache->plan_next] = key;
        cache->plan_val[cache->plan_next] = plan;
        cache->plan_next = (cache->plan_next + 1) % kPlanCache;
        cache->plan_count = std::min(cache->plan_count + 1, kPlanCache);
    }
    return NBODY_OK;
}

// ---------------------------------------------------------------- launching

// Launch a planned force evaluation.  `ws` holds plan.scratch_bytes when that
// is not 0.  With `eu`, the Euler update is applied to every body as its
// final result is formed when the plan ends in a reduction kernel; *fused
// tells whether that happened (otherwise the caller launches the update).
cudaError_t launch_planned(const nbody_plan &plan, const nbody::Problem &pr, float4 *out,
                           void *ws, int sm_count, cudaStream_t stream,
                           const nbody::EulerFuse *eu = nullptr, bool *fused = nullptr) {
    if (fused != nullptr) *fused = false;
    float4 *parts = static_cast<float4 *>(ws);
    const int64_t nt = pr.nt;
    if (plan.path == NBODY_PATH_SYMMETRIC) {
        nbody::SymLaunch sl = {plan.num_iblocks, plan.splits, plan.dists, 0, 1, 0};
        if (plan.scratch_bytes == 0)   // one block, one piece: no partials
            return nbody::launch_sym(plan.variant, pr.targets, pr.nt, pr.eps2, pr.pot, sl, out,
                                     stream);
        const int js = nbody::sym_group_jslots(plan.num_iblocks, plan.dists);
        sl.gstride = static_cast<int64_t>(plan.splits + js) * nt;
        float4 *lo = parts + static_cast<int64_t>(plan.groups_per_pass) * sl.gstride;
        for (int pass = 0; pass < plan.passes; ++pass) {
            sl.g0 = pass * plan.groups_per_pass;
            sl.groups = std::min(plan.groups_per_pass, plan.groups - sl.g0);
            cudaError_t e = nbody::launch_sym(plan.variant, pr.targets, pr.nt, pr.eps2, pr.pot, sl,
                                              parts, stream);
            if (e != cudaSuccess) return e;
            const bool last = pass + 1 == plan.passes;
            const nbody::ReducePass rp = {parts, sl.gstride, plan.splits, true, plan.dists,
                                          plan.num_iblocks, plan.threads * plan.i_per_thread,
                                          sl.g0, sl.groups, pr.nt, out, lo, pass > 0, last};
            e = nbody::launch_reduce_pass(rp, sm_count, stream, last ? eu : nullptr);
            if (e != cudaSuccess) return e;
        }
        if (fused != nullptr) *fused = eu != nullptr;
        return cudaSuccess;
    }
    if (plan.path == NBODY_PATH_ROWS)
        return nbody::launch_rows(plan.variant, pr, rows_launch(plan), out, stream);
    const int ntiles = static_cast<int>(ceil_div(pr.ns, plan.tile));
    if (plan.path == NBODY_PATH_CLUSTER)
        return nbody::launch_cluster(plan.variant, pr, plan.num_iblocks, plan.cluster,
                                     plan.tiles_per_split, ntiles, out, stream);
    if (plan.splits == 1)
        return nbody::launch_tiled(plan.variant, pr, plan.num_iblocks, 0, 1, plan.tiles_per_split,
                                   ntiles, out, stream);
    float4 *lo = parts + static_cast<int64_t>(plan.groups_per_pass) * nt;
    for (int pass = 0; pass < plan.passes; ++pass) {
        const int piece0 = pass * plan.groups_per_pass;
        const int pieces = std::min(plan.groups_per_pass, plan.splits - piece0);
        cudaError_t e = nbody::launch_tiled(plan.variant, pr, plan.num_iblocks, piece0, pieces,
                                            plan.tiles_per_split, ntiles, parts, stream);
        if (e != cudaSuccess) return e;
        const bool last = pass + 1 == plan.passes;
        const nbody::ReducePass rp = {parts, nt, 1, false, 0, 1, 1, piece0, pieces, pr.nt,
                                      out, lo, pass > 0, last};
        e = nbody::launch_reduce_pass(rp, sm_count, stream, last ? eu : nullptr);
        if (e != cudaSuccess) return e;
    }
    if (fused != nullptr) *fused = eu != nullptr;
    return cudaSuccess;
}

// One time step: the planned force evaluation, then the Euler update (inside
// the last reduction pass where the plan has one, otherwise its own kernel).
cudaError_t launch_step(const nbody_plan &plan, const nbody::Problem &pr, float4 *acc, void *ws,
                        int sm_count, float4 *pos, float4 *vel, float dt, cudaStream_t stream) {
    const nbody::EulerFuse eu = {pos, vel, dt};
    bool fused = false;
    cudaError_t e = launch_planned(plan, pr, acc, ws, sm_count, stream, &eu, &fused);
    if (e == cudaSuccess && !fused) e = nbody::launch_euler(pos, vel, acc, pr.nt, dt, sm_count, stream);
    return e;
}

Occupancy device_occupancy(const DeviceState *dev) {
    return {dev->tiled_occ, dev->cluster_occ, dev->sym_occ};
}

bool is_oom(cudaError_t e) { return e == cudaErrorMemoryAllocation; }

// One planned force evaluation (targets x sources) on `stream`.  With a
// caller's workspace (ws_bytes >= 0) it plans within it and allocates
// nothing; otherwise it takes the workspace from the device's pool, within
// the default budget, and re-plans within less if the pool cannot supply it.
nbody_status run_forces(const nbody::Problem &pr, const nbody_forces_opts *opts, float *result,
                        void *ws, int64_t ws_bytes, cudaStream_t stream) {
    DeviceState *dev = nullptr;
    nbody_status st = device_state(&dev);
    if (st != NBODY_OK) return st;
    nbody_plan plan;
    const bool all_pairs = pr.targets == pr.sources && pr.nt == pr.ns;
    const Occupancy occ = device_occupancy(dev);
    float4 *out = reinterpret_cast<float4 *>(result);
    cudaError_t e;
    if (ws_bytes >= 0) {
        if ((st = make_plan(pr.nt, pr.ns, all_pairs, dev->sm_count, occ, opts,
                            ws == nullptr ? 0 : ws_bytes, &plan, dev)) != NBODY_OK)
            return st;
        e = launch_planned(plan, pr, out, ws, dev->sm_count, stream);
        return e == cudaSuccess ? NBODY_OK : cuda_fail(e);
    }
    if ((st = make_plan(pr.nt, pr.ns, all_pairs, dev->sm_count, occ, opts, pool_budget(pr.nt),
                        &plan, dev)) != NBODY_OK)
        return st;
    void *scratch = nullptr;
    if (plan.scratch_bytes > 0) {
        cudaMemPool_t pool = nullptr;
        if ((st = device_pool(dev, &pool)) != NBODY_OK) return st;
        e = cudaMallocFromPoolAsync(&scratch, static_cast<size_t>(plan.scratch_bytes), pool, stream);
        // Short of memory: the least workspace of the same decomposition, then none.
        for (int64_t fallback : {plan.scratch_min_bytes, int64_t(0)}) {
            if (!is_oom(e)) break;
            cudaGetLastError();   // clear the allocation failure
            scratch = nullptr;
            if ((st = make_plan(pr.nt, pr.ns, all_pairs, dev->sm_count, occ, opts, fallback, &plan,
                                dev)) != NBODY_OK)
                return st;
            e = plan.scratch_bytes > 0
                    ? cudaMallocFromPoolAsync(&scratch, static_cast<size_t>(plan.scratch_bytes),
                                              pool, stream)
                    : cudaSuccess;
        }
        if (e != cudaSuccess) return cuda_fail(e);
    }
    e = launch_planned(plan, pr, out, scratch, dev->sm_count, stream);
    if (scratch != nullptr) {
        const cudaError_t ef = cudaFreeAsync(scratch, stream);
        if (e == cudaSuccess) e = ef;
    }
    return e == cudaSuccess ? NBODY_OK : cuda_fail(e);
}

// Workspace a call would take by default on the current device.
nbody_status default_workspace(int64_t nt, int64_t ns, bool all_pairs,
                               const nbody_forces_opts *opts, int64_t *bytes) {
    DeviceState *dev = nullptr;
    nbody_status st = device_state(&dev);
    if (st != NBODY_OK) return st;
    nbody_plan plan;
    if ((st = make_plan(nt, ns, all_pairs, dev->sm_count, device_occupancy(dev), opts,
                        pool_budget(nt), &plan, dev)) != NBODY_OK)
        return st;
    *bytes = plan.scratch_bytes;
    return NBODY_OK;
}

// ---------------------------------------------------------------- multi-step driver
//
// One step (forces, then Euler) is captured once into a CUDA graph on an
// internal stream and replayed `steps` times on the caller's stream, so a
// step costs one graph launch instead of several kernel launches from the
// host.  Where the forces end in a reduction kernel, the Euler update runs
// inside its last pass.  On the small-N paths (row-split, cluster) a second graph holds
// two steps whose Euler update is fused into the force kernel, the positions
// going from pos_mass to a second buffer and back; steps run in pairs
// through it, and an odd last step through the one-step graph.  One graph
// per device is cached, keyed by every argument but the step count; its
// workspace (pool memory, or the caller's) lives as long as the graph.  Each
// call waits on the GPU for the previous one (event `done`), whatever its
// stream, so two replays never share the workspace at the same time.  When
// the key changes, the old graph is destroyed and its pool memory freed in
// stream order behind its last replay.

// Steps per batch graph, and the largest n that gets one.
constexpr int kSimBatch = 16;
constexpr int64_t kSimBatchMaxN = 65536;

struct SimKey {
    const float *pm;
    float *vel;
    float *acc;
    int64_t n;
    float eps2;
    float dt;
    void *ws;           // the caller's workspace, or nullptr for pool memory
    int64_t ws_bytes;
    bool operator==(const SimKey &o) const {
        return pm == o.pm && vel == o.vel && acc == o.acc && n == o.n &&
               std::memcmp(&eps2, &o.eps2, sizeof(float)) == 0 &&
               std::memcmp(&dt, &o.dt, sizeof(float)) == 0 && ws == o.ws &&
               ws_bytes == o.ws_bytes;
    }
};

struct SimGraph {
    bool valid = false;
    SimKey key = {};
    cudaGraphExec_t exec = nullptr;    // one step: forces (+ reduction), then Euler
    cudaGraphExec_t exec2 = nullptr;   // small N: two steps with Euler fused into the forces
    cudaGraphExec_t execb = nullptr;   // up to 65536 bodies: kSimBatch steps in one graph
    void *pool_mem = nullptr;          // pool memory of the workspace (nullptr: the caller's)
    cudaEvent_t done = nullptr;        // recorded after the latest replay
};

std::mutex g_sim_mu;
SimGraph g_sim[kMaxDevices];
cudaStream_t g_capture[kMaxDevices] = {};

nbody_status sim_release(SimGraph &g, cudaStream_t stream) {
    cudaError_t e = cudaSuccess;
    for (cudaGraphExec_t *x : {&g.exec, &g.exec2, &g.execb}) {
        if (*x != nullptr) {
            const cudaError_t ex = cudaGraphExecDestroy(*x);
            if (e == cudaSuccess) e = ex;
            *x = nullptr;
        }
    }
    if (g.pool_mem != nullptr) {
        if (g.done != nullptr) cudaStreamWaitEvent(stream, g.done, 0);
        const cudaError_t ef = cudaFreeAsync(g.pool_mem, stream);
        if (e == cudaSuccess) e = ef;
        g.pool_mem = nullptr;
    }
    g.valid = false;
    return e == cudaSuccess ? NBODY_OK : cuda_fail(e);
}

// Capture `body` on the device's capture stream and instantiate it.
template <typename Body>
cudaError_t capture_graph(cudaStream_t cap, Body body, cudaGraphExec_t *exec) {
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return e;
    const cudaError_t el = body(cap);
    e = cudaStreamEndCapture(cap, &graph);
    if (el != cudaSuccess) e = el;
    if (e == cudaSuccess) e = cudaGraphInstantiate(exec, graph, 0);
    if (graph != nullptr) cudaGraphDestroy(graph);
    return e;
}

// Small-N paths, whose force kernel can apply the Euler step as it stores
// each body's result (into a second position buffer).
bool fuses_euler(const nbody_plan &plan) {
    return plan.path == NBODY_PATH_CLUSTER || plan.path == NBODY_PATH_ROWS;
}

// The force kernel of a small-N plan with the Euler step fused.
cudaError_t launch_fused(const nbody_plan &plan, const nbody::Problem &pr, float4 *acc,
                         const nbody::EulerFuse &eu, cudaStream_t s) {
    if (plan.path == NBODY_PATH_ROWS)
        return nbody::launch_rows(plan.variant, pr, rows_launch(plan), acc, s, &eu);
    const int ntiles = static_cast<int>(ceil_div(pr.ns, plan.tile));
    return nbody::launch_cluster(plan.variant, pr, plan.num_iblocks, plan.cluster,
                                 plan.tiles_per_split, ntiles, acc, s, &eu);
}

// The plan of one simulation step and the workspace it needs (the plan's
// partials, then at small n the second position buffer).
nbody_status sim_plan(DeviceState *dev, int64_t n, int64_t budget, nbody_plan *plan,
                      int64_t *bytes) {
    nbody_status st = make_plan(n, n, true, dev->sm_count, device_occupancy(dev), nullptr, budget,
                                plan, dev);
    if (st != NBODY_OK) return st;
    *bytes = plan->scratch_bytes + (fuses_euler(*plan) ? 16 * n : 0);
    return NBODY_OK;
}

nbody_status sim_build(int dev_id, DeviceState *dev, const SimKey &k, SimGraph &g,
                       cudaStream_t stream) {
    nbody_plan plan;
    int64_t need = 0;
    nbody_status st;
    cudaError_t e;
    if (g_capture[dev_id] == nullptr &&
        (e = cudaStreamCreateWithFlags(&g_capture[dev_id], cudaStreamNonBlocking)) != cudaSuccess)
        return cuda_fail(e);
    if (g.done == nullptr && (e = cudaEventCreateWithFlags(&g.done, cudaEventDisableTiming)) != cudaSuccess)
        return cuda_fail(e);
    void *ws = nullptr;          // the plan's partials, then (small n) the second buffer
    void *pool_mem = nullptr;
    int64_t room = 0;            // bytes at ws
    if (k.ws_bytes >= 0) {
        // the caller's workspace (a null one has no room at all)
        room = k.ws != nullptr ? k.ws_bytes : 0;
        if ((st = sim_plan(dev, k.n, room, &plan, &need)) != NBODY_OK) return st;
        ws = k.ws;
    } else {
        if ((st = sim_plan(dev, k.n, pool_budget(k.n), &plan, &need)) != NBODY_OK) return st;
        if (need > 0) {
            cudaMemPool_t pool = nullptr;
            if ((st = device_pool(dev, &pool)) != NBODY_OK) return st;
            e = cudaMallocFromPoolAsync(&pool_mem, static_cast<size_t>(need), pool, stream);
            if (is_oom(e)) {   // the least workspace of the same plan, then none
                cudaGetLastError();
                pool_mem = nullptr;
                if ((st = sim_plan(dev, k.n, plan.scratch_min_bytes, &plan, &need)) != NBODY_OK)
                    return st;
                e = need > 0 ? cudaMallocFromPoolAsync(&pool_mem, static_cast<size_t>(need), pool,
                                                       stream)
                             : cudaSuccess;
                if (is_oom(e)) {
                    cudaGetLastError();
                    pool_mem = nullptr;
                    if ((st = sim_plan(dev, k.n, 0, &plan, &need)) != NBODY_OK) return st;
                    e = cudaSuccess;
                }
            }
            if (e != cudaSuccess) return cuda_fail(e);
            ws = pool_mem;
            room = pool_mem != nullptr ? need : 0;
        }
    }
    // the first replay waits for the allocation, on whatever stream it runs
    if ((e = cudaEventRecord(g.done, stream)) != cudaSuccess) {
        if (pool_mem != nullptr) cudaFreeAsync(pool_mem, stream);
        return cuda_fail(e);
    }
    const cudaStream_t cap = g_capture[dev_id];
    const int ni = static_cast<int>(k.n);
    float4 *pos = reinterpret_cast<float4 *>(const_cast<float *>(k.pm));
    float4 *vel = reinterpret_cast<float4 *>(k.vel);
    float4 *acc = reinterpret_cast<float4 *>(k.acc);
    const nbody::Problem pr = {k.pm, k.pm, ni, ni, k.eps2, true};
    void *parts = plan.scratch_bytes > 0 ? ws : nullptr;
    cudaGraphExec_t exec = nullptr, exec2 = nullptr;
    e = capture_graph(cap, [&](cudaStream_t s) {
        return launch_step(plan, pr, acc, parts, dev->sm_count, pos, vel, k.dt, s);
    }, &exec);
    // Small N: two steps per replay with the Euler update fused into the
    // force kernel, positions alternating between pos_mass and pos_b.
    float4 *pb = nullptr;
    if (e == cudaSuccess && fuses_euler(plan) && ws != nullptr &&
        room >= plan.scratch_bytes + 16 * k.n)
        pb = reinterpret_cast<float4 *>(static_cast<char *>(ws) + plan.scratch_bytes);
    const nbody::Problem pr_b = {reinterpret_cast<const float *>(pb),
                                 reinterpret_cast<const float *>(pb), ni, ni, k.eps2, true};
    const nbody::EulerFuse to_b = {pb, vel, k.dt};
    const nbody::EulerFuse to_a = {pos, vel, k.dt};
    if (pb != nullptr) {
        e = capture_graph(cap, [&](cudaStream_t s) {
            cudaError_t el = launch_fused(plan, pr, acc, to_b, s);
            if (el == cudaSuccess) el = launch_fused(plan, pr_b, acc, to_a, s);
            return el;
        }, &exec2);
    }
    // Up to 65536 bodies a step is short enough that launching one graph per
    // step (or pair) shows: kSimBatch steps are captured into one graph,
    // where each kernel's launch overlaps the previous one's tail.
    cudaGraphExec_t execb = nullptr;
    if (e == cudaSuccess && k.n <= kSimBatchMaxN) {
        if (exec2 != nullptr) {
            e = capture_graph(cap, [&](cudaStream_t s) {
                cudaError_t el = cudaSuccess;
                for (int t = 0; t < kSimBatch / 2 && el == cudaSuccess; ++t) {
                    el = launch_fused(plan, pr, acc, to_b, s);
                    if (el == cudaSuccess) el = launch_fused(plan, pr_b, acc, to_a, s);
                }
                return el;
            }, &execb);
        } else {
            e = capture_graph(cap, [&](cudaStream_t s) {
                cudaError_t el = cudaSuccess;
                for (int t = 0; t < kSimBatch && el == cudaSuccess; ++t)
                    el = launch_step(plan, pr, acc, parts, dev->sm_count, pos, vel, k.dt, s);
                return el;
            }, &execb);
        }
    }
    if (e != cudaSuccess) {
        if (exec != nullptr) cudaGraphExecDestroy(exec);
        if (exec2 != nullptr) cudaGraphExecDestroy(exec2);
        if (pool_mem != nullptr) cudaFreeAsync(pool_mem, stream);
        return cuda_fail(e);
    }
    g.key = k;
    g.exec = exec;
    g.exec2 = exec2;
    g.execb = execb;
    g.pool_mem = pool_mem;
    g.valid = true;
    return NBODY_OK;
}

nbody_status run_simulate(float *pos_mass, float *vel, float *acc_pot, int64_t n, float eps2,
                          float dt, int64_t steps, void *ws, int64_t ws_bytes, cudaStream_t stream) {
    nbody_status st = check_forces(pos_mass, n, eps2, acc_pot);
    if (st != NBODY_OK) return st;
    if (steps < 0 || !std::isfinite(dt)) return NBODY_ERR_INVALID_ARG;
    if (n == 0 || steps == 0) return NBODY_OK;
    if (vel == nullptr) return NBODY_ERR_INVALID_ARG;
    if (!aligned16(vel)) return NBODY_ERR_MISALIGNED;
    if (overlap(vel, pos_mass, 16 * n) || overlap(vel, acc_pot, 16 * n)) return NBODY_ERR_ALIAS;
    if (ws_bytes >= 0 &&
        (st = check_workspace(ws, static_cast<size_t>(ws_bytes),
                              {{pos_mass, 16 * n}, {vel, 16 * n}, {acc_pot, 16 * n}})) != NBODY_OK)
        return st;
    DeviceState *dev = nullptr;
    if ((st = device_state(&dev)) != NBODY_OK) return st;
    int dev_id = 0;
    if ((st = current_device(&dev_id)) != NBODY_OK) return st;
    std::lock_guard<std::mutex> lock(g_sim_mu);
    SimGraph &g = g_sim[dev_id];
    const SimKey key = {pos_mass, vel, acc_pot, n, eps2, dt, ws_bytes >= 0 ? ws : nullptr,
                        ws_bytes >= 0 ? (ws == nullptr ? 0 : ws_bytes) : -1};
    if (!(g.valid && g.key == key)) {
        if (g.valid && (st = sim_release(g, stream)) != NBODY_OK) return st;
        if ((st = sim_build(dev_id, dev, key, g, stream)) != NBODY_OK) return st;
    }
    cudaError_t e = cudaStreamWaitEvent(stream, g.done, 0);   // after the previous replay
    if (e != cudaSuccess) return cuda_fail(e);
    int64_t left = steps;
    if (g.execb != nullptr)
        for (; left >= kSimBatch; left -= kSimBatch)
            if ((e = cudaGraphLaunch(g.execb, stream)) != cudaSuccess) return cuda_fail(e);
    if (g.exec2 != nullptr)
        for (; left >= 2; left -= 2)
            if ((e = cudaGraphLaunch(g.exec2, stream)) != cudaSuccess) return cuda_fail(e);
    for (; left > 0; --left)
        if ((e = cudaGraphLaunch(g.exec, stream)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaEventRecord(g.done, stream)) != cudaSuccess) return cuda_fail(e);
    return NBODY_OK;
}

// Nominal occupancy of each tiled variant (used by the host-only planner
// entry point when the caller gives none): register-limited at 64K per SM.
int nominal_occ(int i_per_thread, int threads) {
    const int regs = i_per_thread >= 8 ? 168 : (i_per_thread >= 4 ? 96 : 64);
    int occ = 65536 / (regs * threads);
    return occ < 1 ? 1 : occ;
}

nbody_status host_plan(int64_t nt, int64_t ns, bool all_pairs, int32_t sm_count,
                       int32_t ctas_per_sm, const nbody_forces_opts *opts, int64_t budget,
                       nbody_plan *plan) {
    int occ[kMaxVariants], cocc[kMaxVariants], socc[kMaxVariants];
    for (int v = 0; v < nbody::tiled_variant_count() && v < kMaxVariants; ++v) {
        const nbody::TiledVariant &tv = nbody::tiled_variant(v);
        occ[v] = ctas_per_sm > 0 ? ctas_per_sm : nominal_occ(tv.i_per_thread, tv.threads);
    }
    for (int v = 0; v < nbody::cluster_variant_count() && v < kMaxVariants; ++v) {
        const nbody::ClusterVariant &cv = nbody::cluster_variant(v);
        cocc[v] = ctas_per_sm > 0 ? ctas_per_sm : nominal_occ(cv.i_per_thread, cv.warps * 32);
    }
    for (int v = 0; v < nbody::sym_variant_count() && v < kMaxVariants; ++v) {
        const nbody::SymVariant &sv = nbody::sym_variant(v);
        const int by_smem = static_cast<int>(kSmemPerSm / static_cast<int64_t>(sv.smem + 1024));
        socc[v] = ctas_per_sm > 0 ? ctas_per_sm : std::max(1, std::min(sv.min_ctas, by_smem));
    }
    return make_plan(nt, ns, all_pairs, sm_count, Occupancy{occ, cocc, socc}, opts, budget, plan);
}

nbody_forces_opts with_quantities(const nbody_forces_opts *opts, int quantities) {
    nbody_forces_opts o = {NBODY_PATH_AUTO, -1, 0, NBODY_PRECISION_DEFAULT, quantities, 0};
    if (opts != nullptr) {
        o = *opts;
        if (quantities != NBODY_QUANTITIES_ACC_POT) o.quantities = quantities;
    }
    return o;
}

bool wants_pot(const nbody_forces_opts *opts) {
    return opts == nullptr || opts->quantities != NBODY_QUANTITIES_ACC;
}

nbody_status forces_common(const float *pos_mass, int64_t n, float eps2, float *acc_pot,
                           const nbody_forces_opts *opts, void *ws, int64_t ws_bytes,
                           cudaStream_t stream) {
    nbody_status st = check_forces(pos_mass, n, eps2, acc_pot);
    if (st != NBODY_OK || n == 0) return st;
    if (ws_bytes >= 0 &&
        (st = check_workspace(ws, static_cast<size_t>(ws_bytes),
                              {{pos_mass, 16 * n}, {acc_pot, 16 * n}})) != NBODY_OK)
        return st;
    const nbody::Problem pr = {pos_mass, pos_mass, static_cast<int>(n), static_cast<int>(n), eps2,
                               wants_pot(opts)};
    return run_forces(pr, opts, acc_pot, ws, ws_bytes, stream);
}

nbody_status forces_ts_common(const float *targets, int64_t nt, const float *sources, int64_t ns,
                              float eps2, float *out, const nbody_forces_opts *opts, void *ws,
                              int64_t ws_bytes, cudaStream_t stream) {
    if (check_n(nt) != NBODY_OK || check_n(ns) != NBODY_OK) return NBODY_ERR_INVALID_ARG;
    if (nt == 0) return NBODY_OK;
    if (targets == nullptr || out == nullptr || (ns > 0 && sources == nullptr))
        return NBODY_ERR_INVALID_ARG;
    if (!eps2_ok(eps2)) return NBODY_ERR_INVALID_ARG;
    if (!aligned16(targets) || !aligned16(out) || (ns > 0 && !aligned16(sources)))
        return NBODY_ERR_MISALIGNED;
    if (overlap(out, targets, 16 * nt)) return NBODY_ERR_ALIAS;
    if (ns > 0 && overlap2(out, 16 * nt, sources, 16 * ns)) return NBODY_ERR_ALIAS;
    nbody_status st;
    if (ws_bytes >= 0 &&
        (st = check_workspace(ws, static_cast<size_t>(ws_bytes),
                              {{targets, 16 * nt}, {sources, 16 * ns}, {out, 16 * nt}})) != NBODY_OK)
        return st;
    if (ns == 0) {   // no sources: every sum is empty
        const cudaError_t e = cudaMemsetAsync(out, 0, static_cast<size_t>(16 * nt), stream);
        return e == cudaSuccess ? NBODY_OK : cuda_fail(e);
    }
    const nbody::Problem pr = {targets, sources, static_cast<int>(nt), static_cast<int>(ns), eps2,
                               wants_pot(opts)};
    return run_forces(pr, opts, out, ws, ws_bytes, stream);
}

}  // namespace

namespace nbody {
void record_cuda_error(int e) { g_last_cuda_error = e; }
}  // namespace nbody

// ======================================================================= C ABI

extern "C" {

const char *nbody_status_string(nbody_status s) {
    switch (s) {
        case NBODY_OK: return "NBODY_OK";
        case NBODY_ERR_INVALID_ARG: return "NBODY_ERR_INVALID_ARG: invalid argument";
        case NBODY_ERR_MISALIGNED: return "NBODY_ERR_MISALIGNED: array not 16-byte aligned";
        case NBODY_ERR_ALIAS: return "NBODY_ERR_ALIAS: output or workspace overlaps another array";
        case NBODY_ERR_CUDA: return "NBODY_ERR_CUDA: CUDA runtime error";
        case NBODY_ERR_TIMEOUT: return "NBODY_ERR_TIMEOUT: bounded device wait ran out";
        case NBODY_ERR_DEVICE: return "NBODY_ERR_DEVICE: current device is not sm_103";
        case NBODY_ERR_TOO_LARGE:
            return "NBODY_ERR_TOO_LARGE: n exceeds the fixed scratch of nbody_forces_noalloc";
        case NBODY_ERR_WORKSPACE:
            return "NBODY_ERR_WORKSPACE: the forced path cannot run within the given workspace";
    }
    return "NBODY_ERR_UNKNOWN";
}

int nbody_last_cuda_error(void) { return g_last_cuda_error; }

nbody_status nbody_plan_forces(int64_t n, int32_t sm_count, int32_t ctas_per_sm,
                               const nbody_forces_opts *opts, nbody_plan *plan) {
    return host_plan(n, n, true, sm_count, ctas_per_sm, opts, n > 0 ? pool_budget(n) : 0, plan);
}

nbody_status nbody_plan_forces_ws(int64_t n, int32_t sm_count, int32_t ctas_per_sm,
                                  const nbody_forces_opts *opts, int64_t workspace_bytes,
                                  nbody_plan *plan) {
    if (workspace_bytes < 0) return NBODY_ERR_INVALID_ARG;
    return host_plan(n, n, true, sm_count, ctas_per_sm, opts, workspace_bytes, plan);
}

nbody_status nbody_plan_forces_ts(int64_t nt, int64_t ns, int32_t sm_count, int32_t ctas_per_sm,
                                  const nbody_forces_opts *opts, int64_t workspace_bytes,
                                  nbody_plan *plan) {
    if (workspace_bytes < -1) return NBODY_ERR_INVALID_ARG;
    return host_plan(nt, ns, false, sm_count, ctas_per_sm, opts,
                     workspace_bytes >= 0 ? workspace_bytes : (nt > 0 ? pool_budget(nt) : 0), plan);
}

nbody_status nbody_forces_ex(const float *pos_mass, int64_t n, float eps2, float *acc_pot,
                             const nbody_forces_opts *opts, cudaStream_t stream) {
    return forces_common(pos_mass, n, eps2, acc_pot, opts, nullptr, -1, stream);
}

nbody_status nbody_forces(const float *pos_mass, int64_t n, float eps2, float *acc_pot,
                          cudaStream_t stream) {
    return forces_common(pos_mass, n, eps2, acc_pot, nullptr, nullptr, -1, stream);
}

nbody_status nbody_forces_acc(const float *pos_mass, int64_t n, float eps2, float *acc_pot,
                              cudaStream_t stream) {
    const nbody_forces_opts o = with_quantities(nullptr, NBODY_QUANTITIES_ACC);
    return forces_common(pos_mass, n, eps2, acc_pot, &o, nullptr, -1, stream);
}

nbody_status nbody_forces_ts(const float *targets, int64_t nt, const float *sources, int64_t ns,
                             float eps2, float *out, cudaStream_t stream) {
    return forces_ts_common(targets, nt, sources, ns, eps2, out, nullptr, nullptr, -1, stream);
}

nbody_status nbody_forces_ws(const float *pos_mass, int64_t n, float eps2, float *acc_pot,
                             const nbody_forces_opts *opts, void *workspace,
                             size_t *workspace_bytes, cudaStream_t stream) {
    if (workspace_bytes == nullptr) return NBODY_ERR_INVALID_ARG;
    if (workspace == nullptr) {   // size query
        if (check_n(n) != NBODY_OK || !eps2_ok(eps2)) return NBODY_ERR_INVALID_ARG;
        int64_t b = 0;
        nbody_status st = n == 0 ? NBODY_OK : default_workspace(n, n, true, opts, &b);
        if (st == NBODY_OK) *workspace_bytes = static_cast<size_t>(b);
        return st;
    }
    if (*workspace_bytes > static_cast<size_t>(INT64_MAX)) return NBODY_ERR_INVALID_ARG;
    return forces_common(pos_mass, n, eps2, acc_pot, opts, workspace,
                         static_cast<int64_t>(*workspace_bytes), stream);
}

nbody_status nbody_forces_ts_ws(const float *targets, int64_t nt, const float *sources,
                                int64_t ns, float eps2, float *out,
                                const nbody_forces_opts *opts, void *workspace,
                                size_t *workspace_bytes, cudaStream_t stream) {
    if (workspace_bytes == nullptr) return NBODY_ERR_INVALID_ARG;
    if (workspace == nullptr) {   // size query
        if (check_n(nt) != NBODY_OK || check_n(ns) != NBODY_OK || !eps2_ok(eps2))
            return NBODY_ERR_INVALID_ARG;
        int64_t b = 0;
        nbody_status st = NBODY_OK;
        if (nt > 0 && ns > 0)
            st = default_workspace(nt, ns, targets != nullptr && targets == sources, opts, &b);
        if (st == NBODY_OK) *workspace_bytes = static_cast<size_t>(b);
        return st;
    }
    if (*workspace_bytes > static_cast<size_t>(INT64_MAX)) return NBODY_ERR_INVALID_ARG;
    return forces_ts_common(targets, nt, sources, ns, eps2, out, opts, workspace,
                            static_cast<int64_t>(*workspace_bytes), stream);
}

nbody_status nbody_simulate(float *pos_mass, float *vel, float *acc_pot, int64_t n, float eps2,
                            float dt, int64_t steps, cudaStream_t stream) {
    return run_simulate(pos_mass, vel, acc_pot, n, eps2, dt, steps, nullptr, -1, stream);
}

nbody_status nbody_simulate_ws(float *pos_mass, float *vel, float *acc_pot, int64_t n,
                               float eps2, float dt, int64_t steps, void *workspace,
                               size_t *workspace_bytes, cudaStream_t stream) {
    if (workspace_bytes == nullptr) return NBODY_ERR_INVALID_ARG;
    if (workspace == nullptr) {   // size query
        if (check_n(n) != NBODY_OK || !eps2_ok(eps2)) return NBODY_ERR_INVALID_ARG;
        if (n == 0) {
            *workspace_bytes = 0;
            return NBODY_OK;
        }
        DeviceState *dev = nullptr;
        nbody_status st = device_state(&dev);
        if (st != NBODY_OK) return st;
        nbody_plan plan;
        int64_t need = 0;
        if ((st = sim_plan(dev, n, pool_budget(n), &plan, &need)) != NBODY_OK) return st;
        *workspace_bytes = static_cast<size_t>(need);
        return NBODY_OK;
    }
    if (*workspace_bytes > static_cast<size_t>(INT64_MAX)) return NBODY_ERR_INVALID_ARG;
    return run_simulate(pos_mass, vel, acc_pot, n, eps2, dt, steps, workspace,
                        static_cast<int64_t>(*workspace_bytes), stream);
}

nbody_status nbody_release_cached(void) {
    int dev_id = 0;
    nbody_status st = current_device(&dev_id);
    if (st != NBODY_OK) return st;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
    {
        std::lock_guard<std::mutex> lock(g_sim_mu);
        SimGraph &g = g_sim[dev_id];
        if (g.valid || g.pool_mem != nullptr) {
            if ((st = sim_release(g, 0)) != NBODY_OK) return st;
            if ((e = cudaStreamSynchronize(0)) != cudaSuccess) return cuda_fail(e);
        }
    }
    cudaMemPool_t pool = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        pool = g_dev[dev_id].pool;
    }
    if (pool != nullptr && (e = cudaMemPoolTrimTo(pool, 0)) != cudaSuccess) return cuda_fail(e);
    return NBODY_OK;
}

nbody_status nbody_euler_step(float *pos_mass, float *vel, const float *acc_pot, int64_t n,
                              float dt, cudaStream_t stream) {
    if (check_n(n) != NBODY_OK) return NBODY_ERR_INVALID_ARG;
    if (n == 0) return NBODY_OK;
    if (pos_mass == nullptr || vel == nullptr || acc_pot == nullptr) return NBODY_ERR_INVALID_ARG;
    if (!std::isfinite(dt)) return NBODY_ERR_INVALID_ARG;
    if (!aligned16(pos_mass) || !aligned16(vel) || !aligned16(acc_pot)) return NBODY_ERR_MISALIGNED;
    const int64_t bytes = 16 * n;
    if (overlap(pos_mass, vel, bytes) || overlap(pos_mass, acc_pot, bytes) ||
        overlap(vel, acc_pot, bytes))
        return NBODY_ERR_ALIAS;
    DeviceState *dev = nullptr;
    nbody_status st = device_state(&dev);
    if (st != NBODY_OK) return st;
    const cudaError_t e = nbody::launch_euler(reinterpret_cast<float4 *>(pos_mass),
                                              reinterpret_cast<float4 *>(vel),
                                              reinterpret_cast<const float4 *>(acc_pot),
                                              static_cast<int>(n), dt, dev->sm_count, stream);
    return e == cudaSuccess ? NBODY_OK : cuda_fail(e);
}

}  // extern "C"
