// nbody_api.cu -- the C ABI: argument checks, the launch planner, per-device
// state and dispatch.  See include/nbody.h for the contract of each call.
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

bool overlap(const void *a, const void *b, int64_t bytes) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a);
    const uintptr_t y = reinterpret_cast<uintptr_t>(b);
    const uintptr_t len = static_cast<uintptr_t>(bytes);
    return x < y + len && y < x + len;
}

// [a, a + a_bytes) and [b, b + b_bytes) share a byte.
bool overlap2(const void *a, int64_t a_bytes, const void *b, int64_t b_bytes) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a);
    const uintptr_t y = reinterpret_cast<uintptr_t>(b);
    return x < y + static_cast<uintptr_t>(b_bytes) && y < x + static_cast<uintptr_t>(a_bytes);
}

nbody_status check_n(int64_t n) {
    return (n < 0 || n > INT32_MAX) ? NBODY_ERR_INVALID_ARG : NBODY_OK;
}

nbody_status check_forces(const float *pm, int64_t n, float eps2, const float *acc) {
    if (check_n(n) != NBODY_OK) return NBODY_ERR_INVALID_ARG;
    if (n == 0) return NBODY_OK;
    if (pm == nullptr || acc == nullptr) return NBODY_ERR_INVALID_ARG;
    if (!std::isfinite(eps2) || !(eps2 >= FLT_MIN)) return NBODY_ERR_INVALID_ARG;
    if (!aligned16(pm) || !aligned16(acc)) return NBODY_ERR_MISALIGNED;
    if (overlap(pm, acc, 16 * n)) return NBODY_ERR_ALIAS;
    return NBODY_OK;
}

// ---------------------------------------------------------------- per-device state

constexpr int kMaxDevices = 64;
constexpr int kMaxVariants = 32;

struct DeviceState {
    bool ready = false;
    int sm_count = 0;
    int tiled_occ[kMaxVariants] = {0};
    int cluster_occ[kMaxVariants] = {0};
    int sym_occ[kMaxVariants] = {0};
    cudaMemPool_t pool = nullptr;     // stream-ordered scratch for split partials
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

nbody_status device_state(DeviceState **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return NBODY_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &d = g_dev[dev];
    if (!d.ready) {
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
            if (cv.whole &&
                (e = cudaFuncSetAttribute(cv.fn_pot, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(nbody::kWholeSmemMax))) != cudaSuccess)
                return cuda_fail(e);
            // register-limited residency (whole-range launches are further
            // limited by their shared memory, see plan_cluster_variant)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.cluster_occ[v], cv.fn_pot,
                                                              cv.warps * 32, 0);
            if (e != cudaSuccess) return cuda_fail(e);
        }
        for (int v = 0; v < nbody::sym_variant_count() && v < kMaxVariants; ++v) {
            const nbody::SymVariant &sv = nbody::sym_variant(v);
            if ((e = cudaFuncSetAttribute(sv.fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(sv.smem))) != cudaSuccess)
                return cuda_fail(e);
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.sym_occ[v], sv.fn, sv.warps * 32,
                                                              sv.smem);
            if (e != cudaSuccess) return cuda_fail(e);
        }
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        if ((e = cudaMemPoolCreate(&d.pool, &props)) != cudaSuccess) return cuda_fail(e);
        uint64_t keep = UINT64_MAX;   // keep freed blocks for the next call
        if ((e = cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess)
            return cuda_fail(e);
        d.ready = true;
    }
    *out = &d;
    return NBODY_OK;
}

// ---------------------------------------------------------------- planner

constexpr int kDefaultTiledVariant = 0;
constexpr int kDefaultClusterVariant = 0;
constexpr int kCompensatedTiledVariant = 7;
constexpr int kMaxSplits = 1024;
constexpr int64_t kMaxScratchBytes = int64_t(2) << 30;
// Relative cost model (only ratios matter): pair rate of one SM, the fixed
// cost of a work item in source-body equivalents, one launch, scratch traffic.
constexpr double kPairsPerSmSecond = 1.4e10;
constexpr int kItemOverheadBodies = 96;
constexpr double kLaunchSeconds = 2.5e-6;
constexpr double kScratchBytesPerSecond = 5.0e12;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

void plan_tiled(int64_t nt, int64_t ns, int sm, int occ, int variant, int splits_req,
                nbody_plan *p) {
    const nbody::TiledVariant &v = nbody::tiled_variant(variant);
    const int64_t bi = static_cast<int64_t>(v.threads) * v.i_per_thread;
    const int64_t num_ib = ceil_div(nt, bi);
    const int64_t ntiles = ceil_div(ns, v.tile);
    const int64_t slots = static_cast<int64_t>(sm > 0 ? sm : 1) * (occ > 0 ? occ : 1);
    const double slot_rate = kPairsPerSmSecond / (occ > 0 ? occ : 1);

    int64_t s_lo = 1, s_hi = std::min<int64_t>(ntiles, kMaxSplits);
    s_hi = std::max<int64_t>(1, std::min<int64_t>(s_hi, kMaxScratchBytes / (16 * nt)));
    if (splits_req > 0) s_lo = s_hi = std::min<int64_t>(splits_req, ntiles);

    double best_t = INFINITY;
    int64_t best_s = 1, best_tps = ntiles, best_waves = 1;
    for (int64_t s = s_lo; s <= s_hi; ++s) {
        const int64_t tps = ceil_div(ntiles, s);
        const int64_t used = ceil_div(ntiles, tps);
        if (used != s && splits_req <= 0) continue;   // same as a smaller S
        const int64_t items = num_ib * used;
        const int64_t waves = ceil_div(items, slots);
        double t = static_cast<double>(waves) *
                   static_cast<double>(tps * v.tile + kItemOverheadBodies) * bi / slot_rate;
        if (used > 1) t += kLaunchSeconds + 32.0 * used * nt / kScratchBytesPerSecond;
        if (t < best_t * (1.0 - 1e-3)) {
            best_t = t;
            best_s = used;
            best_tps = tps;
            best_waves = waves;
        }
    }
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
    p->grid = num_ib * best_s;
    p->scratch_bytes = best_s > 1 ? 16 * best_s * nt : 0;
    p->fill = static_cast<double>(num_ib * best_s) / static_cast<double>(best_waves * slots);
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
    p->grid = num_ib * best_c;
    p->scratch_bytes = 0;
    p->fill = best_fill > 1.0 ? 1.0 : best_fill;
    *t_out = best_t;
}

// Largest n the automatic choice sends to the cluster path (measured on
// GB300 inside CUDA graphs: the cluster path is ahead up to 4096 bodies, the
// tiled one from 8192).
constexpr int64_t kClusterMaxN = 6144;

// Symmetric path (each unordered pair once).  Smallest n the automatic choice
// sends to it, and the variant it takes by size, measured on GB300 inside
// CUDA graphs: from 10240 bodies every shape below beats the tiled path
// (54.5 against 57.6 us at 10240; 221 against 264 us at 24576), 512-body
// blocks win up to about 45K bodies (better filled waves), 1024-body blocks
// up to about 160K, and 2048-body blocks above (fewer partial slots); each
// choice is within 4.5 % of the fastest shape at every size measured.  The
// j-side partials take (nb - 1) / 2 (+1) records per body, so they grow as
// n^2 / T: the cap below bounds them.
constexpr int64_t kSymMinN = 10240;
constexpr int64_t kSymMidN = 45056;     // from here 1024-body blocks
constexpr int64_t kSymLargeN = 163840;  // from here 2048-body blocks
constexpr int kSymSmallVariant = 2;     // K = 8, 2 warps: 512-body blocks
constexpr int kSymMidVariant = 1;       // K = 8, 4 warps: 1024-body blocks
constexpr int kDefaultSymVariant = 0;   // K = 8, 8 warps: 2048-body blocks
constexpr int64_t kMaxSymScratchBytes = int64_t(24) << 30;
// Relative cost model of the symmetric path: evaluations (two interactions
// each) per SM-second, the fixed cost of a CTA in evaluations, scratch traffic.
constexpr double kSymEvalsPerSmSecond = 1.1e10;
constexpr double kSymItemOverheadEvals = 64.0 * 1024.0;

struct Occupancy {
    const int *tiled;
    const int *cluster;
    const int *sym;
};

// Block count, j-side slots per body (the largest), and units per row (the
// largest) of the symmetric decomposition.
struct SymGeometry {
    int64_t block, nb, jslots, units;
};

SymGeometry sym_geometry(const nbody::SymVariant &v, int64_t n) {
    SymGeometry g;
    g.block = 32LL * v.warps * v.i_per_thread;
    g.nb = ceil_div(n, g.block);
    const int64_t h = (g.nb - 1) / 2;
    g.jslots = h + (g.nb % 2 == 0 ? 1 : 0);
    g.units = (1 + g.jslots) * (g.block / v.sub);
    return g;
}

bool plan_sym(int64_t n, int sm, int occ, int variant, int splits_req, nbody_plan *p) {
    const nbody::SymVariant &v = nbody::sym_variant(variant);
    const SymGeometry g = sym_geometry(v, n);
    const int64_t jbytes = 16 * g.jslots * n;
    if (jbytes + 16 * n > kMaxSymScratchBytes) return false;
    const int64_t slots = static_cast<int64_t>(sm > 0 ? sm : 1) * (occ > 0 ? occ : 1);
    const double slot_rate = kSymEvalsPerSmSecond / (occ > 0 ? occ : 1);
    const double unit_evals = static_cast<double>(g.block) * v.sub;

    // pieces allowed by the partials' cap (each piece adds one i-side slot)
    const int64_t s_cap = std::max<int64_t>(1, (kMaxSymScratchBytes - jbytes) / (16 * n));
    int64_t s_lo = 1, s_hi = std::min<int64_t>(std::min<int64_t>(g.units, kMaxSplits), s_cap);
    if (splits_req > 0) s_lo = s_hi = std::min<int64_t>(std::min<int64_t>(splits_req, g.units), s_cap);

    double best_t = INFINITY;
    int64_t best_s = 1, best_upp = g.units, best_waves = 1;
    for (int64_t s = s_lo; s <= s_hi; ++s) {
        const int64_t upp = ceil_div(g.units, s);   // units of the largest piece
        const int64_t waves = ceil_div(g.nb * s, slots);
        double t = static_cast<double>(waves) * (upp * unit_evals + kSymItemOverheadEvals) /
                   slot_rate;
        const bool reduce = s > 1 || g.jslots > 0;
        if (reduce) t += kLaunchSeconds + 16.0 * (s + g.jslots + 1) * n / kScratchBytesPerSecond;
        if (t < best_t * (1.0 - 1e-3)) {
            best_t = t;
            best_s = s;
            best_upp = upp;
            best_waves = waves;
        }
    }
    p->path = NBODY_PATH_SYMMETRIC;
    p->variant = variant;
    p->i_per_thread = v.i_per_thread;
    p->threads = v.warps * 32;
    p->tile = v.sub;
    p->num_iblocks = static_cast<int32_t>(g.nb);
    p->splits = static_cast<int32_t>(best_s);
    p->tiles_per_split = static_cast<int32_t>(best_upp);
    p->cluster = 1;
    p->warps_j = 1;
    p->grid = g.nb * best_s;
    p->scratch_bytes = (best_s > 1 || g.jslots > 0) ? 16 * (best_s + g.jslots) * n : 0;
    p->fill = static_cast<double>(g.nb * best_s) / static_cast<double>(best_waves * slots);
    return true;
}

int auto_sym_variant(int64_t n) {
    return n < kSymMidN ? kSymSmallVariant : (n < kSymLargeN ? kSymMidVariant : kDefaultSymVariant);
}

// all_pairs: the targets are the sources (same array, nt == ns), the case the
// symmetric path needs.
nbody_status make_plan(int64_t nt, int64_t ns, bool all_pairs, int sm, const Occupancy &occ,
                       const nbody_forces_opts *opts, nbody_plan *p) {
    if (nt <= 0 || nt > INT32_MAX || ns <= 0 || ns > INT32_MAX || sm <= 0 || p == nullptr)
        return NBODY_ERR_INVALID_ARG;
    nbody_forces_opts o = {NBODY_PATH_AUTO, -1, 0, 0};
    if (opts != nullptr) o = *opts;
    if (o.path < NBODY_PATH_AUTO || o.path > NBODY_PATH_SYMMETRIC || o.splits < 0)
        return NBODY_ERR_INVALID_ARG;
    if (o.precision < 0 || o.precision > 1) return NBODY_ERR_INVALID_ARG;
    if (o.precision == 1) {   // compensated: the tiled path's compensated kernel
        if (o.path == NBODY_PATH_CLUSTER || o.path == NBODY_PATH_SYMMETRIC ||
            (o.variant >= 0 && o.variant != kCompensatedTiledVariant))
            return NBODY_ERR_INVALID_ARG;
        o.path = NBODY_PATH_TILED;
        o.variant = kCompensatedTiledVariant;
    }
    all_pairs = all_pairs && nt == ns;
    if (o.path == NBODY_PATH_SYMMETRIC && !all_pairs) return NBODY_ERR_INVALID_ARG;
    int path = o.path;
    if (path == NBODY_PATH_AUTO) {
        if (nt <= kClusterMaxN && ns <= kClusterMaxN) {
            path = NBODY_PATH_CLUSTER;
        } else if (all_pairs && nt >= kSymMinN &&
                   plan_sym(nt, sm, occ.sym[auto_sym_variant(nt)], auto_sym_variant(nt), o.splits,
                            p)) {
            return NBODY_OK;
        } else {
            path = NBODY_PATH_TILED;
        }
    }
    if (path == NBODY_PATH_SYMMETRIC) {
        const int variant = o.variant < 0 ? auto_sym_variant(nt) : o.variant;
        if (variant >= nbody::sym_variant_count() || variant >= kMaxVariants)
            return NBODY_ERR_INVALID_ARG;
        return plan_sym(nt, sm, occ.sym[variant], variant, o.splits, p) ? NBODY_OK
                                                                        : NBODY_ERR_INVALID_ARG;
    }
    if (path == NBODY_PATH_TILED) {
        const int variant = o.variant < 0 ? kDefaultTiledVariant : o.variant;
        if (variant >= nbody::tiled_variant_count() || variant >= kMaxVariants)
            return NBODY_ERR_INVALID_ARG;
        plan_tiled(nt, ns, sm, occ.tiled[variant], variant, o.splits, p);
        return NBODY_OK;
    }
    if (o.splits != 0) return NBODY_ERR_INVALID_ARG;   // the cluster path plans its own split
    if (o.variant >= nbody::cluster_variant_count()) return NBODY_ERR_INVALID_ARG;
    // The cost model picks the cluster size well but ranks the kernel
    // variants poorly; measured inside CUDA graphs on GB300, variant 0 is the
    // fastest or within a few percent from 1024 to 6144 bodies, so automatic
    // planning uses it and a forced variant is honoured.
    const int only = o.variant >= 0 ? o.variant : kDefaultClusterVariant;
    double best = INFINITY;
    for (int v = 0; v < nbody::cluster_variant_count(); ++v) {
        if (v != only) continue;
        nbody_plan cand;
        double t;
        plan_cluster_variant(nt, ns, sm, occ.cluster[v], v, &cand, &t);
        if (t < best * (1.0 - 1e-3)) {
            best = t;
            *p = cand;
        }
    }
    // a forced whole-range variant whose range cannot fit shared memory
    return std::isfinite(best) ? NBODY_OK : NBODY_ERR_INVALID_ARG;
}

// Launch a planned force evaluation; `scratch` holds plan.scratch_bytes when
// that is not 0.
cudaError_t launch_planned(const nbody_plan &plan, const nbody::Problem &pr, float4 *out,
                           float4 *scratch, int sm_count, cudaStream_t stream) {
    if (plan.path == NBODY_PATH_SYMMETRIC) {
        const int block = plan.threads * plan.i_per_thread;
        if (plan.scratch_bytes == 0)   // one block, one piece: no partials
            return nbody::launch_sym(plan.variant, pr.targets, pr.nt, pr.eps2, plan.num_iblocks, 1,
                                     out, nullptr, stream);
        float4 *jpart = scratch + static_cast<int64_t>(plan.splits) * pr.nt;
        cudaError_t e = nbody::launch_sym(plan.variant, pr.targets, pr.nt, pr.eps2,
                                          plan.num_iblocks, plan.splits, scratch, jpart, stream);
        if (e == cudaSuccess)
            e = nbody::launch_reduce_sym(scratch, plan.splits, jpart, pr.nt, block,
                                         plan.num_iblocks, out, sm_count, stream);
        return e;
    }
    const int ntiles = static_cast<int>(ceil_div(pr.ns, plan.tile));
    if (plan.path == NBODY_PATH_CLUSTER)
        return nbody::launch_cluster(plan.variant, pr, plan.num_iblocks, plan.cluster,
                                     plan.tiles_per_split, ntiles, out, stream);
    if (plan.splits == 1)
        return nbody::launch_tiled(plan.variant, pr, plan.num_iblocks, 1, plan.tiles_per_split,
                                   ntiles, out, stream);
    cudaError_t e = nbody::launch_tiled(plan.variant, pr, plan.num_iblocks, plan.splits,
                                        plan.tiles_per_split, ntiles, scratch, stream);
    if (e == cudaSuccess) e = nbody::launch_reduce_splits(scratch, pr.nt, plan.splits, out, sm_count, stream);
    return e;
}

// One time step: the planned force evaluation, then the Euler update.  When
// the plan ends in a reduction kernel, the update runs inside it, body by
// body, as each final (a, p) is formed (same arithmetic, one launch and one
// pass over the bodies fewer); otherwise the Euler kernel follows.
cudaError_t launch_step(const nbody_plan &plan, const nbody::Problem &pr, float4 *acc,
                        float4 *scratch, int sm_count, float4 *pos, float4 *vel, float dt,
                        cudaStream_t stream) {
    const nbody::EulerFuse eu = {pos, vel, dt};
    if (plan.path == NBODY_PATH_SYMMETRIC && plan.scratch_bytes > 0) {
        const int block = plan.threads * plan.i_per_thread;
        float4 *jpart = scratch + static_cast<int64_t>(plan.splits) * pr.nt;
        cudaError_t e = nbody::launch_sym(plan.variant, pr.targets, pr.nt, pr.eps2,
                                          plan.num_iblocks, plan.splits, scratch, jpart, stream);
        if (e == cudaSuccess)
            e = nbody::launch_reduce_sym(scratch, plan.splits, jpart, pr.nt, block,
                                         plan.num_iblocks, acc, sm_count, stream, &eu);
        return e;
    }
    if (plan.path == NBODY_PATH_TILED && plan.splits > 1) {
        const int ntiles = static_cast<int>(ceil_div(pr.ns, plan.tile));
        cudaError_t e = nbody::launch_tiled(plan.variant, pr, plan.num_iblocks, plan.splits,
                                            plan.tiles_per_split, ntiles, scratch, stream);
        if (e == cudaSuccess)
            e = nbody::launch_reduce_splits(scratch, pr.nt, plan.splits, acc, sm_count, stream, &eu);
        return e;
    }
    cudaError_t e = launch_planned(plan, pr, acc, scratch, sm_count, stream);
    if (e == cudaSuccess) e = nbody::launch_euler(pos, vel, acc, pr.nt, dt, sm_count, stream);
    return e;
}

Occupancy device_occupancy(const DeviceState *dev) {
    return {dev->tiled_occ, dev->cluster_occ, dev->sym_occ};
}

// Launch one planned force evaluation (targets x sources) on `stream`, with
// its split partials in stream-ordered memory from the device's pool.
nbody_status run_forces(const nbody::Problem &pr, const nbody_forces_opts *opts, float *result,
                        cudaStream_t stream) {
    DeviceState *dev = nullptr;
    nbody_status st = device_state(&dev);
    if (st != NBODY_OK) return st;
    nbody_plan plan;
    const bool all_pairs = pr.targets == pr.sources && pr.nt == pr.ns;
    if ((st = make_plan(pr.nt, pr.ns, all_pairs, dev->sm_count, device_occupancy(dev), opts,
                        &plan)) != NBODY_OK)
        return st;
    float4 *out = reinterpret_cast<float4 *>(result);
    void *scratch = nullptr;
    cudaError_t e;
    if (plan.scratch_bytes > 0) {
        e = cudaMallocFromPoolAsync(&scratch, static_cast<size_t>(plan.scratch_bytes), dev->pool,
                                    stream);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    e = launch_planned(plan, pr, out, static_cast<float4 *>(scratch), dev->sm_count, stream);
    if (scratch != nullptr) {
        const cudaError_t ef = cudaFreeAsync(scratch, stream);
        if (e == cudaSuccess) e = ef;
    }
    return e == cudaSuccess ? NBODY_OK : cuda_fail(e);
}

// ---------------------------------------------------------------- multi-step driver
//
// One step (forces, then Euler) is captured once into a CUDA graph on an
// internal stream and replayed `steps` times on the caller's stream, so a
// step costs one graph launch instead of two or three kernel launches from
// the host.  Where the forces end in a reduction kernel (the symmetric path,
// or the tiled path with split sources), the Euler update runs inside it.
// On the cluster path (small N) a second graph holds two steps whose Euler
// update is fused into the force kernel, the positions going from pos_mass
// to a library-owned second buffer and back; steps run in pairs through it,
// and an odd last step through the one-step graph.  One graph per device is
// cached, keyed by every argument but the step count; its split scratch (if
// any) lives as long as the graph.  When the key changes, the old graph is
// destroyed (deferred until it finishes) and its scratch freed in stream
// order behind its last launch.

struct SimKey {
    const float *pm;
    float *vel;
    float *acc;
    int64_t n;
    float eps2;
    float dt;
    bool operator==(const SimKey &o) const {
        return pm == o.pm && vel == o.vel && acc == o.acc && n == o.n &&
               std::memcmp(&eps2, &o.eps2, sizeof(float)) == 0 &&
               std::memcmp(&dt, &o.dt, sizeof(float)) == 0;
    }
};

struct SimGraph {
    bool valid = false;
    SimKey key = {};
    cudaGraphExec_t exec = nullptr;    // one step: forces (+ reduction), then Euler
    cudaGraphExec_t exec2 = nullptr;   // small N: two steps with Euler fused into the forces
    void *scratch = nullptr;           // split partials (tiled path)
    void *pos_b = nullptr;             // second position buffer of the fused steps
    cudaEvent_t done = nullptr;        // recorded after the latest replay
};

std::mutex g_sim_mu;
SimGraph g_sim[kMaxDevices];
cudaStream_t g_capture[kMaxDevices] = {};

nbody_status sim_release(SimGraph &g, cudaStream_t stream) {
    cudaError_t e = cudaSuccess;
    for (cudaGraphExec_t *x : {&g.exec, &g.exec2}) {
        if (*x != nullptr) {
            const cudaError_t ex = cudaGraphExecDestroy(*x);
            if (e == cudaSuccess) e = ex;
            *x = nullptr;
        }
    }
    if ((g.scratch != nullptr || g.pos_b != nullptr) && g.done != nullptr)
        cudaStreamWaitEvent(stream, g.done, 0);
    for (void **b : {&g.scratch, &g.pos_b}) {
        if (*b != nullptr) {
            const cudaError_t ef = cudaFreeAsync(*b, stream);
            if (e == cudaSuccess) e = ef;
            *b = nullptr;
        }
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

nbody_status sim_build(int dev_id, DeviceState *dev, const SimKey &k, SimGraph &g,
                       cudaStream_t stream) {
    nbody_plan plan;
    nbody_status st = make_plan(k.n, k.n, true, dev->sm_count, device_occupancy(dev), nullptr,
                                &plan);
    if (st != NBODY_OK) return st;
    cudaError_t e;
    if (g_capture[dev_id] == nullptr &&
        (e = cudaStreamCreateWithFlags(&g_capture[dev_id], cudaStreamNonBlocking)) != cudaSuccess)
        return cuda_fail(e);
    if (g.done == nullptr && (e = cudaEventCreateWithFlags(&g.done, cudaEventDisableTiming)) != cudaSuccess)
        return cuda_fail(e);
    void *scratch = nullptr;
    if (plan.scratch_bytes > 0) {
        e = cudaMallocFromPoolAsync(&scratch, static_cast<size_t>(plan.scratch_bytes), dev->pool,
                                    stream);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    const cudaStream_t cap = g_capture[dev_id];
    const int ni = static_cast<int>(k.n);
    float4 *pos = reinterpret_cast<float4 *>(const_cast<float *>(k.pm));
    float4 *vel = reinterpret_cast<float4 *>(k.vel);
    float4 *acc = reinterpret_cast<float4 *>(k.acc);
    const nbody::Problem pr = {k.pm, k.pm, ni, ni, k.eps2};
    cudaGraphExec_t exec = nullptr, exec2 = nullptr;
    e = capture_graph(cap, [&](cudaStream_t st) {
        return launch_step(plan, pr, acc, static_cast<float4 *>(scratch), dev->sm_count, pos, vel,
                           k.dt, st);
    }, &exec);
    // Small N: two steps per replay with the Euler update fused into the
    // cluster kernel, positions alternating between pos_mass and pos_b.
    void *pos_b = nullptr;
    if (e == cudaSuccess && plan.path == NBODY_PATH_CLUSTER) {
        e = cudaMallocFromPoolAsync(&pos_b, static_cast<size_t>(16 * k.n), dev->pool, stream);
        if (e == cudaSuccess) {
            float4 *pb = static_cast<float4 *>(pos_b);
            const nbody::Problem pr_b = {reinterpret_cast<const float *>(pb),
                                         reinterpret_cast<const float *>(pb), ni, ni, k.eps2};
            const int ntiles = static_cast<int>(ceil_div(k.n, plan.tile));
            const nbody::EulerFuse to_b = {pb, vel, k.dt};
            const nbody::EulerFuse to_a = {pos, vel, k.dt};
            e = capture_graph(cap, [&](cudaStream_t st) {
                cudaError_t el = nbody::launch_cluster(plan.variant, pr, plan.num_iblocks,
                                                       plan.cluster, plan.tiles_per_split, ntiles,
                                                       acc, st, &to_b);
                if (el == cudaSuccess)
                    el = nbody::launch_cluster(plan.variant, pr_b, plan.num_iblocks, plan.cluster,
                                               plan.tiles_per_split, ntiles, acc, st, &to_a);
                return el;
            }, &exec2);
        }
    }
    if (e != cudaSuccess) {
        if (exec != nullptr) cudaGraphExecDestroy(exec);
        if (scratch != nullptr) cudaFreeAsync(scratch, stream);
        if (pos_b != nullptr) cudaFreeAsync(pos_b, stream);
        return cuda_fail(e);
    }
    g.key = k;
    g.exec = exec;
    g.exec2 = exec2;
    g.scratch = scratch;
    g.pos_b = pos_b;
    g.valid = true;
    return NBODY_OK;
}

// Nominal occupancy of each tiled variant (used by the host-only planner
// entry point when the caller gives none): register-limited at 64K per SM.
int nominal_occ(int i_per_thread, int threads) {
    const int regs = i_per_thread >= 8 ? 168 : (i_per_thread >= 4 ? 96 : 64);
    int occ = 65536 / (regs * threads);
    return occ < 1 ? 1 : occ;
}

}  // namespace

// ======================================================================= C ABI

extern "C" {

const char *nbody_status_string(nbody_status s) {
    switch (s) {
        case NBODY_OK: return "NBODY_OK";
        case NBODY_ERR_INVALID_ARG: return "NBODY_ERR_INVALID_ARG: invalid argument";
        case NBODY_ERR_MISALIGNED: return "NBODY_ERR_MISALIGNED: body array not 16-byte aligned";
        case NBODY_ERR_ALIAS: return "NBODY_ERR_ALIAS: output overlaps an input";
        case NBODY_ERR_CUDA: return "NBODY_ERR_CUDA: CUDA runtime error";
        case NBODY_ERR_TIMEOUT: return "NBODY_ERR_TIMEOUT: bounded device wait ran out";
        case NBODY_ERR_DEVICE: return "NBODY_ERR_DEVICE: current device is not sm_103";
        case NBODY_ERR_TOO_LARGE:
            return "NBODY_ERR_TOO_LARGE: n exceeds the fixed scratch of nbody_forces_noalloc";
    }
    return "NBODY_ERR_UNKNOWN";
}

int nbody_last_cuda_error(void) { return g_last_cuda_error; }

nbody_status nbody_plan_forces(int64_t n, int32_t sm_count, int32_t ctas_per_sm,
                               const nbody_forces_opts *opts, nbody_plan *plan) {
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
    return make_plan(n, n, true, sm_count, Occupancy{occ, cocc, socc}, opts, plan);
}

nbody_status nbody_forces_ex(const float *pos_mass, int64_t n, float eps2, float *acc_pot,
                             const nbody_forces_opts *opts, cudaStream_t stream) {
    nbody_status st = check_forces(pos_mass, n, eps2, acc_pot);
    if (st != NBODY_OK || n == 0) return st;
    const nbody::Problem pr = {pos_mass, pos_mass, static_cast<int>(n), static_cast<int>(n), eps2};
    return run_forces(pr, opts, acc_pot, stream);
}

nbody_status nbody_forces_ts(const float *targets, int64_t nt, const float *sources, int64_t ns,
                             float eps2, float *out, cudaStream_t stream) {
    if (check_n(nt) != NBODY_OK || check_n(ns) != NBODY_OK) return NBODY_ERR_INVALID_ARG;
    if (nt == 0) return NBODY_OK;
    if (targets == nullptr || out == nullptr || (ns > 0 && sources == nullptr))
        return NBODY_ERR_INVALID_ARG;
    if (!std::isfinite(eps2) || !(eps2 >= FLT_MIN)) return NBODY_ERR_INVALID_ARG;
    if (!aligned16(targets) || !aligned16(out) || (ns > 0 && !aligned16(sources)))
        return NBODY_ERR_MISALIGNED;
    if (overlap(out, targets, 16 * nt)) return NBODY_ERR_ALIAS;
    if (ns > 0 && overlap2(out, 16 * nt, sources, 16 * ns)) return NBODY_ERR_ALIAS;
    if (ns == 0) {   // no sources: every sum is empty
        const cudaError_t e = cudaMemsetAsync(out, 0, static_cast<size_t>(16 * nt), stream);
        return e == cudaSuccess ? NBODY_OK : cuda_fail(e);
    }
    const nbody::Problem pr = {targets, sources, static_cast<int>(nt), static_cast<int>(ns), eps2};
    return run_forces(pr, nullptr, out, stream);
}

nbody_status nbody_simulate(float *pos_mass, float *vel, float *acc_pot, int64_t n, float eps2,
                            float dt, int64_t steps, cudaStream_t stream) {
    nbody_status st = check_forces(pos_mass, n, eps2, acc_pot);
    if (st != NBODY_OK) return st;
    if (steps < 0 || !std::isfinite(dt)) return NBODY_ERR_INVALID_ARG;
    if (n == 0 || steps == 0) return NBODY_OK;
    if (vel == nullptr) return NBODY_ERR_INVALID_ARG;
    if (!aligned16(vel)) return NBODY_ERR_MISALIGNED;
    if (overlap(vel, pos_mass, 16 * n) || overlap(vel, acc_pot, 16 * n)) return NBODY_ERR_ALIAS;
    DeviceState *dev = nullptr;
    if ((st = device_state(&dev)) != NBODY_OK) return st;
    int dev_id = 0;
    cudaError_t e = cudaGetDevice(&dev_id);
    if (e != cudaSuccess) return cuda_fail(e);
    std::lock_guard<std::mutex> lock(g_sim_mu);
    SimGraph &g = g_sim[dev_id];
    const SimKey key = {pos_mass, vel, acc_pot, n, eps2, dt};
    if (!(g.valid && g.key == key)) {
        if (g.valid && (st = sim_release(g, stream)) != NBODY_OK) return st;
        if ((st = sim_build(dev_id, dev, key, g, stream)) != NBODY_OK) return st;
    }
    int64_t left = steps;
    if (g.exec2 != nullptr)
        for (; left >= 2; left -= 2)
            if ((e = cudaGraphLaunch(g.exec2, stream)) != cudaSuccess) return cuda_fail(e);
    for (; left > 0; --left)
        if ((e = cudaGraphLaunch(g.exec, stream)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaEventRecord(g.done, stream)) != cudaSuccess) return cuda_fail(e);
    return NBODY_OK;
}

nbody_status nbody_forces(const float *pos_mass, int64_t n, float eps2, float *acc_pot,
                          cudaStream_t stream) {
    return nbody_forces_ex(pos_mass, n, eps2, acc_pot, nullptr, stream);
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
