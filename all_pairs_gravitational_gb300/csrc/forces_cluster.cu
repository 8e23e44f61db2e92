// forces_cluster.cu -- all-pairs softened gravity for small N: the source
// range of one target block is split across the warps of a CTA and across
// the CTAs of a thread-block cluster, and the partial sums are added back in
// a fixed order through shared memory and distributed shared memory (DSMEM).
// A forced path (NBODY_PATH_CLUSTER): the automatic choice takes the
// row-split kernel (forces_rows.cu), faster at every small size.
//
// With one thread per target, N = 1024 bodies would occupy a few SMs of 152
// (the GPU Gems 3 ch.31 study page, section 4, splits a body's row over
// several threads below about 4096 bodies and merges the partial
// accelerations).  Here a cluster of C CTAs shares one block of BI = 32 K
// targets; CTA c takes source tiles [c T, c T + T) and warp w of it takes
// the w-th slice of them, so C * W pieces of the source range run in
// parallel, for N * BI / (C * W) pairs each.
//
// Two ways to feed the warps:
//   * tiled (forces_cluster_kernel): 128-body tiles through a 3-stage cp.async
//     ring, warp w taking the w-th slice of every tile;
//   * whole range (forces_cluster_whole_kernel): the CTA's entire range staged
//     into dynamic shared memory at once, one barrier, warp w taking the
//     w-th contiguous slice.
//
// Optionally (nbody_simulate) the kernel also applies the Euler step to each
// target as it stores its result, writing the new position to a second
// buffer, so that a small-N time step is one launch instead of two.
//
// Reduction, deterministic and without atomics or global scratch:
//   0. every thread arrives at a cluster barrier when the kernel starts;
//   1. after the pair loop each warp folds its fp32 partials into Kahan
//      totals and writes them to shared memory, and the CTA adds its W warp
//      partials in the order w = 0 .. W-1;
//   2. after waiting on the start barrier (every CTA of the cluster has
//      started, so its shared memory exists), the CTA stores each target's
//      partial straight into the inbox of the CTA that owns that target
//      (CTA c owns slice c of the target block), in the sender's slot;
//   3. a second cluster barrier (release / acquire) makes the stores
//      visible, and each owner adds its inbox in rank order 0 .. C-1,
//      compensated, and stores the result.
//   No CTA touches another's shared memory after step 3's barrier, so none
//   has to wait for the others before exiting (one cluster barrier fewer
//   than reading the partials from the other CTAs).
#include <algorithm>

#include "nbody_device.cuh"
#include "nbody_internal.h"

namespace nbody {

// Dynamic shared memory of the whole-range kernel: the staged range, the
// per-warp partials and the inbox of the cluster reduction.
size_t whole_smem_bytes(int K, int W, int tiles_per_cta) {
    return static_cast<size_t>(tiles_per_cta) * 128 * 32 + static_cast<size_t>(W + 1) * 32 * K * 16;
}

namespace {

constexpr int kStages = 3;
constexpr int kClusterTile = 128;   // source tile of the cluster path (both kernels)
constexpr int kFoldJ = 32;          // sources between folds of a warp's partials

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

__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Store a float4 into the shared memory of CTA `rank` of this cluster, at
// the offset `local` has in this CTA's shared memory.
__device__ __forceinline__ void st_dsmem_f4(void *local, uint32_t rank, float4 v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};"
                 :: "r"(remote), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w) : "memory");
}

__device__ __forceinline__ void kahan4(float4 &h, float4 &c, const float4 &v) {
    kahan1(h.x, c.x, v.x);
    kahan1(h.y, c.y, v.y);
    kahan1(h.z, c.z, v.z);
    kahan1(h.w, c.w, v.w);
}

// One warp's accumulators for K targets per lane, KP = K/2 f32x2 pairs.
template <int KP>
struct WarpAcc {
    f2 ax[KP], ay[KP], az[KP], pp[KP];   // fp32 partials since the last fold
    f2 hx[KP], hy[KP], hz[KP], hp[KP];   // Kahan totals ...
    f2 lx[KP], ly[KP], lz[KP], lp[KP];   // ... and corrections

    __device__ __forceinline__ void init() {
#pragma unroll
        for (int q = 0; q < KP; ++q) {
            ax[q] = ay[q] = az[q] = pp[q] = 0ull;
            hx[q] = hy[q] = hz[q] = hp[q] = 0ull;
            lx[q] = ly[q] = lz[q] = lp[q] = 0ull;
        }
    }

    // Sources [j_begin, j_end) of a duplicated shared-memory run.
    template <bool POT>
    __device__ __forceinline__ void run(const float4 *s4, int j_begin, int j_end, const f2 (&xi)[KP],
                                        const f2 (&yi)[KP], const f2 (&zi)[KP], f2 e2) {
#pragma unroll 4
        for (int jj = j_begin; jj < j_end; ++jj) {
            const Src sj = load_src(s4, jj);
#pragma unroll
            for (int q = 0; q < KP; ++q) {
                const Geom g = pair_geom(sj, xi[q], yi[q], zi[q], e2);
                const f2 tm = pair_accumulate(g, sj.m, ax[q], ay[q], az[q]);
                if (POT) pp[q] = f2_add(pp[q], tm);
            }
        }
    }

    __device__ __forceinline__ void fold_acc() {
#pragma unroll
        for (int q = 0; q < KP; ++q) {
            f2_kahan_fold(hx[q], lx[q], ax[q]);
            f2_kahan_fold(hy[q], ly[q], ay[q]);
            f2_kahan_fold(hz[q], lz[q], az[q]);
        }
    }

    __device__ __forceinline__ void fold_pot() {
#pragma unroll
        for (int q = 0; q < KP; ++q) f2_kahan_fold(hp[q], lp[q], pp[q]);
    }
};

// Steps 1-3 of the reduction: warp partials -> CTA partial -> the owner
// CTAs' inboxes -> out[ib * BI + slot] for this CTA's slice of the target
// block.  `red` holds W * 32 K records (warp partials), `box` 32 K (the
// inbox: [sender rank][slot within a slice]).
template <int K, int W, bool POT, bool EULER>
__device__ __forceinline__ void reduce_and_store(WarpAcc<K / 2> &acc, float4 *red, float4 *box,
                                                 int ib, const Problem &pr,
                                                 float4 *__restrict__ out, const EulerFuse &eu) {
    constexpr int KP = K / 2;
    constexpr int BI = 32 * K;
    constexpr int NT = W * 32;
    const int tid = static_cast<int>(threadIdx.x);
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const uint32_t crank = cluster_ctarank();
    const uint32_t csize = cluster_nctarank();
    const int per = BI / static_cast<int>(csize);
    // 1. warp partials to shared memory: slot k * 32 + lane is target ib * BI + slot
#pragma unroll
    for (int q = 0; q < KP; ++q) {
        float x0, x1, y0, y1, z0, z1, p0 = 0.f, p1 = 0.f;
        f2_unpack(f2_sub(acc.hx[q], acc.lx[q]), x0, x1);
        f2_unpack(f2_sub(acc.hy[q], acc.ly[q]), y0, y1);
        f2_unpack(f2_sub(acc.hz[q], acc.lz[q]), z0, z1);
        if (POT) f2_unpack(f2_sub(acc.hp[q], acc.lp[q]), p0, p1);
        red[warp * BI + (2 * q) * 32 + lane] = make_float4(x0, y0, z0, p0);
        red[warp * BI + (2 * q + 1) * 32 + lane] = make_float4(x1, y1, z1, p1);
    }
    __syncthreads();
    // 2. the CTA partial over warps 0 .. W-1, stored into the owner's inbox
    cluster_wait();   // every CTA of the cluster has started
    for (int slot = tid; slot < BI; slot += NT) {
        float4 h = red[slot];
        float4 c = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 1; w < W; ++w) kahan4(h, c, red[w * BI + slot]);
        st_dsmem_f4(&box[static_cast<int>(crank) * per + slot % per],
                    static_cast<uint32_t>(slot / per),
                    make_float4(__fsub_rn(h.x, c.x), __fsub_rn(h.y, c.y), __fsub_rn(h.z, c.z),
                                __fsub_rn(h.w, c.w)));
    }
    // 3. every store of the cluster is visible: this CTA's slice, rank order
    cluster_sync();
    for (int t = tid; t < per; t += NT) {
        float4 h = make_float4(0.f, 0.f, 0.f, 0.f);
        float4 c = h;
        for (uint32_t r = 0; r < csize; ++r) kahan4(h, c, box[static_cast<int>(r) * per + t]);
        const int slot = static_cast<int>(crank) * per + t;
        const int64_t i = static_cast<int64_t>(ib) * BI + slot;
        if (i < pr.nt) {
            const float4 a = make_float4(__fsub_rn(h.x, c.x), __fsub_rn(h.y, c.y),
                                         __fsub_rn(h.z, c.z), POT ? -__fsub_rn(h.w, c.w) : 0.f);
            out[i] = a;
            if (EULER) {   // the step of euler.cu, on this body, positions first
                float4 x = __ldg(reinterpret_cast<const float4 *>(pr.targets) + i);
                float4 v = eu.vel[i];
                euler_body(x, v, a, eu.dt);
                eu.pos_out[i] = x;
                eu.vel[i] = v;
            }
        }
    }
}

template <int K, int W, int P, bool POT, bool EULER>
__global__ void __launch_bounds__(W * 32)
forces_cluster_kernel(const Problem pr, int tiles_per_cta, int ntiles,
                      float4 *__restrict__ out, const EulerFuse eu) {
    static_assert(K % 2 == 0, "targets are processed in f32x2 pairs");
    constexpr int KP = K / 2;
    constexpr int NT = W * 32;
    constexpr int BI = 32 * K;          // targets per cluster
    constexpr int JW = P / W;           // sources per warp per tile
    constexpr int FOLD_P = 8;           // tiles between folds of the potential
    static_assert(P % W == 0 && JW <= kFoldJ, "tile must split evenly, <= 32 sources per warp");

    __shared__ __align__(16) float sdup[kStages][P * 8];
    __shared__ __align__(16) float4 red[W * BI];
    __shared__ __align__(16) float4 box[BI];
    pdl_wait_and_release();
    cluster_arrive_relaxed();   // matched by the wait before the partials are pushed

    const int warp = static_cast<int>(threadIdx.x) >> 5;
    const int lane = static_cast<int>(threadIdx.x) & 31;
    const int ib = static_cast<int>(blockIdx.x / cluster_nctarank());
    const int t_begin = static_cast<int>(cluster_ctarank()) * tiles_per_cta;
    const int t_end = min(t_begin + tiles_per_cta, ntiles);

    f2 xi[KP], yi[KP], zi[KP];
    load_targets<KP>(pr.targets, pr.nt, static_cast<int64_t>(ib) * BI + lane, 32, xi, yi, zi);
    const f2 e2 = f2_pack(pr.eps2, pr.eps2);
    WarpAcc<KP> acc;
    acc.init();

    if (t_begin < t_end) stage_tile<NT, P>(sdup[0], pr.sources, pr.ns, t_begin);
    cp_async_commit();
    if (t_begin + 1 < t_end) stage_tile<NT, P>(sdup[1], pr.sources, pr.ns, t_begin + 1);
    cp_async_commit();

    int stage = 0;
    for (int t = t_begin; t < t_end; ++t) {
        const int k = t - t_begin;
        cp_async_wait<1>();
        __syncthreads();
        {
            int s2 = stage + 2;
            if (s2 >= kStages) s2 -= kStages;
            if (t + 2 < t_end) stage_tile<NT, P>(sdup[s2], pr.sources, pr.ns, t + 2);
            cp_async_commit();
        }
        const float4 *s4 = reinterpret_cast<const float4 *>(sdup[stage]);
        acc.template run<POT>(s4, warp * JW, (warp + 1) * JW, xi, yi, zi, e2);
        acc.fold_acc();                                   // every warp slice (<= 32 sources)
        if (POT && ((k + 1) % FOLD_P == 0 || t + 1 == t_end)) acc.fold_pot();
        stage = (stage + 1 == kStages) ? 0 : stage + 1;
    }
    cp_async_wait<0>();
    reduce_and_store<K, W, POT, EULER>(acc, red, box, ib, pr, out, eu);
}

// Whole-range variant: see the file header.  The CTA's range is
// tiles_per_cta * 128 bodies (a few thousand at most for the N this path
// serves), zero-filled past ns.
template <int K, int W, bool POT, bool EULER>
__global__ void __launch_bounds__(W * 32)
forces_cluster_whole_kernel(const Problem pr, int tiles_per_cta, float4 *__restrict__ out,
                            const EulerFuse eu) {
    static_assert(K % 2 == 0, "targets are processed in f32x2 pairs");
    constexpr int KP = K / 2;
    constexpr int NT = W * 32;
    constexpr int BI = 32 * K;

    extern __shared__ __align__(16) float4 dyn[];
    pdl_wait_and_release();
    cluster_arrive_relaxed();   // matched by the wait before the partials are pushed
    const int jc = tiles_per_cta * kClusterTile;          // sources staged by this CTA
    float *sdup = reinterpret_cast<float *>(dyn);          // jc bodies x 8 floats
    float4 *red = dyn + 2 * jc;
    float4 *box = red + W * BI;

    const int warp = static_cast<int>(threadIdx.x) >> 5;
    const int lane = static_cast<int>(threadIdx.x) & 31;
    const int ib = static_cast<int>(blockIdx.x / cluster_nctarank());
    const int64_t j0 = static_cast<int64_t>(cluster_ctarank()) * jc;

    stage_sources<NT>(sdup, pr.sources, pr.ns, j0, jc);
    cp_async_commit();

    f2 xi[KP], yi[KP], zi[KP];
    load_targets<KP>(pr.targets, pr.nt, static_cast<int64_t>(ib) * BI + lane, 32, xi, yi, zi);
    const f2 e2 = f2_pack(pr.eps2, pr.eps2);
    WarpAcc<KP> acc;
    acc.init();

    cp_async_wait<0>();
    __syncthreads();

    // warp slice: jw sources (jc / W, a multiple of 16), folded every 32
    const int jw = jc / W;
    const float4 *s4 = reinterpret_cast<const float4 *>(sdup) + 2 * (warp * jw);
    for (int jb = 0; jb < jw; jb += kFoldJ) {
        acc.template run<POT>(s4, jb, min(jb + kFoldJ, jw), xi, yi, zi, e2);
        acc.fold_acc();
        if (POT) acc.fold_pot();
    }
    reduce_and_store<K, W, POT, EULER>(acc, red, box, ib, pr, out, eu);
}

template <int K, int W, int P>
cudaError_t launch_tiled_cluster(const Problem &pr, int num_ib, int cluster, int tpc, int ntiles,
                                 float4 *out, cudaStream_t stream, const EulerFuse *eu) {
    const dim3 grid(static_cast<unsigned>(num_ib) * static_cast<unsigned>(cluster));
    const dim3 block(W * 32);
    const unsigned cx = static_cast<unsigned>(cluster);
    const EulerFuse none = {nullptr, nullptr, 0.f};
    if (eu != nullptr)
        return pr.pot ? launch_pdl(forces_cluster_kernel<K, W, P, true, true>, grid, block, 0,
                                   stream, cx, pr, tpc, ntiles, out, *eu)
                      : launch_pdl(forces_cluster_kernel<K, W, P, false, true>, grid, block, 0,
                                   stream, cx, pr, tpc, ntiles, out, *eu);
    return pr.pot ? launch_pdl(forces_cluster_kernel<K, W, P, true, false>, grid, block, 0, stream,
                               cx, pr, tpc, ntiles, out, none)
                  : launch_pdl(forces_cluster_kernel<K, W, P, false, false>, grid, block, 0, stream,
                               cx, pr, tpc, ntiles, out, none);
}

template <int K, int W>
cudaError_t launch_whole(const Problem &pr, int num_ib, int cluster, int tpc, float4 *out,
                         cudaStream_t stream, const EulerFuse *eu) {
    const dim3 grid(static_cast<unsigned>(num_ib) * static_cast<unsigned>(cluster));
    const dim3 block(W * 32);
    const size_t smem = whole_smem_bytes(K, W, tpc);
    const unsigned cx = static_cast<unsigned>(cluster);
    const EulerFuse none = {nullptr, nullptr, 0.f};
    if (eu != nullptr)
        return pr.pot ? launch_pdl(forces_cluster_whole_kernel<K, W, true, true>, grid, block,
                                   smem, stream, cx, pr, tpc, out, *eu)
                      : launch_pdl(forces_cluster_whole_kernel<K, W, false, true>, grid, block,
                                   smem, stream, cx, pr, tpc, out, *eu);
    return pr.pot ? launch_pdl(forces_cluster_whole_kernel<K, W, true, false>, grid, block, smem,
                               stream, cx, pr, tpc, out, none)
                  : launch_pdl(forces_cluster_whole_kernel<K, W, false, false>, grid, block, smem,
                               stream, cx, pr, tpc, out, none);
}

#define NBODY_CLUSTER(K, W, P)                                                             \
    {K, W, P, false, reinterpret_cast<const void *>(&forces_cluster_kernel<K, W, P, true, false>), \
     reinterpret_cast<const void *>(&forces_cluster_kernel<K, W, P, false, false>)}
#define NBODY_CLUSTER_WHOLE(K, W)                                                          \
    {K, W, kClusterTile, true,                                                             \
     reinterpret_cast<const void *>(&forces_cluster_whole_kernel<K, W, true, false>),      \
     reinterpret_cast<const void *>(&forces_cluster_whole_kernel<K, W, false, false>)}

const ClusterVariant kVariants[] = {
    NBODY_CLUSTER(2, 4, 128),   // 0: default
    NBODY_CLUSTER(4, 4, 128),   // 1
    NBODY_CLUSTER(2, 8, 128),   // 2
    NBODY_CLUSTER(4, 8, 128),   // 3
    NBODY_CLUSTER_WHOLE(2, 4),  // 4: whole source range staged at once
    NBODY_CLUSTER_WHOLE(4, 4),  // 5
    NBODY_CLUSTER_WHOLE(2, 8),  // 6
    NBODY_CLUSTER_WHOLE(4, 8),  // 7
};

#undef NBODY_CLUSTER
#undef NBODY_CLUSTER_WHOLE

}  // namespace

int cluster_variant_count() { return static_cast<int>(sizeof(kVariants) / sizeof(kVariants[0])); }

const ClusterVariant &cluster_variant(int v) { return kVariants[v]; }

cudaError_t launch_cluster(int variant, const Problem &pr, int num_ib, int cluster,
                           int tiles_per_cta, int ntiles, float4 *out, cudaStream_t stream,
                           const EulerFuse *eu) {
    const int tpc = tiles_per_cta;
    switch (variant) {
        case 0: return launch_tiled_cluster<2, 4, 128>(pr, num_ib, cluster, tpc, ntiles, out, stream, eu);
        case 1: return launch_tiled_cluster<4, 4, 128>(pr, num_ib, cluster, tpc, ntiles, out, stream, eu);
        case 2: return launch_tiled_cluster<2, 8, 128>(pr, num_ib, cluster, tpc, ntiles, out, stream, eu);
        case 3: return launch_tiled_cluster<4, 8, 128>(pr, num_ib, cluster, tpc, ntiles, out, stream, eu);
        case 4: return launch_whole<2, 4>(pr, num_ib, cluster, tpc, out, stream, eu);
        case 5: return launch_whole<4, 4>(pr, num_ib, cluster, tpc, out, stream, eu);
        case 6: return launch_whole<2, 8>(pr, num_ib, cluster, tpc, out, stream, eu);
        case 7: return launch_whole<4, 8>(pr, num_ib, cluster, tpc, out, stream, eu);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace nbody
