// forces_rows.cu -- softened gravity for few sources: the row of each target
// (its sum over every source) is split over the 32 lanes of a warp, and over
// S pieces of the source range, with every source held in shared memory.
//
// Below about ten thousand bodies, one thread per target leaves most of the
// GPU idle.  The GPU Gems 3 ch.31 study page (section 4) therefore splits a
// body's row over several threads and adds their partial accelerations.
// Here:
//   * the targets are cut into consecutive runs of TB = ceil(nt / SMs), one
//     CTA each, so that every SM gets the same share of the pairs;
//   * the CTA stages all ns sources into shared memory once, as four arrays
//     x[], y[], z[], m[], zero past ns (a zero mass adds exactly 0, since
//     |r|^2 + eps^2 > 0);
//   * a warp item is K targets, their coordinates the same in every lane,
//     against one piece of the sources.  Lane l takes the source pairs
//     (2c, 2c + 1) of the columns c = l, l + 32, ... of the piece: one f32x2
//     operation serves two sources, and a warp's 8-byte loads are
//     contiguous;
//   * at the end of an item, each lane adds its two halves, and the 4 K
//     values of the item (a and p of K targets) are added across the warp
//     by a fixed recursive-halving shuffle exchange (warp_sum_transposed);
//     the lanes holding the totals store the piece's sums in shared memory;
//   * after a barrier, thread t adds target t's S piece sums in order,
//     compensated, and stores (ax, ay, az, p); in nbody_simulate it then
//     applies the Euler step to that body.
// No atomics, no global scratch and no cluster: the results are
// deterministic.  A piece holds at most 2048 sources (the planner's rule;
// a forced piece count may exceed it), so a lane sums at most 32 terms per
// half before the exchange: the run length between the compensated folds of
// the other kernels.
#include <algorithm>

#include "nbody_device.cuh"
#include "nbody_internal.h"

namespace nbody {

size_t rows_smem_bytes(int ns_pad, int pieces, int tb_pad) {
    return 16ull * static_cast<size_t>(ns_pad) +
           16ull * static_cast<size_t>(pieces) * static_cast<size_t>(tb_pad);
}

namespace {

constexpr int kLoadBatch = 16;   // sources each thread loads before storing them

__device__ __forceinline__ void kahan4r(float4 &h, float4 &c, const float4 &v) {
    kahan1(h.x, c.x, v.x);
    kahan1(h.y, c.y, v.y);
    kahan1(h.z, c.z, v.z);
    kahan1(h.w, c.w, v.w);
}

__device__ __forceinline__ float4 source_or_zero(const float4 *__restrict__ src4, int j, int ns) {
    return j < ns ? __ldg(src4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
}

// Source j into the arrays x, y, z, m (stride sp floats).
__device__ __forceinline__ void put_source(float *xs, int sp, int j, const float4 &b) {
    xs[j] = b.x;
    xs[sp + j] = b.y;
    xs[2 * sp + j] = b.z;
    xs[3 * sp + j] = b.w;
}

// Sums each of the M values v[0..M) (M a power of two <= 32) over the 32
// lanes of the warp, in a fixed order, by recursive halving: at the exchange
// with the lane `o` away, the lower lane keeps the first half of its values
// and the upper lane the second, each adding its partner's copy of the half
// it keeps (M - 1 shuffles in all, against 5 M for a tree per value); plain
// butterfly exchanges finish once one value is left.  Afterwards lane l
// holds the total of value l / (32 / M).
template <int M>
__device__ __forceinline__ float warp_sum_transposed(float (&v)[M], int lane) {
#pragma unroll
    for (int h = M / 2, o = 16; h >= 1; h /= 2, o /= 2) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int q = 0; q < h; ++q) {
            const float send = up ? v[q] : v[q + h];
            const float keep = up ? v[q + h] : v[q];
            v[q] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, o));
        }
    }
    float x = v[0];
#pragma unroll
    for (int o = 16 / M; o >= 1; o /= 2) x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

// Smallest power of two >= x (x <= 32).
__host__ __device__ constexpr int pow2_at_least(int x) { return x <= 1 ? 1 : 2 * pow2_at_least((x + 1) / 2); }

// One warp item: K targets (the same in every lane) and their partial sums
// over the source columns this lane meets.
template <int K, int U, bool POT>
struct RowItem {
    f2 xi[K], yi[K], zi[K];
    f2 ax[K], ay[K], az[K], pp[K];

    __device__ __forceinline__ void init(const float4 (&tgt)[K]) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
            xi[k] = f2_pack(tgt[k].x, tgt[k].x);
            yi[k] = f2_pack(tgt[k].y, tgt[k].y);
            zi[k] = f2_pack(tgt[k].z, tgt[k].z);
            ax[k] = ay[k] = az[k] = pp[k] = 0ull;
        }
    }

    // Columns c, c + 32, ..., nsteps of them; column c holds sources 2c, 2c + 1.
    __device__ __forceinline__ void run(const float *xs, int sp, int c, int nsteps, f2 e2) {
        const f2 *xs2 = reinterpret_cast<const f2 *>(xs);
        const f2 *ys2 = reinterpret_cast<const f2 *>(xs + sp);
        const f2 *zs2 = reinterpret_cast<const f2 *>(xs + 2 * sp);
        const f2 *ms2 = reinterpret_cast<const f2 *>(xs + 3 * sp);
#pragma unroll U
        for (int st = 0; st < nsteps; ++st, c += 32) {
            const Src sj = {xs2[c], ys2[c], zs2[c], ms2[c]};
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const Geom gm = pair_geom(sj, xi[k], yi[k], zi[k], e2);
                const f2 tm = pair_accumulate(gm, sj.m, ax[k], ay[k], az[k]);
                if (POT) pp[k] = f2_add(pp[k], tm);
            }
        }
    }

    // Each lane's two halves, then the warp sums of the 4 K values (value
    // 4 k + c: component c of target k; zeros pad to M), stored as the
    // piece sums of the item's targets at `slot` (4 K floats).
    __device__ __forceinline__ void finish(float *slot, int lane) {
        constexpr int M = pow2_at_least(4 * K);
        float v[M];
#pragma unroll
        for (int k = 0; k < K; ++k) {
            float lo, hi;
            f2_unpack(ax[k], lo, hi);
            v[4 * k] = __fadd_rn(lo, hi);
            f2_unpack(ay[k], lo, hi);
            v[4 * k + 1] = __fadd_rn(lo, hi);
            f2_unpack(az[k], lo, hi);
            v[4 * k + 2] = __fadd_rn(lo, hi);
            f2_unpack(pp[k], lo, hi);
            v[4 * k + 3] = POT ? __fadd_rn(lo, hi) : 0.f;
        }
#pragma unroll
        for (int q = 4 * K; q < M; ++q) v[q] = 0.f;
        const float tot = warp_sum_transposed<M>(v, lane);
        constexpr int kLanesPerValue = 32 / M;
        const int idx = lane / kLanesPerValue;
        if (lane % kLanesPerValue == 0 && idx < 4 * K) slot[idx] = tot;
    }
};

template <int K, int W, int U, bool POT, bool EULER>
__global__ void __launch_bounds__(W * 32, 1)
forces_rows_kernel(const Problem pr, const RowsLaunch rl, float4 *__restrict__ out,
                   const EulerFuse eu) {
    constexpr int NT = W * 32;
    extern __shared__ __align__(16) float rsm[];
    const int sp = rl.ns_pad;                             // x, y, z, m at 0, sp, 2 sp, 3 sp
    float4 *red = reinterpret_cast<float4 *>(rsm + 4 * sp);   // [pieces][tb_pad]
    float *redf = rsm + 4 * sp;
    pdl_wait_and_release();

    const int tid = static_cast<int>(threadIdx.x);
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * rl.tb;
    const int tb = static_cast<int>(min(static_cast<int64_t>(rl.tb), static_cast<int64_t>(pr.nt) - t0));
    const float4 *t4 = reinterpret_cast<const float4 *>(pr.targets) + t0;
    const int items = rl.groups * rl.pieces;
    const f2 e2 = f2_pack(pr.eps2, pr.eps2);

    // The targets of this warp's first item, requested before the sources
    // (past the CTA's last target: copies of it, never stored).
    float4 tgt[K];
    if (warp < items) {
        const int g = warp / rl.pieces;
#pragma unroll
        for (int k = 0; k < K; ++k) tgt[k] = __ldg(t4 + min(g * K + k, tb - 1));
    }
    RowItem<K, U, POT> acc;
    // nbody_simulate: the position and velocity of the first target this
    // thread finishes, requested now so that the Euler step at the end does
    // not wait for them
    float4 x_pre = make_float4(0.f, 0.f, 0.f, 0.f), v_pre = x_pre;
    if (EULER && tid < tb) {
        x_pre = __ldg(t4 + tid);
        v_pre = eu.vel[t0 + tid];
    }

    // every source into the four arrays (zero past ns), then the warps'
    // items in turn
    const float4 *src4 = reinterpret_cast<const float4 *>(pr.sources);
    for (int j0 = 0; j0 < rl.ns_pad; j0 += NT * kLoadBatch) {
        float4 b[kLoadBatch];
#pragma unroll
        for (int r = 0; r < kLoadBatch; ++r) b[r] = source_or_zero(src4, j0 + r * NT + tid, pr.ns);
#pragma unroll
        for (int r = 0; r < kLoadBatch; ++r)
            if (j0 + r * NT + tid < rl.ns_pad) put_source(rsm, sp, j0 + r * NT + tid, b[r]);
    }
    __syncthreads();
    for (int it = warp; it < items; it += W) {
        const int g = it / rl.pieces;
        const int s = it - g * rl.pieces;
        if (it != warp) {
#pragma unroll
            for (int k = 0; k < K; ++k) tgt[k] = __ldg(t4 + min(g * K + k, tb - 1));
        }
        acc.init(tgt);
        acc.run(rsm, sp, s * rl.cols + lane, rl.cols / 32, e2);
        acc.finish(redf + 4 * (s * rl.tb_pad + g * K), lane);
    }
    __syncthreads();

    // each target's piece sums in order, compensated
    for (int t = tid; t < tb; t += NT) {
        float4 h = red[t];
        float4 c = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s = 1; s < rl.pieces; ++s) kahan4r(h, c, red[s * rl.tb_pad + t]);
        const float4 a = make_float4(__fsub_rn(h.x, c.x), __fsub_rn(h.y, c.y), __fsub_rn(h.z, c.z),
                                     POT ? -__fsub_rn(h.w, c.w) : 0.f);
        const int64_t i = t0 + t;
        out[i] = a;
        if (EULER) {   // the step of euler.cu, on this body, positions first
            float4 x = t == tid ? x_pre : __ldg(t4 + t);
            float4 v = t == tid ? v_pre : eu.vel[i];
            euler_body(x, v, a, eu.dt);
            eu.pos_out[i] = x;
            eu.vel[i] = v;
        }
    }
}

template <int K, int W, int U>
cudaError_t launch_rows_kw(const Problem &pr, const RowsLaunch &rl, float4 *out,
                           cudaStream_t stream, const EulerFuse *eu) {
    const dim3 grid(static_cast<unsigned>((static_cast<int64_t>(pr.nt) + rl.tb - 1) / rl.tb));
    const dim3 block(W * 32);
    const size_t smem = rows_smem_bytes(rl.ns_pad, rl.pieces, rl.tb_pad);
    const EulerFuse none = {nullptr, nullptr, 0.f};
    if (eu != nullptr)
        return pr.pot ? launch_pdl(forces_rows_kernel<K, W, U, true, true>, grid, block, smem,
                                   stream, 1u, pr, rl, out, *eu)
                      : launch_pdl(forces_rows_kernel<K, W, U, false, true>, grid, block, smem,
                                   stream, 1u, pr, rl, out, *eu);
    return pr.pot ? launch_pdl(forces_rows_kernel<K, W, U, true, false>, grid, block, smem,
                               stream, 1u, pr, rl, out, none)
                  : launch_pdl(forces_rows_kernel<K, W, U, false, false>, grid, block, smem,
                               stream, 1u, pr, rl, out, none);
}

#define NBODY_ROWS(K, W, U)                                                                  \
    {K, W, reinterpret_cast<const void *>(&forces_rows_kernel<K, W, U, true, false>),        \
     reinterpret_cast<const void *>(&forces_rows_kernel<K, W, U, false, false>),             \
     reinterpret_cast<const void *>(&forces_rows_kernel<K, W, U, true, true>),               \
     reinterpret_cast<const void *>(&forces_rows_kernel<K, W, U, false, true>),              \
     &launch_rows_kw<K, W, U>}

const RowsVariant kRowsVariants[] = {
    NBODY_ROWS(7, 8, 1),    // 0: default
    NBODY_ROWS(6, 8, 1),    // 1
    NBODY_ROWS(4, 12, 1),   // 2
    NBODY_ROWS(2, 8, 2),    // 3
};

#undef NBODY_ROWS

}  // namespace

int rows_variant_count() { return static_cast<int>(sizeof(kRowsVariants) / sizeof(kRowsVariants[0])); }

const RowsVariant &rows_variant(int v) { return kRowsVariants[v]; }

cudaError_t launch_rows(int variant, const Problem &pr, const RowsLaunch &rl, float4 *out,
                        cudaStream_t stream, const EulerFuse *eu) {
    if (variant < 0 || variant >= rows_variant_count()) return cudaErrorInvalidValue;
    return kRowsVariants[variant].launch(pr, rl, out, stream, eu);
}

}  // namespace nbody
