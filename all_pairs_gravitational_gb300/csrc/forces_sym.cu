// forces_sym.cu -- all-pairs softened gravity with every unordered pair
// evaluated once and applied to both of its bodies.
//
// The pull of j on i and the pull of i on j share r = x_j - x_i, |r|^2 + eps^2
// and its reciprocal square root; only the masses differ (Newton's third law:
// a_j gets -m_i r / d^3 where a_i gets +m_j r / d^3, and the potential terms
// are m_j / d and m_i / d).  One evaluation therefore serves two
// interactions: 18 fp32 lane operations and 1 MUFU rsqrt instead of 2 x 13
// and 2.  The pages' kernels evaluate every ordered pair (the j-loop of
// calculate_forces in the GPU Gems 3 ch.31 notes; the lecture's kernels); the
// sum each body receives is the same.
//
// Decomposition.  Bodies are cut into nb blocks of T = 32 W K.  Block pair
// (I, J), I != J, is evaluated once, by row I when J = I + d (mod nb) with
// 1 <= d <= H = (nb - 1) / 2, and for even nb also d = nb / 2 by the row
// I < nb / 2 only.  Row I also evaluates its own block against itself (d = 0),
// one way only (the i-side), which includes every self pair: it adds 0 to a
// and -m_i / eps to p, with no branch (lecture slide 12).  The distances are
// taken in groups of D; in each group a row's work is a list of units -- SUB
// bodies of one block J -- cut into P pieces, one CTA each, so that the
// launch fills the GPU.  A launch evaluates one or more consecutive groups.
//
// Per CTA: W warps, each holding K targets per lane (K/2 packed f32x2 pairs)
// for the whole piece.  A unit is streamed 32 bodies at a time: lane l loads
// body c + l (its "home" source) and, over 32 steps s, meets the home body of
// lane l ^ s, fetched by a shuffle.  The j-side terms a lane computes for that
// body are shuffled back to its home lane, which sums them.  So every target
// of a warp meets every source of a chunk exactly once, and every source's
// j-side sum stays in one register.
//
// Sums and determinism.  The i-side is folded into Kahan totals every 32
// sources (the acceleration) and every 1024 (the potential), as in the tiled
// kernel.  After each unit, the warps' j-side sums for its SUB sources are
// added in warp order and written to the group's j-side slot of distance d;
// the i-side totals of piece k go to the group's i-side slot k.  The
// reduction kernel (reduce.cu) adds, for every body, each group's i-side
// slots and then the j-side slots that reach it, group by group, in a fixed
// order, Kahan-compensated.  No atomics: results are bit-reproducible.
//
// Bodies past n are loaded as zeros: a zero mass adds exactly 0 to the other
// body's sums, and the phantom's own sums are never stored.
#include <algorithm>

#include "nbody_device.cuh"
#include "nbody_internal.h"

namespace nbody {

namespace {

template <int K, int W, int SUB>
struct SymShape {
    static constexpr int KP = K / 2;
    static constexpr int NT = W * 32;
    static constexpr int T = W * 32 * K;   // bodies per block
    static constexpr int SPB = T / SUB;    // units per block
    static constexpr int CPU = SUB / 32;   // 32-body chunks per unit
    static constexpr size_t jacc_bytes = 2ull * W * SUB * sizeof(float4);
    static constexpr size_t tot_bytes = static_cast<size_t>(KP) * 8 * NT * sizeof(f2);
    static constexpr size_t smem_bytes = jacc_bytes + tot_bytes;
    static_assert(K % 2 == 0, "targets are processed in f32x2 pairs");
    static_assert(SUB % 32 == 0 && T % SUB == 0, "units hold whole chunks and tile a block");
    static_assert(SUB <= NT, "one thread per source in the unit reduction");
};

__device__ __forceinline__ float4 body_or_zero(const float4 *__restrict__ bodies, int64_t i, int n) {
    return i < n ? __ldg(bodies + i) : make_float4(0.f, 0.f, 0.f, 0.f);
}

// One chunk both ways: the lane's targets against the 32 home sources of the
// warp, i-side into (ax, ay, az, pp), j-side returned for this lane's home
// source as (ax, ay, az, -p) (-p = 0 without the potential).
template <int KP, int U, bool GF, bool POT>
__device__ __forceinline__ float4 chunk_sym(float4 home, const f2 (&xi)[KP], const f2 (&yi)[KP],
                                            const f2 (&zi)[KP], const f2 (&nmi)[KP], f2 e2,
                                            f2 (&ax)[KP], f2 (&ay)[KP], f2 (&az)[KP],
                                            f2 (&pp)[KP]) {
    float jx = 0.f, jy = 0.f, jz = 0.f, jp = 0.f;
#pragma unroll U
    for (int s = 0; s < 32; ++s) {
        const float xj = __shfl_xor_sync(0xffffffffu, home.x, s);
        const float yj = __shfl_xor_sync(0xffffffffu, home.y, s);
        const float zj = __shfl_xor_sync(0xffffffffu, home.z, s);
        const float mj = __shfl_xor_sync(0xffffffffu, home.w, s);
        const Src sj = {f2_pack(xj, xj), f2_pack(yj, yj), f2_pack(zj, zj), f2_pack(mj, mj)};
        f2 tx = 0ull, ty = 0ull, tz = 0ull, tp = 0ull;
        Geom gq[KP];
        if constexpr (GF) {   // every pair's geometry and rsqrt before any accumulation
#pragma unroll
            for (int q = 0; q < KP; ++q) gq[q] = pair_geom(sj, xi[q], yi[q], zi[q], e2);
        }
#pragma unroll
        for (int q = 0; q < KP; ++q) {
            const Geom g = GF ? gq[q] : pair_geom(sj, xi[q], yi[q], zi[q], e2);
            const f2 inv2 = f2_mul(g.inv, g.inv);
            const f2 inv3 = f2_mul(inv2, g.inv);          // 1 / d^3
            const f2 sc = f2_mul(sj.m, inv3);             // m_j / d^3
            ax[q] = f2_fma(sc, g.dx, ax[q]);
            ay[q] = f2_fma(sc, g.dy, ay[q]);
            az[q] = f2_fma(sc, g.dz, az[q]);
            if (POT) pp[q] = f2_fma(sj.m, g.inv, pp[q]);  // + m_j / d
            const f2 nsc = f2_mul(nmi[q], inv3);          // -m_i / d^3
            tx = f2_fma(nsc, g.dx, tx);
            ty = f2_fma(nsc, g.dy, ty);
            tz = f2_fma(nsc, g.dz, tz);
            if (POT) tp = f2_fma(nmi[q], g.inv, tp);      // - m_i / d
        }
        float a, b;
        f2_unpack(tx, a, b);
        jx += __shfl_xor_sync(0xffffffffu, a + b, s);
        f2_unpack(ty, a, b);
        jy += __shfl_xor_sync(0xffffffffu, a + b, s);
        f2_unpack(tz, a, b);
        jz += __shfl_xor_sync(0xffffffffu, a + b, s);
        if (POT) {
            f2_unpack(tp, a, b);
            jp += __shfl_xor_sync(0xffffffffu, a + b, s);
        }
    }
    return make_float4(jx, jy, jz, jp);
}

// One chunk of the row's own block: i-side only (the pair law of the tiled
// kernel), self pairs included.
template <int KP, int U, bool POT>
__device__ __forceinline__ void chunk_diag(float4 home, const f2 (&xi)[KP], const f2 (&yi)[KP],
                                           const f2 (&zi)[KP], f2 e2, f2 (&ax)[KP], f2 (&ay)[KP],
                                           f2 (&az)[KP], f2 (&pp)[KP]) {
#pragma unroll U
    for (int s = 0; s < 32; ++s) {
        const float xj = __shfl_xor_sync(0xffffffffu, home.x, s);
        const float yj = __shfl_xor_sync(0xffffffffu, home.y, s);
        const float zj = __shfl_xor_sync(0xffffffffu, home.z, s);
        const float mj = __shfl_xor_sync(0xffffffffu, home.w, s);
        const Src sj = {f2_pack(xj, xj), f2_pack(yj, yj), f2_pack(zj, zj), f2_pack(mj, mj)};
#pragma unroll
        for (int q = 0; q < KP; ++q) {
            const Geom g = pair_geom(sj, xi[q], yi[q], zi[q], e2);
            const f2 tm = pair_accumulate(g, sj.m, ax[q], ay[q], az[q]);
            if (POT) pp[q] = f2_add(pp[q], tm);
        }
    }
}

template <int K, int W, int SUB, int MINB, int U, bool GF, bool POT>
__global__ void __launch_bounds__(W * 32, MINB)
forces_sym_kernel(const float4 *__restrict__ bodies, int n, float eps2, int nb, int P, int D,
                  int g0, float4 *__restrict__ parts, int64_t gstride) {
    using S = SymShape<K, W, SUB>;
    constexpr int KP = S::KP, NT = S::NT, T = S::T, SPB = S::SPB, CPU = S::CPU;
    constexpr int FOLD_P = 32;   // chunks between folds of the potential (1024 sources)

    extern __shared__ __align__(16) unsigned char smem[];
    float4 (*jacc)[W][SUB] = reinterpret_cast<float4 (*)[W][SUB]>(smem);
    pdl_wait_and_release();

    const int tid = static_cast<int>(threadIdx.x);
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const unsigned b = blockIdx.x;
    const int row = static_cast<int>(b % static_cast<unsigned>(nb));
    const unsigned rest = b / static_cast<unsigned>(nb);
    const int piece = static_cast<int>(rest % static_cast<unsigned>(P));
    const int gl = static_cast<int>(rest / static_cast<unsigned>(P));
    // this group's distances for this row: [dlo, dhi)
    const int dlo = (g0 + gl) * D;
    const int H = (nb - 1) / 2;
    const int dmax = H + ((nb % 2 == 0 && row < nb / 2) ? 1 : 0);
    const int dhi = min(dlo + D, dmax + 1);
    const int64_t units = dhi > dlo ? static_cast<int64_t>(dhi - dlo) * SPB : 0;
    const int64_t u0 = units * piece / P;
    const int64_t u1 = units * (piece + 1) / P;
    const int jbase = max(dlo, 1);          // distance of the group's first j-side slot
    float4 *gparts = parts + static_cast<int64_t>(gl) * gstride;

    Totals<KP, NT, true> tot;
    tot.s = reinterpret_cast<f2 (*)[NT]>(smem + S::jacc_bytes);
    tot.tid = tid;
    tot.init();

    // Targets: lane 0/1 of pair q are bodies ibase + 64 q and ibase + 64 q + 32.
    const int64_t ibase = static_cast<int64_t>(row) * T + warp * (32 * K) + lane;
    f2 xi[KP], yi[KP], zi[KP], nmi[KP];
#pragma unroll
    for (int q = 0; q < KP; ++q) {
        const float4 b0 = body_or_zero(bodies, ibase + 64 * q, n);
        const float4 b1 = body_or_zero(bodies, ibase + 64 * q + 32, n);
        xi[q] = f2_pack(b0.x, b1.x);
        yi[q] = f2_pack(b0.y, b1.y);
        zi[q] = f2_pack(b0.z, b1.z);
        nmi[q] = f2_pack(-b0.w, -b1.w);
    }
    const f2 e2 = f2_pack(eps2, eps2);

    f2 ax[KP], ay[KP], az[KP], pp[KP];
#pragma unroll
    for (int q = 0; q < KP; ++q) ax[q] = ay[q] = az[q] = pp[q] = 0ull;

    // Home source of chunk k of this piece, for this lane.
    auto home_index = [&](int64_t k) -> int64_t {
        const int64_t u = u0 + k / CPU;
        const int c = static_cast<int>(k % CPU);
        const int d = dlo + static_cast<int>(u / SPB);
        const int sub = static_cast<int>(u % SPB);
        int J = row + d;
        if (J >= nb) J -= nb;
        return static_cast<int64_t>(J) * T + sub * SUB + c * 32 + lane;
    };
    const int64_t nchunks = (u1 - u0) * CPU;
    float4 next = nchunks > 0 ? body_or_zero(bodies, home_index(0), n) : make_float4(0.f, 0.f, 0.f, 0.f);

    int64_t k = 0;
    int since_p = 0;
    for (int64_t u = u0; u < u1; ++u) {
        const int d = dlo + static_cast<int>(u / SPB);
        const int buf = static_cast<int>(u & 1);
#pragma unroll 1
        for (int c = 0; c < CPU; ++c, ++k) {
            const float4 home = next;
            if (k + 1 < nchunks) next = body_or_zero(bodies, home_index(k + 1), n);
            if (d != 0) {
                jacc[buf][warp][c * 32 + lane] =
                    chunk_sym<KP, U, GF, POT>(home, xi, yi, zi, nmi, e2, ax, ay, az, pp);
            } else {
                chunk_diag<KP, U, POT>(home, xi, yi, zi, e2, ax, ay, az, pp);
            }
#pragma unroll
            for (int q = 0; q < KP; ++q) {
                tot.fold(q, 0, ax[q]);
                tot.fold(q, 1, ay[q]);
                tot.fold(q, 2, az[q]);
            }
            if (POT && ++since_p == FOLD_P) {
                since_p = 0;
#pragma unroll
                for (int q = 0; q < KP; ++q) tot.fold(q, 3, pp[q]);
            }
        }
        // Every warp's j-side sums of this unit are in jacc[buf]; the buffer
        // is written again two units later, after the next barrier, which no
        // thread passes before finishing the reduction below.
        __syncthreads();
        if (d != 0 && tid < SUB) {
            float hx = 0.f, hy = 0.f, hz = 0.f, hw = 0.f;
            float cx = 0.f, cy = 0.f, cz = 0.f, cw = 0.f;
#pragma unroll
            for (int w = 0; w < W; ++w) {
                const float4 v = jacc[buf][w][tid];
                kahan1(hx, cx, v.x);
                kahan1(hy, cy, v.y);
                kahan1(hz, cz, v.z);
                if (POT) kahan1(hw, cw, v.w);
            }
            int J = row + d;
            if (J >= nb) J -= nb;
            const int64_t j = static_cast<int64_t>(J) * T + static_cast<int>(u % SPB) * SUB + tid;
            if (j < n)
                gparts[static_cast<int64_t>(P + d - jbase) * n + j] =
                    make_float4(__fsub_rn(hx, cx), __fsub_rn(hy, cy), __fsub_rn(hz, cz),
                                __fsub_rn(hw, cw));
        }
    }
    if (POT) {
#pragma unroll
        for (int q = 0; q < KP; ++q) tot.fold(q, 3, pp[q]);
    }

    float4 *dst = gparts + static_cast<int64_t>(piece) * n;
#pragma unroll
    for (int q = 0; q < KP; ++q) {
        float x0, x1, y0, y1, z0, z1, p0 = 0.f, p1 = 0.f;
        f2_unpack(tot.value(q, 0), x0, x1);
        f2_unpack(tot.value(q, 1), y0, y1);
        f2_unpack(tot.value(q, 2), z0, z1);
        if (POT) f2_unpack(tot.value(q, 3), p0, p1);
        const int64_t i0 = ibase + 64 * q;
        const int64_t i1 = i0 + 32;
        if (i0 < n) dst[i0] = make_float4(x0, y0, z0, POT ? -p0 : 0.f);
        if (i1 < n) dst[i1] = make_float4(x1, y1, z1, POT ? -p1 : 0.f);
    }
}

// Instantiated shapes: K targets per lane, W warps per CTA, SUB sources per
// unit, the minimum resident CTAs per SM asked of the register allocator, the
// unroll factor of the 32-step chunk loop, and GF: the geometry and rsqrt of
// all K/2 target pairs computed before any of their accumulations (the
// rsqrt latencies overlap).  Each shape is built with and without the
// potential.  The variants differ only in the block size (W = 8, 4, 2 warps:
// 2048, 1024, 512 bodies); the planner takes the smaller blocks for smaller
// n, whose waves they fill better, and variant 0 from about 160K bodies,
// where fewer partial slots win (3.31e12 interactions/s at 2^20; 118
// registers).
// Measured and dropped, each relative to the best shape of its time:
//   128-body units (1.5-2.5 % slower), 32-body units (2-3 % slower);
//   K = 6 or 4 (6-12 % slower); K = 12 with 8 or 4 warps (204-228
//   registers, 8 warps per SM: 10-11 % slower at 2^20, equal without the
//   potential); K = 2 or 4 with 32-body units and 256- or
//   512-body blocks (slower than variant 2 at every size from 2048 bodies);
//   the chunk loop unrolled by 2 or 4 (2-4 % slower);
//   each target pair's geometry and accumulation in turn (2.4 % slower);
//   two partners per step side by side (1-9 % slower);
//   1/d^2 from a MUFU reciprocal instead of a packed multiply, one FMA-pipe
//   operation fewer per pair (2.5 % slower);
//   the next step's partner shuffled a step ahead (1.5-5 % slower);
//   the i-side folded every 64 sources instead of 32 (1.2 % slower);
//   3 CTAs per SM at K = 4 (12 % slower);
//   each unit's cross-warp j-side sums spread over all threads, one component
//   each, instead of one thread per source (1.2 % slower);
//   the two halves of each j-side term shuffled back separately and added
//   by the home lane as one packed add per step (halves added once per
//   chunk): 6 % slower with the potential, equal without it;
//   the potential terms or the j-side sums as scalar fp32 FMAs (6-10 %
//   slower: packed f32x2 instructions occupy both halves of the FMA pipe, so
//   no half is left idle for scalar work);
//   each source's packed j-side sum carried round the warp with it (lane
//   l + 1 takes it after lane l's FMAs), which removes the 8 scalar adds per
//   step for 4 more shuffles: 2.3 % slower at 2^20 (3.3 % without the
//   potential).
#define NBODY_SYM_LIST(X)                     \
    X(8, 8, 64, 2, 1, true)   /* 0: default */ \
    X(8, 4, 64, 4, 1, true)   /* 1 */          \
    X(8, 2, 64, 8, 1, true)   /* 2 */

#define NBODY_SYM_ENTRY(K, W, SUB, MINB, U, GF)                                      \
    {K, W, SUB, MINB, SymShape<K, W, SUB>::smem_bytes,                                 \
     reinterpret_cast<const void *>(&forces_sym_kernel<K, W, SUB, MINB, U, GF, true>), \
     reinterpret_cast<const void *>(&forces_sym_kernel<K, W, SUB, MINB, U, GF, false>)},

const SymVariant kSymVariants[] = {NBODY_SYM_LIST(NBODY_SYM_ENTRY)};

template <int K, int W, int SUB, int MINB, int U, bool GF>
cudaError_t launch_sym_variant(const float *bodies, int n, float eps2, bool pot,
                               const SymLaunch &sl, float4 *parts, cudaStream_t stream) {
    const unsigned grid = static_cast<unsigned>(sl.nb) * static_cast<unsigned>(sl.P) *
                          static_cast<unsigned>(sl.groups);
    const float4 *b4 = reinterpret_cast<const float4 *>(bodies);
    constexpr size_t smem = SymShape<K, W, SUB>::smem_bytes;
    return pot ? launch_pdl(forces_sym_kernel<K, W, SUB, MINB, U, GF, true>, dim3(grid),
                            dim3(W * 32), smem, stream, 1, b4, n, eps2, sl.nb, sl.P, sl.D, sl.g0,
                            parts, sl.gstride)
               : launch_pdl(forces_sym_kernel<K, W, SUB, MINB, U, GF, false>, dim3(grid),
                            dim3(W * 32), smem, stream, 1, b4, n, eps2, sl.nb, sl.P, sl.D, sl.g0,
                            parts, sl.gstride);
}

typedef cudaError_t (*SymLauncher)(const float *, int, float, bool, const SymLaunch &, float4 *,
                                   cudaStream_t);

#define NBODY_SYM_LAUNCHER(K, W, SUB, MINB, U, GF) &launch_sym_variant<K, W, SUB, MINB, U, GF>,

const SymLauncher kSymLaunchers[] = {NBODY_SYM_LIST(NBODY_SYM_LAUNCHER)};

#undef NBODY_SYM_ENTRY
#undef NBODY_SYM_LAUNCHER

}  // namespace

int sym_variant_count() { return static_cast<int>(sizeof(kSymVariants) / sizeof(kSymVariants[0])); }

const SymVariant &sym_variant(int v) { return kSymVariants[v]; }

int sym_group_jslots(int nb, int D) {
    const int nd = sym_ndist(nb);
    const int groups = (nd + D - 1) / D;
    int best = 0;
    for (int g = 0; g < groups && g < 2; ++g) {   // group 0 lacks d = 0's slot; group 1 is full
        const int lo = std::max(g * D, 1);
        const int hi = std::min((g + 1) * D, nd);
        best = std::max(best, hi - lo);
    }
    return best;
}

cudaError_t launch_sym(int variant, const float *bodies, int n, float eps2, bool pot,
                       const SymLaunch &sl, float4 *parts, cudaStream_t stream) {
    if (variant < 0 || variant >= sym_variant_count()) return cudaErrorInvalidValue;
    if (sl.nb < 1 || sl.P < 1 || sl.D < 1 || sl.groups < 1) return cudaErrorInvalidValue;
    return kSymLaunchers[variant](bodies, n, eps2, pot, sl, parts, stream);
}

}  // namespace nbody
