// forces_tiled.cu -- all-pairs softened gravity, tiled over the whole GPU.
//
// Work decomposition.  Targets are cut into i-blocks of K * NT bodies, one
// CTA each; the sources are cut into tiles of P bodies, and the tile range
// may be split into S pieces so that (i-blocks x pieces) fills the GPU's CTA
// slots evenly (with one piece per i-block, N = 2^20 would leave part of the
// last wave idle on 152 SMs).  S > 1 writes fp32 partials, which a second
// kernel (reduce.cu) adds in a fixed order; a launch may cover a subset of
// the pieces when the workspace holds fewer than S partial arrays.
//
// Per CTA:
//   * each thread keeps K targets in registers, as K/2 packed f32x2 pairs
//     (targets i and i + NT share one register pair), so that one source
//     body read from shared memory feeds K pair terms -- the register
//     blocking of several targets per thread in the Aizu slides No.13-16;
//   * source tiles are staged in shared memory (the tile of the lecture's
//     slides 44-54 and of calculate_forces in the GPU Gems 3 ch.31 notes)
//     by cp.async, three stages deep: tile t+2 is in flight while tile t is
//     computed, with one barrier per tile instead of load-sync-compute-sync;
//   * a tile is stored duplicated, (x, x, y, y, z, z, m, m) per body, so that
//     two 16-byte shared loads hand the pair arithmetic its packed operands;
//   * the last tile is zero-filled past ns: a zero-mass body at the origin
//     adds exactly 0 to a and p, so the inner loop has no tail branch (the
//     tail rule of the GPU Gems 3 ch.31 study page, section 3); the self pair
//     needs no branch either (lecture slide 12);
//   * each pair is the rsqrt form of bodyBodyInteraction: 13 fp32 lane
//     operations, 6.5 issued f32x2 instructions, and 1 MUFU rsqrt;
//   * pair terms are summed in fp32 over 32 sources (the acceleration) or
//     about 1024 sources (the potential, a sum of like-signed terms), then
//     folded into Kahan-compensated totals, so the error grows neither with N
//     nor with the size of a near neighbour's term.
#include <algorithm>

#include "nbody_device.cuh"
#include "nbody_internal.h"

namespace nbody {

namespace {

constexpr int kStages = 3;
// Sources between compensated folds of the acceleration.  A near neighbour
// can contribute a term thousands of times |a_i|; while it sits in an fp32
// running sum, every later addition rounds at its scale.  Restarting the
// fp32 sum every 32 sources bounds that loss (the Kahan totals absorb the
// large term exactly enough); it costs 12 fp32 operations per 32 x 13.
constexpr int kFoldJ = 32;

// Loop modes:
//   0: one source per step of the unrolled loop;
//   2: two sources per step, their pairs computed side by side (more
//      independent instructions in flight per warp);
//   3: compensated -- the rsqrt is refined by one Newton step and every
//      acceleration term goes to a Kahan sum (29 fp32 lane-operations per pair
//      instead of 13), for bodies whose sum cancels heavily.
template <int K, int NT, int P, int MINB, bool TSMEM, int U, int MODE, bool POT>
__global__ void __launch_bounds__(NT, MINB)
forces_tiled_kernel(const Problem pr, int num_ib, int piece0, int tiles_per_split, int ntiles,
                    float4 *__restrict__ out) {
    static_assert(K % 2 == 0, "targets are processed in f32x2 pairs");
    static_assert(MODE == 0 || MODE == 2 || MODE == 3, "unknown loop mode");
    constexpr int KP = K / 2;
    constexpr int FOLD_P = (1024 + P - 1) / P;   // tiles between folds of the potential
    static_assert(P % kFoldJ == 0, "tile must hold whole fold intervals");

    __shared__ __align__(16) float sdup[kStages][P * 8];
    __shared__ __align__(16) f2 stot[TSMEM ? KP * 8 : 1][TSMEM ? NT : 1];
    pdl_wait_and_release();

    const int tid = static_cast<int>(threadIdx.x);
    const int ib = static_cast<int>(blockIdx.x % static_cast<unsigned>(num_ib));
    const int split = static_cast<int>(blockIdx.x / static_cast<unsigned>(num_ib));
    const int t_begin = (piece0 + split) * tiles_per_split;
    const int t_end = min(t_begin + tiles_per_split, ntiles);
    const int64_t ibase = static_cast<int64_t>(ib) * (NT * K) + tid;

    f2 xi[KP], yi[KP], zi[KP];
    load_targets<KP>(pr.targets, pr.nt, ibase, NT, xi, yi, zi);
    const f2 e2 = f2_pack(pr.eps2, pr.eps2);

    f2 ax[KP], ay[KP], az[KP], pp[KP];          // fp32 partials of the current fold
#pragma unroll
    for (int q = 0; q < KP; ++q) ax[q] = ay[q] = az[q] = pp[q] = 0ull;
    Totals<KP, NT, TSMEM> tot;
    if constexpr (TSMEM) {
        tot.s = stot;
        tot.tid = tid;
    }
    tot.init();

    // Prologue: two tiles in flight (one commit group per tile, empty past the end).
    if (t_begin < t_end) stage_tile<NT, P>(sdup[0], pr.sources, pr.ns, t_begin);
    cp_async_commit();
    if (t_begin + 1 < t_end) stage_tile<NT, P>(sdup[1], pr.sources, pr.ns, t_begin + 1);
    cp_async_commit();

    int stage = 0;
    for (int t = t_begin; t < t_end; ++t) {
        const int k = t - t_begin;
        cp_async_wait<1>();        // this thread's copies of tile t have landed
        __syncthreads();           // ... everyone's have, and tile t-1 is no longer read
        {
            int s2 = stage + 2;
            if (s2 >= kStages) s2 -= kStages;
            if (t + 2 < t_end) stage_tile<NT, P>(sdup[s2], pr.sources, pr.ns, t + 2);
            cp_async_commit();
        }
        const float4 *s4 = reinterpret_cast<const float4 *>(sdup[stage]);

        if constexpr (MODE == 3) {
            const f2 one = f2_pack(1.0f, 1.0f);
            const f2 half = f2_pack(0.5f, 0.5f);
#pragma unroll U
            for (int jj = 0; jj < P; ++jj) {
                const Src sj = load_src(s4, jj);
#pragma unroll
                for (int q = 0; q < KP; ++q) {
                    Geom g = pair_geom(sj, xi[q], yi[q], zi[q], e2);
                    // Newton: r = r0 + (r0 / 2)(1 - d2 r0^2)
                    const f2 res = f2_fma(f2_sub(0ull, f2_mul(g.d2, g.inv)), g.inv, one);
                    g.inv = f2_fma(f2_mul(half, g.inv), res, g.inv);
                    const f2 tm = f2_mul(sj.m, g.inv);
                    const f2 sc = f2_mul(tm, f2_mul(g.inv, g.inv));
                    f2 tx = f2_mul(sc, g.dx), ty = f2_mul(sc, g.dy), tz = f2_mul(sc, g.dz);
                    tot.fold(q, 0, tx);
                    tot.fold(q, 1, ty);
                    tot.fold(q, 2, tz);
                    if (POT) pp[q] = f2_add(pp[q], tm);
                }
            }
        } else {
#pragma unroll 1
            for (int jb = 0; jb < P; jb += kFoldJ) {
                if constexpr (MODE == 2) {
#pragma unroll U
                    for (int jj = jb; jj < jb + kFoldJ; jj += 2) {
                        const Src s0 = load_src(s4, jj);
                        const Src s1 = load_src(s4, jj + 1);
#pragma unroll
                        for (int q = 0; q < KP; ++q) {
                            const Geom g0 = pair_geom(s0, xi[q], yi[q], zi[q], e2);
                            const Geom g1 = pair_geom(s1, xi[q], yi[q], zi[q], e2);
                            const f2 t0 = pair_accumulate(g0, s0.m, ax[q], ay[q], az[q]);
                            const f2 t1 = pair_accumulate(g1, s1.m, ax[q], ay[q], az[q]);
                            if (POT) pp[q] = f2_add(pp[q], f2_add(t0, t1));
                        }
                    }
                } else {
#pragma unroll U
                    for (int jj = jb; jj < jb + kFoldJ; ++jj) {
                        const Src sj = load_src(s4, jj);
#pragma unroll
                        for (int q = 0; q < KP; ++q) {
                            const Geom g = pair_geom(sj, xi[q], yi[q], zi[q], e2);
                            const f2 tm = pair_accumulate(g, sj.m, ax[q], ay[q], az[q]);
                            if (POT) pp[q] = f2_add(pp[q], tm);
                        }
                    }
                }
#pragma unroll
                for (int q = 0; q < KP; ++q) {
                    tot.fold(q, 0, ax[q]);
                    tot.fold(q, 1, ay[q]);
                    tot.fold(q, 2, az[q]);
                }
            }
        }
        if (POT && ((k + 1) % FOLD_P == 0 || t + 1 == t_end)) {
#pragma unroll
            for (int q = 0; q < KP; ++q) tot.fold(q, 3, pp[q]);
        }
        stage = (stage + 1 == kStages) ? 0 : stage + 1;
    }
    cp_async_wait<0>();

    float4 *dst = out + static_cast<int64_t>(split) * pr.nt;
#pragma unroll
    for (int q = 0; q < KP; ++q) {
        float x0, x1, y0, y1, z0, z1, p0 = 0.f, p1 = 0.f;
        f2_unpack(tot.value(q, 0), x0, x1);
        f2_unpack(tot.value(q, 1), y0, y1);
        f2_unpack(tot.value(q, 2), z0, z1);
        if (POT) f2_unpack(tot.value(q, 3), p0, p1);
        const int64_t i0 = ibase + (2 * q) * NT;
        const int64_t i1 = ibase + (2 * q + 1) * NT;
        if (i0 < pr.nt) dst[i0] = make_float4(x0, y0, z0, POT ? -p0 : 0.f);
        if (i1 < pr.nt) dst[i1] = make_float4(x1, y1, z1, POT ? -p1 : 0.f);
    }
}

// Instantiated shapes: K targets per thread, NT threads, P-body tiles, the
// minimum resident CTAs per SM asked of the register allocator, where the
// compensated totals live (true: shared memory), the unroll factor U and the
// loop MODE.  Variant 0 is the default: the fastest of the shapes measured on
// GB300 from N = 2^18 to 2^20 (2.50e12 pairs/s at N = 2^20; packed FMA with
// three fresh operands tops out near 90 % of the pipe, and this reaches
// about 92 % of that).  Variant 7 is the compensated kernel that
// precision = 1 selects.  The others stay selectable for tuning and tests.
#define NBODY_TILED_LIST(X)                                 \
    X(4, 256, 128, 2, true, 4, 2)   /* 0: default */         \
    X(4, 256, 128, 2, false, 8, 0)  /* 1 */                  \
    X(4, 128, 128, 5, false, 8, 0)  /* 2 */                  \
    X(2, 128, 128, 8, false, 8, 0)  /* 3 */                  \
    X(8, 128, 128, 3, false, 8, 0)  /* 4 */                  \
    X(4, 256, 128, 3, true, 8, 0)   /* 5 */                  \
    X(2, 256, 128, 4, false, 4, 2)  /* 6 */                  \
    X(4, 256, 128, 2, false, 4, 3)  /* 7: compensated */

#define NBODY_TILED_ENTRY(K, NT, P, MINB, TS, U, MODE)                                  \
    {K, NT, P,                                                                         \
     reinterpret_cast<const void *>(&forces_tiled_kernel<K, NT, P, MINB, TS, U, MODE, true>), \
     reinterpret_cast<const void *>(&forces_tiled_kernel<K, NT, P, MINB, TS, U, MODE, false>)},

const TiledVariant kVariants[] = {NBODY_TILED_LIST(NBODY_TILED_ENTRY)};

template <int K, int NT, int P, int MINB, bool TS, int U, int MODE>
cudaError_t launch_variant(const Problem &pr, int num_ib, int piece0, int pieces, int tps,
                           int ntiles, float4 *out, cudaStream_t stream) {
    const unsigned grid = static_cast<unsigned>(num_ib) * static_cast<unsigned>(pieces);
    return pr.pot ? launch_pdl(forces_tiled_kernel<K, NT, P, MINB, TS, U, MODE, true>, dim3(grid),
                               dim3(NT), 0, stream, 1, pr, num_ib, piece0, tps, ntiles, out)
                  : launch_pdl(forces_tiled_kernel<K, NT, P, MINB, TS, U, MODE, false>, dim3(grid),
                               dim3(NT), 0, stream, 1, pr, num_ib, piece0, tps, ntiles, out);
}

typedef cudaError_t (*TiledLauncher)(const Problem &, int, int, int, int, int, float4 *,
                                     cudaStream_t);

#define NBODY_TILED_LAUNCHER(K, NT, P, MINB, TS, U, MODE) &launch_variant<K, NT, P, MINB, TS, U, MODE>,

const TiledLauncher kLaunchers[] = {NBODY_TILED_LIST(NBODY_TILED_LAUNCHER)};

#undef NBODY_TILED_ENTRY
#undef NBODY_TILED_LAUNCHER

}  // namespace

int tiled_variant_count() { return static_cast<int>(sizeof(kVariants) / sizeof(kVariants[0])); }

const TiledVariant &tiled_variant(int v) { return kVariants[v]; }

cudaError_t launch_tiled(int variant, const Problem &pr, int num_ib, int piece0, int pieces,
                         int tps, int ntiles, float4 *out, cudaStream_t stream) {
    if (variant < 0 || variant >= tiled_variant_count()) return cudaErrorInvalidValue;
    if (num_ib < 1 || pieces < 1 || piece0 < 0) return cudaErrorInvalidValue;
    return kLaunchers[variant](pr, num_ib, piece0, pieces, tps, ntiles, out, stream);
}

}  // namespace nbody
