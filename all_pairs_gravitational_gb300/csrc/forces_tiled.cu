// forces_tiled.cu -- all-pairs softened gravity, tiled over the whole GPU.
//
// Work decomposition.  Targets are cut into i-blocks of K * NT bodies, one
// CTA each; the sources are cut into tiles of P bodies, and the tile range
// may be split into S pieces so that (i-blocks x pieces) fills the GPU's CTA
// slots evenly (with one piece per i-block, N = 2^20 would leave a third of
// the last wave idle on 152 SMs).  S > 1 writes fp32 partials, which a
// second kernel adds in a fixed order.
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
//     two 16-byte shared loads hand the pair arithmetic its operands {x_j,
//     x_j}, {y_j, y_j}, ... without register shuffling;
//   * the last tile is zero-filled by cp.async past n: a zero-mass body at the
//     origin adds exactly 0 to a and p (|r|^2 + eps^2 >= eps^2 > 0), so the
//     inner loop has no tail branch (the tail rule of the GPU Gems 3 ch.31
//     study page, section 3);
//   * the self pair needs no branch either (lecture slide 12);
//   * each pair is the rsqrt form of bodyBodyInteraction (GPU Gems 3 ch.31
//     study page, section 1): r = x_j - x_i (3), d2 = r.r + eps^2 (3 FMA),
//     inv = rsqrt(d2) (MUFU), t = m_j inv, inv^2, s = t inv^2 (3),
//     a += s r (3 FMA), p += t (1): 13 fp32 lane operations, 6.5 issued
//     f32x2 instructions;
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

// Stage source tile `tile` (bodies [tile * P, tile * P + P)) into `sbuf` in
// the duplicated layout.  Each 4-byte copy moves one component into one of
// its two slots; bodies past n are written as zeros.
template <int NT, int P>
__device__ __forceinline__ void stage_tile(float *sbuf, const float *src_bodies, int ns, int tile) {
    static_assert((8 * P) % NT == 0, "tile copies must divide evenly among threads");
    const uint32_t sbase = smem_u32(sbuf);
    const int64_t j0 = static_cast<int64_t>(tile) * P;
#pragma unroll
    for (int r = 0; r < (8 * P) / NT; ++r) {
        const int idx = r * NT + static_cast<int>(threadIdx.x);   // float slot in the tile
        const int64_t j = j0 + (idx >> 3);
        const int comp = (idx >> 1) & 3;
        const bool ok = j < ns;
        const float *src = src_bodies + (ok ? j * 4 + comp : 0);
        cp_async_4(sbase + 4u * static_cast<uint32_t>(idx), src, ok ? 4 : 0);
    }
}

// Compensated totals of one thread: in registers, or (TSMEM) in shared
// memory, one column per thread so that a warp's accesses are contiguous.
// Shared-memory totals free 8 registers per target pair for occupancy at
// the cost of 4 shared accesses per component per fold.
template <int KP, int NT, bool TSMEM>
struct Totals;

template <int KP, int NT>
struct Totals<KP, NT, false> {
    f2 h[KP][4], l[KP][4];
    __device__ __forceinline__ void init() {
#pragma unroll
        for (int q = 0; q < KP; ++q)
#pragma unroll
            for (int c = 0; c < 4; ++c) h[q][c] = l[q][c] = 0ull;
    }
    __device__ __forceinline__ void fold(int q, int c, f2 &part) { f2_kahan_fold(h[q][c], l[q][c], part); }
    __device__ __forceinline__ f2 value(int q, int c) { return f2_sub(h[q][c], l[q][c]); }
};

template <int KP, int NT>
struct Totals<KP, NT, true> {
    f2 (*s)[NT];     // [KP * 4 * 2][NT]: (hi, lo) of component c of pair q
    int tid;
    __device__ __forceinline__ void init() {
#pragma unroll
        for (int r = 0; r < KP * 8; ++r) s[r][tid] = 0ull;
    }
    __device__ __forceinline__ void fold(int q, int c, f2 &part) {
        f2 hi = s[(q * 4 + c) * 2][tid];
        f2 lo = s[(q * 4 + c) * 2 + 1][tid];
        f2_kahan_fold(hi, lo, part);
        s[(q * 4 + c) * 2][tid] = hi;
        s[(q * 4 + c) * 2 + 1][tid] = lo;
    }
    __device__ __forceinline__ f2 value(int q, int c) {
        return f2_sub(s[(q * 4 + c) * 2][tid], s[(q * 4 + c) * 2 + 1][tid]);
    }
};

// MODE 0: one source per step of the unrolled loop; 1: software-pipelined
// (rsqrt of source j+1 issued before source j is finished); 2: two sources
// per step, their instructions interleaved in source order.
// MODE 3: compensated -- the rsqrt is refined by one Newton step and every
// acceleration term is added to a Kahan sum (29 fp32 lane-operations per pair
// instead of 13), for systems whose bodies see extreme cancellation.
template <int K, int NT, int P, int MINB, bool TSMEM, int U, int MODE, bool POT>
__global__ void __launch_bounds__(NT, MINB)
forces_tiled_kernel(const Problem pr, int num_ib, int tiles_per_split, int ntiles,
                    float4 *__restrict__ out) {
    static_assert(K % 2 == 0, "targets are processed in f32x2 pairs");
    constexpr int KP = K / 2;
    constexpr int FOLD_P = (1024 + P - 1) / P;   // tiles between folds of the potential
    static_assert(P % kFoldJ == 0, "tile must hold whole fold intervals");

    // One spare body per stage: the software-pipelined loop reads source
    // jj + 1 ahead of finishing jj, and the last look-ahead lands on the spare
    // slot; its values are never used.
    __shared__ __align__(16) float sdup[kStages][(P + 1) * 8];
    __shared__ __align__(16) f2 stot[TSMEM ? KP * 8 : 1][TSMEM ? NT : 1];

    const int tid = static_cast<int>(threadIdx.x);
    const int ib = static_cast<int>(blockIdx.x % static_cast<unsigned>(num_ib));
    const int split = static_cast<int>(blockIdx.x / static_cast<unsigned>(num_ib));
    const int t_begin = split * tiles_per_split;
    const int t_end = min(t_begin + tiles_per_split, ntiles);
    const int64_t ibase = static_cast<int64_t>(ib) * (NT * K) + tid;
    const float4 *tg4 = reinterpret_cast<const float4 *>(pr.targets);
    const int n = pr.nt;   // targets

    // Targets: lane 0 of pair q is body ibase + 2q*NT, lane 1 is ibase + (2q+1)*NT.
    f2 xi[KP], yi[KP], zi[KP];
#pragma unroll
    for (int q = 0; q < KP; ++q) {
        const int64_t i0 = min(ibase + (2 * q) * NT, static_cast<int64_t>(n) - 1);
        const int64_t i1 = min(ibase + (2 * q + 1) * NT, static_cast<int64_t>(n) - 1);
        const float4 b0 = __ldg(tg4 + i0);
        const float4 b1 = __ldg(tg4 + i1);
        xi[q] = f2_pack(b0.x, b1.x);
        yi[q] = f2_pack(b0.y, b1.y);
        zi[q] = f2_pack(b0.z, b1.z);
    }
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
        if constexpr (MODE == 1) {
            // front(j): r = x_j - x_i, d2, rsqrt(d2) -- issued one source
            // ahead, so the MUFU work of j+1 overlaps the FMA work of j.
            f2 cdx[KP], cdy[KP], cdz[KP], cinv[KP], cm;
            auto front = [&](int j, f2 (&dx)[KP], f2 (&dy)[KP], f2 (&dz)[KP], f2 (&inv)[KP], f2 &m) {
                const float4 a = s4[2 * j];
                const float4 b = s4[2 * j + 1];
                const f2 xj = f2_pack(a.x, a.y);
                const f2 yj = f2_pack(a.z, a.w);
                const f2 zj = f2_pack(b.x, b.y);
                m = f2_pack(b.z, b.w);
#pragma unroll
                for (int q = 0; q < KP; ++q) {
                    dx[q] = f2_sub(xj, xi[q]);
                    dy[q] = f2_sub(yj, yi[q]);
                    dz[q] = f2_sub(zj, zi[q]);
                    f2 d2 = f2_fma(dx[q], dx[q], e2);
                    d2 = f2_fma(dy[q], dy[q], d2);
                    d2 = f2_fma(dz[q], dz[q], d2);
                    float d2a, d2b;
                    f2_unpack(d2, d2a, d2b);
                    inv[q] = f2_pack(rsqrt_hw(d2a), rsqrt_hw(d2b));
                }
            };
            front(0, cdx, cdy, cdz, cinv, cm);
#pragma unroll U
            for (int jj = 0; jj < P; ++jj) {
                f2 ndx[KP], ndy[KP], ndz[KP], ninv[KP], nm;
                front(jj + 1, ndx, ndy, ndz, ninv, nm);     // jj + 1 == P: the spare slot
#pragma unroll
                for (int q = 0; q < KP; ++q) {
                    const f2 tm = f2_mul(cm, cinv[q]);
                    const f2 inv2 = f2_mul(cinv[q], cinv[q]);
                    const f2 sc = f2_mul(tm, inv2);
                    ax[q] = f2_fma(sc, cdx[q], ax[q]);
                    ay[q] = f2_fma(sc, cdy[q], ay[q]);
                    az[q] = f2_fma(sc, cdz[q], az[q]);
                    if (POT) pp[q] = f2_add(pp[q], tm);
                    cdx[q] = ndx[q];
                    cdy[q] = ndy[q];
                    cdz[q] = ndz[q];
                    cinv[q] = ninv[q];
                }
                cm = nm;
                if ((jj % kFoldJ) == kFoldJ - 1) {
#pragma unroll
                    for (int q = 0; q < KP; ++q) {
                        tot.fold(q, 0, ax[q]);
                        tot.fold(q, 1, ay[q]);
                        tot.fold(q, 2, az[q]);
                    }
                }
            }
        } else if constexpr (MODE == 3) {
            const f2 one = f2_pack(1.0f, 1.0f);
            const f2 half = f2_pack(0.5f, 0.5f);
#pragma unroll U
            for (int jj = 0; jj < P; ++jj) {
                const float4 a = s4[2 * jj];
                const float4 b = s4[2 * jj + 1];
                const f2 xj = f2_pack(a.x, a.y);
                const f2 yj = f2_pack(a.z, a.w);
                const f2 zj = f2_pack(b.x, b.y);
                const f2 mj = f2_pack(b.z, b.w);
#pragma unroll
                for (int q = 0; q < KP; ++q) {
                    const f2 dx = f2_sub(xj, xi[q]);
                    const f2 dy = f2_sub(yj, yi[q]);
                    const f2 dz = f2_sub(zj, zi[q]);
                    f2 d2 = f2_fma(dx, dx, e2);
                    d2 = f2_fma(dy, dy, d2);
                    d2 = f2_fma(dz, dz, d2);
                    float d2a, d2b;
                    f2_unpack(d2, d2a, d2b);
                    const f2 r0 = f2_pack(rsqrt_hw(d2a), rsqrt_hw(d2b));
                    // Newton: r = r0 + (r0 / 2) (1 - d2 r0^2)
                    const f2 h = f2_mul(d2, r0);
                    const f2 res = f2_fma(f2_sub(0ull, h), r0, one);
                    const f2 inv = f2_fma(f2_mul(half, r0), res, r0);
                    const f2 tm = f2_mul(mj, inv);
                    const f2 inv2 = f2_mul(inv, inv);
                    const f2 sc = f2_mul(tm, inv2);
                    f2 tx = f2_mul(sc, dx), ty = f2_mul(sc, dy), tz = f2_mul(sc, dz);
                    tot.fold(q, 0, tx);
                    tot.fold(q, 1, ty);
                    tot.fold(q, 2, tz);
                    if (POT) pp[q] = f2_add(pp[q], tm);
                }
            }
        } else if constexpr (MODE == 2) {
#pragma unroll 1
            for (int jb = 0; jb < P; jb += kFoldJ) {
#pragma unroll U
                for (int jj = jb; jj < jb + kFoldJ; jj += 2) {
                    const float4 a0 = s4[2 * jj], b0 = s4[2 * jj + 1];
                    const float4 a1 = s4[2 * jj + 2], b1 = s4[2 * jj + 3];
                    const f2 xj0 = f2_pack(a0.x, a0.y), xj1 = f2_pack(a1.x, a1.y);
                    const f2 yj0 = f2_pack(a0.z, a0.w), yj1 = f2_pack(a1.z, a1.w);
                    const f2 zj0 = f2_pack(b0.x, b0.y), zj1 = f2_pack(b1.x, b1.y);
                    const f2 mj0 = f2_pack(b0.z, b0.w), mj1 = f2_pack(b1.z, b1.w);
#pragma unroll
                    for (int q = 0; q < KP; ++q) {
                        const f2 dx0 = f2_sub(xj0, xi[q]), dx1 = f2_sub(xj1, xi[q]);
                        const f2 dy0 = f2_sub(yj0, yi[q]), dy1 = f2_sub(yj1, yi[q]);
                        const f2 dz0 = f2_sub(zj0, zi[q]), dz1 = f2_sub(zj1, zi[q]);
                        f2 d20 = f2_fma(dx0, dx0, e2), d21 = f2_fma(dx1, dx1, e2);
                        d20 = f2_fma(dy0, dy0, d20);
                        d21 = f2_fma(dy1, dy1, d21);
                        d20 = f2_fma(dz0, dz0, d20);
                        d21 = f2_fma(dz1, dz1, d21);
                        float u0, v0, u1, v1;
                        f2_unpack(d20, u0, v0);
                        f2_unpack(d21, u1, v1);
                        const f2 inv0 = f2_pack(rsqrt_hw(u0), rsqrt_hw(v0));
                        const f2 inv1 = f2_pack(rsqrt_hw(u1), rsqrt_hw(v1));
                        const f2 tm0 = f2_mul(mj0, inv0), tm1 = f2_mul(mj1, inv1);
                        const f2 iq0 = f2_mul(inv0, inv0), iq1 = f2_mul(inv1, inv1);
                        const f2 s0 = f2_mul(tm0, iq0), s1 = f2_mul(tm1, iq1);
                        ax[q] = f2_fma(s0, dx0, ax[q]);
                        ay[q] = f2_fma(s0, dy0, ay[q]);
                        az[q] = f2_fma(s0, dz0, az[q]);
                        ax[q] = f2_fma(s1, dx1, ax[q]);
                        ay[q] = f2_fma(s1, dy1, ay[q]);
                        az[q] = f2_fma(s1, dz1, az[q]);
                        if (POT) pp[q] = f2_add(pp[q], f2_add(tm0, tm1));
                    }
                }
#pragma unroll
                for (int q = 0; q < KP; ++q) {
                    tot.fold(q, 0, ax[q]);
                    tot.fold(q, 1, ay[q]);
                    tot.fold(q, 2, az[q]);
                }
            }
        } else {
#pragma unroll 1
        for (int jb = 0; jb < P; jb += kFoldJ) {
#pragma unroll U
            for (int jj = jb; jj < jb + kFoldJ; ++jj) {
                const float4 a = s4[2 * jj];       // x, x, y, y
                const float4 b = s4[2 * jj + 1];   // z, z, m, m
                const f2 xj = f2_pack(a.x, a.y);
                const f2 yj = f2_pack(a.z, a.w);
                const f2 zj = f2_pack(b.x, b.y);
                const f2 mj = f2_pack(b.z, b.w);
#pragma unroll
                for (int q = 0; q < KP; ++q) {
                    const f2 dx = f2_sub(xj, xi[q]);
                    const f2 dy = f2_sub(yj, yi[q]);
                    const f2 dz = f2_sub(zj, zi[q]);
                    f2 d2 = f2_fma(dx, dx, e2);
                    d2 = f2_fma(dy, dy, d2);
                    d2 = f2_fma(dz, dz, d2);
                    float d2a, d2b;
                    f2_unpack(d2, d2a, d2b);
                    const f2 inv = f2_pack(rsqrt_hw(d2a), rsqrt_hw(d2b));
                    const f2 tm = f2_mul(mj, inv);        // m_j / sqrt(d2)
                    const f2 inv2 = f2_mul(inv, inv);     // 1 / d2
                    const f2 s = f2_mul(tm, inv2);        // m_j / d2^(3/2)
                    ax[q] = f2_fma(s, dx, ax[q]);
                    ay[q] = f2_fma(s, dy, ay[q]);
                    az[q] = f2_fma(s, dz, az[q]);
                    if (POT) pp[q] = f2_add(pp[q], tm);
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

    float4 *dst = out + static_cast<int64_t>(split) * n;
#pragma unroll
    for (int q = 0; q < KP; ++q) {
        float x0, x1, y0, y1, z0, z1, p0 = 0.f, p1 = 0.f;
        f2_unpack(tot.value(q, 0), x0, x1);
        f2_unpack(tot.value(q, 1), y0, y1);
        f2_unpack(tot.value(q, 2), z0, z1);
        if (POT) f2_unpack(tot.value(q, 3), p0, p1);
        const int64_t i0 = ibase + (2 * q) * NT;
        const int64_t i1 = ibase + (2 * q + 1) * NT;
        if (i0 < n) dst[i0] = make_float4(x0, y0, z0, -p0);
        if (i1 < n) dst[i1] = make_float4(x1, y1, z1, -p1);
    }
}

// Fixed-order compensated sum of the S partials of each body.
__global__ void reduce_splits_kernel(const float4 *__restrict__ part, int n, int splits,
                                     float4 *__restrict__ out) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += stride) {
        float hx = 0.f, hy = 0.f, hz = 0.f, hw = 0.f;
        float cx = 0.f, cy = 0.f, cz = 0.f, cw = 0.f;
        for (int s = 0; s < splits; ++s) {
            const float4 v = __ldg(part + static_cast<int64_t>(s) * n + i);
            float y, t;
            y = __fsub_rn(v.x, cx); t = __fadd_rn(hx, y); cx = __fsub_rn(__fsub_rn(t, hx), y); hx = t;
            y = __fsub_rn(v.y, cy); t = __fadd_rn(hy, y); cy = __fsub_rn(__fsub_rn(t, hy), y); hy = t;
            y = __fsub_rn(v.z, cz); t = __fadd_rn(hz, y); cz = __fsub_rn(__fsub_rn(t, hz), y); hz = t;
            y = __fsub_rn(v.w, cw); t = __fadd_rn(hw, y); cw = __fsub_rn(__fsub_rn(t, hw), y); hw = t;
        }
        out[i] = make_float4(__fsub_rn(hx, cx), __fsub_rn(hy, cy), __fsub_rn(hz, cz),
                             __fsub_rn(hw, cw));
    }
}

// Instantiated shapes: K targets per thread, NT threads, P-body tiles, the
// minimum resident CTAs per SM asked of the register allocator, where the
// compensated totals live (true: shared memory), the unroll factor U and the
// loop MODE.  Variant 0 is the default: the fastest on GB300 from N = 2^18
// to 2^20 (2.50e12 pairs/s at N = 2^20; packed FMA with three fresh
// operands tops out near 90 % of the pipe, and this reaches about 89 % of
// that).  Variant 8 is the compensated kernel that precision = 1 selects.
// The others stay selectable for tuning and tests.
#define NBODY_TILED_LIST(X)                                 \
    X(4, 256, 128, 2, true, 4, 2)   /* 0: default */         \
    X(4, 256, 128, 2, false, 8, 0)  /* 1 */                  \
    X(4, 128, 128, 5, false, 8, 0)  /* 2 */                  \
    X(2, 128, 128, 8, false, 8, 0)  /* 3 */                  \
    X(8, 128, 128, 3, false, 8, 0)  /* 4 */                  \
    X(4, 256, 128, 3, true, 8, 0)   /* 5 */                  \
    X(4, 256, 128, 2, false, 8, 1)  /* 6 */                  \
    X(2, 256, 128, 4, false, 4, 2)  /* 7 */                  \
    X(4, 256, 128, 2, false, 4, 3)  /* 8: compensated (precision 1) */

#define NBODY_TILED_ENTRY(K, NT, P, MINB, TS, U, MODE) \
    {K, NT, P, reinterpret_cast<const void *>(&forces_tiled_kernel<K, NT, P, MINB, TS, U, MODE, true>)},

const TiledVariant kVariants[] = {NBODY_TILED_LIST(NBODY_TILED_ENTRY)};

template <int K, int NT, int P, int MINB, bool TS, int U, int MODE>
cudaError_t launch_variant(const Problem &pr, int num_ib, int splits, int tps, int ntiles,
                           float4 *out, cudaStream_t stream) {
    const unsigned grid = static_cast<unsigned>(num_ib) * static_cast<unsigned>(splits);
    forces_tiled_kernel<K, NT, P, MINB, TS, U, MODE, true><<<grid, NT, 0, stream>>>(
        pr, num_ib, tps, ntiles, out);
    return cudaGetLastError();
}

typedef cudaError_t (*TiledLauncher)(const Problem &, int, int, int, int, float4 *, cudaStream_t);

#define NBODY_TILED_LAUNCHER(K, NT, P, MINB, TS, U, MODE) &launch_variant<K, NT, P, MINB, TS, U, MODE>,

const TiledLauncher kLaunchers[] = {NBODY_TILED_LIST(NBODY_TILED_LAUNCHER)};

}  // namespace

int tiled_variant_count() { return static_cast<int>(sizeof(kVariants) / sizeof(kVariants[0])); }

const TiledVariant &tiled_variant(int v) { return kVariants[v]; }

cudaError_t launch_tiled(int variant, const Problem &pr, int num_ib, int splits, int tps,
                         int ntiles, float4 *out, cudaStream_t stream) {
    if (variant < 0 || variant >= tiled_variant_count()) return cudaErrorInvalidValue;
    return kLaunchers[variant](pr, num_ib, splits, tps, ntiles, out, stream);
}

cudaError_t launch_reduce_splits(const float4 *part, int n, int splits, float4 *out, int sm_count,
                                 cudaStream_t stream) {
    const int threads = 256;
    const int64_t want = (static_cast<int64_t>(n) + threads - 1) / threads;
    const int grid = static_cast<int>(std::min<int64_t>(want, static_cast<int64_t>(sm_count) * 8));
    reduce_splits_kernel<<<grid, threads, 0, stream>>>(part, n, splits, out);
    return cudaGetLastError();
}

}  // namespace nbody
