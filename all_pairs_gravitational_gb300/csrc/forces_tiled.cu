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
__device__ __forceinline__ void stage_tile(float *sbuf, const float *pm, int n, int tile) {
    static_assert((8 * P) % NT == 0, "tile copies must divide evenly among threads");
    const uint32_t sbase = smem_u32(sbuf);
    const int64_t j0 = static_cast<int64_t>(tile) * P;
#pragma unroll
    for (int r = 0; r < (8 * P) / NT; ++r) {
        const int idx = r * NT + static_cast<int>(threadIdx.x);   // float slot in the tile
        const int64_t j = j0 + (idx >> 3);
        const int comp = (idx >> 1) & 3;
        const bool ok = j < n;
        const float *src = pm + (ok ? j * 4 + comp : 0);
        cp_async_4(sbase + 4u * static_cast<uint32_t>(idx), src, ok ? 4 : 0);
    }
}

template <int K, int NT, int P, bool POT>
__global__ void __launch_bounds__(NT)
forces_tiled_kernel(const float *__restrict__ pm, int n, float eps2, int num_ib,
                    int tiles_per_split, int ntiles, float4 *__restrict__ out) {
    static_assert(K % 2 == 0, "targets are processed in f32x2 pairs");
    constexpr int KP = K / 2;
    constexpr int FOLD_P = (1024 + P - 1) / P;   // tiles between folds of the potential
    static_assert(P % kFoldJ == 0, "tile must hold whole fold intervals");

    __shared__ __align__(16) float sdup[kStages][P * 8];

    const int tid = static_cast<int>(threadIdx.x);
    const int ib = static_cast<int>(blockIdx.x % static_cast<unsigned>(num_ib));
    const int split = static_cast<int>(blockIdx.x / static_cast<unsigned>(num_ib));
    const int t_begin = split * tiles_per_split;
    const int t_end = min(t_begin + tiles_per_split, ntiles);
    const int64_t ibase = static_cast<int64_t>(ib) * (NT * K) + tid;
    const float4 *pm4 = reinterpret_cast<const float4 *>(pm);

    // Targets: lane 0 of pair q is body ibase + 2q*NT, lane 1 is ibase + (2q+1)*NT.
    f2 xi[KP], yi[KP], zi[KP];
#pragma unroll
    for (int q = 0; q < KP; ++q) {
        const int64_t i0 = min(ibase + (2 * q) * NT, static_cast<int64_t>(n) - 1);
        const int64_t i1 = min(ibase + (2 * q + 1) * NT, static_cast<int64_t>(n) - 1);
        const float4 b0 = __ldg(pm4 + i0);
        const float4 b1 = __ldg(pm4 + i1);
        xi[q] = f2_pack(b0.x, b1.x);
        yi[q] = f2_pack(b0.y, b1.y);
        zi[q] = f2_pack(b0.z, b1.z);
    }
    const f2 e2 = f2_pack(eps2, eps2);

    f2 ax[KP], ay[KP], az[KP], pp[KP];          // fp32 partial over the current fold
    f2 hx[KP], hy[KP], hz[KP], hp[KP];          // compensated totals: hi ...
    f2 lx[KP], ly[KP], lz[KP], lp[KP];          // ... and the Kahan correction
#pragma unroll
    for (int q = 0; q < KP; ++q) {
        ax[q] = ay[q] = az[q] = pp[q] = 0ull;
        hx[q] = hy[q] = hz[q] = hp[q] = 0ull;
        lx[q] = ly[q] = lz[q] = lp[q] = 0ull;
    }

    // Prologue: two tiles in flight (one commit group per tile, empty past the end).
    if (t_begin < t_end) stage_tile<NT, P>(sdup[0], pm, n, t_begin);
    cp_async_commit();
    if (t_begin + 1 < t_end) stage_tile<NT, P>(sdup[1], pm, n, t_begin + 1);
    cp_async_commit();

    int stage = 0;
    for (int t = t_begin; t < t_end; ++t) {
        const int k = t - t_begin;
        cp_async_wait<1>();        // this thread's copies of tile t have landed
        __syncthreads();           // ... everyone's have, and tile t-1 is no longer read
        {
            int s2 = stage + 2;
            if (s2 >= kStages) s2 -= kStages;
            if (t + 2 < t_end) stage_tile<NT, P>(sdup[s2], pm, n, t + 2);
            cp_async_commit();
        }

        const float4 *s4 = reinterpret_cast<const float4 *>(sdup[stage]);
#pragma unroll 1
        for (int jb = 0; jb < P; jb += kFoldJ) {
#pragma unroll 8
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
                f2_kahan_fold(hx[q], lx[q], ax[q]);
                f2_kahan_fold(hy[q], ly[q], ay[q]);
                f2_kahan_fold(hz[q], lz[q], az[q]);
            }
        }
        if (POT && ((k + 1) % FOLD_P == 0 || t + 1 == t_end)) {
#pragma unroll
            for (int q = 0; q < KP; ++q) f2_kahan_fold(hp[q], lp[q], pp[q]);
        }
        stage = (stage + 1 == kStages) ? 0 : stage + 1;
    }
    cp_async_wait<0>();

    float4 *dst = out + static_cast<int64_t>(split) * n;
#pragma unroll
    for (int q = 0; q < KP; ++q) {
        float x0, x1, y0, y1, z0, z1, p0 = 0.f, p1 = 0.f;
        f2_unpack(f2_sub(hx[q], lx[q]), x0, x1);
        f2_unpack(f2_sub(hy[q], ly[q]), y0, y1);
        f2_unpack(f2_sub(hz[q], lz[q]), z0, z1);
        if (POT) f2_unpack(f2_sub(hp[q], lp[q]), p0, p1);
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

#define NBODY_TILED(K, NT, P) {K, NT, P, reinterpret_cast<const void *>(&forces_tiled_kernel<K, NT, P, true>)}

const TiledVariant kVariants[] = {
    NBODY_TILED(4, 128, 128),   // 0: default
    NBODY_TILED(8, 128, 128),   // 1
    NBODY_TILED(2, 128, 128),   // 2
    NBODY_TILED(4, 256, 128),   // 3
};

#undef NBODY_TILED

template <int K, int NT, int P>
cudaError_t launch_variant(const float *pm, int n, float eps2, int num_ib, int splits, int tps,
                           int ntiles, float4 *out, cudaStream_t stream) {
    const unsigned grid = static_cast<unsigned>(num_ib) * static_cast<unsigned>(splits);
    forces_tiled_kernel<K, NT, P, true><<<grid, NT, 0, stream>>>(pm, n, eps2, num_ib, tps,
                                                                 ntiles, out);
    return cudaGetLastError();
}

}  // namespace

int tiled_variant_count() { return static_cast<int>(sizeof(kVariants) / sizeof(kVariants[0])); }

const TiledVariant &tiled_variant(int v) { return kVariants[v]; }

cudaError_t launch_tiled(int variant, const float *pm, int n, float eps2, int num_ib, int splits,
                         int tps, int ntiles, float4 *out, cudaStream_t stream) {
    switch (variant) {
        case 0: return launch_variant<4, 128, 128>(pm, n, eps2, num_ib, splits, tps, ntiles, out, stream);
        case 1: return launch_variant<8, 128, 128>(pm, n, eps2, num_ib, splits, tps, ntiles, out, stream);
        case 2: return launch_variant<2, 128, 128>(pm, n, eps2, num_ib, splits, tps, ntiles, out, stream);
        case 3: return launch_variant<4, 256, 128>(pm, n, eps2, num_ib, splits, tps, ntiles, out, stream);
        default: return cudaErrorInvalidValue;
    }
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
