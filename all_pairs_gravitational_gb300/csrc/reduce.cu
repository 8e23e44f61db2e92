// reduce.cu -- the fixed-order, compensated sum of split partials, one pass
// of groups at a time.
//
// When a force launch splits the sources of a target over several CTAs, each
// writes an fp32 partial record; this kernel adds them.  Per body, in an
// order fixed by the decomposition alone: the running total of the earlier
// passes, then for each group of this pass its i-side slots and (symmetric
// path) the j-side slots of the group's distances that reach the body's
// block, in increasing distance.  The total is a Kahan pair (high, low);
// between passes the high part waits in the output record and the low part in
// a workspace slot, both stored exactly, so the arithmetic does not depend on
// how many groups a pass holds.  The last pass stores high - low and, for
// nbody_simulate, applies the body's Euler step (the force kernel has
// finished reading the positions).
//
// HBM-bound: every slot record is read once (16 bytes), the carry read and
// written once per pass.  A grid-stride loop over bodies, one thread per
// body; the slots a body reads in a group are consecutive records at stride
// n (the i-side slots, then the j-side ones), read as runs with up to sixteen
// loads in flight ahead of the dependent compensated adds.
#include <algorithm>

#include "nbody_device.cuh"
#include "nbody_internal.h"

namespace nbody {

namespace {

struct Kahan4 {
    float hx = 0.f, hy = 0.f, hz = 0.f, hw = 0.f;
    float cx = 0.f, cy = 0.f, cz = 0.f, cw = 0.f;
    __device__ __forceinline__ void add(const float4 &v) {
        kahan1(hx, cx, v.x);
        kahan1(hy, cy, v.y);
        kahan1(hz, cz, v.z);
        kahan1(hw, cw, v.w);
    }
};

// Add records p[0], p[n], ..., p[(cnt - 1) n] in that order, B loads at a
// time ahead of the adds.
template <int B>
__device__ __forceinline__ void add_run_b(Kahan4 &k, const float4 *p, int64_t n, int cnt) {
    int s = 0;
    for (; s + B <= cnt; s += B) {
        float4 v[B];
#pragma unroll
        for (int u = 0; u < B; ++u) v[u] = __ldg(p + static_cast<int64_t>(s + u) * n);
#pragma unroll
        for (int u = 0; u < B; ++u) k.add(v[u]);
    }
    for (; s < cnt; ++s) k.add(__ldg(p + static_cast<int64_t>(s) * n));
}

__device__ __forceinline__ void add_run(Kahan4 &k, const float4 *p, int64_t n, int cnt) {
    if (cnt >= 16)
        add_run_b<16>(k, p, n, cnt);
    else
        add_run_b<4>(k, p, n, cnt);
}

constexpr int kReduceThreads = 128;

template <bool SYM, bool EULER>
__global__ void __launch_bounds__(kReduceThreads)
reduce_pass_kernel(const ReducePass rp, const EulerFuse eu) {
    pdl_wait_and_release();
    const int64_t n = rp.n;
    const int H = (rp.nb - 1) / 2;
    const bool even = rp.nb % 2 == 0;
    const int nd = SYM ? sym_ndist(rp.nb) : 0;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += stride) {
        Kahan4 k;
        if (rp.carry_in) {
            const float4 h = rp.out[i];
            const float4 c = rp.lo[i];
            k.hx = h.x; k.hy = h.y; k.hz = h.z; k.hw = h.w;
            k.cx = c.x; k.cy = c.y; k.cz = c.z; k.cw = c.w;
        }
        // the extra distance nb / 2 of an even block count reaches only the
        // blocks nb / 2 .. nb - 1 (it is evaluated by the rows below nb / 2)
        const bool upper = SYM && even && (i / rp.block) >= rp.nb / 2;
        if (!SYM && rp.gstride == static_cast<int64_t>(rp.islots) * n) {
            // the tiled path: every group's slots follow one another
            add_run(k, rp.parts + i, n, rp.groups * rp.islots);
        } else {
            for (int gl = 0; gl < rp.groups; ++gl) {
                const float4 *base = rp.parts + static_cast<int64_t>(gl) * rp.gstride + i;
                int cnt = rp.islots;
                if (SYM) {   // j-side slots of distances jbase .. dhi - 1 follow the i-side ones
                    const int dlo = (rp.g0 + gl) * rp.D;
                    const int jbase = max(dlo, 1);
                    int dhi = min(dlo + rp.D, nd);
                    if (even && !upper) dhi = min(dhi, H + 1);
                    cnt += max(0, dhi - jbase);
                }
                add_run(k, base, n, cnt);
            }
        }
        if (rp.final_pass) {
            const float4 a = make_float4(__fsub_rn(k.hx, k.cx), __fsub_rn(k.hy, k.cy),
                                         __fsub_rn(k.hz, k.cz), __fsub_rn(k.hw, k.cw));
            rp.out[i] = a;
            if (EULER) {
                float4 x = eu.pos_out[i];
                float4 v = eu.vel[i];
                euler_body(x, v, a, eu.dt);
                eu.pos_out[i] = x;
                eu.vel[i] = v;
            }
        } else {
            rp.out[i] = make_float4(k.hx, k.hy, k.hz, k.hw);
            rp.lo[i] = make_float4(k.cx, k.cy, k.cz, k.cw);
        }
    }
}

template <bool SYM>
cudaError_t launch_one(const ReducePass &rp, int grid, cudaStream_t stream, const EulerFuse *eu) {
    if (eu != nullptr)
        return launch_pdl(reduce_pass_kernel<SYM, true>, dim3(grid), dim3(kReduceThreads), 0,
                          stream, 1, rp, *eu);
    return launch_pdl(reduce_pass_kernel<SYM, false>, dim3(grid), dim3(kReduceThreads), 0, stream,
                      1, rp, EulerFuse{nullptr, nullptr, 0.f});
}

}  // namespace

cudaError_t launch_reduce_pass(const ReducePass &rp, int sm_count, cudaStream_t stream,
                               const EulerFuse *euler) {
    if (rp.n <= 0 || rp.groups < 1 || rp.islots < 0) return cudaErrorInvalidValue;
    if (euler != nullptr && !rp.final_pass) return cudaErrorInvalidValue;
    const int64_t want = (static_cast<int64_t>(rp.n) + kReduceThreads - 1) / kReduceThreads;
    const int grid = static_cast<int>(std::min<int64_t>(want, static_cast<int64_t>(sm_count) * 16));
    return rp.sym ? launch_one<true>(rp, grid, stream, euler)
                  : launch_one<false>(rp, grid, stream, euler);
}

}  // namespace nbody
