// euler.cu -- explicit Euler step, in place, one body per thread iteration.
//
// x <- x + dt * v with the old v, then v <- v + dt * a: the lecture's
// integrate() kernel (slides 15 and 40), which advances the positions before
// the velocities.  __fmul_rn/__fadd_rn round each product and sum on its
// own, so the compiler cannot contract them into an FMA and the result is
// bit-identical to separately rounded fp32 arithmetic.  Mass (pos_mass.w)
// and vel.w are stored back unchanged.
//
// Traffic: 48 bytes read + 32 bytes written per body, as float4 accesses; a
// grid-stride loop with a few CTAs per SM keeps enough loads in flight to
// stream HBM.
#include <algorithm>

#include "nbody_device.cuh"
#include "nbody_internal.h"

namespace nbody {

namespace {

__global__ void __launch_bounds__(256)
euler_kernel(float4 *__restrict__ pm, float4 *__restrict__ vel,
             const float4 *__restrict__ acc, int n, float dt) {
    pdl_wait_and_release();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += stride) {
        float4 p = pm[i];
        float4 v = vel[i];
        euler_body(p, v, __ldg(acc + i), dt);
        pm[i] = p;
        vel[i] = v;
    }
}

}  // namespace

cudaError_t launch_euler(float4 *pm, float4 *vel, const float4 *acc, int n, float dt,
                         int sm_count, cudaStream_t stream) {
    const int threads = 256;
    const int64_t want = (static_cast<int64_t>(n) + threads - 1) / threads;
    const int grid = static_cast<int>(std::min<int64_t>(want, static_cast<int64_t>(sm_count) * 8));
    return launch_pdl(euler_kernel, dim3(grid), dim3(threads), 0, stream, 1, pm, vel, acc, n, dt);
}

}  // namespace nbody
