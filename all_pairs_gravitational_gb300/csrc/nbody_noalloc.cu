// nbody_noalloc.cu -- nbody_forces_noalloc: the tiled force path with its
// split partials kept in one fixed, library-owned device array instead of
// memory obtained per call.
//
// Who needs it: callers that may not allocate device memory themselves or
// through a library -- a host framework that owns every byte of GPU memory
// and forbids plug-ins from allocating, code under a hard latency budget
// (cudaMalloc and cudaFree can synchronise the whole device), and code
// whose memory budget is fixed before it starts.
//
// The scratch below is a file-scope __device__ array: every GPU that loads
// libnbody.so holds it (NBODY_NOALLOC_MAX_N float4 records, 64 MiB) until
// the process exits.  Host code must never pass the array's name to a
// kernel: on the host that name is only a stand-in, not a device address.
// The device address is looked up once per device with cudaGetSymbolAddress
// during set-up, which is done by the first call on that device.
//
// All calls share the array and it keeps whatever the last call wrote.
// Nothing in it has to start at zero: the force kernel writes every partial
// record the reduction reads.  Two calls whose kernels overlap on the GPU
// (different streams, or several host threads) race on the array and give
// wrong results; serialise them.
#include <algorithm>
#include <cfloat>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "nbody.h"
#include "nbody_internal.h"

namespace {

constexpr int64_t kScratchRecords = NBODY_NOALLOC_MAX_N;

static __device__ __align__(256) float4 g_noalloc_scratch[kScratchRecords];

constexpr int kMaxDevices = 64;
constexpr int kMaxSplitsTried = 256;

struct NoAllocDevice {
    bool ready = false;
    float4 *scratch = nullptr;   // device address of g_noalloc_scratch on this device
    int sm_count = 0;
    int occ = 0;                 // resident CTAs per SM of the default tiled kernel
};

std::mutex g_mu;
NoAllocDevice g_dev[kMaxDevices];

// Record the CUDA error for nbody_last_cuda_error (defined with the other
// entry points) and report it.
nbody_status fail(cudaError_t e) {
    nbody::record_cuda_error(static_cast<int>(e));
    return NBODY_ERR_CUDA;
}

// Per-device set-up, with that device current: no allocation of any kind.
nbody_status setup(NoAllocDevice **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(e);
    if (dev < 0 || dev >= kMaxDevices) return NBODY_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    NoAllocDevice &d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return fail(e);
        if (major != 10 || minor != 3) return NBODY_ERR_DEVICE;
        const nbody::TiledVariant &tv = nbody::tiled_variant(0);
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.occ, tv.fn_pot, tv.threads, 0)) != cudaSuccess)
            return fail(e);
        void *ptr = nullptr;
        if ((e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch)) != cudaSuccess) return fail(e);
        d.scratch = static_cast<float4 *>(ptr);
        d.ready = true;
    }
    *out = &d;
    return NBODY_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void *a, const void *b, int64_t bytes) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a);
    const uintptr_t y = reinterpret_cast<uintptr_t>(b);
    const uintptr_t len = static_cast<uintptr_t>(bytes);
    return x < y + len && y < x + len;
}

}  // namespace

extern "C" nbody_status nbody_forces_noalloc(const float *pos_mass, int64_t n, float eps2,
                                             float *acc_pot, cudaStream_t stream) {
    if (n < 0 || n > INT32_MAX) return NBODY_ERR_INVALID_ARG;
    if (n == 0) return NBODY_OK;
    if (pos_mass == nullptr || acc_pot == nullptr) return NBODY_ERR_INVALID_ARG;
    if (!std::isfinite(eps2) || !(eps2 >= NBODY_MIN_EPS2)) return NBODY_ERR_INVALID_ARG;
    if (!aligned16(pos_mass) || !aligned16(acc_pot)) return NBODY_ERR_MISALIGNED;
    if (overlap(pos_mass, acc_pot, 16 * n)) return NBODY_ERR_ALIAS;
    if (n > NBODY_NOALLOC_MAX_N) return NBODY_ERR_TOO_LARGE;

    NoAllocDevice *dev = nullptr;
    nbody_status st = setup(&dev);
    if (st != NBODY_OK) return st;

    // Split the source range as far as the fixed scratch allows (S * n
    // partial records), keeping the split count with the best predicted fill.
    const int64_t s_max = std::min<int64_t>(kScratchRecords / n, kMaxSplitsTried);
    nbody_plan best = {};
    bool have = false;
    for (int64_t s = 1; s <= s_max; ++s) {
        nbody_forces_opts opts = {NBODY_PATH_TILED, -1, static_cast<int32_t>(s),
                                  NBODY_PRECISION_DEFAULT, NBODY_QUANTITIES_ACC_POT, 0};
        nbody_plan p;
        if (nbody_plan_forces(n, dev->sm_count, dev->occ, &opts, &p) != NBODY_OK) continue;
        if (p.splits > s_max) continue;
        if (!have || p.fill > best.fill * (1.0 + 1e-3)) {
            best = p;
            have = true;
        }
    }
    if (!have) return NBODY_ERR_INVALID_ARG;

    const int ni = static_cast<int>(n);
    const int ntiles = static_cast<int>((n + best.tile - 1) / best.tile);
    float4 *out = reinterpret_cast<float4 *>(acc_pot);
    const nbody::Problem pr = {pos_mass, pos_mass, ni, ni, eps2, true};
    cudaError_t e;
    if (best.splits == 1) {
        e = nbody::launch_tiled(best.variant, pr, best.num_iblocks, 0, 1, best.tiles_per_split,
                                ntiles, out, stream);
    } else {
        // every piece in one launch, their partials in the fixed array, then
        // one reduction pass that adds them in piece order
        e = nbody::launch_tiled(best.variant, pr, best.num_iblocks, 0, best.splits,
                                best.tiles_per_split, ntiles, dev->scratch, stream);
        const nbody::ReducePass rp = {dev->scratch, n, 1, false, 0, 1, 1, 0, best.splits, ni,
                                      out, nullptr, false, true};
        if (e == cudaSuccess) e = nbody::launch_reduce_pass(rp, dev->sm_count, stream);
    }
    return e == cudaSuccess ? NBODY_OK : fail(e);
}
