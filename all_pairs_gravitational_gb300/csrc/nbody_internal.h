// nbody_internal.h -- launchers behind the C ABI (not part of the public API).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace nbody {

// Launch `kernel` on `stream` with programmatic stream serialization allowed
// (the kernel begins with pdl_wait_and_release, nbody_device.cuh), plus an
// optional cluster shape (cluster_x > 1).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, unsigned cluster_x, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    unsigned na = 1;
    if (cluster_x > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = cluster_x;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        na = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// One force evaluation: every target against every source.  The all-pairs
// call passes the same array as targets and sources.
struct Problem {
    const float *targets;   // nt records (x, y, z, w); w is not read
    const float *sources;   // ns records (x, y, z, m)
    int nt;
    int ns;
    float eps2;
    bool pot;               // compute the potential (false: .w of every result is 0)
};

// A compiled instantiation of the tiled force kernel.
struct TiledVariant {
    int i_per_thread;   // K target bodies per thread (even: lanes of f32x2 pairs)
    int threads;        // threads per CTA
    int tile;           // source bodies per shared-memory tile
    const void *fn_pot; // kernel computing a and p
    const void *fn_acc; // kernel computing a only
};

int tiled_variant_count();
const TiledVariant &tiled_variant(int v);

// Force kernel over grid = num_ib * pieces CTAs; CTA b handles i-block
// b % num_ib and source tiles [s * tps, min((s + 1) * tps, ntiles)) with
// s = piece0 + b / num_ib.  Writes out[(b / num_ib) * nt + i] (out = the
// result when the whole source range is one piece).
cudaError_t launch_tiled(int variant, const Problem &pr, int num_ib, int piece0, int pieces,
                         int tiles_per_split, int ntiles, float4 *out, cudaStream_t stream);

// Euler update applied by a kernel as it stores each body's result:
// pos_out = pos + dt * vel (old vel), then vel += dt * a, every product and
// sum rounded on its own; the mass is copied.  In a force kernel pos_out must
// not be the targets array (other CTAs are still reading it); in a reduction
// kernel, which runs after the force kernel, it is the positions themselves.
struct EulerFuse {
    float4 *pos_out;
    float4 *vel;
    float dt;
};

// A compiled instantiation of the small-N cluster kernel.
struct ClusterVariant {
    int i_per_thread;   // K targets per lane (even); the cluster's target block is 32 K
    int warps;          // W warps per CTA, each taking a slice of every source tile
    int tile;           // source bodies per shared-memory tile
    bool whole;         // stages the CTA's whole source range at once (dynamic smem)
    const void *fn_pot;
    const void *fn_acc;
};

// Dynamic shared memory a whole-range cluster launch needs.
size_t whole_smem_bytes(int K, int W, int tiles_per_cta);

// Largest dynamic shared memory a whole-range CTA may use (the sm_103 opt-in
// limit is 227 KB per block).
constexpr size_t kWholeSmemMax = 200 * 1024;

int cluster_variant_count();
const ClusterVariant &cluster_variant(int v);

// Cluster kernel over grid = num_ib * cluster CTAs in clusters of `cluster`;
// cluster b handles targets [b * 32K, (b + 1) * 32K), its CTA of rank c the
// source tiles [c * tpc, min((c + 1) * tpc, ntiles)).  Writes out[i] directly.
cudaError_t launch_cluster(int variant, const Problem &pr, int num_ib, int cluster,
                           int tiles_per_cta, int ntiles, float4 *out, cudaStream_t stream,
                           const EulerFuse *euler = nullptr);

// The row-split kernel's decomposition: CTA b takes targets [b tb, (b + 1) tb)
// (fewer in the last CTA); its warp items are `groups` runs of K targets
// (tb_pad = groups K >= tb) times `pieces` pieces of `cols` source pairs each
// (cols a multiple of 32; ns_pad = 2 pieces cols >= ns, zero past ns).
struct RowsLaunch {
    int tb;
    int groups;
    int tb_pad;
    int pieces;
    int cols;
    int ns_pad;
};

// A compiled instantiation of the row-split kernel.
struct RowsVariant {
    int i_per_warp;       // K targets per warp item
    int warps;            // W warps per CTA
    const void *fn_pot;   // a and p
    const void *fn_acc;   // a only
    const void *fn_pot_euler;   // the same with the Euler step fused
    const void *fn_acc_euler;
    cudaError_t (*launch)(const struct Problem &, const struct RowsLaunch &, float4 *,
                          cudaStream_t, const struct EulerFuse *);
};

int rows_variant_count();
const RowsVariant &rows_variant(int v);

// Dynamic shared memory of a row-split launch: the sources and the piece sums.
size_t rows_smem_bytes(int ns_pad, int pieces, int tb_pad);

// Largest dynamic shared memory of a row-split CTA (the sm_103 opt-in limit
// of 227 KB per block).
constexpr size_t kRowsSmemMax = 227 * 1024;

// Row-split kernel over ceil(nt / tb) CTAs; writes out[i] directly.
cudaError_t launch_rows(int variant, const Problem &pr, const RowsLaunch &rl, float4 *out,
                        cudaStream_t stream, const EulerFuse *euler = nullptr);

// A compiled instantiation of the symmetric (each unordered pair once) kernel.
struct SymVariant {
    int i_per_thread;   // K targets per lane (even)
    int warps;          // W warps per CTA; a block is T = 32 W K bodies
    int sub;            // sources per unit (a barrier and a j-side write-back per unit)
    int min_ctas;       // resident CTAs per SM the register allocation was bounded for
    size_t smem;        // dynamic shared memory per CTA
    const void *fn_pot;
    const void *fn_acc;
};

int sym_variant_count();
const SymVariant &sym_variant(int v);

// The symmetric decomposition of n bodies into nb blocks of T: block row I
// evaluates, both ways, the blocks at circular distance d = 1 .. H from it
// (H = (nb - 1) / 2), and d = nb / 2 as well for I < nb / 2 when nb is even;
// d = 0 is its own block, evaluated one way.  Distances 0 .. ndist - 1 are
// taken in groups of D; in each group a row's units (SUB sources of one
// block) are cut into P pieces.
struct SymLaunch {
    int nb;         // blocks
    int P;          // pieces per row per group
    int D;          // distances per group
    int g0;         // first group of this launch
    int groups;     // groups of this launch: grid = nb * P * groups CTAs
    int64_t gstride;// records between the partial slots of consecutive groups
};

// Distances of the decomposition: 0 .. ndist - 1.
__host__ __device__ inline int sym_ndist(int nb) {
    return (nb - 1) / 2 + 1 + (nb % 2 == 0 ? 1 : 0);
}

// The largest j-side slot count of any group (the slot layout's stride is
// P + that many records per body).
int sym_group_jslots(int nb, int D);

// Symmetric kernel: CTA b takes row b % nb, piece (b / nb) % P of group
// g0 + b / (nb P).  Writes the group's i-side partials to
// parts[gl * gstride + piece * n + i] and its j-side partials to
// parts[gl * gstride + (P + d - max(dlo, 1)) * n + j] (gl = group - g0, dlo
// = the group's first distance).  With nb == 1 and P == 1, parts may be the
// result itself.
cudaError_t launch_sym(int variant, const float *bodies, int n, float eps2, bool pot,
                       const SymLaunch &sl, float4 *parts, cudaStream_t stream);

// One pass of the fixed-order compensated reduction.  For every body i, in
// this order: the running total carried in from the previous pass (its high
// part in out[i], its low part in lo[i]); then, for each group of the pass,
// its i-side slots 0 .. islots - 1 and (symmetric path) the j-side slots of
// the group's distances that reach the body's block, in increasing distance.
// A final pass stores high - low (and applies `euler` if given); any other
// stores the high and low parts for the next pass.
struct ReducePass {
    const float4 *parts;
    int64_t gstride;    // records between the slots of consecutive groups
    int islots;         // i-side slots per group (tiled path: 1)
    bool sym;           // symmetric path: j-side slots follow the i-side ones
    int D;              // symmetric: distances per group
    int nb;             // symmetric: blocks
    int block;          // symmetric: bodies per block
    int g0;             // first group of the pass
    int groups;         // groups in the pass
    int n;
    float4 *out;
    float4 *lo;
    bool carry_in;
    bool final_pass;
};

cudaError_t launch_reduce_pass(const ReducePass &rp, int sm_count, cudaStream_t stream,
                               const EulerFuse *euler = nullptr);

// Record a CUDA error for nbody_last_cuda_error (this host thread).
void record_cuda_error(int e);

cudaError_t launch_euler(float4 *pos_mass, float4 *vel, const float4 *acc_pot, int n,
                         float dt, int sm_count, cudaStream_t stream);

}  // namespace nbody
