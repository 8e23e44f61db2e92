// nbody_internal.h -- launchers behind the C ABI (not part of the public API).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace nbody {

// One force evaluation: every target against every source.  The all-pairs
// call passes the same array as targets and sources.
struct Problem {
    const float *targets;   // nt records (x, y, z, w); w is not read
    const float *sources;   // ns records (x, y, z, m)
    int nt;
    int ns;
    float eps2;
};

// A compiled instantiation of the tiled force kernel.
struct TiledVariant {
    int i_per_thread;   // K target bodies per thread (even: lanes of f32x2 pairs)
    int threads;        // threads per CTA
    int tile;           // source bodies per shared-memory tile
    const void *fn_pot; // kernel computing a and p
};

int tiled_variant_count();
const TiledVariant &tiled_variant(int v);

// Force kernel over grid = num_ib * splits CTAs; CTA b handles i-block
// b % num_ib and source tiles [s * tps, min((s + 1) * tps, ntiles)) with
// s = b / num_ib.  Writes out[s * nt + i] (out = the result when splits == 1).
cudaError_t launch_tiled(int variant, const Problem &pr, int num_ib, int splits,
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

// A compiled instantiation of the symmetric (each unordered pair once) kernel.
struct SymVariant {
    int i_per_thread;   // K targets per lane (even)
    int warps;          // W warps per CTA; a block is T = 32 W K bodies
    int sub;            // sources per unit (a barrier and a j-side write-back per unit)
    int min_ctas;       // resident CTAs per SM the register allocation was bounded for
    size_t smem;        // dynamic shared memory per CTA
    const void *fn;
};

int sym_variant_count();
const SymVariant &sym_variant(int v);

// Symmetric kernel over grid = nb * splits CTAs, nb = ceil(n / T): CTA b
// takes row b % nb, piece b / nb of that row's units.  Writes the i-side
// partials ipart[piece * n + i] and the j-side partials jpart[(d - 1) * n + j].
cudaError_t launch_sym(int variant, const float *bodies, int n, float eps2, int nb, int splits,
                       float4 *ipart, float4 *jpart, cudaStream_t stream);

// out[i] = the splits i-side slots of body i, then its j-side slots, in a
// fixed order, compensated (block = T bodies).  With `euler`, each body's
// Euler step follows in place (euler->pos_out = the positions the force
// kernel read, which it has finished reading).
cudaError_t launch_reduce_sym(const float4 *ipart, int splits, const float4 *jpart, int n,
                              int block, int nb, float4 *out, int sm_count, cudaStream_t stream,
                              const EulerFuse *euler = nullptr);

// out[i] = sum over s of part[s * n + i], in the order s = 0, 1, ..., compensated;
// with `euler`, each body's Euler step follows in place, as above.
cudaError_t launch_reduce_splits(const float4 *part, int n, int splits, float4 *out,
                                 int sm_count, cudaStream_t stream,
                                 const EulerFuse *euler = nullptr);

cudaError_t launch_euler(float4 *pos_mass, float4 *vel, const float4 *acc_pot, int n,
                         float dt, int sm_count, cudaStream_t stream);

}  // namespace nbody
