/*
 * nbody.h -- C ABI of the GB300 all-pairs softened gravity library (libnbody.so).
 *
 * The operation (G = 1), for every target body i of n bodies:
 *
 *   a_i =  sum_j m_j (x_j - x_i) / (|x_j - x_i|^2 + eps^2)^(3/2)
 *   p_i = -sum_j m_j             / (|x_j - x_i|^2 + eps^2)^(1/2)
 *
 * with the sum over every j, i itself included and no branch: the self term
 * adds exactly 0 to a_i and -m_i/eps to p_i.
 *
 *   - Softened pair law and the branch-free self term: "N体問題" lecture slides
 *     (Nagaoka), slides 4 and 12.  Pair routine with the 20-flop count:
 *     bodyBodyInteraction in the "Cuda Nbody笔记" notes (GPU Gems 3 ch.31).
 *   - Potential, and the float4 (x, y, z, m) in / (ax, ay, az, p) out layout:
 *     "ATI Stream SDK による天文物理計算の高速化" slides (Aizu), No.4 and No.5.
 *   - Explicit Euler, positions first: the lecture's slides 6 and 15 and its
 *     integrate() kernel (slide 40).
 *
 * Conventions shared by every call:
 *   - Bodies are float4 records in arrays of n * 4 fp32 values, 16-byte aligned,
 *     in DEVICE memory owned by the caller.  The library keeps no pointer after
 *     a call returns (nbody_simulate's cached graph excepted, see there).
 *   - Calls are asynchronous on `stream` (0 = the legacy default stream) and
 *     never synchronise the host.  Results are ready when the stream reaches
 *     them.
 *   - Arguments are checked on the host before any launch; a rejected call
 *     launches nothing and leaves every buffer untouched.  No kernel traps,
 *     asserts or spins on a flag.
 *   - n is an int64_t; n == 0 is a successful no-op; 0 < n <= 2^31 - 1.
 *   - Every kernel is launched with programmatic stream serialization and
 *     lets the next kernel of its stream be scheduled once it has started;
 *     it waits for the previous kernel to complete before touching memory.
 *     A caller's own kernel launched with that attribute after a library
 *     call must wait likewise (cudaGridDependencySynchronize) before reading
 *     the results.
 *
 * Device memory.  Large problems add partial sums in a second kernel; the
 * partials need a workspace.  Two ways to provide it:
 *   - the *_ws calls take a caller-owned workspace and allocate nothing; with
 *     a NULL workspace they only report the size they would use;
 *   - the other calls take the workspace from a library-owned, stream-ordered
 *     memory pool for the duration of the call (freed in stream order at its
 *     end; nbody_simulate keeps it with its cached graph).  The pool keeps at
 *     most NBODY_POOL_KEEP_BYTES of freed memory across synchronisations and
 *     returns the rest to the system; nbody_release_cached returns all of it.
 * A workspace of any size works: the library plans the decomposition to fit
 * it (with none at all, partials are not used).  The default budget is
 * NBODY_DEFAULT_WORKSPACE_BYTES.
 */
#ifndef NBODY_H
#define NBODY_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum nbody_status {
    NBODY_OK = 0,
    NBODY_ERR_INVALID_ARG = 1,  /* n < 0 or > 2^31-1, null pointer, eps2 or dt out of range */
    NBODY_ERR_MISALIGNED = 2,   /* a body array or the workspace not 16-byte aligned */
    NBODY_ERR_ALIAS = 3,        /* an output or the workspace overlaps a buffer it must not */
    NBODY_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed (see nbody_last_cuda_error) */
    NBODY_ERR_TIMEOUT = 5,      /* reserved: a bounded device-side wait ran out */
    NBODY_ERR_DEVICE = 6,       /* the current device is not an sm_103 GPU */
    NBODY_ERR_TOO_LARGE = 7,    /* n above NBODY_NOALLOC_MAX_N (nbody_forces_noalloc only) */
    NBODY_ERR_WORKSPACE = 8     /* a forced path cannot run within the given workspace */
} nbody_status;

/* Workspace budget of the calls that take it from the library's pool: at
 * n = 2^20 the symmetric path then holds about 0.95 GB of partials. */
#define NBODY_DEFAULT_WORKSPACE_BYTES 1000000000LL

/* Freed pool memory kept for the next call across synchronisations. */
#define NBODY_POOL_KEEP_BYTES (64LL << 20)

/* Smallest accepted eps^2.  The branch-free self term (and any two bodies at
 * the same point) evaluates m * (eps^2)^(-3/2) * 0, which is 0 only while
 * m * (eps^2)^(-3/2) is finite in fp32: here (eps^2)^(-3/2) = 3.2e37, so
 * masses up to about 10 are safe; with larger masses eps^2 must grow with
 * them (m * (eps^2)^(-3/2) < 3.4e38), or those accelerations are NaN. */
#define NBODY_MIN_EPS2 1.0e-25f

/*
 * nbody_forces -- acceleration and potential of every body from every body.
 *
 *   pos_mass : device, n records (x, y, z, m), fp32, 16-byte aligned.  Read only.
 *   n        : number of bodies.
 *   eps2     : softening eps^2 (not eps), fp32.  Must be finite and
 *              >= NBODY_MIN_EPS2 (the branch-free self term needs
 *              |r|^2 + eps^2 > 0 and m (eps^2)^(-3/2) finite; see there).
 *   acc_pot  : device, n records (ax, ay, az, p), fp32, 16-byte aligned.
 *              Written in full; must not overlap pos_mass.
 *   stream   : CUDA stream of the launch.
 *
 * Arithmetic: fp32 pair terms (hardware rsqrt), fp32 partial sums over
 * sources folded into compensated (Kahan) totals.  Large n splits the source
 * range over CTAs and adds the fp32 partials in a fixed order, compensated,
 * in a second kernel.  From n = 10240 each unordered pair is evaluated once
 * for both bodies (the symmetric path below).  A run is bit-reproducible for
 * the same n, inputs, GPU model and plan; every workspace large enough for
 * one group of the plan (nbody_plan.scratch_min_bytes) gives the same plan
 * and the same bits.
 *
 * Workspace: from the library's pool, at most NBODY_DEFAULT_WORKSPACE_BYTES
 * (more only where a single group of partials is larger, from n of about
 * 20 million).  If the pool cannot supply it, the call re-plans within the
 * smallest workspace of the same decomposition and then within none, so it
 * fails with NBODY_ERR_CUDA only where no plan can run.
 *
 * Errors: NBODY_ERR_INVALID_ARG, _MISALIGNED, _ALIAS (host checks, nothing
 * launched); NBODY_ERR_DEVICE; NBODY_ERR_CUDA.
 */
nbody_status nbody_forces(const float *pos_mass, int64_t n, float eps2,
                          float *acc_pot, cudaStream_t stream);

/*
 * nbody_forces_acc -- nbody_forces without the potential: acc_pot gets
 * (ax, ay, az, 0).  The acceleration-only kernels of the lecture's slides
 * 13-57; they skip the potential's fp32 operations (12 instead of 13 per
 * ordered pair, 16 instead of 18 per unordered pair on the symmetric path).
 * Arguments, workspace and errors as nbody_forces.
 */
nbody_status nbody_forces_acc(const float *pos_mass, int64_t n, float eps2,
                              float *acc_pot, cudaStream_t stream);

/*
 * nbody_euler_step -- one explicit Euler step, in place:
 *   x <- x + dt * v   (with the velocity from before this call), then
 *   v <- v + dt * a,
 * per component in fp32, each product and each sum rounded on its own (no
 * fused multiply-add), so the result is bit-identical to that arithmetic.
 *
 *   pos_mass : device, n records (x, y, z, m); x, y, z updated, m untouched.
 *   vel      : device, n records (vx, vy, vz, w); vx, vy, vz updated, w untouched.
 *   acc_pot  : device, n records (ax, ay, az, p) from nbody_forces; p not read.
 *   dt       : time step, finite (any sign).
 *
 * All three arrays 16-byte aligned; none may overlap another.  No workspace.
 * Errors: as nbody_forces.
 */
nbody_status nbody_euler_step(float *pos_mass, float *vel, const float *acc_pot,
                              int64_t n, float dt, cudaStream_t stream);

/*
 * nbody_forces_ts -- target/source form: the acceleration and potential at
 * each of nt targets from all ns sources, the same pair law and arithmetic
 * as nbody_forces (which is the case targets == sources).  This is the
 * near-field leaf interaction of hierarchical codes, which keep all-pairs for
 * close cells (GPU Gems 3 ch.31 study page, section 6; Aizu slides No.30-34).
 *
 *   targets : device, nt records (x, y, z, w); w is not read.
 *   sources : device, ns records (x, y, z, m).  May be the targets array.
 *   out     : device, nt records (ax, ay, az, p); must overlap neither input.
 *
 * Every source counts, including one that sits exactly on a target (it adds
 * 0 to a and -m/eps to p).  ns == 0 writes zeros; nt == 0 is a no-op.
 * Workspace and errors: as nbody_forces.
 */
nbody_status nbody_forces_ts(const float *targets, int64_t nt, const float *sources, int64_t ns,
                             float eps2, float *out, cudaStream_t stream);

/*
 * nbody_simulate -- `steps` explicit Euler steps of the self-gravitating
 * system, device-resident: each step is nbody_forces(pos_mass -> acc_pot)
 * followed by nbody_euler_step, with the same arithmetic as the two calls and
 * bit-identical results (where the forces end in a reduction kernel, the
 * Euler update runs inside its last pass; at small n it runs inside the force
 * kernel).  It replaces the host loop of the lecture's program (slide 13, the
 * commented time loop) and of the Aizu host flow (No.10, upload / run / read
 * back / integrate on the host).
 *
 *   pos_mass, vel : device, n records each; updated in place.
 *   acc_pot       : device, n records; on return it holds (a, p) of the last
 *                   step's starting positions.
 *   steps         : >= 0 (0 is a no-op).
 *
 * One step is captured once into a CUDA graph and replayed on `stream`; up
 * to 65536 bodies a second graph holds 16 steps (and on the small-n path a
 * third holds two with the Euler update fused into the force kernel), and
 * `steps` runs as batches of 16, then pairs, then single steps.  The
 * library keeps one set of graphs per device, keyed by the
 * pointers, n, eps2, dt and the workspace; a call with other arguments
 * rebuilds it (tens of microseconds).  The graph's workspace (the partials,
 * and at small n a second position buffer) comes from the library's pool and
 * is held with the graph until it is rebuilt or nbody_release_cached is
 * called.  Successive calls on one device are ordered on the GPU after one
 * another, whatever their streams (each waits for the previous replay), so
 * the shared workspace is never used by two replays at once.  Do not call it
 * inside a stream capture of your own.
 * Errors: as nbody_forces and nbody_euler_step.
 */
nbody_status nbody_simulate(float *pos_mass, float *vel, float *acc_pot, int64_t n, float eps2,
                            float dt, int64_t steps, cudaStream_t stream);

/* Human-readable name of a status code; never NULL. */
const char *nbody_status_string(nbody_status s);

/* The cudaError_t of the most recent NBODY_ERR_CUDA on this host thread. */
int nbody_last_cuda_error(void);

/*
 * nbody_release_cached -- return the current device's memory held by the
 * library: wait until the device is idle (this call blocks the host), destroy
 * nbody_simulate's cached graph and free its workspace, and return every
 * free block of the library's pool to the system.  Afterwards the library
 * holds no device memory of that device except the fixed array of
 * nbody_forces_noalloc (64 MiB, for the lifetime of the process, once that
 * call has been used).  Errors: NBODY_ERR_DEVICE, NBODY_ERR_CUDA.
 */
nbody_status nbody_release_cached(void);

/* ------------------------------------------------------------------------
 * Launch control (tuning sweeps and tests).  Same operation as nbody_forces.
 * ------------------------------------------------------------------------ */

enum {
    NBODY_PATH_AUTO = 0,     /* the library's choice from n and the SM count */
    NBODY_PATH_TILED = 1,    /* i-blocks x j-splits over the whole grid (any n) */
    NBODY_PATH_CLUSTER = 2,  /* small n: warps and a CTA cluster split j, DSMEM reduction */
    NBODY_PATH_SYMMETRIC = 3,/* all-pairs only: each unordered pair evaluated once and
                                applied to both bodies (see below) */
    NBODY_PATH_ROWS = 4      /* few sources: each target's row split over the lanes of a
                                warp, every source in shared memory (see below) */
};

/*
 * The row-split path.  Below about ten thousand bodies one thread per target
 * leaves most of the GPU idle; the GPU Gems 3 ch.31 study page (section 4)
 * splits a body's row over several threads instead.  One CTA per SM takes
 * ceil(nt / SMs) consecutive targets and stages every source into shared
 * memory (so ns is limited to about 14000 sources: NBODY_ERR_INVALID_ARG
 * beyond).  A warp takes K targets against one of S pieces of at most 2048
 * sources, its lanes striding over the piece two sources per f32x2
 * operation; each target's lane sums are added by a fixed shuffle tree and
 * its S piece sums in order, compensated.  No workspace, no atomics:
 * deterministic.  opts.splits forces S.  The automatic choice takes it when
 * the sources number fewer than 10240 and the targets fewer than 10240, or
 * (separate target and source arrays) up to 131072 where its piece sums fit.
 */

/*
 * The symmetric path.  The pull of j on i and of i on j share r, |r|^2 + eps^2
 * and its rsqrt (Newton's third law), so one evaluation of the pair law
 * serves both bodies: 18 fp32 operations per unordered pair instead of 2 x 13.
 * The pages' kernels evaluate every ordered pair; the sums are the same up to
 * rounding order, and parity with them is held to the same bounds.  Bodies
 * are cut into nb blocks of T = 32 * warps * i_per_thread; block pairs at
 * circular distance 1..(nb-1)/2 (and nb/2 once, for even nb) are evaluated
 * both ways, each block against itself one way.  The distances are taken in
 * groups of D; within a group each block row is cut into P pieces (one CTA
 * each), whose partials -- P per body for the i-side, one per distance for
 * the j-side -- are added per body in a fixed order, compensated, by a
 * second kernel.  The groups run in passes of as many as the workspace
 * holds; the running compensated total passes from one pass to the next
 * exactly (its high part in the output, its low part in the workspace), so
 * every workspace that holds one group gives the same bits.  It needs
 * targets == sources (nbody_forces, or nbody_forces_ts with the same array
 * and nt == ns) and default precision; automatic planning uses it for
 * n >= 10240, with blocks of 512, 1024 or 2048 bodies as n grows.
 */

typedef struct nbody_forces_opts {
    int32_t path;       /* NBODY_PATH_* */
    int32_t variant;    /* kernel variant of the path; -1 = library default */
    int32_t splits;     /* tiled and row-split paths: pieces S of the source range;
                           symmetric path: pieces P of a row per group (0 = planner's
                           choice) */
    int32_t precision;  /* NBODY_PRECISION_* */
    int32_t quantities; /* NBODY_QUANTITIES_* */
    int32_t dists;      /* symmetric path: distances D per group (0 = planner's choice) */
} nbody_forces_opts;

enum {
    /* fp32 pair terms, fp32 partial sums folded into Kahan totals every 32
     * sources (acceleration) or 1024 (potential): the default. */
    NBODY_PRECISION_DEFAULT = 0,
    /* fp32 pair terms with a Newton-refined rsqrt, and every acceleration term
     * added to a Kahan sum: for bodies whose sum cancels heavily (near
     * neighbours far stronger than the total).  About 2.2x the time; tiled
     * path only.  The double-double arithmetic of the Aizu slides (No.21-22)
     * is the model for compensated sums of fp32 terms. */
    NBODY_PRECISION_COMPENSATED = 1
};

enum {
    NBODY_QUANTITIES_ACC_POT = 0,  /* (ax, ay, az, p): the default */
    NBODY_QUANTITIES_ACC = 1       /* (ax, ay, az, 0): the potential is not computed */
};

/* The decomposition nbody_forces would launch; host-only, needs no GPU. */
typedef struct nbody_plan {
    int32_t path;            /* NBODY_PATH_TILED, _CLUSTER, _SYMMETRIC or _ROWS */
    int32_t variant;         /* kernel variant index of that path */
    int32_t i_per_thread;    /* target bodies held in registers by each thread (row-split:
                                by each warp item) */
    int32_t threads;         /* threads per CTA computing pairs */
    int32_t tile;            /* source bodies per shared-memory tile (symmetric: per unit;
                                row-split: per piece, padded) */
    int32_t num_iblocks;     /* CTAs along the targets (symmetric: the nb blocks;
                                row-split: the CTAs, one per SM at most) */
    int32_t splits;          /* tiled, row-split: pieces S of the source range; symmetric:
                                pieces P of a row per group; cluster: CTAs x warps
                                splitting j */
    int32_t tiles_per_split; /* tiled: source tiles per piece; symmetric: units of
                                the largest piece; row-split: targets per CTA */
    int32_t cluster;         /* cluster path: CTAs per cluster */
    int32_t warps_j;         /* cluster path: warps splitting j inside a CTA; row-split:
                                warps per CTA */
    int32_t dists;           /* symmetric: distances D per group; 0 otherwise */
    int32_t groups;          /* symmetric: groups of distances; tiled: S; cluster, row-split: 1 */
    int32_t groups_per_pass; /* groups evaluated by one force launch */
    int32_t passes;          /* force launches (each followed by its reduction if any) */
    int64_t grid;            /* CTAs of the largest force launch */
    int64_t scratch_bytes;   /* workspace the plan uses (0 if none) */
    int64_t scratch_min_bytes; /* least workspace that keeps this decomposition and
                                  its results (one group per pass; 0 if none) */
    double fill;             /* predicted fraction of CTA slots doing useful work */
} nbody_plan;

/*
 * nbody_plan_forces -- the plan for n bodies on a GPU with `sm_count` SMs,
 * `ctas_per_sm` resident force CTAs per SM (0 = the value the library's
 * occupancy model gives), and the given options (NULL = defaults), within
 * the default workspace budget.  Host only.  Errors: NBODY_ERR_INVALID_ARG.
 */
nbody_status nbody_plan_forces(int64_t n, int32_t sm_count, int32_t ctas_per_sm,
                               const nbody_forces_opts *opts, nbody_plan *plan);

/* nbody_plan_forces within a workspace of `workspace_bytes` (>= 0).  Errors:
 * NBODY_ERR_INVALID_ARG; NBODY_ERR_WORKSPACE if a forced path cannot run in it. */
nbody_status nbody_plan_forces_ws(int64_t n, int32_t sm_count, int32_t ctas_per_sm,
                                  const nbody_forces_opts *opts, int64_t workspace_bytes,
                                  nbody_plan *plan);

/* The plan of nbody_forces_ts for nt targets and ns sources held in separate
 * arrays (the symmetric path is not open to it), within `workspace_bytes`
 * (>= 0), or the default budget for -1.  Host only.  Errors:
 * NBODY_ERR_INVALID_ARG; NBODY_ERR_WORKSPACE if a forced path cannot run in it. */
nbody_status nbody_plan_forces_ts(int64_t nt, int64_t ns, int32_t sm_count, int32_t ctas_per_sm,
                                  const nbody_forces_opts *opts, int64_t workspace_bytes,
                                  nbody_plan *plan);

/* nbody_forces with explicit launch options (NULL = defaults). */
nbody_status nbody_forces_ex(const float *pos_mass, int64_t n, float eps2, float *acc_pot,
                             const nbody_forces_opts *opts, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Caller-owned workspace: the same operations with no allocation by the
 * library.  Shared rules:
 *   - workspace == NULL: nothing is launched; *workspace_bytes receives the
 *     size the call would use by default on the current device (the one the
 *     pool-based call would take).  Pointers to bodies may be NULL then.
 *   - otherwise the call uses at most *workspace_bytes bytes at `workspace`
 *     (device memory, 16-byte aligned, overlapping no other argument) and
 *     plans within them; its contents on entry do not matter and are
 *     garbage on exit.  *workspace_bytes is not changed.  With
 *     *workspace_bytes == 0 the pointer is never dereferenced: any non-NULL
 *     value runs the call without partials.
 *   - The workspace is in use until the stream passes the call: do not reuse
 *     it on another stream before that.
 * ------------------------------------------------------------------------ */

/* nbody_forces_ex with a caller-owned workspace (opts NULL = defaults). */
nbody_status nbody_forces_ws(const float *pos_mass, int64_t n, float eps2, float *acc_pot,
                             const nbody_forces_opts *opts, void *workspace,
                             size_t *workspace_bytes, cudaStream_t stream);

/* nbody_forces_ts with a caller-owned workspace and options. */
nbody_status nbody_forces_ts_ws(const float *targets, int64_t nt, const float *sources,
                                int64_t ns, float eps2, float *out,
                                const nbody_forces_opts *opts, void *workspace,
                                size_t *workspace_bytes, cudaStream_t stream);

/*
 * nbody_simulate with a caller-owned workspace: the cached graph uses it
 * instead of pool memory, so it must stay valid, and untouched by anything
 * else, until a call with other arguments, nbody_release_cached, or the end
 * of the process.
 */
nbody_status nbody_simulate_ws(float *pos_mass, float *vel, float *acc_pot, int64_t n,
                               float eps2, float dt, int64_t steps, void *workspace,
                               size_t *workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * No-allocation variant.  The pages have no counterpart to this call: it
 * exists for callers that cannot allocate device memory -- a host framework
 * that owns all GPU memory and forbids libraries from allocating, code under
 * a hard latency budget (cudaMalloc/cudaFree can synchronise the device), or
 * code whose memory budget is fixed up front.
 * ------------------------------------------------------------------------ */

/* Largest n nbody_forces_noalloc accepts: its fixed scratch holds this many
 * float4 partial records (64 MiB), and it splits the source range into S
 * pieces only while S * n fits. */
#define NBODY_NOALLOC_MAX_N 4194304

/*
 * nbody_forces_noalloc -- the same operation, arguments and result layout as
 * nbody_forces, computed by the tiled path with its split partials in a
 * fixed array inside the library instead of memory obtained per call.  It
 * calls no cudaMalloc, cudaFree or other allocating routine.
 *
 *   - Every GPU that loads libnbody.so holds that array (64 MiB) until the
 *     process exits.
 *   - The first call on a device does a one-time set-up for it (device
 *     attributes, occupancy, and the array's device address); make that first
 *     call before any stream capture.
 *   - All calls share the array and it keeps the last call's contents;
 *     nothing in it needs to start at zero.  Calls whose kernels overlap on
 *     the GPU (other streams, other host threads) race on it: serialise them.
 *   - n > NBODY_NOALLOC_MAX_N returns NBODY_ERR_TOO_LARGE and launches
 *     nothing; the other errors are those of nbody_forces.
 */
nbody_status nbody_forces_noalloc(const float *pos_mass, int64_t n, float eps2,
                                  float *acc_pot, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NBODY_H */
