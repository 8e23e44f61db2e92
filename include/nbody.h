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
 *     a call returns.
 *   - Calls are asynchronous on `stream` (0 = the legacy default stream) and
 *     never synchronise the host.  Results are ready when the stream reaches
 *     them.
 *   - Arguments are checked on the host before any launch; a rejected call
 *     launches nothing and leaves every buffer untouched.  No kernel traps,
 *     asserts or spins on a flag.
 *   - n is an int64_t; n == 0 is a successful no-op; 0 < n <= 2^31 - 1.
 */
#ifndef NBODY_H
#define NBODY_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum nbody_status {
    NBODY_OK = 0,
    NBODY_ERR_INVALID_ARG = 1,  /* n < 0 or > 2^31-1, null pointer, eps2 or dt out of range */
    NBODY_ERR_MISALIGNED = 2,   /* a body array not 16-byte aligned */
    NBODY_ERR_ALIAS = 3,        /* an output overlaps an input it must not overlap */
    NBODY_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed (see nbody_last_cuda_error) */
    NBODY_ERR_TIMEOUT = 5,      /* reserved: a bounded device-side wait ran out */
    NBODY_ERR_DEVICE = 6,       /* the current device is not an sm_103 GPU */
    NBODY_ERR_TOO_LARGE = 7     /* n above NBODY_NOALLOC_MAX_N (nbody_forces_noalloc only) */
} nbody_status;

/*
 * nbody_forces -- acceleration and potential of every body from every body.
 *
 *   pos_mass : device, n records (x, y, z, m), fp32, 16-byte aligned.  Read only.
 *   n        : number of bodies.
 *   eps2     : softening eps^2 (not eps), fp32.  Must be finite and >= FLT_MIN
 *              (the branch-free self term needs |r|^2 + eps^2 > 0).
 *   acc_pot  : device, n records (ax, ay, az, p), fp32, 16-byte aligned.
 *              Written in full; must not overlap pos_mass.
 *   stream   : CUDA stream of the launch.
 *
 * Arithmetic: fp32 pair terms (hardware rsqrt), fp32 partial sums over j-tiles
 * folded into compensated (Kahan) totals; a run is bit-reproducible for the
 * same n, inputs and GPU model.  Large n may split the source range over
 * CTAs and add the fp32 partials in a fixed order in a second kernel; the
 * partials live in stream-ordered memory from a library-owned pool.  From
 * n = 10240 each unordered pair is evaluated once for both bodies (the
 * symmetric path below).
 *
 * Errors: NBODY_ERR_INVALID_ARG, _MISALIGNED, _ALIAS (host checks, nothing
 * launched); NBODY_ERR_DEVICE; NBODY_ERR_CUDA.
 */
nbody_status nbody_forces(const float *pos_mass, int64_t n, float eps2,
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
 * All three arrays 16-byte aligned; none may overlap another.
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
 * Errors: as nbody_forces.
 */
nbody_status nbody_forces_ts(const float *targets, int64_t nt, const float *sources, int64_t ns,
                             float eps2, float *out, cudaStream_t stream);

/*
 * nbody_simulate -- `steps` explicit Euler steps of the self-gravitating
 * system, device-resident: each step is nbody_forces(pos_mass -> acc_pot)
 * followed by nbody_euler_step, with the same arithmetic as the two calls and
 * bit-identical results (where the forces end in a reduction kernel, the
 * Euler update runs inside it; at small n it runs inside the force kernel).
 * It replaces the host loop of the
 * lecture's program (slide 13, the commented time loop) and of the Aizu host
 * flow (No.10, upload / run / read back / integrate on the host).
 *
 *   pos_mass, vel : device, n records each; updated in place.
 *   acc_pot       : device, n records; on return it holds (a, p) of the last
 *                   step's starting positions.
 *   steps         : >= 0 (0 is a no-op).
 *
 * One step is captured once into a CUDA graph and replayed `steps` times on
 * `stream`.  The library keeps one such graph per device, keyed by the
 * pointers, n, eps2 and dt; a call with other arguments rebuilds it (tens of
 * microseconds).  Its split scratch comes from the library's pool and lives
 * with the graph.  Do not call it inside a stream capture of your own.
 * Errors: as nbody_forces and nbody_euler_step.
 */
nbody_status nbody_simulate(float *pos_mass, float *vel, float *acc_pot, int64_t n, float eps2,
                            float dt, int64_t steps, cudaStream_t stream);

/* Human-readable name of a status code; never NULL. */
const char *nbody_status_string(nbody_status s);

/* The cudaError_t of the most recent NBODY_ERR_CUDA on this host thread. */
int nbody_last_cuda_error(void);

/* ------------------------------------------------------------------------
 * Launch control (tuning sweeps and tests).  Same operation as nbody_forces.
 * ------------------------------------------------------------------------ */

enum {
    NBODY_PATH_AUTO = 0,     /* the library's choice from n and the SM count */
    NBODY_PATH_TILED = 1,    /* i-blocks x j-splits over the whole grid (any n) */
    NBODY_PATH_CLUSTER = 2,  /* small n: warps and a CTA cluster split j, DSMEM reduction */
    NBODY_PATH_SYMMETRIC = 3 /* all-pairs only: each unordered pair evaluated once and
                                applied to both bodies (see below) */
};

/*
 * The symmetric path.  The pull of j on i and of i on j share r, |r|^2 + eps^2
 * and its rsqrt (Newton's third law), so one evaluation of the pair law
 * serves both bodies: 18 fp32 operations per unordered pair instead of 2 x 13.
 * The pages' kernels evaluate every ordered pair; the sums are the same up to
 * rounding order, and parity with them is held to the same bounds.  Bodies
 * are cut into nb blocks of T = 32 * warps * i_per_thread; block pairs at
 * circular distance 1..(nb-1)/2 (and nb/2 once, for even nb) are evaluated
 * both ways, each block against itself one way.  The partials (S per body
 * for the i-side, about nb/2 per body for the j-side, n * 16 bytes each) come
 * from the library's pool and are added in a fixed order: results are
 * bit-reproducible.  It needs targets == sources (nbody_forces, or
 * nbody_forces_ts with the same array and nt == ns), default precision, and
 * partials within 24 GiB (n up to about 2.5 million); automatic planning uses
 * it for n >= 10240 when those hold, with blocks of 512, 1024 or 2048 bodies
 * as n grows.
 */

typedef struct nbody_forces_opts {
    int32_t path;       /* NBODY_PATH_* */
    int32_t variant;    /* kernel variant of the path; -1 = library default */
    int32_t splits;     /* tiled and symmetric paths: pieces S of the source range
                           (0 = planner's choice, 1 = none) */
    int32_t precision;  /* NBODY_PRECISION_* */
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

/* The decomposition nbody_forces would launch; host-only, needs no GPU. */
typedef struct nbody_plan {
    int32_t path;            /* NBODY_PATH_TILED, _CLUSTER or _SYMMETRIC */
    int32_t variant;         /* kernel variant index of that path */
    int32_t i_per_thread;    /* target bodies held in registers by each thread */
    int32_t threads;         /* threads per CTA computing pairs */
    int32_t tile;            /* source bodies per shared-memory tile (symmetric: per unit) */
    int32_t num_iblocks;     /* CTAs along the targets (symmetric: the nb blocks) */
    int32_t splits;          /* pieces of the source range (S) */
    int32_t tiles_per_split; /* tiled path: source tiles per piece; symmetric: units of
                                the largest piece */
    int32_t cluster;         /* cluster path: CTAs per cluster */
    int32_t warps_j;         /* cluster path: warps splitting j inside a CTA */
    int64_t grid;            /* CTAs launched by the force kernel */
    int64_t scratch_bytes;   /* stream-ordered scratch for the partials (0 if none) */
    double fill;             /* predicted fraction of CTA slots doing useful work */
} nbody_plan;

/*
 * nbody_plan_forces -- the plan for n bodies on a GPU with `sm_count` SMs,
 * `ctas_per_sm` resident force CTAs per SM (0 = the value the library's
 * occupancy model gives), and the given options (NULL = defaults).
 * Host only.  Errors: NBODY_ERR_INVALID_ARG.
 */
nbody_status nbody_plan_forces(int64_t n, int32_t sm_count, int32_t ctas_per_sm,
                               const nbody_forces_opts *opts, nbody_plan *plan);

/* nbody_forces with explicit launch options (NULL = defaults). */
nbody_status nbody_forces_ex(const float *pos_mass, int64_t n, float eps2, float *acc_pot,
                             const nbody_forces_opts *opts, cudaStream_t stream);

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
