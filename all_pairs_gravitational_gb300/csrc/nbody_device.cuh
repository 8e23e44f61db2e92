// nbody_device.cuh -- device helpers shared by the force kernels.
//
// Blackwell executes add/sub/mul/fma on a pair of fp32 lanes held in one
// 64-bit register pair (PTX .f32x2) as ONE issued instruction.  The FMA pipe
// still does 128 fp32 lane-operations per clock per SM, so the pair law's 13
// fp32 operations keep the same pipe time, but they take half the issue
// slots; the freed slots absorb the rsqrt (MUFU), the shared-memory loads
// and the loop bookkeeping, which otherwise compete with the arithmetic.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace nbody {

// Two fp32 lanes: bits 0..31 are lane 0, bits 32..63 lane 1.
typedef unsigned long long f2;

__device__ __forceinline__ f2 f2_pack(float lo, float hi) {
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f2_unpack(f2 v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ f2 f2_add(f2 a, f2 b) {
    f2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ f2 f2_sub(f2 a, f2 b) {
    f2 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ f2 f2_mul(f2 a, f2 b) {
    f2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// a * b + c, one rounding per lane.
__device__ __forceinline__ f2 f2_fma(f2 a, f2 b, f2 c) {
    f2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// Hardware reciprocal square root (one MUFU operation).  Its argument here is
// |r|^2 + eps^2 >= eps^2 >= FLT_MIN, always a normal number, so flushing
// subnormals changes nothing.
__device__ __forceinline__ float rsqrt_hw(float x) {
    float r;
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Kahan step: fold the partial sum `part` into (hi, lo), where the running
// total is hi - lo, then clear `part`.  Each lane independently.
__device__ __forceinline__ void f2_kahan_fold(f2 &hi, f2 &lo, f2 &part) {
    const f2 y = f2_sub(part, lo);
    const f2 t = f2_add(hi, y);
    lo = f2_sub(f2_sub(t, hi), y);
    hi = t;
    part = 0ull;
}

// Scalar Kahan step: add x to the total hi - lo.
__device__ __forceinline__ void kahan1(float &hi, float &lo, float x) {
    const float y = __fsub_rn(x, lo);
    const float t = __fadd_rn(hi, y);
    lo = __fsub_rn(__fsub_rn(t, hi), y);
    hi = t;
}

// One body's explicit Euler step, positions first: x <- x + dt v with the old
// v, then v <- v + dt a, every product and sum rounded on its own
// (__fmul_rn/__fadd_rn cannot be contracted into an FMA); x.w and v.w pass
// through.  The lecture's integrate() kernel (slides 15 and 40).
__device__ __forceinline__ void euler_body(float4 &x, float4 &v, const float4 &a, float dt) {
    x.x = __fadd_rn(x.x, __fmul_rn(dt, v.x));
    x.y = __fadd_rn(x.y, __fmul_rn(dt, v.y));
    x.z = __fadd_rn(x.z, __fmul_rn(dt, v.z));
    v.x = __fadd_rn(v.x, __fmul_rn(dt, a.x));
    v.y = __fadd_rn(v.y, __fmul_rn(dt, a.y));
    v.z = __fadd_rn(v.z, __fmul_rn(dt, a.z));
}

// Programmatic dependent launch.  Every kernel of the library is launched
// with programmatic stream serialization allowed, so the hardware may start
// scheduling its CTAs while the previous kernel in the stream is finishing.
// Each kernel first waits for the previous grid to complete with its memory
// visible -- before touching any global memory, so the ordering is the same
// as plain stream order -- and only then lets the next grid be scheduled
// (so at most one grid waits ahead of a running one).  Only the launch and
// CTA scheduling latency overlap.
__device__ __forceinline__ void pdl_wait_and_release() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 4-byte asynchronous global->shared copy; src_bytes = 0 writes a zero
// without reading global memory.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src, int src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;"
                 :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory");
}

// Compensated totals of one thread: in registers, or (TSMEM) in shared
// memory, one column per thread so that a warp's accesses are contiguous.
// Shared-memory totals free 8 registers per target pair for more
// instruction-level parallelism at the cost of 4 shared accesses per
// component per fold.
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

// ---------------------------------------------------------------- pair law
//
// Source tiles live in shared memory duplicated, (x, x, y, y, z, z, m, m)
// per body, so that two 16-byte loads give the packed operands {x_j, x_j},
// ... that pair a source with the two targets of an f32x2 register pair.

struct Src {
    f2 x, y, z, m;
};

__device__ __forceinline__ Src load_src(const float4 *s4, int j) {
    const float4 a = s4[2 * j];       // x, x, y, y
    const float4 b = s4[2 * j + 1];   // z, z, m, m
    return {f2_pack(a.x, a.y), f2_pack(a.z, a.w), f2_pack(b.x, b.y), f2_pack(b.z, b.w)};
}

// The geometry of a source against two targets: r = x_j - x_i (3 packed
// subtractions), |r|^2 + eps^2 (3 packed FMAs) and its reciprocal square
// root (2 MUFU operations) -- the rsqrt form of bodyBodyInteraction in the
// GPU Gems 3 ch.31 study page, section 1.
struct Geom {
    f2 dx, dy, dz, d2, inv;
};

__device__ __forceinline__ Geom pair_geom(const Src &s, f2 xi, f2 yi, f2 zi, f2 e2) {
    Geom g;
    g.dx = f2_sub(s.x, xi);
    g.dy = f2_sub(s.y, yi);
    g.dz = f2_sub(s.z, zi);
    g.d2 = f2_fma(g.dx, g.dx, e2);
    g.d2 = f2_fma(g.dy, g.dy, g.d2);
    g.d2 = f2_fma(g.dz, g.dz, g.d2);
    float lo, hi;
    f2_unpack(g.d2, lo, hi);
    g.inv = f2_pack(rsqrt_hw(lo), rsqrt_hw(hi));
    return g;
}

// a += m inv^3 r (3 packed multiplies, 3 packed FMAs); returns m inv, the
// potential term.  With pair_geom: 12 of the 13 fp32 lane operations of a
// pair (the 13th adds the returned term to the potential).
__device__ __forceinline__ f2 pair_accumulate(const Geom &g, f2 m, f2 &ax, f2 &ay, f2 &az) {
    const f2 tm = f2_mul(m, g.inv);        // m_j / sqrt(d2)
    const f2 inv2 = f2_mul(g.inv, g.inv);  // 1 / d2
    const f2 sc = f2_mul(tm, inv2);        // m_j / d2^(3/2)
    ax = f2_fma(sc, g.dx, ax);
    ay = f2_fma(sc, g.dy, ay);
    az = f2_fma(sc, g.dz, az);
    return tm;
}

// Stage source bodies [j0, j0 + count) into `sbuf` in the duplicated layout,
// NT threads cooperating; each 4-byte copy moves one component into one of
// its two slots, and bodies at or past `ns` are written as zeros (a zero-mass
// body at the origin adds exactly 0 to a and p, since |r|^2 + eps^2 > 0).
template <int NT>
__device__ __forceinline__ void stage_sources(float *sbuf, const float *src_bodies, int ns,
                                              int64_t j0, int count) {
    const uint32_t sbase = smem_u32(sbuf);
    for (int idx = static_cast<int>(threadIdx.x); idx < 8 * count; idx += NT) {
        const int64_t j = j0 + (idx >> 3);
        const int comp = (idx >> 1) & 3;
        const bool ok = j < ns;
        const float *src = src_bodies + (ok ? j * 4 + comp : 0);
        cp_async_4(sbase + 4u * static_cast<uint32_t>(idx), src, ok ? 4 : 0);
    }
}

// Same, for a whole tile of P bodies; the copy loop is fully unrolled.
template <int NT, int P>
__device__ __forceinline__ void stage_tile(float *sbuf, const float *src_bodies, int ns, int tile) {
    static_assert((8 * P) % NT == 0, "tile copies must divide evenly among threads");
    const uint32_t sbase = smem_u32(sbuf);
    const int64_t j0 = static_cast<int64_t>(tile) * P;
#pragma unroll
    for (int r = 0; r < (8 * P) / NT; ++r) {
        const int idx = r * NT + static_cast<int>(threadIdx.x);
        const int64_t j = j0 + (idx >> 3);
        const int comp = (idx >> 1) & 3;
        const bool ok = j < ns;
        const float *src = src_bodies + (ok ? j * 4 + comp : 0);
        cp_async_4(sbase + 4u * static_cast<uint32_t>(idx), src, ok ? 4 : 0);
    }
}

// Load K targets per thread as K/2 f32x2 pairs: lane 0 of pair q is target
// base + 2q*stride, lane 1 is base + (2q+1)*stride; indices past nt are
// clamped (their results are never stored).
template <int KP>
__device__ __forceinline__ void load_targets(const float *targets, int nt, int64_t base,
                                             int stride, f2 (&xi)[KP], f2 (&yi)[KP],
                                             f2 (&zi)[KP]) {
    const float4 *t4 = reinterpret_cast<const float4 *>(targets);
#pragma unroll
    for (int q = 0; q < KP; ++q) {
        const int64_t i0 = min(base + (2 * q) * stride, static_cast<int64_t>(nt) - 1);
        const int64_t i1 = min(base + (2 * q + 1) * stride, static_cast<int64_t>(nt) - 1);
        const float4 b0 = __ldg(t4 + i0);
        const float4 b1 = __ldg(t4 + i1);
        xi[q] = f2_pack(b0.x, b1.x);
        yi[q] = f2_pack(b0.y, b1.y);
        zi[q] = f2_pack(b0.z, b1.z);
    }
}

}  // namespace nbody
