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

}  // namespace nbody
