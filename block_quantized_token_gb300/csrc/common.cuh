// Device helpers shared by the kernels: PTX wrappers (mbarrier, bulk copy,
// programmatic dependent launch, tensor-core MMA) and the exact small-integer
// to fp16 conversions used to dequantise blocks in registers.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define ER_DEV __device__ __forceinline__

// device flag bits (see er_get_device_error)
#define ER_FLAG_TOKEN 1
#define ER_FLAG_POS 2
#define ER_FLAG_WAIT 4
#define ER_FLAG_NONFINITE 8

// bounded waits give up after this many nanoseconds of %globaltimer by default
#define ER_WAIT_NS 1000000000ull

namespace er {

// The limit of every bounded wait, in ns.  Each translation unit holds its own
// copy (the library is compiled without relocatable device code); the host
// sets all of them through er_set_wait_limit_ns, for tests of the give-up path.
static __device__ unsigned long long g_wait_ns = ER_WAIT_NS;
ER_DEV unsigned long long wait_limit_ns() { return *reinterpret_cast<volatile unsigned long long *>(&g_wait_ns); }
// Sets this translation unit's copy on the current device (synchronous).
static inline cudaError_t set_wait_limit_here(unsigned long long ns) {
    return cudaMemcpyToSymbol(g_wait_ns, &ns, sizeof ns);
}

// ---------------------------------------------------------------------------
// programmatic dependent launch (PDL)
// ---------------------------------------------------------------------------
// Blocks until the grids this grid depends on have completed and their memory
// is visible.  A no-op when the kernel was launched without the PDL attribute.
ER_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel in the stream start its independent prologue.
ER_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// mbarrier + bulk async copy (the TMA engine's non-tensor form)
// ---------------------------------------------------------------------------
ER_DEV uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

ER_DEV void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
ER_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
ER_DEV void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

ER_DEV void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// Returns true once the phase with parity `parity` has completed; a thread may
// be suspended for up to about 20 us inside the call while it waits (rather
// than spinning and taking issue slots from the warps that compute).
ER_DEV bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(20000)
        : "memory");
    return ok != 0;
}

// atomic add with acquire-release semantics at GPU scope (returns the old value)
ER_DEV int atom_add_acq_rel_gpu(int *p, int v) {
    int old;
    asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

ER_DEV void red_add_release_gpu(unsigned *p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
ER_DEV unsigned ld_acquire_gpu(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

ER_DEV uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait: false after the wait limit without completion (the caller
// records an error and stops waiting).
ER_DEV bool mbar_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    const unsigned long long lim = wait_limit_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255) == 0 && globaltimer_ns() - t0 > lim) return false;
    }
}

// global -> shared bulk copy completing on `bar` (16-byte aligned, size % 16 == 0)
ER_DEV void bulk_g2s(void *dst_smem, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

ER_DEV void prefetch_l2_bulk(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------------------
// shared-memory vector loads
// ---------------------------------------------------------------------------
ER_DEV uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
ER_DEV uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

// ---------------------------------------------------------------------------
// tensor core: D[16x8] = A[16x16] B[16x8] + C, fp16 inputs, fp32 accumulate
// ---------------------------------------------------------------------------
ER_DEV void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1, const float (&c)[4]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
          "f"(c[3]));
}

// ---------------------------------------------------------------------------
// exact integer -> fp16 pairs.  An fp16 with exponent field 25 (bits 0x6400)
// is 1024 + m for its 10-bit mantissa m, so OR-ing a small unsigned integer
// into the mantissa and subtracting the bias gives the integer exactly.
// ---------------------------------------------------------------------------
ER_DEV uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
ER_DEV uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t orv) {
    uint32_t d;
    // d = (a & mask) | orv  (truth table 0xEA for (a & b) | c)
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(orv));
    return d;
}
ER_DEV uint32_t h2_sub(uint32_t a, uint32_t b) {
    __half2 r = __hsub2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}
ER_DEV uint32_t h2_fma(uint32_t a, uint32_t b, uint32_t c) {
    __half2 r = __hfma2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b),
                        *reinterpret_cast<__half2 *>(&c));
    return *reinterpret_cast<uint32_t *>(&r);
}

// Q8_0 word of 4 stored bytes u_i = q_i ^ 0x80 -> two half2 (q0,q1), (q2,q3)
ER_DEV void q8_word_to_h2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t k1152 = 0x64806480u;  // half2(1152, 1152) = 1024 + 128
    lo = h2_sub(prmt(w, 0x64646464u, 0x4140u), k1152);
    hi = h2_sub(prmt(w, 0x64646464u, 0x4342u), k1152);
}

// Q4_0 word of 8 stored nibbles n_p at bits 4p -> four half2 of (n - 8):
//   r0 = (n0, n4), r1 = (n1, n5), r2 = (n2, n6), r3 = (n3, n7)
ER_DEV void q4_word_to_h2(uint32_t w, uint32_t (&r)[4]) {
    const uint32_t magic = 0x64006400u;
    const uint32_t k1032 = 0x64086408u;        // half2(1032, 1032) = 1024 + 8
    const uint32_t k1_16 = 0x2C002C00u;        // half2(1/16, 1/16)
    const uint32_t km72 = 0xD480D480u;         // half2(-72, -72) = -(64 + 8)
    const uint32_t w8 = w >> 8;
    r[0] = h2_sub(lop3_and_or(w, 0x000F000Fu, magic), k1032);
    r[1] = h2_fma(lop3_and_or(w, 0x00F000F0u, magic), k1_16, km72);
    r[2] = h2_sub(lop3_and_or(w8, 0x000F000Fu, magic), k1032);
    r[3] = h2_fma(lop3_and_or(w8, 0x00F000F0u, magic), k1_16, km72);
}

ER_DEV float h2f_lo(uint32_t h) { return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFF))); }
ER_DEV float h2f_hi(uint32_t h) { return __half2float(__ushort_as_half((unsigned short)(h >> 16))); }

// order-preserving map of a finite float to uint32 (for packed argmax keys)
ER_DEV uint32_t float_order_key(float v) {
    uint32_t b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

}  // namespace er
