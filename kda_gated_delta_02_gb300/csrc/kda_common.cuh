// kda_common.cuh -- device helpers shared by the KDA kernels (sm_103a).
//
// Warp-level bf16 tensor-core products (mma.sync m16n8k16, fp32 accumulate),
// ldmatrix fragment loads, 16-byte cp.async staging and small conversions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

// ------------------------------------------------------------------ conversions
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low 16 bits)
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&u);
    return __bfloat1622float2(v);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ tensor cores
// D = A(16x16, row) * B(16x8, col) + C, bf16 inputs, fp32 accumulate.
// Fragment ownership (g = lane/4, q = lane%4):
//   A: a0 (g, 2q..2q+1)  a1 (g+8, 2q..)  a2 (g, 2q+8..)  a3 (g+8, 2q+8..)
//   B: b0 (k 2q..2q+1, n g)  b1 (k 2q+8.., n g)
//   C: c0 (g, 2q)  c1 (g, 2q+1)  c2 (g+8, 2q)  c3 (g+8, 2q+1)
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D = A(16x8, row) * B(8x8, col) + C in tf32 with fp32 accumulate.
//   A: a0 (g, q)  a1 (g+8, q)  a2 (g, q+4)  a3 (g+8, q+4);  B: b0 (k q, n g)  b1 (k q+4, n g)
//   C: as for the bf16 shape.
__device__ __forceinline__ void mma_tf32(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// x = hi + lo with hi, lo representable in tf32: products hi*hi + hi*lo + lo*hi
// keep about 21 mantissa bits (fp32-level accuracy from tf32 tensor products).
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
    uint32_t h;
    asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(h) : "f"(x));
    const float r = x - __uint_as_float(h);
    uint32_t l;
    asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(l) : "f"(r));
    hi = h;
    lo = l;
}

// Four 8x8 b16 matrices; lane l supplies the row address of matrix l/8, row l%8.
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// A fragment (16x16) of a row-major [m][k] bf16 array with row stride `ld`
// elements, tile origin (m0, k0).
__device__ __forceinline__ void ld_a_rowmajor(uint32_t (&a)[4], const __nv_bfloat16 *base, int ld,
                                              int m0, int k0, int lane) {
    int mi = lane >> 3, r = lane & 7;
    const __nv_bfloat16 *p = base + (size_t)(m0 + r + 8 * (mi & 1)) * ld + k0 + 8 * (mi >> 1);
    ldsm_x4(a, smem_u32(p));
}

// A fragment of A = X^T where X is a row-major [k][m] bf16 array.
__device__ __forceinline__ void ld_a_transposed(uint32_t (&a)[4], const __nv_bfloat16 *base, int ld,
                                                int m0, int k0, int lane) {
    int mi = lane >> 3, r = lane & 7;
    const __nv_bfloat16 *p = base + (size_t)(k0 + r + 8 * (mi >> 1)) * ld + m0 + 8 * (mi & 1);
    ldsm_x4_t(a, smem_u32(p));
}

// B fragments of two adjacent n8 tiles (n0..n0+15), k16 step at k0, from a
// row-major [k][n] bf16 array.  b[0],b[1] -> tile n0; b[2],b[3] -> tile n0+8.
__device__ __forceinline__ void ld_b_kmajor_rows(uint32_t (&b)[4], const __nv_bfloat16 *base, int ld,
                                                 int k0, int n0, int lane) {
    int mi = lane >> 3, r = lane & 7;
    const __nv_bfloat16 *p = base + (size_t)(k0 + r + 8 * (mi & 1)) * ld + n0 + 8 * (mi >> 1);
    ldsm_x4_t(b, smem_u32(p));
}

// ------------------------------------------------------------------ async copies
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src, bool valid) {
    uint32_t d = smem_u32(smem_dst);
    int n = valid ? 16 : 0;  // 0 source bytes: the 16 destination bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(gmem_src), "r"(n));
}
__device__ __forceinline__ void cp_async4(void *smem_dst, const void *gmem_src, bool valid) {
    uint32_t d = smem_u32(smem_dst);
    int n = valid ? 4 : 0;
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(d), "l"(gmem_src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::); }

// 32-bit shared-state-space accesses by address (keeps address math 32-bit)
__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void sts16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.b16 [%0], %1;\n" ::"r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ void sts64(uint32_t addr, uint32_t a, uint32_t b) {
    asm volatile("st.shared.v2.b32 [%0], {%1, %2};\n" ::"r"(addr), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ uint16_t lds16(uint32_t addr) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];\n" : "=h"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];\n" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void report_status(uint32_t *status, uint32_t bits) {
    if (status) atomicOr(status, bits);
}

}  // namespace kda
