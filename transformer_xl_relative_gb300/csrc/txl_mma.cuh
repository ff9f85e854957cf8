// txl_mma.cuh -- warp-level bf16 tensor-core helpers (mma.sync m16n8k16, ldmatrix, cp.async) and
// the swizzled shared-memory layout of 64- and 128-element bf16 rows they read, shared by the
// tensor-core backward and the learned-table kernel.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>

namespace txl {
namespace mma {

// Rows of 64 bf16 are stored as 128-byte rows with the 16-byte chunk index xor-ed with the row
// (mod 8), so that ldmatrix reads of eight rows hit eight different bank groups; rows of 128 bf16
// xor the low three chunk bits.
__device__ __forceinline__ uint32_t swz64(int row, int col)        // byte offset, 64-wide rows
{
    return static_cast<uint32_t>(row * 128 + ((((col >> 3) ^ row) & 7) << 4) + (col & 7) * 2);
}
__device__ __forceinline__ uint32_t swz128(int row, int col)       // byte offset, 128-wide rows
{
    const int c = col >> 3;
    return static_cast<uint32_t>(row * 256 + (((c & 8) | ((c ^ row) & 7)) << 4) + (col & 7) * 2);
}

__device__ __forceinline__ uint32_t cvta_smem(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// D += A B: m16n8k16, A row-major bf16, B column-major bf16, fp32 accumulators.
__device__ __forceinline__ void mma16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float ex2(float x)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Fragment addresses (lane l) for ldmatrix.x4, see the fragment layouts of mma.m16n8k16:
//  A 16x16 at (r0, c0) of a row-major [m][k] tile (non-transposed load)
__device__ __forceinline__ void a_rc(int lane, int r0, int c0, int& r, int& c)
{
    r = r0 + (lane & 7) + ((lane >> 3) & 1) * 8;
    c = c0 + (lane >> 4) * 8;
}
//  B of two n-tiles (n0 .. n0+15) x k16 (k0 ..) from an [n][k] tile (non-transposed load)
__device__ __forceinline__ void b_nk(int lane, int n0, int k0, int& r, int& c)
{
    r = n0 + (lane & 7) + (lane >> 4) * 8;
    c = k0 + ((lane >> 3) & 1) * 8;
}
//  B of two n-tiles from a [k][n] tile (transposed load)
__device__ __forceinline__ void b_kn(int lane, int k0, int n0, int& r, int& c)
{
    r = k0 + (lane & 7) + ((lane >> 3) & 1) * 8;
    c = n0 + (lane >> 4) * 8;
}
//  A 16x16 at (m0, k0) from a [k][m] tile (transposed load)
__device__ __forceinline__ void a_km(int lane, int m0, int k0, int& r, int& c)
{
    r = k0 + (lane & 7) + (lane >> 4) * 8;
    c = m0 + ((lane >> 3) & 1) * 8;
}

// 16-byte asynchronous copy into shared memory; src_bytes = 0 fills the 16 bytes with zeros.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(cvta_smem(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

}  // namespace mma
}  // namespace txl
