// txl_attn_simt.cu -- relative attention, one warp per (batch, head, query), any layout.
//
// Serves the fp32 path and every bf16 request the fused tensor-core kernel does not take
// (D > 128, strides that are not 16-byte aligned, a ring memory whose write pointer is not a
// multiple of 128).  Lane l owns head dimensions l, l+32, l+64, l+96.  Keys are visited in
// order with an online softmax; each score is the four-term sum of
// "跨窗口的相对位置编码" §3, written as (q+u).k + (q+v).r[delta_c], scaled, and masked keys are
// never visited ("TransformerXL 相对位置编码" §4.2-4.3).
#include <cuda_bf16.h>

#include "txl_internal.h"

namespace txl {

namespace {

constexpr int kSimtWarps = 4;

template <typename T> __device__ __forceinline__ float ld_f(const T* p);
template <> __device__ __forceinline__ float ld_f<float>(const float* p) { return __ldg(p); }
template <> __device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16* p)
{
    return __bfloat162float(*p);
}
template <typename T> __device__ __forceinline__ void st_f(T* p, float v);
template <> __device__ __forceinline__ void st_f<float>(float* p, float v) { *p = v; }
template <> __device__ __forceinline__ void st_f<__nv_bfloat16>(__nv_bfloat16* p, float v)
{
    *p = __float2bfloat16_rn(v);
}

template <typename T>
__global__ void __launch_bounds__(32 * kSimtWarps) attn_simt_kernel(AttnSimtParams p)
{
    const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t total = static_cast<int64_t>(p.B) * p.H * p.L;
    if (gw >= total) return;
    const int i = static_cast<int>(gw % p.L);
    const int h = static_cast<int>((gw / p.L) % p.H);
    const int b = static_cast<int>(gw / (static_cast<int64_t>(p.L) * p.H));

    const T* q = static_cast<const T*>(p.q) + b * p.q_sb + i * p.q_st + h * p.q_sh;
    float qu[4], qv[4], o[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int d = lane + 32 * c;
        float x = 0.f, uu = 0.f, vv = 0.f;
        if (d < p.D) {
            x = ld_f(q + d);
            uu = __ldg(p.u + h * p.D + d);
            vv = __ldg(p.vb + h * p.D + d);
        }
        qu[c] = x + uu;
        qv[c] = x + vv;
        o[c] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    const int qpos = p.M + i;
    for (int j = p.lo; j <= qpos; ++j) {
        const T* kp;
        const T* vp;
        if (j < p.M) {
            int slot = static_cast<int>((static_cast<int64_t>(p.wp) + j) % p.M);
            if (!in_range(slot, 0, p.M, p.chk)) slot = 0;
            const int64_t off = b * p.m_sb + slot * p.m_st + h * p.m_sh;
            kp = static_cast<const T*>(p.kmem) + off;
            vp = static_cast<const T*>(p.vmem) + off;
        } else {
            const int t = j - p.M;
            kp = static_cast<const T*>(p.kcur) + b * p.kc_sb + t * p.kc_st + h * p.kc_sh;
            vp = static_cast<const T*>(p.vcur) + b * p.vc_sb + t * p.vc_st + h * p.vc_sh;
        }
        const int delta = qpos - j;
        int dc = delta < p.C ? delta : p.C;
        if (!in_range(dc, 0, p.n_rows, p.chk)) dc = 0;
        const T* rp = static_cast<const T*>(p.r) + dc * p.r_row + h * p.r_head;
        float part = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int d = lane + 32 * c;
            if (d < p.D) part = fmaf(qu[c], ld_f(kp + d), fmaf(qv[c], ld_f(rp + d), part));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        const float s = part * p.scale;
        const float m_new = fmaxf(m, s);
        const float alpha = expf(m - m_new);
        const float pe = expf(s - m_new);
        l = fmaf(l, alpha, pe);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int d = lane + 32 * c;
            const float vv = d < p.D ? ld_f(vp + d) : 0.f;
            o[c] = fmaf(o[c], alpha, pe * vv);
        }
        m = m_new;
    }
    T* out = static_cast<T*>(p.out) + b * p.o_sb + i * p.o_st + h * p.o_sh;
    const float inv = 1.f / l;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int d = lane + 32 * c;
        if (d < p.D) st_f(out + d, o[c] * inv);
    }
}

}  // namespace

cudaError_t launch_attn_simt(const AttnSimtParams& p, txl_dtype dtype, cudaStream_t s)
{
    const int64_t warps = static_cast<int64_t>(p.B) * p.H * p.L;
    if (warps == 0) return cudaSuccess;
    const int64_t blocks = (warps + kSimtWarps - 1) / kSimtWarps;
    if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
    if (dtype == TXL_F32)
        attn_simt_kernel<float><<<static_cast<unsigned>(blocks), 32 * kSimtWarps, 0, s>>>(p);
    else
        attn_simt_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), 32 * kSimtWarps, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace txl
