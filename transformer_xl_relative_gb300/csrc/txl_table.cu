// txl_table.cu -- the learned-table variant of the relative attention ("TransformerXL 相对位置编码"
// §3.1): bidirectional attention over one sequence (no memory), the position vector of a pair read
// from a projected lookup table at rel(i, j) = clamp(i - j + max_len - 1, 0, 2 max_len - 2) (§2: the
// distance shifted to a non-negative index and clamped), and the score
//   scale q_i.k_j + scale q_i.r_rel + u.k_j + v.r_rel  =  (scale q_i + u).k_j + (scale q_i + v).r_rel
// with the scale on the first two terms only, as that page computes it; keys whose mask entry is 0
// take the score -1e9 (so a row with every key masked averages the values uniformly).
//
// One warp per four consecutive queries of one (b, h), lane l owning dimensions l, l+32, l+64,
// l+96; keys in increasing order with an online softmax per query.  The table row of query g at
// key j + 1 is the row query g - 1 used at key j, so a key costs its k and v rows and one new
// table row.
#include <cuda_bf16.h>

#include "txl_internal.h"

namespace txl {

namespace {

constexpr int kTabWarps = 4;
constexpr int kTG = 4;

template <typename T> __device__ __forceinline__ float tldf(const T* p);
template <> __device__ __forceinline__ float tldf<float>(const float* p) { return __ldg(p); }
template <> __device__ __forceinline__ float tldf<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }
template <typename T> __device__ __forceinline__ void tstf(T* p, float v);
template <> __device__ __forceinline__ void tstf<float>(float* p, float v) { *p = v; }
template <> __device__ __forceinline__ void tstf<__nv_bfloat16>(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

template <typename T, int DC>
__device__ __forceinline__ void tload(const T* p, int D, int lane, float* x)
{
#pragma unroll
    for (int c = 0; c < DC; ++c) {
        const int d = lane + 32 * c;
        x[c] = d < D ? tldf(p + d) : 0.f;
    }
}

// Sums of the warp's kTG partial dot products, left in every lane (transposing butterfly: two
// exchanges that halve the values per lane, three plain ones, one broadcast per value).
__device__ __forceinline__ void tsum4(float* v, int lane)
{
    float w0, w1;
    {
        const bool hi = lane & 16;
        w0 = (hi ? v[2] : v[0]) + __shfl_xor_sync(0xffffffffu, hi ? v[0] : v[2], 16);
        w1 = (hi ? v[3] : v[1]) + __shfl_xor_sync(0xffffffffu, hi ? v[1] : v[3], 16);
    }
    {
        const bool hi = lane & 8;
        w0 = (hi ? w1 : w0) + __shfl_xor_sync(0xffffffffu, hi ? w0 : w1, 8);
    }
#pragma unroll
    for (int bit = 4; bit > 0; bit >>= 1) w0 += __shfl_xor_sync(0xffffffffu, w0, bit);
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = __shfl_sync(0xffffffffu, w0, k << 3);
}

template <typename T, int DC>
__global__ void __launch_bounds__(32 * kTabWarps) table_attn_kernel(const TableParams p)
{
    const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int nq = (p.L + kTG - 1) / kTG;
    if (gw >= static_cast<int64_t>(p.B) * p.H * nq) return;
    const int i0 = static_cast<int>(gw % nq) * kTG;
    const int h = static_cast<int>((gw / nq) % p.H);
    const int b = static_cast<int>(gw / (static_cast<int64_t>(nq) * p.H));
    const int top = 2 * p.max_len - 2;
    auto trow = [&](int idx) {
        const int c = idx < 0 ? 0 : (idx > top ? top : idx);
        return static_cast<const T*>(p.r) + c * p.r_row + h * p.r_head;
    };
    float qa[kTG][DC], qb[kTG][DC], o[kTG][DC], m[kTG], l[kTG], rx[kTG][DC];
#pragma unroll
    for (int g = 0; g < kTG; ++g) {
        const int i = min(i0 + g, p.L - 1);
        const T* qp = static_cast<const T*>(p.q) + b * p.q_sb + i * p.q_st + h * p.q_sh;
#pragma unroll
        for (int c = 0; c < DC; ++c) {
            const int d = lane + 32 * c;
            float x = 0.f, uu = 0.f, vv = 0.f;
            if (d < p.D) {
                x = tldf(qp + d) * p.scale;
                uu = __ldg(p.u + h * p.D + d);
                vv = __ldg(p.vb + h * p.D + d);
            }
            qa[g][c] = x + uu;
            qb[g][c] = x + vv;
            o[g][c] = 0.f;
        }
        m[g] = -INFINITY;
        l[g] = 0.f;
        tload<T, DC>(trow(i0 + g + p.max_len - 1), p.D, lane, rx[g]);     // key 0
    }
    for (int j = 0; j < p.L; ++j) {
        const T* kp = static_cast<const T*>(p.k) + b * p.k_sb + j * p.k_st + h * p.k_sh;
        const T* vp = static_cast<const T*>(p.v) + b * p.v_sb + j * p.v_st + h * p.v_sh;
        float kx[DC], vx[DC], rn[DC];
        tload<T, DC>(kp, p.D, lane, kx);
        tload<T, DC>(vp, p.D, lane, vx);
        tload<T, DC>(trow(i0 - j - 1 + p.max_len - 1), p.D, lane, rn);      // query 0 at key j + 1
        const bool masked = p.mask && p.mask[static_cast<int64_t>(b) * p.L + j] == 0;
        float s[kTG];
#pragma unroll
        for (int g = 0; g < kTG; ++g) {
            float x = 0.f;
#pragma unroll
            for (int c = 0; c < DC; ++c) x = fmaf(qa[g][c], kx[c], fmaf(qb[g][c], rx[g][c], x));
            s[g] = x;
        }
        tsum4(s, lane);
#pragma unroll
        for (int g = 0; g < kTG; ++g) {
            const float sg = masked ? -1e9f : s[g];
            const float mn = fmaxf(m[g], sg);
            const float alpha = __expf(m[g] - mn), pe = __expf(sg - mn);
            l[g] = fmaf(l[g], alpha, pe);
#pragma unroll
            for (int c = 0; c < DC; ++c) o[g][c] = fmaf(o[g][c], alpha, pe * vx[c]);
            m[g] = mn;
        }
#pragma unroll
        for (int g = kTG - 1; g > 0; --g)
#pragma unroll
            for (int c = 0; c < DC; ++c) rx[g][c] = rx[g - 1][c];
#pragma unroll
        for (int c = 0; c < DC; ++c) rx[0][c] = rn[c];
    }
#pragma unroll
    for (int g = 0; g < kTG; ++g) {
        const int i = i0 + g;
        if (i >= p.L) break;
        T* op = static_cast<T*>(p.out) + b * p.o_sb + i * p.o_st + h * p.o_sh;
        const float inv = 1.f / l[g];
#pragma unroll
        for (int c = 0; c < DC; ++c) {
            const int d = lane + 32 * c;
            if (d < p.D) tstf(op + d, o[g][c] * inv);
        }
    }
}

template <typename T>
cudaError_t launch_t(const TableParams& p, cudaStream_t s)
{
    const int64_t warps = static_cast<int64_t>(p.B) * p.H * ((p.L + kTG - 1) / kTG);
    const int64_t blocks = (warps + kTabWarps - 1) / kTabWarps;
    if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
    if (p.D <= 64)
        table_attn_kernel<T, 2><<<static_cast<unsigned>(blocks), 32 * kTabWarps, 0, s>>>(p);
    else
        table_attn_kernel<T, 4><<<static_cast<unsigned>(blocks), 32 * kTabWarps, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_table_attn(const TableParams& p, txl_dtype dtype, cudaStream_t s)
{
    if (static_cast<int64_t>(p.B) * p.H * p.L == 0) return cudaSuccess;
    if (table_tc_eligible(p, dtype)) return launch_table_tc(p, s);
    return dtype == TXL_F32 ? launch_t<float>(p, s) : launch_t<__nv_bfloat16>(p, s);
}

}  // namespace txl
