// txl_bwd.cu -- gradients of the relative attention (the backward of txl_rel_attn_fwd).
//
// With q' = q + u, q'' = q + v_bias, s_ij = scale (q'_i . k_j + q''_i . r[min(M + i - j, C)]),
// P = softmax over the visible keys and out = P V, an upstream gradient dO gives
//   D_i = dO_i . out_i,  dP_ij = dO_i . v_j,  dS_ij = scale P_ij (dP_ij - D_i)
//   dq_i = sum_j dS_ij (k_j + r[delta_ij]),  dk_j = sum_i dS_ij q'_i,  dv_j = sum_i P_ij dO_i,
//   du = sum dS_ij k_j,  dv_bias = sum dS_ij r[delta_ij],  dr[delta] = sum_{delta_ij = delta} dS_ij q''_i
// (the chain rule through the four-term score of "Transformer-XL 和相对位置编码" §2.3.2 and the
// softmax).  Keys and values of the memory get no gradient: the memory is the stop-gradient
// part of the extended sequence ("Transformer-XL 和相对位置编码" §2.3.1).
//
// Every pass recomputes the scores it needs instead of storing P (fp32 arithmetic throughout),
// one warp per row of work, lane l owning head dimensions l, l+32, l+64, l+96:
//   rows  (b, h, i): log-sum-exp and D_i, then dq_i; the per-query parts of du and dv_bias
//   keys  (b, h, j) of the current segment: dk_j, dv_j
//   dist  (h, delta) for distances below the clamp: dr[delta] over every (b, i)
//   clamp (b, h, i): the pairs whose distance reaches clamp_len, added into dr[C] atomically
//   bias  (h, d): du and dv_bias from the per-query parts
// and the position table's backward dW_R = sum_delta R_delta^T dr[delta] with R the sinusoid.
#include <cmath>

#include <cuda_bf16.h>

#include "txl_internal.h"

namespace txl {

namespace {

constexpr int kBwdWarps = 4;

template <typename T> __device__ __forceinline__ float ldf(const T* p);
template <> __device__ __forceinline__ float ldf<float>(const float* p) { return __ldg(p); }
template <> __device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// Key j (logical, 0 <= j < M + L) of (b, h): the memory ring for j < M, the current segment after.
template <typename T>
__device__ __forceinline__ void key_ptrs(const AttnSimtParams& a, int b, int h, int j, const T*& kp, const T*& vp)
{
    if (j < a.M) {
        const int slot = static_cast<int>((static_cast<int64_t>(a.wp) + j) % a.M);
        const int64_t off = b * a.m_sb + slot * a.m_st + h * a.m_sh;
        kp = static_cast<const T*>(a.kmem) + off;
        vp = static_cast<const T*>(a.vmem) + off;
    } else {
        const int t = j - a.M;
        kp = static_cast<const T*>(a.kcur) + b * a.kc_sb + t * a.kc_st + h * a.kc_sh;
        vp = static_cast<const T*>(a.vcur) + b * a.vc_sb + t * a.vc_st + h * a.vc_sh;
    }
}

// Query i of (b, h): q' = q + u and q'' = q + v_bias in the lane's dimensions.
template <typename T>
__device__ __forceinline__ void load_query(const AttnSimtParams& a, int b, int h, int i, int lane, float* qu, float* qv)
{
    const T* q = static_cast<const T*>(a.q) + b * a.q_sb + i * a.q_st + h * a.q_sh;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int d = lane + 32 * c;
        float x = 0.f, uu = 0.f, vv = 0.f;
        if (d < a.D) {
            x = ldf(q + d);
            uu = __ldg(a.u + h * a.D + d);
            vv = __ldg(a.vb + h * a.D + d);
        }
        qu[c] = x + uu;
        qv[c] = x + vv;
    }
}

template <typename T>
__device__ __forceinline__ void load_vec(const T* p, int D, int lane, float* x)
{
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int d = lane + 32 * c;
        x[c] = d < D ? ldf(p + d) : 0.f;
    }
}

// scale * (q' . k + q'' . r) for the (query, key) pair, reduced over the warp.
template <typename T>
__device__ __forceinline__ float score(const AttnSimtParams& a, const float* qu, const float* qv, const T* kp,
                                       const T* rp, int lane, float* kx, float* rx)
{
    float part = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int d = lane + 32 * c;
        kx[c] = d < a.D ? ldf(kp + d) : 0.f;
        rx[c] = d < a.D ? ldf(rp + d) : 0.f;
        part = fmaf(qu[c], kx[c], fmaf(qv[c], rx[c], part));
    }
    return warp_sum(part) * a.scale;
}

template <typename T>
__device__ __forceinline__ const T* rrow(const AttnSimtParams& a, int h, int delta)
{
    const int dc = delta < a.C ? delta : a.C;
    return static_cast<const T*>(a.r) + dc * a.r_row + h * a.r_head;
}

// ---------------------------------------------------------------------------- rows: dq, lse, D
template <typename T>
__global__ void __launch_bounds__(32 * kBwdWarps) bwd_rows_kernel(const BwdParams p)
{
    const AttnSimtParams& a = p.a;
    const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (gw >= static_cast<int64_t>(a.B) * a.H * a.L) return;
    const int i = static_cast<int>(gw % a.L);
    const int h = static_cast<int>((gw / a.L) % a.H);
    const int b = static_cast<int>(gw / (static_cast<int64_t>(a.L) * a.H));
    float qu[4], qv[4], g[4], o[4], kx[4], rx[4], vx[4];
    load_query<T>(a, b, h, i, lane, qu, qv);
    load_vec(static_cast<const T*>(p.dout) + b * p.g_sb + i * p.g_st + h * p.g_sh, a.D, lane, g);
    load_vec(static_cast<const T*>(a.out) + b * a.o_sb + i * a.o_st + h * a.o_sh, a.D, lane, o);
    float dd = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) dd = fmaf(g[c], o[c], dd);
    dd = warp_sum(dd);
    const int qpos = a.M + i;
    // pass 1: log-sum-exp of the visible scores (online)
    float m = -INFINITY, l = 0.f;
    for (int j = a.lo; j <= qpos; ++j) {
        const T *kp, *vp;
        key_ptrs<T>(a, b, h, j, kp, vp);
        const float s = score<T>(a, qu, qv, kp, rrow<T>(a, h, qpos - j), lane, kx, rx);
        const float mn = fmaxf(m, s);
        l = l * expf(m - mn) + expf(s - mn);
        m = mn;
    }
    const float lse = m + logf(l);
    // pass 2: dS and dq
    float dac[4] = {0.f, 0.f, 0.f, 0.f}, dbd[4] = {0.f, 0.f, 0.f, 0.f};
    for (int j = a.lo; j <= qpos; ++j) {
        const T *kp, *vp;
        key_ptrs<T>(a, b, h, j, kp, vp);
        const float s = score<T>(a, qu, qv, kp, rrow<T>(a, h, qpos - j), lane, kx, rx);
        load_vec(vp, a.D, lane, vx);
        float dp = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) dp = fmaf(g[c], vx[c], dp);
        dp = warp_sum(dp);
        const float ds = a.scale * expf(s - lse) * (dp - dd);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            dac[c] = fmaf(ds, kx[c], dac[c]);
            dbd[c] = fmaf(ds, rx[c], dbd[c]);
        }
    }
    const int64_t row = (static_cast<int64_t>(b) * a.L + i) * a.H + h;     // [B][L][H] row of D
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int d = lane + 32 * c;
        if (d < a.D) {
            p.dq[row * a.D + d] = dac[c] + dbd[c];
            p.pac[row * a.D + d] = dac[c];
            p.pbd[row * a.D + d] = dbd[c];
        }
    }
    if (lane == 0) {
        p.lse[row] = lse;
        p.dd[row] = dd;
    }
}

// ---------------------------------------------------------------------------- keys: dk, dv
template <typename T>
__global__ void __launch_bounds__(32 * kBwdWarps) bwd_keys_kernel(const BwdParams p)
{
    const AttnSimtParams& a = p.a;
    const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (gw >= static_cast<int64_t>(a.B) * a.H * a.L) return;
    const int jc = static_cast<int>(gw % a.L);                 // key of the current segment
    const int h = static_cast<int>((gw / a.L) % a.H);
    const int b = static_cast<int>(gw / (static_cast<int64_t>(a.L) * a.H));
    const T *kp, *vp;
    key_ptrs<T>(a, b, h, a.M + jc, kp, vp);
    float kx[4], vx[4], qu[4], qv[4], g[4], rx[4];
    load_vec(kp, a.D, lane, kx);
    load_vec(vp, a.D, lane, vx);
    float dk[4] = {0.f, 0.f, 0.f, 0.f}, dv[4] = {0.f, 0.f, 0.f, 0.f};
    for (int i = jc; i < a.L; ++i) {                            // queries that see key M + jc
        load_query<T>(a, b, h, i, lane, qu, qv);
        load_vec(static_cast<const T*>(p.dout) + b * p.g_sb + i * p.g_st + h * p.g_sh, a.D, lane, g);
        load_vec(rrow<T>(a, h, i - jc), a.D, lane, rx);
        float part = 0.f, dp = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            part = fmaf(qu[c], kx[c], fmaf(qv[c], rx[c], part));
            dp = fmaf(g[c], vx[c], dp);
        }
        part = warp_sum(part);
        dp = warp_sum(dp);
        const int64_t row = (static_cast<int64_t>(b) * a.L + i) * a.H + h;
        const float pr = expf(part * a.scale - p.lse[row]);
        const float ds = a.scale * pr * (dp - p.dd[row]);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            dk[c] = fmaf(ds, qu[c], dk[c]);
            dv[c] = fmaf(pr, g[c], dv[c]);
        }
    }
    const int64_t row = (static_cast<int64_t>(b) * a.L + jc) * a.H + h;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int d = lane + 32 * c;
        if (d < a.D) {
            p.dk[row * a.D + d] = dk[c];
            p.dv[row * a.D + d] = dv[c];
        }
    }
}

// dS_ij of one visible (query, key) pair, with q''_i of the query left in qv.
template <typename T>
__device__ __forceinline__ float pair_ds(const BwdParams& p, int b, int h, int i, int j, int lane, float* qv)
{
    const AttnSimtParams& a = p.a;
    float qu[4], g[4], kx[4], rx[4], vx[4];
    load_query<T>(a, b, h, i, lane, qu, qv);
    const T *kp, *vp;
    key_ptrs<T>(a, b, h, j, kp, vp);
    const float s = score<T>(a, qu, qv, kp, rrow<T>(a, h, a.M + i - j), lane, kx, rx);
    load_vec(static_cast<const T*>(p.dout) + b * p.g_sb + i * p.g_st + h * p.g_sh, a.D, lane, g);
    load_vec(vp, a.D, lane, vx);
    float dp = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) dp = fmaf(g[c], vx[c], dp);
    dp = warp_sum(dp);
    const int64_t row = (static_cast<int64_t>(b) * a.L + i) * a.H + h;
    return a.scale * expf(s - p.lse[row]) * (dp - p.dd[row]);
}

// ---------------------------------------------------------------------------- distances below the clamp
template <typename T>
__global__ void __launch_bounds__(32 * kBwdWarps) bwd_dist_kernel(const BwdParams p, int n_exact)
{
    const AttnSimtParams& a = p.a;
    const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (gw >= static_cast<int64_t>(a.H) * n_exact) return;
    const int delta = static_cast<int>(gw % n_exact);
    const int h = static_cast<int>(gw / n_exact);
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, qv[4];
    for (int b = 0; b < a.B; ++b)
        for (int i = 0; i < a.L; ++i) {
            const int j = a.M + i - delta;
            if (j < a.lo) continue;                       // before the valid memory (or the sequence)
            const float ds = pair_ds<T>(p, b, h, i, j, lane, qv);
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[c] = fmaf(ds, qv[c], acc[c]);
        }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int d = lane + 32 * c;
        if (d < a.D) p.dr[(static_cast<int64_t>(delta) * a.H + h) * a.D + d] = acc[c];
    }
}

// ---------------------------------------------------------------------------- distances at the clamp
template <typename T>
__global__ void __launch_bounds__(32 * kBwdWarps) bwd_clamp_kernel(const BwdParams p)
{
    const AttnSimtParams& a = p.a;
    const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (gw >= static_cast<int64_t>(a.B) * a.H * a.L) return;
    const int i = static_cast<int>(gw % a.L);
    const int h = static_cast<int>((gw / a.L) % a.H);
    const int b = static_cast<int>(gw / (static_cast<int64_t>(a.L) * a.H));
    const int j_hi = a.M + i - a.C;                       // keys at distance >= clamp_len
    if (j_hi < a.lo) return;
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, qv[4];
    for (int j = a.lo; j <= j_hi; ++j) {
        const float ds = pair_ds<T>(p, b, h, i, j, lane, qv);
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[c] = fmaf(ds, qv[c], acc[c]);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int d = lane + 32 * c;
        if (d < a.D) atomicAdd(p.dr + (static_cast<int64_t>(a.C) * a.H + h) * a.D + d, acc[c]);
    }
}

// ---------------------------------------------------------------------------- du, dv_bias
__global__ void bwd_bias_kernel(const BwdParams p)
{
    const AttnSimtParams& a = p.a;
    const int hd = blockIdx.x * blockDim.x + threadIdx.x;
    const int HD = a.H * a.D;
    if (hd >= HD) return;
    float su = 0.f, sv = 0.f;
    const int64_t rows = static_cast<int64_t>(a.B) * a.L;
    for (int64_t r = 0; r < rows; ++r) {
        su += p.pac[r * HD + hd];
        sv += p.pbd[r * HD + hd];
    }
    p.du[hd] = su;
    p.dvb[hd] = sv;
}

// ---------------------------------------------------------------------------- dW_R = R^T dr
// Block (64 model columns m, 64 columns n = h*D + d); the sinusoid rows R_delta[m] of a chunk of
// 32 distances are evaluated in double precision and rounded to fp32 (as the fp32 forward does).
constexpr int kPosBwdT = 64, kPosBwdChunk = 32;

__global__ void __launch_bounds__(256) pos_bwd_kernel(PosBwdParams p)
{
    __shared__ float Rs[kPosBwdChunk][kPosBwdT + 1];
    __shared__ float Gs[kPosBwdChunk][kPosBwdT + 1];
    const int m0 = blockIdx.y * kPosBwdT, n0 = blockIdx.x * kPosBwdT;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;      // 16 x 16 threads, 4 x 4 outputs each
    float acc[4][4] = {};
    const int HD = p.H * p.D;
    for (int d0 = 0; d0 < p.n_rows; d0 += kPosBwdChunk) {
        for (int e = threadIdx.x; e < kPosBwdChunk * kPosBwdT; e += blockDim.x) {
            const int rr = e / kPosBwdT, cc = e % kPosBwdT;
            const int delta = d0 + rr, m = m0 + cc, n = n0 + cc;
            float rv = 0.f, gv = 0.f;
            if (delta < p.n_rows) {
                if (m < p.d_model) {
                    const int k = m >> 1;
                    const double w = pow(10000.0, -(2.0 * k) / static_cast<double>(p.d_model));
                    const double x = static_cast<double>(delta) * w;
                    rv = static_cast<float>((m & 1) ? cos(x) : sin(x));
                }
                if (n < HD) gv = p.dr[static_cast<int64_t>(delta) * HD + n];
            }
            Rs[rr][cc] = rv;
            Gs[rr][cc] = gv;
        }
        __syncthreads();
#pragma unroll 4
        for (int rr = 0; rr < kPosBwdChunk; ++rr) {
            float rv[4], gv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                rv[e] = Rs[rr][ty + 16 * e];
                gv[e] = Gs[rr][tx + 16 * e];
            }
#pragma unroll
            for (int e = 0; e < 4; ++e)
#pragma unroll
                for (int f = 0; f < 4; ++f) acc[e][f] = fmaf(rv[e], gv[f], acc[e][f]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int f = 0; f < 4; ++f) {
            const int m = m0 + ty + 16 * e, n = n0 + tx + 16 * f;
            if (m < p.d_model && n < HD) p.dW[static_cast<int64_t>(m) * p.ld_dw + n] = acc[e][f];
        }
}

template <typename T>
cudaError_t launch_all(const BwdParams& p, cudaStream_t s)
{
    const AttnSimtParams& a = p.a;
    const int64_t row_warps = static_cast<int64_t>(a.B) * a.H * a.L;
    const int64_t row_blocks = (row_warps + kBwdWarps - 1) / kBwdWarps;
    if (row_blocks > 0x7fffffffll) return cudaErrorInvalidValue;
    const int thr = 32 * kBwdWarps;
    const int n_need = (a.M + a.L < a.C + 1) ? a.M + a.L : a.C + 1;
    const bool clamped = a.C < a.M + a.L - 1;
    const int n_exact = clamped ? a.C : n_need;
    cudaError_t e = cudaMemsetAsync(p.dr, 0, static_cast<size_t>(p.n_rows) * a.H * a.D * sizeof(float), s);
    if (e != cudaSuccess) return e;
    bwd_rows_kernel<T><<<static_cast<unsigned>(row_blocks), thr, 0, s>>>(p);
    bwd_keys_kernel<T><<<static_cast<unsigned>(row_blocks), thr, 0, s>>>(p);
    const int64_t dist_blocks = (static_cast<int64_t>(a.H) * n_exact + kBwdWarps - 1) / kBwdWarps;
    if (dist_blocks > 0) bwd_dist_kernel<T><<<static_cast<unsigned>(dist_blocks), thr, 0, s>>>(p, n_exact);
    if (clamped) bwd_clamp_kernel<T><<<static_cast<unsigned>(row_blocks), thr, 0, s>>>(p);
    const int HD = a.H * a.D;
    bwd_bias_kernel<<<(HD + 127) / 128, 128, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rel_attn_bwd(const BwdParams& p, txl_dtype dtype, cudaStream_t s)
{
    if (static_cast<int64_t>(p.a.B) * p.a.H * p.a.L == 0) return cudaSuccess;
    return dtype == TXL_F32 ? launch_all<float>(p, s) : launch_all<__nv_bfloat16>(p, s);
}

cudaError_t launch_pos_bwd(const PosBwdParams& p, cudaStream_t s)
{
    if (p.d_model == 0) return cudaSuccess;
    if (p.n_rows == 0)
        return cudaMemset2DAsync(p.dW, static_cast<size_t>(p.ld_dw) * sizeof(float), 0,
                                 sizeof(float) * p.H * p.D, p.d_model, s);
    dim3 grid((p.H * p.D + kPosBwdT - 1) / kPosBwdT, (p.d_model + kPosBwdT - 1) / kPosBwdT);
    pos_bwd_kernel<<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace txl
