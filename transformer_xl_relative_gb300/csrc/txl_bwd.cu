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
// and the launch of the position table's backward dW_R = sum_delta R_delta^T dr[delta]
// (txl_pos_bwd_tc.cu).
#include <cmath>

#include <cuda_bf16.h>

#include "txl_internal.h"

namespace txl {

namespace {

constexpr int kBwdWarps = 4;
constexpr int kG = 4;          // queries, keys or distances per warp: neighbours share operand rows

template <typename T> __device__ __forceinline__ float ldf(const T* p);
template <> __device__ __forceinline__ float ldf<float>(const float* p) { return __ldg(p); }
template <> __device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// Warp-wide sums of 2^LOG values at once, left in every lane.  A transposing butterfly halves the
// values each lane carries per exchange (xor 16, 8, ... : lane l ends with value index taken from
// its high bits), plain exchanges finish the sums, and one shuffle per value broadcasts it:
// for 8 values 4 + 2 + 1 + 2 + 8 = 17 shuffles instead of 8 x 5 = 40.
template <int LOG>
__device__ __forceinline__ void warp_sums(float* v, int lane)
{
    constexpr int N = 1 << LOG;
    float w[N];
#pragma unroll
    for (int k = 0; k < N; ++k) w[k] = v[k];
    int n = N;
#pragma unroll
    for (int r = 0; r < LOG; ++r) {
        const int bit = 16 >> r;                       // lane bit of this exchange
        const bool hi = lane & bit;
        n >>= 1;
#pragma unroll
        for (int m = 0; m < N / 2; ++m) {
            if (m < n) {
                const float keep = hi ? w[m + n] : w[m];
                const float send = hi ? w[m] : w[m + n];
                w[m] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
            }
        }
    }
#pragma unroll
    for (int bit = 16 >> LOG; bit > 0; bit >>= 1) w[0] += __shfl_xor_sync(0xffffffffu, w[0], bit);
    // lane l now holds the sum of value k = (l >> (5 - LOG)); broadcast each
#pragma unroll
    for (int k = 0; k < N; ++k) v[k] = __shfl_sync(0xffffffffu, w[0], k << (5 - LOG));
}

// Key j (logical, 0 <= j < M + L) of (b, h): the memory ring for j < M, the current segment after.
template <typename T>
__device__ __forceinline__ void key_ptrs(const AttnSimtParams& a, int b, int h, int j, const T*& kp, const T*& vp)
{
    if (j < a.M) {
        int slot = a.wp + j;                              // wp < M and j < M: one subtraction wraps it
        if (slot >= a.M) slot -= a.M;
        const int64_t off = b * a.m_sb + slot * a.m_st + h * a.m_sh;
        kp = static_cast<const T*>(a.kmem) + off;
        vp = static_cast<const T*>(a.vmem) + off;
    } else {
        const int t = j - a.M;
        kp = static_cast<const T*>(a.kcur) + b * a.kc_sb + t * a.kc_st + h * a.kc_sh;
        vp = static_cast<const T*>(a.vcur) + b * a.vc_sb + t * a.vc_st + h * a.vc_sh;
    }
}

template <typename T, int DC>
__device__ __forceinline__ void load_vec(const T* p, int D, int lane, float* x)
{
#pragma unroll
    for (int c = 0; c < DC; ++c) {
        const int d = lane + 32 * c;
        x[c] = d < D ? ldf(p + d) : 0.f;
    }
}

// Query i of (b, h): q' = q + u and q'' = q + v_bias in the lane's dimensions.
template <typename T, int DC>
__device__ __forceinline__ void load_query(const AttnSimtParams& a, int b, int h, int i, int lane, float* qu, float* qv)
{
    const T* q = static_cast<const T*>(a.q) + b * a.q_sb + i * a.q_st + h * a.q_sh;
#pragma unroll
    for (int c = 0; c < DC; ++c) {
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
__device__ __forceinline__ const T* rrow(const AttnSimtParams& a, int h, int delta)
{
    const int dc = delta < 0 ? 0 : (delta < a.C ? delta : a.C);       // negative: a masked pair
    return static_cast<const T*>(a.r) + dc * a.r_row + h * a.r_head;
}

template <typename T>
__device__ __forceinline__ const T* gout(const BwdParams& p, int b, int h, int i)
{
    return static_cast<const T*>(p.dout) + b * p.g_sb + i * p.g_st + h * p.g_sh;
}

__device__ __forceinline__ int64_t qrow(const AttnSimtParams& a, int b, int i, int h)
{
    return (static_cast<int64_t>(b) * a.L + i) * a.H + h;                // [B][L][H] row
}

// ---------------------------------------------------------------------------- rows: dq, lse, D
// Warp = kG consecutive queries i0 + g of one (b, h).  Keys are visited in increasing order; the
// position row of query g at key j + 1 is the row query g - 1 used at key j, so each key costs
// one new r row (for g = 0), its k row, and (second pass) its v row.
template <typename T, int DC>
__global__ void __launch_bounds__(32 * kBwdWarps) bwd_rows_kernel(const BwdParams p)
{
    const AttnSimtParams& a = p.a;
    const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int nq = (a.L + kG - 1) / kG;
    if (gw >= static_cast<int64_t>(a.B) * a.H * nq) return;
    const int i0 = static_cast<int>(gw % nq) * kG;
    const int h = static_cast<int>((gw / nq) % a.H);
    const int b = static_cast<int>(gw / (static_cast<int64_t>(nq) * a.H));
    float qu[kG][DC], qv[kG][DC], go[kG][DC], dd[kG];
#pragma unroll
    for (int g = 0; g < kG; ++g) {
        const int i = min(i0 + g, a.L - 1);               // rows past L repeat the last (not stored)
        load_query<T, DC>(a, b, h, i, lane, qu[g], qv[g]);
        float o[DC];
        load_vec<T, DC>(gout<T>(p, b, h, i), a.D, lane, go[g]);
        load_vec<T, DC>(static_cast<const T*>(a.out) + b * a.o_sb + i * a.o_st + h * a.o_sh, a.D, lane, o);
        float x = 0.f;
#pragma unroll
        for (int c = 0; c < DC; ++c) x = fmaf(go[g][c], o[c], x);
        dd[g] = warp_sum(x);
    }
    const int j_end = a.M + min(i0 + kG - 1, a.L - 1);  // the last query's diagonal
    float lse[kG];
    {
        float m[kG], l[kG], rx[kG][DC];
#pragma unroll
        for (int g = 0; g < kG; ++g) {
            m[g] = -INFINITY;
            l[g] = 0.f;
            load_vec<T, DC>(rrow<T>(a, h, a.M + i0 + g - a.lo), a.D, lane, rx[g]);
        }
        // software pipeline: the next key's k row and the next r row are requested before the
        // current key's arithmetic
        float kn[DC], rn[DC];
        {
            const T *kp, *vp;
            key_ptrs<T>(a, b, h, a.lo, kp, vp);
            load_vec<T, DC>(kp, a.D, lane, kn);
        }
        for (int j = a.lo; j <= j_end; ++j) {
            float kx[DC];
#pragma unroll
            for (int c = 0; c < DC; ++c) kx[c] = kn[c];
            if (j < j_end) {
                const T *kp, *vp;
                key_ptrs<T>(a, b, h, j + 1, kp, vp);
                load_vec<T, DC>(kp, a.D, lane, kn);
            }
            load_vec<T, DC>(rrow<T>(a, h, a.M + i0 - j - 1), a.D, lane, rn);
            float part[kG];
#pragma unroll
            for (int g = 0; g < kG; ++g) {
                float x = 0.f;
#pragma unroll
                for (int c = 0; c < DC; ++c) x = fmaf(qu[g][c], kx[c], fmaf(qv[g][c], rx[g][c], x));
                part[g] = x;
            }
            warp_sums<2>(part, lane);
#pragma unroll
            for (int g = 0; g < kG; ++g) {
                if (j <= a.M + i0 + g) {                  // visible to query g
                    const float s = part[g] * a.scale;
                    const float mn = fmaxf(m[g], s);
                    l[g] = l[g] * __expf(m[g] - mn) + __expf(s - mn);
                    m[g] = mn;
                }
            }
            // next key: query g takes query g-1's row, query 0 its next (smaller) distance
#pragma unroll
            for (int g = kG - 1; g > 0; --g)
#pragma unroll
                for (int c = 0; c < DC; ++c) rx[g][c] = rx[g - 1][c];
#pragma unroll
            for (int c = 0; c < DC; ++c) rx[0][c] = rn[c];
        }
#pragma unroll
        for (int g = 0; g < kG; ++g) lse[g] = m[g] + __logf(l[g]);
    }
    float dac[kG][DC], dbd[kG][DC], rx[kG][DC];
#pragma unroll
    for (int g = 0; g < kG; ++g) {
#pragma unroll
        for (int c = 0; c < DC; ++c) dac[g][c] = dbd[g][c] = 0.f;
        load_vec<T, DC>(rrow<T>(a, h, a.M + i0 + g - a.lo), a.D, lane, rx[g]);
    }
    float kn[DC], vn[DC], rn[DC];
    {
        const T *kp, *vp;
        key_ptrs<T>(a, b, h, a.lo, kp, vp);
        load_vec<T, DC>(kp, a.D, lane, kn);
        load_vec<T, DC>(vp, a.D, lane, vn);
    }
    for (int j = a.lo; j <= j_end; ++j) {
        float kx[DC], vx[DC];
#pragma unroll
        for (int c = 0; c < DC; ++c) {
            kx[c] = kn[c];
            vx[c] = vn[c];
        }
        if (j < j_end) {
            const T *kp, *vp;
            key_ptrs<T>(a, b, h, j + 1, kp, vp);
            load_vec<T, DC>(kp, a.D, lane, kn);
            load_vec<T, DC>(vp, a.D, lane, vn);
        }
        load_vec<T, DC>(rrow<T>(a, h, a.M + i0 - j - 1), a.D, lane, rn);
        float part[kG], dp[kG];
#pragma unroll
        for (int g = 0; g < kG; ++g) {
            float x = 0.f, y = 0.f;
#pragma unroll
            for (int c = 0; c < DC; ++c) {
                x = fmaf(qu[g][c], kx[c], fmaf(qv[g][c], rx[g][c], x));
                y = fmaf(go[g][c], vx[c], y);
            }
            part[g] = x;
            dp[g] = y;
        }
        {
            float both[2 * kG];
#pragma unroll
            for (int g = 0; g < kG; ++g) {
                both[g] = part[g];
                both[kG + g] = dp[g];
            }
            warp_sums<3>(both, lane);
#pragma unroll
            for (int g = 0; g < kG; ++g) {
                part[g] = both[g];
                dp[g] = both[kG + g];
            }
        }
#pragma unroll
        for (int g = 0; g < kG; ++g) {
            const float ds = (j <= a.M + i0 + g) ? a.scale * __expf(part[g] * a.scale - lse[g]) * (dp[g] - dd[g]) : 0.f;
#pragma unroll
            for (int c = 0; c < DC; ++c) {
                dac[g][c] = fmaf(ds, kx[c], dac[g][c]);
                dbd[g][c] = fmaf(ds, rx[g][c], dbd[g][c]);
            }
        }
#pragma unroll
        for (int g = kG - 1; g > 0; --g)
#pragma unroll
            for (int c = 0; c < DC; ++c) rx[g][c] = rx[g - 1][c];
#pragma unroll
        for (int c = 0; c < DC; ++c) rx[0][c] = rn[c];
    }
#pragma unroll
    for (int g = 0; g < kG; ++g) {
        const int i = i0 + g;
        if (i >= a.L) break;
        const int64_t row = qrow(a, b, i, h);
#pragma unroll
        for (int c = 0; c < DC; ++c) {
            const int d = lane + 32 * c;
            if (d < a.D) {
                p.dq[row * a.D + d] = dac[g][c] + dbd[g][c];
                p.pac[row * a.D + d] = dac[g][c];
                p.pbd[row * a.D + d] = dbd[g][c];
            }
        }
        if (lane == 0) {
            p.lse[row] = lse[g];
            p.dd[row] = dd[g];
        }
    }
}

// ---------------------------------------------------------------------------- keys: dk, dv
// Warp = kG consecutive keys jc0 + g of the current segment of one (b, h).  Queries are visited
// in increasing order (query i sees key jc iff i >= jc); key g's position row at query i + 1 is
// key g - 1's row at query i, so each query costs its q and dO rows and one new r row.
template <typename T, int DC>
__global__ void __launch_bounds__(32 * kBwdWarps) bwd_keys_kernel(const BwdParams p)
{
    const AttnSimtParams& a = p.a;
    const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int nk = (a.L + kG - 1) / kG;
    if (gw >= static_cast<int64_t>(a.B) * a.H * nk) return;
    const int jc0 = static_cast<int>(gw % nk) * kG;
    const int h = static_cast<int>((gw / nk) % a.H);
    const int b = static_cast<int>(gw / (static_cast<int64_t>(nk) * a.H));
    float kx[kG][DC], vx[kG][DC], dk[kG][DC], dv[kG][DC], rx[kG][DC];
#pragma unroll
    for (int g = 0; g < kG; ++g) {
        const T *kp, *vp;
        key_ptrs<T>(a, b, h, a.M + min(jc0 + g, a.L - 1), kp, vp);
        load_vec<T, DC>(kp, a.D, lane, kx[g]);
        load_vec<T, DC>(vp, a.D, lane, vx[g]);
#pragma unroll
        for (int c = 0; c < DC; ++c) dk[g][c] = dv[g][c] = 0.f;
        load_vec<T, DC>(rrow<T>(a, h, -g), a.D, lane, rx[g]);        // distance at query jc0
    }
    // software pipeline: the next query's rows and r row are requested before this query's arithmetic
    float qun[DC], qvn[DC], gon[DC], rn[DC], lsen, ddn;
    load_query<T, DC>(a, b, h, jc0, lane, qun, qvn);
    load_vec<T, DC>(gout<T>(p, b, h, jc0), a.D, lane, gon);
    lsen = p.lse[qrow(a, b, jc0, h)];
    ddn = p.dd[qrow(a, b, jc0, h)];
    for (int i = jc0; i < a.L; ++i) {
        float qu[DC], qv[DC], go[DC];
#pragma unroll
        for (int c = 0; c < DC; ++c) {
            qu[c] = qun[c];
            qv[c] = qvn[c];
            go[c] = gon[c];
        }
        const float lse = lsen, ddi = ddn;
        if (i + 1 < a.L) {
            load_query<T, DC>(a, b, h, i + 1, lane, qun, qvn);
            load_vec<T, DC>(gout<T>(p, b, h, i + 1), a.D, lane, gon);
            lsen = p.lse[qrow(a, b, i + 1, h)];
            ddn = p.dd[qrow(a, b, i + 1, h)];
        }
        load_vec<T, DC>(rrow<T>(a, h, i + 1 - jc0), a.D, lane, rn);
        float part[kG], dp[kG];
#pragma unroll
        for (int g = 0; g < kG; ++g) {
            float x = 0.f, y = 0.f;
#pragma unroll
            for (int c = 0; c < DC; ++c) {
                x = fmaf(qu[c], kx[g][c], fmaf(qv[c], rx[g][c], x));
                y = fmaf(go[c], vx[g][c], y);
            }
            part[g] = x;
            dp[g] = y;
        }
        {
            float both[2 * kG];
#pragma unroll
            for (int g = 0; g < kG; ++g) {
                both[g] = part[g];
                both[kG + g] = dp[g];
            }
            warp_sums<3>(both, lane);
#pragma unroll
            for (int g = 0; g < kG; ++g) {
                part[g] = both[g];
                dp[g] = both[kG + g];
            }
        }
#pragma unroll
        for (int g = 0; g < kG; ++g) {
            const bool vis = i >= jc0 + g;
            const float pr = vis ? __expf(part[g] * a.scale - lse) : 0.f;
            const float ds = a.scale * pr * (dp[g] - ddi);
#pragma unroll
            for (int c = 0; c < DC; ++c) {
                dk[g][c] = fmaf(ds, qu[c], dk[g][c]);
                dv[g][c] = fmaf(pr, go[c], dv[g][c]);
            }
        }
#pragma unroll
        for (int g = kG - 1; g > 0; --g)
#pragma unroll
            for (int c = 0; c < DC; ++c) rx[g][c] = rx[g - 1][c];
#pragma unroll
        for (int c = 0; c < DC; ++c) rx[0][c] = rn[c];
    }
#pragma unroll
    for (int g = 0; g < kG; ++g) {
        const int jc = jc0 + g;
        if (jc >= a.L) break;
        const int64_t row = qrow(a, b, jc, h);
#pragma unroll
        for (int c = 0; c < DC; ++c) {
            const int d = lane + 32 * c;
            if (d < a.D) {
                p.dk[row * a.D + d] = dk[g][c];
                p.dv[row * a.D + d] = dv[g][c];
            }
        }
    }
}

// ---------------------------------------------------------------------------- distances below the clamp
// Warp = kG consecutive distances delta0 + g of one head; over every (b, i), distance g pairs query
// i with key M + i - delta0 - g.  Key g at query i + 1 is key g - 1 at query i, so each query costs
// its q and dO rows and one new k, v row.
template <typename T, int DC>
__global__ void __launch_bounds__(32 * kBwdWarps) bwd_dist_kernel(const BwdParams p, int n_exact)
{
    const AttnSimtParams& a = p.a;
    const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int nd = (n_exact + kG - 1) / kG;
    if (gw >= static_cast<int64_t>(a.H) * nd) return;
    const int d0 = static_cast<int>(gw % nd) * kG;
    const int h = static_cast<int>(gw / nd);
    float rx[kG][DC], acc[kG][DC];
#pragma unroll
    for (int g = 0; g < kG; ++g) {
        load_vec<T, DC>(rrow<T>(a, h, min(d0 + g, n_exact - 1)), a.D, lane, rx[g]);
#pragma unroll
        for (int c = 0; c < DC; ++c) acc[g][c] = 0.f;
    }
    // queries with at least one of the warp's keys visible: M + i - d0 >= lo
    const int i_start = max(0, a.lo + d0 - a.M);
    for (int b = 0; b < a.B; ++b) {
        float kx[kG][DC], vx[kG][DC];
#pragma unroll
        for (int g = 0; g < kG; ++g) {
            const int j = a.M + i_start - d0 - g;
            const T *kp, *vp;
            key_ptrs<T>(a, b, h, max(j, 0), kp, vp);
            load_vec<T, DC>(kp, a.D, lane, kx[g]);
            load_vec<T, DC>(vp, a.D, lane, vx[g]);
        }
        if (i_start >= a.L) continue;
        float qun[DC], qvn[DC], gon[DC], knx[DC], vnx[DC], lsen, ddn;
        load_query<T, DC>(a, b, h, i_start, lane, qun, qvn);
        load_vec<T, DC>(gout<T>(p, b, h, i_start), a.D, lane, gon);
        lsen = p.lse[qrow(a, b, i_start, h)];
        ddn = p.dd[qrow(a, b, i_start, h)];
        for (int i = i_start; i < a.L; ++i) {
            float qu[DC], qv[DC], go[DC];
#pragma unroll
            for (int c = 0; c < DC; ++c) {
                qu[c] = qun[c];
                qv[c] = qvn[c];
                go[c] = gon[c];
            }
            const float lse = lsen, ddi = ddn;
            if (i + 1 < a.L) {                               // the next query's rows and its new key
                load_query<T, DC>(a, b, h, i + 1, lane, qun, qvn);
                load_vec<T, DC>(gout<T>(p, b, h, i + 1), a.D, lane, gon);
                lsen = p.lse[qrow(a, b, i + 1, h)];
                ddn = p.dd[qrow(a, b, i + 1, h)];
                const T *kp, *vp;
                key_ptrs<T>(a, b, h, max(a.M + i + 1 - d0, 0), kp, vp);
                load_vec<T, DC>(kp, a.D, lane, knx);
                load_vec<T, DC>(vp, a.D, lane, vnx);
            }
            float part[kG], dp[kG];
#pragma unroll
            for (int g = 0; g < kG; ++g) {
                float x = 0.f, y = 0.f;
#pragma unroll
                for (int c = 0; c < DC; ++c) {
                    x = fmaf(qu[c], kx[g][c], fmaf(qv[c], rx[g][c], x));
                    y = fmaf(go[c], vx[g][c], y);
                }
                part[g] = x;
                dp[g] = y;
            }
            {
                float both[2 * kG];
#pragma unroll
                for (int g = 0; g < kG; ++g) {
                    both[g] = part[g];
                    both[kG + g] = dp[g];
                }
                warp_sums<3>(both, lane);
#pragma unroll
                for (int g = 0; g < kG; ++g) {
                    part[g] = both[g];
                    dp[g] = both[kG + g];
                }
            }
#pragma unroll
            for (int g = 0; g < kG; ++g) {
                const bool vis = (d0 + g < n_exact) && (a.M + i - d0 - g >= a.lo);
                const float ds = vis ? a.scale * __expf(part[g] * a.scale - lse) * (dp[g] - ddi) : 0.f;
#pragma unroll
                for (int c = 0; c < DC; ++c) acc[g][c] = fmaf(ds, qv[c], acc[g][c]);
            }
#pragma unroll
            for (int g = kG - 1; g > 0; --g)
#pragma unroll
                for (int c = 0; c < DC; ++c) {
                    kx[g][c] = kx[g - 1][c];
                    vx[g][c] = vx[g - 1][c];
                }
#pragma unroll
            for (int c = 0; c < DC; ++c) {
                kx[0][c] = knx[c];
                vx[0][c] = vnx[c];
            }
        }
    }
#pragma unroll
    for (int g = 0; g < kG; ++g) {
        const int delta = d0 + g;
        if (delta >= n_exact) break;
#pragma unroll
        for (int c = 0; c < DC; ++c) {
            const int d = lane + 32 * c;
            if (d < a.D) p.dr[(static_cast<int64_t>(delta) * a.H + h) * a.D + d] = acc[g][c];
        }
    }
}

// ---------------------------------------------------------------------------- distances at the clamp
// Warp per (b, h, i): the keys j <= M + i - C all use r[C]; their dS q''_i is added into dr[C].
template <typename T, int DC>
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
    float qu[DC], qv[DC], go[DC], rx[DC], acc[DC];
    load_query<T, DC>(a, b, h, i, lane, qu, qv);
    load_vec<T, DC>(gout<T>(p, b, h, i), a.D, lane, go);
    load_vec<T, DC>(rrow<T>(a, h, a.C), a.D, lane, rx);
    const int64_t row = qrow(a, b, i, h);
    const float lse = p.lse[row], ddi = p.dd[row];
    float bd = 0.f;
#pragma unroll
    for (int c = 0; c < DC; ++c) {
        bd = fmaf(qv[c], rx[c], bd);
        acc[c] = 0.f;
    }
    bd = warp_sum(bd);                                    // the position term is the same for all these keys
    float dssum = 0.f;
    for (int j = a.lo; j <= j_hi; ++j) {
        const T *kp, *vp;
        key_ptrs<T>(a, b, h, j, kp, vp);
        float kx[DC], vx[DC];
        load_vec<T, DC>(kp, a.D, lane, kx);
        load_vec<T, DC>(vp, a.D, lane, vx);
        float x = 0.f, y = 0.f;
#pragma unroll
        for (int c = 0; c < DC; ++c) {
            x = fmaf(qu[c], kx[c], x);
            y = fmaf(go[c], vx[c], y);
        }
        x = warp_sum(x);
        y = warp_sum(y);
        dssum += a.scale * __expf((x + bd) * a.scale - lse) * (y - ddi);
    }
#pragma unroll
    for (int c = 0; c < DC; ++c) {
        const int d = lane + 32 * c;
        if (d < a.D) atomicAdd(p.dr + (static_cast<int64_t>(a.C) * a.H + h) * a.D + d, dssum * qv[c]);
    }
}

// ---------------------------------------------------------------------------- du, dv_bias
// Grid (column blocks of 128 (h, d), row chunks): each thread sums its column over one chunk of the
// B*L per-query rows and adds the partial sums into du, dv_bias (zeroed before).
constexpr int kBiasRowsPerChunk = 96;

__global__ void bwd_bias_kernel(const BwdParams p, int64_t chunk)
{
    const AttnSimtParams& a = p.a;
    const int hd = blockIdx.x * blockDim.x + threadIdx.x;
    const int HD = a.H * a.D;
    if (hd >= HD) return;
    const int64_t rows = static_cast<int64_t>(a.B) * a.L;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * chunk;
    const int64_t r1 = r0 + chunk < rows ? r0 + chunk : rows;
    float su = 0.f, sv = 0.f;
    for (int64_t r = r0; r < r1; ++r) {
        su += p.pac[r * HD + hd];
        sv += p.pbd[r * HD + hd];
    }
    atomicAdd(p.du + hd, su);
    atomicAdd(p.dvb + hd, sv);
}

// The bias reduction: du and dv_bias from the per-query parts in the workspace.
cudaError_t launch_bias(const BwdParams& p, cudaStream_t s)
{
    const AttnSimtParams& a = p.a;
    const int HD = a.H * a.D;
    const int64_t rows = static_cast<int64_t>(a.B) * a.L;
    int64_t chunk = kBiasRowsPerChunk;
    if ((rows + chunk - 1) / chunk > 65535) chunk = (rows + 65534) / 65535;
    const int64_t chunks = (rows + chunk - 1) / chunk;
    cudaError_t e = cudaMemsetAsync(p.du, 0, sizeof(float) * HD, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(p.dvb, 0, sizeof(float) * HD, s);
    if (e != cudaSuccess) return e;
    bwd_bias_kernel<<<dim3((HD + 127) / 128, static_cast<unsigned>(chunks)), 128, 0, s>>>(p, chunk);
    return cudaGetLastError();
}

template <typename T, int DC>
cudaError_t launch_all(const BwdParams& p, cudaStream_t s)
{
    const AttnSimtParams& a = p.a;
    const int thr = 32 * kBwdWarps;
    auto blocks = [](int64_t warps) { return (warps + kBwdWarps - 1) / kBwdWarps; };
    const int64_t grp = static_cast<int64_t>(a.B) * a.H * ((a.L + kG - 1) / kG);
    const int64_t row_warps = static_cast<int64_t>(a.B) * a.H * a.L;
    if (blocks(row_warps) > 0x7fffffffll) return cudaErrorInvalidValue;
    const int n_need = (a.M + a.L < a.C + 1) ? a.M + a.L : a.C + 1;
    const bool clamped = a.C < a.M + a.L - 1;
    const int n_exact = clamped ? a.C : n_need;
    cudaError_t e = cudaMemsetAsync(p.dr, 0, static_cast<size_t>(p.n_rows) * a.H * a.D * sizeof(float), s);
    if (e != cudaSuccess) return e;
    bwd_rows_kernel<T, DC><<<static_cast<unsigned>(blocks(grp)), thr, 0, s>>>(p);
    bwd_keys_kernel<T, DC><<<static_cast<unsigned>(blocks(grp)), thr, 0, s>>>(p);
    const int64_t dist_warps = static_cast<int64_t>(a.H) * ((n_exact + kG - 1) / kG);
    if (n_exact > 0) bwd_dist_kernel<T, DC><<<static_cast<unsigned>(blocks(dist_warps)), thr, 0, s>>>(p, n_exact);
    if (clamped) bwd_clamp_kernel<T, DC><<<static_cast<unsigned>(blocks(row_warps)), thr, 0, s>>>(p);
    return launch_bias(p, s);
}

template <typename T>
cudaError_t launch_t(const BwdParams& p, cudaStream_t s)
{
    return p.a.D <= 64 ? launch_all<T, 2>(p, s) : launch_all<T, 4>(p, s);
}

}  // namespace

cudaError_t launch_rel_attn_bwd(const BwdParams& p, txl_dtype dtype, cudaStream_t s)
{
    if (static_cast<int64_t>(p.a.B) * p.a.H * p.a.L == 0) return cudaSuccess;
    if (bwd_tc_eligible(p, dtype)) {
        const AttnSimtParams& a = p.a;
        const size_t cur = static_cast<size_t>(a.B) * a.L * a.H * a.D * sizeof(float);
        cudaError_t e = cudaMemsetAsync(p.dr, 0, static_cast<size_t>(p.n_rows) * a.H * a.D * sizeof(float), s);
        if (bwd_umma_eligible(p, dtype)) {
            // du and dv_bias come out of the gradient kernel itself
            const size_t hd = static_cast<size_t>(a.H) * a.D * sizeof(float);
            if (e == cudaSuccess) e = cudaMemsetAsync(p.du, 0, hd, s);
            if (e == cudaSuccess) e = cudaMemsetAsync(p.dvb, 0, hd, s);
            if (e == cudaSuccess) e = launch_bwd_umma(p, s);
            return e;
        }
        if (e == cudaSuccess) e = cudaMemsetAsync(p.dk, 0, cur, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(p.dv, 0, cur, s);
        if (e == cudaSuccess) e = launch_bwd_tc(p, s);
        if (e == cudaSuccess) e = launch_bias(p, s);
        return e;
    }
    return dtype == TXL_F32 ? launch_t<float>(p, s) : launch_t<__nv_bfloat16>(p, s);
}

cudaError_t launch_pos_bwd(const PosBwdParams& p, cudaStream_t s)
{
    if (p.d_model == 0) return cudaSuccess;
    const cudaError_t e = cudaMemset2DAsync(p.dW, static_cast<size_t>(p.ld_dw) * sizeof(float), 0,
                                            sizeof(float) * p.H * p.D, p.d_model, s);
    if (e != cudaSuccess || p.n_rows == 0) return e;
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorUnknown;
    return launch_pos_bwd_tc(p, sms, s);
}

}  // namespace txl
