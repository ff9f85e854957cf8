// txl_decode.cu -- relative attention for a few queries (L <= 16) over a long memory: split-K
// ("flash decoding").  The incremental-generation case of "Transformer-XL架构解析" §3.2 and
// "Transformer-XL 和相对位置编码" §2.2: each new token attends to the cached memory plus itself.
//
// Same arithmetic as the other attention paths ("跨窗口的相对位置编码" §3, terms (a)-(d); the clamp
// of "TransformerXL 相对位置编码" §2.4; the causal-with-memory mask of §4.2/§4.3):
//     s_ij = scale * [ (q_i+u).k_j + (q_i+v).r[min(M+i-j, C)] ],  out_i = softmax_j(s_ij) V
// With a handful of queries per (b, h) there is almost no reuse of K and V: the work is bound by
// HBM (about one flop per byte at L = 1), so it runs on the CUDA cores and spreads the keys of each
// (b, h) over many CTAs.
//
// decode_partial_kernel: one CTA per (chunk of 256 keys, h, b), 256 threads.
//   1. q+u and q+v in fp32 shared memory.
//   2. The position term of the chunk as a band: the chunk's keys and the L queries touch the
//      CK + L - 1 distances delta_top - rho (rho = 0 ..), delta_top = M + L - 1 - j0; thread rho
//      reads r[min(delta, C)] once and forms e(i, rho) = (q_i+v).r for every query.  Query i and
//      key j meet at rho = (L - 1 - i) + (j - j0): the relative shift is this index.
//   3. One key per thread: (q_i+u).k_j + e(i, rho) for every query, masked (key before the valid
//      memory, or in the future of the query) to -inf, in the log2 domain.
//   4. Per query: the chunk's maximum m and sum l of 2^(s - m) (block reductions).
//   5. O_i = sum_j 2^(s_ij - m_i) v_j: each warp takes 32 keys, lane = head dimension pairs; the
//      eight warps' partial sums meet in shared memory.  (m, l, O) go to the workspace.
// decode_combine_kernel: per (b, h, i), merges the chunks: M = max m_c, w_c = 2^(m_c - M),
//   out = sum w_c O_c / sum w_c l_c.
#include <mutex>

#include <cuda_bf16.h>

#include "txl_internal.h"
#include "txl_ptx.cuh"

namespace txl {

namespace {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kCopyRows = kDecThreads / 8;         // rows one pass of 16-byte copies covers
static_assert(kDecThreads == kDecodeChunk, "one thread per key of a chunk");

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// Eight consecutive elements d0 .. d0+7 of a row as fp32; elements at or past D read as 0.
// vec: the row start and d0 are 16-byte aligned and d0 + 8 <= D may use one or two vector loads.
template <typename T>
__device__ __forceinline__ void load8(const T* row, int d0, int D, bool vec, float* o)
{
    if (vec && d0 + 8 <= D) {
        if constexpr (sizeof(T) == 2) {
            const uint4 x = __ldg(reinterpret_cast<const uint4*>(row + d0));
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                o[2 * e] = __uint_as_float(w[e] << 16);
                o[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
            }
        } else {
            const float4 a = __ldg(reinterpret_cast<const float4*>(row + d0));
            const float4 b = __ldg(reinterpret_cast<const float4*>(row + d0 + 4));
            o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
            o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = d0 + e < D ? to_f(row[d0 + e]) : 0.f;
    }
}

// Key/value row of logical key j (memory slot (wp + j) mod M, or current-segment row j - M).
template <typename T>
__device__ __forceinline__ const T* kv_row(const DecodeParams& p, int b, int h, int j, bool values)
{
    if (j < p.M) {
        const int slot = p.wp + j >= p.M ? p.wp + j - p.M : p.wp + j;   // wp < M and j < M
        const T* base = static_cast<const T*>(values ? p.vmem : p.kmem);
        return base + b * p.m_sb + static_cast<int64_t>(slot) * p.m_st + h * p.m_sh;
    }
    const int t = j - p.M;
    if (values)
        return static_cast<const T*>(p.vcur) + b * p.vc_sb + static_cast<int64_t>(t) * p.vc_st + h * p.vc_sh;
    return static_cast<const T*>(p.kcur) + b * p.kc_sb + static_cast<int64_t>(t) * p.kc_st + h * p.kc_sh;
}

template <typename T, int LQ>
__global__ void __launch_bounds__(kDecThreads) decode_partial_kernel(const __grid_constant__ DecodeParams p)
{
    extern __shared__ __align__(16) float dsm[];
    pdl_launch_dependents();                       // the merge may launch (it waits for this grid)
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int L = p.L, D = p.D, Dp = p.Dp;
    const int K = p.M + L;
    const int j0 = c * kDecodeChunk;
    const int BW = kDecodeChunk + LQ;                         // band row pitch
    float* qu = dsm;                                          // [LQ][Dp]
    float* qv = qu + LQ * Dp;                                 // [LQ][Dp]
    float* band = qv + LQ * Dp;                               // [LQ][BW]
    float* sp = band + LQ * BW;                               // [LQ][kDecodeChunk]
    float* red = sp + LQ * kDecodeChunk;                      // [2][kDecWarps][LQ]
    float* obuf = red + 2 * kDecWarps * LQ;                   // [kDecWarps][LQ][Do]

    // 1. q + u, q + v (fp32)
    for (int x = tid; x < LQ * Dp; x += kDecThreads) {
        const int i = x / Dp, d = x - i * Dp;
        float qq = 0.f, uu = 0.f, vv = 0.f;
        if (i < L && d < D) {
            qq = to_f(static_cast<const T*>(p.q)[b * p.q_sb + static_cast<int64_t>(i) * p.q_st + h * p.q_sh + d]);
            uu = __ldg(p.u + h * D + d);
            vv = __ldg(p.vb + h * D + d);
        }
        qu[x] = (i < L && d < D) ? qq + uu : 0.f;
        qv[x] = (i < L && d < D) ? qq + vv : 0.f;
    }
    __syncthreads();

    // Rows are read cooperatively: the eight lanes of group rg = lane / 8 read one row together,
    // lane part = lane mod 8 taking the 16-byte pieces part, part + 8, ... (four whole rows per
    // warp instruction), and their partial dot products meet in three shuffles.
    const int rg = lane >> 3, part = lane & 7;

    // 2. position band e(i, rho) = (q_i + v) . r[min(delta_top - rho, C)]
    const int delta_top = p.M + L - 1 - j0;
    const int n_band = kDecodeChunk + L - 1;
    for (int rho0 = 4 * warp; rho0 < n_band; rho0 += 4 * kDecWarps) {
        const int rho = rho0 + rg;
        const int delta = delta_top - rho;
        float acc[LQ];
#pragma unroll
        for (int i = 0; i < LQ; ++i) acc[i] = 0.f;
        if (rho < n_band && delta >= 0) {
            const int dc = delta < p.C ? delta : p.C;
            const T* rrow = static_cast<const T*>(p.r) + static_cast<int64_t>(dc) * p.r_row + h * p.r_head;
            for (int d0 = 8 * part; d0 < D; d0 += 64) {
                float r8[8];
                load8(rrow, d0, D, p.vec_r, r8);
#pragma unroll
                for (int i = 0; i < LQ; ++i) {
                    const float4 a = *reinterpret_cast<const float4*>(qv + i * Dp + d0);
                    const float4 e = *reinterpret_cast<const float4*>(qv + i * Dp + d0 + 4);
                    acc[i] = fmaf(a.x, r8[0], fmaf(a.y, r8[1], fmaf(a.z, r8[2], fmaf(a.w, r8[3], acc[i]))));
                    acc[i] = fmaf(e.x, r8[4], fmaf(e.y, r8[5], fmaf(e.z, r8[6], fmaf(e.w, r8[7], acc[i]))));
                }
            }
        }
#pragma unroll
        for (int i = 0; i < LQ; ++i) {
            float x = acc[i];
            x += __shfl_xor_sync(0xffffffffu, x, 1);
            x += __shfl_xor_sync(0xffffffffu, x, 2);
            x += __shfl_xor_sync(0xffffffffu, x, 4);
            if (part == 0 && rho < n_band) band[i * BW + rho] = x;
        }
    }
    __syncthreads();

    // 3. scores of every key of the chunk against every query (log2 domain), masked keys -inf:
    //    key t = t0 + rg of this warp's 32 in groups of four, into sp[i][t]
    for (int t0 = 32 * warp; t0 < 32 * warp + 32; t0 += 4) {
        const int t = t0 + rg;
        const int jj = j0 + t;
        const bool live = jj < K && jj >= p.lo;
        float acc[LQ];
#pragma unroll
        for (int i = 0; i < LQ; ++i) acc[i] = 0.f;
        if (live) {
            const T* krow = kv_row<T>(p, b, h, jj, false);
            for (int d0 = 8 * part; d0 < D; d0 += 64) {
                float k8[8];
                load8(krow, d0, D, p.vec_kv, k8);
#pragma unroll
                for (int i = 0; i < LQ; ++i) {
                    const float4 a = *reinterpret_cast<const float4*>(qu + i * Dp + d0);
                    const float4 e = *reinterpret_cast<const float4*>(qu + i * Dp + d0 + 4);
                    acc[i] = fmaf(a.x, k8[0], fmaf(a.y, k8[1], fmaf(a.z, k8[2], fmaf(a.w, k8[3], acc[i]))));
                    acc[i] = fmaf(e.x, k8[4], fmaf(e.y, k8[5], fmaf(e.z, k8[6], fmaf(e.w, k8[7], acc[i]))));
                }
            }
        }
#pragma unroll
        for (int i = 0; i < LQ; ++i) {
            float x = acc[i];
            x += __shfl_xor_sync(0xffffffffu, x, 1);
            x += __shfl_xor_sync(0xffffffffu, x, 2);
            x += __shfl_xor_sync(0xffffffffu, x, 4);
            const bool vis = live && i < L && jj <= p.M + i;
            if (part == 0) sp[i * kDecodeChunk + t] = vis ? (x + band[i * BW + (L - 1 - i) + t]) * p.qscale : -INFINITY;
        }
    }
    __syncthreads();
    float s[LQ];
#pragma unroll
    for (int i = 0; i < LQ; ++i) s[i] = sp[i * kDecodeChunk + tid];

    // 4. per query: chunk maximum, probabilities, chunk sum
    float m[LQ];
#pragma unroll
    for (int i = 0; i < LQ; ++i) {
        float x = s[i];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
        if (lane == 0) red[warp * LQ + i] = x;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < LQ; ++i) {
        float x = red[i];
#pragma unroll
        for (int w = 1; w < kDecWarps; ++w) x = fmaxf(x, red[w * LQ + i]);
        m[i] = x;
        const float pv = x == -INFINITY ? 0.f : exp2f(s[i] - x);
        sp[i * kDecodeChunk + tid] = pv;
        float y = pv;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) y += __shfl_xor_sync(0xffffffffu, y, off);
        if (lane == 0) red[(kDecWarps + warp) * LQ + i] = y;
    }
    __syncthreads();

    // 5. O_i over this warp's 32 keys; lane owns dims 2 lane + 64 g, 2 lane + 1 + 64 g.  Rows are
    //    requested eight at a time before any of them is used (a key outside [lo, K) reads the
    //    chunk's first valid row and weighs 0), so each lane keeps eight loads in flight.
    constexpr int kG = 2;                                     // D <= 128
    constexpr int kBatch = 8;
    const int ng = D > 64 ? 2 : 1;
    float o[LQ][2 * kG];
#pragma unroll
    for (int i = 0; i < LQ; ++i)
#pragma unroll
        for (int e = 0; e < 2 * kG; ++e) o[i][e] = 0.f;
    const int kb = 32 * warp;
    const int jfirst = max(j0, p.lo);                         // some valid key of the chunk
    if (jfirst < K && j0 + kb < K) {
#pragma unroll
        for (int g = 0; g < kG; ++g) {
            if (g >= ng) break;
            const int d = 2 * lane + 64 * g;
            const bool vec = p.vec_kv && d + 1 < D;
#pragma unroll 1
            for (int k8 = 0; k8 < 32; k8 += kBatch) {
                float v0[kBatch], v1[kBatch];
#pragma unroll
                for (int e = 0; e < kBatch; ++e) {
                    const int jj0 = j0 + kb + k8 + e;
                    const int jj = (jj0 >= K || jj0 < p.lo) ? jfirst : jj0;
                    const T* vrow = kv_row<T>(p, b, h, jj, true);
                    if (vec) {
                        if constexpr (sizeof(T) == 2) {
                            const uint32_t w = __ldg(reinterpret_cast<const unsigned int*>(vrow + d));
                            v0[e] = __uint_as_float(w << 16);
                            v1[e] = __uint_as_float(w & 0xffff0000u);
                        } else {
                            const float2 w = __ldg(reinterpret_cast<const float2*>(vrow + d));
                            v0[e] = w.x;
                            v1[e] = w.y;
                        }
                    } else {
                        v0[e] = d < D ? to_f(vrow[d]) : 0.f;
                        v1[e] = d + 1 < D ? to_f(vrow[d + 1]) : 0.f;
                    }
                }
#pragma unroll
                for (int e = 0; e < kBatch; ++e) {
                    const int t = kb + k8 + e;
#pragma unroll
                    for (int i = 0; i < LQ; ++i) {
                        const float pij = sp[i * kDecodeChunk + t];   // 0 for masked and absent keys
                        o[i][2 * g] = fmaf(pij, v0[e], o[i][2 * g]);
                        o[i][2 * g + 1] = fmaf(pij, v1[e], o[i][2 * g + 1]);
                    }
                }
            }
        }
    }
    constexpr int Do = 64 * kG;
#pragma unroll
    for (int i = 0; i < LQ; ++i)
#pragma unroll
        for (int g = 0; g < kG; ++g) {
            obuf[(warp * LQ + i) * Do + 2 * lane + 64 * g] = o[i][2 * g];
            obuf[(warp * LQ + i) * Do + 2 * lane + 1 + 64 * g] = o[i][2 * g + 1];
        }
    __syncthreads();

    // partial (m, l, O) of every query of this chunk
    const int Dw = D + 2;
    for (int x = tid; x < L * Dw; x += kDecThreads) {
        const int i = x / Dw, e = x - i * Dw;
        float val;
        if (e == 0) {
            val = red[i];
#pragma unroll
            for (int w = 1; w < kDecWarps; ++w) val = fmaxf(val, red[w * LQ + i]);
        } else if (e == 1) {
            val = 0.f;
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w) val += red[(kDecWarps + w) * LQ + i];
        } else {
            val = 0.f;
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w) val += obuf[(w * LQ + i) * Do + (e - 2)];
        }
        p.part[((static_cast<int64_t>(b) * p.H + h) * L + i) * p.n_chunks * Dw + static_cast<int64_t>(c) * Dw + e] = val;
    }
    (void)m;
}

// ------------------------------------------------------------------------------------------
// Staged variant for bf16 rows of D <= 64 (D a multiple of 8) whose starts are 16-byte aligned:
// every thread first requests its share of the chunk's key rows, value rows and position-band
// rows as 16-byte asynchronous copies into shared memory (absent rows are zero-filled without
// reading memory), so a CTA has its ~96 KB in flight at once; the phases then read shared memory.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool live)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 ::"r"(dst), "l"(src), "r"(live ? 16 : 0) : "memory");
}

constexpr int kStRowBytes = 128;                     // 64 bf16 per staged row

__device__ __forceinline__ void unpack8(uint4 x, float* o)
{
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        o[2 * e] = __uint_as_float(w[e] << 16);
        o[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    }
}

template <int LQ>
__global__ void __launch_bounds__(kDecThreads) decode_staged_kernel(const __grid_constant__ DecodeParams p)
{
    extern __shared__ __align__(16) float dsm[];
    pdl_launch_dependents();                       // the merge may launch (it waits for this grid)
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rg = lane >> 3, part = lane & 7;
    const int L = p.L, D = p.D, dch = D >> 3;
    const int K = p.M + L;
    const int j0 = c * kDecodeChunk;
    uint8_t* ks = reinterpret_cast<uint8_t*>(dsm);                       // [CK][128 B]
    uint8_t* vs = ks + kDecodeChunk * kStRowBytes;                         // [CK][128 B]
    float* qu = reinterpret_cast<float*>(vs + kDecodeChunk * kStRowBytes); // [LQ][64]
    float* qv = qu + LQ * 64;
    const int BW = kDecodeChunk + LQ;
    float* band = qv + LQ * 64;                                            // [LQ][BW]
    float* sp = band + LQ * BW;                                            // [LQ][CK]
    float* red = sp + LQ * kDecodeChunk;                                   // [2][warps][LQ]
    float* obuf = red + 2 * kDecWarps * LQ;                                // [warps][LQ][64]

    // 0. all copies of the chunk in flight at once.  Thread tid moves 16-byte piece pc = tid mod 8
    //    of rows tid/8 + 32 k (k = 0..7) of K and V.  (The position band reads r, small and
    //    L2-resident, straight from global memory; when every distance of the chunk reaches
    //    clamp_len it is one value per query.)
    const int delta_top = p.M + L - 1 - j0;
    const int n_band = kDecodeChunk + L - 1;
    const bool band_const = delta_top - (n_band - 1) >= p.C;
    const int pc = tid & 7, r0 = tid >> 3;
    if (pc < dch) {
        const __nv_bfloat16* kmem = static_cast<const __nv_bfloat16*>(p.kmem) + b * p.m_sb + h * p.m_sh + 8 * pc;
        const __nv_bfloat16* vmem = static_cast<const __nv_bfloat16*>(p.vmem) + b * p.m_sb + h * p.m_sh + 8 * pc;
        const __nv_bfloat16* kcur = static_cast<const __nv_bfloat16*>(p.kcur) + b * p.kc_sb + h * p.kc_sh + 8 * pc;
        const __nv_bfloat16* vcur = static_cast<const __nv_bfloat16*>(p.vcur) + b * p.vc_sb + h * p.vc_sh + 8 * pc;
        const __nv_bfloat16* dummy = static_cast<const __nv_bfloat16*>(p.q);
        const uint32_t ks_s = static_cast<uint32_t>(__cvta_generic_to_shared(ks)) + r0 * kStRowBytes + 16 * pc;
        const uint32_t vs_s = static_cast<uint32_t>(__cvta_generic_to_shared(vs)) + r0 * kStRowBytes + 16 * pc;
#pragma unroll
        for (int k = 0; k < kDecodeChunk / kCopyRows; ++k) {
            const int j = j0 + r0 + kCopyRows * k;
            const bool live = j < K && j >= p.lo;
            const __nv_bfloat16* ksrc = dummy;
            const __nv_bfloat16* vsrc = dummy;
            if (live) {
                if (j < p.M) {
                    const int slot = p.wp + j >= p.M ? p.wp + j - p.M : p.wp + j;
                    ksrc = kmem + static_cast<int64_t>(slot) * p.m_st;
                    vsrc = vmem + static_cast<int64_t>(slot) * p.m_st;
                } else {
                    ksrc = kcur + static_cast<int64_t>(j - p.M) * p.kc_st;
                    vsrc = vcur + static_cast<int64_t>(j - p.M) * p.vc_st;
                }
            }
            cp_async16(ks_s + kCopyRows * k * kStRowBytes, ksrc, live);
            cp_async16(vs_s + kCopyRows * k * kStRowBytes, vsrc, live);
        }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");

    // 1. q + u, q + v (fp32) while the copies fly (staged rows: Dp = 64)
    for (int x = tid; x < LQ * 64; x += kDecThreads) {
        const int i = x >> 6, d = x & 63;
        const bool in = i < L && d < D;
        const float qq = in ? __bfloat162float(static_cast<const __nv_bfloat16*>(p.q)[
                                  b * p.q_sb + static_cast<int64_t>(i) * p.q_st + h * p.q_sh + d]) : 0.f;
        qu[x] = in ? qq + __ldg(p.u + h * D + d) : 0.f;
        qv[x] = in ? qq + __ldg(p.vb + h * D + d) : 0.f;
    }
    if (band_const) {
        // every key of the chunk sits at distance >= clamp_len: e(i) = (q_i + v) . r[clamp_len]
        __syncthreads();
        if (warp == 0) {
            const __nv_bfloat16* rrow = static_cast<const __nv_bfloat16*>(p.r) + static_cast<int64_t>(p.C) * p.r_row + h * p.r_head;
            for (int i = 0; i < L; ++i) {
                float x = 0.f;
                for (int d = lane; d < D; d += 32) x = fmaf(qv[i * 64 + d], __bfloat162float(rrow[d]), x);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
                if (lane == 0) band[i * BW] = x;
            }
        }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();

    // 2. position band, eight lanes per row (lane part holds 16-byte piece part); each lane
    //    requests its pieces of all its rows before using any
    if (!band_const) {
        constexpr int kBandIter = (kDecodeChunk + kDecodeMaxL + 4 * kDecWarps - 1) / (4 * kDecWarps);
        uint4 raw[kBandIter];
#pragma unroll
        for (int k = 0; k < kBandIter; ++k) {
            const int rho = 4 * warp + 4 * kDecWarps * k + rg;
            const int delta = delta_top - rho;
            raw[k] = make_uint4(0u, 0u, 0u, 0u);
            if (rho < n_band && delta >= 0 && part < dch) {
                const int dc = delta < p.C ? delta : p.C;
                raw[k] = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.r) +
                                                              static_cast<int64_t>(dc) * p.r_row + h * p.r_head + 8 * part));
            }
        }
#pragma unroll
        for (int k = 0; k < kBandIter; ++k) {
            const int rho = 4 * warp + 4 * kDecWarps * k + rg;
            float acc[LQ];
#pragma unroll
            for (int i = 0; i < LQ; ++i) acc[i] = 0.f;
            if (part < dch) {
                float r8[8];
                unpack8(raw[k], r8);
#pragma unroll
                for (int i = 0; i < LQ; ++i) {
                    const float4 a = *reinterpret_cast<const float4*>(qv + i * 64 + 8 * part);
                    const float4 e = *reinterpret_cast<const float4*>(qv + i * 64 + 8 * part + 4);
                    acc[i] = fmaf(a.x, r8[0], fmaf(a.y, r8[1], fmaf(a.z, r8[2], fmaf(a.w, r8[3], acc[i]))));
                    acc[i] = fmaf(e.x, r8[4], fmaf(e.y, r8[5], fmaf(e.z, r8[6], fmaf(e.w, r8[7], acc[i]))));
                }
            }
#pragma unroll
            for (int i = 0; i < LQ; ++i) {
                float x = acc[i];
                x += __shfl_xor_sync(0xffffffffu, x, 1);
                x += __shfl_xor_sync(0xffffffffu, x, 2);
                x += __shfl_xor_sync(0xffffffffu, x, 4);
                if (part == 0 && rho < n_band) band[i * BW + rho] = x;
            }
        }
    }
    __syncthreads();

    // 3. scores, eight lanes per key row
    if constexpr (LQ <= 4) {
        // q + u of the lane's piece stays in registers; lane (rg, part) forms the partial dots of
        // its piece for rows t = 32 warp + 4 k + rg (k = 0..7), then a transposing butterfly over
        // the group's eight lanes leaves lane part with the whole dot of row k = part.
        float qr[LQ][8];
#pragma unroll
        for (int i = 0; i < LQ; ++i)
#pragma unroll
            for (int e = 0; e < 8; ++e) qr[i][e] = part < dch ? qu[i * 64 + 8 * part + e] : 0.f;
        float acc[LQ][8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int t = 32 * warp + 4 * k + rg;
            float k8[8];
            if (part < dch) {
                unpack8(*reinterpret_cast<const uint4*>(ks + t * kStRowBytes + 16 * part), k8);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) k8[e] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < LQ; ++i) {
                float x = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) x = fmaf(qr[i][e], k8[e], x);
                acc[i][k] = x;
            }
        }
        const bool b4 = part & 4, b2 = part & 2, b1 = part & 1;
        const int t = 32 * warp + 4 * part + rg;
        const int jj = j0 + t;
        const bool live = jj < K && jj >= p.lo;
#pragma unroll
        for (int i = 0; i < LQ; ++i) {
            float v4[4], v2[2];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float keep = b4 ? acc[i][m + 4] : acc[i][m];
                const float send = b4 ? acc[i][m] : acc[i][m + 4];
                v4[m] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
            }
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const float keep = b2 ? v4[m + 2] : v4[m];
                const float send = b2 ? v4[m] : v4[m + 2];
                v2[m] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
            }
            const float keep = b1 ? v2[1] : v2[0];
            const float send = b1 ? v2[0] : v2[1];
            const float x = keep + __shfl_xor_sync(0xffffffffu, send, 1);
            const bool vis = live && i < L && jj <= p.M + i;
            const float e = band[i * BW + (band_const ? 0 : (L - 1 - i) + t)];
            sp[i * kDecodeChunk + t] = vis ? (x + e) * p.qscale : -INFINITY;
        }
    } else {
        for (int t0 = 32 * warp; t0 < 32 * warp + 32; t0 += 4) {
            const int t = t0 + rg;
            const int jj = j0 + t;
            const bool live = jj < K && jj >= p.lo;
            float acc[LQ];
    #pragma unroll
            for (int i = 0; i < LQ; ++i) acc[i] = 0.f;
            if (part < dch) {
                float k8[8];
                unpack8(*reinterpret_cast<const uint4*>(ks + t * kStRowBytes + 16 * part), k8);
    #pragma unroll
                for (int i = 0; i < LQ; ++i) {
                    const float4 a = *reinterpret_cast<const float4*>(qu + i * 64 + 8 * part);
                    const float4 e = *reinterpret_cast<const float4*>(qu + i * 64 + 8 * part + 4);
                    acc[i] = fmaf(a.x, k8[0], fmaf(a.y, k8[1], fmaf(a.z, k8[2], fmaf(a.w, k8[3], acc[i]))));
                    acc[i] = fmaf(e.x, k8[4], fmaf(e.y, k8[5], fmaf(e.z, k8[6], fmaf(e.w, k8[7], acc[i]))));
                }
            }
    #pragma unroll
            for (int i = 0; i < LQ; ++i) {
                float x = acc[i];
                x += __shfl_xor_sync(0xffffffffu, x, 1);
                x += __shfl_xor_sync(0xffffffffu, x, 2);
                x += __shfl_xor_sync(0xffffffffu, x, 4);
                const bool vis = live && i < L && jj <= p.M + i;
                const float e = band[i * BW + (band_const ? 0 : (L - 1 - i) + t)];
                if (part == 0) sp[i * kDecodeChunk + t] = vis ? (x + e) * p.qscale : -INFINITY;
            }
        }
    }
    __syncthreads();

    // 4. per query: chunk maximum, probabilities, chunk sum
    float s[LQ];
#pragma unroll
    for (int i = 0; i < LQ; ++i) {
        s[i] = sp[i * kDecodeChunk + tid];
        float x = s[i];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
        if (lane == 0) red[warp * LQ + i] = x;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < LQ; ++i) {
        float x = red[i];
#pragma unroll
        for (int w = 1; w < kDecWarps; ++w) x = fmaxf(x, red[w * LQ + i]);
        const float pv = x == -INFINITY ? 0.f : exp2f(s[i] - x);
        sp[i * kDecodeChunk + tid] = pv;
        float y = pv;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) y += __shfl_xor_sync(0xffffffffu, y, off);
        if (lane == 0) red[(kDecWarps + warp) * LQ + i] = y;
    }
    __syncthreads();

    // 5. O_i over this warp's 32 keys from shared memory; lane owns dims 2 lane, 2 lane + 1
    //    (zero-filled absent rows weigh 0)
    float o[LQ][2];
#pragma unroll
    for (int i = 0; i < LQ; ++i) o[i][0] = o[i][1] = 0.f;
    if (2 * lane < D) {
#pragma unroll 8
        for (int kk = 0; kk < 32; ++kk) {
            const int t = 32 * warp + kk;
            const uint32_t w = *reinterpret_cast<const uint32_t*>(vs + t * kStRowBytes + 4 * lane);
            const float v0 = __uint_as_float(w << 16), v1 = __uint_as_float(w & 0xffff0000u);
#pragma unroll
            for (int i = 0; i < LQ; ++i) {
                const float pij = sp[i * kDecodeChunk + t];
                o[i][0] = fmaf(pij, v0, o[i][0]);
                o[i][1] = fmaf(pij, v1, o[i][1]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < LQ; ++i) {
        obuf[(warp * LQ + i) * 64 + 2 * lane] = o[i][0];
        obuf[(warp * LQ + i) * 64 + 2 * lane + 1] = o[i][1];
    }
    __syncthreads();

    const int Dw = D + 2;
    for (int x = tid; x < L * Dw; x += kDecThreads) {
        const int i = x / Dw, e = x - i * Dw;
        float val;
        if (e == 0) {
            val = red[i];
#pragma unroll
            for (int w = 1; w < kDecWarps; ++w) val = fmaxf(val, red[w * LQ + i]);
        } else if (e == 1) {
            val = 0.f;
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w) val += red[(kDecWarps + w) * LQ + i];
        } else {
            val = 0.f;
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w) val += obuf[(w * LQ + i) * 64 + (e - 2)];
        }
        p.part[((static_cast<int64_t>(b) * p.H + h) * L + i) * p.n_chunks * Dw + static_cast<int64_t>(c) * Dw + e] = val;
    }
}

size_t decode_staged_smem_bytes(int lq)
{
    return static_cast<size_t>(2 * kDecodeChunk) * kStRowBytes +
           (2ull * lq * 64 + static_cast<size_t>(lq) * (kDecodeChunk + lq) + static_cast<size_t>(lq) * kDecodeChunk +
            2ull * kDecWarps * lq + static_cast<size_t>(kDecWarps) * lq * 64) * sizeof(float);
}

template <typename T>
__global__ void __launch_bounds__(128) decode_combine_kernel(const __grid_constant__ DecodeParams p)
{
    // weights of the chunks first (in parallel), then every output dimension reads its chunks'
    // partial sums with independent loads
    __shared__ float wsh[1024];
    __shared__ float mred[4];
    pdl_wait();                                               // the partials are complete
    const int bhi = blockIdx.x;                               // (b * H + h) * L + i
    const int i = bhi % p.L;
    const int bh = bhi / p.L;
    const int h = bh % p.H, b = bh / p.H;
    const int Dw = p.D + 2;
    const int nc = p.n_chunks;
    const float* part = p.part + static_cast<int64_t>(bhi) * nc * Dw;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float mx = -INFINITY;
    for (int c = tid; c < nc; c += blockDim.x) mx = fmaxf(mx, part[c * Dw]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) mred[warp] = mx;
    __syncthreads();
    mx = fmaxf(fmaxf(mred[0], mred[1]), fmaxf(mred[2], mred[3]));
    float den = 0.f;
    const bool in_smem = nc <= 1024;
    for (int c = tid; c < nc; c += blockDim.x) {
        const float mc = part[c * Dw];
        const float w = mc == -INFINITY ? 0.f : exp2f(mc - mx);
        if (in_smem) wsh[c] = w;
        den = fmaf(w, part[c * Dw + 1], den);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
    __syncthreads();
    if (lane == 0) mred[warp] = den;
    __syncthreads();
    den = (mred[0] + mred[1]) + (mred[2] + mred[3]);
    for (int d = tid; d < p.D; d += blockDim.x) {
        float num = 0.f;
#pragma unroll 4
        for (int c = 0; c < nc; ++c) {
            float w;
            if (in_smem) {
                w = wsh[c];
            } else {
                const float mc = part[c * Dw];
                w = mc == -INFINITY ? 0.f : exp2f(mc - mx);
            }
            num = fmaf(w, part[c * Dw + 2 + d], num);
        }
        T* o = static_cast<T*>(p.out) + b * p.o_sb + static_cast<int64_t>(i) * p.o_st + h * p.o_sh + d;
        const float val = num / den;
        if constexpr (sizeof(T) == 2) *o = __float2bfloat16_rn(val);
        else *o = val;
    }
}

template <typename T, int LQ>
cudaError_t launch_lq(const DecodeParams& p, cudaStream_t s)
{
    dim3 grid(p.n_chunks, p.H, p.B);
    const bool staged = sizeof(T) == 2 && p.vec_kv && p.vec_r && (p.D % 8) == 0 && p.D <= 64;
    if (staged) {
        static bool attr_st = false;
        if (!attr_st) {
            cudaError_t e = cudaFuncSetAttribute(decode_staged_kernel<LQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(decode_staged_smem_bytes(LQ)));
            if (e != cudaSuccess) return e;
            attr_st = true;
        }
        decode_staged_kernel<LQ><<<grid, kDecThreads, decode_staged_smem_bytes(LQ), s>>>(p);
    } else {
        static bool attr_done = false;
        if (!attr_done) {
            cudaError_t e = cudaFuncSetAttribute(decode_partial_kernel<T, LQ>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(decode_smem_bytes(LQ, 128)));
            if (e != cudaSuccess) return e;
            attr_done = true;
        }
        decode_partial_kernel<T, LQ><<<grid, kDecThreads, decode_smem_bytes(LQ, p.Dp), s>>>(p);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // launched as a dependent of the partial kernel: its launch overlaps that grid's tail
    return launch_dependent(decode_combine_kernel<T>, dim3(p.B * p.H * p.L), dim3(128), 0, s, p);
}

template <typename T>
cudaError_t launch_t(const DecodeParams& p, cudaStream_t s)
{
    if (p.L <= 1) return launch_lq<T, 1>(p, s);
    if (p.L <= 2) return launch_lq<T, 2>(p, s);
    if (p.L <= 4) return launch_lq<T, 4>(p, s);
    if (p.L <= 8) return launch_lq<T, 8>(p, s);
    return launch_lq<T, 16>(p, s);
}

// Scratch of the variant of the decode path that allocates nothing (txl_rel_attn_decode_noalloc):
// every GPU that loads the library holds these kDecodeStaticScratchBytes until the process exits.
// All calls share it; the partial kernel writes every entry the merge reads, so nothing in it has
// to start at zero, but two calls that overlap on the GPU overwrite each other's partials.
static __device__ __align__(256) float g_decode_scratch[kDecodeStaticScratchBytes / sizeof(float)];

}  // namespace

// Device address of the static scratch on the current device.  In host code the array's name is
// only a host-side stand-in, so the address is looked up with cudaGetSymbolAddress with the device
// current and cached per device.  The cache entry carries the unique id of the context it was
// looked up in: after cudaDeviceReset the device gets a new primary context (the library's module
// is loaded again, possibly elsewhere), the id differs, and the first call in the new context looks
// the address up again instead of using a stale one.
namespace {
using PFN_ctx_get_current = CUresult (*)(CUcontext*);
using PFN_ctx_get_id = CUresult (*)(CUcontext, unsigned long long*);
}  // namespace

bool current_context_id(unsigned long long* id)
{
    static PFN_ctx_get_current get_current = nullptr;
    static PFN_ctx_get_id get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_ctx_get_current>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_ctx_get_id>(fn);
    });
    if (!get_current || !get_id) return false;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

cudaError_t decode_static_scratch(float** out)
{
    static std::mutex mu;
    static float* addr[kMaxDevices] = {};
    static unsigned long long ctx_of[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    // no context may be current yet on this thread: the runtime creates (or binds) the device's
    // primary context in cudaGetSymbolAddress, after which the id is read
    unsigned long long ctx = 0;
    const bool have_ctx = current_context_id(&ctx);
    std::lock_guard<std::mutex> lock(mu);
    if (!have_ctx || !addr[dev] || ctx_of[dev] != ctx) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
        if (e != cudaSuccess) return e;
        if (!have_ctx && !current_context_id(&ctx)) return cudaErrorDeviceUninitialized;
        addr[dev] = static_cast<float*>(ptr);
        ctx_of[dev] = ctx;
    }
    *out = addr[dev];
    return cudaSuccess;
}

size_t decode_smem_bytes(int lq, int Dp)
{
    const size_t floats = 2ull * lq * Dp + static_cast<size_t>(lq) * (kDecodeChunk + lq) +
                          static_cast<size_t>(lq) * kDecodeChunk + 2ull * kDecWarps * lq +
                          static_cast<size_t>(kDecWarps) * lq * 128;
    return floats * sizeof(float);
}

cudaError_t launch_decode(const DecodeParams& p, txl_dtype dtype, cudaStream_t s)
{
    if (p.B == 0 || p.L == 0) return cudaSuccess;
    return dtype == TXL_F32 ? launch_t<float>(p, s) : launch_t<__nv_bfloat16>(p, s);
}

}  // namespace txl
