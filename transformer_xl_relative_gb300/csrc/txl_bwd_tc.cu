// txl_bwd_tc.cu -- gradients of the relative attention on the tensor cores (bf16, d_head = 64).
//
// The same gradients as txl_bwd.cu (the chain rule through the four-term score of
// "Transformer-XL 和相对位置编码" §2.3.2 and the softmax; the memory's keys and values are the
// stop-gradient part, §2.3.1):
//   P_ij = 2^(c s_ij - L2_i),  dS_ij = P_ij (dO_i . v_j - dO_i . out_i)   (c = scale log2 e)
//   dq_i = scale sum_j dS_ij (k_j + r[delta_ij]),  dk_j = scale sum_i dS_ij q'_i,  dv_j = sum_i P_ij dO_i,
//   dr[delta] = scale sum_{delta_ij = delta} dS_ij q''_i,   q' = q + u,  q'' = q + v_bias,
// with delta_ij = min(M + i - j, clamp_len).
//
// This is the mma.sync path: txl_bwd_umma.cu's tcgen05 kernel takes the bf16 d_head 64 calls whose
// row log-sum-exp is given and whose gradient buffers are 16-byte aligned; the rest come here.
//
// One CTA of four warps per (query tile of 64, head, batch entry); warp w owns query rows
// 16w .. 16w + 15.  Key tiles of 64 are aligned to the query tile (tile t covers keys
// j0 = M + i0 - 64 t ...), so the distances of tile t fill a window of 127 position rows starting
// at 64 t - 63.  Every product is a bf16 mma.sync with fp32 accumulation:
//   S = Q' K^T and BD = Q'' R_win^T (the relative shift as a per-row index remap through shared
//   memory, as in the forward), dP = dO V^T, dq += dS K + G R_win where G is dS scattered by
//   distance (G[i][i - j + 63] = dS_ij), and, over the whole CTA, dv_tile = P^T dO, dk_tile = dS^T Q'
//   and dr_win = G^T Q'', added into global fp32 gradients with vector atomics.
// Pairs whose distance reaches clamp_len all share r[clamp_len]; their dS nearly cancel (each row of
// dS sums to zero), so they stay out of the bf16 G: their fp32 sum per row c_i enters dq_i as
// c_i r[clamp_len] and dr[clamp_len] as sum_i c_i q''_i.
// The scores use the forward kernel's query forms Qc' = bf16(c q') and Qc'' = bf16(c q''), so the
// row log-sum-exp L2_i the persistent forward kernel writes (txl_rel_attn_bwd has it computed when
// that kernel takes the inputs) belongs to them; otherwise a first sweep over the key tiles takes
// it here.  The sweep over the key tiles then computes the gradients.
// dq goes straight to its rows (one CTA per query row); the per-query parts of du and dv_bias go
// to the workspace the bias reduction of txl_bwd.cu sums.
#include <cuda_bf16.h>

#include "txl_internal.h"
#include "txl_mma.cuh"

namespace txl {

namespace {

using namespace mma;

constexpr int kBT = 128;                 // threads: four warps
constexpr float kLn2 = 0.693147180559945309f;   // scale / c: the gradients through Qc' and Qc''
constexpr int kQT = 64;                  // queries per CTA
constexpr int kKT = 64;                  // keys per tile
constexpr int kWin = 128;                // position rows per tile window (127 used)
constexpr int kBdRing = 192;             // BD ring columns per query row
constexpr int kBdPitch = 196;            // bf16 per ring row (padded; two CTAs still fit an SM)

// Shared memory (bytes).  Tiles of 64 bf16 per row are stored as 128-byte rows with the 16-byte
// chunk index xor-ed with the row (mod 8), so that ldmatrix reads of eight rows hit eight
// different bank groups; the G buffer (128 bf16 per row) xors the low three chunk bits.
struct BSmem {
    static constexpr int QU = 0;                         // [64][64] q + u
    static constexpr int QV = QU + kQT * 128;            // [64][64] q + v_bias
    static constexpr int GO = QV + kQT * 128;            // [64][64] dO
    static constexpr int K = GO + kQT * 128;             // [64][64] key tile
    static constexpr int V = K + kKT * 128;              // [64][64] value tile
    static constexpr int R = V + kKT * 128;              // [128][64] position window
    static constexpr int P = R + kWin * 128;             // [64][64] P (bf16)
    static constexpr int DS = P + kQT * 128;             // [64][64] dS (bf16)
    static constexpr int G = DS + kQT * 128;             // [64][128] dS by distance
    static constexpr int BD = G + kQT * 256;             // [64][kBdPitch] ring of BD window products (bf16)
    static constexpr int Size = BD + kQT * kBdPitch * 2;
};

// Key j of (b, h): memory ring slot for 0 <= j < M, current segment for M <= j < M + L, else null.
__device__ __forceinline__ void key_rows(const AttnSimtParams& a, int b, int h, int j, const __nv_bfloat16*& kp,
                                         const __nv_bfloat16*& vp)
{
    kp = vp = nullptr;
    if (j < 0 || j >= a.M + a.L) return;
    if (j < a.M) {
        int slot = a.wp + j;
        if (slot >= a.M) slot -= a.M;
        const int64_t off = b * a.m_sb + static_cast<int64_t>(slot) * a.m_st + h * a.m_sh;
        kp = static_cast<const __nv_bfloat16*>(a.kmem) + off;
        vp = static_cast<const __nv_bfloat16*>(a.vmem) + off;
    } else {
        const int t = j - a.M;
        kp = static_cast<const __nv_bfloat16*>(a.kcur) + b * a.kc_sb + static_cast<int64_t>(t) * a.kc_st + h * a.kc_sh;
        vp = static_cast<const __nv_bfloat16*>(a.vcur) + b * a.vc_sb + static_cast<int64_t>(t) * a.vc_st + h * a.vc_sh;
    }
}

// Issue the copies of the key tile (and the value tile) starting at key j0 and of the position
// window whose row 0 is distance tb (rows clamped into [0, min(C, n_rows - 1)]: rows outside pair
// only with masked (query, key) pairs, rows past clamp_len repeat r[clamp_len]).  Keys outside
// [0, M + L) are zero-filled.
__device__ __forceinline__ void issue_tiles(const BwdParams& p, uint8_t* sm, int b, int h, int j0, int tb, bool values,
                                            int tid)
{
    const AttnSimtParams& a = p.a;
    const int rmax = min(a.C, p.n_rows - 1);
#pragma unroll
    for (int x = 0; x < (kKT * 8) / kBT; ++x) {
        const int id = tid + kBT * x;
        const int row = id >> 3, ch = id & 7;
        const __nv_bfloat16 *kp, *vp;
        key_rows(a, b, h, j0 + row, kp, vp);
        const uint32_t nb = kp ? 16u : 0u;
        cp_async16(sm + BSmem::K + swz64(row, 8 * ch), kp ? static_cast<const void*>(kp + 8 * ch) : a.r, nb);
        if (values)
            cp_async16(sm + BSmem::V + swz64(row, 8 * ch), vp ? static_cast<const void*>(vp + 8 * ch) : a.r, nb);
    }
#pragma unroll
    for (int x = 0; x < (kWin * 8) / kBT; ++x) {
        const int id = tid + kBT * x;
        const int row = id >> 3, ch = id & 7;
        const int rr = min(max(tb + row, 0), rmax);
        cp_async16(sm + BSmem::R + swz64(row, 8 * ch),
                   static_cast<const __nv_bfloat16*>(a.r) + static_cast<int64_t>(rr) * a.r_row + h * a.r_head + 8 * ch,
                   16u);
    }
    cp_async_commit();
}

// Scores of this warp's 16 rows against key tile t (keys from j0), in the log2 domain (c s), masked
// to -inf: S = Qc' K^T from the tensor cores plus BD remapped from the window product Qc'' R_win^T,
// with the scaled query forms Qc' = bf16(c q'), Qc'' = bf16(c q'') of the forward kernel.
// Window row w of tile t + 1 is window row w + 64 of tile t, so the products live in a per-row ring
// (row w of tile t in column (w + 64 t) mod 192) and every tile after a sweep's first multiplies
// only its 64 new rows.
__device__ __forceinline__ void tile_scores(const BwdParams& p, uint8_t* sm, int warp, int lane, int i0, int j0,
                                            int t, float (&s)[8][4])
{
    const AttnSimtParams& a = p.a;
    const uint32_t sbase = cvta_smem(sm);
    const int g = lane >> 2, tg = lane & 3;
#pragma unroll
    for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
    // S = Q' K^T: A = Q' rows 16w.., B = K tile as [key][d]
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        int r, cc;
        a_rc(lane, 16 * warp, 16 * kk, r, cc);
        uint32_t a0, a1, a2, a3;
        ldsm_x4(sbase + BSmem::QU + swz64(r, cc), a0, a1, a2, a3);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
            b_nk(lane, 16 * np, 16 * kk, r, cc);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(sbase + BSmem::K + swz64(r, cc), b0, b1, b2, b3);
            mma16816(s[2 * np], a0, a1, a2, a3, b0, b1);
            mma16816(s[2 * np + 1], a0, a1, a2, a3, b2, b3);
        }
    }
    // BD over the window's new rows (both halves on the first tile, rows 64..127 after), staged as
    // bf16 in this warp's ring rows
    __nv_bfloat16* bd = reinterpret_cast<__nv_bfloat16*>(sm + BSmem::BD);
    const int roff = (kKT * t) % kBdRing;
#pragma unroll 1
    for (int half = t == 0 ? 0 : 1; half < 2; ++half) {
        float w[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n) w[n][0] = w[n][1] = w[n][2] = w[n][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            int r, cc;
            a_rc(lane, 16 * warp, 16 * kk, r, cc);
            uint32_t a0, a1, a2, a3;
            ldsm_x4(sbase + BSmem::QV + swz64(r, cc), a0, a1, a2, a3);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                b_nk(lane, 64 * half + 16 * np, 16 * kk, r, cc);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(sbase + BSmem::R + swz64(r, cc), b0, b1, b2, b3);
                mma16816(w[2 * np], a0, a1, a2, a3, b0, b1);
                mma16816(w[2 * np + 1], a0, a1, a2, a3, b2, b3);
            }
        }
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const int col = (64 * half + 8 * n + 2 * tg + roff) % kBdRing;
            const int r0 = 16 * warp + g;
            *reinterpret_cast<uint32_t*>(bd + r0 * kBdPitch + col) = pack2(w[n][0], w[n][1]);
            *reinterpret_cast<uint32_t*>(bd + (r0 + 8) * kBdPitch + col) = pack2(w[n][2], w[n][3]);
        }
    }
    __syncwarp();
    // s_ij = S_ij + BD[i][i - j + 63] (both already scaled by c) for visible pairs, -inf otherwise
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const int il = 16 * warp + g + 8 * hr;
        const int i = i0 + il;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int jl = 8 * n + 2 * tg + e;
                const int j = j0 + jl;
                const bool vis = i < a.L && j >= a.lo && j <= a.M + i && j < a.M + a.L;
                int cw = il - jl + 63 + roff;
                cw = cw >= kBdRing ? cw - kBdRing : cw;
                const float x = s[n][2 * hr + e] + __bfloat162float(bd[il * kBdPitch + cw]);
                s[n][2 * hr + e] = vis ? x : -INFINITY;
            }
        }
    }
}

__global__ void __launch_bounds__(kBT) bwd_tc_kernel(const BwdParams p)
{
    extern __shared__ __align__(128) uint8_t sm[];
    const AttnSimtParams& a = p.a;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, tg = lane & 3;
    // grid (H, B, query tiles) with the query tile slowest and reversed: the CTAs with the most key
    // tiles are dispatched first, the short ones fill the last wave
    const int h = blockIdx.x, b = blockIdx.y, qt = gridDim.z - 1 - blockIdx.z;
    const int i0 = kQT * qt;
    const uint32_t sbase = cvta_smem(sm);
    const float c = a.scale * 1.4426950408889634f;

    // ---- Qc' = c (q + u), Qc'' = c (q + v_bias) and dO of the CTA's rows (bf16, zero past L), the
    //      query forms rounded exactly as the forward kernel rounds them (one fma of q with c and the
    //      product c u), so that the forward's log-sum-exp belongs to these scores
#pragma unroll
    for (int x = 0; x < (kQT * 8) / kBT; ++x) {
        const int id = tid + kBT * x;
        const int row = id >> 3, ch = id & 7;
        const int i = i0 + row;
        uint4 wu = make_uint4(0, 0, 0, 0), wv = wu, wg = wu;
        if (i < a.L) {
            const uint4 qq = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) + b * a.q_sb +
                                                                  static_cast<int64_t>(i) * a.q_st + h * a.q_sh) + ch);
            wg = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.dout) + b * p.g_sb +
                                                      static_cast<int64_t>(i) * p.g_st + h * p.g_sh) + ch);
            const uint32_t qw[4] = {qq.x, qq.y, qq.z, qq.w};
            uint32_t ou[4], ov[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int d = 8 * ch + 2 * e;
                const float x0 = bf16_lo(qw[e]), x1 = bf16_hi(qw[e]);
                ou[e] = pack2(fmaf(x0, c, __ldg(a.u + h * 64 + d) * c), fmaf(x1, c, __ldg(a.u + h * 64 + d + 1) * c));
                ov[e] = pack2(fmaf(x0, c, __ldg(a.vb + h * 64 + d) * c), fmaf(x1, c, __ldg(a.vb + h * 64 + d + 1) * c));
            }
            wu = make_uint4(ou[0], ou[1], ou[2], ou[3]);
            wv = make_uint4(ov[0], ov[1], ov[2], ov[3]);
        }
        *reinterpret_cast<uint4*>(sm + BSmem::QU + swz64(row, 8 * ch)) = wu;
        *reinterpret_cast<uint4*>(sm + BSmem::QV + swz64(row, 8 * ch)) = wv;
        *reinterpret_cast<uint4*>(sm + BSmem::GO + swz64(row, 8 * ch)) = wg;
    }

    // ---- D_i = dO_i . out_i for this thread's rows (16 dimensions per lane of a quad)
    float Dd[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const int i = i0 + 16 * warp + g + 8 * hr;
        float acc = 0.f;
        if (i < a.L) {
            const __nv_bfloat16* go = static_cast<const __nv_bfloat16*>(p.dout) + b * p.g_sb +
                                      static_cast<int64_t>(i) * p.g_st + h * p.g_sh + 16 * tg;
            const __nv_bfloat16* oo = static_cast<const __nv_bfloat16*>(a.out) + b * a.o_sb +
                                      static_cast<int64_t>(i) * a.o_st + h * a.o_sh + 16 * tg;
#pragma unroll
            for (int d = 0; d < 16; ++d) acc = fmaf(__bfloat162float(go[d]), __bfloat162float(oo[d]), acc);
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        Dd[hr] = acc;
    }

    const int n_t = (a.M + i0 + kQT - 1 - a.lo) / kKT + 1;

    // ---- sweep 1: row log-sum-exp (log2 domain), unless the fused forward kernel has written it
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
    for (int t = 0; t < (p.lse_given ? 0 : n_t); ++t) {
        const int j0 = a.M + i0 - kKT * t;
        __syncthreads();
        issue_tiles(p, sm, b, h, j0, kKT * t - (kKT - 1), false, tid);
        cp_async_wait_all();
        __syncthreads();
        float s[8][4];
        tile_scores(p, sm, warp, lane, i0, j0, t, s);
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            float mx = -INFINITY;
#pragma unroll
            for (int n = 0; n < 8; ++n) mx = fmaxf(mx, fmaxf(s[n][2 * hr], s[n][2 * hr + 1]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mnew = fmaxf(mrow[hr], mx);
            // a row with nothing visible yet keeps a zero sum (every lane takes every shuffle)
            const float mref = mnew == -INFINITY ? 0.f : mnew;
            float sum = 0.f;
#pragma unroll
            for (int n = 0; n < 8; ++n) sum += ex2(s[n][2 * hr] - mref) + ex2(s[n][2 * hr + 1] - mref);
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            lrow[hr] = lrow[hr] * ex2(mrow[hr] - mref) + sum;
            mrow[hr] = mnew;
        }
    }
    float L2[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const int i = i0 + 16 * warp + g + 8 * hr;
        if (p.lse_given)
            L2[hr] = i < a.L ? p.lse[(static_cast<int64_t>(b) * a.L + i) * a.H + h] : 0.f;
        else
            L2[hr] = lrow[hr] > 0.f ? mrow[hr] + __log2f(lrow[hr]) : 0.f;
    }

    // ---- sweep 2: gradients
    float dqa[8][4], dqb[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) dqa[n][e] = dqb[n][e] = 0.f;
    float csum[2] = {0.f, 0.f};                          // fp32 dS of the pairs at or past clamp_len
    const float scale = a.scale;
    // tile t + 1's keys, values and window are copied in while tile t's dv, dk and dr products run
    __syncthreads();
    issue_tiles(p, sm, b, h, a.M + i0, -(kKT - 1), true, tid);
    for (int t = 0; t < n_t; ++t) {
        const int j0 = a.M + i0 - kKT * t;
        const int tb = kKT * t - (kKT - 1);                  // distance of window row 0
        cp_async_wait_all();
        __syncthreads();
        float s[8][4];
        tile_scores(p, sm, warp, lane, i0, j0, t, s);
        // P, in place
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[n][e] = ex2(s[n][e] - L2[e >> 1]);
        // dP = dO V^T
        float dp[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n) dp[n][0] = dp[n][1] = dp[n][2] = dp[n][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            int r, cc;
            a_rc(lane, 16 * warp, 16 * kk, r, cc);
            uint32_t a0, a1, a2, a3;
            ldsm_x4(sbase + BSmem::GO + swz64(r, cc), a0, a1, a2, a3);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                b_nk(lane, 16 * np, 16 * kk, r, cc);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(sbase + BSmem::V + swz64(r, cc), b0, b1, b2, b3);
                mma16816(dp[2 * np], a0, a1, a2, a3, b0, b1);
                mma16816(dp[2 * np + 1], a0, a1, a2, a3, b2, b3);
            }
        }
        // dS = P (dP - D), bf16 pairs (row g: e = 0, 1; row g + 8: e = 2, 3); P and dS to shared
        // memory for the CTA-wide products, dS by distance into G (this warp's rows, zeroed first)
        // for distances below clamp_len, the rest summed in fp32
        uint32_t dsw[8][2];
        {
            uint4* grow = reinterpret_cast<uint4*>(sm + BSmem::G + (16 * warp) * 256);
#pragma unroll
            for (int x = 0; x < 8; ++x) grow[lane + 32 * x] = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const int jl = 8 * n + 2 * tg;
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int il = 16 * warp + g + 8 * hr;
                const float d0 = s[n][2 * hr] * (dp[n][2 * hr] - Dd[hr]);
                const float d1 = s[n][2 * hr + 1] * (dp[n][2 * hr + 1] - Dd[hr]);
                dsw[n][hr] = pack2(d0, d1);
                *reinterpret_cast<uint32_t*>(sm + BSmem::P + swz64(il, jl)) = pack2(s[n][2 * hr], s[n][2 * hr + 1]);
                *reinterpret_cast<uint32_t*>(sm + BSmem::DS + swz64(il, jl)) = dsw[n][hr];
                // key jl (distance 64 t + il - jl) goes to window column il - jl + 63, key jl + 1 to
                // the column before it
                const int dist = kKT * t + il - jl;
                if (dist < a.C)
                    *reinterpret_cast<__nv_bfloat16*>(sm + BSmem::G + swz128(il, il - jl + 63)) =
                        __ushort_as_bfloat16(static_cast<unsigned short>(dsw[n][hr] & 0xffffu));
                else
                    csum[hr] += d0;
                if (dist - 1 < a.C)
                    *reinterpret_cast<__nv_bfloat16*>(sm + BSmem::G + swz128(il, il - jl + 62)) =
                        __ushort_as_bfloat16(static_cast<unsigned short>(dsw[n][hr] >> 16));
                else
                    csum[hr] += d1;
            }
        }
        // dq_ac += dS K: A = dS from the accumulator layout (n-tiles 2kk, 2kk + 1 form k-step kk)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint32_t a0 = dsw[2 * kk][0], a1 = dsw[2 * kk][1], a2 = dsw[2 * kk + 1][0], a3 = dsw[2 * kk + 1][1];
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                int r, cc;
                b_kn(lane, 16 * kk, 16 * np, r, cc);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(sbase + BSmem::K + swz64(r, cc), b0, b1, b2, b3);
                mma16816(dqa[2 * np], a0, a1, a2, a3, b0, b1);
                mma16816(dqa[2 * np + 1], a0, a1, a2, a3, b2, b3);
            }
        }
        __syncwarp();
        // dq_bd += G R_win: A = this warp's G rows, B = the window as [distance][d]
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            int r, cc;
            a_rc(lane, 16 * warp, 16 * kk, r, cc);
            uint32_t a0, a1, a2, a3;
            ldsm_x4(sbase + BSmem::G + swz128(r, cc), a0, a1, a2, a3);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                b_kn(lane, 16 * kk, 16 * np, r, cc);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(sbase + BSmem::R + swz64(r, cc), b0, b1, b2, b3);
                mma16816(dqb[2 * np], a0, a1, a2, a3, b0, b1);
                mma16816(dqb[2 * np + 1], a0, a1, a2, a3, b2, b3);
            }
        }
        __syncthreads();                                    // P, dS and G of all rows are in place
        if (t + 1 < n_t) issue_tiles(p, sm, b, h, j0 - kKT, tb + kKT, true, tid);   // K, V, R are free
        // dv, dk of the current keys j0 + 16w .. (warp w): P^T dO and scale dS^T Q'
        const int jw = j0 + 16 * warp;
        if (jw + 15 >= a.M && jw < a.M + a.L) {
            float acc[8][4];
#pragma unroll
            for (int pass = 0; pass < 2; ++pass) {
#pragma unroll
                for (int n = 0; n < 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
                const uint32_t asrc = sbase + (pass == 0 ? BSmem::P : BSmem::DS);
                const uint32_t bsrc = sbase + (pass == 0 ? BSmem::GO : BSmem::QU);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    int r, cc;
                    a_km(lane, 16 * warp, 16 * kk, r, cc);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(asrc + swz64(r, cc), a0, a1, a2, a3);
#pragma unroll
                    for (int np = 0; np < 4; ++np) {
                        b_kn(lane, 16 * kk, 16 * np, r, cc);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(bsrc + swz64(r, cc), b0, b1, b2, b3);
                        mma16816(acc[2 * np], a0, a1, a2, a3, b0, b1);
                        mma16816(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
                    }
                }
                float* dst = pass == 0 ? p.dv : p.dk;
                const float f = pass == 0 ? 1.f : kLn2;     // scale dS^T q' = ln 2 dS^T Qc'
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int j = jw + g + 8 * hr;
                    if (j < a.M || j >= a.M + a.L) continue;
                    float* row = dst + ((static_cast<int64_t>(b) * a.L + (j - a.M)) * a.H + h) * 64;
#pragma unroll
                    for (int n = 0; n < 8; ++n)
                        atomicAdd(reinterpret_cast<float2*>(row + 8 * n + 2 * tg),
                                  make_float2(f * acc[n][2 * hr], f * acc[n][2 * hr + 1]));
                }
            }
        }
        // dr over the window: warp w takes window rows 32w .. 32w + 31, G^T Q''
        {
            float acc[2][8][4];
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int n = 0; n < 8; ++n) acc[m][n][0] = acc[m][n][1] = acc[m][n][2] = acc[m][n][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    int r, cc;
                    a_km(lane, 32 * warp + 16 * m, 16 * kk, r, cc);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(sbase + BSmem::G + swz128(r, cc), a0, a1, a2, a3);
#pragma unroll
                    for (int np = 0; np < 4; ++np) {
                        b_kn(lane, 16 * kk, 16 * np, r, cc);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(sbase + BSmem::QV + swz64(r, cc), b0, b1, b2, b3);
                        mma16816(acc[m][2 * np], a0, a1, a2, a3, b0, b1);
                        mma16816(acc[m][2 * np + 1], a0, a1, a2, a3, b2, b3);
                    }
                }
            }
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int td = tb + 32 * warp + 16 * m + g + 8 * hr;
                    // rows past the clamp are empty in G; rows past the table pair with no visible key
                    if (td < 0 || td >= a.C || td >= p.n_rows) continue;
                    float* dst = p.dr + (static_cast<int64_t>(td) * a.H + h) * 64;
#pragma unroll
                    for (int n = 0; n < 8; ++n)
                        atomicAdd(reinterpret_cast<float2*>(dst + 8 * n + 2 * tg),
                                  make_float2(kLn2 * acc[m][n][2 * hr], kLn2 * acc[m][n][2 * hr + 1]));
                }
        }
    }

    // ---- the clamped pairs: c_i r[C] into dq_bd, sum_i c_i q''_i into dr[C]
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        csum[hr] += __shfl_xor_sync(0xffffffffu, csum[hr], 1);
        csum[hr] += __shfl_xor_sync(0xffffffffu, csum[hr], 2);
    }
    if (a.C < p.n_rows) {                                // else no distance reaches clamp_len
        const __nv_bfloat16* rc = static_cast<const __nv_bfloat16*>(a.r) + static_cast<int64_t>(a.C) * a.r_row +
                                  h * a.r_head;
        float part[8][2];
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const int d = 8 * n + 2 * tg;
            const float r0 = __bfloat162float(rc[d]), r1 = __bfloat162float(rc[d + 1]);
            dqb[n][0] += csum[0] * r0;
            dqb[n][1] += csum[0] * r1;
            dqb[n][2] += csum[1] * r0;
            dqb[n][3] += csum[1] * r1;
            const uint32_t q0 = *reinterpret_cast<const uint32_t*>(sm + BSmem::QV + swz64(16 * warp + g, d));
            const uint32_t q1 = *reinterpret_cast<const uint32_t*>(sm + BSmem::QV + swz64(16 * warp + g + 8, d));
            part[n][0] = csum[0] * bf16_lo(q0) + csum[1] * bf16_lo(q1);
            part[n][1] = csum[0] * bf16_hi(q0) + csum[1] * bf16_hi(q1);
        }
        // sum over the warp's 16 rows (lanes of equal tg), one atomic pair per column pair
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                part[n][e] += __shfl_xor_sync(0xffffffffu, part[n][e], 4);
                part[n][e] += __shfl_xor_sync(0xffffffffu, part[n][e], 8);
                part[n][e] += __shfl_xor_sync(0xffffffffu, part[n][e], 16);
            }
        if (g == 0) {
            float* dst = p.dr + (static_cast<int64_t>(a.C) * a.H + h) * 64;
#pragma unroll
            for (int n = 0; n < 8; ++n)
                atomicAdd(reinterpret_cast<float2*>(dst + 8 * n + 2 * tg),
                          make_float2(kLn2 * part[n][0], kLn2 * part[n][1]));
        }
    }

    // ---- dq and the per-query parts of du (dS K) and dv_bias (dS r)
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const int i = i0 + 16 * warp + g + 8 * hr;
        if (i >= a.L) continue;
        const int64_t row = ((static_cast<int64_t>(b) * a.L + i) * a.H + h) * 64;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const int d = 8 * n + 2 * tg;
            const float xa0 = scale * dqa[n][2 * hr], xa1 = scale * dqa[n][2 * hr + 1];
            const float xb0 = scale * dqb[n][2 * hr], xb1 = scale * dqb[n][2 * hr + 1];
            *reinterpret_cast<float2*>(p.dq + row + d) = make_float2(xa0 + xb0, xa1 + xb1);
            *reinterpret_cast<float2*>(p.pac + row + d) = make_float2(xa0, xa1);
            *reinterpret_cast<float2*>(p.pbd + row + d) = make_float2(xb0, xb1);
        }
    }
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool st8(int64_t s) { return (s & 7) == 0; }

}  // namespace

bool bwd_tc_eligible(const BwdParams& p, txl_dtype dtype)
{
    const AttnSimtParams& a = p.a;
    if (dtype != TXL_BF16 || a.D != 64 || a.H > 65535 || a.B > 65535) return false;
    bool ok = al16(a.q) && st8(a.q_sb) && st8(a.q_st) && st8(a.q_sh) && al16(a.kcur) && st8(a.kc_sb) &&
              st8(a.kc_st) && st8(a.kc_sh) && al16(a.vcur) && st8(a.vc_sb) && st8(a.vc_st) && st8(a.vc_sh) &&
              al16(p.dout) && st8(p.g_sb) && st8(p.g_st) && st8(p.g_sh) && al16(a.r) && st8(a.r_row) && st8(a.r_head);
    if (a.M > 0) ok = ok && al16(a.kmem) && al16(a.vmem) && st8(a.m_sb) && st8(a.m_st) && st8(a.m_sh);
    return ok;
}

// dq, pac, pbd are written; dk, dv and dr must be zero on entry (atomic accumulation).
cudaError_t launch_bwd_tc(const BwdParams& p, cudaStream_t s)
{
    static bool attr_done = false;
    if (!attr_done) {
        const cudaError_t e = cudaFuncSetAttribute(bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, BSmem::Size);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    const dim3 grid(p.a.H, p.a.B, (p.a.L + kQT - 1) / kQT);
    bwd_tc_kernel<<<grid, kBT, BSmem::Size, s>>>(p);
    return cudaGetLastError();
}

}  // namespace txl
