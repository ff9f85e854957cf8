// txl_table_tc.cu -- the learned-table variant of the relative attention on the tensor cores
// (bf16, d_head = 64): the same scores as txl_table.cu ("TransformerXL 相对位置编码" §3.1)
//   s_ij = (scale q_i + u) . k_j + (scale q_i + v) . r_table[clamp(i - j + max_len - 1, 0, 2 max_len - 2)]
// over one bidirectional sequence, masked keys scored -1e9, out_i = softmax_j(s_ij) v_j.
//
// One CTA of four warps per (query tile of 64, head, batch entry); warp w owns query rows
// 16w .. 16w + 15.  For key tile j0 the table indices of the pairs fill a window of 127 rows
// starting at i0 - j0 - 63 + max_len - 1 (clamped into the table), so the table term is the window
// product (scale q + v) W^T remapped per row through shared memory, exactly as the relative shift
// of the Transformer-XL kernels.  The window of tile t + 1 shares 64 rows with the window of tile t
// (for the same query rows), so the window products live in a per-row ring of 192 columns and every
// tile after the first loads and multiplies only its 64 new rows.  bf16 mma.sync products with fp32
// accumulation, an online softmax in the log2 domain, O += P V with P taken straight from the
// accumulators; the next key tile, value tile and window rows are copied in with cp.async while the
// current tile is computed.
#include <cuda_bf16.h>

#include "txl_internal.h"
#include "txl_mma.cuh"

namespace txl {

namespace {

using namespace mma;

constexpr int kTT = 128;                 // threads: four warps
constexpr int kTQ = 64;                  // queries per CTA
constexpr int kTK = 64;                  // keys per tile
constexpr int kTWin = 128;               // table rows per window (127 used)
constexpr int kTRing = 192;              // window-product ring columns per query row
constexpr int kTBdPitch = 200;           // bf16 per ring row (padded)
constexpr float kLog2e = 1.4426950408889634f;

struct TSmem {
    static constexpr int QA = 0;                         // [64][64] scale q + u
    static constexpr int QB = QA + kTQ * 128;            // [64][64] scale q + v
    static constexpr int BUF = QB + kTQ * 128;           // two buffers of: key tile, value tile, window
    static constexpr int K = 0, V = kTK * 128, W = 2 * kTK * 128;
    static constexpr int BufBytes = W + kTWin * 128;
    static constexpr int BD = BUF + 2 * BufBytes;        // [64][kTBdPitch] ring of window products (bf16)
    static constexpr int Size = BD + kTQ * kTBdPitch * 2;
};

// Copies of key tile j0, its value tile and the first n_win (64 or 128) rows of its table window.
__device__ __forceinline__ void issue_table_tiles(const TableParams& p, uint8_t* buf, int b, int h, int i0, int j0,
                                                  int n_win, int tid)
{
    const __nv_bfloat16* kb = static_cast<const __nv_bfloat16*>(p.k);
    const __nv_bfloat16* vb = static_cast<const __nv_bfloat16*>(p.v);
#pragma unroll
    for (int x = 0; x < (kTK * 8) / kTT; ++x) {
        const int id = tid + kTT * x;
        const int row = id >> 3, ch = id & 7;
        const int j = j0 + row;
        const bool in = j < p.L;
        const int64_t kof = b * p.k_sb + static_cast<int64_t>(in ? j : 0) * p.k_st + h * p.k_sh + 8 * ch;
        const int64_t vof = b * p.v_sb + static_cast<int64_t>(in ? j : 0) * p.v_st + h * p.v_sh + 8 * ch;
        cp_async16(buf + TSmem::K + swz64(row, 8 * ch), kb + kof, in ? 16u : 0u);
        cp_async16(buf + TSmem::V + swz64(row, 8 * ch), vb + vof, in ? 16u : 0u);
    }
    const int top = 2 * p.max_len - 2;
    const int w0 = i0 - j0 - (kTK - 1) + p.max_len - 1;  // table index of window row 0
#pragma unroll
    for (int x = 0; x < (kTWin * 8) / kTT; ++x) {
        const int id = tid + kTT * x;
        const int row = id >> 3, ch = id & 7;
        if (row >= n_win) break;
        const int rr = min(max(w0 + row, 0), top);
        cp_async16(buf + TSmem::W + swz64(row, 8 * ch),
                   static_cast<const __nv_bfloat16*>(p.r) + static_cast<int64_t>(rr) * p.r_row + h * p.r_head + 8 * ch,
                   16u);
    }
    cp_async_commit();
}

__global__ void __launch_bounds__(kTT) table_tc_kernel(const TableParams p)
{
    extern __shared__ __align__(128) uint8_t sm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, tg = lane & 3;
    const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int i0 = kTQ * qt;
    const uint32_t sbase = cvta_smem(sm);
    const int n_kt = (p.L + kTK - 1) / kTK;

    issue_table_tiles(p, sm + TSmem::BUF, b, h, i0, 0, kTWin, tid);

    // scale q + u and scale q + v of the CTA's rows (bf16, zero past L)
#pragma unroll
    for (int x = 0; x < (kTQ * 8) / kTT; ++x) {
        const int id = tid + kTT * x;
        const int row = id >> 3, ch = id & 7;
        const int i = i0 + row;
        uint4 wa = make_uint4(0, 0, 0, 0), wb = wa;
        if (i < p.L) {
            const uint4 qq = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) + b * p.q_sb +
                                                                  static_cast<int64_t>(i) * p.q_st + h * p.q_sh) + ch);
            const uint32_t qw[4] = {qq.x, qq.y, qq.z, qq.w};
            uint32_t oa[4], ob[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int d = 8 * ch + 2 * e;
                const float x0 = bf16_lo(qw[e]) * p.scale, x1 = bf16_hi(qw[e]) * p.scale;
                oa[e] = pack2(x0 + __ldg(p.u + h * 64 + d), x1 + __ldg(p.u + h * 64 + d + 1));
                ob[e] = pack2(x0 + __ldg(p.vb + h * 64 + d), x1 + __ldg(p.vb + h * 64 + d + 1));
            }
            wa = make_uint4(oa[0], oa[1], oa[2], oa[3]);
            wb = make_uint4(ob[0], ob[1], ob[2], ob[3]);
        }
        *reinterpret_cast<uint4*>(sm + TSmem::QA + swz64(row, 8 * ch)) = wa;
        *reinterpret_cast<uint4*>(sm + TSmem::QB + swz64(row, 8 * ch)) = wb;
    }

    float o[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY}, lpart[2] = {0.f, 0.f};
    __nv_bfloat16* bd = reinterpret_cast<__nv_bfloat16*>(sm + TSmem::BD);

    for (int t = 0; t < n_kt; ++t) {
        const int j0 = kTK * t;
        cp_async_wait_all();
        __syncthreads();                 // tile t landed; every warp is done with buffer (t + 1) & 1
        if (t + 1 < n_kt)
            issue_table_tiles(p, sm + TSmem::BUF + ((t + 1) & 1) * TSmem::BufBytes, b, h, i0, j0 + kTK, kTK, tid);
        // window row w of this tile sits in ring column (w + 128 t) mod 192: tile t + 1's rows 64..127
        // are tile t's rows 0..63, already in the ring
        const int roff = (128 * t) % kTRing;
        const uint32_t buf = sbase + TSmem::BUF + (t & 1) * TSmem::BufBytes;

        // S = Qa K^T
        float s[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            int r, cc;
            a_rc(lane, 16 * warp, 16 * kk, r, cc);
            uint32_t a0, a1, a2, a3;
            ldsm_x4(sbase + TSmem::QA + swz64(r, cc), a0, a1, a2, a3);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                b_nk(lane, 16 * np, 16 * kk, r, cc);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(buf + TSmem::K + swz64(r, cc), b0, b1, b2, b3);
                mma16816(s[2 * np], a0, a1, a2, a3, b0, b1);
                mma16816(s[2 * np + 1], a0, a1, a2, a3, b2, b3);
            }
        }
        // window product Qb W^T of the new rows (both halves on the first tile, rows 0..63 after),
        // staged as bf16 in this warp's ring rows
#pragma unroll 1
        for (int half = 0; half < (t == 0 ? 2 : 1); ++half) {
            float w[8][4];
#pragma unroll
            for (int n = 0; n < 8; ++n) w[n][0] = w[n][1] = w[n][2] = w[n][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                int r, cc;
                a_rc(lane, 16 * warp, 16 * kk, r, cc);
                uint32_t a0, a1, a2, a3;
                ldsm_x4(sbase + TSmem::QB + swz64(r, cc), a0, a1, a2, a3);
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    b_nk(lane, 64 * half + 16 * np, 16 * kk, r, cc);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(buf + TSmem::W + swz64(r, cc), b0, b1, b2, b3);
                    mma16816(w[2 * np], a0, a1, a2, a3, b0, b1);
                    mma16816(w[2 * np + 1], a0, a1, a2, a3, b2, b3);
                }
            }
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                const int col = (64 * half + 8 * n + 2 * tg + roff) % kTRing;
                const int r0 = 16 * warp + g;
                *reinterpret_cast<uint32_t*>(bd + r0 * kTBdPitch + col) = pack2(w[n][0], w[n][1]);
                *reinterpret_cast<uint32_t*>(bd + (r0 + 8) * kTBdPitch + col) = pack2(w[n][2], w[n][3]);
            }
        }
        __syncwarp();
        // log2-domain scores: keys past L excluded, masked keys -1e9 (natural units)
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int jl = 8 * n + 2 * tg + e;
                const int j = j0 + jl;
                const bool in = j < p.L;
                const bool keep = in && (!p.mask || p.mask[static_cast<int64_t>(b) * p.L + j] != 0);
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int il = 16 * warp + g + 8 * hr;
                    int c = il - jl + 63 + roff;
                    c = c >= kTRing ? c - kTRing : c;
                    const float x = s[n][2 * hr + e] + __bfloat162float(bd[il * kTBdPitch + c]);
                    s[n][2 * hr + e] = keep ? kLog2e * x : (in ? -1e9f * kLog2e : -INFINITY);
                }
            }
        // online softmax: per-thread partial row sums, quad-wide maxima
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            float mx = -INFINITY;
#pragma unroll
            for (int n = 0; n < 8; ++n) mx = fmaxf(mx, fmaxf(s[n][2 * hr], s[n][2 * hr + 1]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mnew = fmaxf(mrow[hr], mx);
            const float mref = mnew == -INFINITY ? 0.f : mnew;
            const float alpha = ex2(mrow[hr] - mref);
            mrow[hr] = mnew;
            lpart[hr] *= alpha;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                o[n][2 * hr] *= alpha;
                o[n][2 * hr + 1] *= alpha;
                s[n][2 * hr] = ex2(s[n][2 * hr] - mref);
                s[n][2 * hr + 1] = ex2(s[n][2 * hr + 1] - mref);
            }
        }
        // P (bf16, the accumulator layout re-used as the A operand) times V; the row sums add
        // the same bf16 values
        uint32_t pw[8][2];
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                pw[n][hr] = pack2(s[n][2 * hr], s[n][2 * hr + 1]);
                lpart[hr] += bf16_lo(pw[n][hr]) + bf16_hi(pw[n][hr]);
            }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint32_t a0 = pw[2 * kk][0], a1 = pw[2 * kk][1], a2 = pw[2 * kk + 1][0], a3 = pw[2 * kk + 1][1];
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                int r, cc;
                b_kn(lane, 16 * kk, 16 * np, r, cc);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(buf + TSmem::V + swz64(r, cc), b0, b1, b2, b3);
                mma16816(o[2 * np], a0, a1, a2, a3, b0, b1);
                mma16816(o[2 * np + 1], a0, a1, a2, a3, b2, b3);
            }
        }
    }

    // out = O / l (bf16 pairs)
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        float l = lpart[hr];
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        const int i = i0 + 16 * warp + g + 8 * hr;
        if (i >= p.L) continue;
        const float inv = 1.f / l;
        __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) + b * p.o_sb + static_cast<int64_t>(i) * p.o_st +
                              h * p.o_sh;
#pragma unroll
        for (int n = 0; n < 8; ++n)
            *reinterpret_cast<uint32_t*>(orow + 8 * n + 2 * tg) = pack2(o[n][2 * hr] * inv, o[n][2 * hr + 1] * inv);
    }
}

inline bool al16(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }
inline bool st8(int64_t s) { return (s & 7) == 0; }

}  // namespace

bool table_tc_eligible(const TableParams& p, txl_dtype dtype)
{
    if (dtype != TXL_BF16 || p.D != 64 || p.H > 65535 || p.B > 65535) return false;
    return al16(p.q) && st8(p.q_sb) && st8(p.q_st) && st8(p.q_sh) && al16(p.k) && st8(p.k_sb) && st8(p.k_st) &&
           st8(p.k_sh) && al16(p.v) && st8(p.v_sb) && st8(p.v_st) && st8(p.v_sh) && al16(p.out) && st8(p.o_sb) &&
           st8(p.o_st) && st8(p.o_sh) && al16(p.r) && st8(p.r_row) && st8(p.r_head);
}

cudaError_t launch_table_tc(const TableParams& p, cudaStream_t s)
{
    static bool attr_done = false;
    if (!attr_done) {
        const cudaError_t e = cudaFuncSetAttribute(table_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, TSmem::Size);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    const dim3 grid((p.L + kTQ - 1) / kTQ, p.H, p.B);
    table_tc_kernel<<<grid, kTT, TSmem::Size, s>>>(p);
    return cudaGetLastError();
}

}  // namespace txl
