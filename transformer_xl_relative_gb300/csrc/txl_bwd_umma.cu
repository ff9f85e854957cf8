// txl_bwd_umma.cu -- gradients of the relative attention on the 5th-generation tensor cores
// (bf16, d_head = 64): every product a tcgen05 MMA with its fp32 accumulator in tensor memory.
//
// The gradients are those of txl_bwd_tc.cu: the chain rule through the four-term score of
// "Transformer-XL 和相对位置编码" §2.3.2 and the softmax, the memory's keys and values being the
// stop-gradient part of §2.3.1.  With the forward kernel's row log-sum-exp L2_i (log2 domain) and
// its query forms Qc' = bf16(c (q + u)), Qc'' = bf16(c (q + v_bias)), c = scale log2 e:
//   s_ij = Qc'_i . k_j + Qc''_i . r[delta_ij],   P_ij = 2^(s_ij - L2_i),
//   dS_ij = P_ij (dO_i . v_j - dO_i . out_i),
//   dq_i = scale sum_j dS_ij (k_j + r[delta_ij]),   dk_j = ln 2 sum_i dS_ij Qc'_i,
//   dv_j = sum_i P_ij dO_i,   dr[delta] = ln 2 sum_{delta_ij = delta} dS_ij Qc''_i,
// delta_ij = min(M + i - j, clamp_len).
//
// One launch holds two kinds of CTA, each on 128 rows of one (b, h):
//  * a query CTA owns a query tile and sweeps the key tiles of 128 its queries see, newest
//    first (tile t starts at key M + i0 - 128 t, so its distances are 128 t + i - j with i, j
//    local, window column c = i - j + 127 in [0, 255) over position rows 128 t - 127 + c).  It
//    accumulates dq_ac = dS K and dq_bd = G R_win in TMEM over the sweep, where G, dS scattered
//    by distance (G[i][i - j + 127] = dS_ij), sits in shared memory as the A operand of that
//    product and, read transposed, of dr_win = G^T Qc''.  The window's lower 128 rows are the
//    upper 128 of the tile before, so every block of 128 distance rows receives the products of
//    two consecutive tiles and is added to dr (fp32 atomics) once, while the next tile's score
//    products run.  The sums of dq_ac and dq_bd over the CTA's queries are added into du and
//    dv_bias.
//  * a key CTA owns a key tile of the current segment and sweeps the query tiles that see it,
//    with dv += P^T dO and dk += dS^T Qc' accumulated in TMEM (P and dS in shared memory, read
//    transposed): every key has one owner, so dk and dv are written once, without atomics.
// Both recompute, per (query tile, key tile), S = Qc' K^T, the window products W = Qc'' R_win^T
// (both 128-row halves), P and dP = dO V^T.  W reaches each row's positions through a shared-
// memory stage (the relative shift as a per-row index remap, bf16 like the forward's ring), so
// the scores are the forward kernel's and L2_i belongs to them.
// Pairs whose distance reaches clamp_len share r[clamp_len]; their dS nearly cancel, so they stay
// out of the bf16 G and enter dq_i as c_i r[clamp_len] and dr[clamp_len] as ln 2 sum_i c_i Qc''_i
// with c_i their fp32 sum per row.
//
// 512 threads: thread (li, q) serves TMEM lane / tile row li and the column quarter q of every
// 128-column product; thread 0 issues the MMAs.  Steps run in phases separated by CTA barriers
// and one mbarrier that each group of MMAs commits to; every wait is bounded (2 s).
#include <cuda_bf16.h>

#include "txl_internal.h"
#include "txl_ptx.cuh"
#include "txl_mma.cuh"

namespace txl {

namespace {

constexpr int kUThreads = 512;
constexpr int kTileBytes = 16384;                  // 128 rows x 128 B, one 128-byte swizzle atom wide
constexpr int kStagePitch = 84;                    // 32-bit words per stage row (80 used)
constexpr int kDrPitch = 272;                      // bytes per staged fp32 dr row (256 used)
constexpr float kLn2u = 0.693147180559945309f;
constexpr uint64_t kUWaitNs = 2000000000ull;

// TMEM columns.  Query CTA: S, then dr_win (lower block in 0..63, upper in 64..127); W over
// 128..383, then dP in 128..255 and dS (bf16 pairs) in 256..319; dq_ac, dq_bd.  Key CTA: S; W,
// then dP; dv, dk.
constexpr uint32_t kColS = 0, kColW = 128, kColDP = 128, kColDS = 256, kColA0 = 384, kColA1 = 448;

struct USmem {
    static constexpr int QU = 0;                           // [128][64] Qc'  (query rows)
    static constexpr int QV = QU + kTileBytes;             // [128][64] Qc''
    static constexpr int GO = QV + kTileBytes;             // [128][64] dO (key CTA: even steps)
    static constexpr int K0 = GO + kTileBytes;             // key tiles, two slots (key CTA: K0 only,
    static constexpr int K1 = K0 + kTileBytes;             //   K1 takes the next query tile's raw q)
    static constexpr int V0 = K1 + kTileBytes;             // value tiles, two slots (key CTA: V0 only,
    static constexpr int V1 = V0 + kTileBytes;             //   V1 takes dO of the odd steps)
    static constexpr int R = V1 + kTileBytes;              // three [128][64] blocks of position rows
    static constexpr int X = R + 3 * kTileBytes;           // query CTA: G, 4 atoms [128][64];
                                                           // key CTA: P, 2 atoms, then dS, 2 atoms;
                                                           // first the W stage [128][kStagePitch] words
    static constexpr int Bar = X + 4 * kTileBytes;         // MMA completion, drain
    static constexpr int Misc = Bar + 16;                  // TMEM base, abort flag
    static constexpr int Csum = Misc + 16;                 // float [4][128]
    static constexpr int Bias = Csum + 4 * 128 * 4;        // float [2][64]: c u, c v_bias
    static constexpr int Size = Bias + 2 * 64 * 4;
};
static_assert(128 * kStagePitch * 4 <= 4 * kTileBytes && 128 * kDrPitch <= 4 * kTileBytes, "stage, dr rows inside X");
static_assert(USmem::Size <= 232448, "shared memory per CTA");

// Key j of (b, h): memory ring slot for lo <= j < M, current segment for M <= j < M + L, else
// null (zero-filled: such keys are masked, and zeros keep their products finite).
__device__ __forceinline__ void kv_rows(const AttnSimtParams& a, int b, int h, int j, const __nv_bfloat16*& kp,
                                        const __nv_bfloat16*& vp)
{
    kp = vp = nullptr;
    if (j < a.lo || j >= a.M + a.L) return;
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

// Keys j0 .. j0 + 127 into a K and a V slot (128-byte swizzled rows, the K-major layout of the
// MMA descriptors).
__device__ __forceinline__ void load_keys(const AttnSimtParams& a, uint8_t* kdst, uint8_t* vdst, int b, int h, int j0,
                                          int tid)
{
#pragma unroll
    for (int x = 0; x < 1024 / kUThreads; ++x) {
        const int id = tid + kUThreads * x;
        const int row = id >> 3, ch = id & 7;
        const __nv_bfloat16 *kp, *vp;
        kv_rows(a, b, h, j0 + row, kp, vp);
        const uint32_t nb = kp ? 16u : 0u;
        mma::cp_async16(kdst + mma::swz64(row, 8 * ch), kp ? static_cast<const void*>(kp + 8 * ch) : a.r, nb);
        mma::cp_async16(vdst + mma::swz64(row, 8 * ch), vp ? static_cast<const void*>(vp + 8 * ch) : a.r, nb);
    }
}

// Raw q and dO of query rows i0 .. i0 + 127 (zero past L) into two slots.
__device__ __forceinline__ void load_query_raw(const BwdParams& p, uint8_t* qdst, uint8_t* gdst, int b, int h, int i0,
                                               int tid)
{
    const AttnSimtParams& a = p.a;
#pragma unroll
    for (int x = 0; x < 1024 / kUThreads; ++x) {
        const int id = tid + kUThreads * x;
        const int row = id >> 3, ch = id & 7;
        const int i = i0 + row;
        const bool in = i < a.L;
        const __nv_bfloat16* qp = static_cast<const __nv_bfloat16*>(a.q) + b * a.q_sb + static_cast<int64_t>(in ? i : 0) * a.q_st +
                                  h * a.q_sh + 8 * ch;
        const __nv_bfloat16* gp = static_cast<const __nv_bfloat16*>(p.dout) + b * p.g_sb +
                                  static_cast<int64_t>(in ? i : 0) * p.g_st + h * p.g_sh + 8 * ch;
        mma::cp_async16(qdst + mma::swz64(row, 8 * ch), qp, in ? 16u : 0u);
        mma::cp_async16(gdst + mma::swz64(row, 8 * ch), gp, in ? 16u : 0u);
    }
}

// Position block beta (distances 128 beta - 127 + x, x = 0 .. 127, clamped into [0, min(C,
// n_rows - 1)]: rows below 0 pair only with masked keys, rows past clamp_len repeat r[clamp_len])
// into R slot beta mod 3.
__device__ __forceinline__ void load_rblock(const BwdParams& p, uint8_t* sm, int h, int beta, int tid)
{
    const AttnSimtParams& a = p.a;
    const int rmax = min(a.C, p.n_rows - 1);
    uint8_t* dst = sm + USmem::R + (beta % 3) * kTileBytes;
#pragma unroll
    for (int x = 0; x < 1024 / kUThreads; ++x) {
        const int id = tid + kUThreads * x;
        const int row = id >> 3, ch = id & 7;
        const int rr = min(max(128 * beta - 127 + row, 0), rmax);
        mma::cp_async16(dst + mma::swz64(row, 8 * ch),
                        static_cast<const __nv_bfloat16*>(a.r) + static_cast<int64_t>(rr) * a.r_row + h * a.r_head +
                            8 * ch,
                        16u);
    }
}

// Qc' = c (q + u) and Qc'' = c (q + v_bias) of query rows i0 .. i0 + 127 from their raw q (in
// shared memory, swizzled), rounded as the forward kernel rounds them (one fma of q with c and the
// product c u, c v_bias, held per dimension in shared memory); rows past L stay zero.
__device__ __forceinline__ void convert_queries(const AttnSimtParams& a, uint8_t* sm, const uint8_t* qraw, int i0, int tid)
{
    const float* uc = reinterpret_cast<const float*>(sm + USmem::Bias);
    const float* vc = uc + 64;
#pragma unroll
    for (int x = 0; x < 1024 / kUThreads; ++x) {
        const int id = tid + kUThreads * x;
        const int row = id >> 3, ch = id & 7;
        const uint32_t off = mma::swz64(row, 8 * ch);
        uint4 wu = make_uint4(0, 0, 0, 0), wv = wu;
        if (i0 + row < a.L) {
            const uint4 qq = *reinterpret_cast<const uint4*>(qraw + off);
            const uint32_t qw[4] = {qq.x, qq.y, qq.z, qq.w};
            uint32_t ou[4], ov[4];
            const float c = a.scale * 1.4426950408889634f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float x0 = mma::bf16_lo(qw[e]), x1 = mma::bf16_hi(qw[e]);
                const int d = 8 * ch + 2 * e;
                ou[e] = pack_bf16x2(fmaf(x0, c, uc[d]), fmaf(x1, c, uc[d + 1]));
                ov[e] = pack_bf16x2(fmaf(x0, c, vc[d]), fmaf(x1, c, vc[d + 1]));
            }
            wu = make_uint4(ou[0], ou[1], ou[2], ou[3]);
            wv = make_uint4(ov[0], ov[1], ov[2], ov[3]);
        }
        *reinterpret_cast<uint4*>(sm + USmem::QU + off) = wu;
        *reinterpret_cast<uint4*>(sm + USmem::QV + off) = wv;
    }
}

// D_i = dO_i . out_i of every query row (four rows per warp, eight lanes per row), for the
// gradient kernel's dS = P (dP - D).
__global__ void __launch_bounds__(256) bwd_rowdot_kernel(const BwdParams p)
{
    const AttnSimtParams& a = p.a;
    const int64_t rows = static_cast<int64_t>(a.B) * a.L * a.H;
    const int64_t row = (static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x) >> 3;
    const int ch = threadIdx.x & 7;
    float acc = 0.f;
    if (row < rows) {
        const int h = static_cast<int>(row % a.H);
        const int64_t bi = row / a.H;
        const int i = static_cast<int>(bi % a.L), b = static_cast<int>(bi / a.L);
        const uint4 g = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.dout) + b * p.g_sb +
                                                             static_cast<int64_t>(i) * p.g_st + h * p.g_sh) + ch);
        const uint4 o = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.out) + b * a.o_sb +
                                                             static_cast<int64_t>(i) * a.o_st + h * a.o_sh) + ch);
        const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            acc = fmaf(mma::bf16_lo(gw[e]), mma::bf16_lo(ow[e]), acc);
            acc = fmaf(mma::bf16_hi(gw[e]), mma::bf16_hi(ow[e]), acc);
        }
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    if (row < rows && ch == 0) p.dd[row] = acc;
}

// D_i and the log-sum-exp of query row i of (b, h) (zero past L).
__device__ __forceinline__ void row_stats(const BwdParams& p, int b, int h, int i, float& dd, float& l2)
{
    const AttnSimtParams& a = p.a;
    dd = 0.f;
    l2 = 0.f;
    if (i >= a.L) return;
    const int64_t row = (static_cast<int64_t>(b) * a.L + i) * a.H + h;
    dd = __ldg(p.dd + row);
    l2 = __ldg(p.lse + row);
}

// Byte offset of G[li][c] (window column c of query row li): four K-major swizzle atoms of 64
// columns.
__device__ __forceinline__ uint32_t g_off(int li, int c)
{
    return static_cast<uint32_t>((c >> 6) * kTileBytes + li * 128 + (((((c >> 3) & 7) ^ li) & 7) << 4) + ((c & 7) << 1));
}

// Add 128 staged dr rows (fp32, kDrPitch bytes apart in X) to dr rows delta0 .. delta0 + 127 of
// head h, skipping distances outside [0, min(clamp_len, n_rows)): warp w takes rows w, w + 16, ...
__device__ __forceinline__ void flush_dr_rows(const BwdParams& p, const uint8_t* sm, int h, int delta0, int warp,
                                              int lane)
{
    const AttnSimtParams& a = p.a;
    const int lim = min(a.C, p.n_rows);
#pragma unroll
    for (int k = 0; k < 128 / (kUThreads / 32); ++k) {
        const int r = warp + (kUThreads / 32) * k;
        const int delta = delta0 + r;
        if (delta >= 0 && delta < lim) {
            const float2 v = *reinterpret_cast<const float2*>(sm + USmem::X + r * kDrPitch + 8 * lane);
            atomicAdd(reinterpret_cast<float2*>(p.dr + (static_cast<int64_t>(delta) * a.H + h) * 64 + 2 * lane), v);
        }
    }
}

__global__ void __launch_bounds__(kUThreads, 1) bwd_umma_kernel(const __grid_constant__ BwdParams p)
{
    extern __shared__ __align__(1024) uint8_t sm[];
    const AttnSimtParams& a = p.a;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int li = tid & 127, qt4 = tid >> 7;             // TMEM lane / tile row, column quarter
    if ((smem_u32(sm) & 1023u) != 0) {
        if (tid == 0 && p.err_flag) atomicCAS(p.err_flag, 0, TXL_ERR_ALIGNMENT);
        return;
    }
    const int h = blockIdx.x, b = blockIdx.y;
    const int n_qt = (a.L + 127) / 128;
    // work classes, longest first: query tiles from the last, then key tiles from the first
    const bool key_cta = static_cast<int>(blockIdx.z) >= n_qt;
    const int own = key_cta ? static_cast<int>(blockIdx.z) - n_qt : n_qt - 1 - static_cast<int>(blockIdx.z);
    const int M = a.M, L = a.L, C = a.C;
    const float c = a.scale * 1.4426950408889634f;

    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + USmem::Bar);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + USmem::Misc);
    int* abort_flag = reinterpret_cast<int*>(sm + USmem::Misc + 4);
    float* csum_s = reinterpret_cast<float*>(sm + USmem::Csum);
    uint32_t* srow = reinterpret_cast<uint32_t*>(sm + USmem::X) + li * kStagePitch;
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(bar + 1, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tmem_holder, 512);
    // set (by thread 0, only inside its bounded waits, read by all after the CTA barrier that
    // follows them) once a wait gave up: every later wait returns at once, so the sweep runs out
    // without waiting, and no result is written
    auto aborted = [&]() { return *reinterpret_cast<volatile int*>(abort_flag) != 0; };

    // sweep geometry: step t pairs query tile i0 with the key tile starting at j0 = M + i0 - 128 t
    const int n_steps = key_cta ? n_qt - own : (M + 128 * own + 127 - a.lo) / 128 + 1;
    int i0 = 128 * own;                                    // key CTA: the first query tile = own
    const int jk = M + 128 * own;                          // key CTA: its key tile
    if (tid < 64) {
        float* bias = reinterpret_cast<float*>(sm + USmem::Bias);
        bias[tid] = __ldg(a.u + h * 64 + tid) * c;
        bias[64 + tid] = __ldg(a.vb + h * 64 + tid) * c;
    }

    // step 0's operands: raw q through the K1 slot, dO, keys, position blocks 0 and 1
    load_query_raw(p, sm + USmem::K1, sm + USmem::GO, b, h, i0, tid);
    load_keys(a, sm + USmem::K0, sm + USmem::V0, b, h, key_cta ? jk : M + i0, tid);
    load_rblock(p, sm, h, 0, tid);
    load_rblock(p, sm, h, 1, tid);
    mma::cp_async_commit();
    float dd, l2;
    row_stats(p, b, h, i0 + li, dd, l2);
    mma::cp_async_wait_all();
    __syncthreads();
    convert_queries(a, sm, sm + USmem::K1, i0, tid);

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const WaitCtl wc{abort_flag, p.err_flag, kUWaitNs};
    const int sh = lane & 1;                              // stage position parity of this row
    const int wq = warp & 3;

    constexpr uint32_t id_nn = idesc_bf16(128, 128, 0, 0);   // K-major A and B
    constexpr uint32_t id_kn = idesc_bf16(128, 64, 0, 1);    // A K-major (or TMEM), B MN-major
    constexpr uint32_t id_mm = idesc_bf16(128, 64, 1, 1);    // A and B MN-major
    const uint32_t s_qu = smem_u32(sm + USmem::QU), s_qv = smem_u32(sm + USmem::QV);
    const uint32_t s_r = smem_u32(sm + USmem::R), s_x = smem_u32(sm + USmem::X);

    uint32_t mph = 0;
    bool ok = true;
    float csum = 0.f;                                     // fp32 dS of this thread's pairs at or past clamp_len
    float carry[16];                                      // upper-block dr_win of the previous tile
#pragma unroll
    for (int e = 0; e < 16; ++e) carry[e] = 0.f;

    // operand slots of step t: a query CTA's key and value tiles alternate between two slots, a key
    // CTA's dO between two; position block beta sits in R slot beta mod 3
    auto slot_k = [&](int t) { return smem_u32(sm + ((key_cta || (t & 1) == 0) ? USmem::K0 : USmem::K1)); };
    auto slot_v = [&](int t) { return smem_u32(sm + ((key_cta || (t & 1) == 0) ? USmem::V0 : USmem::V1)); };
    auto slot_go = [&](int t) { return smem_u32(sm + ((!key_cta || (t & 1) == 0) ? USmem::GO : USmem::V1)); };
    // ---- S = Qc' K^T, W = Qc'' R_win^T (two halves of 128 window rows) of step t: thread 0, once the
    //      step's operands are in shared memory and the TMEM columns are free
    auto issue_scores = [&](int t) {
        tc_fence_after();
        const uint32_t sk = slot_k(t), ra = s_r + (t % 3) * kTileBytes, rb = s_r + ((t + 1) % 3) * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint32_t acc = kk > 0 ? 1u : 0u;
            umma_ss(tmem + kColS, sdesc_k_sw128(s_qu) + 2 * kk, sdesc_k_sw128(sk) + 2 * kk, id_nn, acc);
            umma_ss(tmem + kColW, sdesc_k_sw128(s_qv) + 2 * kk, sdesc_k_sw128(ra) + 2 * kk, id_nn, acc);
            umma_ss(tmem + kColW + 128, sdesc_k_sw128(s_qv) + 2 * kk, sdesc_k_sw128(rb) + 2 * kk, id_nn, acc);
        }
        umma_commit(bar);
    };
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) issue_scores(0);

    for (int t = 0; t < n_steps; ++t) {
        const int j0 = key_cta ? jk : M + i0 - 128 * t;
        const uint32_t s_k = slot_k(t), s_v = slot_v(t), s_go = slot_go(t);
        const uint32_t s_ra = s_r + (t % 3) * kTileBytes, s_rb = s_r + ((t + 1) % 3) * kTileBytes;
        // ---- the next step's operands, into slots the step before released
        float dd_next = 0.f, l2_next = 0.f;
        if (t + 1 < n_steps) {
            if (key_cta) {
                load_query_raw(p, sm + USmem::K1, sm + ((t & 1) ? USmem::GO : USmem::V1), b, h, i0 + 128, tid);
                row_stats(p, b, h, i0 + 128 + li, dd_next, l2_next);
            } else {
                load_keys(a, sm + ((t & 1) ? USmem::K0 : USmem::K1), sm + ((t & 1) ? USmem::V0 : USmem::V1), b, h,
                          j0 - 128, tid);
            }
            load_rblock(p, sm, h, t + 2, tid);
        }
        mma::cp_async_commit();
        if (tid == 0) ok = mbar_spin(bar, mph & 1, wc, 1) && ok;
        ++mph;
        __syncthreads();
        tc_fence_after();
        // ---- W to the stage: row li keeps window columns [32 wq, 32 wq + 160) (every column its
        //      rows read) at position c - 32 wq + sh, two bf16 per word, the even position in the
        //      low half.  Quarter 0 writes span chunks 0 and 1 (words 0 .. 31), quarter q > 0 chunk
        //      q + 1 (words 16 q + 16 ..), with column 32 q + 31 of the chunk before for sh = 1.
        {
            const int q0 = qt4 == 0 ? 0 : qt4 + 1, nq = qt4 == 0 ? 2 : 1;
            float prev = 0.f;
            if (qt4 > 0) {
                uint32_t v0;
                tmem_ld1(tmem + lane_base + kColW + 32 * wq + 32 * q0 - 1, v0);
                tmem_ld_wait();
                prev = __uint_as_float(v0);
            }
#pragma unroll 1
            for (int qi = 0; qi < nq; ++qi) {
                const int q = q0 + qi;
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + kColW + 32 * wq + 32 * q, v);
                tmem_ld_wait();
                uint4* dst = reinterpret_cast<uint4*>(srow + 16 * q);
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int k = 4 * k4 + e;
                        const float lo = sh ? (k == 0 ? prev : __uint_as_float(v[2 * k - 1])) : __uint_as_float(v[2 * k]);
                        const float hi = sh ? __uint_as_float(v[2 * k]) : __uint_as_float(v[2 * k + 1]);
                        w[e] = pack_bf16x2(lo, hi);
                    }
                    dst[k4] = make_uint4(w[0], w[1], w[2], w[3]);
                }
                prev = __uint_as_float(v[31]);
            }
        }
        tc_fence_before();
        __syncthreads();
        // ---- dP = dO V^T (into W's lower half, read above)
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                umma_ss(tmem + kColDP, sdesc_k_sw128(s_go) + 2 * kk, sdesc_k_sw128(s_v) + 2 * kk, id_nn,
                        kk > 0 ? 1u : 0u);
            umma_commit(bar);
        }
        // ---- P of this thread's 32 keys jl = 32 q + k: s = S + BD, BD[k] = W[li][li + 127 - jl]
        //      from stage word (lane + sh)/2 + 63 - 16 q - m (hi half: k = 2m, lo half: k = 2m + 1)
        float pv[32];
        {
            uint32_t sv[32];
            tmem_ld32(tmem + lane_base + kColS + 32 * qt4, sv);
            tmem_ld_wait();
            const int i = i0 + li;
            const int jb = j0 + 32 * qt4;
            // visible keys: lo <= j <= M + i, j < M + L (none past L)
            const int klo = max(a.lo - jb, 0);
            const int khi = i < L ? min(min(M + i, M + L - 1) - jb, 31) : -1;
            const int wb = ((lane + sh) >> 1) + 63 - 16 * qt4;
            if (klo == 0 && khi == 31) {
                const uint64_t nl2 = f2_pack(-l2, -l2);
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const uint32_t w = srow[wb - m];
                    const uint64_t x = f2_add(f2_pack(add_bf16hi_f32(w, __uint_as_float(sv[2 * m])),
                                                      add_bf16lo_f32(w, __uint_as_float(sv[2 * m + 1]))), nl2);
                    float x0, x1;
                    f2_unpack(x, x0, x1);
                    pv[2 * m] = ex2_approx(x0);
                    pv[2 * m + 1] = ex2_approx(x1);
                }
            } else {
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const uint32_t w = srow[wb - m];
                    const float x0 = add_bf16hi_f32(w, __uint_as_float(sv[2 * m]));
                    const float x1 = add_bf16lo_f32(w, __uint_as_float(sv[2 * m + 1]));
                    pv[2 * m] = (2 * m >= klo && 2 * m <= khi) ? ex2_approx(x0 - l2) : 0.f;
                    pv[2 * m + 1] = (2 * m + 1 >= klo && 2 * m + 1 <= khi) ? ex2_approx(x1 - l2) : 0.f;
                }
            }
        }
        if (tid == 0) ok = mbar_spin(bar, mph & 1, wc, 2) && ok;
        ++mph;
        __syncthreads();
        tc_fence_after();
        // ---- dS = P (dP - D)
        float dsv[32];
        {
            uint32_t dpv[32];
            tmem_ld32(tmem + lane_base + kColDP + 32 * qt4, dpv);
            tmem_ld_wait();
            const uint64_t nd = f2_pack(-dd, -dd);
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const uint64_t x = f2_mul(f2_pack(pv[2 * m], pv[2 * m + 1]),
                                          f2_add(f2_pack(__uint_as_float(dpv[2 * m]), __uint_as_float(dpv[2 * m + 1])), nd));
                f2_unpack(x, dsv[2 * m], dsv[2 * m + 1]);
            }
        }
        // every thread is past its stage reads: X takes G (query CTA) or P and dS (key CTA)
        tc_fence_before();
        __syncthreads();
        if (!key_cta) {
            // dS (bf16 pairs) to TMEM, the A operand of dq_ac += dS K
            {
                uint32_t w[16];
#pragma unroll
                for (int m = 0; m < 16; ++m) w[m] = pack_bf16x2(dsv[2 * m], dsv[2 * m + 1]);
                tmem_st16(tmem + lane_base + kColDS + 16 * qt4, w);
            }
            // pairs at or past clamp_len (k < kc) leave G for the fp32 sum
            const int kc = 128 * t + li - 32 * qt4 - C + 1;
            if (kc > 0) {
#pragma unroll
                for (int k = 0; k < 32; ++k)
                    if (k < kc) {
                        csum += dsv[k];
                        dsv[k] = 0.f;
                    }
            }
            // row li of G is zero outside its band [li, li + 127]: quarter 3 clears the 16-byte chunks
            // below the band (up to the one holding column li), quarter 0 those above it (from the
            // one holding column li + 128), each before writing its own band columns there
            if (qt4 == 3 || qt4 == 0) {
                const int a0 = qt4 == 3 ? 0 : (li + 128) >> 3, a1 = qt4 == 3 ? (li >> 3) + 1 : 32;
                for (int ch = a0; ch < a1; ++ch)
                    *reinterpret_cast<uint4*>(sm + USmem::X + (ch >> 3) * kTileBytes + li * 128 + (((ch ^ li) & 7) << 4)) =
                        make_uint4(0, 0, 0, 0);
            }
            // G[li][c] = dS[k], c = cb - k: 32-bit words (even c, c + 1) = (dS[k], dS[k - 1]) with k
            // odd when cb is odd; when cb is even, k = 0 and k = 31 are half words (the other half
            // of each belongs to the row's neighbouring quarter or lies outside the band, already zero)
            const int cb = li + 127 - 32 * qt4;
            const int odd = cb & 1;
            const uint32_t grow = s_x + li * 128;
#pragma unroll
            for (int w = 1; w < 16; ++w) {
                const float lo = odd ? dsv[2 * w + 1] : dsv[2 * w];
                const float hi = odd ? dsv[2 * w] : dsv[2 * w - 1];
                const int cw = cb - 2 * w - odd;
                const uint32_t addr = grow + (cw >> 6) * kTileBytes + (((((cw >> 3) & 7) ^ li) & 7) << 4) + ((cw & 7) << 1);
                asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(pack_bf16x2(lo, hi)) : "memory");
            }
            if (odd) {
                const int cw = cb - 1;
                const uint32_t addr = grow + (cw >> 6) * kTileBytes + (((((cw >> 3) & 7) ^ li) & 7) << 4) + ((cw & 7) << 1);
                asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(pack_bf16x2(dsv[1], dsv[0])) : "memory");
            } else {
                sts_u16(s_x + g_off(li, cb), __bfloat16_as_ushort(__float2bfloat16_rn(dsv[0])));
                sts_u16(s_x + g_off(li, cb - 31), __bfloat16_as_ushort(__float2bfloat16_rn(dsv[31])));
            }
            tmem_st_wait();
        } else {
            // P and dS as [query][key] rows: atom q/2 holds keys 64 (q/2) .. + 63; this quarter's
            // 32 keys are its 16-byte chunks 4 (q & 1) .. + 3
            uint8_t* prow = sm + USmem::X + (qt4 >> 1) * kTileBytes + li * 128;
            uint8_t* drow = prow + 2 * kTileBytes;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t wp[4], wd[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    wp[e] = pack_bf16x2(pv[8 * j + 2 * e], pv[8 * j + 2 * e + 1]);
                    wd[e] = pack_bf16x2(dsv[8 * j + 2 * e], dsv[8 * j + 2 * e + 1]);
                }
                const int off = (((4 * (qt4 & 1) + j) ^ li) & 7) << 4;
                *reinterpret_cast<uint4*>(prow + off) = make_uint4(wp[0], wp[1], wp[2], wp[3]);
                *reinterpret_cast<uint4*>(drow + off) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- gradient products
        if (tid == 0) {
            tc_fence_after();
            if (!key_cta) {
                // dq_ac += dS K (A: dS in TMEM, 8 columns per 16 keys; B: K as [key][d], MN-major)
                const uint64_t kd = sdesc_mn_sw128(s_k, kTileBytes);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    umma_ts(tmem + kColA0, tmem + kColDS + 8 * kk, kd + 128 * kk, id_kn, (t > 0 || kk > 0) ? 1u : 0u);
                // dq_bd += G R_win (A: G K-major over 256 window columns; B: the two R blocks as
                // [row][d], MN-major)
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) {
                    const uint64_t ad = sdesc_k_sw128(s_x + (kk >> 2) * kTileBytes) + 2 * (kk & 3);
                    const uint64_t bd = sdesc_mn_sw128(kk < 8 ? s_ra : s_rb, kTileBytes) + 128 * (kk & 7);
                    umma_ss(tmem + kColA1, ad, bd, id_kn, (t > 0 || kk > 0) ? 1u : 0u);
                }
                // dr_win = G^T Qc'' (A: G read MN-major, 128 window rows = two atoms; B: Qc''
                // as [query][d], MN-major), lower block into columns 0..63, upper into 64..127
                const uint64_t qvd = sdesc_mn_sw128(s_qv, kTileBytes);
#pragma unroll
                for (int kq = 0; kq < 8; ++kq) {
                    umma_ss(tmem + kColS, sdesc_mn_sw128(s_x, kTileBytes) + 128 * kq, qvd + 128 * kq, id_mm,
                            kq > 0 ? 1u : 0u);
                    umma_ss(tmem + kColS + 64, sdesc_mn_sw128(s_x + 2 * kTileBytes, kTileBytes) + 128 * kq,
                            qvd + 128 * kq, id_mm, kq > 0 ? 1u : 0u);
                }
            } else {
                // dv += P^T dO, dk += dS^T Qc' (A: P / dS read MN-major; B: dO / Qc' MN-major)
                const uint64_t pd = sdesc_mn_sw128(s_x, kTileBytes), dsd = sdesc_mn_sw128(s_x + 2 * kTileBytes, kTileBytes);
                const uint64_t god = sdesc_mn_sw128(s_go, kTileBytes), qud = sdesc_mn_sw128(s_qu, kTileBytes);
#pragma unroll
                for (int kq = 0; kq < 8; ++kq) {
                    const uint32_t acc = (t > 0 || kq > 0) ? 1u : 0u;
                    umma_ss(tmem + kColA0, pd + 128 * kq, god + 128 * kq, id_mm, acc);
                    umma_ss(tmem + kColA1, dsd + 128 * kq, qud + 128 * kq, id_mm, acc);
                }
            }
            umma_commit(bar);
        }
        if (tid == 0) ok = mbar_spin(bar, mph & 1, wc, 3) && ok;
        ++mph;
        __syncthreads();
        tc_fence_after();
        if (!key_cta) {
            // dr rows of block t (distances 128 t - 127 + li): this tile's lower block plus the
            // previous tile's upper block, staged as fp32 rows in X (G is no longer read), then
            // added to dr a whole row per warp instruction (lane l: dimensions 2l, 2l + 1) while the
            // next step's score products run
            uint32_t lo[16], hi[16];
            tmem_ld16(tmem + lane_base + kColS + 16 * qt4, lo);
            tmem_ld16(tmem + lane_base + kColS + 64 + 16 * qt4, hi);
            tmem_ld_wait();
            float4* st = reinterpret_cast<float4*>(sm + USmem::X + li * kDrPitch + 64 * qt4);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                st[e] = make_float4(kLn2u * (__uint_as_float(lo[4 * e]) + carry[4 * e]),
                                    kLn2u * (__uint_as_float(lo[4 * e + 1]) + carry[4 * e + 1]),
                                    kLn2u * (__uint_as_float(lo[4 * e + 2]) + carry[4 * e + 2]),
                                    kLn2u * (__uint_as_float(lo[4 * e + 3]) + carry[4 * e + 3]));
#pragma unroll
            for (int e = 0; e < 16; ++e) carry[e] = __uint_as_float(hi[e]);
        }
        if (t + 1 < n_steps) {
            mma::cp_async_wait_all();                     // the next step's operands have landed
            if (key_cta) {
                // the next query tile: its raw q in the K1 slot, its dO in the other dO slot
                __syncthreads();
                i0 += 128;
                convert_queries(a, sm, sm + USmem::K1, i0, tid);
                dd = dd_next;
                l2 = l2_next;
            }
            fence_proxy_async_smem();
        }
        tc_fence_before();
        __syncthreads();
        if (tid == 0 && t + 1 < n_steps) issue_scores(t + 1);
        if (!key_cta) flush_dr_rows(p, sm, h, 128 * t - 127, warp, lane);
        tc_fence_before();
    }

    const bool failed = aborted();
    if (failed) {
        // a wait gave up: no result is written; every copy and product in flight lands first
    } else if (!key_cta) {
        // the last tile's upper block
        {
            __syncthreads();                              // the last step's staged rows are added
            float4* st = reinterpret_cast<float4*>(sm + USmem::X + li * kDrPitch + 64 * qt4);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                st[e] = make_float4(kLn2u * carry[4 * e], kLn2u * carry[4 * e + 1], kLn2u * carry[4 * e + 2],
                                    kLn2u * carry[4 * e + 3]);
            __syncthreads();
            flush_dr_rows(p, sm, h, 128 * n_steps - 127, warp, lane);
        }
        // the clamped pairs: c_i r[C] into dq_bd, ln 2 sum_i c_i Qc''_i into dr[C]
        csum_s[qt4 * 128 + li] = csum;
        __syncthreads();
        const float crow = csum_s[li] + csum_s[128 + li] + csum_s[256 + li] + csum_s[384 + li];
        uint32_t qa[16], qb[16];
        tmem_ld16(tmem + lane_base + kColA0 + 16 * qt4, qa);
        tmem_ld16(tmem + lane_base + kColA1 + 16 * qt4, qb);
        tmem_ld_wait();
        const bool clamped = C < p.n_rows;                // else no distance reaches clamp_len
        if (clamped) {
            const __nv_bfloat16* rc =
                static_cast<const __nv_bfloat16*>(a.r) + static_cast<int64_t>(C) * a.r_row + h * a.r_head + 16 * qt4;
            const uint8_t* qvrow = sm + USmem::QV + li * 128;
            float* dst = p.dr + (static_cast<int64_t>(C) * a.H + h) * 64 + 16 * qt4;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                qb[e] = __float_as_uint(__uint_as_float(qb[e]) + crow * __bfloat162float(rc[e]));
                const int d = 16 * qt4 + e;
                const uint16_t qbits =
                    *reinterpret_cast<const uint16_t*>(qvrow + ((((d >> 3) ^ li) & 7) << 4) + ((d & 7) << 1));
                float part = crow * __uint_as_float(static_cast<uint32_t>(qbits) << 16);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
                if (lane == 0) atomicAdd(dst + e, kLn2u * part);
            }
        }
        // dq; du (sum of the dq_ac rows) and dv_bias (sum of the dq_bd rows) over this tile's queries
        const int i = i0 + li;
        const float scale = a.scale;
        float part[32];                                   // scale dq_ac, then scale dq_bd, of this row
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            part[e] = i < L ? scale * __uint_as_float(qa[e]) : 0.f;
            part[16 + e] = i < L ? scale * __uint_as_float(qb[e]) : 0.f;
        }
        if (i < L) {
            const int64_t row = ((static_cast<int64_t>(b) * L + i) * a.H + h) * 64 + 16 * qt4;
#pragma unroll
            for (int e = 0; e < 16; e += 4)
                *reinterpret_cast<float4*>(p.dq + row + e) =
                    make_float4(part[e] + part[16 + e], part[e + 1] + part[17 + e], part[e + 2] + part[18 + e],
                                part[e + 3] + part[19 + e]);
        }
        // the warp's 32 rows summed by a transposing butterfly (lane l ends with the sum of value l),
        // then the four warps of each column quarter through shared memory
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const bool up = (lane & o) != 0;
#pragma unroll
            for (int k = 0; k < o; ++k) {
                const float keep = up ? part[k + o] : part[k];
                const float send = up ? part[k] : part[k + o];
                part[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
        }
        __syncthreads();                                  // X's dr rows have been added
        float* red = reinterpret_cast<float*>(sm + USmem::X);    // [quarter][lane quarter][32]
        red[(qt4 * 4 + (warp & 3)) * 32 + lane] = part[0];
        __syncthreads();
        if (tid < 128) {
            const int q = tid >> 5, v = tid & 31;
            const float sum = red[(q * 4) * 32 + v] + red[(q * 4 + 1) * 32 + v] + red[(q * 4 + 2) * 32 + v] +
                              red[(q * 4 + 3) * 32 + v];
            float* dst = v < 16 ? p.du : p.dvb;
            atomicAdd(dst + h * 64 + 16 * q + (v & 15), sum);
        }
    } else {
        // dv and dk of the owned keys (TMEM lane li = key jk + li)
        uint32_t va[16], ka[16];
        tmem_ld16(tmem + lane_base + kColA0 + 16 * qt4, va);
        tmem_ld16(tmem + lane_base + kColA1 + 16 * qt4, ka);
        tmem_ld_wait();
        const int jt = 128 * own + li;                    // key index inside the current segment
        if (jt < L) {
            const int64_t row = ((static_cast<int64_t>(b) * L + jt) * a.H + h) * 64 + 16 * qt4;
#pragma unroll
            for (int e = 0; e < 16; e += 4) {
                *reinterpret_cast<float4*>(p.dv + row + e) =
                    make_float4(__uint_as_float(va[e]), __uint_as_float(va[e + 1]), __uint_as_float(va[e + 2]),
                                __uint_as_float(va[e + 3]));
                *reinterpret_cast<float4*>(p.dk + row + e) =
                    make_float4(kLn2u * __uint_as_float(ka[e]), kLn2u * __uint_as_float(ka[e + 1]),
                                kLn2u * __uint_as_float(ka[e + 2]), kLn2u * __uint_as_float(ka[e + 3]));
            }
        }
    }
    (void)ok;
    mma::cp_async_wait_all();
    if (failed && tid == 0) {
        int never = 0;
        const WaitCtl dw{&never, nullptr, 100000000ull};
        umma_commit(bar + 1);                             // arrives once every issued MMA is complete
        (void)mbar_wait(bar + 1, 0, dw, 9);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

inline bool al16u(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }
inline bool st8u(int64_t s) { return (s & 7) == 0; }

}  // namespace

bool bwd_umma_eligible(const BwdParams& p, txl_dtype dtype)
{
    const AttnSimtParams& a = p.a;
    if (!p.lse_given || !bwd_tc_eligible(p, dtype)) return false;
    if (2 * ((a.L + 127) / 128) > 65535) return false;
    return al16u(a.out) && st8u(a.o_sb) && st8u(a.o_st) && st8u(a.o_sh) && al16u(p.dq) && al16u(p.dk) &&
           al16u(p.dv) && al16u(p.dr);
}

// D_i of every row into the workspace (dd), then the gradient kernel: dq, dk, dv are written; dr,
// du and dv_bias must be zero on entry (atomic accumulation).
cudaError_t launch_bwd_umma(const BwdParams& p, cudaStream_t s)
{
    static bool attr_done = false;
    if (!attr_done) {
        const cudaError_t e =
            cudaFuncSetAttribute(bwd_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, USmem::Size);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    const int64_t rows = static_cast<int64_t>(p.a.B) * p.a.L * p.a.H;
    bwd_rowdot_kernel<<<static_cast<unsigned>((rows + 31) / 32), 256, 0, s>>>(p);
    const int n_qt = (p.a.L + 127) / 128;
    const dim3 grid(p.a.H, p.a.B, 2 * n_qt);
    bwd_umma_kernel<<<grid, kUThreads, USmem::Size, s>>>(p);
    return cudaGetLastError();
}

}  // namespace txl
