// txl_attn_tc.cu -- fused relative attention for sm_103a: TMA tiles, tcgen05 UMMA with TMEM
// accumulators, the relative shift as an index remap, online softmax, P.V on tensor cores.
// It serves 64 < d_head <= 128 (two 64-column atoms per row); d_head <= 64 takes the persistent
// kernel of txl_attn_persist.cu, and the one-atom branches below are kept only as that template
// parameter's other value (not instantiated).
//
// Per CTA: one tile of 128 queries of one (batch, head).  Score of query i and key j
// ("跨窗口的相对位置编码" §3, "Transformer-XL 和相对位置编码" §2.3.2 terms (a)-(d)):
//     s_ij = c * [ (q_i+u).k_j + (q_i+v).r[min(M+i-j, C)] ]        c = scale * log2(e)
// computed as two dense contractions per key tile,
//     AC = Qu K^T          Qu = bf16(c (q+u))            -> TMEM, 128 x 128 fp32
//     BD = Qv R_chunk^T    Qv = bf16(c (q+v))            -> TMEM, 128 x 128 fp32
// then mask, online softmax and O += P V (P bf16 written back into the AC columns of TMEM).
//
// Key tiles are aligned to the query tile: tile t covers keys [j0, j0+128) with
// j0 = M + i0 - 128 t, processed t = 0 (the diagonal, newest keys) upward in distance.  With this
// alignment the distances of tile t are 128t + (li - lj), so tile t needs exactly the rows
// [128(t-1), 128(t+1)) of r: the chunk of tile t-1 and one new chunk of 128 rows.  Each chunk's
// BD values are computed once by UMMA and kept per row in a shared-memory ring; the relative shift
// is then a per-row index remap (row li reads entry (li - lj) of chunk t, or 128 + li - lj of
// chunk t-1) instead of the pad-and-reshape "Relative Shift" trick the qidao123 page names.
// Distances >= clamp_len all use r[clamp_len] ("TransformerXL 相对位置编码" §2.4): one extra
// UMMA of Qv against the rows starting at clamp_len gives that per-row value; chunks that lie
// entirely beyond clamp_len are never loaded or multiplied.
//
// Softmax: two warpgroups split every 128-column tile; thread (row li, half hf) owns columns
// [64 hf, 64 hf + 64).  TMEM lane li holds query pi(li) = 2*(li mod 64) + li/64: warps of rows
// 0..63 hold even queries, rows 64..127 odd ones, so the parity of every per-row shift is
// warp-uniform and the remap needs no divergent code.  The two threads of a row exchange their
// tile maxima through shared memory at a 64-thread named barrier and keep separate partial row
// sums until the epilogue.
//
// Roles (352 threads): warps 0-7 softmax / correction / epilogue (two warpgroups), warp 8 TMA
// producer of q, K and r tiles, warp 9 TMEM owner and issuer of the S and BD products, warp 10
// TMA producer of V tiles (kept apart so that K and r prefetch is never held up behind a V slot).
// For D <= 64 warp 10 also issues P.V, so the S/BD issue of the next tile and the P.V issue of
// the current one proceed in two threads.  Every wait is bounded (2 s) and aborts the CTA
// cleanly; every softmax thread executes every named barrier of the tile loop even after an
// abort, so no warp can be left behind at a barrier.
#include <cuda_bf16.h>

#include "txl_internal.h"
#include "txl_ptx.cuh"
#include "txl_attn_common.cuh"

namespace txl {

namespace {

using namespace attn;

constexpr int kThreads = 352;
constexpr int kSoftmaxThreads = 256;
constexpr int kProducerWarp = 8;             // q, K and r tiles
constexpr int kMmaWarp = 9;
constexpr int kValueWarp = 10;               // V tiles, decoupled so K/r can run ahead
template <int NA>
struct AttnSmem {
    static constexpr int NS = (NA == 1) ? 3 : 1;    // pipeline stages for K and r tiles
    static constexpr int NV = (NA == 1) ? 2 : 1;    // pipeline stages for V tiles
    static constexpr int Qu = 0;
    static constexpr int Qv = Qu + NA * kTile;
    static constexpr int K = Qv + NA * kTile;
    static constexpr int V = K + NS * NA * kTile;
    static constexpr int R = V + NV * NA * kTile;
    static constexpr int BD = R + NS * NA * kTile;     // also the raw-Q staging area
    static constexpr int Bars = BD + kBdBytes;
    // q_full q_ready | k_full k_empty r_full r_empty (NS each) v_full v_empty (NV each) |
    // s_full[2] bd_full bd_free p_full[2] pv_done o_full drain s_free[2] drain_v
    static constexpr int NumBars = 2 + 4 * NS + 2 * NV + 12;
    static constexpr int Misc = Bars + NumBars * 8;
    static constexpr int Size = Misc + 16;
};

struct Bars {
    uint64_t *q_full, *q_ready, *k_full, *k_empty, *v_full, *v_empty, *r_full, *r_empty;
    uint64_t *s_full, *bd_full, *bd_free, *p_full, *pv_done, *o_full, *drain, *s_free, *drain_v;
};

template <int NS, int NV>
__device__ __forceinline__ Bars carve_bars(uint8_t* base)
{
    uint64_t* b = reinterpret_cast<uint64_t*>(base);
    Bars r;
    r.q_full = b; r.q_ready = b + 1;
    r.k_full = b + 2; r.k_empty = r.k_full + NS;
    r.v_full = r.k_empty + NS; r.v_empty = r.v_full + NV;
    r.r_full = r.v_empty + NV; r.r_empty = r.r_full + NS;
    r.s_full = r.r_empty + NS;
    r.bd_full = r.s_full + 2; r.bd_free = r.bd_full + 1;
    r.p_full = r.bd_free + 1;
    r.pv_done = r.p_full + 2; r.o_full = r.pv_done + 1; r.drain = r.o_full + 1;
    r.s_free = r.drain + 1;
    r.drain_v = r.s_free + 2;
    return r;
}

// Tile plan shared by every role of the CTA.
struct Plan {
    int i0, n_t, max_delta;
    bool clampc;
    __device__ bool need_chunk(int t, int C) const { return 128 * t < C; }
};

template <int NA>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(const __grid_constant__ AttnTcParams p)
{
    using S = AttnSmem<NA>;
    constexpr int NS = S::NS;
    constexpr int NV = S::NV;
    constexpr int NPV = 64 * NA;
    // D <= 64: P gets TMEM columns of its own, so the S buffers are free as soon as the softmax
    // has read them and S(t+1) can be computed while the softmax of tile t runs.  D = 128 needs
    // all 128 O columns, so P is written over the S buffer it came from.
    constexpr bool kSeparateP = (NA == 1);
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if ((smem_u32(smem) & 1023u) != 0) {
        if (tid == 0 && p.err_flag) atomicCAS(p.err_flag, 0, TXL_ERR_ALIGNMENT);
        return;
    }
    const Bars bar = carve_bars<NS, NV>(smem + S::Bars);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + S::Misc);
    int* abort_flag = reinterpret_cast<int*>(smem + S::Misc + 4);

    if (tid == 0) {
        mbar_init(bar.q_full, 1);
        mbar_init(bar.q_ready, 8);
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bar.k_full[s], 1); mbar_init(&bar.k_empty[s], 1);
            mbar_init(&bar.r_full[s], 1); mbar_init(&bar.r_empty[s], 1);
        }
        for (int s = 0; s < NV; ++s) { mbar_init(&bar.v_full[s], 1); mbar_init(&bar.v_empty[s], 1); }
        mbar_init(&bar.s_full[0], 1); mbar_init(&bar.s_full[1], 1);
        mbar_init(bar.bd_full, 1); mbar_init(bar.bd_free, 8);
        mbar_init(&bar.p_full[0], 8); mbar_init(&bar.p_full[1], 8);
        mbar_init(bar.pv_done, 1); mbar_init(bar.o_full, 1); mbar_init(bar.drain, 1);
        mbar_init(&bar.s_free[0], 8); mbar_init(&bar.s_free[1], 8);
        mbar_init(bar.drain_v, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) tmem_alloc(tmem_holder, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const WaitCtl wc{abort_flag, p.err_flag, kWaitTimeoutNs};

    const int qt = p.n_qt - 1 - static_cast<int>(blockIdx.x);     // longest tiles first
    const int h = blockIdx.y, b = blockIdx.z;
    const int M = p.M, lo = p.lo, C = p.C;
    Plan plan;
    plan.i0 = qt * 128;
    plan.n_t = (M + plan.i0 + 127 - lo) / 128 + 1;
    plan.max_delta = M + min(plan.i0 + 127, p.L - 1) - lo;
    plan.clampc = C <= plan.max_delta;
    const int n_t = plan.n_t;

    // Key tile t covers keys j0 = M + i0 - 128 t; memory keys come from the ring slot
    // (wp + j0) mod M (or j0 itself for a plain memory; a negative j0 reads TMA zero fill).
    auto key_tile = [&](int t, const CUtensorMap*& km, const CUtensorMap*& vm, int& row) {
        const int j0 = M + plan.i0 - 128 * t;
        if (j0 >= M) {
            km = &p.tm_kcur; vm = &p.tm_vcur; row = j0 - M;
            if (!in_range(row, 0, p.L, p.chk)) row = 0;
        }
        else {
            km = &p.tm_kmem; vm = &p.tm_vmem;
            row = p.wp ? static_cast<int>((static_cast<int64_t>(p.wp) + j0) % M) : j0;
            if (!in_range(row, p.wp ? 0 : -127, M, p.chk)) row = 0;
        }
    };

    if (warp == kProducerWarp) {
        // =========================================================== TMA producer: q, K, r
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_q);
            tma_prefetch_desc(&p.tm_kcur);
            tma_prefetch_desc(&p.tm_r);
            if (M > 0) tma_prefetch_desc(&p.tm_kmem);
            uint8_t* staging = smem + S::BD;
            mbar_expect_tx(bar.q_full, NA * kTile);
            for (int a = 0; a < NA; ++a)
                tma_load_4d(staging + a * kTile, &p.tm_q, 64 * a, h, plan.i0, b, bar.q_full);
            int rs = 0, kc = 0;                       // loads issued per pipeline
            bool ok = true;
            auto load_r = [&](int row0) -> bool {
                const int s = rs % NS;
                if (!mbar_wait(&bar.r_empty[s], ((rs / NS) & 1) ^ 1, wc, 10)) return false;
                mbar_expect_tx(&bar.r_full[s], NA * kTile);
                for (int a = 0; a < NA; ++a)
                    tma_load_3d(smem + S::R + (s * NA + a) * kTile, &p.tm_r, 64 * a, h, row0,
                                &bar.r_full[s]);
                ++rs;
                return true;
            };
            if (plan.clampc) ok = load_r(C);
            for (int t = 0; t < n_t && ok; ++t) {
                if (plan.need_chunk(t, C)) { ok = load_r(128 * t); if (!ok) break; }
                const CUtensorMap* km;
                const CUtensorMap* vm;
                int row;
                key_tile(t, km, vm, row);
                const int s = t % NS;
                if (!(ok = mbar_wait(&bar.k_empty[s], ((t / NS) & 1) ^ 1, wc, 11))) break;
                mbar_expect_tx(&bar.k_full[s], NA * kTile);
                for (int a = 0; a < NA; ++a)
                    tma_load_4d(smem + S::K + (s * NA + a) * kTile, km, 64 * a, h, row, b, &bar.k_full[s]);
                ++kc;
            }
            if (*abort_flag) {
                // wait (bounded) for the loads already issued, so that no TMA write lands in
                // shared memory after this CTA has exited
                int never = 0;
                const WaitCtl dw{&never, nullptr, 100000000ull};
                (void)mbar_wait(bar.q_full, 0, dw, 13);
                for (int x = rs - NS; x < rs; ++x)
                    if (x >= 0) (void)mbar_wait(&bar.r_full[x % NS], (x / NS) & 1, dw, 14);
                for (int x = kc - NS; x < kc; ++x)
                    if (x >= 0) (void)mbar_wait(&bar.k_full[x % NS], (x / NS) & 1, dw, 15);
            }
        }
    } else if (warp == kValueWarp) {
        // =========================================================== TMA producer: V (+ P.V)
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_vcur);
            if (M > 0) tma_prefetch_desc(&p.tm_vmem);
            int vc = 0;
            auto load_v = [&](int t) -> bool {
                const CUtensorMap* km;
                const CUtensorMap* vm;
                int row;
                key_tile(t, km, vm, row);
                const int s = t % NV;
                if (!mbar_wait(&bar.v_empty[s], ((t / NV) & 1) ^ 1, wc, 12)) return false;
                mbar_expect_tx(&bar.v_full[s], NA * kTile);
                for (int a = 0; a < NA; ++a)
                    tma_load_4d(smem + S::V + (s * NA + a) * kTile, vm, 64 * a, h, row, b, &bar.v_full[s]);
                ++vc;
                return true;
            };
            if (!kSeparateP) {
                for (int t = 0; t < n_t; ++t)
                    if (!load_v(t)) break;
            } else {
                // O += P_t V_t from the P buffer, V of tile t + 1 requested before P_t is awaited
                constexpr uint32_t idesc_pv = idesc_bf16(128, NPV, 0, 1);
                const uint64_t v_d = sdesc_mn_sw128(smem_u32(smem + S::V), kTile);
                constexpr uint64_t kStage = (NA * kTile) >> 4;
                const uint32_t b_vempty = smem_u32(bar.v_empty), b_pvdone = smem_u32(bar.pv_done);
                bool ok = load_v(0);
                for (int t = 0; t < n_t && ok; ++t) {
                    if (t + 1 < n_t && !(ok = load_v(t + 1))) break;
                    const int s = t % NV;
                    if (!(ok = mbar_wait(&bar.p_full[t & 1], (t >> 1) & 1, wc, 23))) break;
                    if (!(ok = mbar_wait(&bar.v_full[s], (t / NV) & 1, wc, 24))) break;
                    tc_fence_after();
                    const uint64_t vb = v_d + kStage * s;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        umma_ts(tmem + kColO, tmem + kColP + (kk >> 2) * 32 + (kk & 3) * 8,
                                vb + kk * (2048 >> 4), idesc_pv, (t > 0 || kk > 0) ? 1u : 0u);
                    umma_commit_addr(b_vempty + 8 * s);
                    umma_commit_addr(b_pvdone);
                }
                umma_commit(ok ? bar.o_full : bar.drain_v);
                if (!ok) {
                    int never = 0;
                    const WaitCtl dw{&never, nullptr, 100000000ull};
                    (void)mbar_wait(bar.drain_v, 0, dw, 28);
                }
            }
            if (*abort_flag) {
                int never = 0;
                const WaitCtl dw{&never, nullptr, 100000000ull};
                for (int x = vc - NV; x < vc; ++x)
                    if (x >= 0) (void)mbar_wait(&bar.v_full[x % NV], (x / NV) & 1, dw, 16);
            }
        }
    } else if (warp == kMmaWarp) {
        // =========================================================== UMMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16(128, 128, 0, 0);
            constexpr uint32_t idesc_pv = idesc_bf16(128, NPV, 0, 1);
            const uint32_t qu = smem_u32(smem + S::Qu), qv = smem_u32(smem + S::Qv);
            const int ksteps = p.k_steps;
            int rs = 0, bd_uses = 0;
            bool ok = mbar_wait(bar.q_ready, 0, wc, 20);
            // Every descriptor is fixed per CTA up to a stage offset: build them once, then each
            // UMMA is one instruction plus an independent add (the start-address field counts
            // 16-byte units, so a 32-byte K step is +2 and a 16 KB atom is +1024).
            // (A fully unrolled K loop with a runtime guard around the UMMA asm gave wrong
            // results on sm_103a; the K loop stays a runtime loop.)
            constexpr int KMAX = 4 * NA;                        // k steps of a full atom set
            const uint64_t qu_d = sdesc_k_sw128(qu), qv_d = sdesc_k_sw128(qv);
            const uint64_t k_d = sdesc_k_sw128(smem_u32(smem + S::K));
            const uint64_t r_d = sdesc_k_sw128(smem_u32(smem + S::R));
            const uint64_t v_d = sdesc_mn_sw128(smem_u32(smem + S::V), kTile);
            constexpr uint64_t kStage = (NA * kTile) >> 4;      // one stage in descriptor units
            const uint32_t b_kempty = smem_u32(bar.k_empty), b_sfull = smem_u32(bar.s_full);
            const uint32_t b_rempty = smem_u32(bar.r_empty), b_bdfull = smem_u32(bar.bd_full);
            const uint32_t b_vempty = smem_u32(bar.v_empty), b_pvdone = smem_u32(bar.pv_done);
            auto mma_bd = [&]() -> bool {
                const int s = rs % NS;
                if (!mbar_wait(&bar.r_full[s], (rs / NS) & 1, wc, 21)) return false;
                if (!mbar_wait(bar.bd_free, (bd_uses & 1) ^ 1, wc, 22)) return false;
                tc_fence_after();
                const uint64_t rb = r_d + kStage * s;
#pragma unroll 1
                for (int kk = 0; kk < ksteps; ++kk) {
                    const uint64_t off = (kk >> 2) * (kTile >> 4) + (kk & 3) * 2;
                    if (kk < KMAX)
                        umma_ss(tmem + kColBD, qv_d + off, rb + off, idesc_qk, kk > 0 ? 1u : 0u);
                }
                umma_commit_addr(b_rempty + 8 * s);
                umma_commit_addr(b_bdfull);
                ++rs;
                ++bd_uses;
                return true;
            };
            // P of tile t (D = 128; for D <= 64 the V warp issues P.V from the separate P buffer,
            // keys 0-63 in its columns 0-31 and keys 64-127 in 32-63): in the S buffer of t, keys
            // 0-63 in columns 0-31 and keys 64-127 in columns 64-95 (each softmax half writes
            // inside its own S columns).
            auto mma_pv = [&](int t) -> bool {
                const int s = t % NV;
                if (!mbar_wait(&bar.p_full[t & 1], (t >> 1) & 1, wc, 23)) return false;
                if (!mbar_wait(&bar.v_full[s], (t / NV) & 1, wc, 24)) return false;
                tc_fence_after();
                const uint64_t vb = v_d + kStage * s;
                const uint32_t pcol = tmem + ((t & 1) ? kColS1 : kColS0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    umma_ts(tmem + kColO, pcol + (kk >> 2) * 64 + (kk & 3) * 8,
                            vb + kk * (2048 >> 4), idesc_pv, (t > 0 || kk > 0) ? 1u : 0u);
                umma_commit_addr(b_vempty + 8 * s);
                umma_commit_addr(b_pvdone);
                return true;
            };
            // S_t into S[t & 1]; with a separate P it waits until the softmax has read S_{t-2}
            auto mma_s = [&](int t) -> bool {
                const int s = t % NS;
                if (!mbar_wait(&bar.k_full[s], (t / NS) & 1, wc, 25)) return false;
                if (kSeparateP && !mbar_wait(&bar.s_free[t & 1], ((t >> 1) & 1) ^ 1, wc, 27)) return false;
                tc_fence_after();
                const uint64_t kb = k_d + kStage * s;
                const uint32_t scol = tmem + ((t & 1) ? kColS1 : kColS0);
#pragma unroll 1
                for (int kk = 0; kk < ksteps; ++kk) {
                    const uint64_t off = (kk >> 2) * (kTile >> 4) + (kk & 3) * 2;
                    if (kk < KMAX)
                        umma_ss(scol, qu_d + off, kb + off, idesc_qk, kk > 0 ? 1u : 0u);
                }
                umma_commit_addr(b_kempty + 8 * s);
                umma_commit_addr(b_sfull + 8 * (t & 1));
                return true;
            };
            if (ok) {
                tc_fence_after();
                if (plan.clampc) ok = mma_bd();
            }
            if (ok) ok = mma_s(0);
            if (ok && plan.need_chunk(0, C)) ok = mma_bd();
            // tile t + 1's products are issued while the softmax of tile t runs; P.V of tile t
            // (D = 128) follows once its P is in TMEM
            for (int t = 0; t < n_t && ok; ++t) {
                if (t + 1 < n_t) {
                    if (!(ok = mma_s(t + 1))) break;
                    if (plan.need_chunk(t + 1, C) && !(ok = mma_bd())) break;
                }
                if (!kSeparateP && !(ok = mma_pv(t))) break;
            }
            // every S and BD product is awaited by the softmax before the CTA ends; O is complete
            // when the issuer of P.V commits o_full
            if (!kSeparateP || !ok) umma_commit(ok ? bar.o_full : bar.drain);
            if (!ok) {
                int never = 0;
                const WaitCtl dw{&never, nullptr, 100000000ull};
                (void)mbar_wait(bar.drain, 0, dw, 26);
            }
        }
        __syncwarp();
    } else {
        // =========================================================== softmax warps 0-7
        const int hf = tid >> 7;                     // column half of every tile
        const int li = tid & 127;                    // TMEM lane == tile row
        const int pi = query_of_row(li);             // query offset inside the tile
        const int sh = (li >> 6) ? 0 : 1;            // odd queries: 0, even queries: 1
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        bool ok = true;

        // ---- prologue: Qu = c(q+u), Qv = c(q+v) in bf16, rows permuted to pi(li); each half
        // converts 4 of the 8 16-byte chunks of every 64-column atom.  u and v of this head are
        // staged in shared memory (after the raw-q staging area) while the q tile is in flight.
        float* uv = reinterpret_cast<float*>(smem + S::BD + NA * kTile);    // [2][128]
        {
            const int d = tid & 127;
            const float* src_uv = (tid < 128 ? p.u : p.vb) + static_cast<int64_t>(h) * p.D;
            uv[tid] = d < p.D ? __ldg(src_uv + d) : 0.f;
        }
        named_bar_sync(1, kSoftmaxThreads);
        ok = warp_wait(bar.q_full, 0, wc, 30);
        if (ok) {
            const uint8_t* staging = smem + S::BD;
            const int src = pi;
            const float* uh = uv;
            const float* vh = uv + 128;
#pragma unroll
            for (int a = 0; a < NA; ++a) {
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const int c = 4 * hf + c4;
                    const uint4 raw = *reinterpret_cast<const uint4*>(
                        staging + a * kTile + src * 128 + ((c ^ (src & 7)) << 4));
                    const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
                    uint32_t wu[4], wv[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int d0 = 64 * a + 8 * c + 2 * e;
                        const float q0 = __uint_as_float(rw[e] << 16);
                        const float q1 = __uint_as_float(rw[e] & 0xffff0000u);
                        const bool z0 = d0 >= p.D, z1 = d0 + 1 >= p.D;
                        const float u0 = uh[d0], u1 = uh[d0 + 1];
                        const float v0 = vh[d0], v1 = vh[d0 + 1];
                        wu[e] = pack_bf16x2(z0 ? 0.f : (q0 + u0) * p.qscale, z1 ? 0.f : (q1 + u1) * p.qscale);
                        wv[e] = pack_bf16x2(z0 ? 0.f : (q0 + v0) * p.qscale, z1 ? 0.f : (q1 + v1) * p.qscale);
                    }
                    const int off = a * kTile + li * 128 + ((c ^ (li & 7)) << 4);
                    *reinterpret_cast<uint4*>(smem + S::Qu + off) = make_uint4(wu[0], wu[1], wu[2], wu[3]);
                    *reinterpret_cast<uint4*>(smem + S::Qv + off) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            mbar_arrive_if(bar.q_ready, lane == 0);
        }
        named_bar_sync(1, kSoftmaxThreads);    // all staging reads done before the ring reuses it

        uint32_t* bdrow = reinterpret_cast<uint32_t*>(smem + S::BD) + li * kBdPitchWords;
        const uint32_t row_saddr = smem_u32(bdrow);
        float* xchg = reinterpret_cast<float*>(bdrow + 128);          // 4 exchange words per row
        const int wbase_row = (li & 63) - 32 * hf;                   // (pi + sh - 1)/2 - 32 hf
        float m_run = -INFINITY, l_half = 0.f;
        uint32_t bdc_bits = 0;                  // fp32 bits of (q+v).r[clamp_len] for this row
        int bd_uses = 0;

        // The ring starts as bf16 -inf.  The positions the diagonal tile reads for future keys
        // (lj > pi) are never written before that tile, so those keys come out masked.
        {
            uint4* w = reinterpret_cast<uint4*>(bdrow + 64 * hf);
            const uint4 ninf = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
#pragma unroll
            for (int q4 = 0; q4 < 16; ++q4) w[q4] = ninf;
        }
        pair_bar(li);

        if (plan.clampc) {
            if (ok) ok = warp_wait(bar.bd_full, bd_uses & 1, wc, 31);
            if (ok) {
                tc_fence_after();
                uint32_t v0;
                tmem_ld1(tmem + lane_base + kColBD, v0);
                tmem_ld_wait();
                bdc_bits = v0;
                tc_fence_before();
                __syncwarp();
                mbar_arrive_if(bar.bd_free, lane == 0);
            }
            ++bd_uses;
        }

        for (int t = 0; t < n_t; ++t) {
            const bool chunk = plan.need_chunk(t, C);
            // a slot whose distances all reach clamp_len holds r[clamp_len]'s value everywhere;
            // it is written once, unless two tiles ago it already held that fill
            const bool fill = plan.clampc && !chunk && (t < 2 || plan.need_chunk(t - 2, C));
            const uint32_t scol = tmem + lane_base + ((t & 1) ? kColS1 : kColS0) + 64 * hf;
            float s[64];
            if (chunk && ok) ok = warp_wait(bar.bd_full, bd_uses & 1, wc, 32);
            if (ok) ok = warp_wait(&bar.s_full[t & 1], (t >> 1) & 1, wc, 33);
            if (ok) {
                tc_fence_after();
                if (chunk || fill) {
                    // this half's chunk columns (or the clamp value) -> ring first, which keeps
                    // register use low
                    uint32_t bdv[64];
                    if (chunk) {
                        tmem_ld64(tmem + lane_base + kColBD + 64 * hf, bdv);
                        tmem_ld_wait();
                        tc_fence_before();
                        __syncwarp();
                        mbar_arrive_if(bar.bd_free, lane == 0);
                        const int cc = C - 128 * t - 64 * hf;   // first local column at the clamp
                        if (plan.clampc && cc < 64) {
#pragma unroll
                            for (int k = 0; k < 64; ++k) bdv[k] = k >= cc ? bdc_bits : bdv[k];
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < 64; ++k) bdv[k] = bdc_bits;
                    }
                    ring_write_half(bdrow, row_saddr, bdv, t, hf, sh);
                }
                uint32_t su[64];
                tmem_ld64(scol, su);
                tmem_ld_wait();
                if (kSeparateP) {                       // S buffer may now take S_{t+2}
                    tc_fence_before();
                    __syncwarp();
                    mbar_arrive_if(&bar.s_free[t & 1], lane == 0);
                }
#pragma unroll
                for (int k = 0; k < 64; ++k) s[k] = __uint_as_float(su[k]);
            }
            if (chunk) ++bd_uses;
            if (chunk || fill) pair_bar(li);            // both halves of the slot are in the ring
            const int j0 = M + plan.i0 - 128 * t;
            const int lm = lo - j0;                     // keys lj < lm precede the valid memory
            const int wbase = 64 * (t & 1) + wbase_row;
            if (ok && lm > 0) {
                // only the last (oldest) tile can start before the valid memory: its invalid keys
                // read -inf; each thread writes exactly the positions it reads itself
                const int hi_lj = min(lm, 64 * hf + 64);
#pragma unroll 1
                for (int lj = 64 * hf; lj < hi_lj; ++lj)
                    sts_u16(row_saddr + 2u * ((128 * (t & 1) + pi - lj + sh) & 255), 0xFF80);
            }
            float mloc = -INFINITY;
            if (ok) {
                mloc = logits_interior(s, bdrow, wbase);
                xchg[2 * (t & 1) + hf] = mloc;
            }
            pair_bar(li);                               // exchange the two halves' maxima
            if (ok) {
                const float mt = fmaxf(mloc, xchg[2 * (t & 1) + (hf ^ 1)]);
                float alpha = 1.f;
                bool rescale_o = false;
                if (t == 0) {
                    m_run = mt;
                } else if (mt > m_run + kRescaleThreshold) {
                    alpha = ex2_approx(m_run - mt);
                    m_run = mt;
                    rescale_o = true;
                }
                const uint64_t negm = f2_pack(-m_run, -m_run);
                uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0;
                uint32_t pw[32];
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    float y0, y1;
                    f2_unpack(f2_add(f2_pack(s[2 * k], s[2 * k + 1]), negm), y0, y1);
                    const float p0 = ex2_approx(y0), p1 = ex2_approx(y1);
                    if (k & 1) acc1 = f2_add(acc1, f2_pack(p0, p1));
                    else acc0 = f2_add(acc0, f2_pack(p0, p1));
                    pw[k] = pack_bf16x2(p0, p1);
                }
                float a0, a1, b0, b1;
                f2_unpack(acc0, a0, a1);
                f2_unpack(acc1, b0, b1);
                l_half = fmaf(l_half, alpha, (a0 + a1) + (b0 + b1));
                // P.V of the previous tile must be complete before its P buffer (separate P) or
                // O (rescale) is touched
                const bool rescale_any = t >= 1 && __any_sync(0xffffffffu, rescale_o);
                if (t >= 1 && (kSeparateP || rescale_any)) {
                    ok = warp_wait(bar.pv_done, (t - 1) & 1, wc, 34);
                    if (ok) tc_fence_after();
                }
                if (ok) {
                    // P (bf16): keys 64hf.. at column 32hf of the P buffer, or at column 64hf of
                    // this tile's S buffer
                    tmem_st32(kSeparateP ? tmem + lane_base + kColP + 32 * hf : scol, pw);
                }
                if (ok && rescale_any) {
                    const uint64_t al2 = f2_pack(alpha, alpha);
#pragma unroll 1
                    for (int cb = 0; cb < NPV / 64; ++cb) {
                        uint32_t o[32];
                        const uint32_t oaddr = tmem + lane_base + kColO + (NPV / 2) * hf + 32 * cb;
                        tmem_ld32(oaddr, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            float x0, x1;
                            f2_unpack(f2_mul(f2_pack(__uint_as_float(o[2 * k]), __uint_as_float(o[2 * k + 1])), al2),
                                      x0, x1);
                            o[2 * k] = __float_as_uint(x0);
                            o[2 * k + 1] = __float_as_uint(x1);
                        }
                        tmem_st32(oaddr, o);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                mbar_arrive_if(&bar.p_full[t & 1], lane == 0 && ok);
            }
        }

        // ---- epilogue: O / (l_0 + l_1) -> bf16 -> out[b, i0 + pi, h, :]; each half stores half
        // of the columns
        if (ok) ok = warp_wait(bar.o_full, 0, wc, 35);
        xchg[2 * (n_t & 1) + hf] = l_half;
        pair_bar(li);
        if (ok) {
            tc_fence_after();
            const float l_row = l_half + xchg[2 * (n_t & 1) + (hf ^ 1)];
            const int i = plan.i0 + pi;
            const float inv_l = 1.f / l_row;
            __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) + b * p.o_sb +
                                  static_cast<int64_t>(i) * p.o_st + h * p.o_sh;
            const bool vec = p.out_vec != 0;
#pragma unroll 1
            for (int cb = 0; cb < NPV / 64; ++cb) {
                uint32_t o[32];
                const int d0 = (NPV / 2) * hf + 32 * cb;
                tmem_ld32(tmem + lane_base + kColO + d0, o);
                tmem_ld_wait();
                if (i >= p.L) continue;
                if (vec && d0 + 32 <= p.D) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w[e] = pack_bf16x2(__uint_as_float(o[8 * q4 + 2 * e]) * inv_l,
                                               __uint_as_float(o[8 * q4 + 2 * e + 1]) * inv_l);
                        *reinterpret_cast<uint4*>(orow + d0 + 8 * q4) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                } else {
                    for (int k = 0; k < 32 && d0 + k < p.D; ++k)
                        orow[d0 + k] = __float2bfloat16_rn(__uint_as_float(o[k]) * inv_l);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int NA>
cudaError_t launch_na(const AttnTcParams& p, cudaStream_t s)
{
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<NA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             AttnSmem<NA>::Size);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    dim3 grid(p.n_qt, p.H, p.B);
    attn_tc_kernel<NA><<<grid, kThreads, AttnSmem<NA>::Size, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

// 64 < d_head <= 128 (two 64-column atoms).  d_head <= 64 takes the persistent kernel
// (txl_attn_persist.cu); the one-atom form of this kernel is not instantiated.
cudaError_t launch_attn_tc(const AttnTcParams& p, cudaStream_t s)
{
    if (p.B == 0 || p.L == 0 || p.H == 0) return cudaSuccess;
    if (p.n_atoms != 2) return cudaErrorInvalidValue;
    return launch_na<2>(p, s);
}

}  // namespace txl
