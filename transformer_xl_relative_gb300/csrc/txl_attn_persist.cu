// txl_attn_persist.cu -- persistent fused relative attention for d_head <= 64 on sm_103a.
//
// Same arithmetic as the one-CTA-per-query-tile kernel (txl_attn_tc.cu): per key tile
//     AC = Qu K^T,  BD = Qv R_chunk^T   (tcgen05, fp32 in TMEM),  Qu = bf16(c(q+u)), Qv = bf16(c(q+v))
// ("跨窗口的相对位置编码" §3; "Transformer-XL 和相对位置编码" §2.3.2 terms (a)-(d)), the relative
// shift as a per-row index remap through a shared-memory ring of BD values, the clamp of
// distances at clamp_len ("TransformerXL 相对位置编码" §2.4), the causal-with-memory mask, an
// online softmax in the log2 domain and O += P V on the tensor cores.
//
// What differs is the schedule.  One CTA per SM loops over work items (b, h, query tile), longest
// first, in serpentine rounds (round n gives CTA c item n G + c for even n and n G + G - 1 - c for
// odd n).  Every pipeline (K, r and V stages, the two S buffers, the BD buffer, the P buffer)
// keeps one counter across items, so the TMA producer, the UMMA issuers and the q converter start
// on item n + 1 while the softmax warps finish item n: the q load, the Qu/Qv conversion and the
// first S and BD products of an item hide behind the last tiles and the epilogue of the one
// before, and no CTA launch separates them.
//
// The same kernel also serves the learned-table variant ("TransformerXL 相对位置编码" §3.1, the index
// of §2): attn_persist_kernel<true> attends bidirectionally over the current sequence, reads the
// position vector of pair (i, j) from table row i - j + max_len - 1 (every row of the sequence's
// pairs exists when L <= max_len, so nothing clamps) and scales only the q terms: Qu = bf16(log2 e
// (scale q + u)), Qv = bf16(log2 e (scale q + v)).  Its key tiles run from the sequence's last to its
// first, so that the distance grows with the tile index as it does with memory, and one extra BD
// chunk (the distances just below the first tile's) precedes every item.
//
// Roles (384 threads): warps 0-7 softmax / correction / epilogue (two warpgroups splitting each
// tile's columns), warp 8 TMA producer of raw q, K and r tiles, warp 9 TMEM owner and issuer of
// S and BD, warp 10 TMA producer of V tiles and issuer of P.V, warp 11 converter of raw q into
// Qu and Qv.  Every wait is bounded (2 s); an abort drains every role and every softmax thread
// still executes every named barrier of the loops.
#include <cuda_bf16.h>

#include "txl_internal.h"
#include "txl_ptx.cuh"
#include "txl_attn_common.cuh"

namespace txl {

namespace {

using namespace attn;

constexpr int kPThreads = 384;
constexpr int kPProducerWarp = 8;
constexpr int kPMmaWarp = 9;
constexpr int kPValueWarp = 10;
constexpr int kPConvWarp = 11;
constexpr int kNK = 2;                      // K stages
constexpr int kNR = 2;                      // r stages
constexpr int kNV = 2;                      // V stages

struct PSmem {
    // two (Qu, Qv) buffers: item n uses buffer n mod 2; raw q lands in its Qu slot and is
    // converted in place while the item before is still being computed
    static constexpr int Q = 0;                          // Qu0 Qv0 Qu1 Qv1
    static constexpr int K = Q + 4 * kTile;
    static constexpr int R = K + kNK * kTile;
    static constexpr int V = R + kNR * kTile;
    static constexpr int BD = V + kNV * kTile;
    static constexpr int Bars = BD + kBdBytes;
    // qraw_full[2] q_ready[2] q_free[2] | k_full/k_empty (kNK each) r_full/r_empty (kNR each)
    // v_full/v_empty (kNV each) | s_full[2] s_free[2] bd_full bd_free p_full[2] pv_done o_full
    // o_free drain drain_v
    static constexpr int NumBars = 6 + 2 * (kNK + kNR + kNV) + 13;
    __device__ static constexpr int qu(int qb) { return Q + 2 * qb * kTile; }
    __device__ static constexpr int qv(int qb) { return Q + (2 * qb + 1) * kTile; }
    static constexpr int Misc = Bars + NumBars * 8;
    static constexpr int Sched = Misc + 16;             // int first[32], int count[32]
    static constexpr int Size = Sched + 2 * kMaxSchedClasses * 4;
};

struct PBars {
    uint64_t *qraw_full, *q_ready, *q_free;              // two each, one per (Qu, Qv) buffer
    uint64_t *k_full, *k_empty, *r_full, *r_empty, *v_full, *v_empty;
    uint64_t *s_full, *s_free, *bd_full, *bd_free, *p_full, *pv_done, *o_full, *o_free, *drain, *drain_v;
};

__device__ __forceinline__ PBars carve_pbars(uint8_t* base)
{
    uint64_t* b = reinterpret_cast<uint64_t*>(base);
    PBars r;
    r.qraw_full = b; r.q_ready = b + 2; r.q_free = b + 4;
    r.k_full = b + 6; r.k_empty = r.k_full + kNK;
    r.r_full = r.k_empty + kNK; r.r_empty = r.r_full + kNR;
    r.v_full = r.r_empty + kNR; r.v_empty = r.v_full + kNV;
    r.s_full = r.v_empty + kNV; r.s_free = r.s_full + 2;
    r.bd_full = r.s_free + 2; r.bd_free = r.bd_full + 1;
    r.p_full = r.bd_free + 1; r.pv_done = r.p_full + 2;
    r.o_full = r.pv_done + 1; r.o_free = r.o_full + 1;
    r.drain = r.o_free + 1; r.drain_v = r.drain + 1;
    return r;
}

// One work item: query tile qt of head h of batch entry b, with its key-tile plan.
struct Item {
    int b, h, i0, n_t;
    bool clampc;             // some distance of the item reaches clamp_len
};

// The n-th item of this CTA (false once the CTA has none left), longest first.  With a count table
// (sched_mode 1) the CTA takes count[qt] items of each query tile qt, items first[qt] .. of that
// tile's (b, h) list (first/count: this CTA's row of the table and its prefix sums, in shared
// memory).  Otherwise items are numbered longest first (every (b, h) of qt = n_qt - 1, then of
// qt = n_qt - 2, ...) and dealt in serpentine rounds.
template <bool kTab>
__device__ __forceinline__ bool item_at(const AttnTcParams& p, const int* first, const int* count, int n, Item& it)
{
    int qt, rem;
    if (p.sched_mode) {
        qt = p.n_qt - 1;
        while (qt >= 0 && n >= count[qt]) {
            n -= count[qt];
            --qt;
        }
        if (qt < 0) return false;
        rem = first[qt] + n;
    } else {
        const int G = gridDim.x, c = blockIdx.x;
        const int64_t per_qt = static_cast<int64_t>(p.H) * p.B;
        const int64_t idx = static_cast<int64_t>(n) * G + ((n & 1) ? (G - 1 - c) : c);
        if (idx >= per_qt * p.n_qt) return false;
        const int64_t g = idx / per_qt;
        rem = static_cast<int>(idx - g * per_qt);
        qt = p.n_qt - 1 - static_cast<int>(g);
    }
    it.h = rem % p.H;
    it.b = rem / p.H;
    it.i0 = qt * 128;
    if constexpr (kTab) {
        it.n_t = p.n_qt;                     // every key tile of the sequence
        it.clampc = true;                    // one extra BD chunk precedes the tiles (chunk -1)
    } else {
        it.n_t = (p.M + it.i0 + 127 - p.lo) / 128 + 1;
        const int max_delta = p.M + min(it.i0 + 127, p.L - 1) - p.lo;
        it.clampc = p.C <= max_delta;
    }
    return true;
}

__device__ __forceinline__ bool need_chunk(int t, int C) { return 128 * t < C; }

// Key tile t of an item covers keys j0 = M + i0 - 128 t; memory keys come from the ring slot
// (wp + j0) mod slots (or j0 itself for a plain memory; a negative j0 reads TMA zero fill), and so
// do the current segment's keys when the whole sequence lives in the ring (ring_all).
// In learned-table mode tile t covers keys 128 (n_qt - 1 - t) ..: the last key tile first, so that
// the distances i - j grow with t as they do with memory.
template <bool kTab>
__device__ __forceinline__ void key_tile(const AttnTcParams& p, const Item& it, int t, bool values,
                                         const CUtensorMap*& map, int& row)
{
    if constexpr (kTab) {
        map = values ? &p.tm_vcur : &p.tm_kcur;
        row = 128 * (p.n_qt - 1 - t);
        if (!in_range(row, 0, p.L, p.chk)) row = 0;
        return;
    }
    const int j0 = p.M + it.i0 - 128 * t;
    if (j0 >= p.M && !p.ring_all) {
        map = values ? &p.tm_vcur : &p.tm_kcur;
        row = j0 - p.M;
        if (!in_range(row, 0, p.L, p.chk)) row = 0;
    } else {
        map = values ? &p.tm_vmem : &p.tm_kmem;
        if (p.wp || p.ring_all) {
            row = static_cast<int>((static_cast<int64_t>(p.wp) + j0) % p.slots);
            if (!in_range(row, 0, p.slots, p.chk)) row = 0;
        } else {
            row = j0;                                   // a plain memory: rows before 0 read zero fill
            if (!in_range(row, -127, p.M, p.chk)) row = 0;
        }
    }
}

// kMask (learned-table mode with a key mask): keys whose mask byte is 0 read a score of about -1e30
// from the ring (bf16 0xF14A); added to any finite logit it stays exactly that value, so such keys
// get weight 0 beside any unmasked key, and a row whose keys are all masked weighs them equally.
constexpr uint16_t kMaskedKeyBf16 = 0xF14A;

// kLse = 1: the row statistics alone (log-sum-exp for the gradient kernels): no output is written.
// kLse = 2: the forward output and, besides it, every row's log-sum-exp.
template <bool kTab, bool kMask = false, int kLse = 0>
__global__ void __launch_bounds__(kPThreads, 1) attn_persist_kernel(const __grid_constant__ AttnTcParams p)
{
    constexpr int NPV = 64;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    pdl_launch_dependents();
    if ((smem_u32(smem) & 1023u) != 0) {
        pdl_wait();
        if (tid == 0 && p.err_flag) atomicCAS(p.err_flag, 0, TXL_ERR_ALIGNMENT);
        return;
    }
    const PBars bar = carve_pbars(smem + PSmem::Bars);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + PSmem::Misc);
    int* abort_flag = reinterpret_cast<int*>(smem + PSmem::Misc + 4);

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar.qraw_full[s], 1); mbar_init(&bar.q_ready[s], 1); mbar_init(&bar.q_free[s], 1);
        }
        for (int s = 0; s < kNK; ++s) { mbar_init(&bar.k_full[s], 1); mbar_init(&bar.k_empty[s], 1); }
        for (int s = 0; s < kNR; ++s) { mbar_init(&bar.r_full[s], 1); mbar_init(&bar.r_empty[s], 1); }
        for (int s = 0; s < kNV; ++s) { mbar_init(&bar.v_full[s], 1); mbar_init(&bar.v_empty[s], 1); }
        mbar_init(&bar.s_full[0], 1); mbar_init(&bar.s_full[1], 1);
        mbar_init(&bar.s_free[0], 8); mbar_init(&bar.s_free[1], 8);
        mbar_init(bar.bd_full, 1); mbar_init(bar.bd_free, 8);
        mbar_init(&bar.p_full[0], 8); mbar_init(&bar.p_full[1], 8);
        mbar_init(bar.pv_done, 1); mbar_init(bar.o_full, 1); mbar_init(bar.o_free, 8);
        mbar_init(bar.drain, 1); mbar_init(bar.drain_v, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    int* sched_first = reinterpret_cast<int*>(smem + PSmem::Sched);
    int* sched_count = sched_first + kMaxSchedClasses;
    if (p.sched_mode) {
        // this CTA's row of the count table and its prefix sums over the CTAs before it: one warp
        // per query-tile class, lanes striding over the CTAs
        for (int q = warp; q < p.n_qt; q += kPThreads / 32) {
            int f = 0;
            for (int c = lane; c < static_cast<int>(blockIdx.x); c += 32) f += p.sched_counts[c * p.n_qt + q];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) f += __shfl_xor_sync(0xffffffffu, f, o);
            if (lane == 0) {
                sched_first[q] = f;
                sched_count[q] = p.sched_counts[blockIdx.x * p.n_qt + q];
            }
        }
    }
    // the tensor maps are kernel parameters, valid before the previous grid ends: start fetching
    // them now so that the first loads do not wait for them
    if (warp == kPProducerWarp && lane == 0) {
        tma_prefetch_desc(&p.tm_qe);
        tma_prefetch_desc(&p.tm_qo);
        tma_prefetch_desc(&p.tm_kcur);
        tma_prefetch_desc(&p.tm_r);
        if (p.M > 0) tma_prefetch_desc(&p.tm_kmem);
    } else if (warp == kPValueWarp && lane == 0) {
        tma_prefetch_desc(&p.tm_vcur);
        if (p.M > 0) tma_prefetch_desc(&p.tm_vmem);
    }
    if (warp == kPMmaWarp) tmem_alloc(tmem_holder, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // inputs (q, k, v, r, the memory) may come from the previous grid, which may also still read
    // the output buffer: no global access before this point
    pdl_wait();
    const uint32_t tmem = *tmem_holder;
    const WaitCtl wc{abort_flag, p.err_flag, kWaitTimeoutNs};
    const int C = p.C;
    // bounded waits for work already in flight when an abort drains a role
    int never = 0;
    const WaitCtl dw{&never, nullptr, 100000000ull};

    if (warp == kPProducerWarp) {
        // =========================================================== TMA producer: raw q, K, r
        if (lane == 0) {
            int nq = 0, rc = 0, kc = 0;               // loads issued per pipeline
            bool ok = true;
            auto load_r = [&](int row0, int h) -> bool {
                const int s = rc % kNR;
                if (!mbar_wait(&bar.r_empty[s], ((rc / kNR) & 1) ^ 1, wc, 10)) return false;
                mbar_expect_tx(&bar.r_full[s], kTile);
                tma_load_3d(smem + PSmem::R + s * kTile, &p.tm_r, 0, h, row0, &bar.r_full[s]);
                ++rc;
                return true;
            };
            Item it;
            for (int n = 0; ok && item_at<kTab>(p, sched_first, sched_count, n, it); ++n) {
                // raw q rows in TMEM-lane order: even queries of the tile to rows 0-63, odd
                // queries to rows 64-127 (the even and odd row maps both step two tokens per row)
                const int qb = n & 1;
                if (!(ok = mbar_wait(&bar.q_free[qb], ((n >> 1) & 1) ^ 1, wc, 11))) break;
                mbar_expect_tx(&bar.qraw_full[qb], kTile);
                tma_load_4d(smem + PSmem::qu(qb), &p.tm_qe, 0, it.h, it.i0 >> 1, it.b, &bar.qraw_full[qb]);
                tma_load_4d(smem + PSmem::qu(qb) + kTile / 2, &p.tm_qo, 0, it.h, it.i0 >> 1, it.b,
                            &bar.qraw_full[qb]);
                ++nq;
                // r row of chunk t's first distance: 128 t (learned table: 128 t + roff of the item)
                const int roff = kTab ? p.roff + it.i0 - 128 * (p.n_qt - 1) : 0;
                if (it.clampc && !(ok = load_r(kTab ? roff - 128 : C, it.h))) break;
                for (int t = 0; t < it.n_t; ++t) {
                    if (need_chunk(t, C) && !(ok = load_r(128 * t + roff, it.h))) break;
                    const CUtensorMap* km;
                    int row;
                    key_tile<kTab>(p, it, t, false, km, row);
                    const int s = kc % kNK;
                    if (!(ok = mbar_wait(&bar.k_empty[s], ((kc / kNK) & 1) ^ 1, wc, 12))) break;
                    mbar_expect_tx(&bar.k_full[s], kTile);
                    tma_load_4d(smem + PSmem::K + s * kTile, km, 0, it.h, row, it.b, &bar.k_full[s]);
                    ++kc;
                }
            }
            if (*abort_flag) {
                // no TMA write may land in shared memory after the CTA has exited
                for (int x = nq - 2; x < nq; ++x)
                    if (x >= 0) (void)mbar_wait(&bar.qraw_full[x & 1], (x >> 1) & 1, dw, 13);
                for (int x = rc - kNR; x < rc; ++x)
                    if (x >= 0) (void)mbar_wait(&bar.r_full[x % kNR], (x / kNR) & 1, dw, 14);
                for (int x = kc - kNK; x < kc; ++x)
                    if (x >= 0) (void)mbar_wait(&bar.k_full[x % kNK], (x / kNK) & 1, dw, 15);
            }
        }
    } else if (warp == kPConvWarp) {
        // =========================================================== raw q -> Qu, Qv (in place)
        // Lane l converts 16-byte chunk c = l mod 8 (dims 8c .. 8c+7) of rows l/8 + 4k, k = 0..31:
        // Qu = c(q + u) and Qv = c(q + v), each as one fma of q with the pre-scaled bias.
        const int c = lane & 7;
        bool ok = true;
        Item it;
        for (int n = 0; ok && item_at<kTab>(p, sched_first, sched_count, n, it); ++n) {
            const int qb = n & 1;
            float us[8], vs[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int d = 8 * c + e;
                const bool in = d < p.D;
                const float bs = kTab ? p.bscale : p.qscale;
                us[e] = in ? __ldg(p.u + static_cast<int64_t>(it.h) * p.D + d) * bs : 0.f;
                vs[e] = in ? __ldg(p.vb + static_cast<int64_t>(it.h) * p.D + d) * bs : 0.f;
            }
            const uint64_t sc2 = f2_pack(p.qscale, p.qscale);
            if (!(ok = warp_wait(&bar.qraw_full[qb], (n >> 1) & 1, wc, 40))) break;
            uint8_t* qu = smem + PSmem::qu(qb);
            uint8_t* qv = smem + PSmem::qv(qb);
#pragma unroll 4
            for (int k = 0; k < 32; ++k) {
                const int li = (lane >> 3) + 4 * k;
                const int off = li * 128 + ((c ^ (li & 7)) << 4);
                const uint4 x = *reinterpret_cast<const uint4*>(qu + off);
                const uint32_t rw[4] = {x.x, x.y, x.z, x.w};
                uint32_t wu[4], wv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    // dims past D hold zeros in q and in the biases, so they stay zero
                    const uint64_t q2 = f2_pack(__uint_as_float(rw[e] << 16), __uint_as_float(rw[e] & 0xffff0000u));
                    float a0, a1, b0, b1;
                    f2_unpack(f2_fma(q2, sc2, f2_pack(us[2 * e], us[2 * e + 1])), a0, a1);
                    f2_unpack(f2_fma(q2, sc2, f2_pack(vs[2 * e], vs[2 * e + 1])), b0, b1);
                    wu[e] = pack_bf16x2(a0, a1);
                    wv[e] = pack_bf16x2(b0, b1);
                }
                *reinterpret_cast<uint4*>(qu + off) = make_uint4(wu[0], wu[1], wu[2], wu[3]);
                *reinterpret_cast<uint4*>(qv + off) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            mbar_arrive_if(&bar.q_ready[qb], lane == 0);
        }
    } else if (warp == kPMmaWarp) {
        // =========================================================== UMMA issuer: S and BD
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16(128, 128, 0, 0);
            const uint64_t qu_d0 = sdesc_k_sw128(smem_u32(smem + PSmem::qu(0)));
            const uint64_t qv_d0 = sdesc_k_sw128(smem_u32(smem + PSmem::qv(0)));
            constexpr uint64_t kQBuf = (2 * kTile) >> 4;           // next (Qu, Qv) buffer
            uint64_t qu_d = qu_d0, qv_d = qv_d0;
            const uint64_t k_d = sdesc_k_sw128(smem_u32(smem + PSmem::K));
            const uint64_t r_d = sdesc_k_sw128(smem_u32(smem + PSmem::R));
            constexpr uint64_t kStage = kTile >> 4;                // one stage in descriptor units
            const uint32_t b_kempty = smem_u32(bar.k_empty), b_sfull = smem_u32(bar.s_full);
            const uint32_t b_rempty = smem_u32(bar.r_empty), b_bdfull = smem_u32(bar.bd_full);
            const int ksteps = p.k_steps;
            int kc = 0, rc = 0, bd = 0, T = 0;       // K tiles, r chunks, BD products, tiles so far
            bool ok = true;
            // The K loop stays a runtime loop (a fully unrolled one with a runtime guard around
            // the UMMA asm gave wrong results on sm_103a).
            auto mma_bd = [&]() -> bool {
                const int s = rc % kNR;
                if (!mbar_wait(&bar.r_full[s], (rc / kNR) & 1, wc, 21)) return false;
                if (!mbar_wait(bar.bd_free, (bd & 1) ^ 1, wc, 22)) return false;
                tc_fence_after();
                const uint64_t rb = r_d + kStage * s;
#pragma unroll 1
                for (int kk = 0; kk < ksteps; ++kk)
                    if (kk < 4) umma_ss(tmem + kColBD, qv_d + kk * 2, rb + kk * 2, idesc_qk, kk > 0 ? 1u : 0u);
                umma_commit_addr(b_rempty + 8 * s);
                umma_commit_addr(b_bdfull);
                ++rc;
                ++bd;
                return true;
            };
            // S of global tile number tg into S[tg & 1], once the softmax has read S of tg - 2
            auto mma_s = [&](int tg) -> bool {
                const int s = kc % kNK;
                if (!mbar_wait(&bar.k_full[s], (kc / kNK) & 1, wc, 25)) return false;
                if (!mbar_wait(&bar.s_free[tg & 1], ((tg >> 1) & 1) ^ 1, wc, 27)) return false;
                tc_fence_after();
                const uint64_t kb = k_d + kStage * s;
                const uint32_t scol = tmem + ((tg & 1) ? kColS1 : kColS0);
#pragma unroll 1
                for (int kk = 0; kk < ksteps; ++kk)
                    if (kk < 4) umma_ss(scol, qu_d + kk * 2, kb + kk * 2, idesc_qk, kk > 0 ? 1u : 0u);
                umma_commit_addr(b_kempty + 8 * s);
                umma_commit_addr(b_sfull + 8 * (tg & 1));
                ++kc;
                return true;
            };
            Item it;
            for (int n = 0; ok && item_at<kTab>(p, sched_first, sched_count, n, it); ++n) {
                const int qb = n & 1;
                if (!(ok = mbar_wait(&bar.q_ready[qb], (n >> 1) & 1, wc, 20))) break;
                tc_fence_after();
                qu_d = qu_d0 + kQBuf * qb;
                qv_d = qv_d0 + kQBuf * qb;
                if (it.clampc && !(ok = mma_bd())) break;
                if (!(ok = mma_s(T))) break;
                if (need_chunk(0, C) && !(ok = mma_bd())) break;
                // tile t + 1's products are issued while the softmax works on tile t
                for (int t = 0; t + 1 < it.n_t; ++t) {
                    if (!(ok = mma_s(T + t + 1))) break;
                    if (need_chunk(t + 1, C) && !(ok = mma_bd())) break;
                }
                if (!ok) break;
                umma_commit(&bar.q_free[qb]);        // Qu and Qv of this item are read for good
                T += it.n_t;
            }
            // every S and BD product is awaited by the softmax before the CTA ends
            if (!ok) {
                umma_commit(bar.drain);
                (void)mbar_wait(bar.drain, 0, dw, 26);
            }
        }
        __syncwarp();
    } else if (warp == kPValueWarp) {
        // =========================================================== V tiles + P.V
        if (lane == 0) {
            constexpr uint32_t idesc_pv = idesc_bf16(128, NPV, 0, 1);
            const uint64_t v_d = sdesc_mn_sw128(smem_u32(smem + PSmem::V), kTile);
            constexpr uint64_t kStage = kTile >> 4;
            const uint32_t b_vempty = smem_u32(bar.v_empty), b_pvdone = smem_u32(bar.pv_done);
            // two cursors over the flattened (item, tile) sequence: V loads run one tile ahead
            struct Cursor {
                int n, t;
                Item it;
                bool valid;
            };
            auto advance = [&](Cursor& cu) {
                if (++cu.t >= cu.it.n_t) {
                    ++cu.n;
                    cu.t = 0;
                    cu.valid = item_at<kTab>(p, sched_first, sched_count, cu.n, cu.it);
                }
            };
            Cursor ld, cs;
            ld.n = 0; ld.t = 0; ld.valid = item_at<kTab>(p, sched_first, sched_count, 0, ld.it);
            cs = ld;
            int vc = 0, T = 0;
            bool ok = true;
            auto load_v = [&](const Cursor& cu) -> bool {
                const CUtensorMap* vm;
                int row;
                key_tile<kTab>(p, cu.it, cu.t, true, vm, row);
                const int s = vc % kNV;
                if (!mbar_wait(&bar.v_empty[s], ((vc / kNV) & 1) ^ 1, wc, 16)) return false;
                mbar_expect_tx(&bar.v_full[s], kTile);
                tma_load_4d(smem + PSmem::V + s * kTile, vm, 0, cu.it.h, row, cu.it.b, &bar.v_full[s]);
                ++vc;
                return true;
            };
            if (ld.valid) {
                ok = load_v(ld);
                advance(ld);
            }
            while (ok && cs.valid) {
                if (ld.valid) {
                    if (!(ok = load_v(ld))) break;
                    advance(ld);
                }
                const int s = T % kNV;
                // O of the previous item must have been read by the epilogue before it is reset
                if (cs.t == 0 && cs.n > 0 && !(ok = mbar_wait(bar.o_free, (cs.n - 1) & 1, wc, 29))) break;
                if (!(ok = mbar_wait(&bar.p_full[T & 1], (T >> 1) & 1, wc, 23))) break;
                if (!(ok = mbar_wait(&bar.v_full[s], (T / kNV) & 1, wc, 24))) break;
                tc_fence_after();
                const uint64_t vb = v_d + kStage * s;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    umma_ts(tmem + kColO, tmem + kColP + (kk >> 2) * 32 + (kk & 3) * 8,
                            vb + kk * (2048 >> 4), idesc_pv, (cs.t > 0 || kk > 0) ? 1u : 0u);
                umma_commit_addr(b_vempty + 8 * s);
                umma_commit_addr(b_pvdone);
                if (cs.t + 1 == cs.it.n_t) umma_commit(bar.o_full);
                ++T;
                advance(cs);
            }
            if (!ok) {
                umma_commit(bar.drain_v);
                (void)mbar_wait(bar.drain_v, 0, dw, 28);
            }
            if (*abort_flag) {
                for (int x = vc - kNV; x < vc; ++x)
                    if (x >= 0) (void)mbar_wait(&bar.v_full[x % kNV], (x / kNV) & 1, dw, 17);
            }
        }
    } else {
        // =========================================================== softmax warps 0-7
        const int hf = tid >> 7;                     // column half of every tile
        const int li = tid & 127;                    // TMEM lane == tile row
        const int pi = query_of_row(li);             // query offset inside the tile
        const int sh = (li >> 6) ? 0 : 1;            // odd queries: 0, even queries: 1
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        uint32_t* bdrow = reinterpret_cast<uint32_t*>(smem + PSmem::BD) + li * kBdPitchWords;
        const uint32_t row_saddr = smem_u32(bdrow);
        float* xchg = reinterpret_cast<float*>(bdrow + 128);          // 4 exchange words per row
        const int wbase_row = (li & 63) - 32 * hf;                   // (pi + sh - 1)/2 - 32 hf
        bool ok = true;
        int T = 0, bd = 0;                           // tiles and BD products consumed so far
        Item it;
        for (int n = 0; item_at<kTab>(p, sched_first, sched_count, n, it); ++n) {
            const int M = p.M;
            float m_run = -INFINITY, l_half = 0.f;
            uint32_t bdc_bits = 0;                  // fp32 bits of (q+v).r[clamp_len] for this row
            if constexpr (kTab) {
                // learned table: chunk -1, the distances just below the first key tile's, goes
                // into ring slot 1 (no key is masked by position)
                if (ok) ok = warp_wait(bar.bd_full, bd & 1, wc, 31);
                if (ok) {
                    tc_fence_after();
                    uint32_t bdv[64];
                    tmem_ld64(tmem + lane_base + kColBD + 64 * hf, bdv);
                    tmem_ld_wait();
                    tc_fence_before();
                    __syncwarp();
                    mbar_arrive_if(bar.bd_free, lane == 0);
                    ring_write_half(bdrow, row_saddr, bdv, -1, hf, sh);
                }
                ++bd;
            } else {
            // The ring starts as bf16 -inf.  The positions the diagonal tile reads for future
            // keys (lj > pi) are never written before that tile, so those keys come out masked.
            {
                uint4* w = reinterpret_cast<uint4*>(bdrow + 64 * hf);
                const uint4 ninf = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
#pragma unroll
                for (int q4 = 0; q4 < 16; ++q4) w[q4] = ninf;
            }
            pair_bar(li);
            if (it.clampc) {
                if (ok) ok = warp_wait(bar.bd_full, bd & 1, wc, 31);
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
                ++bd;
            }
            }

            for (int t = 0; t < it.n_t; ++t, ++T) {
                const bool chunk = need_chunk(t, C);
                // a slot whose distances all reach clamp_len holds r[clamp_len]'s value
                // everywhere; it is written once, unless two tiles ago it already held that fill
                const bool fill = it.clampc && !chunk && (t < 2 || need_chunk(t - 2, C));
                const uint32_t scol = tmem + lane_base + ((T & 1) ? kColS1 : kColS0) + 64 * hf;
                float s[64];
                bool kz0 = false, kz1 = false;              // keys lane, lane + 32 of this half masked
                if constexpr (kMask) {
                    // requested now, used after the ring write: the loads fly during the waits
                    const int jk = 128 * (p.n_qt - 1 - t) + 64 * hf + lane;
                    const uint8_t* km = p.key_mask + static_cast<int64_t>(it.b) * p.L;
                    kz0 = jk < p.L && __ldg(km + jk) == 0;
                    kz1 = jk + 32 < p.L && __ldg(km + jk + 32) == 0;
                }
                if (chunk && ok) ok = warp_wait(bar.bd_full, bd & 1, wc, 32);
                if (ok) ok = warp_wait(&bar.s_full[T & 1], (T >> 1) & 1, wc, 33);
                if (ok) {
                    tc_fence_after();
                    if (chunk || fill) {
                        uint32_t bdv[64];
                        if (chunk) {
                            tmem_ld64(tmem + lane_base + kColBD + 64 * hf, bdv);
                            tmem_ld_wait();
                            tc_fence_before();
                            __syncwarp();
                            mbar_arrive_if(bar.bd_free, lane == 0);
                            const int cc = C - 128 * t - 64 * hf;   // first local column at the clamp
                            if (it.clampc && cc < 64) {
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
                    tc_fence_before();                  // the S buffer may now take S of T + 2
                    __syncwarp();
                    mbar_arrive_if(&bar.s_free[T & 1], lane == 0);
#pragma unroll
                    for (int k = 0; k < 64; ++k) s[k] = __uint_as_float(su[k]);
                }
                if (chunk) ++bd;
                if (chunk || fill) pair_bar(li);            // both halves of the slot are in the ring
                const int wbase = 64 * (t & 1) + wbase_row;
                if constexpr (kTab) {
                    // keys past the sequence's end (only in the first tile, the last key tile)
                    // read -inf; each thread writes exactly the positions it reads itself
                    const int lk = p.L - 128 * (p.n_qt - 1 - t);
                    if (ok && lk < 64 * hf + 64) {
#pragma unroll 1
                        for (int lj = max(lk, 64 * hf); lj < 64 * hf + 64; ++lj)
                            sts_u16(row_saddr + 2u * ((128 * (t & 1) + pi - lj + sh) & 255), 0xFF80);
                    }
                    if constexpr (kMask) {
                        // masked keys of this half (the same for every row: a warp-uniform loop)
                        uint64_t z = (static_cast<uint64_t>(__ballot_sync(0xffffffffu, kz1)) << 32) |
                                     __ballot_sync(0xffffffffu, kz0);
                        while (ok && z) {
                            const int lj = 64 * hf + __ffsll(static_cast<long long>(z)) - 1;
                            z &= z - 1;
                            sts_u16(row_saddr + 2u * ((128 * (t & 1) + pi - lj + sh) & 255), kMaskedKeyBf16);
                        }
                    }
                } else {
                    const int j0 = M + it.i0 - 128 * t;
                    const int lm = p.lo - j0;               // keys lj < lm precede the valid memory
                    if (ok && lm > 0) {
                        // only the last (oldest) tile can start before the valid memory: its
                        // invalid keys read -inf; each thread writes exactly the positions it
                        // reads itself
                        const int hi_lj = min(lm, 64 * hf + 64);
#pragma unroll 1
                        for (int lj = 64 * hf; lj < hi_lj; ++lj)
                            sts_u16(row_saddr + 2u * ((128 * (t & 1) + pi - lj + sh) & 255), 0xFF80);
                    }
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
                    // P = 2^(s - m) is taken on bf16 pairs: P.V consumes bf16 P, so the pair is
                    // rounded once before the exponential instead of after it, and one
                    // special-function instruction serves two keys.  The row sum adds exactly the
                    // bf16 values P.V multiplies.
                    const uint64_t negm = f2_pack(-m_run, -m_run);
                    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
                    uint32_t pw[32];
                    if constexpr (kLse == 1) {
                        // the row sum alone, from fp32 exponentials of the fp32 logits (P is not
                        // needed: zeros go through P.V)
#pragma unroll
                        for (int k = 0; k < 32; ++k) {
                            a0 += ex2_approx(s[2 * k] - m_run);
                            b0 += ex2_approx(s[2 * k + 1] - m_run);
                            pw[k] = 0u;
                        }
                    } else {
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        float y0, y1;
                        f2_unpack(f2_add(f2_pack(s[2 * k], s[2 * k + 1]), negm), y0, y1);
                        pw[k] = ex2_bf16x2(pack_bf16x2(y0, y1));
                        if (k & 1) {
                            b0 = add_bf16lo_f32(pw[k], b0);
                            b1 = add_bf16hi_f32(pw[k], b1);
                        } else {
                            a0 = add_bf16lo_f32(pw[k], a0);
                            a1 = add_bf16hi_f32(pw[k], a1);
                        }
                    }
                    }
                    l_half = fmaf(l_half, alpha, (a0 + a1) + (b0 + b1));
                    // P.V of the previous tile (of this item or the one before) must be complete
                    // before the P buffer, or O (rescale), is touched
                    const bool rescale_any = t >= 1 && __any_sync(0xffffffffu, rescale_o);
                    if (T >= 1) {
                        ok = warp_wait(bar.pv_done, (T - 1) & 1, wc, 34);
                        if (ok) tc_fence_after();
                    }
                    // P (bf16): keys 64hf.. at column 32hf of the P buffer
                    if (ok) tmem_st32(tmem + lane_base + kColP + 32 * hf, pw);
                    if (ok && rescale_any) {
                        const uint64_t al2 = f2_pack(alpha, alpha);
                        uint32_t o[32];
                        const uint32_t oaddr = tmem + lane_base + kColO + (NPV / 2) * hf;
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
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    mbar_arrive_if(&bar.p_full[T & 1], lane == 0 && ok);
                }
            }

            // ---- epilogue: O / (l_0 + l_1) -> bf16 -> out[b, i0 + pi, h, :].  O is released to the
            // next item's P.V as soon as it is read.  With 16-byte aligned output rows each thread
            // stages its normalised half row in the front of its (now dead) ring row; the pair of
            // warps then writes its 32 rows as whole 128-byte lines, four rows per store
            // instruction instead of 32 half lines (a chunk past d_head's end, when D % 8 != 0,
            // element by element).  Other layouts store element by element from registers.
            if (ok) ok = warp_spin(bar.o_full, n & 1, wc, 35);
            xchg[2 * (it.n_t & 1) + hf] = l_half;
            pair_bar(li);
            const bool staged = p.out_a16 != 0;
            if (ok && kLse == 1) {
                // log2-domain log-sum-exp of the row, in the scaled score units of the logits
                __syncwarp();
                mbar_arrive_if(bar.o_free, lane == 0);
                const int i = it.i0 + pi;
                if (hf == 0 && i < p.L)
                    p.lse[(static_cast<int64_t>(it.b) * p.L + i) * p.H + it.h] =
                        m_run + __log2f(l_half + xchg[2 * (it.n_t & 1) + 1]);
            } else if (ok) {
                uint32_t o[32];
                tc_fence_after();
                tmem_ld32(tmem + lane_base + kColO + (NPV / 2) * hf, o);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                mbar_arrive_if(bar.o_free, lane == 0);
                const float inv_l = rcp_approx(l_half + xchg[2 * (it.n_t & 1) + (hf ^ 1)]);
                if constexpr (kLse == 2) {
                    // the row sum of the bf16 P that P.V multiplied, the normaliser of out
                    const int i = it.i0 + pi;
                    if (hf == 0 && i < p.L)
                        p.lse[(static_cast<int64_t>(it.b) * p.L + i) * p.H + it.h] =
                            m_run + __log2f(l_half + xchg[2 * (it.n_t & 1) + 1]);
                }
                if (staged) {
                    uint4* st = reinterpret_cast<uint4*>(bdrow + 16 * hf);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w[e] = pack_bf16x2(__uint_as_float(o[8 * q4 + 2 * e]) * inv_l,
                                               __uint_as_float(o[8 * q4 + 2 * e + 1]) * inv_l);
                        st[q4] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                } else {
                    const int i = it.i0 + pi, d0 = (NPV / 2) * hf;
                    if (i < p.L) {
                        __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) + it.b * p.o_sb +
                                              static_cast<int64_t>(i) * p.o_st + it.h * p.o_sh;
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            if (d0 + k < p.D) orow[d0 + k] = __float2bfloat16_rn(__uint_as_float(o[k]) * inv_l);
                    }
                }
            }
            pair_bar(li);                                   // both halves of every row are staged
            if (kLse != 1 && ok && staged) {
                // this warp stores rows (li & ~31) + 16 hf + 0..15: lane -> row + lane / 8, chunk
                // of 8 columns lane mod 8
                const uint32_t* bd0 = reinterpret_cast<const uint32_t*>(smem + PSmem::BD);
                const int c = lane & 7;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int r = (li & ~31) + 16 * hf + 4 * k + (lane >> 3);
                    const int i = it.i0 + query_of_row(r);
                    if (i < p.L && 8 * c < p.D) {
                        const uint4 v = *reinterpret_cast<const uint4*>(bd0 + r * kBdPitchWords + 4 * c);
                        __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) + it.b * p.o_sb +
                                              static_cast<int64_t>(i) * p.o_st + it.h * p.o_sh;
                        if (8 * c + 8 <= p.D) {
                            *reinterpret_cast<uint4*>(orow + 8 * c) = v;
                        } else {                    // the chunk holding d_head's end (D % 8 != 0)
                            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                if (8 * c + e < p.D)
                                    orow[8 * c + e] = __ushort_as_bfloat16(static_cast<unsigned short>(w[e >> 1] >> (16 * (e & 1))));
                        }
                    }
                }
            }
            pair_bar(li);                                   // staged rows read before the ring reset
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kPMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

cudaError_t launch_attn_persist(const AttnTcParams& p, int sm_count, cudaStream_t s)
{
    if (p.B == 0 || p.L == 0 || p.H == 0) return cudaSuccess;
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(attn_persist_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             PSmem::Size);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(attn_persist_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, PSmem::Size);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(attn_persist_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 PSmem::Size);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(attn_persist_kernel<false, false, 1>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, PSmem::Size);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(attn_persist_kernel<false, false, 2>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, PSmem::Size);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    const int64_t items = static_cast<int64_t>(p.n_qt) * p.H * p.B;
    const int grid = static_cast<int>(items < sm_count ? items : sm_count);
    if (p.lse && !p.table && p.lse_out)
        return launch_dependent(attn_persist_kernel<false, false, 2>, dim3(grid), dim3(kPThreads), PSmem::Size,
                                s, p);
    if (p.lse && !p.table)
        return launch_dependent(attn_persist_kernel<false, false, 1>, dim3(grid), dim3(kPThreads), PSmem::Size,
                                s, p);
    if (p.table == 2)
        return launch_dependent(attn_persist_kernel<true, true>, dim3(grid), dim3(kPThreads), PSmem::Size, s, p);
    if (p.table) return launch_dependent(attn_persist_kernel<true>, dim3(grid), dim3(kPThreads), PSmem::Size, s, p);
    return launch_dependent(attn_persist_kernel<false>, dim3(grid), dim3(kPThreads), PSmem::Size, s, p);
}

}  // namespace txl
