// txl_attn_tc.cu -- fused relative attention for sm_103a: TMA tiles, tcgen05 UMMA with TMEM
// accumulators, the relative shift as an index remap, online softmax, P.V on tensor cores.
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
// BD values are computed once by UMMA and kept per thread in shared memory; the relative shift is
// then a per-row index remap (thread li reads entry (li - lj) of chunk t, or 128 + li - lj of
// chunk t-1) instead of the pad-and-reshape "Relative Shift" trick the qidao123 page names.
// Distances >= clamp_len all use r[clamp_len] ("TransformerXL 相对位置编码" §2.4): one extra
// UMMA of Qv against the rows starting at clamp_len gives that per-row value; chunks that lie
// entirely beyond clamp_len are never loaded or multiplied.
//
// Thread li of warps 0-3 owns TMEM lane li, i.e. query row li of the tile, which holds query
// pi(li) = 2*(li mod 64) + li/64: warps 0-1 hold the even queries, warps 2-3 the odd ones, so the
// parity of every per-thread shift is warp-uniform and the remap needs no divergent code.
//
// Roles (192 threads): warps 0-3 softmax / correction / epilogue, warp 4 TMA producer, warp 5
// UMMA issuer (and TMEM owner).  Every wait is bounded (2 s) and aborts the CTA cleanly.
#include <cuda_bf16.h>

#include "txl_internal.h"
#include "txl_ptx.cuh"

namespace txl {

namespace {

constexpr int kThreads = 192;
constexpr int kTile = 16384;                 // 128 rows x 128 B: one swizzle-atom column
constexpr int kBdPitchWords = 132;           // per-thread ring of 256 bf16 + 4 words of padding
constexpr int kBdBytes = 128 * kBdPitchWords * 4;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColBD = 256, kColO = 384;
constexpr float kRescaleThreshold = 8.0f;    // log2 units: P values stay below 2^8

template <int NA>
struct AttnSmem {
    static constexpr int NS = (NA == 1) ? 2 : 1;    // pipeline stages for K, V and r tiles
    static constexpr int Qu = 0;
    static constexpr int Qv = Qu + NA * kTile;
    static constexpr int K = Qv + NA * kTile;
    static constexpr int V = K + NS * NA * kTile;
    static constexpr int R = V + NS * NA * kTile;
    static constexpr int BD = R + NS * NA * kTile;     // also the raw-Q staging area
    static constexpr int Bars = BD + kBdBytes;
    // q_full q_ready | k_full k_empty v_full v_empty r_full r_empty (NS each) |
    // s_full[2] bd_full bd_free p_full[2] pv_done o_full drain
    static constexpr int NumBars = 2 + 6 * NS + 9;
    static constexpr int Misc = Bars + NumBars * 8;
    static constexpr int Size = Misc + 16;
};

struct Bars {
    uint64_t *q_full, *q_ready, *k_full, *k_empty, *v_full, *v_empty, *r_full, *r_empty;
    uint64_t *s_full, *bd_full, *bd_free, *p_full, *pv_done, *o_full, *drain;
};

template <int NS>
__device__ __forceinline__ Bars carve_bars(uint8_t* base)
{
    uint64_t* b = reinterpret_cast<uint64_t*>(base);
    Bars r;
    r.q_full = b; r.q_ready = b + 1;
    r.k_full = b + 2; r.k_empty = r.k_full + NS;
    r.v_full = r.k_empty + NS; r.v_empty = r.v_full + NS;
    r.r_full = r.v_empty + NS; r.r_empty = r.r_full + NS;
    r.s_full = r.r_empty + NS;
    r.bd_full = r.s_full + 2; r.bd_free = r.bd_full + 1;
    r.p_full = r.bd_free + 1;
    r.pv_done = r.p_full + 2; r.o_full = r.pv_done + 1; r.drain = r.o_full + 1;
    return r;
}

// Tile plan shared by every role of the CTA.
struct Plan {
    int i0, n_t, max_delta;
    bool clampc;
    __device__ bool need_chunk(int t, int C) const { return 128 * t < C; }
};

__device__ __forceinline__ int query_of_row(int li) { return 2 * (li & 63) + (li >> 6); }

// ---------------------------------------------------------------------------------------------
// Softmax step on one tile for one thread.  MODE bits: 1 = diagonal tile (mask lj > pi),
// 2 = low mask (lj < lm), 4 = some distances clamped (lj <= thr), 8 = all clamped (no buffer).
template <int MODE>
__device__ __forceinline__ float tile_logits(float* s, const uint32_t* bdrow, int wbase, int pi,
                                             int lm, int thr, float bd_clamp)
{
    float mx = -INFINITY;
#pragma unroll
    for (int m = 0; m < 64; ++m) {
        const int l0 = 2 * m, l1 = 2 * m + 1;
        float x0, x1;
        if (MODE & 8) {
            x0 = s[l0] + bd_clamp;
            x1 = s[l1] + bd_clamp;
        } else {
            const uint32_t w = bdrow[(wbase - m) & 127];
            x0 = add_bf16hi_f32(w, s[l0]);
            x1 = add_bf16lo_f32(w, s[l1]);
            if (MODE & 4) {
                x0 = (l0 <= thr) ? s[l0] + bd_clamp : x0;
                x1 = (l1 <= thr) ? s[l1] + bd_clamp : x1;
            }
        }
        if (MODE & 1) {
            x0 = (l0 <= pi) ? x0 : -INFINITY;
            x1 = (l1 <= pi) ? x1 : -INFINITY;
        }
        if (MODE & 2) {
            x0 = (l0 >= lm) ? x0 : -INFINITY;
            x1 = (l1 >= lm) ? x1 : -INFINITY;
        }
        s[l0] = x0;
        s[l1] = x1;
        mx = fmaxf(mx, fmaxf(x0, x1));
    }
    return mx;
}

__device__ __forceinline__ float dispatch_logits(int mode, float* s, const uint32_t* bdrow,
                                                 int wbase, int pi, int lm, int thr, float bdc)
{
    switch (mode) {
    case 0: return tile_logits<0>(s, bdrow, wbase, pi, lm, thr, bdc);
    case 1: return tile_logits<1>(s, bdrow, wbase, pi, lm, thr, bdc);
    case 2: return tile_logits<2>(s, bdrow, wbase, pi, lm, thr, bdc);
    case 4: return tile_logits<4>(s, bdrow, wbase, pi, lm, thr, bdc);
    case 5: return tile_logits<5>(s, bdrow, wbase, pi, lm, thr, bdc);
    case 6: return tile_logits<6>(s, bdrow, wbase, pi, lm, thr, bdc);
    case 8: return tile_logits<8>(s, bdrow, wbase, pi, lm, thr, bdc);
    case 9: return tile_logits<9>(s, bdrow, wbase, pi, lm, thr, bdc);
    case 10: return tile_logits<10>(s, bdrow, wbase, pi, lm, thr, bdc);
    case 3: return tile_logits<3>(s, bdrow, wbase, pi, lm, thr, bdc);
    case 7: return tile_logits<7>(s, bdrow, wbase, pi, lm, thr, bdc);
    default: return tile_logits<11>(s, bdrow, wbase, pi, lm, thr, bdc);
    }
}

template <int NA>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(const __grid_constant__ AttnTcParams p)
{
    using S = AttnSmem<NA>;
    constexpr int NS = S::NS;
    constexpr int NPV = 64 * NA;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if ((smem_u32(smem) & 1023u) != 0) {
        if (tid == 0 && p.err_flag) atomicCAS(p.err_flag, 0, TXL_ERR_ALIGNMENT);
        return;
    }
    const Bars bar = carve_bars<NS>(smem + S::Bars);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + S::Misc);
    int* abort_flag = reinterpret_cast<int*>(smem + S::Misc + 4);

    if (tid == 0) {
        mbar_init(bar.q_full, 1);
        mbar_init(bar.q_ready, 4);
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bar.k_full[s], 1); mbar_init(&bar.k_empty[s], 1);
            mbar_init(&bar.v_full[s], 1); mbar_init(&bar.v_empty[s], 1);
            mbar_init(&bar.r_full[s], 1); mbar_init(&bar.r_empty[s], 1);
        }
        mbar_init(&bar.s_full[0], 1); mbar_init(&bar.s_full[1], 1);
        mbar_init(bar.bd_full, 1); mbar_init(bar.bd_free, 4);
        mbar_init(&bar.p_full[0], 4); mbar_init(&bar.p_full[1], 4);
        mbar_init(bar.pv_done, 1); mbar_init(bar.o_full, 1); mbar_init(bar.drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 5) tmem_alloc(tmem_holder, 512);
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

    if (warp == 4) {
        // =========================================================== TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_q);
            tma_prefetch_desc(&p.tm_kcur);
            tma_prefetch_desc(&p.tm_vcur);
            tma_prefetch_desc(&p.tm_r);
            if (M > 0) { tma_prefetch_desc(&p.tm_kmem); tma_prefetch_desc(&p.tm_vmem); }
            uint8_t* staging = smem + S::BD;
            mbar_expect_tx(bar.q_full, NA * kTile);
            for (int a = 0; a < NA; ++a)
                tma_load_4d(staging + a * kTile, &p.tm_q, 64 * a, h, plan.i0, b, bar.q_full);
            int rs = 0, kc = 0, vc = 0;               // loads issued per pipeline
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
                const int j0 = M + plan.i0 - 128 * t;
                const CUtensorMap* km;
                const CUtensorMap* vm;
                int row;
                if (j0 >= M) { km = &p.tm_kcur; vm = &p.tm_vcur; row = j0 - M; }
                else {
                    km = &p.tm_kmem; vm = &p.tm_vmem;
                    row = p.wp ? static_cast<int>((static_cast<int64_t>(p.wp) + j0) % M) : j0;
                }
                const int s = t % NS;
                const uint32_t par = ((t / NS) & 1) ^ 1;
                if (!(ok = mbar_wait(&bar.k_empty[s], par, wc, 11))) break;
                mbar_expect_tx(&bar.k_full[s], NA * kTile);
                for (int a = 0; a < NA; ++a)
                    tma_load_4d(smem + S::K + (s * NA + a) * kTile, km, 64 * a, h, row, b, &bar.k_full[s]);
                ++kc;
                if (!(ok = mbar_wait(&bar.v_empty[s], par, wc, 12))) break;
                mbar_expect_tx(&bar.v_full[s], NA * kTile);
                for (int a = 0; a < NA; ++a)
                    tma_load_4d(smem + S::V + (s * NA + a) * kTile, vm, 64 * a, h, row, b, &bar.v_full[s]);
                ++vc;
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
                for (int x = vc - NS; x < vc; ++x)
                    if (x >= 0) (void)mbar_wait(&bar.v_full[x % NS], (x / NS) & 1, dw, 16);
            }
        }
    } else if (warp == 5) {
        // =========================================================== UMMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16(128, 128, 0, 0);
            constexpr uint32_t idesc_pv = idesc_bf16(128, NPV, 0, 1);
            const uint32_t qu = smem_u32(smem + S::Qu), qv = smem_u32(smem + S::Qv);
            const int ksteps = p.k_steps;
            int rs = 0, bd_uses = 0;
            bool ok = mbar_wait(bar.q_ready, 0, wc, 20);
            auto mma_bd = [&]() -> bool {
                const int s = rs % NS;
                if (!mbar_wait(&bar.r_full[s], (rs / NS) & 1, wc, 21)) return false;
                if (!mbar_wait(bar.bd_free, (bd_uses & 1) ^ 1, wc, 22)) return false;
                tc_fence_after();
                const uint32_t rb = smem_u32(smem + S::R + s * NA * kTile);
                for (int kk = 0; kk < ksteps; ++kk) {
                    const uint32_t off = (kk >> 2) * kTile + (kk & 3) * 32;
                    umma_ss(tmem + kColBD, sdesc_k_sw128(qv + off), sdesc_k_sw128(rb + off), idesc_qk,
                            kk > 0 ? 1u : 0u);
                }
                umma_commit(&bar.r_empty[s]);
                umma_commit(bar.bd_full);
                ++rs;
                ++bd_uses;
                return true;
            };
            auto mma_pv = [&](int t) -> bool {
                const int s = t % NS;
                if (!mbar_wait(&bar.p_full[t & 1], (t >> 1) & 1, wc, 23)) return false;
                if (!mbar_wait(&bar.v_full[s], (t / NS) & 1, wc, 24)) return false;
                tc_fence_after();
                const uint32_t vb = smem_u32(smem + S::V + s * NA * kTile);
                const uint32_t pcol = tmem + ((t & 1) ? kColS1 : kColS0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    umma_ts(tmem + kColO, pcol + kk * 8, sdesc_mn_sw128(vb + kk * 2048, kTile), idesc_pv,
                            (t > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&bar.v_empty[s]);
                umma_commit(bar.pv_done);
                return true;
            };
            if (ok) {
                tc_fence_after();
                if (plan.clampc) ok = mma_bd();
            }
            for (int t = 0; t < n_t && ok; ++t) {
                const int s = t % NS;
                if (!(ok = mbar_wait(&bar.k_full[s], (t / NS) & 1, wc, 25))) break;
                tc_fence_after();
                const uint32_t kb = smem_u32(smem + S::K + s * NA * kTile);
                const uint32_t scol = tmem + ((t & 1) ? kColS1 : kColS0);
                for (int kk = 0; kk < ksteps; ++kk) {
                    const uint32_t off = (kk >> 2) * kTile + (kk & 3) * 32;
                    umma_ss(scol, sdesc_k_sw128(qu + off), sdesc_k_sw128(kb + off), idesc_qk,
                            kk > 0 ? 1u : 0u);
                }
                umma_commit(&bar.k_empty[s]);
                umma_commit(&bar.s_full[t & 1]);
                if (plan.need_chunk(t, C) && !(ok = mma_bd())) break;
                if (t >= 1 && !(ok = mma_pv(t - 1))) break;
            }
            if (ok) ok = mma_pv(n_t - 1);
            umma_commit(ok ? bar.o_full : bar.drain);
            if (!ok) {
                int never = 0;
                const WaitCtl dw{&never, nullptr, 100000000ull};
                (void)mbar_wait(bar.drain, 0, dw, 26);
            }
        }
        __syncwarp();
    } else {
        // =========================================================== softmax warps 0-3
        const int li = tid;                          // TMEM lane == tile row
        const int pi = query_of_row(li);             // query offset inside the tile
        const int sh = (warp >> 1) ? 0 : 1;          // odd queries: 0, even queries: 1
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        bool ok = true;

        // ---- prologue: Qu = c(q+u), Qv = c(q+v) in bf16, rows permuted to pi(li)
        ok = warp_wait(bar.q_full, 0, wc, 30);
        if (ok) {
            const uint8_t* staging = smem + S::BD;
            const int src = pi;
            const float* uh = p.u + static_cast<int64_t>(h) * p.D;
            const float* vh = p.vb + static_cast<int64_t>(h) * p.D;
#pragma unroll
            for (int a = 0; a < NA; ++a) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 raw = *reinterpret_cast<const uint4*>(
                        staging + a * kTile + src * 128 + ((c ^ (src & 7)) << 4));
                    const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
                    uint32_t wu[4], wv[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int d0 = 64 * a + 8 * c + 2 * e;
                        const float q0 = __uint_as_float(rw[e] << 16);
                        const float q1 = __uint_as_float(rw[e] & 0xffff0000u);
                        const float u0 = d0 < p.D ? __ldg(uh + d0) : 0.f;
                        const float u1 = d0 + 1 < p.D ? __ldg(uh + d0 + 1) : 0.f;
                        const float v0 = d0 < p.D ? __ldg(vh + d0) : 0.f;
                        const float v1 = d0 + 1 < p.D ? __ldg(vh + d0 + 1) : 0.f;
                        const bool z0 = d0 >= p.D, z1 = d0 + 1 >= p.D;
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
            if (lane == 0) mbar_arrive(bar.q_ready);
        }
        named_bar_sync(1, 128);       // all staging reads done before the BD ring reuses it

        uint32_t* bdrow = reinterpret_cast<uint32_t*>(smem + S::BD) + li * kBdPitchWords;
        const int base_w = li & 63;                   // (pi + sh - 1) / 2
        float m_run = -INFINITY, l_run = 0.f, bd_clamp = 0.f, carry = 0.f;
        int bd_uses = 0;

        if (ok && plan.clampc) {
            ok = warp_wait(bar.bd_full, bd_uses & 1, wc, 31);
            if (ok) {
                tc_fence_after();
                uint32_t v0;
                tmem_ld1(tmem + lane_base + kColBD, v0);
                tmem_ld_wait();
                bd_clamp = __uint_as_float(v0);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar.bd_free);
                ++bd_uses;
            }
        }

        for (int t = 0; t < n_t && ok; ++t) {
            // ---- new BD chunk: TMEM -> per-thread ring in shared memory (bf16, remap-ready)
            if (plan.need_chunk(t, C)) {
                ok = warp_wait(bar.bd_full, bd_uses & 1, wc, 32);
                if (!ok) break;
                tc_fence_after();
                uint32_t* slot = bdrow + 64 * (t & 1);
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t v[32];
                    tmem_ld32(tmem + lane_base + kColBD + 32 * cb, v);
                    tmem_ld_wait();
                    uint32_t w[16];
                    if (sh == 0) {
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            w[k] = pack_bf16x2(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1]));
                    } else {
                        w[0] = pack_bf16x2(carry, __uint_as_float(v[0]));
#pragma unroll
                        for (int k = 1; k < 16; ++k)
                            w[k] = pack_bf16x2(__uint_as_float(v[2 * k - 1]), __uint_as_float(v[2 * k]));
                        carry = __uint_as_float(v[31]);
                    }
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        *reinterpret_cast<uint4*>(slot + 16 * cb + 4 * q4) =
                            make_uint4(w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
                }
                if (sh == 1) bdrow[64 * ((t + 1) & 1)] = pack_bf16x2(carry, 0.f);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar.bd_free);
                ++bd_uses;
            }

            // ---- scores of tile t
            ok = warp_wait(&bar.s_full[t & 1], (t >> 1) & 1, wc, 33);
            if (!ok) break;
            tc_fence_after();
            const uint32_t scol = tmem + lane_base + ((t & 1) ? kColS1 : kColS0);
            uint32_t su[128];
            tmem_ld32(scol + 0, su);
            tmem_ld32(scol + 32, su + 32);
            tmem_ld32(scol + 64, su + 64);
            tmem_ld32(scol + 96, su + 96);
            tmem_ld_wait();
            float s[128];
#pragma unroll
            for (int k = 0; k < 128; ++k) s[k] = __uint_as_float(su[k]);
            const int j0 = M + plan.i0 - 128 * t;
            const int lm = lo - j0;                       // first visible column of this tile
            const int thr = 128 * t + pi - C;             // columns <= thr are clamped
            int mode = 0;
            if (t == 0) mode |= 1;
            if (lm > 0) mode |= 2;
            if (__all_sync(0xffffffffu, thr >= 127)) mode |= 8;
            else if (__any_sync(0xffffffffu, thr >= 0)) mode |= 4;
            const int wbase = 64 * (t & 1) + base_w;
            const float mt = dispatch_logits(mode, s, bdrow, wbase, pi, lm, thr, bd_clamp);

            // ---- online softmax with a lazily refreshed running max
            float alpha = 1.f;
            bool rescale_o = false;
            if (t == 0) {
                m_run = mt;
            } else if (mt > m_run + kRescaleThreshold) {
                alpha = ex2_approx(m_run - mt);
                m_run = mt;
                rescale_o = true;
            }
            float sum = 0.f;
            uint32_t pw[64];
#pragma unroll
            for (int k = 0; k < 64; ++k) {
                const float p0 = ex2_approx(s[2 * k] - m_run);
                const float p1 = ex2_approx(s[2 * k + 1] - m_run);
                sum += p0 + p1;
                pw[k] = pack_bf16x2(p0, p1);
            }
            l_run = fmaf(l_run, alpha, sum);
            tmem_st32(scol + 0, pw);
            tmem_st32(scol + 32, pw + 32);
            if (t >= 1 && __any_sync(0xffffffffu, rescale_o)) {
                // O may only be touched once PV of the previous tile has completed
                ok = warp_wait(bar.pv_done, (t - 1) & 1, wc, 34);
                if (!ok) break;
                tc_fence_after();
#pragma unroll 1
                for (int cb = 0; cb < NPV / 32; ++cb) {
                    uint32_t o[32];
                    tmem_ld32(tmem + lane_base + kColO + 32 * cb, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                    tmem_st32(tmem + lane_base + kColO + 32 * cb, o);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.p_full[t & 1]);
        }

        // ---- epilogue: O / l -> bf16 -> out[b, i0 + pi, h, :]
        if (ok) {
            ok = warp_wait(bar.o_full, 0, wc, 35);
        }
        if (ok) {
            tc_fence_after();
            const int i = plan.i0 + pi;
            const float inv_l = 1.f / l_run;
            __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) + b * p.o_sb +
                                  static_cast<int64_t>(i) * p.o_st + h * p.o_sh;
            const bool vec = (p.D % 8) == 0;
#pragma unroll 1
            for (int cb = 0; cb < NPV / 32; ++cb) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_base + kColO + 32 * cb, o);
                tmem_ld_wait();
                if (i >= p.L) continue;
                const int d0 = 32 * cb;
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
    if (warp == 5) {
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

cudaError_t launch_attn_tc(const AttnTcParams& p, cudaStream_t s)
{
    if (p.B == 0 || p.L == 0 || p.H == 0) return cudaSuccess;
    return p.n_atoms == 1 ? launch_na<1>(p, s) : launch_na<2>(p, s);
}

}  // namespace txl
