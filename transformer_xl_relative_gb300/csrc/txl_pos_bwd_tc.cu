// txl_pos_bwd_tc.cu -- dW_R = R^T dr on the 5th-generation tensor cores (tcgen05.mma kind::tf32,
// three products per K step for fp32-level accuracy).
//
// R is the interleaved sinusoid of the relative positions ("Transformer-XL 和相对位置编码" §2.3.2,
// the encoding R_{i-j} that W_R projects), dr the gradient of the position rows the attention
// backward writes; dW_R[m][n] = sum_delta R_delta[m] dr[delta][n] with n = h D + d.  Each CTA owns a
// 128 (model columns m) x 256 (columns n) tile over a share of the distances, in chunks of 32:
//  * its threads generate the chunk of R^T with the arithmetic of the position table (frequencies in
//    double precision, here as exp(-2k ln(10000) / d_model), the angle of every fourth distance
//    reduced modulo 2 pi in double precision, the three after it offset in fp32, the fp32 sine or
//    cosine, both from one sincosf: entries within 6e-7 of the exact sinusoid), and load the chunk
//    of dr;
//  * both are split into tf32 parts, x = hi + lo with hi = x rounded to tf32 and lo = x - hi (exact
//    in fp32), and R_hi dr_hi + R_hi dr_lo + R_lo dr_hi run as UMMAs (A: R^T and B: dr^T, both
//    K-major, the distances along the 128-byte swizzled rows, 32 fp32 per row) into one 128 x 256
//    fp32 TMEM accumulator.  The dropped lo.lo term and the tf32 reading of the lo parts leave about
//    2^-21 relative per product.
// Two stages: the threads fill one while the products of the other run.  The tile is then added
// into the zeroed dW_R through shared memory, one row segment per warp instruction (the distance
// shares of one tile add up there).
#include <cmath>

#include "txl_internal.h"
#include "txl_ptx.cuh"

namespace txl {

namespace {

constexpr int kPBThreads = 512;
constexpr int kPBChunk = 32;                        // distances per chunk: one 128-byte row of fp32
constexpr int kPBM = 128, kPBN = 256;
constexpr int kATile = kPBM * 128;                  // R^T chunk, [m][32 fp32]
constexpr int kBTile = kPBN * 128;                  // dr^T chunk, [n][32 fp32]
constexpr int kPBStage = 2 * kATile + 2 * kBTile;   // hi and lo of each
constexpr int kOutPitch = kPBN + 4;                 // fp32 per staged output row

struct PBSmem {
    static constexpr int Stages = 0;                 // two stages: A_hi, A_lo, B_hi, B_lo
    static constexpr int Ws = Stages + 2 * kPBStage; // double [128]
    static constexpr int Wf = Ws + kPBM * 8;         // float [128]
    static constexpr int Bars = Wf + kPBM * 4;       // two stage mbarriers, drain
    static constexpr int Misc = Bars + 24;           // TMEM base, abort flag
    static constexpr int Size = Misc + 16;
};
static_assert(kPBM * kOutPitch * 4 <= 2 * kPBStage, "output staging inside the stages");
static_assert(PBSmem::Size <= 232448, "shared memory per CTA");

__global__ void __launch_bounds__(kPBThreads, 1) pos_bwd_tc_kernel(const __grid_constant__ PosBwdParams p)
{
    extern __shared__ __align__(1024) uint8_t sm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if ((smem_u32(sm) & 1023u) != 0) return;
    const int n0 = blockIdx.x * kPBN, m0 = blockIdx.y * kPBM;
    const int HD = p.H * p.D;
    double* Ws = reinterpret_cast<double*>(sm + PBSmem::Ws);
    float* Wf = reinterpret_cast<float*>(sm + PBSmem::Wf);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + PBSmem::Bars);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + PBSmem::Misc);
    int* abort_flag = reinterpret_cast<int*>(sm + PBSmem::Misc + 4);
    if (tid < kPBM / 2) {
        // the tile's 64 frequencies 10000^(-2k / d_model), each shared by columns 2k and 2k + 1
        const int k = (m0 >> 1) + tid;
        const double w = exp(-(2.0 * k) / static_cast<double>(p.d_model) * 9.210340371976182736);   // ln 10000
        Ws[2 * tid] = Ws[2 * tid + 1] = w;
        Wf[2 * tid] = Wf[2 * tid + 1] = static_cast<float>(w);
    }
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        mbar_init(&bar[2], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tmem_holder, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const WaitCtl wc{abort_flag, nullptr, kWaitTimeoutNs};

    // this CTA's share of the distances, whole chunks
    const int per = (p.n_rows + kPBChunk * gridDim.z - 1) / (kPBChunk * gridDim.z) * kPBChunk;
    const int d_lo = blockIdx.z * per, d_hi = min(p.n_rows, d_lo + per);
    const int nch = d_hi > d_lo ? (d_hi - d_lo + kPBChunk - 1) / kPBChunk : 0;
    constexpr double kTwoPi = 6.283185307179586476925;
    constexpr double kInvTwoPi = 0.159154943091895335768884;   // the quotient only picks the multiple of 2 pi
    constexpr uint32_t idesc = idesc_tf32(kPBM, kPBN, 0, 0);

    // generation roles.  A: the frequency kl = tid mod 64 of the tile (columns 2 kl, 2 kl + 1: its sine and
    // cosine from one sincosf), distances 4 (tid / 64) .. + 3 of the chunk; B: row tid mod 256 (column
    // n0 + tid mod 256 of dr), distances 16 (tid / 256) .. + 15 (each load coalesced across the warp)
    const int kl = tid & 63, ag = tid >> 6;
    const int ms = 2 * kl;                                // the sine's row; the cosine's is ms + 1
    const bool m_in = m0 + ms < p.d_model;
    const int bl = tid & (kPBN - 1), bq = tid >> 8;
    const int nt = n0 + bl;
    for (int c = 0; c < nch; ++c) {
        const int s = c & 1;
        uint8_t* st = sm + PBSmem::Stages + s * kPBStage;
        if (c >= 2) {                                     // the products that read this stage are done
            if (tid == 0) (void)mbar_spin(&bar[s], ((c - 2) >> 1) & 1, wc, 1);
            __syncthreads();
            if (*reinterpret_cast<volatile int*>(abort_flag)) break;
        }
        const int d0 = d_lo + c * kPBChunk;
        // ---- R^T chunk: A[ms][dl] = sin, A[ms + 1][dl] = cos, dl = 4 ag + e (anchor distance 4 ag)
        {
            const int dl = 4 * ag;
            const int da = d0 + dl;
            const double x = static_cast<double>(da) * Ws[ms];
            const float base = static_cast<float>(fma(-rint(x * kInvTwoPi), kTwoPi, x));
            float sh[4], sl[4], ch[4], cl[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float sv = 0.f, cv = 0.f;
                if (da + e < d_hi && m_in) sincosf(fmaf(static_cast<float>(e), Wf[ms], base), &sv, &cv);
                sh[e] = round_tf32(sv);
                sl[e] = sv - sh[e];
                ch[e] = round_tf32(cv);
                cl[e] = cv - ch[e];
            }
            const uint32_t offs = ms * 128 + ((((dl >> 2) ^ ms) & 7) << 4);
            const uint32_t offc = (ms + 1) * 128 + ((((dl >> 2) ^ (ms + 1)) & 7) << 4);
            *reinterpret_cast<float4*>(st + offs) = make_float4(sh[0], sh[1], sh[2], sh[3]);
            *reinterpret_cast<float4*>(st + kATile + offs) = make_float4(sl[0], sl[1], sl[2], sl[3]);
            *reinterpret_cast<float4*>(st + offc) = make_float4(ch[0], ch[1], ch[2], ch[3]);
            *reinterpret_cast<float4*>(st + kATile + offc) = make_float4(cl[0], cl[1], cl[2], cl[3]);
        }
        // ---- dr^T chunk: B[bl][dl] = dr[d0 + dl][n0 + bl], dl = 16 bq + 4 q + e
        {
            uint8_t* bhi = st + 2 * kATile + bl * 128;
            uint8_t* blo = bhi + kBTile;
            const float* src = p.dr + static_cast<int64_t>(d0) * HD + nt;
            const bool in_n = nt < HD;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int q4 = 4 * bq + q;
                float g[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int dl = 4 * q4 + e;
                    g[e] = (in_n && d0 + dl < d_hi) ? __ldg(src + static_cast<int64_t>(dl) * HD) : 0.f;
                }
                const float4 h4 = make_float4(round_tf32(g[0]), round_tf32(g[1]), round_tf32(g[2]), round_tf32(g[3]));
                const float4 l4 = make_float4(g[0] - h4.x, g[1] - h4.y, g[2] - h4.z, g[3] - h4.w);
                const uint32_t off = ((q4 ^ bl) & 7) << 4;
                *reinterpret_cast<float4*>(bhi + off) = h4;
                *reinterpret_cast<float4*>(blo + off) = l4;
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t sa = smem_u32(st);
            const uint64_t ahi = sdesc_k_sw128(sa), alo = sdesc_k_sw128(sa + kATile);
            const uint64_t bhi = sdesc_k_sw128(sa + 2 * kATile), blo = sdesc_k_sw128(sa + 2 * kATile + kBTile);
#pragma unroll
            for (int kk = 0; kk < kPBChunk / 8; ++kk) {
                umma_ss_tf32(tmem, ahi + 2 * kk, bhi + 2 * kk, idesc, (c > 0 || kk > 0) ? 1u : 0u);
                umma_ss_tf32(tmem, ahi + 2 * kk, blo + 2 * kk, idesc, 1u);
                umma_ss_tf32(tmem, alo + 2 * kk, bhi + 2 * kk, idesc, 1u);
            }
            umma_commit(&bar[s]);
        }
    }
    if (nch > 0 && !*reinterpret_cast<volatile int*>(abort_flag)) {
        if (tid == 0) (void)mbar_spin(&bar[(nch - 1) & 1], ((nch - 1) >> 1) & 1, wc, 2);
        __syncthreads();
    }
    // set only inside thread 0's bounded waits, read by all after the CTA barrier that follows them
    const bool failed = *reinterpret_cast<volatile int*>(abort_flag) != 0;
    if (nch > 0 && !failed) {
        tc_fence_after();
        // ---- the tile through shared memory: warp w reads lane quarter w mod 4, columns 64 (w / 4) ..
        float* out = reinterpret_cast<float*>(sm + PBSmem::Stages);
        {
            const int q = warp & 3, ch = warp >> 2;
            const int row = 32 * q + lane;
            const uint32_t tb = tmem + (static_cast<uint32_t>(32 * q) << 16) + 64u * ch;
#pragma unroll 1
            for (int k = 0; k < 2; ++k) {
                uint32_t v[32];
                tmem_ld32(tb + 32 * k, v);
                tmem_ld_wait();
                float4* dst = reinterpret_cast<float4*>(out + row * kOutPitch + 64 * ch + 32 * k);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    dst[e] = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                         __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
            }
        }
        __syncthreads();
        // ---- added into dW_R: warp w takes rows w, w + 16, ..; lane l columns 8 l .. 8 l + 7
        const bool vec_out = (p.ld_dw & 3) == 0 && (reinterpret_cast<uintptr_t>(p.dW) & 15u) == 0;
#pragma unroll 1
        for (int r = warp; r < kPBM; r += kPBThreads / 32) {
            const int mm = m0 + r;
            if (mm >= p.d_model) break;
            float* drow = p.dW + static_cast<int64_t>(mm) * p.ld_dw;
            const float* srow = out + r * kOutPitch;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int cl = 8 * lane + 4 * e, n = n0 + cl;
                const float4 v = *reinterpret_cast<const float4*>(srow + cl);
                if (vec_out && n + 3 < HD) {
                    atomicAdd(reinterpret_cast<float4*>(drow + n), v);
                } else {
                    if (n < HD) atomicAdd(drow + n, v.x);
                    if (n + 1 < HD) atomicAdd(drow + n + 1, v.y);
                    if (n + 2 < HD) atomicAdd(drow + n + 2, v.z);
                    if (n + 3 < HD) atomicAdd(drow + n + 3, v.w);
                }
            }
        }
    }
    if (failed && tid == 0) {
        // a wait gave up: every issued product completes before the TMEM is released
        int never = 0;
        const WaitCtl dw{&never, nullptr, 100000000ull};
        umma_commit(&bar[2]);
        (void)mbar_wait(&bar[2], 0, dw, 3);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

}  // namespace

// dW must be zero on entry (the distance shares add into it).
cudaError_t launch_pos_bwd_tc(const PosBwdParams& p, int sm_count, cudaStream_t s)
{
    static bool attr_done = false;
    if (!attr_done) {
        const cudaError_t e =
            cudaFuncSetAttribute(pos_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PBSmem::Size);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    const int tn = (p.H * p.D + kPBN - 1) / kPBN, tm = (p.d_model + kPBM - 1) / kPBM;
    const int chunks = (p.n_rows + kPBChunk - 1) / kPBChunk;
    // one CTA per SM (its shared memory): as many distance shares as fit one wave
    int splits = sm_count / (tn * tm);
    splits = splits < 1 ? 1 : (splits > chunks ? chunks : splits);
    if (splits > 65535) splits = 65535;
    pos_bwd_tc_kernel<<<dim3(tn, tm, splits), kPBThreads, PBSmem::Size, s>>>(p);
    return cudaGetLastError();
}

}  // namespace txl
