// txl_pos.cu -- relative position key vectors r[delta][h][d] = sum_m R_delta[m] W_R[m][h*D+d].
//
//   R_delta[2k] = sin(delta * w_k), R_delta[2k+1] = cos(delta * w_k), w_k = 10000^(-2k/d_model)
//   ("跨窗口的相对位置编码" §2; "Transformer-XL 和相对位置编码" §2.3.2), projected by W_R (the
//   position projection W_{k,R}, r_proj without bias in "TransformerXL 相对位置编码" §3.1).
//
// bf16 path: one tcgen05 GEMM per 128 x 128 output tile.  The A operand (128 distances x 64
// sinusoid columns) is generated on chip by four warps straight into the 128-byte-swizzled
// shared-memory layout the tensor core reads; it never exists in HBM.  W_R tiles arrive by TMA.
// Generation uses angle addition from two small tables per K tile:
//   angle(delta0 + 16a + b) = angle(delta0 + 16a) + angle(b),  a in [0,8), b in [0,16)
// so each CTA evaluates 768 sin/cos pairs per 64-column K tile instead of 4096, and each element
// costs one complex multiply.  Warp 4 issues TMA, warp 5 issues UMMA (fp32 accumulator in TMEM).
#include <cmath>

#include <cuda_bf16.h>

#include "txl_internal.h"
#include "txl_ptx.cuh"

namespace txl {

namespace {

// ------------------------------------------------------------------------------- fp32 SIMT
// One CTA per distance row: R_delta is evaluated in double precision and rounded once to fp32,
// then every (h, d) column is a dot product over d_model.
constexpr int kPosF32Threads = 256;

__global__ void __launch_bounds__(kPosF32Threads) pos_gen_f32_kernel(PosGenF32Params p)
{
    extern __shared__ float R[];
    const int delta = blockIdx.x;
    for (int k = threadIdx.x; k < p.d_model / 2; k += blockDim.x) {
        const double w = pow(10000.0, -(2.0 * k) / static_cast<double>(p.d_model));
        const double a = static_cast<double>(delta) * w;
        R[2 * k] = static_cast<float>(sin(a));
        R[2 * k + 1] = static_cast<float>(cos(a));
    }
    __syncthreads();
    const int HD = p.H * p.D;
    for (int n = threadIdx.x; n < HD; n += blockDim.x) {
        float acc = 0.f;
        for (int m = 0; m < p.d_model; ++m) acc = fmaf(R[m], p.W[static_cast<int64_t>(m) * p.ld_w + n], acc);
        const int h = n / p.D, d = n - (n / p.D) * p.D;
        p.r[(static_cast<int64_t>(delta) * p.H + h) * p.ld_r + d] = acc;
    }
}

// ------------------------------------------------------------------------------- bf16 tcgen05
constexpr int kPosStages = 4;
constexpr int kPosThreads = 192;            // warps 0-3 generate + epilogue, 4 TMA, 5 UMMA
constexpr int kTileBytes = 128 * 128;       // 16 KB: 128 rows x 128 B (A tile) or 2 x 8 KB (B)

struct PosSmem {
    // offsets from a 1024-byte aligned base
    static constexpr int A = 0;                                   // kPosStages x 16 KB
    static constexpr int Bt = A + kPosStages * kTileBytes;        // kPosStages x 16 KB
    static constexpr int TabBase = Bt + kPosStages * kTileBytes;  // float2 [32 k][8 a]
    static constexpr int TabStep = TabBase + 32 * 8 * 8;          // float2 [32 k][16 b]
    static constexpr int Bars = TabStep + 32 * 16 * 8;
    static constexpr int NumBars = 3 * kPosStages + 2;
    static constexpr int Misc = Bars + NumBars * 8;                // tmem base, abort flag
    static constexpr int Size = Misc + 16;
};

__global__ void __launch_bounds__(kPosThreads, 1) pos_gen_tc_kernel(const __grid_constant__ PosGenTcParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    uint64_t* full_a = reinterpret_cast<uint64_t*>(smem + PosSmem::Bars);
    uint64_t* full_b = full_a + kPosStages;
    uint64_t* empty = full_b + kPosStages;
    uint64_t* acc_full = empty + kPosStages;
    uint64_t* drain = acc_full + 1;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + PosSmem::Misc);
    int* abort_flag = reinterpret_cast<int*>(smem + PosSmem::Misc + 4);

    if ((smem_u32(smem) & 1023u) != 0) {        // the swizzled layouts need a 1 KB aligned base
        if (tid == 0 && p.err_flag) atomicCAS(p.err_flag, 0, TXL_ERR_ALIGNMENT);
        return;
    }
    if (tid == 0) {
        for (int s = 0; s < kPosStages; ++s) {
            mbar_init(&full_a[s], 4);
            mbar_init(&full_b[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 5) tmem_alloc(tmem_holder, 128);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const WaitCtl wc{abort_flag, p.err_flag, kWaitTimeoutNs};

    const int delta0 = blockIdx.x * 128;
    const int n0 = blockIdx.y * 128;
    const int nk = p.n_ktiles;

    if (warp == 4) {
        // ------------------------------------------------ TMA producer: W_R tiles
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_w);
            int issued = 0;
            for (int kt = 0; kt < nk; ++kt) {
                const int s = kt % kPosStages;
                if (!mbar_wait(&empty[s], ((kt / kPosStages) & 1) ^ 1, wc, 1)) break;
                mbar_expect_tx(&full_b[s], kTileBytes);
                uint8_t* dst = smem + PosSmem::Bt + s * kTileBytes;
                tma_load_2d(dst, &p.tm_w, n0, kt * 64, &full_b[s]);
                tma_load_2d(dst + 8192, &p.tm_w, n0 + 64, kt * 64, &full_b[s]);
                ++issued;
            }
            // after an abort, wait (bounded) until the loads already issued have landed so no
            // TMA write reaches shared memory after the CTA exits
            if (*abort_flag) {
                int never = 0;
                const WaitCtl drain_wc{&never, nullptr, 100000000ull};
                for (int kt = issued - kPosStages; kt < issued; ++kt)
                    if (kt >= 0) (void)mbar_wait(&full_b[kt % kPosStages], (kt / kPosStages) & 1, drain_wc, 2);
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------ UMMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(128, 128, 0, 1);
            bool ok = true;
            for (int kt = 0; kt < nk && ok; ++kt) {
                const int s = kt % kPosStages;
                const uint32_t par = (kt / kPosStages) & 1;
                ok = mbar_wait(&full_a[s], par, wc, 3) && mbar_wait(&full_b[s], par, wc, 4);
                if (!ok) break;
                tc_fence_after();
                const uint32_t a_base = smem_u32(smem + PosSmem::A + s * kTileBytes);
                const uint32_t b_base = smem_u32(smem + PosSmem::Bt + s * kTileBytes);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t ad = sdesc_k_sw128(a_base + kk * 32);
                    const uint64_t bd = sdesc_mn_sw128(b_base + kk * 2048, 8192);
                    umma_ss(tmem, ad, bd, idesc, (kt > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(&empty[s]);
            }
            umma_commit(ok ? acc_full : drain);
            if (!ok) {                                   // every issued UMMA done before dealloc
                int never = 0;
                const WaitCtl drain_wc{&never, nullptr, 100000000ull};
                (void)mbar_wait(drain, 0, drain_wc, 5);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ generators (warps 0-3), row = tid
        float2* tab_base = reinterpret_cast<float2*>(smem + PosSmem::TabBase);   // [k][a]
        float2* tab_step = reinterpret_cast<float2*>(smem + PosSmem::TabStep);   // [k][b]
        const int a = tid >> 4, b = tid & 15;
        const int half = p.d_model >> 1;
        bool ok = true;
        // Every generator warp runs all nk iterations and both named barriers of each, even
        // after an abort (work is then skipped), so no warp can be left at a barrier.
        for (int kt = 0; kt < nk; ++kt) {
            const int s = kt % kPosStages;
            named_bar_sync(1, 128);                      // previous tables fully consumed
            if (ok) {
                for (int e = tid; e < 32 * 24; e += 128) {   // angle tables of this K tile
                    int kl, mult;
                    float2* dst;
                    if (e < 256) { kl = e >> 3; mult = delta0 + 16 * (e & 7); dst = tab_base + e; }
                    else { kl = (e - 256) >> 4; mult = (e - 256) & 15; dst = tab_step + (e - 256); }
                    const int kg = kt * 32 + kl;
                    float sv = 0.f, cv = 1.f;
                    if (kg < half) sincosf(static_cast<float>(mult) * p.inv_freq[kg], &sv, &cv);
                    *dst = make_float2(sv, cv);
                }
            }
            named_bar_sync(1, 128);
            if (ok) ok = warp_wait(&empty[s], ((kt / kPosStages) & 1) ^ 1, wc, 6);
            if (!ok) continue;
            uint8_t* row = smem + PosSmem::A + s * kTileBytes + tid * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {                // 16-byte chunk c = frequencies 4c..4c+3
                uint32_t w[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int kl = 4 * c + j;
                    const int kg = kt * 32 + kl;
                    const float2 x = tab_base[kl * 8 + a];
                    const float2 y = tab_step[kl * 16 + b];
                    float sv = fmaf(x.x, y.y, x.y * y.x);          // sin(A+B)
                    float cv = fmaf(x.y, y.y, -(x.x * y.x));       // cos(A+B)
                    if (kg >= half) { sv = 0.f; cv = 0.f; }
                    w[j] = pack_bf16x2(sv, cv);
                }
                const int pc = c ^ (tid & 7);
                *reinterpret_cast<uint4*>(row + pc * 16) = make_uint4(w[0], w[1], w[2], w[3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&full_a[s]);
        }
        if (ok) {
            ok = warp_wait(acc_full, 0, wc, 7);
        }
        if (ok) {
            tc_fence_after();
            const int delta = delta0 + tid;
            const int HD = p.H * p.D;
            const bool dense = (p.ld_r == p.D) && (HD % 8 == 0);
            __nv_bfloat16* rrow = static_cast<__nv_bfloat16*>(p.r) + static_cast<int64_t>(delta) * p.H * p.ld_r;
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t v[32];
                tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + cb * 32, v);
                tmem_ld_wait();
                if (delta >= p.n_rows) continue;
                const int nb = n0 + cb * 32;
                if (dense && nb + 32 <= HD) {
                    uint4* dst = reinterpret_cast<uint4*>(rrow + nb);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t w[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            w[j] = pack_bf16x2(__uint_as_float(v[8 * q + 2 * j]), __uint_as_float(v[8 * q + 2 * j + 1]));
                        dst[q] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                } else {
                    for (int j = 0; j < 32; ++j) {
                        const int n = nb + j;
                        if (n >= HD) break;
                        const int h = n / p.D, d = n - h * p.D;
                        rrow[static_cast<int64_t>(h) * p.ld_r + d] = __float2bfloat16_rn(__uint_as_float(v[j]));
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
}

}  // namespace

cudaError_t launch_pos_gen_f32(const PosGenF32Params& p, cudaStream_t s)
{
    if (p.n_rows == 0) return cudaSuccess;
    const size_t smem = sizeof(float) * p.d_model;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(pos_gen_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    pos_gen_f32_kernel<<<p.n_rows, kPosF32Threads, smem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_pos_gen_tc(const PosGenTcParams& p, cudaStream_t s)
{
    if (p.n_rows == 0) return cudaSuccess;
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(pos_gen_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             PosSmem::Size);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    dim3 grid((p.n_rows + 127) / 128, (p.H * p.D + 127) / 128);
    pos_gen_tc_kernel<<<grid, kPosThreads, PosSmem::Size, s>>>(p);
    return cudaGetLastError();
}

}  // namespace txl
