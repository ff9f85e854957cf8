// txl_pos.cu -- relative position key vectors r[delta][h][d] = sum_m R_delta[m] W_R[m][h*D+d].
//
//   R_delta[2k] = sin(delta * w_k), R_delta[2k+1] = cos(delta * w_k), w_k = 10000^(-2k/d_model)
//   ("跨窗口的相对位置编码" §2; "Transformer-XL 和相对位置编码" §2.3.2), projected by W_R (the
//   position projection W_{k,R}, r_proj without bias in "TransformerXL 相对位置编码" §3.1).
//
// bf16 path: one tcgen05 GEMM per 128 x 128 output tile.  The A operand (128 distances x 64
// sinusoid columns) is generated on chip by eight warps straight into the 128-byte-swizzled
// shared-memory layout the tensor core reads; it never exists in HBM.  W_R tiles arrive by TMA.
// Generation advances along the distance axis by angle addition,
//   angle((delta + 1) w) = angle(delta w) + angle(w),
// so each thread evaluates two sines/cosines per K tile and each further element costs one
// complex multiply.  Sixteen generator warps (four per scheduler) keep the short dependency
// chains of the generation overlapped; warp 16 issues TMA, warp 17 issues UMMA (fp32
// accumulator in TMEM).
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
constexpr int kPosStages = 6;
constexpr int kPosGenWarps = 16;                            // generate the A operand + epilogue
constexpr int kPosTmaWarp = kPosGenWarps;                   // W_R tiles
constexpr int kPosMmaWarp = kPosGenWarps + 1;               // UMMA issue, TMEM owner
constexpr int kPosThreads = 32 * (kPosGenWarps + 2);
constexpr int kTileBytes = 128 * 128;       // 16 KB: 128 rows x 128 B (A tile) or 2 x 8 KB (B)
constexpr int kRowsPerWarp = 128 / kPosGenWarps;            // distances one generator warp covers

struct PosSmem {
    // offsets from a 1024-byte aligned base
    static constexpr int A = 0;                                   // kPosStages x 16 KB
    static constexpr int Bt = A + kPosStages * kTileBytes;        // kPosStages x 16 KB
    static constexpr int Freq = Bt + kPosStages * kTileBytes;     // float [kMaxDModel / 2]
    static constexpr int Bars = Freq + kMaxDModel / 2 * 4;
    static constexpr int NumBars = 3 * kPosStages + 2;
    static constexpr int Misc = Bars + NumBars * 8;                // tmem base, abort flag
    static constexpr int Size = Misc + 16;
};

// sin and cos of an angle of moderate size (|x| < 2^20): Cody-Waite reduction modulo 2 pi with
// a two-constant split of 2 pi (fp32(2 pi) and the fp32 remainder), then the hardware sine and
// cosine on [-pi, pi], whose absolute error there is about 2^-21.
__device__ __forceinline__ void sincos_reduced(float x, float& sv, float& cv)
{
    constexpr float kTwoPiHi = 6.28318548202514648f;        // fp32(2 pi)
    constexpr float kTwoPiLo = -1.74845553146951717e-07f;   // fp32(2 pi - kTwoPiHi)
    constexpr float kInvTwoPi = 0.159154936671257019f;
    const float n = rintf(x * kInvTwoPi);
    float r = fmaf(-n, kTwoPiHi, x);
    r = fmaf(-n, kTwoPiLo, r);
    sv = __sinf(r);
    cv = __cosf(r);
}

// Grid: (row tiles of 128 distances, column tiles of 128 (h, d) columns).  Per 64-column K tile
// of the sinusoid, generator lane k owns frequency w_k of the tile and warp g the 8 distances
// delta0 + 8 g + b, b = 0..7: it evaluates the angle of the first of them and of one step w_k,
// then advances by rotation, (sin, cos)(x + w) = (s cw + c sw, c cw - s sw), writing each bf16
// (sin, cos) pair as one 32-bit word into the 128-byte-swizzled K-major layout the tensor core
// reads (a warp writes one full 128-byte row per store: no bank conflicts).
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
    float* freq = reinterpret_cast<float*>(smem + PosSmem::Freq);

    if ((smem_u32(smem) & 1023u) != 0) {        // the swizzled layouts need a 1 KB aligned base
        if (tid == 0 && p.err_flag) atomicCAS(p.err_flag, 0, TXL_ERR_ALIGNMENT);
        return;
    }
    const int half = p.d_model >> 1;
    // w_k = 10000^(-2k/d_model) = 2^(k * log2_freq_step)
    for (int k = tid; k < half; k += kPosThreads) freq[k] = exp2f(static_cast<float>(k) * p.log2_freq_step);
    if (tid == 0) {
        for (int s = 0; s < kPosStages; ++s) {
            mbar_init(&full_a[s], kPosGenWarps);
            mbar_init(&full_b[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kPosMmaWarp) tmem_alloc(tmem_holder, 128);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const WaitCtl wc{abort_flag, p.err_flag, kWaitTimeoutNs};

    const int delta0 = blockIdx.x * 128;
    const int n0 = blockIdx.y * 128;
    const int nk = p.n_ktiles;

    if (warp == kPosTmaWarp) {
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
    } else if (warp == kPosMmaWarp) {
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
        // ------------------------------------------------ generators (warps 0-7)
        const int row0 = kRowsPerWarp * warp;                 // first local distance of the warp
        const float first = static_cast<float>(delta0 + row0);
        bool ok = true;
        for (int kt = 0; kt < nk && ok; ++kt) {
            const int s = kt % kPosStages;
            const int kg = kt * 32 + lane;
            float sv = 0.f, cv = 0.f, sw = 0.f, cw = 1.f;     // frequencies past d_model/2: zero
            if (kg < half) {
                const float w = freq[kg];
                sincos_reduced(first * w, sv, cv);
                sincos_reduced(w, sw, cw);
            }
            ok = warp_wait(&empty[s], ((kt / kPosStages) & 1) ^ 1, wc, 6);
            if (!ok) break;
            const uint32_t tile = smem_u32(smem + PosSmem::A + s * kTileBytes);
#pragma unroll
            for (int b = 0; b < kRowsPerWarp; ++b) {
                const int row = row0 + b;
                const uint32_t addr = tile + row * 128 + ((((lane >> 2) ^ (row & 7)) << 4) | ((lane & 3) << 2));
                asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(pack_bf16x2(sv, cv)) : "memory");
                const float sn = fmaf(sv, cw, cv * sw);
                const float cn = fmaf(cv, cw, -(sv * sw));
                sv = sn;
                cv = cn;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&full_a[s]);
        }
        if (ok) ok = warp_wait(acc_full, 0, wc, 7);
        if (ok) {
            // epilogue: warp g reads TMEM lanes 32 (g mod 4) .. +32, columns 32 (g / 4) .. +32
            tc_fence_after();
            const int li = 32 * (warp & 3) + lane;
            const int delta = delta0 + li;
            const int HD = p.H * p.D;
            const bool dense = (p.ld_r == p.D) && (HD % 8 == 0);
            __nv_bfloat16* rrow = static_cast<__nv_bfloat16*>(p.r) + static_cast<int64_t>(delta) * p.H * p.ld_r;
#pragma unroll 1
            constexpr int kColBlocks = 16 / kPosGenWarps;          // 32-column blocks per warp
            for (int cb = (warp >> 2) * kColBlocks; cb < ((warp >> 2) + 1) * kColBlocks; ++cb) {
                uint32_t v[32];
                tmem_ld32(tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + cb * 32, v);
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
    if (warp == kPosMmaWarp) {
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
