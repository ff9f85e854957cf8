// txl_pos.cu -- relative position key vectors r[delta][h][d] = sum_m R_delta[m] W_R[m][h*D+d].
//
//   R_delta[2k] = sin(delta * w_k), R_delta[2k+1] = cos(delta * w_k), w_k = 10000^(-2k/d_model)
//   ("跨窗口的相对位置编码" §2; "Transformer-XL 和相对位置编码" §2.3.2), projected by W_R (the
//   position projection W_{k,R}, r_proj without bias in "TransformerXL 相对位置编码" §3.1).
//
// bf16 path: one tcgen05 GEMM per 128 x 128 output tile, r_tile = R_tile . W_R_tile.  The A
// operand (128 distances x 64 sinusoid columns per K tile) is generated on chip straight into
// tensor memory, which the UMMA reads as its A operand; it never exists in HBM or shared memory,
// so shared memory carries only the W_R tiles (TMA writes, UMMA reads).  Generation advances
// along the distance axis by angle addition, angle((delta + 8) w) = angle(delta w) + angle(8 w):
// a thread evaluates one sine/cosine per frequency and K tile and gets the three further
// distances it owns by complex multiplication.
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
constexpr int kPosGenWarps = 8;                             // generate the A operand + epilogue
constexpr int kPosTmaWarp = kPosGenWarps;                   // W_R tiles
constexpr int kPosMmaWarp = kPosGenWarps + 1;               // UMMA issue, TMEM owner
constexpr int kPosThreads = 32 * (kPosGenWarps + 2);
constexpr int kPosGenThreads = 32 * kPosGenWarps;
constexpr int kPosACols = kPosKTile / 2;                    // TMEM columns of one A stage (bf16 pairs)
constexpr int kStageBytes = 128 * kPosKTile * 2;            // one W_R stage: 2 x (kPosKTile k x 64 n) bf16
constexpr uint32_t kPosColAcc = 0;                          // TMEM: fp32 accumulator, 128 columns
constexpr uint32_t kPosColA = 128;                          // TMEM: A stages, kPosACols columns each
constexpr uint32_t kPosTmemCols = 512;
static_assert(kPosColA + kPosACols * kPosStages <= kPosTmemCols, "A stages exceed the TMEM allocation");
static_assert(kPosACols == 64, "the generator mapping covers 64 columns per stage");

struct PosSmem {
    // offsets from a 1024-byte aligned base
    static constexpr int Bt = 0;                                  // kPosStages x 32 KB (W_R)
    static constexpr int Out = Bt;                                // epilogue staging, 32 KB, reuses Bt
    static constexpr int Freq = Bt + kPosStages * kStageBytes;    // float2 [kMaxDModel / 4]: w of a pair
    static constexpr int Step = Freq + kMaxDModel / 2 * 4;        // float4 [kMaxDModel / 4]: sin, cos 8 w
    static constexpr int Bars = Step + kMaxDModel / 2 * 8;
    static constexpr int NumBars = 3 * kPosStages + 2;
    static constexpr int Misc = Bars + NumBars * 8;                // tmem base, abort flag
    static constexpr int Size = Misc + 16;
};
// more than half of an SM's shared memory: one CTA per SM, so the 512-column TMEM allocation
// never waits for another CTA of this kernel
static_assert(PosSmem::Size > 116 * 1024, "two CTAs could share an SM");

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

// tcgen05.st of 16 TMEM lanes x 8 columns: thread t writes lanes t/4 (a0, a1) and t/4 + 8 (b0, b1),
// columns 2 (t mod 4) and 2 (t mod 4) + 1.
__device__ __forceinline__ void tmem_st_16x256b(uint32_t taddr, uint32_t a0, uint32_t a1, uint32_t b0, uint32_t b1)
{
    asm volatile("tcgen05.st.sync.aligned.16x256b.x1.b32 [%0], {%1, %2, %3, %4};"
                 ::"r"(taddr), "r"(a0), "r"(a1), "r"(b0), "r"(b1) : "memory");
}

// Epilogue of the output tile when r rows are dense (ld_r == D, 16-byte aligned): warp g reads
// TMEM lanes 32 (g mod 4) .. +32, columns 64 (g / 4) .. +64, into a shared staging tile (row li at
// li * 256 bytes, 16-byte chunk c stored at chunk c ^ (li mod 16)), then the generator warps
// store it row-contiguously (a warp writes two full 256-byte row segments per instruction).
__device__ __forceinline__ void pos_store_dense(const PosGenTcParams& p, uint8_t* smem, uint32_t tmem, int warp,
                                                int lane, int delta0, int n0)
{
    const int li = 32 * (warp & 3) + lane;
    const uint32_t stage = smem_u32(smem + PosSmem::Out);
#pragma unroll 1
    for (int cb = 2 * (warp >> 2); cb < 2 * (warp >> 2) + 2; ++cb) {
        uint32_t v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + kPosColAcc + cb * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                w[j] = pack_bf16x2(__uint_as_float(v[8 * q + 2 * j]), __uint_as_float(v[8 * q + 2 * j + 1]));
            const int chunk = 4 * cb + q;
            const uint32_t addr = stage + li * 256 + ((chunk ^ (li & 15)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                         "r"(w[3]) : "memory");
        }
    }
    named_bar_sync(1, kPosGenThreads);
    const int HD = p.H * p.D;
    const int chunk = lane & 15;
    const int n = n0 + 8 * chunk;
#pragma unroll 1
    for (int it = 0; it < 128 / (2 * kPosGenWarps); ++it) {
        const int row = (128 / kPosGenWarps) * warp + 2 * it + (lane >> 4);
        const int delta = delta0 + row;
        if (delta >= p.n_rows || n >= HD) continue;
        uint32_t w0, w1, w2, w3;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                     : "r"(stage + row * 256 + ((chunk ^ (row & 15)) << 4)));
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.r) + static_cast<int64_t>(delta) * HD + n;
        *reinterpret_cast<uint4*>(dst) = make_uint4(w0, w1, w2, w3);
    }
}

// Epilogue for any r layout: element stores straight from TMEM (rows past n_rows are skipped).
__device__ __forceinline__ void pos_store_strided(const PosGenTcParams& p, uint32_t tmem, int warp, int lane,
                                                  int delta0, int n0)
{
    const int li = 32 * (warp & 3) + lane;
    const int delta = delta0 + li;
    const int HD = p.H * p.D;
    __nv_bfloat16* rrow = static_cast<__nv_bfloat16*>(p.r) + static_cast<int64_t>(delta) * p.H * p.ld_r;
#pragma unroll 1
    for (int cb = 2 * (warp >> 2); cb < 2 * (warp >> 2) + 2; ++cb) {
        uint32_t v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + kPosColAcc + cb * 32, v);
        tmem_ld_wait();
        if (delta >= p.n_rows) continue;
        for (int j = 0; j < 32; ++j) {
            const int n = n0 + cb * 32 + j;
            if (n >= HD) break;
            const int h = n / p.D, d = n - h * p.D;
            rrow[static_cast<int64_t>(h) * p.ld_r + d] = __float2bfloat16_rn(__uint_as_float(v[j]));
        }
    }
}

// Grid: (row tiles of 128 distances, column tiles of 128 (h, d) columns); 320 threads.
//   warps 0-7 : generate the A operand into TMEM, then the epilogue.  A K tile is 128 sinusoid
//               columns: TMEM column c of a stage holds the bf16 pair (sin, cos) of frequency
//               64 kt + c.  Warp g = q + 4 hh covers the TMEM lanes (distances) 32 q .. 32 q + 31 and
//               the stage columns 32 hh .. 32 hh + 31.  In the 16x256b store layout lane t of the
//               warp owns distances 32 q + t/4 + {0, 8, 16, 24} and columns 32 hh + 8 jj + 2 (t mod 4)
//               + e (jj < 4, e < 2): per frequency one sine/cosine of the first distance, then three
//               rotations by 8 w.
//   warp 8    : TMA loads of W_R tiles (MN-major B operand, two 64 n x 128 k boxes per stage).
//   warp 9    : TMEM allocation and UMMA issue (A from TMEM, B from shared memory).
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
    float2* freq2 = reinterpret_cast<float2*>(smem + PosSmem::Freq);
    float4* step4 = reinterpret_cast<float4*>(smem + PosSmem::Step);

    pdl_launch_dependents();
    if ((smem_u32(smem) & 1023u) != 0) {        // the swizzled layout needs a 1 KB aligned base
        pdl_wait();
        if (tid == 0 && p.err_flag) atomicCAS(p.err_flag, 0, TXL_ERR_ALIGNMENT);
        return;
    }
    if (tid == 32 * kPosTmaWarp) {
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
    if (warp == kPosMmaWarp) tmem_alloc(tmem_holder, kPosTmemCols);
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
            pdl_wait();                                  // W_R may come from the previous grid
            int issued = 0;
            int s = 0;
            uint32_t par = 0;
            for (int kt = 0; kt < nk; ++kt) {
                if (!mbar_wait(&empty[s], par ^ 1u, wc, 1)) break;
                mbar_expect_tx(&full_b[s], kStageBytes);
                uint8_t* dst = smem + PosSmem::Bt + s * kStageBytes;
                tma_load_2d(dst, &p.tm_w, n0, kt * kPosKTile, &full_b[s]);
                tma_load_2d(dst + kStageBytes / 2, &p.tm_w, n0 + 64, kt * kPosKTile, &full_b[s]);
                ++issued;
                if (++s == kPosStages) {
                    s = 0;
                    par ^= 1u;
                }
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
            // stage 0's descriptor; a stage or K step moves only the 14-bit start-address field
            // (address / 16), which stays below 2^14 for every offset used here
            const uint64_t b_desc0 = sdesc_mn_sw128(smem_u32(smem + PosSmem::Bt), kStageBytes / 2);
            bool ok = true;
            int s = 0;
            uint32_t par = 0;
            for (int kt = 0; kt < nk && ok; ++kt) {
                ok = mbar_wait(&full_a[s], par, wc, 3) && mbar_wait(&full_b[s], par, wc, 4);
                if (!ok) break;
                tc_fence_after();
                const uint64_t bd = b_desc0 + static_cast<uint64_t>(s * (kStageBytes >> 4));
                const uint32_t a_col = tmem + kPosColA + kPosACols * s;
#pragma unroll
                for (int kk = 0; kk < kPosKTile / 16; ++kk)
                    umma_ts(tmem + kPosColAcc, a_col + 8 * kk, bd + 128 * kk, idesc, (kt > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&empty[s]);
                if (++s == kPosStages) {
                    s = 0;
                    par ^= 1u;
                }
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
        // ------------------------------------------------ generators
        const int half = p.d_model >> 1;
        // per frequency pair (2 kp, 2 kp + 1): w_k = 10000^(-2k/d_model) = 2^(k log2_freq_step) and
        // the rotation by 8 distances {sin 8 w_a, sin 8 w_b, cos 8 w_a, cos 8 w_b}, for every
        // frequency of the K tiles.  Frequencies past d_model/2 get w = 0: their A columns are
        // finite and meet W_R rows past d_model, which the TMA loads as zeros.
        const int n_pairs = nk * kPosACols / 2;
        for (int kp = tid; kp < n_pairs; kp += kPosGenThreads) {
            float w[2], s8[2], c8[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int k = 2 * kp + e;
                w[e] = k < half ? exp2f(static_cast<float>(k) * p.log2_freq_step) : 0.f;
                sincos_reduced(8.f * w[e], s8[e], c8[e]);
            }
            freq2[kp] = make_float2(w[0], w[1]);
            step4[kp] = make_float4(s8[0], s8[1], c8[0], c8[1]);
        }
        named_bar_sync(1, kPosGenThreads);
        const int q = warp & 3, hh = warp >> 2;
        const float first = static_cast<float>(delta0 + 32 * q + (lane >> 2));
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q) << 16);
        const int col0 = 32 * hh + 2 * (lane & 3);               // column of (jj, e) = (0, 0)
        const uint64_t minus1 = f2_pack(-1.f, -1.f);
        bool ok = true;
        int s = 0;
        uint32_t par = 0;
        for (int kt = 0; kt < nk && ok; ++kt) {
            // v[m][2 jj + e]: distance first + 8 m, frequency 64 kt + col0 + 8 jj + e.  The two
            // frequencies of a pair advance together in packed fp32x2 arithmetic.
            uint32_t v[4][8];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int kp = (kPosACols * kt + col0 + 8 * jj) >> 1;
                const float2 w2 = freq2[kp];
                const float4 st = step4[kp];
                float sa, ca, sb, cb;
                sincos_reduced(first * w2.x, sa, ca);
                sincos_reduced(first * w2.y, sb, cb);
                uint64_t S = f2_pack(sa, sb), C = f2_pack(ca, cb);
                const uint64_t S8 = f2_pack(st.x, st.y), C8 = f2_pack(st.z, st.w);
                const uint64_t N8 = f2_mul(S8, minus1);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    float s0, s1, c0, c1;
                    f2_unpack(S, s0, s1);
                    f2_unpack(C, c0, c1);
                    v[m][2 * jj] = pack_bf16x2(s0, c0);
                    v[m][2 * jj + 1] = pack_bf16x2(s1, c1);
                    if (m < 3) {
                        // (sin, cos)(x + 8 w) = (s c8 + c s8, c c8 - s s8)
                        const uint64_t Sn = f2_fma(S, C8, f2_mul(C, S8));
                        C = f2_fma(C, C8, f2_mul(S, N8));
                        S = Sn;
                    }
                }
            }
            ok = warp_wait(&empty[s], par ^ 1u, wc, 6);
            if (!ok) break;
            const uint32_t a_col = kPosColA + kPosACols * s + 32 * hh;
#pragma unroll
            for (int g = 0; g < 2; ++g)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    tmem_st_16x256b(lane_base + (static_cast<uint32_t>(16 * g) << 16) + a_col + 8 * jj,
                                    v[2 * g][2 * jj], v[2 * g][2 * jj + 1], v[2 * g + 1][2 * jj],
                                    v[2 * g + 1][2 * jj + 1]);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&full_a[s]);
            if (++s == kPosStages) {
                s = 0;
                par ^= 1u;
            }
        }
        if (ok) ok = warp_wait(acc_full, 0, wc, 7);
        pdl_wait();                                      // the previous grid may still read r
        // every generator warp reaches the staging barrier of the dense epilogue, or none does
        ok = named_bar_and(1, kPosGenThreads, ok);
        if (ok) {
            tc_fence_after();
            if (p.dense) pos_store_dense(p, smem, tmem, warp, lane, delta0, n0);
            else pos_store_strided(p, tmem, warp, lane, delta0, n0);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kPosMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kPosTmemCols);
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
    return launch_dependent(pos_gen_tc_kernel, grid, dim3(kPosThreads), PosSmem::Size, s, p);
}

}  // namespace txl
