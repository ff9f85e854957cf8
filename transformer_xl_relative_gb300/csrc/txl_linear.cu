// txl_linear.cu -- Y = X . W on the 5th-generation tensor cores: the content projections of a
// Transformer-XL attention layer.  Q = h W_q from the current segment and K = h~ W_k, V = h~ W_v
// from the memory-extended hidden states h~ = [SG(h_mem) o h] ("Transformer-XL 和相对位置编码"
// §2.3.1), and the output projection o_proj over the concatenated heads ("TransformerXL 相对位置编码"
// §3.1; q_proj, k_proj, v_proj and o_proj there are linear maps without bias).
//
// bf16 X [m][k] (row stride ld_x), bf16 W [k][n] (row stride ld_w), fp32 accumulation in TMEM,
// bf16 Y [m][n] (row stride ld_y).  Persistent: one CTA per SM walks the 128 x 256 output tiles
// (tile t -> row block t / tiles_n, column block t mod tiles_n, so CTAs of one wave share X rows in
// L2).  Warp 0 streams 64-wide K slices by TMA (X K-major, W MN-major, both 128-byte swizzled) into
// a 4-stage ring; warp 1 issues 128 x 256 x 16 UMMAs into one of two TMEM accumulators; warps 2-5
// drain the other accumulator (TMEM lane quarter = warp mod 4) to bf16 rows of Y while the next
// tile accumulates.  Tails are handled by the TMA zero fill (rows, columns and K past the
// extents read as zeros) and by masking the stores.  Every CTA loads its own X and W boxes; CTAs
// of one wave that share a row or column block find it in L2.
#include <cuda_bf16.h>

#include "txl_internal.h"
#include "txl_ptx.cuh"

namespace txl {

namespace {

constexpr int kLinStages = 4;
constexpr int kLinThreads = 192;                  // TMA, MMA, 4 epilogue warps
constexpr int kLinTmaWarp = 0, kLinMmaWarp = 1;
constexpr int kABytes = 128 * 64 * 2;             // X slice: 128 rows x 64 k
constexpr int kBBytes = 64 * 256 * 2;             // W slice: 64 k x 256 n (four 64-column boxes)
constexpr int kStageBytes = kABytes + kBBytes;
constexpr uint32_t kLinTmemCols = 512;            // two 128 x 256 fp32 accumulators

constexpr int kOutBytes = 32 * 128;              // one epilogue warp's staging: 32 rows x 64 bf16

struct LinSmem {
    static constexpr int Stages = 0;
    static constexpr int Out = Stages + kLinStages * kStageBytes;     // 4 warps x 2 buffers, 1 KB aligned
    static constexpr int Bars = Out + 8 * kOutBytes;
    static constexpr int NumBars = 2 * kLinStages + 4 + 1;
    static constexpr int Misc = Bars + NumBars * 8;           // tmem base, abort flag
    static constexpr int Size = Misc + 16;
};

__global__ void __launch_bounds__(kLinThreads, 1) linear_kernel(const __grid_constant__ LinearParams p)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    pdl_launch_dependents();
    if ((smem_u32(smem) & 1023u) != 0) {
        pdl_wait();
        if (tid == 0 && p.err_flag) atomicCAS(p.err_flag, 0, TXL_ERR_ALIGNMENT);
        return;
    }
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + LinSmem::Bars);
    uint64_t* empty = full + kLinStages;
    uint64_t* acc_full = empty + kLinStages;         // [2]
    uint64_t* acc_empty = acc_full + 2;              // [2]
    uint64_t* drain = acc_empty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + LinSmem::Misc);
    int* abort_flag = reinterpret_cast<int*>(smem + LinSmem::Misc + 4);

    if (tid == 0) {
        for (int s = 0; s < kLinStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kLinMmaWarp) tmem_alloc(tmem_holder, kLinTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    // work units: 128 x 256 output tiles, row block unit / tiles_n, column block unit mod tiles_n
    const int unit0 = blockIdx.x, unit_step = gridDim.x;
    const int n_units = p.n_tiles;
    const WaitCtl wc{abort_flag, p.err_flag, kWaitTimeoutNs};
    int never = 0;
    const WaitCtl dw{&never, nullptr, 100000000ull};

    if (warp == kLinTmaWarp) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_x);
            tma_prefetch_desc(&p.tm_w);
            pdl_wait();                                  // X and W may come from the previous grid
            int it = 0;
            bool ok = true;
            for (int unit = unit0; ok && unit < n_units; unit += unit_step) {
                const int m0 = (unit / p.tiles_n) * 128, n0 = (unit % p.tiles_n) * 256;
                for (int kt = 0; kt < p.k_tiles; ++kt, ++it) {
                    const int s = it % kLinStages;
                    if (!(ok = mbar_wait(&empty[s], ((it / kLinStages) & 1) ^ 1, wc, 1))) break;
                    mbar_expect_tx(&full[s], kStageBytes);
                    uint8_t* a = smem + LinSmem::Stages + s * kStageBytes;
                    tma_load_2d(a, &p.tm_x, kt * 64, m0, &full[s]);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        tma_load_2d(a + kABytes + c * 8192, &p.tm_w, n0 + 64 * c, kt * 64, &full[s]);
                }
            }
            if (!ok) {                                   // loads in flight land before teardown
                for (int j = it - kLinStages; j < it; ++j)
                    if (j >= 0) (void)mbar_wait(&full[j % kLinStages], (j / kLinStages) & 1, dw, 2);
            }
        }
    } else if (warp == kLinMmaWarp) {
        // ------------------------------------------------ UMMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(128, 256, 0, 1);
            // stage 0's descriptors; a stage or K step moves only the 14-bit start-address field
            const uint64_t a_desc0 = sdesc_k_sw128(smem_u32(smem + LinSmem::Stages));
            const uint64_t b_desc0 = sdesc_mn_sw128(smem_u32(smem + LinSmem::Stages + kABytes), 8192);
            int it = 0, tc = 0;
            bool ok = true;
            for (int unit = unit0; ok && unit < n_units; unit += unit_step, ++tc) {
                const int b = tc & 1;
                if (!(ok = mbar_wait(&acc_empty[b], ((tc >> 1) & 1) ^ 1, wc, 3))) break;
                tc_fence_after();
                const uint32_t acc = tmem + 256u * b;
                for (int kt = 0; kt < p.k_tiles; ++kt, ++it) {
                    const int s = it % kLinStages;
                    if (!(ok = mbar_wait(&full[s], (it / kLinStages) & 1, wc, 4))) break;
                    tc_fence_after();
                    const uint64_t off = static_cast<uint64_t>(s * (kStageBytes >> 4));
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_ss(acc, a_desc0 + off + 2 * kk, b_desc0 + off + 128 * kk, idesc,
                                (kt > 0 || kk > 0) ? 1u : 0u);
                    umma_commit(&empty[s]);
                }
                if (ok) umma_commit(&acc_full[b]);
            }
            if (!ok) {                                   // every issued UMMA done before dealloc
                umma_commit(drain);
                (void)mbar_wait(drain, 0, dw, 5);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue: TMEM -> bf16 rows of Y
        // With a TMA map for Y, each warp converts 32 rows x 64 columns at a time into a
        // 128-byte-swizzled staging buffer (two per warp, alternating) and one lane stores it by
        // TMA: whole lines, no store instructions per row.  Otherwise 16-byte (or element)
        // stores straight from registers.
        const int q = warp & 3;
        pdl_wait();                                      // the previous grid may still read Y
        uint8_t* stage_base = smem + LinSmem::Out + (warp - 2) * 2 * kOutBytes;
        int tc = 0, nbuf = 0;
        for (int unit = unit0; unit < n_units; unit += unit_step, ++tc) {
            const int b = tc & 1;
            if (!warp_wait(&acc_full[b], (tc >> 1) & 1, wc, 6)) break;
            tc_fence_after();
            const int m0 = (unit / p.tiles_n) * 128;
            const int row = m0 + 32 * q + lane;
            const int n0 = (unit % p.tiles_n) * 256;
            const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * q) << 16) + 256u * b;
            if (p.tma_store) {
#pragma unroll 1
                for (int c = 0; c < 4; ++c, ++nbuf) {
                    uint8_t* stage = stage_base + (nbuf & 1) * kOutBytes;
                    if (lane == 0) bulk_wait_group_read<1>();   // this buffer's previous store has read it
                    __syncwarp();
                    uint32_t v[64];
                    tmem_ld32(tbase + 64 * c, v);
                    tmem_ld32(tbase + 64 * c + 32, v + 32);
                    tmem_ld_wait();
                    const uint32_t rowaddr = smem_u32(stage) + lane * 128;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w[e] = pack_bf16x2(__uint_as_float(v[8 * j + 2 * e]), __uint_as_float(v[8 * j + 2 * e + 1]));
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                                     ::"r"(rowaddr + ((j ^ (lane & 7)) << 4)), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                                       "r"(w[3]) : "memory");
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const int n = n0 + 64 * c;
                        if (p.split_hd > 0 && n >= p.split_hd) {
                            // a key or value block: rows m0 + 32 q .. of one batch entry, consecutive slots
                            const int row = m0 + 32 * q;
                            const int b = row / p.seg_len, tt = row - b * p.seg_len;
                            const bool val = n >= 2 * p.split_hd;
                            tma_store_3d(val ? &p.tm_v : &p.tm_k, n - (val ? 2 : 1) * p.split_hd,
                                         (p.slot0 + tt) % p.slots, b, stage);
                        } else {
                            tma_store_2d(&p.tm_y, n, m0 + 32 * q, stage);
                        }
                        bulk_commit_group();
                    }
                }
            } else {
                __nv_bfloat16* yrow = static_cast<__nv_bfloat16*>(p.y) + static_cast<int64_t>(row) * p.ld_y;
#pragma unroll 1
                for (int cb = 0; cb < 8; ++cb) {
                    uint32_t v[32];
                    tmem_ld32(tbase + 32 * cb, v);
                    tmem_ld_wait();
                    const int c0 = n0 + 32 * cb;
                    if (row >= p.m || c0 >= p.n) continue;
                    if (p.vec && c0 + 32 <= p.n) {
                        uint4* dst = reinterpret_cast<uint4*>(yrow + c0);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                w[e] = pack_bf16x2(__uint_as_float(v[8 * j + 2 * e]), __uint_as_float(v[8 * j + 2 * e + 1]));
                            dst[j] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (c0 + j < p.n) yrow[c0 + j] = __float2bfloat16_rn(__uint_as_float(v[j]));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            mbar_arrive_if(&acc_empty[b], lane == 0);
        }
        if (lane == 0) bulk_wait_group_all();            // stores complete before the CTA exits
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kLinMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kLinTmemCols);
    }
}

}  // namespace

cudaError_t launch_linear(const LinearParams& p, int sm_count, cudaStream_t s)
{
    if (p.n_tiles == 0) return cudaSuccess;
    static bool attr_done = false;
    if (!attr_done) {
        const cudaError_t e = cudaFuncSetAttribute(linear_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   LinSmem::Size);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    const int grid = p.n_tiles < sm_count ? p.n_tiles : sm_count;
    return launch_dependent(linear_kernel, dim3(grid), dim3(kLinThreads), LinSmem::Size, s, p);
}

}  // namespace txl
