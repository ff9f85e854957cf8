// txl_internal.h -- kernel parameter blocks and launch entry points shared by the C-ABI host
// code (txl_api.cu) and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/txl.h"

namespace txl {

// Launch with programmatic stream serialization: the grid may start (and run its prologue) while
// the previous grid of the stream finishes; the kernel itself calls pdl_wait before it touches
// global memory.  Used for the kernels of one forward step (position table, fused attention,
// memory push), which follow one another on a stream.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Range checks of the checked build (compiled with -DTXL_CHECKED): a computed index outside its
// range adds one to the library's device counter `chk` and the caller falls back to a safe index
// (nothing traps, nothing waits); in the normal build every check is `true` and costs nothing.
#ifdef TXL_CHECKED
constexpr bool kCheckedBuild = true;
__device__ __forceinline__ bool in_range(int64_t x, int64_t lo, int64_t hi, int* chk)
{
    const bool ok = x >= lo && x < hi;
    if (!ok && chk) atomicAdd(chk, 1);
    return ok;
}
#else
constexpr bool kCheckedBuild = false;
__device__ __forceinline__ bool in_range(int64_t, int64_t, int64_t, int*) { return true; }
#endif

// Device address of the range-check counter in the current context (null in the normal build).
int* range_counter();
// Unique id of the current CUDA context (false if none is current).
bool current_context_id(unsigned long long* id);

constexpr int kMaxDModel = 4096;   // the bf16 path keeps d_model/2 frequencies in shared memory
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;   // 2 s: far above any healthy wait
constexpr int kSchedCapacity = 4096;   // bytes of per-CTA item counts carried as kernel parameters
constexpr int kMaxSchedClasses = 32;   // query tiles per sequence the count table can describe

// Balanced static assignment of n_cls classes of per_cls interchangeable items (class q costs
// len0 + q key tiles) to G CTAs: counts[c * n_cls + q].  False if it does not fit `capacity`.
bool schedule_items(int G, int n_cls, int per_cls, int len0, uint8_t* counts, int capacity);

// ---------------------------------------------------------------- relative position table
struct PosGenF32Params {
    const float* W;      // [d_model][ld_w]
    float* r;            // [n_rows][H][ld_r]
    int64_t ld_w, ld_r;
    int n_rows, d_model, H, D;
};

constexpr int kPosKTile = 128;   // sinusoid columns (K) per pipeline stage of the bf16 kernel

struct PosGenTcParams {
    CUtensorMap tm_w;    // W_R as 2D (n = h*D+d, m): box 64 x kPosKTile, 128-byte swizzle
    void* r;             // bf16 [n_rows][H][ld_r]
    int64_t ld_r;
    int n_rows, d_model, H, D;
    int n_ktiles;        // ceil(d_model / kPosKTile)
    int dense;           // ld_r == D, H*D a multiple of 8 and r 16-byte aligned: row-vector stores
    int* err_flag;
    float log2_freq_step;        // -2 log2(10000) / d_model: w_k = 2^(k * log2_freq_step)
};

cudaError_t launch_pos_gen_f32(const PosGenF32Params& p, cudaStream_t s);
cudaError_t launch_pos_gen_tc(const PosGenTcParams& p, cudaStream_t s);

// ---------------------------------------------------------------- attention (general SIMT)
struct AttnSimtParams {
    const void* q; int64_t q_sb, q_st, q_sh;
    const void* kmem; const void* vmem; int64_t m_sb, m_st, m_sh;
    const void* kcur; int64_t kc_sb, kc_st, kc_sh;
    const void* vcur; int64_t vc_sb, vc_st, vc_sh;
    void* out; int64_t o_sb, o_st, o_sh;
    const float* u; const float* vb;
    const void* r; int64_t r_row, r_head;       // element strides of the r table
    int B, L, H, D, M, lo, wp, C;
    float scale;
    int n_rows;                                 // rows of the r table (range checks)
    int* chk;                                   // range-check counter (checked build)
};

cudaError_t launch_attn_simt(const AttnSimtParams& p, txl_dtype dtype, cudaStream_t s);

// ---------------------------------------------------------------- attention (fused tcgen05)
struct AttnTcParams {
    CUtensorMap tm_q;            // (d, h, t, b) box 64 x 1 x 128 x 1
    CUtensorMap tm_kmem, tm_vmem;
    CUtensorMap tm_kcur, tm_vcur;
    CUtensorMap tm_r;            // (d, h, row) box 64 x 1 x 128
    // d_head <= 64 (persistent kernel): q rows i0, i0+2, .. (tm_qe) and i0+1, i0+3, .. (tm_qo),
    // (d, h, t/2, b) box 64 x 1 x 64 x 1, so one tile lands with even queries in rows 0-63 and
    // odd queries in rows 64-127
    CUtensorMap tm_qe, tm_qo;
    const float* u; const float* vb;   // [H][D] fp32
    void* out; int64_t o_sb, o_st, o_sh;
    int B, L, H, D, M, lo, wp, C, n_rows;
    // ring_all (persistent kernel only): every key, the current segment's too, is read from the
    // memory ring: logical key j (0 <= j < M + L) lives in slot (wp + j) mod slots
    int ring_all, slots;
    int* chk;                    // range-check counter (checked build)
    int n_qt;                    // query tiles of 128
    int n_atoms;                 // 64-column atoms per row: 1 (D <= 64) or 2 (D <= 128)
    int k_steps;                 // ceil(D / 16): UMMA K steps for the Q.K and Q.r products
    float qscale;                // scale * log2(e)
    int out_vec;                 // out rows take 16-byte stores: D % 8 == 0, 16-byte base and strides
    int out_a16;                 // out base and strides 16-byte aligned (whole 8-element chunks take 16-byte stores)
    int* err_flag;
    // persistent kernel only: sched_counts[c * n_qt + qt] = items of query tile qt that CTA c
    // processes (0 entries when sched_mode == 0: serpentine order instead)
    int sched_mode;
    uint8_t sched_counts[kSchedCapacity];
    // persistent kernel, learned-table mode (table = 1): bidirectional attention over the current
    // sequence alone (no memory, no causal mask, no clamp: every distance i - j of the sequence has
    // its own row i - j + roff of the table); the biases are scaled by bscale instead of qscale
    int table, roff;
    float bscale;
    const uint8_t* key_mask;     // learned-table mode 2: [B][L], keys with 0 score -1e9
    // persistent kernel, log-sum-exp mode (lse != null): every query row's log2-domain
    // log-sum-exp m + log2(l) is written to lse[(b L + i) H + h]; out is written as well when
    // lse_out is set, not otherwise
    float* lse;
    int lse_out;
};

cudaError_t launch_attn_tc(const AttnTcParams& p, cudaStream_t s);
// d_head <= 64: one persistent CTA per SM (at most sm_count CTAs) over all query tiles
cudaError_t launch_attn_persist(const AttnTcParams& p, int sm_count, cudaStream_t s);

// ---------------------------------------------------------------- backward (SIMT)
struct BwdParams {
    AttnSimtParams a;                           // the forward call's inputs and its output (a.out)
    const void* dout; int64_t g_sb, g_st, g_sh; // upstream gradient, the inputs' dtype
    float* dq; float* dk; float* dv;            // [B][L][H][D] (dk, dv: the current segment's keys)
    float* du; float* dvb;                      // [H][D]
    float* dr; int n_rows;                      // [n_rows][H][D]
    float* lse; float* dd;                      // workspace [B][L][H]: log-sum-exp, dO . out
    float* pac; float* pbd;                     // workspace [B][L][H][D]: per-query parts of du, dv_bias
    int lse_given;                              // lse already holds every row's log-sum-exp
    int* err_flag;                              // device status (TXL_ERR_TIMEOUT on a wait abandoned), may be null
};

struct PosBwdParams {
    const float* dr;                            // [n_rows][H*D]
    float* dW; int64_t ld_dw;                   // [d_model][ld_dw]
    int n_rows, d_model, H, D;
};

cudaError_t launch_rel_attn_bwd(const BwdParams& p, txl_dtype dtype, cudaStream_t s);
// tensor-core backward (bf16, D = 64, 16-byte aligned rows): eligibility and the gradient kernel
// (dq, pac, pbd written; dk, dv, dr accumulated atomically into zeroed buffers)
bool bwd_tc_eligible(const BwdParams& p, txl_dtype dtype);
cudaError_t launch_bwd_tc(const BwdParams& p, cudaStream_t s);
// tcgen05 gradient kernel (the above, with the forward's log-sum-exp given and out, dq, dk, dv, dr,
// pac, pbd 16-byte aligned): dq, dk, dv, pac, pbd written; dr accumulated atomically (zeroed first)
bool bwd_umma_eligible(const BwdParams& p, txl_dtype dtype);
cudaError_t launch_bwd_umma(const BwdParams& p, cudaStream_t s);

// ---------------------------------------------------------------- learned-table variant (SIMT)
struct TableParams {
    const void* q; int64_t q_sb, q_st, q_sh;
    const void* k; int64_t k_sb, k_st, k_sh;
    const void* v; int64_t v_sb, v_st, v_sh;
    void* out; int64_t o_sb, o_st, o_sh;
    const float* u; const float* vb;
    const void* r; int64_t r_row, r_head;       // [2 max_len - 1][H][ld_r]
    const uint8_t* mask;                        // [B][L], 0 = masked key; may be null
    int B, L, H, D, max_len;
    float scale;
};
// tensor-core table variant (bf16, D = 64, 16-byte aligned rows)
bool table_tc_eligible(const TableParams& p, txl_dtype dtype);
cudaError_t launch_table_tc(const TableParams& p, cudaStream_t s);

cudaError_t launch_table_attn(const TableParams& p, txl_dtype dtype, cudaStream_t s);
cudaError_t launch_pos_bwd(const PosBwdParams& p, cudaStream_t s);
// dW_R = R^T dr on the tensor cores (dW zeroed first by the caller)
cudaError_t launch_pos_bwd_tc(const PosBwdParams& p, int sm_count, cudaStream_t s);

// ---------------------------------------------------------------- projections (tcgen05 GEMM)
struct LinearParams {
    CUtensorMap tm_x;    // X as 2D (k, m): box 64 x 128, 128-byte swizzle
    CUtensorMap tm_w;    // W as 2D (n, k): box 64 x 64, 128-byte swizzle
    CUtensorMap tm_y;    // Y as 2D (n, m): box 64 x 32, 128-byte swizzle (when tma_store)
    void* y;             // bf16 [m][ld_y]
    int64_t ld_y;
    int m, n, k;
    int tiles_n;         // ceil(n / 256)
    int m_tiles;         // ceil(m / 128)
    int n_tiles;         // m_tiles * tiles_n
    int k_tiles;         // ceil(k / 64)
    int vec;             // Y 16-byte aligned and ld_y a multiple of 8: 16-byte stores
    int tma_store;       // the same, and tm_y encoded: the epilogue stores tiles by TMA
    int* err_flag;
    // Split output (split_hd > 0, TMA stores only): columns [0, split_hd) go to tm_y; columns
    // [split_hd, 2 split_hd) and [2 split_hd, 3 split_hd) go to the rings tm_k, tm_v, (split_hd,
    // slots, batch) maps, row r = b * seg_len + t into slot (slot0 + t) mod slots of entry b
    int split_hd, seg_len, slot0, slots;
    CUtensorMap tm_k, tm_v;
};

cudaError_t launch_linear(const LinearParams& p, int sm_count, cudaStream_t s);

// ---------------------------------------------------------------- decode (few queries, split keys)
constexpr int kDecodeChunk = 256;   // keys per CTA
constexpr int kDecodeMaxL = 16;     // queries per (b, h) the decode path takes

struct DecodeParams {
    const void* q; int64_t q_sb, q_st, q_sh;
    const void* kmem; const void* vmem; int64_t m_sb, m_st, m_sh;
    const void* kcur; int64_t kc_sb, kc_st, kc_sh;
    const void* vcur; int64_t vc_sb, vc_st, vc_sh;
    void* out; int64_t o_sb, o_st, o_sh;
    const float* u; const float* vb;
    const void* r; int64_t r_row, r_head;       // element strides of the r table
    int B, L, H, D, Dp, M, lo, wp, C;           // Dp: D rounded up to 8
    float qscale;                               // scale * log2(e)
    int n_chunks;                               // ceil((M + L) / kDecodeChunk)
    float* part;                                // [B][H][L][n_chunks][D + 2]: (m, l, O[D])
    int vec_kv, vec_r;                          // rows 16-byte aligned: vector loads allowed
};

size_t decode_smem_bytes(int lq, int Dp);
cudaError_t launch_decode(const DecodeParams& p, txl_dtype dtype, cudaStream_t s);

// Static per-device scratch of txl_rel_attn_decode_noalloc (8 MiB) and its device address.
constexpr size_t kDecodeStaticScratchBytes = 8u << 20;
constexpr int kMaxDevices = 64;
cudaError_t decode_static_scratch(float** out);

// ---------------------------------------------------------------- memory ring
struct MemPushParams {
    const void* k_new; const void* v_new;
    int64_t n_sb, n_st, n_sh;           // strides of the k_new view
    int64_t nv_sb, nv_st, nv_sh;        // strides of the v_new view
    void* k; void* v;
    int64_t m_sb, m_st, m_sh;           // ring strides
    int B, H, D, M, wp, t0, n_t;        // copy positions t0 .. t0+n_t-1 of the segment
    int elem_bytes;
    int vec16;                          // 1: copy 16-byte chunks
    int* chk;                           // range-check counter (checked build)
};

cudaError_t launch_mem_push(const MemPushParams& p, cudaStream_t s);

cudaError_t launch_selftest_wait(int* err_flag, unsigned timeout_us, cudaStream_t s);
// One failing and one passing range check on the device (the checked build's counter gains one).
cudaError_t launch_selftest_range(int* chk, cudaStream_t s);

}  // namespace txl
