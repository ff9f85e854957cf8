/*
 * txl.h -- C ABI of libtxl.so: Transformer-XL relative multi-head attention over
 * [memory ++ current segment] on one NVIDIA GB300 (sm_103a).
 *
 * The operation (citations are page title and section):
 *   "跨窗口的相对位置编码" §3 and "Transformer-XL 和相对位置编码" §2.3.2 (terms (a)-(d)):
 *       A_ij = q_i.k_j + q_i.r_{i-j} + u.k_j + v.r_{i-j}
 *   "跨窗口的相对位置编码" §2, "Transformer-XL 和相对位置编码" §2.3.2:
 *       R_delta[2k] = sin(delta * 10000^(-2k/d_model)), R_delta[2k+1] = cos(same)
 *       r_delta = R_delta W_R                  (W_{k,R}; "TransformerXL 相对位置编码" §3.1 r_proj)
 *   "TransformerXL 相对位置编码" §2.4: distances beyond clamp_len count as clamp_len.
 *   "TransformerXL 相对位置编码" §4.2/§4.3: mask the summed score; keys span memory + current.
 *   "Transformer-XL 和相对位置编码" §2.3.1: K, V from [SG(memory) ∘ current], Q from current.
 *   "Transformer-XL架构解析" §1.1: the memory is a FIFO of mem_len positions.
 *
 * Conventions for every entry point:
 *  - Pointers named "device" are CUDA device addresses; the caller owns all memory.  The library
 *    never allocates, frees or synchronises.  Work is enqueued on `stream` (a cudaStream_t; NULL
 *    is the legacy default stream) on the calling thread's current device, and calls return as
 *    soon as it is enqueued.
 *  - Arguments are validated on the host before anything is launched; a non-TXL_OK status means
 *    nothing was enqueued (except TXL_ERR_CUDA, which reports a failed launch).
 *  - Element strides are in elements, not bytes.  The innermost index (d) is always contiguous.
 *  - No exceptions, no printing, no CPU fallback.
 */
#ifndef TXL_H
#define TXL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TXL_OK = 0,
    TXL_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, inconsistent shapes       */
    TXL_ERR_UNSUPPORTED = 2,   /* valid request this build does not implement                 */
    TXL_ERR_ALIGNMENT = 3,     /* a base address or stride is not 16-byte aligned where needed */
    TXL_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed                            */
    TXL_ERR_TIMEOUT = 5,       /* written to err_flag by a kernel whose bounded wait expired   */
    TXL_ERR_WORKSPACE = 6      /* workspace missing or smaller than txl_rel_attn_workspace_size */
} txl_status;

typedef enum { TXL_F32 = 0, TXL_BF16 = 1 } txl_dtype;

/* A [B][T][H][D] tensor in device memory: element (b,t,h,d) lives at
 * ptr + b*stride_b + t*stride_t + h*stride_h + d   (elements of the call's dtype). */
typedef struct {
    void* ptr;
    int64_t stride_b;
    int64_t stride_t;
    int64_t stride_h;
} txl_view;

/* K/V memory of M positions per batch entry ("Transformer-XL架构解析" §1.1: FIFO cache).
 * k and v are device [B][M][H][D] slot arrays with the strides below (shared by k and v).
 * Logical memory key j (0 <= j < M, j = M-1 newest) lives in physical slot (wp + j) mod M and
 * is valid iff j >= M - valid.  A freshly zeroed ring has wp = 0, valid = 0.  A plain
 * contiguous memory (oldest first) is described by wp = 0, valid = M.  M = 0 means no memory
 * (k, v may then be NULL). */
typedef struct {
    void* k;
    void* v;
    int64_t stride_b;
    int64_t stride_t;
    int64_t stride_h;
    int B, M, H, D;
    txl_dtype dtype;
    int wp;      /* next slot to write == slot of the oldest position once the ring is full */
    int valid;   /* number of valid positions, 0..M */
} txl_mem;

/* Human-readable name of a status code (static string). */
const char* txl_status_str(txl_status status);

/* Library ABI version (major*10000 + minor*100 + patch). */
int txl_version(void);

/*
 * txl_rel_pos_gen -- position key vectors of every distance the attention can see.
 *   r[delta][h][d] = sum_m R_delta[m] * W_R[m][h*d_head + d],  delta = 0 .. n_rows-1,
 * with R_delta the interleaved sinusoid above (fp32 angles, on chip; never stored).
 * Row index == distance.  For one attention call, n_rows = min(M+L, clamp_len+1).
 *   W_R : device [d_model][ld_w], dtype; columns 0 .. n_head*d_head-1 are used; no bias.
 *   r   : device [n_rows][n_head][ld_r], dtype; only d < d_head is written.
 * Limits: d_model even, 2 <= d_model <= 4096; ld_w >= n_head*d_head; ld_r >= d_head.
 * bf16: tensor-core path (fp32 accumulate, R rounded to bf16 before the product, output rounded
 *       to bf16 once); needs W_R 16-byte aligned and ld_w a multiple of 8.
 * f32 : fp32 SIMT path with R rounded once from double precision.
 */
txl_status txl_rel_pos_gen(int n_rows, int d_model, int n_head, int d_head,
                           const void* W_R, int64_t ld_w,
                           void* r, int64_t ld_r,
                           txl_dtype dtype, void* stream);

/*
 * txl_rel_attn_fwd -- one forward call of relative multi-head attention.
 * For every batch b, head h and query i (0 <= i < L, absolute position M+i) over keys
 * j in [memory(0..M-1) ++ current(M..M+L-1)]:
 *   delta = M + i - j,  delta_c = min(delta, clamp_len)
 *   visible(i, j) <=> (M - valid) <= j <= M + i
 *   s_ij  = scale * ( q_i.k_j + q_i.r[delta_c] + u_h.k_j + v_h.r[delta_c] )
 *   out_i = sum_j softmax_j(s_ij over visible j) * v_j          (masked keys weigh exactly 0)
 * Arguments:
 *   q      : view of [B][L][H][D] queries of the current segment (device).
 *   mem    : the memory (see txl_mem); may be NULL when there is no memory (M = 0).
 *   k_cur, v_cur : views of [B][L][H][D] keys/values of the current segment (device).
 *   u, v_bias : device fp32 [H][D] global content / position biases.
 *   r      : device [n_rows][H][ld_r] from txl_rel_pos_gen; n_rows >= min(M+L, clamp_len+1).
 *   scale  : logit scale; <= 0 selects 1/sqrt(D).
 *   out    : view of [B][L][H][D] outputs (device), dtype.
 *   workspace : device scratch of workspace_bytes (txl_rel_attn_workspace_size); may be NULL
 *            when that size is 0.
 *   err_flag : optional device int; a kernel whose bounded wait expires writes TXL_ERR_TIMEOUT
 *            there (and its outputs are then undefined).  Never cleared by the library.
 * Paths:
 *   bf16, D <= 128, every base and stride 16-byte aligned, and a ring whose wp and M are
 *   multiples of 128 (or wp == 0): the fused TMA + tcgen05 kernel (TMEM accumulators; the
 *   relative shift is an index remap; the score matrix never reaches HBM).
 *   otherwise (f32, other layouts, other rings): a warp-per-query SIMT kernel on the GPU.
 */
txl_status txl_rel_attn_fwd(int B, int L, int H, int D, int clamp_len,
                            const txl_view* q, const txl_mem* mem,
                            const txl_view* k_cur, const txl_view* v_cur,
                            const float* u, const float* v_bias,
                            const void* r, int64_t ld_r, int n_rows,
                            float scale, const txl_view* out, txl_dtype dtype,
                            void* workspace, size_t workspace_bytes,
                            int* err_flag, void* stream);

/* Bytes of device workspace txl_rel_attn_fwd needs for this shape (0 for every path of this
 * version; kept so callers can size it once). */
size_t txl_rel_attn_workspace_size(int B, int L, int H, int D, const txl_mem* mem,
                                   txl_dtype dtype);

/* Which kernel txl_rel_attn_fwd would run for these arguments: 1 = fused tcgen05 kernel,
 * 2 = SIMT kernel, or a negative txl_status if the arguments are rejected. */
int txl_rel_attn_path(int B, int L, int H, int D, const txl_view* q, const txl_mem* mem,
                      const txl_view* k_cur, const txl_view* v_cur, const void* r,
                      int64_t ld_r, const txl_view* out, txl_dtype dtype);

/*
 * txl_rel_attn_decode -- the same attention as txl_rel_attn_fwd for a few queries (1 <= L <= 16)
 * over a long memory: the incremental-generation case ("Transformer-XL架构解析" §3.2,
 * "Transformer-XL 和相对位置编码" §2.2: each new token attends to the cached memory and itself).
 * Arguments, layouts, masks, clamp and result are those of txl_rel_attn_fwd (f32 or bf16, any
 * ring), except:
 *   L         : 1 .. 16 queries per (b, h) (TXL_ERR_UNSUPPORTED above).
 *   workspace : device scratch, 16-byte aligned, of at least
 *               txl_rel_attn_decode_workspace_size(B, L, H, D, mem) bytes (TXL_ERR_WORKSPACE
 *               otherwise).  It holds per-chunk partial results between the two kernels of the
 *               call; its contents on entry do not matter and are overwritten.
 * The keys of every (b, h) are split into chunks of 256 processed by separate CTAs on the CUDA
 * cores (the work is bound by HBM bandwidth: about one flop per byte at L = 1), then the chunks
 * are merged (split-K softmax).  Calls that share a workspace must not overlap on the GPU.
 * With L >= 3, bf16, D <= 64 and inputs that txl_rel_attn_fwd's fused kernel takes (16-byte aligned
 * rows and strides; a ring's write pointer and length multiples of 128), the call runs that fused
 * tensor-core kernel instead (one query tile over every key, faster from three queries on) and
 * leaves the workspace untouched; the argument checks, the workspace check included, are the same.
 */
txl_status txl_rel_attn_decode(int B, int L, int H, int D, int clamp_len,
                               const txl_view* q, const txl_mem* mem,
                               const txl_view* k_cur, const txl_view* v_cur,
                               const float* u, const float* v_bias,
                               const void* r, int64_t ld_r, int n_rows,
                               float scale, const txl_view* out, txl_dtype dtype,
                               void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace txl_rel_attn_decode needs: B*H*L*ceil((M+L)/256)*(D+2)*4
 * (0 when the shape is outside the decode path). */
size_t txl_rel_attn_decode_workspace_size(int B, int L, int H, int D, const txl_mem* mem);

/* Which kernels txl_rel_attn_decode (and txl_rel_attn_decode_noalloc) would run for these
 * arguments: 1 = the fused persistent tcgen05 kernel (L >= 3, see txl_rel_attn_decode), 4 = the
 * split-key decode kernels and their merge, or a negative txl_status if the arguments are rejected.
 * Nothing is launched; the workspace is not checked. */
int txl_rel_attn_decode_path(int B, int L, int H, int D, const txl_view* q, const txl_mem* mem,
                             const txl_view* k_cur, const txl_view* v_cur, const void* r,
                             int64_t ld_r, const txl_view* out, txl_dtype dtype);

/*
 * txl_rel_attn_decode_noalloc -- txl_rel_attn_decode without a caller workspace, for callers that
 * cannot obtain device memory at call time.  The pages have no counterpart to this entry point: it
 * is a service of this library.  Examples of such callers: a serving process whose device memory
 * is owned by a pre-sized arena that forbids allocations once it runs; a plugin reached through an
 * interface that passes only inputs and outputs; a per-token generation loop that cannot afford
 * cudaMalloc, which may synchronise the device.  Nothing here allocates: no cudaMalloc, cudaFree
 * or allocating library routine is called.
 * Arguments, layouts and results are those of txl_rel_attn_decode minus the workspace.  The
 * per-chunk partial results live instead in a fixed 8 MiB scratch array inside the library, which
 * every GPU that loads the library holds until the process exits:
 *   - B*H*L*ceil((M+L)/256)*(D+2)*4 must not exceed 8388608 bytes (TXL_ERR_WORKSPACE otherwise;
 *     use txl_rel_attn_decode with a workspace for such shapes);
 *   - the first call on a device looks up the array's device address (cudaGetSymbolAddress, with
 *     that device current) and caches it with the id of the current context; make that first
 *     call before any stream capture.  After cudaDeviceReset the device's new context has another
 *     id, and the first call in it looks the address up again (so that call, too, belongs before
 *     any capture);
 *   - every call shares the array.  Each call writes every partial it reads, so nothing has to
 *     start at zero, but calls that overlap on the GPU (two streams, or two host threads on
 *     different streams) race on it and their results are undefined: keep them ordered, for
 *     instance on one stream.
 * Calls that txl_rel_attn_decode sends to the fused kernel (L >= 3, see there) do so here as well
 * and do not touch the array (the size limit above still applies to them).
 */
txl_status txl_rel_attn_decode_noalloc(int B, int L, int H, int D, int clamp_len,
                                       const txl_view* q, const txl_mem* mem,
                                       const txl_view* k_cur, const txl_view* v_cur,
                                       const float* u, const float* v_bias,
                                       const void* r, int64_t ld_r, int n_rows,
                                       float scale, const txl_view* out, txl_dtype dtype,
                                       void* stream);

/*
 * txl_mem_push -- append L positions to the FIFO memory ("Transformer-XL架构解析" §1.1;
 * "Transformer-XL 和相对位置编码" §2.3.1: the cached states of the previous segment).
 * Copies k_new/v_new [B][L][H][D] (device views) into slots (wp + t) mod M for
 * t = max(0, L-M) .. L-1 (a segment longer than the memory keeps its last M positions), then
 * updates mem->wp = (wp + L) mod M and mem->valid = min(valid + L, M) on the host at enqueue
 * time.  The copy is ordered on `stream`; the attention for this segment must be enqueued
 * before the push if it should see the previous memory.  Bit-exact copy.
 */
txl_status txl_mem_push(txl_mem* mem, const txl_view* k_new, const txl_view* v_new, int L,
                        void* stream);

/*
 * txl_linear -- Y = X W: bf16 inputs, fp32 accumulation on the tensor cores, one rounding of each
 * output to bf16.  The content projections of the attention layer: q_proj, k_proj, v_proj and
 * o_proj of "TransformerXL 相对位置编码" §3.1 (linear maps without bias); Q = h W_q, K = h~ W_k,
 * V = h~ W_v of "Transformer-XL 和相对位置编码" §2.3.1.
 *   X : device [m][ld_x], columns 0..k-1 are read;  W : device [k][ld_w], columns 0..n-1 are read;
 *   Y : device [m][ld_y], columns 0..n-1 are written and nothing else.
 * Limits: m, n >= 0 (either 0: nothing to do), k >= 1; ld_x >= k, ld_w >= n, ld_y >= n; X and W
 * 16-byte aligned with ld_x, ld_w multiples of 8 (TXL_ERR_ALIGNMENT otherwise).  bf16 only
 * (TXL_ERR_UNSUPPORTED for TXL_F32).  err_flag: as txl_rel_attn_fwd.
 */
txl_status txl_linear(int m, int n, int k, const void* X, int64_t ld_x, const void* W, int64_t ld_w,
                      void* Y, int64_t ld_y, txl_dtype dtype, int* err_flag, void* stream);

/*
 * txl_rel_attn_layer -- one attention-layer step of Transformer-XL over hidden states:
 *   Q = h W_q and K = h~ W_k, V = h~ W_v over h~ = [SG(h_mem) o h], the memory-extended states
 *   ("Transformer-XL 和相对位置编码" §2.3.1); the relative attention of txl_rel_attn_fwd with the
 *   memory's keys first; y = concat_heads(attention) W_o ("TransformerXL 相对位置编码" §3.1); then
 *   the segment enters the memory (the FIFO of txl_mem_push; mem->wp and mem->valid advance).
 * The memory caches the projected keys and values of its positions (h_mem W_k, h_mem W_v) rather
 * than h_mem: with the weights fixed this is the same function (a row's projection does not depend
 * on when it is taken), and each position is projected once, when it enters the memory, instead of
 * once for every segment that attends to it.
 *   h      : device bf16 [B*L][ld_h], row b*L + t = position t of batch entry b, d_model columns.
 *   mem    : K/V memory as for txl_rel_attn_fwd (bf16, B, H, D matching), or NULL / M = 0.
 *   W_qkv  : device bf16 [d_model][3*H*D], columns [0,HD) = W_q, [HD,2HD) = W_k, [2HD,3HD) = W_v.
 *   W_o    : device bf16 [H*D][d_model].
 *   u, v_bias, r, ld_r, n_rows, clamp_len, scale : as txl_rel_attn_fwd (r from txl_rel_pos_gen).
 *   y      : device bf16 [B*L][ld_y], d_model columns written.
 *   workspace : device, >= txl_rel_attn_layer_workspace_size(B, L, H, D) bytes, 16-byte aligned
 *            (TXL_ERR_WORKSPACE if missing or smaller): the segment's q|k|v [B*L][3*H*D] and the
 *            attention output [B*L][H*D], bf16.  Its contents after the call are unspecified.
 * Limits: H*D and d_model multiples of 8; the limits of txl_linear and txl_rel_attn_fwd.  bf16
 * only.  Enqueues four launches on `stream` (projection, attention, output projection, push).
 */
txl_status txl_rel_attn_layer(int B, int L, int H, int D, int d_model, int clamp_len,
                              const void* h, int64_t ld_h, txl_mem* mem,
                              const void* W_qkv, const void* W_o,
                              const float* u, const float* v_bias,
                              const void* r, int64_t ld_r, int n_rows, float scale,
                              void* y, int64_t ld_y, void* workspace, size_t workspace_bytes,
                              int* err_flag, void* stream);

/* Bytes of device workspace txl_rel_attn_layer needs: B*L*H*D*8 (0 for an empty shape). */
size_t txl_rel_attn_layer_workspace_size(int B, int L, int H, int D);

/*
 * txl_rel_attn_layer_fused -- the layer step of txl_rel_attn_layer in three launches, with the memory
 * push folded into the projection.  The memory of mem_len positions lives in a ring of at least
 * mem_len + L slots (mem->M slots; mem->wp = slot of the oldest memory position, mem->valid = valid
 * memory positions, 0 .. mem_len): the q|k|v product writes the segment's K and V straight into the
 * L slots after the memory, (wp + mem_len + t) mod mem->M, and Q into the workspace; the fused
 * attention reads memory and segment keys from the ring (logical key j of [memory ++ segment] in
 * slot (wp + j) mod mem->M); the output product follows; then, instead of a copy, the window moves:
 * mem->wp += L (mod mem->M), mem->valid = min(valid + L, mem_len).  The function is that of
 * txl_rel_attn_layer with a memory of mem_len positions ("Transformer-XL 和相对位置编码" §2.3.1: the
 * cached states of the previous segment extend the keys and values; "TransformerXL 相对位置编码" §3.1:
 * projections without bias).
 *   h, W_qkv, W_o, u, v_bias, r, ld_r, n_rows, clamp_len, scale, y, ld_y, err_flag : as txl_rel_attn_layer
 *            (n_rows >= min(mem_len + L, clamp_len + 1)).
 *   mem    : device bf16 rings k, v, dense [B][mem->M][H][D]; a ring starts zeroed (wp = 0, valid = 0):
 *            slots past the valid memory are read (and masked), so they must hold finite values.
 *   workspace : device, >= txl_rel_attn_layer_fused_workspace_size(B, L, H, D) bytes, 16-byte aligned.
 * Limits (TXL_ERR_UNSUPPORTED otherwise; use txl_rel_attn_layer): bf16; D <= 64 and a multiple of 8;
 * H*D a multiple of 64; d_model a multiple of 8; L, mem_len, mem->M and mem->wp multiples of 128.
 */
txl_status txl_rel_attn_layer_fused(int B, int L, int H, int D, int d_model, int clamp_len,
                                    const void* h, int64_t ld_h, txl_mem* mem, int mem_len,
                                    const void* W_qkv, const void* W_o,
                                    const float* u, const float* v_bias,
                                    const void* r, int64_t ld_r, int n_rows, float scale,
                                    void* y, int64_t ld_y, void* workspace, size_t workspace_bytes,
                                    int* err_flag, void* stream);

/* Bytes of device workspace txl_rel_attn_layer_fused needs: B*L*H*D*4 (0 for an empty shape). */
size_t txl_rel_attn_layer_fused_workspace_size(int B, int L, int H, int D);

/*
 * txl_rel_attn_bwd -- gradients of one txl_rel_attn_fwd call for an upstream gradient d_out,
 * by the chain rule through the four-term score ("Transformer-XL 和相对位置编码" §2.3.2) and the
 * softmax: with q' = q + u, q'' = q + v_bias, P the attention weights and dS_ij =
 * scale P_ij (d_out_i . v_j - d_out_i . out_i),
 *   dq_i  = sum_j dS_ij (k_j + r[delta_ij])        dk_j = sum_i dS_ij q'_i      dv_j = sum_i P_ij d_out_i
 *   du    = sum dS_ij k_j     dv_bias = sum dS_ij r[delta_ij]     dr[delta] = sum_{delta_ij = delta} dS_ij q''_i
 * The memory's keys and values get no gradient: the memory is the stop-gradient part of the
 * extended sequence ("Transformer-XL 和相对位置编码" §2.3.1); dk_cur, dv_cur cover the current
 * segment's keys.  Arguments as txl_rel_attn_fwd, plus
 *   out    : the forward call's output (view, dtype);  d_out : upstream gradient (view, dtype).
 *   dq, dk_cur, dv_cur : device fp32 [B][L][H][D] (dense);  du, dv_bias : device fp32 [H][D];
 *   dr     : device fp32 [n_rows][H][D], every row written (rows no pair reaches are zero).
 *   workspace : device, >= txl_rel_attn_bwd_workspace_size(B, L, H, D) bytes, 16-byte aligned.
 * Scores are recomputed and P is never stored.  bf16 with D = 64 and 16-byte aligned rows and
 * strides (q, k, v, the memory, d_out, r): bf16 products on the tensor cores with fp32 accumulation
 * (c(q + u), c(q + v), P and dS rounded to bf16 as product operands, c = scale log2 e; pairs whose
 * distance reaches clamp_len summed in fp32), the row log-sum-exp taken by the fused forward kernel
 * when that kernel takes the inputs (written into the workspace).  With out, the gradients and dr
 * 16-byte aligned as well, the gradient products run as tcgen05 MMAs with TMEM accumulators (a
 * launch of query CTAs for dq and dr, and key CTAs for dk and dv); otherwise as mma.sync products.
 * Every other case: fp32 arithmetic on the CUDA cores.  Enqueues several launches.
 */
txl_status txl_rel_attn_bwd(int B, int L, int H, int D, int clamp_len,
                            const txl_view* q, const txl_mem* mem,
                            const txl_view* k_cur, const txl_view* v_cur,
                            const float* u, const float* v_bias,
                            const void* r, int64_t ld_r, int n_rows, float scale,
                            const txl_view* out, const txl_view* d_out,
                            float* dq, float* dk_cur, float* dv_cur, float* du, float* dv_bias,
                            float* dr, txl_dtype dtype, void* workspace, size_t workspace_bytes,
                            void* stream);

/* Which gradient kernel txl_rel_attn_bwd and txl_rel_attn_bwd_lse would run for these arguments
 * (the addresses of out, d_out and the gradient buffers count: their alignment chooses the kernel):
 * 1 = tcgen05 kernel, 2 = mma.sync kernel, 3 = SIMT kernels, or a negative txl_status if the
 * arguments are rejected.  No launch. */
int txl_rel_attn_bwd_path(int B, int L, int H, int D, const txl_view* q, const txl_mem* mem,
                          const txl_view* k_cur, const txl_view* v_cur, const void* r, int64_t ld_r,
                          const txl_view* out, const txl_view* d_out, const float* dq, const float* dk_cur,
                          const float* dv_cur, const float* dr, txl_dtype dtype);

/* Bytes of device workspace txl_rel_attn_bwd needs: B*L*H*(2 + 2*D)*4 (0 for an empty shape). */
size_t txl_rel_attn_bwd_workspace_size(int B, int L, int H, int D);

/*
 * txl_rel_attn_fwd_lse -- txl_rel_attn_fwd that also saves the statistics of its softmax, as a
 * forward pass does for its backward:
 *   lse : device fp32 [B][L][H] (4-byte aligned), lse[(b L + i) H + h] = m_i + log2 l_i, the
 *         log2-domain log-sum-exp of row i's visible scores in the units c s_ij (c = scale log2 e):
 *         m_i the row maximum, l_i the sum of the bf16 weights 2^(c s_ij - m_i) that the output's
 *         P.V multiplied (the output's own normaliser).
 * out is written exactly as txl_rel_attn_fwd writes it.  Only the fused tcgen05 kernel keeps the
 * statistics: bf16, D <= 64 and the inputs its path takes (txl_rel_attn_path = 1), else
 * TXL_ERR_UNSUPPORTED before any launch; lse NULL: TXL_ERR_INVALID_ARG; misaligned:
 * TXL_ERR_ALIGNMENT.  Other arguments and errors as txl_rel_attn_fwd.
 */
txl_status txl_rel_attn_fwd_lse(int B, int L, int H, int D, int clamp_len,
                                const txl_view* q, const txl_mem* mem,
                                const txl_view* k_cur, const txl_view* v_cur,
                                const float* u, const float* v_bias,
                                const void* r, int64_t ld_r, int n_rows,
                                float scale, const txl_view* out, float* lse, txl_dtype dtype,
                                void* workspace, size_t workspace_bytes,
                                int* err_flag, void* stream);

/*
 * txl_rel_attn_bwd_lse -- txl_rel_attn_bwd given the statistics txl_rel_attn_fwd_lse saved for
 * the same call (same inputs and output): on the tensor-core path the gradient kernels read lse
 * in place of taking the row log-sum-exp again (one pass over the keys fewer).  lse: device fp32
 * [B][L][H] (4-byte aligned, TXL_ERR_ALIGNMENT otherwise), read only; NULL gives
 * txl_rel_attn_bwd.  Paths that do not use the statistics ignore it.  Other arguments, results and
 * errors as txl_rel_attn_bwd.
 */
txl_status txl_rel_attn_bwd_lse(int B, int L, int H, int D, int clamp_len,
                                const txl_view* q, const txl_mem* mem,
                                const txl_view* k_cur, const txl_view* v_cur,
                                const float* u, const float* v_bias,
                                const void* r, int64_t ld_r, int n_rows, float scale,
                                const txl_view* out, const txl_view* d_out, const float* lse,
                                float* dq, float* dk_cur, float* dv_cur, float* du, float* dv_bias,
                                float* dr, txl_dtype dtype, void* workspace, size_t workspace_bytes,
                                void* stream);

/*
 * txl_rel_pos_bwd -- gradient of W_R from the gradient of the position rows:
 *   dW_R[m][h*d_head + d] = sum_delta R_delta[m] * dr[delta][h][d]
 * with R_delta the interleaved sinusoid of txl_rel_pos_gen (frequencies in double precision; the
 * angle of every fourth distance reduced modulo 2 pi in double precision, the other three offset from
 * it in fp32; then the fp32 sine or cosine: entries within 6e-7 of the exact sinusoid).  dr: device fp32 [n_rows][H][D] (as txl_rel_attn_bwd writes it);
 * dW_R: device fp32 [d_model][ld_dw], columns 0..H*D-1 written (zeroed, then partial sums over
 * ranges of distances added atomically: the fp32 summation order may differ from call to call).
 * d_model even, ld_dw >= H*D.  The products run on the tensor cores as three tf32 products per
 * step (R and dr each split into a tf32 part and the fp32 remainder; the remainder product dropped):
 * about 2^-21 relative error per product, fp32 accumulation.
 */
txl_status txl_rel_pos_bwd(int n_rows, int d_model, int n_head, int d_head, const float* dr,
                           float* dW_R, int64_t ld_dw, void* stream);

/*
 * txl_rel_attn_table_fwd -- the learned-table variant of relative attention ("TransformerXL 相对位置编码"
 * §3.1): bidirectional over one sequence of L positions (no memory, no causal mask).  The position
 * vector of a pair is row rel = clamp(i - j + max_len - 1, 0, 2*max_len - 2) of the projected table
 * r_table = pos_emb W_R (the distance shifted to a non-negative index and clamped, §2; project the
 * learned pos_emb [2*max_len - 1][d_model] with txl_linear, the projection commutes with the lookup):
 *   s_ij = scale*q_i.k_j + scale*q_i.r_rel + u_h.k_j + v_h.r_rel
 * (the scale on the first two terms only, as that page computes it), keys with key_mask[b][j] == 0
 * scored -1e9 (a row whose keys are all masked averages every value), out_i = softmax_j(s_ij) v_j.
 *   q, k, v, out : views of [B][L][H][D] (device, dtype).  u, v_bias : device fp32 [H][D].
 *   r_table : device [2*max_len - 1][H][ld_r], dtype.  key_mask : device uint8 [B][L] or NULL.
 *   scale   : <= 0 selects 1/sqrt(D).
 * Limits: 1 <= D <= 128, max_len >= 1.  bf16 with D <= 64, L <= max_len and 16-byte aligned bases
 * and strides (q, k, v, r_table): the persistent tcgen05 kernel of txl_rel_attn_fwd in a learned-table
 * mode (log2(e)(scale*q + u), log2(e)(scale*q + v) and P rounded to bf16 as product operands, fp32
 * accumulation in tensor memory; a masked key's score is about -1e30 there, which gives it the same
 * weight as -1e9: exactly 0 beside any unmasked key, equal weights in a fully masked row).  Other bf16
 * calls with D = 64 and 16-byte aligned
 * rows and strides (q, k, v, out, r_table): bf16 mma.sync products with fp32 accumulation (scale*q + u,
 * scale*q + v and P rounded to bf16).  Every other case: fp32 arithmetic on the CUDA cores.
 */
txl_status txl_rel_attn_table_fwd(int B, int L, int H, int D, int max_len,
                                  const txl_view* q, const txl_view* k, const txl_view* v,
                                  const float* u, const float* v_bias,
                                  const void* r_table, int64_t ld_r, const uint8_t* key_mask,
                                  float scale, const txl_view* out, txl_dtype dtype, void* stream);

/* Which kernel txl_rel_attn_table_fwd would run for these arguments: 1 = the persistent tcgen05
 * kernel (learned-table mode), 3 = the mma.sync tensor-core kernel, 2 = the CUDA-core kernel, or a
 * negative txl_status if the arguments are rejected.  Nothing is launched. */
int txl_rel_attn_table_path(int B, int L, int H, int D, int max_len,
                            const txl_view* q, const txl_view* k, const txl_view* v,
                            const void* r_table, int64_t ld_r, const uint8_t* key_mask,
                            const txl_view* out, txl_dtype dtype);

/*
 * Checked build.  libtxl_checked.so is this library compiled with -DTXL_CHECKED (the package builds
 * it on request: transformer_xl_relative_gb300/_build.py --checked; the binding loads it when the
 * environment variable TXL_CHECKED is 1).  Its kernels range-check the indices they compute before
 * using them (the key row of every TMA key/value tile of the fused attention, the memory ring slot
 * of every key in the other attention kernels and of every pushed position, the remapped r row):
 * an index outside its range is counted in a device counter owned by the library and replaced by a
 * safe one, so the call completes (its results are then meaningless) and nothing traps or waits.
 * It stands in for a memory checker; the pages have no counterpart.
 *   txl_checked_build        : 1 in the checked build, 0 otherwise.
 *   txl_range_errors         : failed checks since the library was loaded or last cleared, into the
 *                              host int *count.  Synchronizes the current device (a debugging call).
 *                              TXL_ERR_UNSUPPORTED (and 0) in the normal build.
 *   txl_range_errors_clear   : resets the counter (synchronizes the current device).
 *   txl_selftest_range_check : enqueues one failing and one passing check on `stream`; the counter
 *                              gains exactly one.  TXL_ERR_UNSUPPORTED in the normal build.
 */
int txl_checked_build(void);
txl_status txl_range_errors(int* count);
txl_status txl_range_errors_clear(void);
txl_status txl_selftest_range_check(void* stream);

/* Self-test of the bounded waits used by every kernel: launches one CTA that waits on an
 * mbarrier nothing will signal, gives up after timeout_us microseconds (1 .. 10^7), writes
 * TXL_ERR_TIMEOUT to the device int err_flag and returns.  The context stays usable. */
txl_status txl_selftest_wait_timeout(int* err_flag, unsigned timeout_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TXL_H */
