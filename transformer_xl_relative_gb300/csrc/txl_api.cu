// txl_api.cu -- the C ABI of libtxl.so (declared in include/txl.h): argument validation, TMA
// descriptor encoding and kernel selection.  Host code only; it never allocates, frees or
// synchronises, and it never prints.
#include <cmath>
#include <cstring>
#include <algorithm>
#include <mutex>

#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "txl_internal.h"

using namespace txl;

#ifdef TXL_CHECKED
// Range-check failures of the checked build's kernels since the library was loaded (or cleared).
__device__ int g_range_errors;
#endif

namespace txl {

// The counter's device address in the current context, looked up once per context (null in the
// normal build, whose kernels check nothing).
int* range_counter()
{
#ifdef TXL_CHECKED
    static std::mutex mu;
    static int* addr = nullptr;
    static unsigned long long ctx_of = 0;
    unsigned long long ctx = 0;
    const bool have = current_context_id(&ctx);
    std::lock_guard<std::mutex> lock(mu);
    if (!have || !addr || ctx != ctx_of) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_range_errors) != cudaSuccess) return nullptr;
        if (!have && !current_context_id(&ctx)) return nullptr;
        addr = static_cast<int*>(p);
        ctx_of = ctx;
    }
    return addr;
#else
    return nullptr;
#endif
}

}  // namespace txl

namespace {

constexpr int kVersion = 10000;   // 1.0.0

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool encoder_ready()
{
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

inline bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool s16(int64_t stride_elems, int elem) { return ((stride_elems * elem) & 15) == 0; }

// [B][T][H][D] view -> TMA dims (d, h, t, b), box (64, 1, box_t, 1), 128-byte swizzle, bf16.
bool encode_view4(CUtensorMap* map, const void* ptr, int D, int H, int T, int B, int64_t sh,
                  int64_t st, int64_t sb, unsigned box_t = 128)
{
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(T > 0 ? T : 1), static_cast<cuuint64_t>(B)};
    // extent-1 dimensions never move the coordinate; give them a harmless aligned stride
    const int64_t biggest = std::max(std::max(sh, st), sb) * 2;
    const cuuint64_t strides[3] = {
        static_cast<cuuint64_t>(H > 1 ? sh * 2 : biggest),
        static_cast<cuuint64_t>(T > 1 ? st * 2 : biggest),
        static_cast<cuuint64_t>(B > 1 ? sb * 2 : biggest)};
    const cuuint32_t box[4] = {64, 1, box_t, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_rtab(CUtensorMap* map, const void* r, int D, int H, int n_rows, int64_t ld_r)
{
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(n_rows)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld_r * 2),
                                   static_cast<cuuint64_t>(static_cast<int64_t>(H) * ld_r * 2)};
    const cuuint32_t box[3] = {64, 1, 128};
    const cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(r), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool view_ok(const txl_view* v) { return v && v->ptr; }

// Streaming multiprocessors of the current device (queried once per device).
int sm_count()
{
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

bool view_tma_ok(const txl_view* v, int T, int H, int B)
{
    return a16(v->ptr) && (H <= 1 || s16(v->stride_h, 2)) && (T <= 1 || s16(v->stride_t, 2)) &&
           (B <= 1 || s16(v->stride_b, 2)) && v->stride_h > 0 && v->stride_t > 0 && v->stride_b > 0;
}

// Shared argument checks of txl_rel_attn_fwd / txl_rel_attn_path.  Returns TXL_OK or an error.
txl_status check_attn(int B, int L, int H, int D, const txl_view* q, const txl_mem* mem,
                      const txl_view* k_cur, const txl_view* v_cur, const void* r, int64_t ld_r,
                      const txl_view* out, txl_dtype dtype)
{
    if (B < 0 || L < 0 || H <= 0 || D <= 0 || D > 128) return D > 128 ? TXL_ERR_UNSUPPORTED : TXL_ERR_INVALID_ARG;
    if (dtype != TXL_F32 && dtype != TXL_BF16) return TXL_ERR_INVALID_ARG;
    if (!view_ok(q) || !view_ok(k_cur) || !view_ok(v_cur) || !view_ok(out) || !r) return TXL_ERR_INVALID_ARG;
    if (ld_r < D) return TXL_ERR_INVALID_ARG;
    if (mem && mem->M > 0) {
        if (!mem->k || !mem->v || mem->B != B || mem->H != H || mem->D != D || mem->dtype != dtype)
            return TXL_ERR_INVALID_ARG;
        if (mem->wp < 0 || mem->wp >= mem->M || mem->valid < 0 || mem->valid > mem->M) return TXL_ERR_INVALID_ARG;
    } else if (mem && (mem->M < 0 || mem->valid != 0)) {
        return TXL_ERR_INVALID_ARG;
    }
    return TXL_OK;
}

bool attn_tc_eligible(int B, int L, int H, int D, const txl_view* q, const txl_mem* mem,
                      const txl_view* k_cur, const txl_view* v_cur, const void* r, int64_t ld_r,
                      txl_dtype dtype)
{
    if (dtype != TXL_BF16 || D > 128) return false;
    if (!view_tma_ok(q, L, H, B) || !view_tma_ok(k_cur, L, H, B) || !view_tma_ok(v_cur, L, H, B)) return false;
    if (!a16(r) || !s16(ld_r, 2)) return false;
    const int M = mem ? mem->M : 0;
    if (M > 0) {
        txl_view km{mem->k, mem->stride_b, mem->stride_t, mem->stride_h};
        txl_view vm{mem->v, mem->stride_b, mem->stride_t, mem->stride_h};
        if (!view_tma_ok(&km, M, H, B) || !view_tma_ok(&vm, M, H, B)) return false;
        if (mem->wp != 0 && ((mem->wp % 128) != 0 || (M % 128) != 0)) return false;
    }
    return true;
}

}  // namespace

extern "C" {

const char* txl_status_str(txl_status status)
{
    switch (status) {
    case TXL_OK: return "ok";
    case TXL_ERR_INVALID_ARG: return "invalid argument";
    case TXL_ERR_UNSUPPORTED: return "unsupported";
    case TXL_ERR_ALIGNMENT: return "misaligned address or stride";
    case TXL_ERR_CUDA: return "CUDA error";
    case TXL_ERR_TIMEOUT: return "device wait timed out";
    case TXL_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

int txl_version(void) { return kVersion; }

txl_status txl_rel_pos_gen(int n_rows, int d_model, int n_head, int d_head, const void* W_R, int64_t ld_w,
                           void* r, int64_t ld_r, txl_dtype dtype, void* stream)
{
    if (n_rows < 0 || d_model < 2 || (d_model & 1) || d_model > kMaxDModel || n_head <= 0 || d_head <= 0)
        return TXL_ERR_INVALID_ARG;
    if (!W_R || !r || ld_w < static_cast<int64_t>(n_head) * d_head || ld_r < d_head) return TXL_ERR_INVALID_ARG;
    if (dtype != TXL_F32 && dtype != TXL_BF16) return TXL_ERR_INVALID_ARG;
    if (n_rows == 0) return TXL_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == TXL_F32) {
        PosGenF32Params p{};
        p.W = static_cast<const float*>(W_R);
        p.r = static_cast<float*>(r);
        p.ld_w = ld_w;
        p.ld_r = ld_r;
        p.n_rows = n_rows;
        p.d_model = d_model;
        p.H = n_head;
        p.D = d_head;
        return launch_pos_gen_f32(p, s) == cudaSuccess ? TXL_OK : TXL_ERR_CUDA;
    }
    if (!a16(W_R) || !s16(ld_w, 2)) return TXL_ERR_ALIGNMENT;
    if (!encoder_ready()) return TXL_ERR_CUDA;
    PosGenTcParams p;
    std::memset(&p, 0, sizeof(p));
    const int HD = n_head * d_head;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(d_model)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld_w * 2)};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kPosKTile)};
    const cuuint32_t estr[2] = {1, 1};
    if (g_encode(&p.tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(W_R), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return TXL_ERR_CUDA;
    p.r = r;
    p.ld_r = ld_r;
    p.n_rows = n_rows;
    p.d_model = d_model;
    p.H = n_head;
    p.D = d_head;
    p.n_ktiles = (d_model + kPosKTile - 1) / kPosKTile;
    p.dense = (ld_r == d_head && HD % 8 == 0 && a16(r)) ? 1 : 0;
    p.err_flag = nullptr;
    p.log2_freq_step = static_cast<float>(-2.0 * std::log2(10000.0) / static_cast<double>(d_model));
    return launch_pos_gen_tc(p, s) == cudaSuccess ? TXL_OK : TXL_ERR_CUDA;
}

size_t txl_rel_attn_workspace_size(int, int, int, int, const txl_mem*, txl_dtype) { return 0; }

int txl_rel_attn_path(int B, int L, int H, int D, const txl_view* q, const txl_mem* mem, const txl_view* k_cur,
                      const txl_view* v_cur, const void* r, int64_t ld_r, const txl_view* out, txl_dtype dtype)
{
    const txl_status st = check_attn(B, L, H, D, q, mem, k_cur, v_cur, r, ld_r, out, dtype);
    if (st != TXL_OK) return -static_cast<int>(st);
    return attn_tc_eligible(B, L, H, D, q, mem, k_cur, v_cur, r, ld_r, dtype) ? 1 : 2;
}

namespace {

// The fused tcgen05 attention (persistent kernel for d_head <= 64, one CTA per query tile above).
// ring_slots > 0: every key lives in the memory ring (mem->k, mem->v of ring_slots slots); logical
// key j (0 <= j < M + L, M = mem->M the memory length) in slot (wp + j) mod ring_slots.
txl_status attn_tc_launch(int B, int L, int H, int D, int clamp_len, const txl_view* q, const txl_mem* mem,
                          const txl_view* k_cur, const txl_view* v_cur, const float* u, const float* v_bias,
                          const void* r, int64_t ld_r, int n_rows, float scale, const txl_view* out, int* err_flag,
                          cudaStream_t s, int ring_slots, float* lse = nullptr, int lse_out = 0)
{
    const int M = (mem && mem->M > 0) ? mem->M : 0;
    const int valid = M > 0 ? mem->valid : 0;
    const int wp = (M > 0 || ring_slots > 0) ? mem->wp : 0;
    if (!encoder_ready()) return TXL_ERR_CUDA;
    AttnTcParams p;
    std::memset(&p, 0, sizeof(p));
    const int slots = ring_slots > 0 ? ring_slots : M;
    bool ok = encode_view4(&p.tm_q, q->ptr, D, H, L, B, q->stride_h, q->stride_t, q->stride_b) &&
              encode_rtab(&p.tm_r, r, D, H, n_rows, ld_r);
    if (ok && ring_slots > 0) {
        ok = encode_view4(&p.tm_kmem, mem->k, D, H, slots, B, mem->stride_h, mem->stride_t, mem->stride_b) &&
             encode_view4(&p.tm_vmem, mem->v, D, H, slots, B, mem->stride_h, mem->stride_t, mem->stride_b);
        p.tm_kcur = p.tm_kmem;
        p.tm_vcur = p.tm_vmem;
    } else if (ok) {
        ok = encode_view4(&p.tm_kcur, k_cur->ptr, D, H, L, B, k_cur->stride_h, k_cur->stride_t, k_cur->stride_b) &&
             encode_view4(&p.tm_vcur, v_cur->ptr, D, H, L, B, v_cur->stride_h, v_cur->stride_t, v_cur->stride_b);
        if (ok && M > 0)
            ok = encode_view4(&p.tm_kmem, mem->k, D, H, M, B, mem->stride_h, mem->stride_t, mem->stride_b) &&
                 encode_view4(&p.tm_vmem, mem->v, D, H, M, B, mem->stride_h, mem->stride_t, mem->stride_b);
        else if (ok) {
            p.tm_kmem = p.tm_kcur;
            p.tm_vmem = p.tm_vcur;
        }
    }
    if (!ok) return TXL_ERR_CUDA;
    p.u = u;
    p.vb = v_bias;
    p.out = out->ptr;
    p.o_sb = out->stride_b;
    p.o_st = out->stride_t;
    p.o_sh = out->stride_h;
    p.out_a16 = a16(out->ptr) && s16(out->stride_b, 2) && s16(out->stride_t, 2) && s16(out->stride_h, 2);
    p.out_vec = (D % 8) == 0 && p.out_a16;
    p.B = B; p.L = L; p.H = H; p.D = D; p.M = M;
    p.lo = M - valid;
    p.wp = wp;
    p.slots = slots;
    p.ring_all = ring_slots > 0 ? 1 : 0;
    p.chk = range_counter();
    p.C = clamp_len;
    p.n_rows = n_rows;
    p.n_qt = (L + 127) / 128;
    p.n_atoms = D <= 64 ? 1 : 2;
    p.k_steps = (D + 15) / 16;
    p.qscale = scale * 1.4426950408889634f;
    p.err_flag = err_flag;
    p.lse = lse;
    p.lse_out = lse_out;
    if (lse && p.n_atoms != 1) return TXL_ERR_UNSUPPORTED;
    if (p.n_atoms == 1) {
        if (static_cast<int64_t>(p.n_qt) * H * B > INT32_MAX) return TXL_ERR_UNSUPPORTED;
        // even and odd query rows as two maps stepping two tokens per row; the odd map starts
        // one token in and has floor(L/2) rows, so no load reads past the tensor (with L = 1
        // the odd rows are taken from the even map: they belong to no query and are not stored)
        const char* q0 = static_cast<const char*>(q->ptr);
        bool okq = encode_view4(&p.tm_qe, q0, D, H, (L + 1) / 2, B, q->stride_h, 2 * q->stride_t,
                                q->stride_b, 64);
        if (okq && L / 2 > 0)
            okq = encode_view4(&p.tm_qo, q0 + q->stride_t * 2, D, H, L / 2, B, q->stride_h,
                               2 * q->stride_t, q->stride_b, 64);
        else
            p.tm_qo = p.tm_qe;
        if (!okq) return TXL_ERR_CUDA;
        const int sms = sm_count();
        if (sms <= 0) return TXL_ERR_CUDA;
        const int64_t items = static_cast<int64_t>(p.n_qt) * H * B;
        const int G = static_cast<int>(std::min<int64_t>(items, sms));
        const int64_t per_cls = static_cast<int64_t>(H) * B;
        p.sched_mode = (p.n_qt <= kMaxSchedClasses && per_cls <= INT32_MAX &&
                        schedule_items(G, p.n_qt, static_cast<int>(per_cls), (M + 127 - p.lo) / 128 + 1,
                                       p.sched_counts, kSchedCapacity))
                           ? 1 : 0;
        return launch_attn_persist(p, sms, s) == cudaSuccess ? TXL_OK : TXL_ERR_CUDA;
    }
    if (B > 65535 || H > 65535) return TXL_ERR_UNSUPPORTED;
    return launch_attn_tc(p, s) == cudaSuccess ? TXL_OK : TXL_ERR_CUDA;
}

// The learned-table variant on the persistent tcgen05 kernel (table mode, with or without a key
// mask): bf16, d_head <= 64, L <= max_len (so no pair's index i - j + max_len - 1 leaves the table and
// no clamp applies), 16-byte aligned bases and strides for q, k, v and the table.
bool table_persist_eligible(int B, int L, int H, int D, int max_len, const txl_view* q, const txl_view* k,
                       const txl_view* v, const void* r_table, int64_t ld_r, const uint8_t* key_mask,
                       txl_dtype dtype)
{
    (void)key_mask;
    if (dtype != TXL_BF16 || D > 64 || L > max_len) return false;
    if (!view_tma_ok(q, L, H, B) || !view_tma_ok(k, L, H, B) || !view_tma_ok(v, L, H, B)) return false;
    if (!a16(r_table) || !s16(ld_r, 2)) return false;
    return static_cast<int64_t>((L + 127) / 128) * H * B <= INT32_MAX;
}

txl_status table_tc_launch(int B, int L, int H, int D, int max_len, const txl_view* q, const txl_view* k,
                           const txl_view* v, const float* u, const float* v_bias, const void* r_table, int64_t ld_r,
                           const uint8_t* key_mask, float scale, const txl_view* out, cudaStream_t s)
{
    if (!encoder_ready()) return TXL_ERR_CUDA;
    AttnTcParams p;
    std::memset(&p, 0, sizeof(p));
    const int n_rows = 2 * max_len - 1;
    bool ok = encode_rtab(&p.tm_r, r_table, D, H, n_rows, ld_r) &&
              encode_view4(&p.tm_kcur, k->ptr, D, H, L, B, k->stride_h, k->stride_t, k->stride_b) &&
              encode_view4(&p.tm_vcur, v->ptr, D, H, L, B, v->stride_h, v->stride_t, v->stride_b);
    // even and odd query rows as two maps stepping two tokens per row (as for the main path)
    const char* q0 = static_cast<const char*>(q->ptr);
    ok = ok && encode_view4(&p.tm_qe, q0, D, H, (L + 1) / 2, B, q->stride_h, 2 * q->stride_t, q->stride_b, 64);
    if (ok && L / 2 > 0)
        ok = encode_view4(&p.tm_qo, q0 + q->stride_t * 2, D, H, L / 2, B, q->stride_h, 2 * q->stride_t,
                          q->stride_b, 64);
    else
        p.tm_qo = p.tm_qe;
    if (!ok) return TXL_ERR_CUDA;
    p.tm_kmem = p.tm_kcur;
    p.tm_vmem = p.tm_vcur;
    p.u = u;
    p.vb = v_bias;
    p.out = out->ptr;
    p.o_sb = out->stride_b;
    p.o_st = out->stride_t;
    p.o_sh = out->stride_h;
    p.out_a16 = a16(out->ptr) && s16(out->stride_b, 2) && s16(out->stride_t, 2) && s16(out->stride_h, 2);
    p.out_vec = (D % 8) == 0 && p.out_a16;
    p.B = B; p.L = L; p.H = H; p.D = D;
    p.chk = range_counter();
    p.C = 1 << 30;                            // no clamp: every chunk is multiplied
    p.n_rows = n_rows;
    p.n_qt = (L + 127) / 128;
    p.n_atoms = 1;
    p.k_steps = (D + 15) / 16;
    // s = scale q.k + scale q.r + u.k + v.r in the log2 domain: Qu = log2(e) (scale q + u) and
    // Qv = log2(e) (scale q + v), the scale on q alone
    p.qscale = scale * 1.4426950408889634f;
    p.bscale = 1.4426950408889634f;
    p.table = key_mask ? 2 : 1;
    p.key_mask = key_mask;
    p.roff = max_len - 1;
    p.sched_mode = 0;                         // every item has the same key tiles: serpentine order
    const int sms = sm_count();
    if (sms <= 0) return TXL_ERR_CUDA;
    return launch_attn_persist(p, sms, s) == cudaSuccess ? TXL_OK : TXL_ERR_CUDA;
}

// Decode calls with three or more new queries per (b, h) take the persistent fused kernel when it
// accepts the inputs: one query tile over every key outruns the chunked decode kernels there (B8
// H16 D64 M4096 bf16: 54 us for any L <= 16, against 76 us at L = 3, 220 us at L = 8 and 574 us at
// L = 16; at L = 1 and 2 the decode kernels take 40 and 49 us).  It needs no workspace.
constexpr int kDecodeFusedMinL = 3;

bool decode_takes_fused(int B, int L, int H, int D, const txl_view* q, const txl_mem* mem, const txl_view* k_cur,
                        const txl_view* v_cur, const void* r, int64_t ld_r, txl_dtype dtype)
{
    return L >= kDecodeFusedMinL && D <= 64 && attn_tc_eligible(B, L, H, D, q, mem, k_cur, v_cur, r, ld_r, dtype);
}

}  // namespace

txl_status txl_rel_attn_fwd_lse(int B, int L, int H, int D, int clamp_len, const txl_view* q, const txl_mem* mem,
                                const txl_view* k_cur, const txl_view* v_cur, const float* u, const float* v_bias,
                                const void* r, int64_t ld_r, int n_rows, float scale, const txl_view* out,
                                float* lse, txl_dtype dtype, void* workspace, size_t workspace_bytes, int* err_flag,
                                void* stream)
{
    if (!lse) return TXL_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return TXL_ERR_ALIGNMENT;
    txl_status st = check_attn(B, L, H, D, q, mem, k_cur, v_cur, r, ld_r, out, dtype);
    if (st != TXL_OK) return st;
    if (clamp_len < 0 || !u || !v_bias) return TXL_ERR_INVALID_ARG;
    const int M = (mem && mem->M > 0) ? mem->M : 0;
    if (n_rows < std::min(M + L, clamp_len + 1)) return TXL_ERR_INVALID_ARG;
    // the statistics come from the persistent fused kernel (bf16, d_head <= 64) alone
    if (D > 64 || !attn_tc_eligible(B, L, H, D, q, mem, k_cur, v_cur, r, ld_r, dtype)) return TXL_ERR_UNSUPPORTED;
    (void)workspace;
    (void)workspace_bytes;
    if (B == 0 || L == 0) return TXL_OK;
    if (scale <= 0.f) scale = 1.0f / std::sqrt(static_cast<float>(D));
    return attn_tc_launch(B, L, H, D, clamp_len, q, mem, k_cur, v_cur, u, v_bias, r, ld_r, n_rows, scale, out, err_flag,
                          static_cast<cudaStream_t>(stream), 0, lse, 1);
}

txl_status txl_rel_attn_fwd(int B, int L, int H, int D, int clamp_len, const txl_view* q, const txl_mem* mem,
                            const txl_view* k_cur, const txl_view* v_cur, const float* u, const float* v_bias,
                            const void* r, int64_t ld_r, int n_rows, float scale, const txl_view* out,
                            txl_dtype dtype, void* workspace, size_t workspace_bytes, int* err_flag, void* stream)
{
    (void)workspace;
    (void)workspace_bytes;
    txl_status st = check_attn(B, L, H, D, q, mem, k_cur, v_cur, r, ld_r, out, dtype);
    if (st != TXL_OK) return st;
    if (clamp_len < 0 || !u || !v_bias) return TXL_ERR_INVALID_ARG;
    const int M = (mem && mem->M > 0) ? mem->M : 0;
    const int valid = M > 0 ? mem->valid : 0;
    const int wp = M > 0 ? mem->wp : 0;
    const int need_rows = std::min(M + L, clamp_len + 1);
    if (n_rows < need_rows) return TXL_ERR_INVALID_ARG;
    if (B == 0 || L == 0) return TXL_OK;
    if (scale <= 0.f) scale = 1.0f / std::sqrt(static_cast<float>(D));
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    if (attn_tc_eligible(B, L, H, D, q, mem, k_cur, v_cur, r, ld_r, dtype))
        return attn_tc_launch(B, L, H, D, clamp_len, q, mem, k_cur, v_cur, u, v_bias, r, ld_r, n_rows, scale, out,
                              err_flag, s, 0);

    AttnSimtParams p;
    std::memset(&p, 0, sizeof(p));
    p.q = q->ptr; p.q_sb = q->stride_b; p.q_st = q->stride_t; p.q_sh = q->stride_h;
    if (M > 0) {
        p.kmem = mem->k; p.vmem = mem->v;
        p.m_sb = mem->stride_b; p.m_st = mem->stride_t; p.m_sh = mem->stride_h;
    }
    p.kcur = k_cur->ptr; p.kc_sb = k_cur->stride_b; p.kc_st = k_cur->stride_t; p.kc_sh = k_cur->stride_h;
    p.vcur = v_cur->ptr; p.vc_sb = v_cur->stride_b; p.vc_st = v_cur->stride_t; p.vc_sh = v_cur->stride_h;
    p.out = out->ptr; p.o_sb = out->stride_b; p.o_st = out->stride_t; p.o_sh = out->stride_h;
    p.u = u; p.vb = v_bias;
    p.r = r; p.r_row = static_cast<int64_t>(H) * ld_r; p.r_head = ld_r;
    p.B = B; p.L = L; p.H = H; p.D = D; p.M = M; p.lo = M - valid; p.wp = wp; p.C = clamp_len;
    p.scale = scale;
    p.n_rows = n_rows;
    p.chk = range_counter();
    return launch_attn_simt(p, dtype, s) == cudaSuccess ? TXL_OK : TXL_ERR_CUDA;
}

size_t txl_rel_attn_decode_workspace_size(int B, int L, int H, int D, const txl_mem* mem)
{
    if (B <= 0 || L <= 0 || H <= 0 || D <= 0 || D > 128 || L > kDecodeMaxL) return 0;
    const int64_t M = (mem && mem->M > 0) ? mem->M : 0;
    const int64_t n_chunks = (M + L + kDecodeChunk - 1) / kDecodeChunk;
    return static_cast<size_t>(B) * H * L * n_chunks * (D + 2) * sizeof(float);
}

txl_status txl_rel_attn_decode(int B, int L, int H, int D, int clamp_len, const txl_view* q, const txl_mem* mem,
                               const txl_view* k_cur, const txl_view* v_cur, const float* u, const float* v_bias,
                               const void* r, int64_t ld_r, int n_rows, float scale, const txl_view* out,
                               txl_dtype dtype, void* workspace, size_t workspace_bytes, void* stream)
{
    txl_status st = check_attn(B, L, H, D, q, mem, k_cur, v_cur, r, ld_r, out, dtype);
    if (st != TXL_OK) return st;
    if (L > kDecodeMaxL) return TXL_ERR_UNSUPPORTED;
    if (clamp_len < 0 || !u || !v_bias) return TXL_ERR_INVALID_ARG;
    const int M = (mem && mem->M > 0) ? mem->M : 0;
    const int valid = M > 0 ? mem->valid : 0;
    const int wp = M > 0 ? mem->wp : 0;
    if (n_rows < std::min(M + L, clamp_len + 1)) return TXL_ERR_INVALID_ARG;
    if (B == 0 || L == 0) return TXL_OK;
    const size_t need = txl_rel_attn_decode_workspace_size(B, L, H, D, mem);
    if (!workspace || workspace_bytes < need || !a16(workspace)) return TXL_ERR_WORKSPACE;
    if (B > 65535 || H > 65535) return TXL_ERR_UNSUPPORTED;
    if (scale <= 0.f) scale = 1.0f / std::sqrt(static_cast<float>(D));
    if (decode_takes_fused(B, L, H, D, q, mem, k_cur, v_cur, r, ld_r, dtype))
        return attn_tc_launch(B, L, H, D, clamp_len, q, mem, k_cur, v_cur, u, v_bias, r, ld_r, n_rows, scale, out,
                              nullptr, static_cast<cudaStream_t>(stream), 0);
    const int elem = dtype == TXL_F32 ? 4 : 2;
    auto rows16 = [&](const void* ptr, int64_t sb, int64_t st_, int64_t sh) {
        return a16(ptr) && s16(sb, elem) && s16(st_, elem) && s16(sh, elem);
    };
    DecodeParams p;
    std::memset(&p, 0, sizeof(p));
    p.q = q->ptr; p.q_sb = q->stride_b; p.q_st = q->stride_t; p.q_sh = q->stride_h;
    if (M > 0) {
        p.kmem = mem->k; p.vmem = mem->v;
        p.m_sb = mem->stride_b; p.m_st = mem->stride_t; p.m_sh = mem->stride_h;
    }
    p.kcur = k_cur->ptr; p.kc_sb = k_cur->stride_b; p.kc_st = k_cur->stride_t; p.kc_sh = k_cur->stride_h;
    p.vcur = v_cur->ptr; p.vc_sb = v_cur->stride_b; p.vc_st = v_cur->stride_t; p.vc_sh = v_cur->stride_h;
    p.out = out->ptr; p.o_sb = out->stride_b; p.o_st = out->stride_t; p.o_sh = out->stride_h;
    p.u = u; p.vb = v_bias;
    p.r = r; p.r_row = static_cast<int64_t>(H) * ld_r; p.r_head = ld_r;
    p.B = B; p.L = L; p.H = H; p.D = D; p.Dp = (D + 7) / 8 * 8; p.M = M; p.lo = M - valid; p.wp = wp;
    p.C = clamp_len;
    p.qscale = scale * 1.4426950408889634f;
    p.n_chunks = static_cast<int>((static_cast<int64_t>(M) + L + kDecodeChunk - 1) / kDecodeChunk);
    p.part = static_cast<float*>(workspace);
    p.vec_kv = rows16(k_cur->ptr, k_cur->stride_b, k_cur->stride_t, k_cur->stride_h) &&
               rows16(v_cur->ptr, v_cur->stride_b, v_cur->stride_t, v_cur->stride_h) &&
               (M == 0 || (rows16(mem->k, mem->stride_b, mem->stride_t, mem->stride_h) &&
                           rows16(mem->v, mem->stride_b, mem->stride_t, mem->stride_h)));
    p.vec_r = a16(r) && s16(ld_r, elem);
    return launch_decode(p, dtype, static_cast<cudaStream_t>(stream)) == cudaSuccess ? TXL_OK : TXL_ERR_CUDA;
}

txl_status txl_rel_attn_decode_noalloc(int B, int L, int H, int D, int clamp_len, const txl_view* q,
                                       const txl_mem* mem, const txl_view* k_cur, const txl_view* v_cur,
                                       const float* u, const float* v_bias, const void* r, int64_t ld_r,
                                       int n_rows, float scale, const txl_view* out, txl_dtype dtype,
                                       void* stream)
{
    txl_status st = check_attn(B, L, H, D, q, mem, k_cur, v_cur, r, ld_r, out, dtype);
    if (st != TXL_OK) return st;
    if (L > kDecodeMaxL) return TXL_ERR_UNSUPPORTED;
    if (clamp_len < 0 || !u || !v_bias) return TXL_ERR_INVALID_ARG;
    const int M = (mem && mem->M > 0) ? mem->M : 0;
    const int valid = M > 0 ? mem->valid : 0;
    const int wp = M > 0 ? mem->wp : 0;
    if (n_rows < std::min(M + L, clamp_len + 1)) return TXL_ERR_INVALID_ARG;
    if (B == 0 || L == 0) return TXL_OK;
    // the partial results must fit the library's static scratch
    const int64_t n_chunks = (static_cast<int64_t>(M) + L + kDecodeChunk - 1) / kDecodeChunk;
    const double need = static_cast<double>(B) * H * L * n_chunks * (D + 2) * sizeof(float);
    if (need > static_cast<double>(kDecodeStaticScratchBytes)) return TXL_ERR_WORKSPACE;
    if (B > 65535 || H > 65535) return TXL_ERR_UNSUPPORTED;
    if (scale <= 0.f) scale = 1.0f / std::sqrt(static_cast<float>(D));
    if (decode_takes_fused(B, L, H, D, q, mem, k_cur, v_cur, r, ld_r, dtype))
        return attn_tc_launch(B, L, H, D, clamp_len, q, mem, k_cur, v_cur, u, v_bias, r, ld_r, n_rows, scale, out,
                              nullptr, static_cast<cudaStream_t>(stream), 0);
    float* scratch = nullptr;
    if (decode_static_scratch(&scratch) != cudaSuccess || !scratch) return TXL_ERR_CUDA;
    const int elem = dtype == TXL_F32 ? 4 : 2;
    auto rows16 = [&](const void* ptr, int64_t sb, int64_t st_, int64_t sh) {
        return a16(ptr) && s16(sb, elem) && s16(st_, elem) && s16(sh, elem);
    };
    DecodeParams p;
    std::memset(&p, 0, sizeof(p));
    p.q = q->ptr; p.q_sb = q->stride_b; p.q_st = q->stride_t; p.q_sh = q->stride_h;
    if (M > 0) {
        p.kmem = mem->k; p.vmem = mem->v;
        p.m_sb = mem->stride_b; p.m_st = mem->stride_t; p.m_sh = mem->stride_h;
    }
    p.kcur = k_cur->ptr; p.kc_sb = k_cur->stride_b; p.kc_st = k_cur->stride_t; p.kc_sh = k_cur->stride_h;
    p.vcur = v_cur->ptr; p.vc_sb = v_cur->stride_b; p.vc_st = v_cur->stride_t; p.vc_sh = v_cur->stride_h;
    p.out = out->ptr; p.o_sb = out->stride_b; p.o_st = out->stride_t; p.o_sh = out->stride_h;
    p.u = u; p.vb = v_bias;
    p.r = r; p.r_row = static_cast<int64_t>(H) * ld_r; p.r_head = ld_r;
    p.B = B; p.L = L; p.H = H; p.D = D; p.Dp = (D + 7) / 8 * 8; p.M = M; p.lo = M - valid; p.wp = wp;
    p.C = clamp_len;
    p.qscale = scale * 1.4426950408889634f;
    p.n_chunks = static_cast<int>(n_chunks);
    p.part = scratch;
    p.vec_kv = rows16(k_cur->ptr, k_cur->stride_b, k_cur->stride_t, k_cur->stride_h) &&
               rows16(v_cur->ptr, v_cur->stride_b, v_cur->stride_t, v_cur->stride_h) &&
               (M == 0 || (rows16(mem->k, mem->stride_b, mem->stride_t, mem->stride_h) &&
                           rows16(mem->v, mem->stride_b, mem->stride_t, mem->stride_h)));
    p.vec_r = a16(r) && s16(ld_r, elem);
    return launch_decode(p, dtype, static_cast<cudaStream_t>(stream)) == cudaSuccess ? TXL_OK : TXL_ERR_CUDA;
}

txl_status txl_mem_push(txl_mem* mem, const txl_view* k_new, const txl_view* v_new, int L, void* stream)
{
    if (!mem || !view_ok(k_new) || !view_ok(v_new) || L < 0) return TXL_ERR_INVALID_ARG;
    if (mem->M < 0 || mem->B < 0 || mem->H <= 0 || mem->D <= 0) return TXL_ERR_INVALID_ARG;
    if (mem->dtype != TXL_F32 && mem->dtype != TXL_BF16) return TXL_ERR_INVALID_ARG;
    if (mem->M == 0) return mem->valid == 0 ? TXL_OK : TXL_ERR_INVALID_ARG;
    if (!mem->k || !mem->v || mem->wp < 0 || mem->wp >= mem->M || mem->valid < 0 || mem->valid > mem->M)
        return TXL_ERR_INVALID_ARG;
    if (L == 0) return TXL_OK;
    const int elem = mem->dtype == TXL_F32 ? 4 : 2;
    MemPushParams p{};
    p.chk = range_counter();
    p.k_new = k_new->ptr; p.v_new = v_new->ptr;
    p.n_sb = k_new->stride_b; p.n_st = k_new->stride_t; p.n_sh = k_new->stride_h;
    p.nv_sb = v_new->stride_b; p.nv_st = v_new->stride_t; p.nv_sh = v_new->stride_h;
    p.k = mem->k; p.v = mem->v;
    p.m_sb = mem->stride_b; p.m_st = mem->stride_t; p.m_sh = mem->stride_h;
    p.B = mem->B; p.H = mem->H; p.D = mem->D; p.M = mem->M; p.wp = mem->wp;
    p.t0 = L > mem->M ? L - mem->M : 0;
    p.n_t = L - p.t0;
    p.elem_bytes = elem;
    const bool rows16 = ((static_cast<int64_t>(mem->D) * elem) & 15) == 0;
    p.vec16 = rows16 && a16(k_new->ptr) && a16(v_new->ptr) && a16(mem->k) && a16(mem->v) &&
              s16(k_new->stride_b, elem) && s16(k_new->stride_t, elem) && s16(k_new->stride_h, elem) &&
              s16(v_new->stride_b, elem) && s16(v_new->stride_t, elem) && s16(v_new->stride_h, elem) &&
              s16(mem->stride_b, elem) && s16(mem->stride_t, elem) && s16(mem->stride_h, elem) &&
              static_cast<int64_t>(mem->B) * p.n_t <= INT32_MAX &&
              static_cast<int64_t>(mem->M) + L <= INT32_MAX;         // 32-bit row and slot arithmetic
    if (launch_mem_push(p, static_cast<cudaStream_t>(stream)) != cudaSuccess) return TXL_ERR_CUDA;
    mem->wp = static_cast<int>((static_cast<int64_t>(mem->wp) + L) % mem->M);
    mem->valid = std::min(mem->valid + L, mem->M);
    return TXL_OK;
}

namespace {

// 2D bf16 tensor map over a row-major [rows][ld] matrix, columns 0..cols-1, box (64, box_rows).
bool encode_rows(CUtensorMap* map, const void* ptr, int64_t cols, int64_t rows, int64_t ld, unsigned box_rows)
{
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * 2)};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace {

// K and V column blocks of the q|k|v product routed into ring slots (the fused layer step).
struct LinearSplit {
    int hd, seg_len, slot0, slots;
    void* k_ring;
    void* v_ring;
    int64_t ring_stride_b;           // elements between batch entries of a ring ([B][slots][H*D])
};

// [B][slots][hd] ring as a 3D TMA map (hd, slots, B) with 64 x 32 x 1 boxes, 128-byte swizzle: the
// layout of one staged 32-row, 64-column block of the product's epilogue.
bool encode_ring_store(CUtensorMap* map, void* ring, int hd, int slots, int B, int64_t stride_b)
{
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(hd), static_cast<cuuint64_t>(slots), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(hd) * 2, static_cast<cuuint64_t>(stride_b) * 2};
    const cuuint32_t box[3] = {64, 32, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ring, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

txl_status linear_launch(int m, int n, int k, const void* X, int64_t ld_x, const void* W, int64_t ld_w, void* Y,
                         int64_t ld_y, int* err_flag, cudaStream_t stream, const LinearSplit* split)
{
    if (!a16(X) || !a16(W) || !s16(ld_x, 2) || !s16(ld_w, 2)) return TXL_ERR_ALIGNMENT;
    if (static_cast<int64_t>(m) + 127 > INT32_MAX || static_cast<int64_t>(n) + 255 > INT32_MAX) return TXL_ERR_INVALID_ARG;
    if (!encoder_ready()) return TXL_ERR_CUDA;
    LinearParams p;
    std::memset(&p, 0, sizeof(p));
    if (!encode_rows(&p.tm_x, X, k, m, ld_x, 128) || !encode_rows(&p.tm_w, W, n, k, ld_w, 64)) return TXL_ERR_CUDA;
    p.y = Y;
    p.ld_y = ld_y;
    p.m = m;
    p.n = n;
    p.k = k;
    p.tiles_n = (n + 255) / 256;
    p.m_tiles = (m + 127) / 128;
    const int64_t tiles = static_cast<int64_t>(p.m_tiles) * p.tiles_n;
    if (tiles > INT32_MAX) return TXL_ERR_INVALID_ARG;
    p.n_tiles = static_cast<int>(tiles);
    p.k_tiles = (k + 63) / 64;
    p.vec = (a16(Y) && s16(ld_y, 2)) ? 1 : 0;
    if (split) {
        // Y receives only the first hd columns; the rest go to the rings
        if (!p.vec || !encode_rows(&p.tm_y, Y, split->hd, m, ld_y, 32) ||
            !encode_ring_store(&p.tm_k, split->k_ring, split->hd, split->slots, m / split->seg_len, split->ring_stride_b) ||
            !encode_ring_store(&p.tm_v, split->v_ring, split->hd, split->slots, m / split->seg_len, split->ring_stride_b))
            return TXL_ERR_CUDA;
        p.tma_store = 1;
        p.split_hd = split->hd;
        p.seg_len = split->seg_len;
        p.slot0 = split->slot0;
        p.slots = split->slots;
    } else {
        p.tma_store = (p.vec && encode_rows(&p.tm_y, Y, n, m, ld_y, 32)) ? 1 : 0;
    }
    p.err_flag = err_flag;
    const int sms = sm_count();
    if (sms <= 0) return TXL_ERR_CUDA;
    return launch_linear(p, sms, stream) == cudaSuccess ? TXL_OK : TXL_ERR_CUDA;
}

}  // namespace

txl_status txl_linear(int m, int n, int k, const void* X, int64_t ld_x, const void* W, int64_t ld_w, void* Y,
                      int64_t ld_y, txl_dtype dtype, int* err_flag, void* stream)
{
    if (m < 0 || n < 0 || k <= 0 || !X || !W || !Y) return TXL_ERR_INVALID_ARG;
    if (ld_x < k || ld_w < n || ld_y < n) return TXL_ERR_INVALID_ARG;
    if (dtype == TXL_F32) return TXL_ERR_UNSUPPORTED;
    if (dtype != TXL_BF16) return TXL_ERR_INVALID_ARG;
    if (m == 0 || n == 0) return TXL_OK;
    return linear_launch(m, n, k, X, ld_x, W, ld_w, Y, ld_y, err_flag, static_cast<cudaStream_t>(stream), nullptr);
}

size_t txl_rel_attn_layer_workspace_size(int B, int L, int H, int D)
{
    if (B <= 0 || L <= 0 || H <= 0 || D <= 0) return 0;
    // q|k|v of the segment [B*L][3*H*D] and the attention output [B*L][H*D], bf16
    return static_cast<size_t>(B) * L * H * D * 4 * 2;
}

txl_status txl_rel_attn_layer(int B, int L, int H, int D, int d_model, int clamp_len, const void* h, int64_t ld_h,
                              txl_mem* mem, const void* W_qkv, const void* W_o, const float* u, const float* v_bias,
                              const void* r, int64_t ld_r, int n_rows, float scale, void* y, int64_t ld_y,
                              void* workspace, size_t workspace_bytes, int* err_flag, void* stream)
{
    if (B < 0 || L < 0 || H <= 0 || D <= 0 || d_model <= 0 || clamp_len < 0) return TXL_ERR_INVALID_ARG;
    if (!h || !W_qkv || !W_o || !u || !v_bias || !r || !y) return TXL_ERR_INVALID_ARG;
    if (ld_h < d_model || ld_y < d_model) return TXL_ERR_INVALID_ARG;
    if (mem && mem->M > 0 && (mem->B != B || mem->H != H || mem->D != D || mem->dtype != TXL_BF16))
        return TXL_ERR_INVALID_ARG;
    const int64_t HD = static_cast<int64_t>(H) * D;
    if ((HD & 7) || (d_model & 7)) return TXL_ERR_ALIGNMENT;      // 16-byte rows of q|k|v, attn, y
    if (B == 0 || L == 0) return TXL_OK;
    const size_t need = txl_rel_attn_layer_workspace_size(B, L, H, D);
    if (!workspace || workspace_bytes < need) return TXL_ERR_WORKSPACE;
    if (!a16(workspace)) return TXL_ERR_ALIGNMENT;
    const int rows = B * L;
    if (static_cast<int64_t>(B) * L > INT32_MAX) return TXL_ERR_INVALID_ARG;
    __nv_bfloat16* qkv = static_cast<__nv_bfloat16*>(workspace);
    __nv_bfloat16* attn = qkv + static_cast<int64_t>(rows) * 3 * HD;
    // Q = h W_q and the segment's K = h W_k, V = h W_v in one product with [W_q W_k W_v]
    txl_status st = txl_linear(rows, static_cast<int>(3 * HD), d_model, h, ld_h, W_qkv, 3 * HD, qkv, 3 * HD,
                               TXL_BF16, err_flag, stream);
    if (st != TXL_OK) return st;
    // the attention over [memory ++ segment]: the memory holds the K, V of earlier positions
    const txl_view q{qkv, L * 3 * HD, 3 * HD, D};
    const txl_view kc{qkv + HD, L * 3 * HD, 3 * HD, D};
    const txl_view vc{qkv + 2 * HD, L * 3 * HD, 3 * HD, D};
    const txl_view out{attn, L * HD, HD, D};
    st = txl_rel_attn_fwd(B, L, H, D, clamp_len, &q, mem, &kc, &vc, u, v_bias, r, ld_r, n_rows, scale, &out,
                          TXL_BF16, nullptr, 0, err_flag, stream);
    if (st != TXL_OK) return st;
    // y = concat_h(attn) W_o
    st = txl_linear(rows, d_model, static_cast<int>(HD), attn, HD, W_o, d_model, y, ld_y, TXL_BF16, err_flag, stream);
    if (st != TXL_OK) return st;
    // the segment's K, V enter the memory (FIFO)
    if (mem && mem->M > 0) return txl_mem_push(mem, &kc, &vc, L, stream);
    return TXL_OK;
}

size_t txl_rel_attn_layer_fused_workspace_size(int B, int L, int H, int D)
{
    if (B <= 0 || L <= 0 || H <= 0 || D <= 0) return 0;
    // q of the segment [B*L][H*D] and the attention output [B*L][H*D], bf16
    return static_cast<size_t>(B) * L * H * D * 2 * 2;
}

txl_status txl_rel_attn_layer_fused(int B, int L, int H, int D, int d_model, int clamp_len, const void* h,
                                    int64_t ld_h, txl_mem* mem, int mem_len, const void* W_qkv, const void* W_o,
                                    const float* u, const float* v_bias, const void* r, int64_t ld_r, int n_rows,
                                    float scale, void* y, int64_t ld_y, void* workspace, size_t workspace_bytes,
                                    int* err_flag, void* stream)
{
    if (B < 0 || L < 0 || H <= 0 || D <= 0 || d_model <= 0 || clamp_len < 0 || mem_len < 0) return TXL_ERR_INVALID_ARG;
    if (!h || !W_qkv || !W_o || !u || !v_bias || !r || !y || !mem || !mem->k || !mem->v) return TXL_ERR_INVALID_ARG;
    if (ld_h < d_model || ld_y < d_model || ld_r < D) return TXL_ERR_INVALID_ARG;
    const int slots = mem->M;
    if (mem->B != B || mem->H != H || mem->D != D || mem->dtype != TXL_BF16) return TXL_ERR_INVALID_ARG;
    if (static_cast<int64_t>(mem_len) + L > slots || mem->valid < 0 || mem->valid > mem_len || mem->wp < 0 ||
        mem->wp >= slots)
        return TXL_ERR_INVALID_ARG;
    if (n_rows < std::min(mem_len + L, clamp_len + 1)) return TXL_ERR_INVALID_ARG;
    const int64_t HD = static_cast<int64_t>(H) * D;
    // the persistent tcgen05 attention with tiles of 128 keys aligned to ring slots, product blocks
    // of 64 columns that never straddle the q, k, v column ranges
    if (D > 64 || (D & 7) || (HD % 64) || (d_model & 7) || (L % 128) || (mem_len % 128) || (slots % 128) ||
        (mem->wp % 128))
        return TXL_ERR_UNSUPPORTED;
    if (mem->stride_h != D || mem->stride_t != HD || mem->stride_b != static_cast<int64_t>(slots) * HD)
        return TXL_ERR_UNSUPPORTED;
    if (!a16(mem->k) || !a16(mem->v) || !a16(r) || !s16(ld_r, 2) || !a16(y) || !s16(ld_y, 2)) return TXL_ERR_ALIGNMENT;
    if (B == 0 || L == 0) return TXL_OK;
    if (static_cast<int64_t>(B) * L > INT32_MAX / 4) return TXL_ERR_INVALID_ARG;
    const size_t need = txl_rel_attn_layer_fused_workspace_size(B, L, H, D);
    if (!workspace || workspace_bytes < need) return TXL_ERR_WORKSPACE;
    if (!a16(workspace)) return TXL_ERR_ALIGNMENT;
    if (scale <= 0.f) scale = 1.0f / std::sqrt(static_cast<float>(D));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int rows = B * L;
    __nv_bfloat16* qbuf = static_cast<__nv_bfloat16*>(workspace);
    __nv_bfloat16* attn = qbuf + static_cast<int64_t>(rows) * HD;
    // Q = h W_q into the workspace; K = h W_k and V = h W_v straight into the ring slots that follow
    // the memory, (wp + mem_len + t) mod slots
    const LinearSplit split{static_cast<int>(HD), L, static_cast<int>((static_cast<int64_t>(mem->wp) + mem_len) % slots),
                            slots, mem->k, mem->v, mem->stride_b};
    txl_status st = linear_launch(rows, static_cast<int>(3 * HD), d_model, h, ld_h, W_qkv, 3 * HD, qbuf, HD, err_flag,
                                  s, &split);
    if (st != TXL_OK) return st;
    // the attention over [memory ++ segment], every key read from the ring
    const txl_view q{qbuf, L * HD, HD, D};
    const txl_view out{attn, L * HD, HD, D};
    txl_mem window = *mem;
    window.M = mem_len;
    st = attn_tc_launch(B, L, H, D, clamp_len, &q, &window, nullptr, nullptr, u, v_bias, r, ld_r, n_rows, scale, &out,
                        err_flag, s, slots);
    if (st != TXL_OK) return st;
    // y = concat_h(attn) W_o
    st = linear_launch(rows, d_model, static_cast<int>(HD), attn, HD, W_o, d_model, y, ld_y, err_flag, s, nullptr);
    if (st != TXL_OK) return st;
    // the segment is now the newest part of the memory: no copy, the window moves
    mem->wp = static_cast<int>((static_cast<int64_t>(mem->wp) + L) % slots);
    mem->valid = std::min(mem->valid + L, mem_len);
    return TXL_OK;
}

size_t txl_rel_attn_bwd_workspace_size(int B, int L, int H, int D)
{
    if (B <= 0 || L <= 0 || H <= 0 || D <= 0) return 0;
    const size_t rows = static_cast<size_t>(B) * L * H;
    return rows * 2 * sizeof(float) + rows * D * 2 * sizeof(float);
}

namespace {

// The gradient kernels' parameters from a backward call's arguments (checked by the caller).
BwdParams bwd_params(int B, int L, int H, int D, int clamp_len, const txl_view* q, const txl_mem* mem,
                     const txl_view* k_cur, const txl_view* v_cur, const float* u, const float* v_bias, const void* r,
                     int64_t ld_r, int n_rows, float scale, const txl_view* out, const txl_view* d_out, float* dq,
                     float* dk_cur, float* dv_cur, float* du, float* dv_bias, float* dr)
{
    const int M = (mem && mem->M > 0) ? mem->M : 0;
    const int valid = M > 0 ? mem->valid : 0;
    BwdParams p;
    std::memset(&p, 0, sizeof(p));
    AttnSimtParams& a = p.a;
    a.q = q->ptr; a.q_sb = q->stride_b; a.q_st = q->stride_t; a.q_sh = q->stride_h;
    if (M > 0) {
        a.kmem = mem->k; a.vmem = mem->v;
        a.m_sb = mem->stride_b; a.m_st = mem->stride_t; a.m_sh = mem->stride_h;
    }
    a.kcur = k_cur->ptr; a.kc_sb = k_cur->stride_b; a.kc_st = k_cur->stride_t; a.kc_sh = k_cur->stride_h;
    a.vcur = v_cur->ptr; a.vc_sb = v_cur->stride_b; a.vc_st = v_cur->stride_t; a.vc_sh = v_cur->stride_h;
    a.out = out->ptr; a.o_sb = out->stride_b; a.o_st = out->stride_t; a.o_sh = out->stride_h;
    a.u = u; a.vb = v_bias;
    a.r = r; a.r_row = static_cast<int64_t>(H) * ld_r; a.r_head = ld_r;
    a.B = B; a.L = L; a.H = H; a.D = D; a.M = M; a.lo = M - valid; a.wp = M > 0 ? mem->wp : 0; a.C = clamp_len;
    a.scale = scale;
    p.dout = d_out->ptr; p.g_sb = d_out->stride_b; p.g_st = d_out->stride_t; p.g_sh = d_out->stride_h;
    p.dq = dq; p.dk = dk_cur; p.dv = dv_cur; p.du = du; p.dvb = dv_bias; p.dr = dr; p.n_rows = n_rows;
    return p;
}

}  // namespace

int txl_rel_attn_bwd_path(int B, int L, int H, int D, const txl_view* q, const txl_mem* mem, const txl_view* k_cur,
                          const txl_view* v_cur, const void* r, int64_t ld_r, const txl_view* out,
                          const txl_view* d_out, const float* dq, const float* dk_cur, const float* dv_cur,
                          const float* dr, txl_dtype dtype)
{
    const txl_status st = check_attn(B, L, H, D, q, mem, k_cur, v_cur, r, ld_r, out, dtype);
    if (st != TXL_OK) return -static_cast<int>(st);
    if (!view_ok(d_out) || !dq || !dk_cur || !dv_cur || !dr) return -static_cast<int>(TXL_ERR_INVALID_ARG);
    static const float bias[1] = {0.f};
    BwdParams p = bwd_params(B, L, H, D, 0, q, mem, k_cur, v_cur, bias, bias, r, ld_r, 1, 1.f, out, d_out,
                             const_cast<float*>(dq), const_cast<float*>(dk_cur), const_cast<float*>(dv_cur), nullptr,
                             nullptr, const_cast<float*>(dr));
    if (!bwd_tc_eligible(p, dtype)) return 3;
    if (!attn_tc_eligible(B, L, H, D, q, mem, k_cur, v_cur, r, ld_r, dtype)) return 2;
    p.lse_given = 1;
    return bwd_umma_eligible(p, dtype) ? 1 : 2;
}

txl_status txl_rel_attn_bwd(int B, int L, int H, int D, int clamp_len, const txl_view* q, const txl_mem* mem,
                            const txl_view* k_cur, const txl_view* v_cur, const float* u, const float* v_bias,
                            const void* r, int64_t ld_r, int n_rows, float scale, const txl_view* out,
                            const txl_view* d_out, float* dq, float* dk_cur, float* dv_cur, float* du,
                            float* dv_bias, float* dr, txl_dtype dtype, void* workspace, size_t workspace_bytes,
                            void* stream)
{
    return txl_rel_attn_bwd_lse(B, L, H, D, clamp_len, q, mem, k_cur, v_cur, u, v_bias, r, ld_r, n_rows, scale, out,
                                d_out, nullptr, dq, dk_cur, dv_cur, du, dv_bias, dr, dtype, workspace, workspace_bytes,
                                stream);
}

txl_status txl_rel_attn_bwd_lse(int B, int L, int H, int D, int clamp_len, const txl_view* q, const txl_mem* mem,
                                const txl_view* k_cur, const txl_view* v_cur, const float* u, const float* v_bias,
                                const void* r, int64_t ld_r, int n_rows, float scale, const txl_view* out,
                                const txl_view* d_out, const float* lse, float* dq, float* dk_cur, float* dv_cur,
                                float* du, float* dv_bias, float* dr, txl_dtype dtype, void* workspace,
                                size_t workspace_bytes, void* stream)
{
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return TXL_ERR_ALIGNMENT;
    txl_status st = check_attn(B, L, H, D, q, mem, k_cur, v_cur, r, ld_r, out, dtype);
    if (st != TXL_OK) return st;
    if (clamp_len < 0 || !u || !v_bias || !view_ok(d_out)) return TXL_ERR_INVALID_ARG;
    if (!dq || !dk_cur || !dv_cur || !du || !dv_bias || !dr) return TXL_ERR_INVALID_ARG;
    const int M = (mem && mem->M > 0) ? mem->M : 0;
    const int need_rows = std::min(M + L, clamp_len + 1);
    if (n_rows < need_rows) return TXL_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (B == 0 || L == 0) {
        // no query: every gradient is zero
        const size_t hd = static_cast<size_t>(H) * D * sizeof(float);
        if (cudaMemsetAsync(du, 0, hd, s) != cudaSuccess || cudaMemsetAsync(dv_bias, 0, hd, s) != cudaSuccess ||
            cudaMemsetAsync(dr, 0, hd * n_rows, s) != cudaSuccess)
            return TXL_ERR_CUDA;
        return TXL_OK;
    }
    const size_t need = txl_rel_attn_bwd_workspace_size(B, L, H, D);
    if (!workspace || workspace_bytes < need) return TXL_ERR_WORKSPACE;
    if (!a16(workspace)) return TXL_ERR_ALIGNMENT;
    if (scale <= 0.f) scale = 1.0f / std::sqrt(static_cast<float>(D));
    BwdParams p = bwd_params(B, L, H, D, clamp_len, q, mem, k_cur, v_cur, u, v_bias, r, ld_r, n_rows, scale, out,
                             d_out, dq, dk_cur, dv_cur, du, dv_bias, dr);
    const size_t rows = static_cast<size_t>(B) * L * H;
    float* ws = static_cast<float*>(workspace);
    p.lse = ws;
    p.dd = ws + rows;
    p.pac = ws + 2 * rows;
    p.pbd = ws + 2 * rows + rows * D;
    // On the tensor-core gradient path the fused forward kernel computes every row's log-sum-exp
    // (its statistics alone, nothing else written), in place of the gradient kernel's own first
    // pass over the keys
    if (bwd_tc_eligible(p, dtype) && attn_tc_eligible(B, L, H, D, q, mem, k_cur, v_cur, r, ld_r, dtype)) {
        if (lse) {
            // the forward's own statistics (txl_rel_attn_fwd_lse), read in place
            p.lse = const_cast<float*>(lse);
        } else {
            const txl_status fs = attn_tc_launch(B, L, H, D, clamp_len, q, mem, k_cur, v_cur, u, v_bias, r, ld_r,
                                                 n_rows, scale, out, nullptr, s, 0, p.lse);
            if (fs != TXL_OK) return fs;
        }
        p.lse_given = 1;
    }
    return launch_rel_attn_bwd(p, dtype, s) == cudaSuccess ? TXL_OK : TXL_ERR_CUDA;
}

txl_status txl_rel_pos_bwd(int n_rows, int d_model, int n_head, int d_head, const float* dr, float* dW_R,
                           int64_t ld_dw, void* stream)
{
    if (n_rows < 0 || d_model < 2 || (d_model & 1) || n_head <= 0 || d_head <= 0) return TXL_ERR_INVALID_ARG;
    if (!dW_R || (n_rows > 0 && !dr) || ld_dw < static_cast<int64_t>(n_head) * d_head) return TXL_ERR_INVALID_ARG;
    PosBwdParams p{dr, dW_R, ld_dw, n_rows, d_model, n_head, d_head};
    return launch_pos_bwd(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? TXL_OK : TXL_ERR_CUDA;
}

namespace {

// Argument checks of txl_rel_attn_table_fwd / txl_rel_attn_table_path.
txl_status check_table(int B, int L, int H, int D, int max_len, const txl_view* q, const txl_view* k,
                       const txl_view* v, const void* r_table, int64_t ld_r, const txl_view* out, txl_dtype dtype)
{
    if (B < 0 || L < 0 || H <= 0 || D <= 0 || max_len < 1) return TXL_ERR_INVALID_ARG;
    if (D > 128) return TXL_ERR_UNSUPPORTED;
    if (dtype != TXL_F32 && dtype != TXL_BF16) return TXL_ERR_INVALID_ARG;
    if (!view_ok(q) || !view_ok(k) || !view_ok(v) || !view_ok(out) || !r_table || ld_r < D)
        return TXL_ERR_INVALID_ARG;
    if (static_cast<int64_t>(max_len) * 2 - 1 > INT32_MAX) return TXL_ERR_INVALID_ARG;
    return TXL_OK;
}

TableParams table_params(int B, int L, int H, int D, int max_len, const txl_view* q, const txl_view* k,
                         const txl_view* v, const float* u, const float* v_bias, const void* r_table, int64_t ld_r,
                         const uint8_t* key_mask, float scale, const txl_view* out)
{
    TableParams p;
    std::memset(&p, 0, sizeof(p));
    p.q = q->ptr; p.q_sb = q->stride_b; p.q_st = q->stride_t; p.q_sh = q->stride_h;
    p.k = k->ptr; p.k_sb = k->stride_b; p.k_st = k->stride_t; p.k_sh = k->stride_h;
    p.v = v->ptr; p.v_sb = v->stride_b; p.v_st = v->stride_t; p.v_sh = v->stride_h;
    p.out = out->ptr; p.o_sb = out->stride_b; p.o_st = out->stride_t; p.o_sh = out->stride_h;
    p.u = u; p.vb = v_bias;
    p.r = r_table; p.r_row = static_cast<int64_t>(H) * ld_r; p.r_head = ld_r;
    p.mask = key_mask;
    p.B = B; p.L = L; p.H = H; p.D = D; p.max_len = max_len;
    p.scale = scale;
    return p;
}

}  // namespace

txl_status txl_rel_attn_table_fwd(int B, int L, int H, int D, int max_len, const txl_view* q, const txl_view* k,
                                  const txl_view* v, const float* u, const float* v_bias, const void* r_table,
                                  int64_t ld_r, const uint8_t* key_mask, float scale, const txl_view* out,
                                  txl_dtype dtype, void* stream)
{
    const txl_status st = check_table(B, L, H, D, max_len, q, k, v, r_table, ld_r, out, dtype);
    if (st != TXL_OK) return st;
    if (!u || !v_bias) return TXL_ERR_INVALID_ARG;
    if (B == 0 || L == 0) return TXL_OK;
    if (scale <= 0.f) scale = 1.0f / std::sqrt(static_cast<float>(D));
    if (table_persist_eligible(B, L, H, D, max_len, q, k, v, r_table, ld_r, key_mask, dtype))
        return table_tc_launch(B, L, H, D, max_len, q, k, v, u, v_bias, r_table, ld_r, key_mask, scale, out,
                               static_cast<cudaStream_t>(stream));
    const TableParams p = table_params(B, L, H, D, max_len, q, k, v, u, v_bias, r_table, ld_r, key_mask, scale, out);
    return launch_table_attn(p, dtype, static_cast<cudaStream_t>(stream)) == cudaSuccess ? TXL_OK : TXL_ERR_CUDA;
}

int txl_rel_attn_table_path(int B, int L, int H, int D, int max_len, const txl_view* q, const txl_view* k,
                            const txl_view* v, const void* r_table, int64_t ld_r, const uint8_t* key_mask,
                            const txl_view* out, txl_dtype dtype)
{
    const txl_status st = check_table(B, L, H, D, max_len, q, k, v, r_table, ld_r, out, dtype);
    if (st != TXL_OK) return -static_cast<int>(st);
    if (table_persist_eligible(B, L, H, D, max_len, q, k, v, r_table, ld_r, key_mask, dtype)) return 1;
    const TableParams p = table_params(B, L, H, D, max_len, q, k, v, nullptr, nullptr, r_table, ld_r, key_mask, 1.f,
                                       out);
    return table_tc_eligible(p, dtype) ? 3 : 2;
}

int txl_rel_attn_decode_path(int B, int L, int H, int D, const txl_view* q, const txl_mem* mem,
                             const txl_view* k_cur, const txl_view* v_cur, const void* r, int64_t ld_r,
                             const txl_view* out, txl_dtype dtype)
{
    const txl_status st = check_attn(B, L, H, D, q, mem, k_cur, v_cur, r, ld_r, out, dtype);
    if (st != TXL_OK) return -static_cast<int>(st);
    if (L > kDecodeMaxL) return -static_cast<int>(TXL_ERR_UNSUPPORTED);
    return decode_takes_fused(B, L, H, D, q, mem, k_cur, v_cur, r, ld_r, dtype) ? 1 : 4;
}

int txl_checked_build(void) { return kCheckedBuild ? 1 : 0; }

txl_status txl_range_errors(int* count)
{
    if (!count) return TXL_ERR_INVALID_ARG;
#ifdef TXL_CHECKED
    if (cudaDeviceSynchronize() != cudaSuccess) return TXL_ERR_CUDA;
    return cudaMemcpyFromSymbol(count, g_range_errors, sizeof(int)) == cudaSuccess ? TXL_OK : TXL_ERR_CUDA;
#else
    *count = 0;
    return TXL_ERR_UNSUPPORTED;
#endif
}

txl_status txl_range_errors_clear(void)
{
#ifdef TXL_CHECKED
    const int zero = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return TXL_ERR_CUDA;
    return cudaMemcpyToSymbol(g_range_errors, &zero, sizeof(int)) == cudaSuccess ? TXL_OK : TXL_ERR_CUDA;
#else
    return TXL_ERR_UNSUPPORTED;
#endif
}

txl_status txl_selftest_range_check(void* stream)
{
    if (!kCheckedBuild) return TXL_ERR_UNSUPPORTED;
    int* chk = range_counter();
    if (!chk) return TXL_ERR_CUDA;
    return launch_selftest_range(chk, static_cast<cudaStream_t>(stream)) == cudaSuccess ? TXL_OK : TXL_ERR_CUDA;
}

txl_status txl_selftest_wait_timeout(int* err_flag, unsigned timeout_us, void* stream)
{
    if (!err_flag || timeout_us == 0 || timeout_us > 10000000u) return TXL_ERR_INVALID_ARG;
    return launch_selftest_wait(err_flag, timeout_us, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? TXL_OK
               : TXL_ERR_CUDA;
}

}  // extern "C"
