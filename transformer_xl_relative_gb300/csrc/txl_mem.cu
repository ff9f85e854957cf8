// txl_mem.cu -- FIFO K/V memory update ("Transformer-XL架构解析" §1.1: the newest segment's
// cached states evict the oldest; "Transformer-XL 和相对位置编码" §2.3.1: the cache holds the
// previous segment for the next one's keys and values).
//
// Pure data movement, HBM-bound: every 16-byte chunk of k_new/v_new that survives the push is
// read once and written once to its ring slot (wp + t) mod M.  Consecutive threads handle
// consecutive chunks of one (b, t) row, so loads and stores are coalesced 16-byte accesses.
#include "txl_internal.h"
#include "txl_ptx.cuh"

namespace txl {

namespace {

constexpr int kPushThreads = 128;
constexpr int kPushRows = 4;            // (b, t) rows per block pass: 4 loads in flight per thread

// Grid (row groups, 2): blockIdx.y selects keys (0) or values (1).  Thread c of a block copies
// 16-byte chunk c (head c / cpr, chunk c mod cpr) of kPushRows consecutive (b, t) rows, issuing
// all loads before the stores.  Index arithmetic is 32-bit (the host guarantees B * n_t and
// M + L fit) and is done once per row, not per byte.
__global__ void __launch_bounds__(kPushThreads) mem_push_vec16(MemPushParams p)
{
    pdl_launch_dependents();
    pdl_wait();
    const int which = blockIdx.y;
    const int eb = p.elem_bytes;
    const int cpr = (p.D * eb) >> 4;                       // 16-byte chunks per head row
    const int per_row = p.H * cpr;
    const char* src = static_cast<const char*>(which ? p.v_new : p.k_new);
    char* dst = static_cast<char*>(which ? p.v : p.k);
    const int64_t ssb = (which ? p.nv_sb : p.n_sb) * eb, sst = (which ? p.nv_st : p.n_st) * eb;
    const int64_t ssh = (which ? p.nv_sh : p.n_sh) * eb;
    const int64_t dsb = p.m_sb * eb, dst_t = p.m_st * eb, dsh = p.m_sh * eb;
    const int rows = p.B * p.n_t;
    for (int c = threadIdx.x; c < per_row; c += kPushThreads) {
        const int h = c / cpr, cc = c - h * cpr;
        const int64_t so = h * ssh + 16 * cc, dso = h * dsh + 16 * cc;
        for (int r0 = blockIdx.x * kPushRows; r0 < rows; r0 += gridDim.x * kPushRows) {
            int b = r0 / p.n_t, t = r0 - b * p.n_t;
            uint4 val[kPushRows];
            int64_t doff[kPushRows];
#pragma unroll
            for (int k = 0; k < kPushRows; ++k) {
                const int tt = t + p.t0;                   // position inside the segment
                if (r0 + k < rows) {
                    int slot = (p.wp + tt) % p.M;
                    if (!in_range(slot, 0, p.M, p.chk)) slot = 0;
                    val[k] = __ldg(reinterpret_cast<const uint4*>(src + b * ssb + tt * sst + so));
                    doff[k] = b * dsb + slot * dst_t + dso;
                }
                if (++t == p.n_t) { t = 0; ++b; }
            }
#pragma unroll
            for (int k = 0; k < kPushRows; ++k)
                if (r0 + k < rows) *reinterpret_cast<uint4*>(dst + doff[k]) = val[k];
        }
    }
}

__global__ void __launch_bounds__(kPushThreads) mem_push_scalar(MemPushParams p)
{
    const int64_t per_tensor = static_cast<int64_t>(p.B) * p.n_t * p.H * p.D;
    const int64_t total = 2 * per_tensor;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int which = idx >= per_tensor;
        int64_t rem = idx - which * per_tensor;
        const int d = static_cast<int>(rem % p.D); rem /= p.D;
        const int h = static_cast<int>(rem % p.H); rem /= p.H;
        const int t = static_cast<int>(rem % p.n_t) + p.t0;
        const int b = static_cast<int>(rem / p.n_t);
        int slot = static_cast<int>((static_cast<int64_t>(p.wp) + t) % p.M);
        if (!in_range(slot, 0, p.M, p.chk)) slot = 0;
        const char* src = static_cast<const char*>(which ? p.v_new : p.k_new);
        char* dst = static_cast<char*>(which ? p.v : p.k);
        const int64_t so = which ? (b * p.nv_sb + t * p.nv_st + h * p.nv_sh)
                                 : (b * p.n_sb + t * p.n_st + h * p.n_sh);
        const int64_t dofs = b * p.m_sb + slot * p.m_st + h * p.m_sh;
        if (p.elem_bytes == 4)
            reinterpret_cast<float*>(dst)[dofs + d] = reinterpret_cast<const float*>(src)[so + d];
        else
            reinterpret_cast<uint16_t*>(dst)[dofs + d] =
                reinterpret_cast<const uint16_t*>(src)[so + d];
    }
}

// One CTA waits on an mbarrier that nothing signals, through the same bounded wait every
// pipeline kernel uses, and must come back with TXL_ERR_TIMEOUT recorded.
__global__ void selftest_wait_kernel(int* err_flag, uint64_t timeout_ns)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    WaitCtl w{&abort_flag, err_flag, timeout_ns};
    if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, w, 0);
    __syncthreads();
}

}  // namespace

cudaError_t launch_mem_push(const MemPushParams& p, cudaStream_t s)
{
    const int64_t work = 2ll * p.B * p.n_t * p.H * (p.vec16 ? (p.D * p.elem_bytes) >> 4 : p.D);
    if (work == 0) return cudaSuccess;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t cap = static_cast<int64_t>(sms) * 16;    // grid-stride beyond 16 CTAs per SM
    if (p.vec16) {
        const int64_t rows = static_cast<int64_t>(p.B) * p.n_t;
        int64_t blocks = (rows + kPushRows - 1) / kPushRows;
        if (blocks > cap / 2) blocks = cap / 2;
        return launch_dependent(mem_push_vec16, dim3(static_cast<unsigned>(blocks), 2), dim3(kPushThreads), 0, s, p);
    } else {
        int64_t blocks = (work + kPushThreads - 1) / kPushThreads;
        if (blocks > cap) blocks = cap;
        mem_push_scalar<<<static_cast<unsigned>(blocks), kPushThreads, 0, s>>>(p);
    }
    return cudaGetLastError();
}

// One index out of its range and one inside it, checked as every kernel of the checked build
// checks its computed indices: the counter gains exactly one.  Nothing is accessed.
__global__ void selftest_range_kernel(int* chk, int x_bad, int x_good)
{
    const bool bad_ok = in_range(x_bad, 0, 4, chk);
    const bool good_ok = in_range(x_good, 0, 4, chk);
    (void)bad_ok;
    (void)good_ok;
}

cudaError_t launch_selftest_range(int* chk, cudaStream_t s)
{
    selftest_range_kernel<<<1, 1, 0, s>>>(chk, 5, 1);
    return cudaGetLastError();
}

cudaError_t launch_selftest_wait(int* err_flag, unsigned timeout_us, cudaStream_t s)
{
    selftest_wait_kernel<<<1, 32, 0, s>>>(err_flag, static_cast<uint64_t>(timeout_us) * 1000ull);
    return cudaGetLastError();
}

}  // namespace txl
