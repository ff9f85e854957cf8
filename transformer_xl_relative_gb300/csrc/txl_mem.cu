// txl_mem.cu -- FIFO K/V memory update ("Transformer-XL架构解析" §1.1: the newest segment's
// cached states evict the oldest; "Transformer-XL 和相对位置编码" §2.3.1: the cache holds the
// previous segment for the next one's keys and values).
//
// Pure data movement, HBM-bound: every 16-byte chunk of k_new/v_new that survives the push is
// read once and written once to its ring slot (wp + t) mod M.  Consecutive threads handle
// consecutive chunks of one (b, t, h) row, so loads and stores are coalesced 16-byte accesses.
#include "txl_internal.h"
#include "txl_ptx.cuh"

namespace txl {

namespace {

constexpr int kPushThreads = 256;

__global__ void __launch_bounds__(kPushThreads) mem_push_vec16(MemPushParams p)
{
    const int cpr = (p.D * p.elem_bytes) >> 4;             // 16-byte chunks per head row
    const int64_t per_tensor = static_cast<int64_t>(p.B) * p.n_t * p.H * cpr;
    const int64_t total = 2 * per_tensor;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int which = idx >= per_tensor;               // 0: keys, 1: values
        int64_t rem = idx - which * per_tensor;
        const int c = static_cast<int>(rem % cpr); rem /= cpr;
        const int h = static_cast<int>(rem % p.H); rem /= p.H;
        const int t = static_cast<int>(rem % p.n_t) + p.t0;
        const int b = static_cast<int>(rem / p.n_t);
        const int slot = static_cast<int>((static_cast<int64_t>(p.wp) + t) % p.M);
        const char* src = static_cast<const char*>(which ? p.v_new : p.k_new);
        char* dst = static_cast<char*>(which ? p.v : p.k);
        const int64_t so = which ? (b * p.nv_sb + t * p.nv_st + h * p.nv_sh)
                                 : (b * p.n_sb + t * p.n_st + h * p.n_sh);
        const int64_t d_off = b * p.m_sb + slot * p.m_st + h * p.m_sh;
        const uint4 val = __ldg(reinterpret_cast<const uint4*>(src + so * p.elem_bytes) + c);
        reinterpret_cast<uint4*>(dst + d_off * p.elem_bytes)[c] = val;
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
        const int slot = static_cast<int>((static_cast<int64_t>(p.wp) + t) % p.M);
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
    int64_t blocks = (work + kPushThreads - 1) / kPushThreads;
    const int64_t cap = static_cast<int64_t>(sms) * 8;     // grid-stride beyond 8 CTAs per SM
    if (blocks > cap) blocks = cap;
    if (p.vec16)
        mem_push_vec16<<<static_cast<unsigned>(blocks), kPushThreads, 0, s>>>(p);
    else
        mem_push_scalar<<<static_cast<unsigned>(blocks), kPushThreads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_selftest_wait(int* err_flag, unsigned timeout_us, cudaStream_t s)
{
    selftest_wait_kernel<<<1, 32, 0, s>>>(err_flag, static_cast<uint64_t>(timeout_us) * 1000ull);
    return cudaGetLastError();
}

}  // namespace txl
