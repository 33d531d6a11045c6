// dq_api.cu -- status strings, the CUDA-error record and the per-device error flag.
#include <mutex>

#include "dq_common.cuh"

// Set by kernels that give up a bounded wait (see dq_common.cuh).
static __device__ int g_dq_device_error;

namespace dqhost {

static thread_local int t_last_cuda_error = 0;

int set_cuda_error(cudaError_t e)
{
    t_last_cuda_error = static_cast<int>(e);
    return DQ_ERR_CUDA;
}

int* device_error_flag()
{
    static std::mutex mu;
    static int* ptrs[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_dq_device_error) != cudaSuccess)
            return nullptr;
        ptrs[dev] = static_cast<int*>(p);
    }
    return ptrs[dev];
}

int sm_count()
{
    static std::mutex mu;
    static int counts[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 1;
    std::lock_guard<std::mutex> lock(mu);
    if (!counts[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
            n = 1;
        counts[dev] = n;
    }
    return counts[dev];
}

}  // namespace dqhost

extern "C" {

DQ_API const char* dq_status_string(int s)
{
    switch (s) {
    case DQ_OK: return "ok";
    case DQ_ERR_NULL: return "a required pointer is NULL";
    case DQ_ERR_SHAPE: return "a size is zero, negative or inconsistent";
    case DQ_ERR_ALIGN: return "a pointer or row is not 16-byte aligned";
    case DQ_ERR_UNSUPPORTED: return "no kernel for this shape";
    case DQ_ERR_CUDA: return "a CUDA runtime call failed";
    case DQ_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
    case DQ_ERR_ALLOC: return "workspace allocation failed";
    default: return "unknown status";
    }
}

DQ_API int dq_last_cuda_error(void) { return dqhost::t_last_cuda_error; }

DQ_API int dq_device_error(void* stream)
{
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return dqhost::set_cuda_error(e);
    int* flag = dqhost::device_error_flag();
    if (!flag)
        return dqhost::set_cuda_error(cudaGetLastError());
    int v = 0;
    e = cudaMemcpy(&v, flag, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess)
        return dqhost::set_cuda_error(e);
    if (v) {
        const int zero = 0;
        e = cudaMemcpy(flag, &zero, sizeof(int), cudaMemcpyHostToDevice);
        if (e != cudaSuccess)
            return dqhost::set_cuda_error(e);
    }
    return v;
}

DQ_API int dq_check_device(void* stream)
{
    const int v = dq_device_error(stream);
    if (v < 0)
        return v;
    if (v == 0)
        return DQ_OK;
    // every bit but "bad argument seen on the device" records a wait that ran out
    return (v & ~dq::DEVERR_BAD_ARG) ? DQ_ERR_TIMEOUT : DQ_ERR_SHAPE;
}

}  // extern "C"
