// dq_norm.cu -- RMSNorm and LayerNorm, one thread block per row.
//
// "one-serial-kernel" (vocodex.ai), section "One thread": a row of 2048 values
// walked by one GPU thread took 231 us; the fix shares the row among a block of
// threads, each summing its part, the parts combined across the block, and the
// layer norm in two passes (the mean, then the variance of x - mean).  The
// block size is a parameter so the one-thread form and the sweep over thread
// counts can be run and checked as well.
#include "dq_common.cuh"

namespace dq {

// Sum over the block; blockDim.x is a power of two in [1, 1024].
__device__ float block_sum(float v, float* scratch)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nt = blockDim.x;
    if (nt < 32) {
        const unsigned mask = (nt == 32) ? 0xffffffffu : ((1u << nt) - 1u);
        for (int o = nt >> 1; o > 0; o >>= 1)
            v += __shfl_xor_sync(mask, v, o);
        return __shfl_sync(mask, v, 0);
    }
    v = warp_sum(v);
    __syncthreads();  // scratch may still be read from a previous call
    if (lane == 0)
        scratch[warp] = v;
    __syncthreads();
    float t = 0.f;
    const int nw = nt >> 5;
    for (int w = 0; w < nw; ++w)
        t += scratch[w];
    return t;
}

template <bool LN>
__global__ void __launch_bounds__(1024) norm_kernel(const float* __restrict__ x, const float* __restrict__ gamma,
                                                     const float* __restrict__ beta, float* y, int n, float eps)
{
    __shared__ float scratch[32];
    pdl_trigger();
    pdl_wait();
    const size_t row = blockIdx.x;
    const float* xr = x + row * n;
    float* yr = y + row * n;
    const int tid = threadIdx.x, nt = blockDim.x;
    const bool vec = ((n & 3) == 0) && (((reinterpret_cast<uintptr_t>(xr) | reinterpret_cast<uintptr_t>(yr)) & 15) == 0);
    const int n4 = vec ? n >> 2 : 0;
    const float4* x4 = reinterpret_cast<const float4*>(xr);

    // pass 1: sum (LayerNorm) or sum of squares (RMSNorm)
    float s = 0.f;
    for (int i = tid; i < n4; i += nt) {
        const float4 v = x4[i];
        s += LN ? (v.x + v.y) + (v.z + v.w) : (v.x * v.x + v.y * v.y) + (v.z * v.z + v.w * v.w);
    }
    for (int i = 4 * n4 + tid; i < n; i += nt) {
        const float v = xr[i];
        s += LN ? v : v * v;
    }
    s = block_sum(s, scratch);

    float mean = 0.f, rstd;
    if (LN) {
        mean = s / static_cast<float>(n);
        // pass 2: variance of (x - mean)
        float q = 0.f;
        for (int i = tid; i < n4; i += nt) {
            const float4 v = x4[i];
            const float a = v.x - mean, b = v.y - mean, c = v.z - mean, d = v.w - mean;
            q += (a * a + b * b) + (c * c + d * d);
        }
        for (int i = 4 * n4 + tid; i < n; i += nt) {
            const float a = xr[i] - mean;
            q += a * a;
        }
        q = block_sum(q, scratch);
        rstd = 1.0f / sqrtf(q / static_cast<float>(n) + eps);
    } else {
        rstd = 1.0f / sqrtf(s / static_cast<float>(n) + eps);
    }

    // last pass: scale (and shift); each element is read and written by one thread
    for (int i = tid; i < n4; i += nt) {
        const float4 v = x4[i];
        const float4 g = reinterpret_cast<const float4*>(gamma)[i];
        float4 o;
        if (LN) {
            const float4 b = reinterpret_cast<const float4*>(beta)[i];
            o.x = (v.x - mean) * rstd * g.x + b.x;
            o.y = (v.y - mean) * rstd * g.y + b.y;
            o.z = (v.z - mean) * rstd * g.z + b.z;
            o.w = (v.w - mean) * rstd * g.w + b.w;
        } else {
            o.x = v.x * rstd * g.x;
            o.y = v.y * rstd * g.y;
            o.z = v.z * rstd * g.z;
            o.w = v.w * rstd * g.w;
        }
        reinterpret_cast<float4*>(yr)[i] = o;
    }
    for (int i = 4 * n4 + tid; i < n; i += nt) {
        const float v = xr[i];
        yr[i] = LN ? (v - mean) * rstd * gamma[i] + beta[i] : v * rstd * gamma[i];
    }
}

}  // namespace dq

static int norm_entry(bool ln, const float* x, const float* gamma, const float* beta, float* y, int rows, int n,
                      float eps, int threads, void* stream)
{
    if (!x || !gamma || !y || (ln && !beta))
        return DQ_ERR_NULL;
    if (rows < 1 || n < 1 || !dqhost::valid_eps(eps))
        return DQ_ERR_SHAPE;
    if (threads < 1 || threads > 1024 || (threads & (threads - 1)))
        return DQ_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(gamma) & 15 || (ln && reinterpret_cast<uintptr_t>(beta) & 15)) {
        // gamma/beta are read as float4 when x and y allow it: require alignment
        return DQ_ERR_ALIGN;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (ln)
        dq::norm_kernel<true><<<rows, threads, 0, s>>>(x, gamma, beta, y, n, eps);
    else
        dq::norm_kernel<false><<<rows, threads, 0, s>>>(x, gamma, nullptr, y, n, eps);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DQ_OK : dqhost::set_cuda_error(e);
}

extern "C" {

DQ_API int dq_rmsnorm(const float* x, const float* gamma, float* y, int rows, int n, float eps, void* stream)
{
    return norm_entry(false, x, gamma, nullptr, y, rows, n, eps, 256, stream);
}

DQ_API int dq_layernorm(const float* x, const float* gamma, const float* beta, float* y, int rows, int n, float eps,
                        void* stream)
{
    return norm_entry(true, x, gamma, beta, y, rows, n, eps, 256, stream);
}

DQ_API int dq_rmsnorm_threads(const float* x, const float* gamma, float* y, int rows, int n, float eps, int threads,
                              void* stream)
{
    return norm_entry(false, x, gamma, nullptr, y, rows, n, eps, threads, stream);
}

DQ_API int dq_layernorm_threads(const float* x, const float* gamma, const float* beta, float* y, int rows, int n,
                                float eps, int threads, void* stream)
{
    return norm_entry(true, x, gamma, beta, y, rows, n, eps, threads, stream);
}

}  // extern "C"
