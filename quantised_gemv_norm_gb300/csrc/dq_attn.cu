// dq_attn.cu -- grouped-query decode attention over an fp16 KV cache.
//
// One token: query head h attends over keys 0 .. n_keys-1 of KV head
// h / (n_q / n_kv) with a max-subtracted softmax ("The roofline holds on a
// second GPU", "Said before the run": every new token reads the conversation's
// keys and values, 75.5 MB at 512 tokens for the Qwen3-8B shape).
//
// Grid: ATT_CHUNKS blocks per KV head; block (c, g) takes one contiguous chunk
// of keys and one warp per query head of the group.  Keys and values are staged
// 32 at a time in shared memory (rows padded by 16 bytes so that lane j reading
// key j's row is conflict-free); lane j scores key j, the warp keeps a running
// max / sum / output (4 dims per lane).  Each block writes (m, l, o) partials;
// the last block of a KV head to finish (a device-scope counter, no waiting)
// merges them and resets the counter for the next call.
#include <mutex>

#include "dq_attn.cuh"

namespace dq {

__global__ void __launch_bounds__(256) attn_decode_kernel(const __grid_constant__ AttnArgs args)
{
    __shared__ __align__(16) AttnSmem sm;
    pdl_trigger();
    const AttnArgs a = args;
    attn_block(a, blockIdx.x, blockIdx.y, blockDim.x >> 5, sm, true);
}

// (cos, sin) of p / theta^(2i / hd) for p < max_ctx, i < hd / 2, in double
// precision, rounded once to fp32.
__global__ void rope_table_kernel(float2* __restrict__ tab, int max_ctx, int hd, double theta)
{
    const int half = hd / 2;
    const size_t n = static_cast<size_t>(max_ctx) * half;
    for (size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < n;
         idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int p = static_cast<int>(idx / half), i = static_cast<int>(idx % half);
        const double ang = static_cast<double>(p) * pow(theta, -2.0 * i / hd);
        double sn, cs;
        sincos(ang, &sn, &cs);
        tab[idx] = make_float2(static_cast<float>(cs), static_cast<float>(sn));
    }
}

}  // namespace dq

namespace dqhost {

cudaError_t launch_rope_table(float2* tab, int max_ctx, int hd, double theta, cudaStream_t stream)
{
    const size_t n = static_cast<size_t>(max_ctx) * (hd / 2);
    const int threads = 256;
    const int blocks = static_cast<int>(n / threads + 1 < 4096 ? n / threads + 1 : 4096);
    dq::rope_table_kernel<<<blocks, threads, 0, stream>>>(tab, max_ctx, hd, theta);
    return cudaGetLastError();
}

size_t attention_workspace_bytes(int n_q, int n_kv)
{
    (void)n_kv;
    return dq::ATT_COUNTER_BYTES + static_cast<size_t>(n_q) * dq::ATT_CHUNKS * dq::ATT_PART * sizeof(float);
}

void attention_bind_workspace(dq::AttnArgs& a, void* ws)
{
    a.counters = static_cast<int*>(ws);
    a.part = reinterpret_cast<float*>(static_cast<char*>(ws) + dq::ATT_COUNTER_BYTES);
}

cudaError_t launch_attention(const dq::AttnArgs& a, cudaStream_t stream, bool pdl)
{
    dq::AttnArgs b = a;
    if (!b.err)
        b.err = device_error_flag();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(dq::ATT_CHUNKS, a.n_kv);
    cfg.blockDim = dim3(32 * (a.n_q / a.n_kv));
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, dq::attn_decode_kernel, b);
}

}  // namespace dqhost

extern "C" {

DQ_API size_t dq_attention_workspace_bytes(int n_q, int n_kv)
{
    if (n_q < 1 || n_kv < 1)
        return 0;
    return dqhost::attention_workspace_bytes(n_q, n_kv);
}

DQ_API int dq_attention_decode(const float* q, const void* k_plane, const void* v_plane, float* out, int n_q,
                               int n_kv, int head_dim, int max_ctx, int n_keys, void* workspace,
                               size_t workspace_bytes, void* stream)
{
    if (!q || !k_plane || !v_plane || !out || !workspace)
        return DQ_ERR_NULL;
    if (n_q < 1 || n_kv < 1 || max_ctx < 1 || n_keys < 1 || n_keys > max_ctx || n_q % n_kv)
        return DQ_ERR_SHAPE;
    if (head_dim != dq::ATT_HD || n_q / n_kv > 8 || n_kv > dq::ATT_COUNTER_BYTES / 4)
        return DQ_ERR_UNSUPPORTED;
    if (workspace_bytes < dqhost::attention_workspace_bytes(n_q, n_kv))
        return DQ_ERR_SHAPE;
    if (!dqhost::aligned16(q) || !dqhost::aligned16(k_plane) || !dqhost::aligned16(v_plane) ||
        !dqhost::aligned16(out) || !dqhost::aligned16(workspace))
        return DQ_ERR_ALIGN;
    dq::AttnArgs a{};
    a.q = q;
    a.kc = static_cast<const __half*>(k_plane);
    a.vc = static_cast<const __half*>(v_plane);
    a.out = out;
    dqhost::attention_bind_workspace(a, workspace);
    a.n_q = n_q;
    a.n_kv = n_kv;
    a.max_ctx = max_ctx;
    a.n_keys = n_keys;
    a.step = nullptr;
    cudaError_t e = dqhost::launch_attention(a, static_cast<cudaStream_t>(stream), false);
    return e == cudaSuccess ? DQ_OK : dqhost::set_cuda_error(e);
}

DQ_API int dq_rope_table(float* table, int max_ctx, int head_dim, double theta, void* stream)
{
    if (!table)
        return DQ_ERR_NULL;
    if (max_ctx < 1 || head_dim < 2 || head_dim % 2 || !(theta > 1.0))
        return DQ_ERR_SHAPE;
    if (!dqhost::aligned16(table))
        return DQ_ERR_ALIGN;
    cudaError_t e = dqhost::launch_rope_table(reinterpret_cast<float2*>(table), max_ctx, head_dim, theta,
                                              static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DQ_OK : dqhost::set_cuda_error(e);
}

DQ_API int dq_attention_decode_rope(const float* q, const float* k_new, void* k_plane, const void* v_plane, float* out,
                                    const float* q_norm, const float* k_norm, const float* rope_table, float eps,
                                    int n_q, int n_kv, int head_dim, int max_ctx, int n_keys, void* workspace,
                                    size_t workspace_bytes, void* stream)
{
    if (!q || !k_new || !k_plane || !v_plane || !out || !q_norm || !k_norm || !rope_table || !workspace)
        return DQ_ERR_NULL;
    if (n_q < 1 || n_kv < 1 || max_ctx < 1 || n_keys < 1 || n_keys > max_ctx || n_q % n_kv ||
        !dqhost::valid_eps(eps))
        return DQ_ERR_SHAPE;
    if (head_dim != dq::ATT_HD || n_q / n_kv > 8 || n_kv > dq::ATT_COUNTER_BYTES / 4)
        return DQ_ERR_UNSUPPORTED;
    if (workspace_bytes < dqhost::attention_workspace_bytes(n_q, n_kv))
        return DQ_ERR_SHAPE;
    if (!dqhost::aligned16(q) || !dqhost::aligned16(k_new) || !dqhost::aligned16(k_plane) ||
        !dqhost::aligned16(v_plane) || !dqhost::aligned16(out) || !dqhost::aligned16(q_norm) ||
        !dqhost::aligned16(k_norm) || !dqhost::aligned16(rope_table) || !dqhost::aligned16(workspace))
        return DQ_ERR_ALIGN;
    dq::AttnArgs a{};
    a.q = q;
    a.kc = static_cast<const __half*>(k_plane);
    a.vc = static_cast<const __half*>(v_plane);
    a.out = out;
    dqhost::attention_bind_workspace(a, workspace);
    a.n_q = n_q;
    a.n_kv = n_kv;
    a.max_ctx = max_ctx;
    a.n_keys = n_keys;
    a.step = nullptr;
    a.k_new = k_new;
    a.q_norm = q_norm;
    a.k_norm = k_norm;
    a.rope = reinterpret_cast<const float2*>(rope_table);
    a.eps = eps;
    cudaError_t e = dqhost::launch_attention(a, static_cast<cudaStream_t>(stream), false);
    return e == cudaSuccess ? DQ_OK : dqhost::set_cuda_error(e);
}

}  // extern "C"

// ------------------------------------------------- attention without allocation
//
// Some callers cannot call cudaMalloc: inference-server plugins whose host
// process owns all device memory through its own pool, and embedded or
// real-time deployments that fix their device memory at start-up.  For them
// the attention scratch (the merge counters and the chunk partials) lives in
// one file-scope device array, sized for up to DQ_STATIC_ATT_MAX_Q query heads
// and DQ_STATIC_ATT_MAX_KV KV heads (include/dq.h).  Every device that loads
// this library holds the array until the process exits.

namespace {

constexpr int STATIC_ATT_MAX_Q = DQ_STATIC_ATT_MAX_Q;
constexpr int STATIC_ATT_MAX_KV = DQ_STATIC_ATT_MAX_KV;
// one merge counter (an int) per KV head in the counter area
static_assert(STATIC_ATT_MAX_KV <= dq::ATT_COUNTER_BYTES / 4, "a merge counter per KV head");
constexpr size_t STATIC_ATT_BYTES =
    dq::ATT_COUNTER_BYTES + static_cast<size_t>(STATIC_ATT_MAX_Q) * dq::ATT_CHUNKS * dq::ATT_PART * sizeof(float);
static_assert(STATIC_ATT_BYTES == 1081600, "the size the header states");

static __device__ __align__(256) unsigned char g_static_att_scratch[STATIC_ATT_BYTES];

constexpr int STATIC_ATT_MAX_DEVICES = 64;

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and kept for the process.  In host code
// the array's name stands for a host-side shadow, never for the device memory,
// so only this address may be handed to a kernel.  Returns DQ_OK, or
// DQ_ERR_UNSUPPORTED for a device index beyond the table, or DQ_ERR_CUDA.
int static_att_scratch(void** out)
{
    static std::mutex mu;
    static void* ptrs[STATIC_ATT_MAX_DEVICES] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return dqhost::set_cuda_error(e);
    if (dev < 0 || dev >= STATIC_ATT_MAX_DEVICES)
        return DQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_static_att_scratch)) != cudaSuccess)
            return dqhost::set_cuda_error(e);
        ptrs[dev] = p;
    }
    *out = ptrs[dev];
    return DQ_OK;
}

}  // namespace

extern "C" {

DQ_API int dq_attention_decode_static(const float* q, const void* k_plane, const void* v_plane, float* out, int n_q,
                                      int n_kv, int head_dim, int max_ctx, int n_keys, void* stream)
{
    if (!q || !k_plane || !v_plane || !out)
        return DQ_ERR_NULL;
    if (n_q < 1 || n_kv < 1 || max_ctx < 1 || n_keys < 1 || n_keys > max_ctx || n_q % n_kv)
        return DQ_ERR_SHAPE;
    if (n_q > STATIC_ATT_MAX_Q || n_kv > STATIC_ATT_MAX_KV)
        return DQ_ERR_SHAPE;  // beyond the fixed scratch array
    if (head_dim != dq::ATT_HD || n_q / n_kv > 8)
        return DQ_ERR_UNSUPPORTED;
    if (!dqhost::aligned16(q) || !dqhost::aligned16(k_plane) || !dqhost::aligned16(v_plane) || !dqhost::aligned16(out))
        return DQ_ERR_ALIGN;
    void* scratch = nullptr;
    const int st = static_att_scratch(&scratch);
    if (st != DQ_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the merge counters must start at zero whatever an earlier call left behind
    cudaError_t e = cudaMemsetAsync(scratch, 0, dq::ATT_COUNTER_BYTES, s);
    if (e != cudaSuccess)
        return dqhost::set_cuda_error(e);
    dq::AttnArgs a{};
    a.q = q;
    a.kc = static_cast<const __half*>(k_plane);
    a.vc = static_cast<const __half*>(v_plane);
    a.out = out;
    dqhost::attention_bind_workspace(a, scratch);
    a.n_q = n_q;
    a.n_kv = n_kv;
    a.max_ctx = max_ctx;
    a.n_keys = n_keys;
    a.step = nullptr;
    e = dqhost::launch_attention(a, s, false);
    return e == cudaSuccess ? DQ_OK : dqhost::set_cuda_error(e);
}

}  // extern "C"
