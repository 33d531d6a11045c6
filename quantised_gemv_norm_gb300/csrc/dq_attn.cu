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

__global__ void __launch_bounds__(256) attn_decode_kernel(const __grid_constant__ AttnArgs a)
{
    __shared__ __align__(16) __half ks[ATT_BATCH][ATT_HD + 8];
    __shared__ __align__(16) __half vs[ATT_BATCH][ATT_HD];
    __shared__ __align__(16) float qs[8][ATT_HD];
    __shared__ int s_last;

    pdl_trigger();
    const int c = blockIdx.x, g = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int group = blockDim.x >> 5;
    const int nthr = blockDim.x;
    // step->pos was written before the token's first kernel: safe before the wait
    const int n_keys = a.step ? a.step->pos + 1 : a.n_keys;
    // chunks of at least ATT_MIN_CHUNK keys: short contexts take one block per KV head
    const int L = max((n_keys + ATT_CHUNKS - 1) / ATT_CHUNKS, ATT_MIN_CHUNK);
    const int j0 = c * L, j1 = min(n_keys, j0 + L);
    const int nact = (n_keys + L - 1) / L;
    pdl_wait();
    if (n_keys < 1 || n_keys > a.max_ctx) {
        if (tid == 0 && c == 0)
            set_error(a.err, DEVERR_BAD_ARG);
        return;
    }
    if (j0 >= n_keys)
        return;

    const int h = g * group + warp;
    {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(a.q + static_cast<size_t>(h) * ATT_HD) + lane);
        *reinterpret_cast<float4*>(&qs[warp][4 * lane]) = v;
    }
    const __half* kbase = a.kc + static_cast<size_t>(g) * a.max_ctx * ATT_HD;
    const __half* vbase = a.vc + static_cast<size_t>(g) * a.max_ctx * ATT_HD;
    const float scale = 0.08838834764831845f;  // 1 / sqrt(128)

    float m = -INFINITY, l = 0.f;
    float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
    for (int jb = j0; jb < j1; jb += ATT_BATCH) {
        const int nb = min(ATT_BATCH, j1 - jb);
        __syncthreads();  // previous batch fully consumed (and qs written on the first)
        for (int idx = tid; idx < nb * (ATT_HD / 8); idx += nthr) {
            const int j = idx >> 4, ch = idx & 15;
            const uint4 kv = __ldcg(reinterpret_cast<const uint4*>(kbase + static_cast<size_t>(jb + j) * ATT_HD) + ch);
            const uint4 vv = __ldcg(reinterpret_cast<const uint4*>(vbase + static_cast<size_t>(jb + j) * ATT_HD) + ch);
            *reinterpret_cast<uint4*>(&ks[j][8 * ch]) = kv;
            *reinterpret_cast<uint4*>(&vs[j][8 * ch]) = vv;
        }
        __syncthreads();
        float s = -INFINITY;
        if (lane < nb) {
            float d0 = 0.f, d1 = 0.f;
#pragma unroll
            for (int ch = 0; ch < ATT_HD / 8; ++ch) {
                const uint4 kr = *reinterpret_cast<const uint4*>(&ks[lane][8 * ch]);
                const float4 qa = *reinterpret_cast<const float4*>(&qs[warp][8 * ch]);
                const float4 qb = *reinterpret_cast<const float4*>(&qs[warp][8 * ch + 4]);
                const float2 k0 = __half22float2(*reinterpret_cast<const __half2*>(&kr.x));
                const float2 k1 = __half22float2(*reinterpret_cast<const __half2*>(&kr.y));
                const float2 k2 = __half22float2(*reinterpret_cast<const __half2*>(&kr.z));
                const float2 k3 = __half22float2(*reinterpret_cast<const __half2*>(&kr.w));
                d0 = fmaf(qa.x, k0.x, d0); d1 = fmaf(qa.y, k0.y, d1);
                d0 = fmaf(qa.z, k1.x, d0); d1 = fmaf(qa.w, k1.y, d1);
                d0 = fmaf(qb.x, k2.x, d0); d1 = fmaf(qb.y, k2.y, d1);
                d0 = fmaf(qb.z, k3.x, d0); d1 = fmaf(qb.w, k3.y, d1);
            }
            s = (d0 + d1) * scale;
        }
        const float mb = warp_max(s);
        const float mnew = fmaxf(m, mb);
        const float p = lane < nb ? expf(s - mnew) : 0.f;
        const float corr = expf(m - mnew);  // 0 on the first batch (m = -inf)
        l = l * corr + warp_sum(p);
        o0 *= corr; o1 *= corr; o2 *= corr; o3 *= corr;
        for (int j = 0; j < nb; ++j) {
            const float pj = __shfl_sync(0xffffffffu, p, j);
            const uint2 vr = *reinterpret_cast<const uint2*>(&vs[j][4 * lane]);
            const float2 va = __half22float2(*reinterpret_cast<const __half2*>(&vr.x));
            const float2 vb = __half22float2(*reinterpret_cast<const __half2*>(&vr.y));
            o0 = fmaf(pj, va.x, o0); o1 = fmaf(pj, va.y, o1);
            o2 = fmaf(pj, vb.x, o2); o3 = fmaf(pj, vb.y, o3);
        }
        m = mnew;
    }

    if (nact == 1) {  // the only block of this KV head: normalise and write directly
        const float inv = 1.0f / l;
        *reinterpret_cast<float4*>(a.out + static_cast<size_t>(h) * ATT_HD + 4 * lane) =
            make_float4(o0 * inv, o1 * inv, o2 * inv, o3 * inv);
        return;
    }
    float* pp = a.part + (static_cast<size_t>(h) * ATT_CHUNKS + c) * ATT_PART;
    if (lane == 0) {
        pp[0] = m;
        pp[1] = l;
    }
    *reinterpret_cast<float4*>(pp + 4 + 4 * lane) = make_float4(o0, o1, o2, o3);
    __threadfence();
    __syncthreads();
    if (tid == 0)
        s_last = (atomicAdd(&a.counters[g], 1) == nact - 1);
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();
    // merge the chunk partials of this warp's head
    const float* hp = a.part + static_cast<size_t>(h) * ATT_CHUNKS * ATT_PART;
    float M = -INFINITY;
    for (int cc = 0; cc < nact; ++cc)
        M = fmaxf(M, __ldcg(hp + cc * ATT_PART));
    float Ls = 0.f, r0 = 0.f, r1 = 0.f, r2 = 0.f, r3 = 0.f;
    for (int cc = 0; cc < nact; ++cc) {
        const float w = expf(__ldcg(hp + cc * ATT_PART) - M);
        Ls = fmaf(__ldcg(hp + cc * ATT_PART + 1), w, Ls);
        const float4 ov = __ldcg(reinterpret_cast<const float4*>(hp + cc * ATT_PART + 4) + lane);
        r0 = fmaf(ov.x, w, r0); r1 = fmaf(ov.y, w, r1);
        r2 = fmaf(ov.z, w, r2); r3 = fmaf(ov.w, w, r3);
    }
    const float inv = 1.0f / Ls;
    *reinterpret_cast<float4*>(a.out + static_cast<size_t>(h) * ATT_HD + 4 * lane) =
        make_float4(r0 * inv, r1 * inv, r2 * inv, r3 * inv);
    __syncthreads();
    if (tid == 0)
        a.counters[g] = 0;
}

}  // namespace dq

namespace dqhost {

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

}  // extern "C"

// ------------------------------------------------- attention without allocation
//
// Some callers cannot call cudaMalloc: code that runs while a stream is being
// captured into a CUDA graph under a capture mode that forbids allocation,
// inference-server plugins whose host owns all device memory through its own
// pool, and embedded or real-time deployments that fix their device memory at
// start-up.  For them the attention scratch (the merge counters and the chunk
// partials) lives in one file-scope device array, sized for up to
// DQ_STATIC_ATT_MAX_Q query heads and DQ_STATIC_ATT_MAX_KV KV heads.  Every
// device that loads this library holds the array until the process exits.

namespace {

constexpr int STATIC_ATT_MAX_Q = 64;
constexpr int STATIC_ATT_MAX_KV = 64;
constexpr size_t STATIC_ATT_BYTES =
    dq::ATT_COUNTER_BYTES + static_cast<size_t>(STATIC_ATT_MAX_Q) * dq::ATT_CHUNKS * dq::ATT_PART * sizeof(float);

static __device__ __align__(256) unsigned char g_static_att_scratch[STATIC_ATT_BYTES];

// Device address of the scratch array on the current device, looked up once
// per device (with that device current); null if the lookup fails.
void* static_att_scratch()
{
    static std::mutex mu;
    static void* ptrs[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_att_scratch) != cudaSuccess)
            return nullptr;
        ptrs[dev] = p;
    }
    return ptrs[dev];
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
    void* scratch = static_att_scratch();
    if (!scratch)
        return dqhost::set_cuda_error(cudaGetLastError());
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
