// dq_gemv_host.cu -- plans and launches the streaming GEMV; the GEMV and
// dequantisation entry points of the C ABI.
#include <mutex>

#include "dq_gemv_host.h"

namespace dqhost {

static int row_bytes_of(int fmt, int K)
{
    if (fmt == DQ_FMT_BF16)
        return 2 * K;
    return (K / 256) * (fmt == DQ_FMT_Q4K ? dq::Q4K_BYTES : fmt == DQ_FMT_Q2K ? dq::Q2K_BYTES : dq::Q6K_BYTES);
}

static GemvKernel kernel_for(int fmt, int ul, int rpt, int nmat, int pl)
{
    if (fmt == DQ_FMT_Q4K)
        return gemv_kernel_q4k(ul, rpt, nmat, pl);
    if (fmt == DQ_FMT_Q6K)
        return gemv_kernel_q6k(ul, rpt, nmat, pl);
    if (fmt == DQ_FMT_Q2K)
        return gemv_kernel_q2k(ul, rpt, nmat, pl);
    return gemv_kernel_bf16(ul, rpt, nmat, pl);
}

static cudaError_t ensure_smem_attr(GemvKernel k, int bytes)
{
    static std::mutex mu;
    static GemvKernel keys[256];
    static int vals[256];
    static int n = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
        if (keys[i] == k) {
            if (vals[i] >= bytes)
                return cudaSuccess;
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
            if (e == cudaSuccess)
                vals[i] = bytes;
            return e;
        }
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && n < 256) {
        keys[n] = k;
        vals[n] = bytes;
        ++n;
    }
    return e;
}

int plan_gemv(int fmt, int rows, int K, int nmat, int planes, bool resid, GemvPlan* plan)
{
    if (rows < 1 || K < 1)
        return DQ_ERR_SHAPE;
    const int unit_w = fmt == DQ_FMT_BF16 ? 8 : 32;
    if (fmt == DQ_FMT_BF16 && K % 8)
        return DQ_ERR_SHAPE;
    if (fmt == DQ_FMT_Q4K && K % 256)
        return DQ_ERR_SHAPE;
    if (fmt == DQ_FMT_Q6K && K % 2048)
        return DQ_ERR_ALIGN;  // 210-byte blocks: rows are 16-byte aligned only when K % 2048 == 0
    if (fmt == DQ_FMT_Q2K && K % 1024)
        return DQ_ERR_ALIGN;  // 84-byte blocks: rows are 16-byte aligned only when K % 1024 == 0
    if (fmt != DQ_FMT_BF16 && K > dq::GEMV_MAX_K)
        return DQ_ERR_UNSUPPORTED;
    const int U = K / unit_w;
    const int rb = row_bytes_of(fmt, K);
    const int pl = (planes == 2 && fmt == DQ_FMT_Q4K) ? 2 : 1;
    static const int ul_q[] = {1, 2, 3, 4};
    static const int ul_q2[] = {1, 2};
    static const int ul_b[] = {1, 2, 4, 8, 12};
    const int* uls = fmt == DQ_FMT_BF16 ? ul_b : (pl == 2 ? ul_q2 : ul_q);
    const int nul = fmt == DQ_FMT_BF16 ? 5 : (pl == 2 ? 2 : 4);
    // Row groups of P threads (P >= 64 so that the groups' named barriers fit).
    // Least masked lanes first, then more groups (smaller P).
    static const int Ps[] = {64, 128, 256, 512};
    // bf16 and Q4_K with at least 64 rows a block: groups of 128 or more (measured:
    // bf16 12288 x 4096 16.7 against 18.6 us with 64-thread groups, Q4_K 12288 x 4096
    // 9.03 against 9.16; bf16 4096 x 4096, 27 rows a block, keeps 64: 7.85 against
    // 7.97; Q6_K keeps 64: the vocabulary shape 79.5 against 86.1 with 128)
    const int sms = sm_count();
    const bool tall_fmt = fmt == DQ_FMT_BF16 || fmt == DQ_FMT_Q4K;
    const int pmin = (tall_fmt && (rows + sms - 1) / sms >= 64) ? 128 : 64;
    int best_P = 0, best_UL = 0, best_waste = 1 << 30;
    for (int pi = 0; pi < 4; ++pi) {
        const int P = Ps[pi];
        if (P < pmin)
            continue;
        const int need = (U + P - 1) / P;
        int UL = 0;
        for (int i = 0; i < nul; ++i)
            if (uls[i] >= need) {
                UL = uls[i];
                break;
            }
        if (!UL)
            continue;
        const int RG = dq::NCONS / P;
        if (static_cast<long long>(RG) * rb * nmat > GEMV_STAGE_MAX)
            continue;
        const int waste = UL * P - U;
        if (waste < best_waste) {
            best_waste = waste;
            best_P = P;
            best_UL = UL;
        }
    }
    if (!best_P)
        return DQ_ERR_UNSUPPORTED;
    GemvPlan p{};
    p.fmt = fmt;
    p.rows = rows;
    p.K = K;
    p.nmat = nmat;
    p.row_bytes = rb;
    p.P = best_P;
    p.RG = dq::NCONS / best_P;
    p.UL = best_UL;
    p.grid = rows < sms ? rows : sms;
    // Stage size: at most GEMV_STAGE_TARGET, and about a quarter of one block's
    // bytes so small matrices still pipeline; rows per thread RPT in {1, 2, 4}.
    const long long per_block = static_cast<long long>((rows + p.grid - 1) / p.grid) * rb * nmat;
    const long long unit_stage = static_cast<long long>(p.RG) * rb * nmat;
#ifndef GEMV_CAP_DIV
#define GEMV_CAP_DIV 4
#endif
    long long cap = per_block / GEMV_CAP_DIV;
    if (cap > GEMV_STAGE_TARGET)
        cap = GEMV_STAGE_TARGET;
    p.RPT = 1;
    for (int r = 4; r >= 1; r >>= 1)
        if (unit_stage * r <= cap) {
            p.RPT = r;
            break;
        }
    p.stage_bytes = p.RG * p.RPT * rb * nmat;
    // as many stages as fit next to the activation buffers (2 .. MAX_STAGES)
    p.resid_rows = resid ? (rows + p.grid - 1) / p.grid : 0;
    const dq::GemvSmem base = dq::gemv_smem_layout(fmt, K, 0, p.stage_bytes, p.RPT, nmat, pl, p.resid_rows);
    const int per_stage = p.stage_bytes + 2 * dq::NCONS_WARPS * p.RPT * nmat * 4;
    int ns = (GEMV_SMEM_MAX - base.total) / per_stage;
    if (ns > GEMV_RING_MAX / p.stage_bytes)
        ns = GEMV_RING_MAX / p.stage_bytes;
    if (ns > dq::MAX_STAGES)
        ns = dq::MAX_STAGES;
    if (ns < 2)
        return DQ_ERR_UNSUPPORTED;
    p.nstage = ns;
    p.smem_bytes = dq::gemv_smem_layout(fmt, K, p.nstage, p.stage_bytes, p.RPT, nmat, pl, p.resid_rows).total;
    p.planes = pl;
    p.kernel = kernel_for(fmt, p.UL, p.RPT, nmat, p.planes);
    if (!p.kernel)
        return DQ_ERR_UNSUPPORTED;
    cudaError_t e = ensure_smem_attr(p.kernel, p.smem_bytes);
    if (e != cudaSuccess)
        return set_cuda_error(e);
    int blocks = 0;  // one block of GEMV_THREADS threads must fit on an SM
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, p.kernel, dq::GEMV_THREADS, p.smem_bytes);
    if (e != cudaSuccess)
        return set_cuda_error(e);
    if (blocks < 1)
        return DQ_ERR_UNSUPPORTED;
    *plan = p;
    return DQ_OK;
}

static unsigned long long* g_trace = nullptr;
static size_t g_trace_next = 0;  // 64-bit words of the buffer used by earlier GEMV launches

void set_gemv_trace(void* buf)
{
    g_trace = static_cast<unsigned long long*>(buf);
    g_trace_next = 0;
}
unsigned long long* gemv_trace() { return g_trace; }

cudaError_t launch_gemv(const GemvPlan& plan, dq::GemvArgs a, cudaStream_t stream, bool pdl)
{
    // each traced launch takes the next slot: 8 words per block, 192 for block 0's stages
    a.trace = g_trace ? g_trace + g_trace_next : nullptr;
    if (g_trace)
        g_trace_next += 8 * static_cast<size_t>(plan.grid) + 192;
    a.rows = plan.rows;
    a.K = plan.K;
    a.row_bytes = plan.row_bytes;
    a.P = plan.P;
    a.RG = plan.RG;
    a.nstage = plan.nstage;
    a.stage_bytes = plan.stage_bytes;
    a.resid_rows = plan.resid_rows;
    if (!a.err)
        a.err = device_error_flag();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(dq::GEMV_THREADS);
    cfg.dynamicSmemBytes = plan.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, plan.kernel, a);
}

}  // namespace dqhost

// ------------------------------------------------------------ dequantisers

namespace dq {

__device__ __forceinline__ uint32_t ldb(const uint8_t* p) { return *p; }

// One thread per 32 weights of Q4_K: w = d * sc_j * q - dmin * m_j in fp32.
__global__ void dequant_q4k_kernel(const uint8_t* __restrict__ blocks, float* __restrict__ out, long long nunits)
{
    const long long u = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (u >= nunits)
        return;
    const uint8_t* b = blocks + (u >> 3) * Q4K_BYTES;
    const int j = static_cast<int>(u & 7);
    const float d = half_bits_to_float(ldb(b) | ldb(b + 1) << 8);
    const float dmin = half_bits_to_float(ldb(b + 2) | ldb(b + 3) << 8);
    int sc = 0, mn = 0;
    for (int k = 0; k < 6; ++k) {
        const int bs = 6 * j + k, bm = 48 + 6 * j + k;
        sc |= ((ldb(b + 4 + (bs >> 3)) >> (bs & 7)) & 1) << k;
        mn |= ((ldb(b + 4 + (bm >> 3)) >> (bm & 7)) & 1) << k;
    }
    const float ds = d * static_cast<float>(sc), dm = dmin * static_cast<float>(mn);
    float* o = out + u * 32;
    for (int i = 0; i < 16; ++i) {
        const uint32_t c = ldb(b + 16 + 16 * j + i);
        o[i] = ds * static_cast<float>(c & 15u) - dm;
        o[16 + i] = ds * static_cast<float>(c >> 4) - dm;
    }
}

// One thread per 32 weights of Q2_K: w = d * sc_j * q - dmin * m_j in fp32.
__global__ void dequant_q2k_kernel(const uint8_t* __restrict__ blocks, float* __restrict__ out, long long nunits)
{
    const long long u = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (u >= nunits)
        return;
    const uint8_t* b = blocks + (u >> 3) * Q2K_BYTES;
    const int h = static_cast<int>(u & 7);
    const float d = half_bits_to_float(ldb(b) | ldb(b + 1) << 8);
    const float dmin = half_bits_to_float(ldb(b + 2) | ldb(b + 3) << 8);
    float* o = out + u * 32;
    for (int s = 0; s < 2; ++s) {
        const int j = 2 * h + s;
        const uint32_t sm = ldb(b + 4 + j);
        const float ds = d * static_cast<float>(sm & 15u), dm = dmin * static_cast<float>(sm >> 4);
        for (int i = 0; i < 16; ++i) {
            const uint32_t c = (ldb(b + 20 + 4 * j + (i & 3)) >> (2 * (i >> 2))) & 3u;
            o[16 * s + i] = ds * static_cast<float>(c) - dm;
        }
    }
}

// One thread per 32 weights of Q6_K: w = d * sc[n/16] * (q - 32) in fp32.
__global__ void dequant_q6k_kernel(const uint8_t* __restrict__ blocks, float* __restrict__ out, long long nunits)
{
    const long long u = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (u >= nunits)
        return;
    const uint8_t* b = blocks + (u >> 3) * Q6K_BYTES;
    const int g = static_cast<int>(u & 7);
    const float d = half_bits_to_float(ldb(b + 208) | ldb(b + 209) << 8);
    const float sa = d * static_cast<float>(static_cast<int8_t>(b[192 + 2 * g]));
    const float sb = d * static_cast<float>(static_cast<int8_t>(b[192 + 2 * g + 1]));
    float* o = out + u * 32;
    for (int h = 0; h < 2; ++h)
        for (int t = 0; t < 4; ++t)
            for (int e = 0; e < 4; ++e) {
                const int r = 16 * h + 4 * t + e;
                const uint32_t lo = (ldb(b + 16 * g + 4 * t + e) >> (4 * h)) & 15u;
                const uint32_t hi = (ldb(b + 128 + 8 * g + 4 * h + e) >> (2 * t)) & 3u;
                const int q = static_cast<int>(lo | hi << 4);
                o[r] = (h ? sb : sa) * static_cast<float>(q - 32);
            }
}

}  // namespace dq

// ------------------------------------------------------------------- C ABI

static int gemv_entry(int fmt, const void* W, const void* x, float* y, int rows, int K, bool static_w,
                      void* stream)
{
    if (!W || !x || !y)
        return DQ_ERR_NULL;
    if (!dqhost::aligned16(W) || !dqhost::aligned16(x))
        return DQ_ERR_ALIGN;
    dqhost::GemvPlan plan;
    int st = dqhost::plan_gemv(fmt, rows, K, 1, 1, false, &plan);
    if (st != DQ_OK)
        return st;
    dq::GemvArgs a{};
    a.W = static_cast<const uint8_t*>(W);
    a.pro = fmt == DQ_FMT_BF16 ? dq::PRO_BF16 : dq::PRO_F32;
    a.epi = dq::EPI_STORE;
    if (fmt == DQ_FMT_BF16)
        a.xb = static_cast<const uint16_t*>(x);
    else
        a.x = static_cast<const float*>(x);
    a.y = y;
    // a dependent launch: its set-up and its first weight requests overlap the
    // previous kernel's tail.  Weights that kernel may write are only prefetched into
    // L2 before the wait and copied after it; static weights are copied at once.
    a.w_late = static_w ? 0 : 1;
    cudaError_t e = dqhost::launch_gemv(plan, a, static_cast<cudaStream_t>(stream), true);
    return e == cudaSuccess ? DQ_OK : dqhost::set_cuda_error(e);
}

static int gemv_k_limit(int fmt) { return fmt == DQ_FMT_BF16 ? 24576 : 16384; }

extern "C" {

DQ_API int dq_debug_trace(void* buffer)
{
    dqhost::set_gemv_trace(buffer);
    return DQ_OK;
}

DQ_API int dq_gemv_bf16(const void* W_bf16, const void* x_bf16, float* y, int rows, int K, void* stream)
{
    if (K > 24576)
        return DQ_ERR_UNSUPPORTED;
    return gemv_entry(DQ_FMT_BF16, W_bf16, x_bf16, y, rows, K, false, stream);
}

DQ_API int dq_gemv_q4k(const void* W_blocks, const float* x, float* y, int rows, int K, void* stream)
{
    if (K > 16384)
        return DQ_ERR_UNSUPPORTED;
    return gemv_entry(DQ_FMT_Q4K, W_blocks, x, y, rows, K, false, stream);
}

DQ_API int dq_gemv_q6k(const void* W_blocks, const float* x, float* y, int rows, int K, void* stream)
{
    if (K > 16384)
        return DQ_ERR_UNSUPPORTED;
    return gemv_entry(DQ_FMT_Q6K, W_blocks, x, y, rows, K, false, stream);
}

DQ_API int dq_gemv_q2k(const void* W_blocks, const float* x, float* y, int rows, int K, void* stream)
{
    if (K > 16384)
        return DQ_ERR_UNSUPPORTED;
    return gemv_entry(DQ_FMT_Q2K, W_blocks, x, y, rows, K, false, stream);
}

DQ_API int dq_gemv_ex(int fmt, const void* W, const void* x, float* y, int rows, int K, int flags, void* stream)
{
    if (fmt != DQ_FMT_BF16 && fmt != DQ_FMT_Q4K && fmt != DQ_FMT_Q6K && fmt != DQ_FMT_Q2K)
        return DQ_ERR_SHAPE;
    if (flags & ~DQ_GEMV_STATIC_WEIGHTS)
        return DQ_ERR_SHAPE;
    if (K > gemv_k_limit(fmt))
        return DQ_ERR_UNSUPPORTED;
    return gemv_entry(fmt, W, x, y, rows, K, (flags & DQ_GEMV_STATIC_WEIGHTS) != 0, stream);
}

static int dequant_entry(int fmt, const void* blocks, float* out, long long nblocks, void* stream)
{
    if (!blocks || !out)
        return DQ_ERR_NULL;
    if (nblocks < 1)
        return DQ_ERR_SHAPE;
    const long long nunits = nblocks * 8;
    const int threads = 256;
    const long long grid = (nunits + threads - 1) / threads;
    if (grid > 0x7fffffffLL)
        return DQ_ERR_SHAPE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (fmt == DQ_FMT_Q6K)
        dq::dequant_q6k_kernel<<<static_cast<unsigned>(grid), threads, 0, s>>>(static_cast<const uint8_t*>(blocks), out,
                                                                              nunits);
    else if (fmt == DQ_FMT_Q2K)
        dq::dequant_q2k_kernel<<<static_cast<unsigned>(grid), threads, 0, s>>>(static_cast<const uint8_t*>(blocks), out,
                                                                              nunits);
    else
        dq::dequant_q4k_kernel<<<static_cast<unsigned>(grid), threads, 0, s>>>(static_cast<const uint8_t*>(blocks), out,
                                                                              nunits);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DQ_OK : dqhost::set_cuda_error(e);
}

DQ_API int dq_dequant_q4k(const void* blocks, float* out, long long nblocks, void* stream)
{
    return dequant_entry(DQ_FMT_Q4K, blocks, out, nblocks, stream);
}

DQ_API int dq_dequant_q6k(const void* blocks, float* out, long long nblocks, void* stream)
{
    return dequant_entry(DQ_FMT_Q6K, blocks, out, nblocks, stream);
}

DQ_API int dq_dequant_q2k(const void* blocks, float* out, long long nblocks, void* stream)
{
    return dequant_entry(DQ_FMT_Q2K, blocks, out, nblocks, stream);
}

}  // extern "C"
