// dq_decode.cu -- one decode token over a pre-norm decoder stack.
//
// Per layer five kernels, chained with programmatic dependent launch:
//   1. RMSNorm(x) fused into the Q|K|V GEMV (Q4_K); the epilogue writes q and
//      appends k, v to the fp16 cache at pos;
//   2. grouped-query attention over keys 0..pos, merged by its last block;
//   3. O projection (Q4_K) + residual add into x;
//   4. RMSNorm(x) fused into the gate and up GEMVs (Q4_K, streamed together),
//      epilogue SiLU(gate) * up;
//   5. down projection (Q4_K or Q6_K) + residual add into x;
// then RMSNorm(x) fused into the vocabulary GEMV (Q6_K).  The 5 L + 1 launches
// are captured once in a CUDA graph.  A small kernel before the graph copies
// x_in and records pos and the logits pointer in device memory, because the
// graph's arguments are fixed.
//
// Where the shape allows, the same phases run instead as one persistent
// cooperative kernel (dq_token.cu), launched directly with x_in, pos and the
// logits pointer as arguments.
//
// Layout follows the Qwen3-8B census of "The roofline holds on a second GPU",
// section "The Math"; the norm placement follows "one-serial-kernel", section
// "One thread" (twice per layer and once at the end).
#include <atomic>
#include <new>
#include <vector>

#include "dq_gemv_host.h"
#include "dq_token.cuh"

namespace dq {

__global__ void step_begin_kernel(const float* __restrict__ x_in, float* __restrict__ x, int n, StepArgs* step,
                                  int pos, float* logits)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n)
        x[i] = x_in[i];
    if (i == 0) {
        step->pos = pos;
        step->logits = logits;
    }
}

}  // namespace dq

struct dq_model {
    int n_layers, hidden, ffn, n_q, n_kv, hd, vocab, max_ctx;
    float eps;
    std::vector<const float*> attn_norm, ffn_norm;
    std::vector<const uint8_t*> wqkv, wo, wgate, wup, wdown;
    std::vector<int> down_fmt;
    std::vector<const float*> q_norm, k_norm;  // Qwen3 attention inputs (empty: plain attention)
    const float* out_norm;
    const uint8_t* wvocab;
    __half* kv;
    // workspace (one allocation)
    void* ws;
    float* x;
    float* q;
    float* attn;
    float* act;
    dq::StepArgs* step;
    void* attn_ws;
    float* k_new;       // Qwen3 attention inputs: the token's projected keys, else null
    float2* rope;       // (cos, sin) [max_ctx][hd / 2] when k_new is set
    float* tk_k;        // fused kernel: tagged copies of the token's keys and values [n_kv hd]
    float* tk_v;
    unsigned* tk_stamps; // fused kernel: attention chunk stamps [n_kv][ATT_CHUNKS]
    float* io_x;         // dq_decode_step_host: the input [hidden] and logits [vocab] on the device
    float* io_logits;
    // fused token kernel
    bool fused;
    dqhost::TokenPlan tplan;
    dq::TokenLayer* layers_dev;
    unsigned* bar;                 // fused kernel launch state (blocks out, token count, fault; the kernel keeps it)
    unsigned long long wait_ns;    // bound on the fused kernel's waits
    int skew_next;                 // diagnostics: the next fused token waits for writes never made
    // plans
    dqhost::GemvPlan p_qkv, p_o, p_gateup, p_down_q4, p_down_q6, p_vocab;
    bool have_down_q4, have_down_q6;
    // graph
    int use_graph;
    bool pdl;
    cudaStream_t cap_stream;
    cudaGraph_t graph;
    cudaGraphExec_t exec;
};

enum { K_QKV = 0, K_ATTN = 1, K_O = 2, K_GATEUP = 3, K_DOWN = 4, K_VOCAB = 5 };

// Workspace allocations of dq_model_create still to fail on purpose (diagnostics).
static std::atomic<int> g_fail_allocs{0};

static cudaError_t launch_kernel(dq_model* m, int l, int kind, cudaStream_t s, bool pdl)
{
    const int qdim = m->n_q * m->hd, kvdim = m->n_kv * m->hd;
    const size_t plane = static_cast<size_t>(m->n_kv) * m->max_ctx * m->hd;
    __half* kc = m->kv + static_cast<size_t>(l) * 2 * plane;
    __half* vc = kc + plane;
    int* err = dqhost::device_error_flag();
    dq::GemvArgs a{};
    a.err = err;
    switch (kind) {
    case K_QKV:  // norm + QKV + cache append
        a.W = m->wqkv[l];
        a.pro = dq::PRO_RMS;
        a.x = m->x;
        a.gamma = m->attn_norm[l];
        a.eps = m->eps;
        a.epi = dq::EPI_QKV;
        a.y = m->q;
        a.step = m->step;
        a.kv_k = kc;
        a.kv_v = vc;
        a.k_new = m->k_new;
        a.qdim = qdim;
        a.kvdim = kvdim;
        a.hd = m->hd;
        a.max_ctx = m->max_ctx;
        return dqhost::launch_gemv(m->p_qkv, a, s, pdl);
    case K_ATTN: {
        dq::AttnArgs t{};
        t.q = m->q;
        t.kc = kc;
        t.vc = vc;
        t.out = m->attn;
        dqhost::attention_bind_workspace(t, m->attn_ws);
        t.n_q = m->n_q;
        t.n_kv = m->n_kv;
        t.max_ctx = m->max_ctx;
        t.step = m->step;
        t.err = err;
        if (m->k_new) {
            t.k_new = m->k_new;
            t.q_norm = m->q_norm[l];
            t.k_norm = m->k_norm[l];
            t.rope = m->rope;
            t.eps = m->eps;
        }
        return dqhost::launch_attention(t, s, pdl);
    }
    case K_O:  // O projection + residual
        a.W = m->wo[l];
        a.pro = dq::PRO_F32;
        a.x = m->attn;
        a.epi = dq::EPI_RESID;
        a.y = m->x;
        return dqhost::launch_gemv(m->p_o, a, s, pdl);
    case K_GATEUP:  // norm + gate/up + SwiGLU
        a.W = m->wgate[l];
        a.W2 = m->wup[l];
        a.pro = dq::PRO_RMS;
        a.x = m->x;
        a.gamma = m->ffn_norm[l];
        a.eps = m->eps;
        a.epi = dq::EPI_SWIGLU;
        a.y = m->act;
        return dqhost::launch_gemv(m->p_gateup, a, s, pdl);
    case K_DOWN:  // down + residual
        a.W = m->wdown[l];
        a.pro = dq::PRO_F32;
        a.x = m->act;
        a.epi = dq::EPI_RESID;
        a.y = m->x;
        return dqhost::launch_gemv(m->down_fmt[l] == DQ_FMT_Q6K ? m->p_down_q6 : m->p_down_q4, a, s, pdl);
    default:  // final norm + vocabulary
        a.W = m->wvocab;
        a.pro = dq::PRO_RMS;
        a.x = m->x;
        a.gamma = m->out_norm;
        a.eps = m->eps;
        a.epi = dq::EPI_STORE;
        a.y_from_step = 1;
        a.step = m->step;
        return dqhost::launch_gemv(m->p_vocab, a, s, pdl);
    }
}

static cudaError_t enqueue_token(dq_model* m, cudaStream_t s)
{
    cudaError_t e;
    for (int l = 0; l < m->n_layers; ++l)
        for (int kind = K_QKV; kind <= K_DOWN; ++kind)
            if ((e = launch_kernel(m, l, kind, s, m->pdl)) != cudaSuccess)
                return e;
    return launch_kernel(m, 0, K_VOCAB, s, m->pdl);
}

static void free_model(dq_model* m)
{
    if (!m)
        return;
    if (m->exec)
        cudaGraphExecDestroy(m->exec);
    if (m->graph)
        cudaGraphDestroy(m->graph);
    if (m->cap_stream)
        cudaStreamDestroy(m->cap_stream);
    if (m->ws)
        cudaFree(m->ws);
    delete m;
}

extern "C" {

DQ_API int dq_model_create(const dq_model_desc* d, dq_model** out)
{
    if (!out)
        return DQ_ERR_NULL;
    *out = nullptr;
    if (!d || !d->attn_norm || !d->wqkv || !d->wo || !d->ffn_norm || !d->wgate || !d->wup || !d->wdown ||
        !d->down_fmt || !d->out_norm || !d->wvocab || !d->kv_cache)
        return DQ_ERR_NULL;
    if (d->n_layers < 1 || d->hidden < 1 || d->ffn < 1 || d->n_q_heads < 1 || d->n_kv_heads < 1 ||
        d->head_dim < 1 || d->vocab < 1 || d->max_ctx < 1 || d->n_q_heads % d->n_kv_heads ||
        !dqhost::valid_eps(d->eps))
        return DQ_ERR_SHAPE;
    if (d->head_dim != dq::ATT_HD || d->n_q_heads / d->n_kv_heads > 8 || d->n_kv_heads > dq::ATT_COUNTER_BYTES / 4)
        return DQ_ERR_UNSUPPORTED;
    const int qdim = d->n_q_heads * d->head_dim, kvdim = d->n_kv_heads * d->head_dim;
    if (d->hidden % 256 || d->ffn % 256 || qdim % 256)
        return DQ_ERR_SHAPE;
    for (int l = 0; l < d->n_layers; ++l) {
        if (!d->attn_norm[l] || !d->wqkv[l] || !d->wo[l] || !d->ffn_norm[l] || !d->wgate[l] || !d->wup[l] ||
            !d->wdown[l])
            return DQ_ERR_NULL;
        if (d->down_fmt[l] != DQ_FMT_Q4K && d->down_fmt[l] != DQ_FMT_Q6K)
            return DQ_ERR_SHAPE;
        if (!dqhost::aligned16(d->attn_norm[l]) || !dqhost::aligned16(d->wqkv[l]) || !dqhost::aligned16(d->wo[l]) ||
            !dqhost::aligned16(d->ffn_norm[l]) || !dqhost::aligned16(d->wgate[l]) || !dqhost::aligned16(d->wup[l]) ||
            !dqhost::aligned16(d->wdown[l]))
            return DQ_ERR_ALIGN;
    }
    if (!dqhost::aligned16(d->out_norm) || !dqhost::aligned16(d->wvocab) || !dqhost::aligned16(d->kv_cache))
        return DQ_ERR_ALIGN;
    const bool qwen3 = d->q_norm != nullptr;
    if (qwen3) {
        if (!d->k_norm)
            return DQ_ERR_NULL;
        if (!(d->rope_theta > 1.0))
            return DQ_ERR_SHAPE;
        for (int l = 0; l < d->n_layers; ++l) {
            if (!d->q_norm[l] || !d->k_norm[l])
                return DQ_ERR_NULL;
            if (!dqhost::aligned16(d->q_norm[l]) || !dqhost::aligned16(d->k_norm[l]))
                return DQ_ERR_ALIGN;
        }
    }

    dq_model* m = new (std::nothrow) dq_model();
    if (!m)
        return DQ_ERR_ALLOC;
    m->n_layers = d->n_layers;
    m->hidden = d->hidden;
    m->ffn = d->ffn;
    m->n_q = d->n_q_heads;
    m->n_kv = d->n_kv_heads;
    m->hd = d->head_dim;
    m->vocab = d->vocab;
    m->max_ctx = d->max_ctx;
    m->eps = d->eps;
    m->use_graph = d->use_graph;
    m->pdl = (d->flags & DQ_MODEL_NO_PDL) == 0;
    for (int l = 0; l < d->n_layers; ++l) {
        m->attn_norm.push_back(d->attn_norm[l]);
        m->ffn_norm.push_back(d->ffn_norm[l]);
        m->wqkv.push_back(static_cast<const uint8_t*>(d->wqkv[l]));
        m->wo.push_back(static_cast<const uint8_t*>(d->wo[l]));
        m->wgate.push_back(static_cast<const uint8_t*>(d->wgate[l]));
        m->wup.push_back(static_cast<const uint8_t*>(d->wup[l]));
        m->wdown.push_back(static_cast<const uint8_t*>(d->wdown[l]));
        m->down_fmt.push_back(d->down_fmt[l]);
        if (qwen3) {
            m->q_norm.push_back(d->q_norm[l]);
            m->k_norm.push_back(d->k_norm[l]);
        }
        if (d->down_fmt[l] == DQ_FMT_Q6K)
            m->have_down_q6 = true;
        else
            m->have_down_q4 = true;
    }
    m->out_norm = d->out_norm;
    m->wvocab = static_cast<const uint8_t*>(d->wvocab);
    m->kv = static_cast<__half*>(d->kv_cache);

    int st;
    // The q|k|v projection feeds the attention, which amplifies input errors: it
    // takes the two-plane (about 30-bit) activation.  So does O here (in the
    // fused token kernel O takes one plane: there it measured faster).
    if ((st = dqhost::plan_gemv(DQ_FMT_Q4K, qdim + 2 * kvdim, d->hidden, 1, 2, false, &m->p_qkv)) != DQ_OK ||
        (st = dqhost::plan_gemv(DQ_FMT_Q4K, d->hidden, qdim, 1, 2, true, &m->p_o)) != DQ_OK ||
        (st = dqhost::plan_gemv(DQ_FMT_Q4K, d->ffn, d->hidden, 2, 1, false, &m->p_gateup)) != DQ_OK ||
        (m->have_down_q4 &&
         (st = dqhost::plan_gemv(DQ_FMT_Q4K, d->hidden, d->ffn, 1, 1, true, &m->p_down_q4)) != DQ_OK) ||
        (m->have_down_q6 &&
         (st = dqhost::plan_gemv(DQ_FMT_Q6K, d->hidden, d->ffn, 1, 1, true, &m->p_down_q6)) != DQ_OK) ||
        (st = dqhost::plan_gemv(DQ_FMT_Q6K, d->vocab, d->hidden, 1, 1, false, &m->p_vocab)) != DQ_OK) {
        free_model(m);
        return st;
    }

    // the fused token kernel on request, where the shape allows (its absence is not an error)
    if (d->flags & DQ_MODEL_FUSED)
        m->fused = dqhost::plan_token(d->n_layers, d->hidden, d->ffn, d->n_q_heads, d->n_kv_heads, d->head_dim,
                                      m->have_down_q6, &m->tplan) == DQ_OK;

    // workspace: x | q | attn | act | step | attention scratch | layer table | barrier
    // [| new keys | rotary table], each 256-byte aligned
    auto up = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
    const size_t bx = up(sizeof(float) * d->hidden), bq = up(sizeof(float) * qdim), ba = bq,
                 bf = up(sizeof(float) * d->ffn), bs = up(sizeof(dq::StepArgs)),
                 bw = up(dqhost::attention_workspace_bytes(d->n_q_heads, d->n_kv_heads)),
                 bl = up(sizeof(dq::TokenLayer) * d->n_layers), bb = 256,
                 bk = (qwen3 || m->fused) ? up(sizeof(float) * kvdim) : 0, bv = m->fused ? up(sizeof(float) * kvdim) : 0,
                 br = qwen3 ? up(sizeof(float2) * static_cast<size_t>(d->max_ctx) * (d->head_dim / 2)) : 0,
                 bt = m->fused ? up(sizeof(unsigned) * d->n_kv_heads * dq::ATT_CHUNKS) : 0,
                 bix = up(sizeof(float) * d->hidden), bil = up(sizeof(float) * d->vocab);
    const size_t total = bx + bq + ba + bf + bs + bw + bl + bb + bk + bv + br + bt + bix + bil;
    // diagnostics: an injected allocation failure (dq_debug_fail_next_allocs)
    int inject = g_fail_allocs.load();
    while (inject > 0 && !g_fail_allocs.compare_exchange_weak(inject, inject - 1)) {
    }
    cudaError_t e = inject > 0 ? cudaErrorMemoryAllocation : cudaMalloc(&m->ws, total);
    if (e != cudaSuccess) {
        cudaGetLastError();
        free_model(m);
        return DQ_ERR_ALLOC;
    }
    char* base = static_cast<char*>(m->ws);
    m->x = reinterpret_cast<float*>(base);
    m->q = reinterpret_cast<float*>(base + bx);
    m->attn = reinterpret_cast<float*>(base + bx + bq);
    m->act = reinterpret_cast<float*>(base + bx + bq + ba);
    m->step = reinterpret_cast<dq::StepArgs*>(base + bx + bq + ba + bf);
    m->attn_ws = base + bx + bq + ba + bf + bs;
    m->layers_dev = reinterpret_cast<dq::TokenLayer*>(base + bx + bq + ba + bf + bs + bw);
    m->bar = reinterpret_cast<unsigned*>(base + bx + bq + ba + bf + bs + bw + bl);
    m->wait_ns = dq::WAIT_LIMIT_NS;
    char* kv_copies = base + bx + bq + ba + bf + bs + bw + bl + bb;
    if (qwen3) {
        m->k_new = reinterpret_cast<float*>(kv_copies);
        m->rope = reinterpret_cast<float2*>(kv_copies + bk + bv);
    }
    if (m->fused) {  // the fused kernel's tagged copies of the token's keys and values, attention stamps
        m->tk_k = reinterpret_cast<float*>(kv_copies);
        m->tk_v = reinterpret_cast<float*>(kv_copies + bk);
        m->tk_stamps = reinterpret_cast<unsigned*>(kv_copies + bk + bv + br);
    }
    // device copies of dq_decode_step_host's input and logits
    m->io_x = reinterpret_cast<float*>(kv_copies + bk + bv + br + bt);
    m->io_logits = reinterpret_cast<float*>(kv_copies + bk + bv + br + bt + bix);
    if ((e = cudaMemset(m->ws, 0, total)) != cudaSuccess ||
        (qwen3 && (e = dqhost::launch_rope_table(m->rope, d->max_ctx, d->head_dim, d->rope_theta, 0)) != cudaSuccess)) {
        free_model(m);
        return dqhost::set_cuda_error(e);
    }
    if (m->fused) {
        std::vector<dq::TokenLayer> tl(d->n_layers);
        for (int l = 0; l < d->n_layers; ++l) {
            tl[l].attn_norm = m->attn_norm[l];
            tl[l].ffn_norm = m->ffn_norm[l];
            tl[l].wqkv = m->wqkv[l];
            tl[l].wo = m->wo[l];
            tl[l].wgate = m->wgate[l];
            tl[l].wup = m->wup[l];
            tl[l].wdown = m->wdown[l];
            tl[l].q_norm = qwen3 ? m->q_norm[l] : nullptr;
            tl[l].k_norm = qwen3 ? m->k_norm[l] : nullptr;
            tl[l].down_fmt = m->down_fmt[l];
            tl[l].pad = 0;
        }
        if ((e = cudaMemcpy(m->layers_dev, tl.data(), sizeof(dq::TokenLayer) * d->n_layers,
                            cudaMemcpyHostToDevice)) != cudaSuccess) {
            free_model(m);
            return dqhost::set_cuda_error(e);
        }
    }
    if (m->use_graph && !m->fused) {
        if ((e = cudaStreamCreateWithFlags(&m->cap_stream, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamBeginCapture(m->cap_stream, cudaStreamCaptureModeRelaxed)) != cudaSuccess) {
            free_model(m);
            return dqhost::set_cuda_error(e);
        }
        cudaError_t e1 = enqueue_token(m, m->cap_stream);
        cudaError_t e2 = cudaStreamEndCapture(m->cap_stream, &m->graph);
        if (e1 != cudaSuccess || e2 != cudaSuccess) {
            free_model(m);
            return dqhost::set_cuda_error(e1 != cudaSuccess ? e1 : e2);
        }
        if ((e = cudaGraphInstantiate(&m->exec, m->graph, 0)) != cudaSuccess) {
            free_model(m);
            return dqhost::set_cuda_error(e);
        }
    }
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) {
        free_model(m);
        return dqhost::set_cuda_error(e);
    }
    *out = m;
    return DQ_OK;
}

DQ_API int dq_decode_step(dq_model* m, const float* x_in, int pos, float* logits, void* stream)
{
    if (!m || !x_in || !logits)
        return DQ_ERR_NULL;
    if (pos < 0 || pos >= m->max_ctx)
        return DQ_ERR_SHAPE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (m->fused) {
        dq::TokenArgs a{};
        a.layers = m->layers_dev;
        a.n_layers = m->n_layers;
        a.hidden = m->hidden;
        a.ffn = m->ffn;
        a.n_q = m->n_q;
        a.n_kv = m->n_kv;
        a.hd = m->hd;
        a.vocab = m->vocab;
        a.max_ctx = m->max_ctx;
        a.eps = m->eps;
        a.out_norm = m->out_norm;
        a.wvocab = m->wvocab;
        a.kv = m->kv;
        a.x = m->x;
        a.q = m->q;
        a.attn = m->attn;
        a.act = m->act;
        dq::AttnArgs t{};
        dqhost::attention_bind_workspace(t, m->attn_ws);
        a.part = t.part;
        a.counters = t.counters;
        a.stamps = m->tk_stamps;
        a.k_new = m->tk_k;
        a.v_new = m->tk_v;
        a.qwen = m->k_new != nullptr;
        a.rope = m->rope;
        a.step = m->step;
        a.bar = m->bar;
        a.wait_ns = m->wait_ns;
        a.skew = m->skew_next;
        a.x_in = x_in;
        a.logits = logits;
        a.pos = pos;
        a.fold = pos + 1 <= dq::TK_FOLD_KEYS ? 1 : 0;
        a.err = dqhost::device_error_flag();
        a.trace = dqhost::gemv_trace();
        cudaError_t e = dqhost::launch_token(m->tplan, a, s);
        if (e != cudaSuccess)
            return dqhost::set_cuda_error(e);
        m->skew_next = 0;
        return DQ_OK;
    }
    const int threads = 256;
    dq::step_begin_kernel<<<(m->hidden + threads - 1) / threads, threads, 0, s>>>(x_in, m->x, m->hidden, m->step,
                                                                                  pos, logits);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return dqhost::set_cuda_error(e);
    e = m->use_graph ? cudaGraphLaunch(m->exec, s) : enqueue_token(m, s);
    return e == cudaSuccess ? DQ_OK : dqhost::set_cuda_error(e);
}

DQ_API int dq_decode_step_host(dq_model* m, const float* x_host, int pos, float* logits_host, void* stream)
{
    if (!m || !x_host || !logits_host)
        return DQ_ERR_NULL;
    if (pos < 0 || pos >= m->max_ctx)
        return DQ_ERR_SHAPE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(m->io_x, x_host, sizeof(float) * m->hidden, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess)
        return dqhost::set_cuda_error(e);
    const int st = dq_decode_step(m, m->io_x, pos, m->io_logits, s);
    if (st != DQ_OK)
        return st;
    if ((e = cudaMemcpyAsync(logits_host, m->io_logits, sizeof(float) * m->vocab, cudaMemcpyDeviceToHost, s)) !=
            cudaSuccess ||
        (e = cudaStreamSynchronize(s)) != cudaSuccess)
        return dqhost::set_cuda_error(e);
    return DQ_OK;
}

DQ_API int dq_model_launches_per_step(const dq_model* m)
{
    return m ? (m->fused ? 1 : 2 + 5 * m->n_layers) : 0;
}

DQ_API int dq_model_fused(const dq_model* m)
{
    return m ? (m->fused ? 1 : 0) : DQ_ERR_NULL;
}

DQ_API int dq_model_enqueue_kernel(dq_model* m, int layer, int kind, void* stream)
{
    if (!m)
        return DQ_ERR_NULL;
    if (kind < K_QKV || kind > K_VOCAB || layer < 0 || layer >= m->n_layers)
        return DQ_ERR_SHAPE;
    cudaError_t e = launch_kernel(m, layer, kind, static_cast<cudaStream_t>(stream), m->pdl);
    return e == cudaSuccess ? DQ_OK : dqhost::set_cuda_error(e);
}

DQ_API int dq_model_buffer(const dq_model* m, int which, void** ptr)
{
    if (!m || !ptr)
        return DQ_ERR_NULL;
    switch (which) {
    case 0: *ptr = m->x; return DQ_OK;
    case 1: *ptr = m->q; return DQ_OK;
    case 2: *ptr = m->attn; return DQ_OK;
    case 3: *ptr = m->act; return DQ_OK;
    default: return DQ_ERR_SHAPE;
    }
}

DQ_API int dq_model_debug_waits(dq_model* m, unsigned long long wait_limit_ns, int skew)
{
    if (!m)
        return DQ_ERR_NULL;
    if (wait_limit_ns < 1000ull || wait_limit_ns > 60000000000ull || skew < 0 || skew > 1000)
        return DQ_ERR_SHAPE;
    if (!m->fused)
        return DQ_ERR_UNSUPPORTED;
    m->wait_ns = wait_limit_ns;
    m->skew_next = skew;
    return DQ_OK;
}

DQ_API int dq_debug_fail_next_allocs(int n)
{
    if (n < 0)
        return DQ_ERR_SHAPE;
    g_fail_allocs.store(n);
    return DQ_OK;
}

DQ_API int dq_model_destroy(dq_model* m)
{
    if (!m)
        return DQ_OK;
    cudaDeviceSynchronize();
    free_model(m);
    return DQ_OK;
}

}  // extern "C"
