// dq_token.cuh -- arguments and host interface of the persistent decode-token kernel.
#pragma once

#include "dq_attn.cuh"

namespace dq {

constexpr int TK_THREADS = 512;    // 16 warps, 128 registers a thread
constexpr int TK_WARPS = TK_THREADS / 32;
constexpr int TK_NSTAGE = 4;       // weight ring slots per block
constexpr int TK_SLOT = 40960;     // bytes per slot (largest tile: 4 Q6_K rows of K = 12288)
// Contexts of at most this many keys skip the attention phase and its barrier:
// every block computes all query heads at the start of the O phase.
constexpr int TK_FOLD_KEYS = 4;
constexpr int TK_RED_STRIDE = 4;   // floats per warp in one partial-sum slot

// Phase kinds.  Per layer: QKV, ATTN, O, GATEUP, DOWN (Q4_K or Q6_K); then VOCAB.
enum { PH_QKV = 0, PH_ATTN, PH_O, PH_GATEUP, PH_DOWN_Q4, PH_DOWN_Q6, PH_VOCAB, PH_KINDS };

// Consumer layout by kind: row groups of tk_p threads (each thread holds tk_ul
// 32-element units of the activation, so K <= 32 tk_p tk_ul), tk_rpt rows per
// thread and matrix; a tile holds TK_THREADS / tk_p * tk_rpt rows of each matrix.
#ifndef TK_GU_P
#define TK_GU_P 64
#define TK_GU_UL 2
#define TK_GU_RPT 1
#endif
#ifndef TK_QKV_P
#define TK_QKV_P 64
#define TK_QKV_UL 2
#define TK_QKV_RPT 2
#endif
#ifndef TK_O_P
#define TK_O_P 128
#define TK_O_UL 1
#define TK_O_RPT 4
#endif
#ifndef TK_VOC_P
#define TK_VOC_P 128
#define TK_VOC_UL 1
#define TK_VOC_RPT 3
#endif
__host__ __device__ constexpr int tk_p(int kind)
{
    return kind == PH_GATEUP ? TK_GU_P
           : kind == PH_QKV  ? TK_QKV_P
           : kind == PH_O    ? TK_O_P
           : kind == PH_VOCAB ? TK_VOC_P
                              : 128;
}
// activation units a thread holds (K <= 32 tk_p tk_ul)
__host__ __device__ constexpr int tk_ul(int kind)
{
    return kind == PH_GATEUP ? TK_GU_UL
           : kind == PH_QKV ? TK_QKV_UL
           : kind == PH_O ? TK_O_UL
           : kind == PH_VOCAB ? TK_VOC_UL
           : kind == PH_DOWN_Q4 || kind == PH_DOWN_Q6 ? 3
                                                      : 1;
}
__host__ __device__ constexpr int tk_rg(int kind) { return TK_THREADS / tk_p(kind); }
__host__ __device__ constexpr int tk_rpt(int kind)
{
    return kind == PH_GATEUP ? TK_GU_RPT
           : kind == PH_QKV ? TK_QKV_RPT
           : kind == PH_O ? TK_O_RPT
           : kind == PH_DOWN_Q4 || kind == PH_DOWN_Q6 ? 1
           : kind == PH_VOCAB ? TK_VOC_RPT
                              : 4;
}
__host__ __device__ constexpr int tk_rows_per_tile(int kind) { return tk_rg(kind) * tk_rpt(kind); }

struct TokenLayer {
    const float* attn_norm;
    const float* ffn_norm;
    const uint8_t* wqkv;
    const uint8_t* wo;
    const uint8_t* wgate;
    const uint8_t* wup;
    const uint8_t* wdown;
    const float* q_norm;  // Qwen3 attention inputs: per-head RMSNorm weights [hd] (null: plain attention)
    const float* k_norm;
    int down_fmt;
    int pad;
};

struct TokenArgs {
    const TokenLayer* layers;  // device [n_layers]
    int n_layers, hidden, ffn, n_q, n_kv, hd, vocab, max_ctx;
    float eps;
    const float* out_norm;
    const uint8_t* wvocab;
    __half* kv;                // [n_layers][2][n_kv][max_ctx][hd]
    float* x;                  // residual stream [hidden]
    float* q;                  // [n_q hd]
    float* attn;               // [n_q hd]
    float* act;                // [ffn]
    float* part;               // attention partials
    int* counters;             // attention merge counters (unused here: zero)
    unsigned* stamps;          // attention chunk stamps [n_kv][ATT_CHUNKS]
    int fold;                  // 1: pos + 1 <= TK_FOLD_KEYS, the attention is folded into the O phase
    float* k_new;              // the token's keys [n_kv hd], tagged: as projected (Qwen3) or their fp16 values
    float* v_new;              // the token's values [n_kv hd], tagged fp16 values
    int qwen;                  // Qwen3 attention inputs (per-head norms and rotation)
    const float2* rope;        // (cos, sin) table [max_ctx][hd / 2] with the Qwen3 inputs
    StepArgs* step;            // pos and logits recorded for the diagnostics entry points
    unsigned* bar;             // launch state: [1] blocks finished, [2] token count, [3] a wait ran out
    unsigned long long wait_ns;  // bound on every wait of the launch (wall-clock ns)
    int skew;                  // diagnostics: not 0 -- every tagged read waits for a write never made
    int pad2;
    const float* x_in;
    float* logits;
    int pos;
    int* err;
    unsigned long long* trace; // diagnostics: 4 timestamps per block and phase when not null
};

struct PhaseEnt {
    const uint8_t* W;
    const uint8_t* W2;
    int T0;    // the block's first tile of the phase (tiles numbered over the whole token)
    int kind;
};

struct KindEnt {
    int rows, K, row_bytes, R, nmat;
    int r0, r1;  // this block's rows [r0, r1) of each matrix
    int pad;
};

// Shared memory of one block, at fixed offsets: the weight ring, the per-warp
// partial sums, barriers and flags, the kind table, the block's residual rows,
// the phase table, then the quantised activation (aliased by the attention
// staging), whose size depends on the model shape.
constexpr int TK_RESID_MAX = 64;   // residual rows of one block at most
constexpr int TK_MAX_LAYERS = 64;
constexpr int TK_OFF_RED = TK_NSTAGE * TK_SLOT;
constexpr int TK_OFF_MISC = TK_OFF_RED + 2 * TK_NSTAGE * TK_WARPS * TK_RED_STRIDE * 4;
constexpr int TK_OFF_ARGS = TK_OFF_MISC + 256;
constexpr int TK_OFF_KTAB = TK_OFF_ARGS + (static_cast<int>(sizeof(TokenArgs)) + 127) / 128 * 128;
constexpr int TK_OFF_RESID = TK_OFF_KTAB + 256;
constexpr int TK_OFF_PTAB = TK_OFF_RESID + TK_RESID_MAX * 4;
constexpr int TK_OFF_XQ = TK_OFF_PTAB + ((5 * TK_MAX_LAYERS + 2) * static_cast<int>(sizeof(PhaseEnt)) + 127) / 128 * 128;

// Bytes of one attention item's staging, rounded to 128: two items run at a time.
constexpr int TK_ATT_STAGING = (static_cast<int>(sizeof(AttnSmem)) + 127) / 128 * 128;

// Shared-memory bytes of the block for a model shape: the quantised
// activation of the largest input (two planes for Q|K|V, one for O and the
// down projection) or the attention staging of two items, whichever is larger.
__host__ __device__ inline int tk_smem_bytes(int hidden, int qdim, int ffn)
{
    int xq = (hidden > qdim ? hidden : qdim) / 32 * xq_words(2) * 4;
    xq = xq > ffn / 32 * xq_words(1) * 4 ? xq : ffn / 32 * xq_words(1) * 4;
    xq = xq > 2 * TK_ATT_STAGING ? xq : 2 * TK_ATT_STAGING;
    return TK_OFF_XQ + xq;
}

}  // namespace dq

namespace dqhost {

using TokenKernel = void (*)(dq::TokenArgs);

struct TokenPlan {
    int nph;          // phases per token (5 per layer + 1)
    int grid;         // one block per SM
    int smem_bytes;
    TokenKernel kernel;
};

// Whether the persistent token kernel covers this model shape (DQ_OK) or not
// (DQ_ERR_UNSUPPORTED): at most 64 layers, hidden and n_q head_dim <= 4096,
// ffn <= 16384 (12288 with a Q6_K down projection), and the block's shared
// memory fits.
int plan_token(int n_layers, int hidden, int ffn, int n_q, int n_kv, int hd, bool any_q6_down, TokenPlan* plan);

// Cooperative launch of one token on `stream` (grid barriers need every block resident).
cudaError_t launch_token(const TokenPlan& plan, const dq::TokenArgs& a, cudaStream_t stream);

}  // namespace dqhost
