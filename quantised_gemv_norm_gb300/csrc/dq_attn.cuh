// dq_attn.cuh -- arguments and launcher of the grouped-query decode attention.
#pragma once

#include "dq_gemv.cuh"

namespace dq {

constexpr int ATT_HD = 128;      // head dimension the kernel is written for (4 dims per lane)
constexpr int ATT_CHUNKS = 16;   // key chunks per KV head (thread blocks per KV head)
constexpr int ATT_BATCH = 32;    // keys staged in shared memory at a time (one per lane)
constexpr int ATT_MIN_CHUNK = 64; // fewest keys per block
constexpr int ATT_PART = 4 + ATT_HD;  // floats per partial: m, l, 2 pad, o[128]
constexpr int ATT_COUNTER_BYTES = 256;

struct AttnArgs {
    const float* q;        // [n_q][128]
    const __half* kc;      // [n_kv][max_ctx][128]
    const __half* vc;
    float* out;            // [n_q][128]
    float* part;           // [n_q][ATT_CHUNKS][ATT_PART]
    int* counters;         // [n_kv], zero between calls
    int n_q, n_kv, max_ctx;
    int n_keys;            // used when step == null
    const StepArgs* step;  // decode graph: n_keys = step->pos + 1
    int* err;
};

}  // namespace dq

namespace dqhost {

size_t attention_workspace_bytes(int n_q, int n_kv);
// Splits a workspace into the counters and the partials.
void attention_bind_workspace(dq::AttnArgs& a, void* ws);
cudaError_t launch_attention(const dq::AttnArgs& a, cudaStream_t stream, bool pdl);

}  // namespace dqhost
