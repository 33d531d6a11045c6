// dq_token.cu -- one decode token as a single persistent kernel (sm_103a).
//
// The token is the chain of phases of the per-kernel path (per layer: norm +
// Q|K|V + cache append, attention, O + residual, norm + gate/up + SwiGLU,
// down + residual; then norm + vocabulary), run by one block per SM that stays
// resident for the whole token.  Every phase reads the whole output of the one
// before, but the weight stream does not wait for it: each block numbers the
// weight tiles of all its phases in one sequence and refills its ring slots in
// that order, so the tiles of the next phase are already in flight while the
// current phase finishes and the next activation arrives and is quantised.
// That removes the per-kernel start-up and drain cost that dominates a chain
// of short launches ("The roofline holds on a second GPU", section "Hiding,
// fusing...": keep the bytes in flight across the whole token; "The Mountain
// Runs", section 3: one output per weight row).
//
// The consumers are those of the streaming GEMV kernel (dq_gemv.cuh): 512
// threads in row groups, each thread holding its 32-element units of the
// quantised activation in registers; tile t is completed (slot refilled, rows'
// epilogue run) by warp t % 16 as soon as every warp has released it.  The
// attention phase runs one (key chunk, KV head) item per block on the first
// n_q / n_kv warps (dq_attn.cuh); contexts of at most TK_FOLD_KEYS keys fold it
// into the O phase instead.
//
// Tagged activations instead of grid barriers.  A grid barrier between two
// phases cost 1.3-2.5 us: a release fence before each block's arrival (it waits
// for the block's outstanding stores under full HBM load, 0.5-1.3 us), the
// counter's round trips, then the activation's load.  The vectors the phases
// hand on (the residual x, the attention output, the SwiGLU activation, q and
// fp32 copies of the new key and value) carry their own validity instead: every
// value is written with its lowest mantissa bit set to the parity of the write
// (one fp32 ulp, far below the activation format's rounding), and a reader
// loads the vector straight away, re-reading values whose bit does not yet show
// the write it waits for.  No grid barrier is needed: a phase reads the whole
// vector the previous one wrote, so a block can only start writing a vector
// again after every block has read its previous contents (those reads came
// before the outputs it waited for), and each location alternates between
// consecutive writes, so one bit tells them apart.  The cache rows of the
// token's position are written, from the tagged copies, by the block that
// stages them for the attention (one block per KV head when the attention is
// folded), and the
// attention's merge counters count on across the layers of a token.
//
// Every wait is bounded.  A block whose wait runs out records the error and
// stops working; blocks that wait on its outputs run out in turn, so the token
// ends (with meaningless output) instead of hanging.  The last block out then
// puts the counters and the tagged vectors back into their initial state, so
// the model stays usable.
#include <algorithm>

#include "dq_token.cuh"

namespace dq {

constexpr int DEVERR_TIMEOUT_TAG = 16;  // a wait for another block's output ran out

// Words of the launch-state area (TokenArgs::bar; word 0 unused).
constexpr int TB_EXIT = 1;    // blocks finished
constexpr int TB_TOKEN = 2;   // tokens run since the tagged vectors were reset
constexpr int TB_FAULT = 3;   // a block of this launch gave up a wait

__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* p)
{
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ float4 ld_relaxed_f4(const float* p)
{
    float4 v;
    asm volatile("ld.relaxed.gpu.global.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_f32(float* p, float v)
{
    asm volatile("st.relaxed.gpu.global.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// v with its lowest mantissa bit set to `par`.
__device__ __forceinline__ float tagged(float v, uint32_t par)
{
    return __uint_as_float((__float_as_uint(v) & ~1u) | par);
}

// Whether all four values carry the tag `par`.
__device__ __forceinline__ bool tags_ok(float4 v, uint32_t par)
{
    const uint32_t x = __float_as_uint(v.x) ^ par, y = __float_as_uint(v.y) ^ par, z = __float_as_uint(v.z) ^ par,
                   w = __float_as_uint(v.w) ^ par;
    return ((x | y | z | w) & 1u) == 0u;
}

// The block's shared memory (layout: dq_token.cuh).
extern __shared__ __align__(128) uint8_t tk_smem[];

struct TkMisc {
    float gred[TK_WARPS];      // norm partial sums
    uint64_t full[TK_NSTAGE];  // stage loaded
    uint64_t empty[TK_NSTAGE]; // stage released by all warps
    int dead;                  // a wait of this block ran out
    int issued_hi;             // one past the highest tile issued
    int sync_ok;
    int ttotal;                // the block's tiles over the token
    unsigned tokpar;           // parity of the token count (tags of vectors written once per layer)
    unsigned tokseq;           // the token count
    int last_out;              // this block finished last
};
static_assert(sizeof(TkMisc) <= 256, "misc region");

__device__ __forceinline__ TkMisc& tk_misc() { return *reinterpret_cast<TkMisc*>(tk_smem + TK_OFF_MISC); }
// The launch arguments, copied to shared memory at kernel start: the phase
// functions read them there instead of holding them in registers.
__device__ __forceinline__ const TokenArgs& tk_args() { return *reinterpret_cast<const TokenArgs*>(tk_smem + TK_OFF_ARGS); }
__device__ __forceinline__ KindEnt* tk_ktab() { return reinterpret_cast<KindEnt*>(tk_smem + TK_OFF_KTAB); }
__device__ __forceinline__ float* tk_resid() { return reinterpret_cast<float*>(tk_smem + TK_OFF_RESID); }
__device__ __forceinline__ uint32_t* tk_xq() { return reinterpret_cast<uint32_t*>(tk_smem + TK_OFF_XQ); }
__device__ __forceinline__ float* tk_red() { return reinterpret_cast<float*>(tk_smem + TK_OFF_RED); }
__device__ __forceinline__ PhaseEnt* tk_ptab() { return reinterpret_cast<PhaseEnt*>(tk_smem + TK_OFF_PTAB); }

// Tag of write `idx` (0-based within a token) of a vector written `per_token`
// times a token.  The count runs on across tokens, so consecutive writes
// alternate whatever the number of layers; the first write after a reset has
// tag 1, and the reset state (all zero) tag 0.
__device__ __forceinline__ uint32_t tk_par(int per_token, int idx)
{
    return (tk_misc().tokpar * static_cast<unsigned>(per_token) + static_cast<unsigned>(idx) + 1u) & 1u;
}
// The residual x is written twice per layer: by O (idx 2l) and by down (2l + 1).
__device__ __forceinline__ uint32_t tk_par_x_o(int l) { return tk_par(2 * tk_args().n_layers, 2 * l); }
__device__ __forceinline__ uint32_t tk_par_x_down(int l) { return tk_par(2 * tk_args().n_layers, 2 * l + 1); }
// act, q and the new key and value: once per layer.
__device__ __forceinline__ uint32_t tk_par_layer(int l) { return tk_par(tk_args().n_layers, l); }

// Stream tile T (numbered over the token) into its ring slot.  `cur` is the
// calling thread's cursor into the phase table (each thread issues tiles in
// increasing order, so it only moves forward).
__device__ __forceinline__ void tk_issue(int T, int& cur)
{
    const PhaseEnt* ptab = tk_ptab();
    while (T >= ptab[cur + 1].T0)
        ++cur;
    const PhaseEnt& e = ptab[cur];
    const KindEnt& k = tk_ktab()[e.kind];
    const int row = k.r0 + (T - e.T0) * k.R;
    const int nr = min(k.R, k.r1 - row);
    const uint32_t bytes = static_cast<uint32_t>(nr * k.row_bytes);
    const int s = T & (TK_NSTAGE - 1);
    uint8_t* dst = tk_smem + s * TK_SLOT;
    TkMisc& m = tk_misc();
    const uint64_t pol = l2_evict_first_policy();
    mbar_arrive_expect_tx(&m.full[s], bytes * k.nmat);
    bulk_g2s(dst, e.W + static_cast<size_t>(row) * k.row_bytes, bytes, &m.full[s], pol);
    if (k.nmat == 2)
        bulk_g2s(dst + k.R * k.row_bytes, e.W2 + static_cast<size_t>(row) * k.row_bytes, bytes, &m.full[s], pol);
    atomicMax(&m.issued_hi, T + 1);
}

// Diagnostics: stamp i (0..7) of phase p of this block; even stamps are the global
// timer (ns), odd ones the SM clock (cycles).
__device__ __forceinline__ void tk_trace(int p, int i)
{
    const TokenArgs& A = tk_args();
    if (A.trace && threadIdx.x == 0)
        A.trace[(static_cast<size_t>(blockIdx.x) * (5 * A.n_layers + 1) + p) * 8 + i] =
            (i & 1) ? clock64() : globaltimer_ns();
}

// A wait of this block ran out: record it for the host and for the launch's
// last block (which then resets the tagged vectors), and stop working.
__device__ __forceinline__ void tk_give_up(int code)
{
    const TokenArgs& A = tk_args();
    set_error(A.err, code);
    atomicExch(A.bar + TB_FAULT, 1u);
    tk_misc().dead = 1;
}

// Load chunks c = tid + NT i (float4, c < nchunks) of a tagged vector, re-reading
// those whose tags do not yet show `par`.  The loop is warp-uniform (the lanes
// wait for each other, so later shuffles see converged warps).  False when the
// wait ran out.
template <int NCH, int NT>
__device__ __forceinline__ bool tk_load_tagged(float4 (&v)[NCH], const float* x, int nchunks, int tid, uint32_t par)
{
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
        const int c = tid + NT * i;
        v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < nchunks)
            v[i] = ld_relaxed_f4(x + 4 * c);
    }
    unsigned long long t0 = 0;
    while (true) {
        bool mine = true;
#pragma unroll
        for (int i = 0; i < NCH; ++i)
            if (tid + NT * i < nchunks)
                mine = mine && tags_ok(v[i], par);
        if (__all_sync(0xffffffffu, mine))
            return true;
        const unsigned long long now = globaltimer_ns();
        if (t0 == 0)
            t0 = now;
        else if (__any_sync(0xffffffffu, now - t0 > tk_args().wait_ns))
            return false;
#pragma unroll
        for (int i = 0; i < NCH; ++i) {
            const int c = tid + NT * i;
            if (c < nchunks && !tags_ok(v[i], par))
                v[i] = ld_relaxed_f4(x + 4 * c);
        }
    }
}

// Attention for a short context (n_keys <= TK_FOLD_KEYS), computed by every
// block at the start of the O phase of layer l and quantised straight into the
// O projection's activation table: no attention phase of its own.  Warp w takes query heads w and w + 16 together (n_q <= 32); lane i
// holds dims 4i..4i+3.  With the Qwen3 inputs each block normalises and
// rotates q and the new key itself; one block per head writes the head's output
// and, for a group's first head, the key's and value's fp16 rows into the cache
// (the other blocks use the same rounded values from registers).
// Same arithmetic as attn_block.
//
// The head-norm weights and the rotary row do not depend on this token's q|k|v
// phase, and their addresses take a load of their own: they are loaded before
// the phase's block barrier (tk_fold_preload).  After it, one round trip brings q, the
// new key and value (tagged copies of what the q|k|v phase wrote) and the
// cache rows of the earlier positions.
struct FoldPre {
    NormRope qn, kn;
};

__device__ __forceinline__ void tk_fold_preload(int l, FoldPre& f)
{
    const TokenArgs& A = tk_args();
    const int lane = threadIdx.x & 31;
    if (A.qwen) {
        const float2* cs = A.rope + static_cast<size_t>(A.pos) * (ATT_HD / 2);
        f.qn = load_norm_rope(A.layers[l].q_norm, cs, lane);
        f.kn = load_norm_rope(A.layers[l].k_norm, cs, lane);
    }
}

__device__ __forceinline__ uint2 half4_bits(float4 v)
{
    const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    return make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
}

template <int PL>
__device__ __forceinline__ bool tk_fold_attention(int l, const FoldPre& f)
{
    // the arguments in registers: the table stores below would otherwise make the
    // compiler reload every field from shared memory inside the chain
    const TokenArgs& A0 = tk_args();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pos = A0.pos, n_keys = pos + 1, n_q = A0.n_q, group = n_q / A0.n_kv, max_ctx = A0.max_ctx;
    const size_t plane = static_cast<size_t>(A0.n_kv) * max_ctx * ATT_HD;
    __half* kc = A0.kv + static_cast<size_t>(l) * 2 * plane;
    const __half* vc = kc + plane;
    const float* Aq = A0.q;
    const float* Ak = A0.k_new;
    const float* Av = A0.v_new;
    const bool qwen = A0.qwen != 0;
    const float eps = A0.eps;
    const unsigned long long wait_ns = A0.wait_ns;
    const uint32_t opar_att = tk_par_layer(l);
    const uint32_t par = opar_att ^ (A0.skew != 0 ? 1u : 0u);  // a skew: a write that never comes
    float* Aatt = A0.attn;
    uint32_t* xq = tk_xq();
    constexpr int NH = 2;  // heads per warp
    bool on[NH];
    int hh[NH], gg[NH];
    float4 q[NH], k[NH], v[NH];
    uint2 kr[NH][TK_FOLD_KEYS - 1], vr[NH][TK_FOLD_KEYS - 1];  // cache rows j < pos
#pragma unroll
    for (int i = 0; i < NH; ++i) {
        hh[i] = warp + TK_WARPS * i;
        on[i] = hh[i] < n_q;
        gg[i] = on[i] ? hh[i] / group : 0;
        const size_t row0 = static_cast<size_t>(gg[i]) * max_ctx * ATT_HD;
        q[i] = k[i] = v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (on[i]) {
            q[i] = ld_relaxed_f4(Aq + static_cast<size_t>(hh[i]) * ATT_HD + 4 * lane);
            k[i] = ld_relaxed_f4(Ak + static_cast<size_t>(gg[i]) * ATT_HD + 4 * lane);
            v[i] = ld_relaxed_f4(Av + static_cast<size_t>(gg[i]) * ATT_HD + 4 * lane);
        }
#pragma unroll
        for (int j = 0; j < TK_FOLD_KEYS - 1; ++j) {
            kr[i][j] = vr[i][j] = make_uint2(0u, 0u);
            if (on[i] && j < pos) {
                kr[i][j] = __ldcg(reinterpret_cast<const uint2*>(kc + row0 + static_cast<size_t>(j) * ATT_HD) + lane);
                vr[i][j] = __ldcg(reinterpret_cast<const uint2*>(vc + row0 + static_cast<size_t>(j) * ATT_HD) + lane);
            }
        }
    }
    // the tagged values: re-read any that does not yet show this layer's write
    unsigned long long t0 = 0;
    while (true) {
        bool mine = true;
#pragma unroll
        for (int i = 0; i < NH; ++i)
            if (on[i])
                mine = mine && tags_ok(q[i], par) && tags_ok(k[i], par) && tags_ok(v[i], par);
        if (__all_sync(0xffffffffu, mine))
            break;
        const unsigned long long now = globaltimer_ns();
        if (t0 == 0)
            t0 = now;
        else if (__any_sync(0xffffffffu, now - t0 > wait_ns))
            return false;
#pragma unroll
        for (int i = 0; i < NH; ++i)
            if (on[i]) {
                if (!tags_ok(q[i], par))
                    q[i] = ld_relaxed_f4(Aq + static_cast<size_t>(hh[i]) * ATT_HD + 4 * lane);
                if (!tags_ok(k[i], par))
                    k[i] = ld_relaxed_f4(Ak + static_cast<size_t>(gg[i]) * ATT_HD + 4 * lane);
                if (!tags_ok(v[i], par))
                    v[i] = ld_relaxed_f4(Av + static_cast<size_t>(gg[i]) * ATT_HD + 4 * lane);
            }
    }
    const float scale = 0.08838834764831845f;  // 1 / sqrt(128)
#pragma unroll
    for (int i = 0; i < NH; ++i) {
        if (!on[i])  // warp-uniform
            continue;
        float4 qi = q[i];
        uint2 knew;  // the current position's key as the cache holds it (fp16)
        if (qwen) {
            qi = head_norm_rope(qi, f.qn, eps, lane);
            knew = half4_bits(head_norm_rope(k[i], f.kn, eps, lane));
        } else {
            knew = half4_bits(k[i]);  // the tagged copy of an fp16 value rounds back to it
        }
        const uint2 vnew = half4_bits(v[i]);
        // head h's output (and, for a group's first head, the position's cache rows) is
        // written by block h % blocks: one block each, spread so no block runs late
        const bool writer = blockIdx.x == hh[i] % gridDim.x;
        if (writer && hh[i] % group == 0) {
            const size_t at = (static_cast<size_t>(gg[i]) * max_ctx + pos) * ATT_HD + 4 * lane;
            *reinterpret_cast<uint2*>(kc + at) = knew;
            *reinterpret_cast<uint2*>(const_cast<__half*>(vc) + at) = vnew;
        }
        float sj[TK_FOLD_KEYS];
        float m = -INFINITY;
#pragma unroll
        for (int j = 0; j < TK_FOLD_KEYS; ++j) {
            sj[j] = -INFINITY;
            if (j < n_keys) {
                const uint2 kb = j == pos ? knew : kr[i][j < TK_FOLD_KEYS - 1 ? j : 0];
                const float2 k0 = __half22float2(*reinterpret_cast<const __half2*>(&kb.x));
                const float2 k1 = __half22float2(*reinterpret_cast<const __half2*>(&kb.y));
                float d = fmaf(qi.x, k0.x, qi.y * k0.y) + fmaf(qi.z, k1.x, qi.w * k1.y);
                d = warp_sum(d) * scale;
                sj[j] = d;
                m = fmaxf(m, d);
            }
        }
        float lsum = 0.f;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < TK_FOLD_KEYS; ++j)
            if (j < n_keys) {
                const float pj = expf(sj[j] - m);
                lsum += pj;
                const uint2 vb = j == pos ? vnew : vr[i][j < TK_FOLD_KEYS - 1 ? j : 0];
                const float2 v0 = __half22float2(*reinterpret_cast<const __half2*>(&vb.x));
                const float2 v1 = __half22float2(*reinterpret_cast<const __half2*>(&vb.y));
                o.x = fmaf(pj, v0.x, o.x); o.y = fmaf(pj, v0.y, o.y);
                o.z = fmaf(pj, v1.x, o.z); o.w = fmaf(pj, v1.y, o.w);
            }
        const float inv = 1.0f / lsum;
        o = make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
        quantise_chunk<FMT_Q4K, PL>(o, hh[i] * (ATT_HD / 4) + lane, xq);
        if (writer)  // the attention output too (its tags then alternate every layer)
            att_st_out(Aatt + static_cast<size_t>(hh[i]) * ATT_HD + 4 * lane, o, 1 + static_cast<int>(opar_att));
    }
    return true;
}

// One matrix phase p of kind KIND: prefetch the norm weight, load the tagged
// activation as it arrives, quantise it, consume the phase's tiles and complete them (refill
// + epilogue).  T is the block's next tile, icur the caller's issue cursor;
// returns both advanced.
template <int KIND, int FMT, int PL, int NMAT, int EPI, bool NORM>
__device__ __forceinline__ int2 tk_gemv(int p, int T, int icur)
{
    constexpr int P = tk_p(KIND);     // threads per row group, one activation unit each
    constexpr int RG = tk_rg(KIND);   // row groups
    constexpr int RP = tk_rpt(KIND);  // rows per thread and matrix
    constexpr int R = RG * RP;        // rows per tile and matrix
    constexpr int UL = tk_ul(KIND);   // activation units a thread holds
    constexpr int NCH = (8 * P * UL + TK_THREADS - 1) / TK_THREADS;  // 4-element chunks a thread quantises
    static_assert(RP * NMAT <= TK_RED_STRIDE, "partial sums per warp");
    const TokenArgs& A = tk_args();
    const KindEnt& ke = tk_ktab()[KIND];
    const int K = ke.K;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const PhaseEnt* ptab = tk_ptab();
    const int T0 = ptab[p].T0, ntiles = ptab[p + 1].T0 - T0;
    const int r0 = ke.r0, r1 = ke.r1;
    TkMisc& m = tk_misc();
    const int l = p / 5;
    const bool fold = KIND == PH_O && A.fold;
    const float* gamma = KIND == PH_QKV ? A.layers[l].attn_norm : KIND == PH_GATEUP ? A.layers[l].ffn_norm : A.out_norm;

    tk_trace(p, 0);
    FoldPre fpre;
    if (fold)
        tk_fold_preload(l, fpre);
    float4 gv[NCH];
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
        const int ch = tid + TK_THREADS * i;
        gv[i] = make_float4(1.f, 1.f, 1.f, 1.f);
        if (NORM && ch < K / 4)
            gv[i] = __ldg(reinterpret_cast<const float4*>(gamma) + ch);
    }
    // What the prologue reads, taken from the argument table before the block
    // barrier (after it, every table read would sit in the prologue's dependency chain):
    // the input vector, whether it carries tags and which, the residual rows.
    const bool from_act = KIND == PH_DOWN_Q4 || KIND == PH_DOWN_Q6;
    const bool untagged_in = KIND == PH_QKV && l == 0;  // x_in, written before the launch
    const float* xsrc = KIND == PH_QKV && l == 0 ? A.x_in : KIND == PH_O ? A.attn : from_act ? A.act : A.x;
    // act and attn: this layer's write; x after the O projection (gate/up), after the
    // previous layer's down (q|k|v, vocabulary)
    const uint32_t ipar = from_act || KIND == PH_O ? tk_par_layer(l)
                          : KIND == PH_GATEUP ? tk_par_x_o(l)
                                              : tk_par_x_down(KIND == PH_VOCAB ? A.n_layers - 1 : l - 1);
    const float* rsrc = (KIND == PH_O && l == 0 ? A.x_in : A.x) + r0;
    // diagnostics: with a skew every tagged read waits for a write that never comes
    const uint32_t ipar_w = ipar ^ (A.skew != 0 ? 1u : 0u);
    const float eps = A.eps;
    // no grid barrier: the input is tagged; the block's own warps finish the previous
    // phase's epilogue first (the prologue reuses its shared memory)
    __syncthreads();
    if (m.dead)
        return make_int2(T, icur);
    tk_trace(p, 2);
    tk_trace(p, 3);

    // the block's residual rows (at most TK_RESID_MAX < TK_THREADS): its own
    // outputs of the previous residual phase (x_in for layer 0's O), loaded now
    // and stored after the activation's loads have gone out
    float rv = 0.f;
    if (EPI == EPI_RESID && tid < r1 - r0)
        rv = __ldcg(rsrc + tid);
    float ss = 0.f;
    bool ok = true;
    if (fold) {
        ok = tk_fold_attention<PL>(l, fpre);
    } else {
        float4 xv[NCH];
        if (untagged_in) {  // the token's input, written before the launch
#pragma unroll
            for (int i = 0; i < NCH; ++i) {
                const int ch = tid + TK_THREADS * i;
                xv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (ch < K / 4)
                    xv[i] = __ldcg(reinterpret_cast<const float4*>(xsrc) + ch);
            }
        } else {
            ok = tk_load_tagged<NCH, TK_THREADS>(xv, xsrc, K / 4, tid, ipar_w);
        }
        ss = quantise_block_il<FMT, PL, NCH, TK_THREADS>(xv, gv, NORM, tk_xq(), K, tid);
    }
    if (EPI == EPI_RESID && tid < r1 - r0)
        tk_resid()[tid] = rv;
    if (NORM) {
        ss = warp_sum(ss);
        if (lane == 0)
            m.gred[warp] = ss;
    }
    if (!ok && lane == 0)
        tk_give_up(DEVERR_TIMEOUT_TAG);
    __syncthreads();  // quantised activation, residual rows and norm partials complete
    if (m.dead) {
        tk_trace(p, 4);
        return make_int2(T, icur);
    }
    tk_trace(p, 5);
    float rstd = 1.f;
    if (NORM) {
        const float4* g4 = reinterpret_cast<const float4*>(m.gred);
        const float4 ga = g4[0], gb = g4[1], gc = g4[2], gd = g4[3];
        const float tot = ((ga.x + ga.y) + (ga.z + ga.w)) + ((gb.x + gb.y) + (gb.z + gb.w)) +
                          (((gc.x + gc.y) + (gc.z + gc.w)) + ((gd.x + gd.y) + (gd.z + gd.w)));
        rstd = rsqrtf(tot / static_cast<float>(K) + eps);
    }
    const int g = tid / P, pp = tid % P;
    UnitState<FMT, PL> us[UL];
    bool have[UL];
    int nidx[UL];
#pragma unroll
    for (int k = 0; k < UL; ++k) {
        have[k] = pp + P * k < K / 32;
        nidx[k] = have[k] ? pp + P * k : K / 32 - 1;  // a stand-in for a missing unit (zero activation)
    }
    load_units<FMT, PL, UL>(us, have, tk_xq(), pp, P, rstd);
    tk_trace(p, 7);

    // tags of this phase's outputs
    const uint32_t opar = EPI == EPI_RESID ? (KIND == PH_O ? tk_par_x_o(l) : tk_par_x_down(l)) : tk_par_layer(l);

    // Complete tile tc (token tile Tc) once every warp has released it: refill
    // its slot with tile Tc + TK_NSTAGE, run the epilogue of its rows.  Tile Tc
    // belongs to warp Tc % 16, which tests the slot's `empty` barrier after each
    // of its stages and while it waits for its next one (no fixed delay; a warp
    // only waits on another when its next stage needs that very refill).
    auto complete = [&](int tc, int Tc) {
        if (lane == 0 && Tc + TK_NSTAGE < m.ttotal)
            tk_issue(Tc + TK_NSTAGE, icur);
        const float* rb = tk_red() + (Tc & (2 * TK_NSTAGE - 1)) * TK_WARPS * TK_RED_STRIDE;
        const int row0 = r0 + tc * R;
        const int nr = min(R, r1 - row0);
        for (int row = lane; row < nr; row += 32) {
            const int rg = row % RG, i = row / RG;
            const float* wb = rb + rg * (P / 32) * TK_RED_STRIDE;
            float v0 = 0.f, v1 = 0.f;
#pragma unroll
            for (int w = 0; w < P / 32; ++w) {
                v0 += wb[w * TK_RED_STRIDE + i];
                if (NMAT == 2)
                    v1 += wb[w * TK_RED_STRIDE + RP + i];
            }
            const int r = row0 + row;
            if (EPI == EPI_STORE) {
                A.logits[r] = v0;
            } else if (EPI == EPI_RESID) {
                st_relaxed_f32(A.x + r, tagged(tk_resid()[r - r0] + v0, opar));
            } else if (EPI == EPI_SWIGLU) {
                st_relaxed_f32(A.act + r, tagged(v0 / (1.0f + expf(-v0)) * v1, opar));
            } else {  // EPI_QKV: q rows, then k and v rows
                const int qdim = A.n_q * ATT_HD, kvdim = A.n_kv * ATT_HD;
                if (r < qdim) {
                    st_relaxed_f32(A.q + r, tagged(v0, opar));
                } else {
                    // k and v: tagged fp32 copies (the key as projected with the Qwen3
                    // inputs, else the fp16 value the cache will hold); the attention
                    // (or the fold) writes the cache rows from them
                    const int idx = r - qdim;
                    const bool is_v = idx >= kvdim;
                    const int rem = idx - (is_v ? kvdim : 0);
                    const float copy = (is_v || !A.qwen) ? __half2float(__float2half_rn(v0)) : v0;
                    st_relaxed_f32((is_v ? A.v_new : A.k_new) + rem, tagged(copy, opar));
                }
            }
        }
    };
    auto released = [&](int Tc) { return mbar_test_wait(&m.empty[Tc & (TK_NSTAGE - 1)], (Tc / TK_NSTAGE) & 1); };

    int pend = -1;  // this warp's tile (phase-local index) still to complete
#pragma unroll 1
    for (int t = 0; t < ntiles; ++t, ++T) {
        const int s = T & (TK_NSTAGE - 1);
        const uint32_t ph = (T / TK_NSTAGE) & 1;
        bool got = false;
        if (pend >= 0 && !mbar_test_wait(&m.full[s], ph)) {  // complete the pending tile while waiting
            const unsigned long long t0 = globaltimer_ns();
            while (pend >= 0) {
                if (released(T0 + pend)) {
                    complete(pend, T0 + pend);
                    pend = -1;
                } else if (mbar_test_wait(&m.full[s], ph)) {
                    got = true;
                    break;
                } else if (globaltimer_ns() - t0 > A.wait_ns) {
                    set_error(A.err, DEVERR_TIMEOUT_EMPTY);
                    ok = false;
                    break;
                }
            }
            if (!ok)
                break;
        } else if (pend >= 0) {
            got = true;
        }
        if (!got && !mbar_wait(&m.full[s], ph, A.wait_ns)) {
            set_error(A.err, DEVERR_TIMEOUT_FULL);
            ok = false;
            break;
        }
        if (t == 0)
            tk_trace(p, 1);
        consume_tile<FMT, PL, UL, RP, NMAT>(
            tk_smem + s * TK_SLOT, R, RG, g, ke.row_bytes, us, nidx,
            tk_red() + ((T & (2 * TK_NSTAGE - 1)) * TK_WARPS + warp) * TK_RED_STRIDE, lane);
        if (lane == 0)
            mbar_arrive(&m.empty[s]);
        if (T % TK_WARPS == warp)
            pend = t;
        if (pend >= 0 && released(T0 + pend)) {
            complete(pend, T0 + pend);
            pend = -1;
        }
    }
    if (ok && pend >= 0) {  // the phase's epilogue must be done before the block moves on
        if (mbar_wait(&m.empty[(T0 + pend) & (TK_NSTAGE - 1)], ((T0 + pend) / TK_NSTAGE) & 1, A.wait_ns))
            complete(pend, T0 + pend);
        else {
            set_error(A.err, DEVERR_TIMEOUT_EMPTY);
            ok = false;
        }
    }
    if (!ok) {
        atomicExch(A.bar + TB_FAULT, 1u);
        m.dead = 1;
    }
    tk_trace(p, 4);
    return make_int2(T0 + ntiles, icur);
}

// Attention phase p: items (key chunk, KV head) spread over the blocks, in the
// tagged mode of attn_block (q and the new key and value are polled by their
// tags, the chunks meet through release/acquire stamps, the output is tagged).
__device__ __forceinline__ void tk_attention(int p)
{
    const TokenArgs& A = tk_args();
    TkMisc& m = tk_misc();
    tk_trace(p, 0);
    __syncthreads();  // the staging below reuses the quantised-activation area
    if (m.dead)
        return;
    tk_trace(p, 2);
    const int group = A.n_q / A.n_kv;
    const int sub = (threadIdx.x >> 5) / group;  // two items at a time: warps [0, group) and [group, 2 group)
    if (sub < 2) {
        const int l = p / 5;
        const size_t plane = static_cast<size_t>(A.n_kv) * A.max_ctx * A.hd;
        const int n_keys = A.pos + 1;
        const int L = max((n_keys + ATT_CHUNKS - 1) / ATT_CHUNKS, ATT_MIN_CHUNK);
        const int nact = (n_keys + L - 1) / L;
        AttnArgs t{};
        t.q = A.q;
        t.kc = A.kv + static_cast<size_t>(l) * 2 * plane;
        t.vc = t.kc + plane;
        t.out = A.attn;
        t.part = A.part;
        t.counters = A.counters;
        t.n_q = A.n_q;
        t.n_kv = A.n_kv;
        t.max_ctx = A.max_ctx;
        t.n_keys = n_keys;
        t.step = nullptr;
        t.err = A.err;
        t.k_new = A.k_new;
        t.q_norm = A.layers[l].q_norm;
        t.k_norm = A.layers[l].k_norm;
        t.rope = A.rope;
        t.eps = A.eps;
        t.tag = 1 + static_cast<int>(tk_par_layer(l) ^ (A.skew != 0 ? 1u : 0u));
        t.stamps = A.stamps;
        t.seq = tk_misc().tokseq * static_cast<unsigned>(A.n_layers) + static_cast<unsigned>(l) + 1u;
        t.v_new = A.v_new;
        t.wait_ns = A.wait_ns;
        if (A.trace && sub == 0)  // the block's first item
            t.trace = A.trace + (static_cast<size_t>(blockIdx.x) * (5 * A.n_layers + 1) + p) * 8;
        AttnSmem& sm = *reinterpret_cast<AttnSmem*>(tk_xq() + sub * (TK_ATT_STAGING / 4));
        const int bar = ATT_BAR - sub;
        // Items are numbered chunks first, merging (last) chunks after them: every
        // warp group takes its items in increasing order, so a merging item only ever
        // waits for items that their groups run before any merging one.
        const int nplain = (nact - 1) * A.n_kv;
        // item b of block b's first warp group, then b + blocks of its second: up to one
        // item a block runs alone (at 512 keys 136 items on 136 blocks rather than two
        // each on 68)
        for (int item = static_cast<int>(blockIdx.x + gridDim.x * sub); item < nact * A.n_kv; item += 2 * gridDim.x) {
            const int c = item < nplain ? item % (nact - 1) : nact - 1;
            const int g = item < nplain ? item / (nact - 1) : item - nplain;
            if (!attn_block(t, c, g, group, sm, false, bar, 32 * group * sub)) {
                if ((threadIdx.x & 31) == 0)
                    tk_give_up(DEVERR_TIMEOUT_TAG);
                break;  // every warp of the item returned false together
            }
            named_bar_sync(bar, 32 * group);  // staging free before the next item
            t.trace = nullptr;
        }
    }
    tk_trace(p, 4);
}

__global__ void __launch_bounds__(TK_THREADS, 1) token_kernel(const __grid_constant__ TokenArgs a)
{
    const int nph = 5 * a.n_layers + 1;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    PhaseEnt* ptab = tk_ptab();
    KindEnt* ktab = tk_ktab();
    TkMisc& m = tk_misc();

    {  // the arguments to shared memory
        const int* src = reinterpret_cast<const int*>(&a);
        int* dst = reinterpret_cast<int*>(tk_smem + TK_OFF_ARGS);
        for (int i = tid; i < static_cast<int>(sizeof(TokenArgs) / 4); i += TK_THREADS)
            dst[i] = src[i];
    }
    if (tid < PH_KINDS) {
        const int qdim = a.n_q * a.hd, kvdim = a.n_kv * a.hd;
        const int q4h = a.hidden / 256 * Q4K_BYTES;
        KindEnt k{};
        k.nmat = 1;
        k.R = tk_rows_per_tile(tid);
        switch (tid) {
        case PH_QKV: k.rows = qdim + 2 * kvdim; k.K = a.hidden; k.row_bytes = q4h; break;
        case PH_ATTN: k.R = 1; break;
        case PH_O: k.rows = a.hidden; k.K = qdim; k.row_bytes = qdim / 256 * Q4K_BYTES; break;
        case PH_GATEUP: k.rows = a.ffn; k.K = a.hidden; k.row_bytes = q4h; k.nmat = 2; break;
        case PH_DOWN_Q4: k.rows = a.hidden; k.K = a.ffn; k.row_bytes = a.ffn / 256 * Q4K_BYTES; break;
        case PH_DOWN_Q6: k.rows = a.hidden; k.K = a.ffn; k.row_bytes = a.ffn / 256 * Q6K_BYTES; break;
        default: k.rows = a.vocab; k.K = a.hidden; k.row_bytes = a.hidden / 256 * Q6K_BYTES; break;
        }
        k.r0 = static_cast<int>(static_cast<long long>(blockIdx.x) * k.rows / gridDim.x);
        k.r1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * k.rows / gridDim.x);
        ktab[tid] = k;
    }
    __syncthreads();
    // phase table: kind, weights and this block's tile count, then a prefix sum
    for (int p = tid; p < nph; p += TK_THREADS) {
        PhaseEnt e{a.wvocab, nullptr, 0, PH_VOCAB};
        if (p < nph - 1) {
            const TokenLayer& ly = a.layers[p / 5];
            switch (p % 5) {
            case 0: e.kind = PH_QKV; e.W = ly.wqkv; break;
            case 1: e.kind = PH_ATTN; e.W = nullptr; break;
            case 2: e.kind = PH_O; e.W = ly.wo; break;
            case 3: e.kind = PH_GATEUP; e.W = ly.wgate; e.W2 = ly.wup; break;
            default: e.kind = ly.down_fmt == FMT_Q6K ? PH_DOWN_Q6 : PH_DOWN_Q4; e.W = ly.wdown; break;
            }
        }
        const KindEnt& k = ktab[e.kind];
        e.T0 = (k.r1 - k.r0 + k.R - 1) / k.R;
        ptab[p] = e;
    }
    __syncthreads();
    if (warp == 0) {
        int run = 0;
        for (int base = 0; base < nph; base += 32) {
            const int p = base + lane;
            const int v = p < nph ? ptab[p].T0 : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += u;
            }
            if (p < nph)
                ptab[p].T0 = run + incl - v;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            ptab[nph] = PhaseEnt{nullptr, nullptr, run, PH_VOCAB};
            m.ttotal = run;
        }
    }
    __syncthreads();
    int icur = 0;
    if (tid == 0) {
        for (int s = 0; s < TK_NSTAGE; ++s) {
            mbar_init(&m.full[s], 1);
            mbar_init(&m.empty[s], TK_WARPS);
        }
        fence_mbar_init();
        m.dead = 0;
        m.issued_hi = 0;
        m.last_out = 0;
        // written only by the previous launch's last block: the same value in every block
        m.tokseq = ld_relaxed_u32(a.bar + TB_TOKEN);
        m.tokpar = m.tokseq & 1u;
        for (int T = 0; T < min(TK_NSTAGE, m.ttotal); ++T)
            tk_issue(T, icur);
        if (blockIdx.x == 0) {
            a.step->pos = a.pos;
            a.step->logits = a.logits;
        }
    }
    __syncthreads();

    // The phases in token order: per layer a straight sequence (a loop over a
    // switch on the phase kind makes the register allocator keep every kind's
    // values live at once).
    int2 st = make_int2(0, icur);  // the block's next tile, this thread's issue cursor
#pragma unroll 1
    for (int l = 0; l < a.n_layers; ++l) {
        const int p = 5 * l;
        st = tk_gemv<PH_QKV, FMT_Q4K, 1, 1, EPI_QKV, true>(p, st.x, st.y);
        if (!a.fold)
            tk_attention(p + 1);
        st = tk_gemv<PH_O, FMT_Q4K, 1, 1, EPI_RESID, false>(p + 2, st.x, st.y);
        st = tk_gemv<PH_GATEUP, FMT_Q4K, 1, 2, EPI_SWIGLU, true>(p + 3, st.x, st.y);
        if (ptab[p + 4].kind == PH_DOWN_Q6)
            st = tk_gemv<PH_DOWN_Q6, FMT_Q6K, 1, 1, EPI_RESID, false>(p + 4, st.x, st.y);
        else
            st = tk_gemv<PH_DOWN_Q4, FMT_Q4K, 1, 1, EPI_RESID, false>(p + 4, st.x, st.y);
    }
    st = tk_gemv<PH_VOCAB, FMT_Q6K, 1, 1, EPI_STORE, true>(nph - 1, st.x, st.y);
    // A block that stopped early may still have copies in flight into its
    // shared memory: wait (bounded) for the last ring-full it issued.
    __syncthreads();
    if (tid == 0 && m.dead) {
        const int hi = m.issued_hi;
        for (int Tq = max(0, hi - TK_NSTAGE); Tq < hi; ++Tq) {
            const unsigned long long t0 = globaltimer_ns();
            while (!mbar_try_wait(&m.full[Tq & (TK_NSTAGE - 1)], (Tq / TK_NSTAGE) & 1))
                if (globaltimer_ns() - t0 > 100000000ull) {
                    set_error(a.err, DEVERR_TIMEOUT_DRAIN);
                    break;
                }
        }
    }
    // The last block to finish puts the launch-state area back for the next launch:
    // every block counts itself out only after its last wait and its last
    // write (dead blocks too), so nothing reads the counters or the tagged vectors
    // any more.  The exit count goes back to zero and the token count advances (the
    // tags of the next token follow from it), so a launch's arguments never
    // depend on host-side state.  After a wait ran out somewhere, writes may be
    // missing and the tags out of step: the tagged vectors and the token count go
    // back to zero instead, the state before the first token.
    if (tid == 0) {
        fence_acq_rel_gpu();
        m.last_out = atomicAdd(a.bar + TB_EXIT, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (m.last_out) {
        fence_acq_rel_gpu();
        const bool fault = ld_relaxed_u32(a.bar + TB_FAULT) != 0u;
        if (fault) {
            const int qdim = a.n_q * a.hd, kvdim = a.n_kv * a.hd;
            for (int i = tid; i < a.hidden; i += TK_THREADS)
                a.x[i] = 0.f;
            for (int i = tid; i < a.ffn; i += TK_THREADS)
                a.act[i] = 0.f;
            for (int i = tid; i < qdim; i += TK_THREADS) {
                a.q[i] = 0.f;
                a.attn[i] = 0.f;
            }
            for (int i = tid; i < kvdim; i += TK_THREADS) {
                a.k_new[i] = 0.f;
                a.v_new[i] = 0.f;
            }
            // the attention's chunk stamps: the token count restarts, so old stamps
            // could match a later token's
            for (int i = tid; i < a.n_kv * ATT_CHUNKS; i += TK_THREADS)
                a.stamps[i] = 0u;
        }
        __syncthreads();
        if (tid == 0) {
            const unsigned tok = ld_relaxed_u32(a.bar + TB_TOKEN);
            atomicExch(a.bar + TB_TOKEN, fault ? 0u : tok + 1u);
            atomicExch(a.bar + TB_FAULT, 0u);
            atomicExch(a.bar + TB_EXIT, 0u);
        }
    }
}

}  // namespace dq

namespace dqhost {

int plan_token(int n_layers, int hidden, int ffn, int n_q, int n_kv, int hd, bool any_q6_down, TokenPlan* plan)
{
    using namespace dq;
    const int qdim = n_q * hd;
    if (n_layers > TK_MAX_LAYERS || hidden > 32 * tk_p(PH_QKV) * tk_ul(PH_QKV) || qdim > 32 * tk_p(PH_O) * tk_ul(PH_O) ||
        hidden > 32 * tk_p(PH_GATEUP) * tk_ul(PH_GATEUP) || hidden > 32 * tk_p(PH_VOCAB) * tk_ul(PH_VOCAB) ||
        ffn > 32 * tk_p(PH_DOWN_Q4) * tk_ul(PH_DOWN_Q4) || hidden % 2048 || qdim % 256 || ffn % 256 || hd != ATT_HD || n_q % n_kv ||
        n_q / n_kv > 8)
        return DQ_ERR_UNSUPPORTED;
    if (any_q6_down && ffn % 2048)
        return DQ_ERR_UNSUPPORTED;
    // tiles fit a ring slot
    const int q4h = hidden / 256 * Q4K_BYTES, q4q = qdim / 256 * Q4K_BYTES;
    const int down_rb = ffn / 256 * (any_q6_down ? Q6K_BYTES : Q4K_BYTES);
    if (tk_rows_per_tile(PH_QKV) * q4h > TK_SLOT || tk_rows_per_tile(PH_O) * q4q > TK_SLOT ||
        2 * tk_rows_per_tile(PH_GATEUP) * q4h > TK_SLOT || tk_rows_per_tile(PH_DOWN_Q6) * down_rb > TK_SLOT ||
        tk_rows_per_tile(PH_VOCAB) * (hidden / 256 * Q6K_BYTES) > TK_SLOT)
        return DQ_ERR_UNSUPPORTED;
    const int grid = sm_count();
    if ((hidden + grid - 1) / grid + 1 > TK_RESID_MAX)
        return DQ_ERR_UNSUPPORTED;
    const int smem = tk_smem_bytes(hidden, qdim, ffn);
    if (smem > 227 * 1024)
        return DQ_ERR_UNSUPPORTED;
    const void* k = reinterpret_cast<const void*>(token_kernel);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return DQ_ERR_UNSUPPORTED;
    }
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, TK_THREADS, smem);
    if (e != cudaSuccess || per_sm < 1) {
        cudaGetLastError();
        return DQ_ERR_UNSUPPORTED;
    }
    plan->nph = 5 * n_layers + 1;
    plan->grid = grid;
    plan->smem_bytes = smem;
    plan->kernel = token_kernel;
    return DQ_OK;
}

cudaError_t launch_token(const TokenPlan& plan, const dq::TokenArgs& a, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(dq::TK_THREADS);
    cfg.dynamicSmemBytes = plan.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, plan.kernel, a);
}

}  // namespace dqhost
