// dq_token.cu -- one decode token as a single persistent kernel (sm_103a).
//
// The token is the chain of phases of the per-kernel path (per layer: norm +
// Q|K|V + cache append, attention, O + residual, norm + gate/up + SwiGLU,
// down + residual; then norm + vocabulary), run by one block per SM that stays
// resident for the whole token.  Phases are separated by grid barriers (every
// phase reads the whole output of the one before), but the weight stream is
// not: each block numbers the weight tiles of all its phases in one sequence
// and refills its ring slots in that order, so the tiles of the next phase are
// already in flight while the current phase finishes, the barrier resolves and
// the next activation is quantised.  That removes the per-kernel start-up and
// drain cost that dominates a chain of short launches ("The roofline holds on
// a second GPU", section "Hiding, fusing...": keep the bytes in flight across
// the whole token; "The Mountain Runs", section 3: one output per weight row).
//
// The consumers are those of the streaming GEMV kernel (dq_gemv.cuh): 512
// threads in four row groups of 128, each thread holding its slice of the
// quantised activation in registers; stage t is completed by warp t % 16 two
// stages later.  The attention phase runs one (key chunk, KV head) item per
// block on the first n_q / n_kv warps (dq_attn.cuh).
//
// Every wait is bounded.  A block whose wait runs out records the error, stops
// working and keeps arriving at the grid barriers without waiting, so the other
// blocks finish the token (with meaningless output) instead of hanging.
#include <algorithm>

#include "dq_token.cuh"

namespace dq {

constexpr int DEVERR_TIMEOUT_BARRIER = 16;

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// The block's shared memory (layout: dq_token.cuh).
extern __shared__ __align__(128) uint8_t tk_smem[];

struct TkMisc {
    float gred[NCONS_WARPS];   // norm partial sums
    uint64_t full[TK_NSTAGE];  // stage loaded
    uint64_t empty[TK_NSTAGE]; // stage released by all warps
    int dead;                  // a wait of this block ran out
    int issued_hi;             // one past the highest tile issued
    int sync_ok;
    int ttotal;                // the block's tiles over the token
    // Epilogue pointers of phase p in slot p & 1: thread 0 writes the next
    // phase's while warps may still complete the current phase's last tiles.
    float* y[2];               // output rows
    __half* kc[2];             // EPI_QKV: the layer's K and V planes
    __half* vc[2];
};
static_assert(sizeof(TkMisc) <= 256, "misc region");

__device__ __forceinline__ TkMisc& tk_misc() { return *reinterpret_cast<TkMisc*>(tk_smem + TK_OFF_MISC); }
__device__ __forceinline__ KindEnt* tk_ktab() { return reinterpret_cast<KindEnt*>(tk_smem + TK_OFF_KTAB); }
__device__ __forceinline__ float* tk_resid() { return reinterpret_cast<float*>(tk_smem + TK_OFF_RESID); }
__device__ __forceinline__ uint32_t* tk_xq() { return reinterpret_cast<uint32_t*>(tk_smem + TK_OFF_XQ); }
__device__ __forceinline__ float* tk_red() { return reinterpret_cast<float*>(tk_smem + TK_OFF_RED); }
template <int ULF>
__device__ __forceinline__ PhaseEnt* tk_ptab() { return reinterpret_cast<PhaseEnt*>(tk_smem + tk_off_ptab(ULF)); }

__device__ __forceinline__ int tk_row0(int rows) { return static_cast<int>(static_cast<long long>(blockIdx.x) * rows / gridDim.x); }
__device__ __forceinline__ int tk_row1(int rows) { return static_cast<int>(static_cast<long long>(blockIdx.x + 1) * rows / gridDim.x); }

// Stream tile T (numbered over the token) into its ring slot.  `cur` is the
// calling thread's cursor into the phase table (each thread issues tiles in
// increasing order, so it only moves forward).
template <int ULF>
__device__ __forceinline__ void tk_issue(int T, int& cur)
{
    const PhaseEnt* ptab = tk_ptab<ULF>();
    while (T >= ptab[cur + 1].T0)
        ++cur;
    const PhaseEnt& e = ptab[cur];
    const KindEnt& k = tk_ktab()[e.kind];
    const int r0 = tk_row0(k.rows), r1 = tk_row1(k.rows);
    const int row = r0 + (T - e.T0) * k.R;
    const int nr = min(k.R, r1 - row);
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

// Grid barrier on a monotonic arrival counter: the block arrives, then waits
// until the counter reaches `target` (all gridDim.x blocks have arrived as
// often as this one).  A dead block arrives without waiting.  Returns false
// when the block is (or has just become) dead.
__device__ __forceinline__ bool tk_sync(const TokenArgs& a, unsigned target)
{
    TkMisc& m = tk_misc();
    __syncthreads();  // the block's phase outputs are written
    if (threadIdx.x == 0) {
        int ok = *reinterpret_cast<volatile int*>(&m.dead) == 0;
        red_release_add(a.bar, 1u);  // release, cumulative over the block's writes through bar.sync
        if (ok && static_cast<int>(ld_acquire_u32(a.bar) - target) < 0) {
            const unsigned long long t0 = globaltimer_ns();
            while (static_cast<int>(ld_acquire_u32(a.bar) - target) < 0) {
                if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
                    set_error(a.err, DEVERR_TIMEOUT_BARRIER);
                    m.dead = 1;
                    ok = 0;
                    break;
                }
            }
        }
        m.sync_ok = ok;
    }
    __syncthreads();
    return m.sync_ok != 0;
}

__device__ __forceinline__ void tk_trace(const TokenArgs& a, int nph, int p, int i)
{
    if (a.trace && threadIdx.x == 0)
        a.trace[(static_cast<size_t>(blockIdx.x) * nph + p) * 4 + i] = globaltimer_ns();
}

// Epilogue of one output row r (value v0, and v1 of the second matrix).
template <int EPI>
__device__ __forceinline__ void tk_epilogue(const TokenArgs& a, int slot, int r, int r0, float v0, float v1)
{
    const TkMisc& m = tk_misc();
    float* y = m.y[slot];
    if (EPI == EPI_STORE) {
        y[r] = v0;
    } else if (EPI == EPI_RESID) {
        y[r] = tk_resid()[r - r0] + v0;
    } else if (EPI == EPI_SWIGLU) {
        y[r] = v0 / (1.0f + expf(-v0)) * v1;
    } else {  // EPI_QKV: q rows, then k and v rows appended to the cache at pos
        const int qdim = a.n_q * a.hd, kvdim = a.n_kv * a.hd;
        if (r < qdim) {
            y[r] = v0;
        } else {
            const int idx = r - qdim;
            const int which = idx / kvdim, rem = idx - which * kvdim;
            const int kvh = rem / a.hd, dd = rem - kvh * a.hd;
            __half* plane = which ? m.vc[slot] : m.kc[slot];
            plane[(static_cast<size_t>(kvh) * a.max_ctx + a.pos) * a.hd + dd] = __float2half_rn(v0);
        }
    }
}

// One matrix phase: prefetch the norm weight, pass the barrier, quantise the
// activation, consume the phase's tiles and complete them (refill + epilogue).
template <int ULF, int KIND, int FMT, int PL, int UL, int NMAT, int EPI, bool NORM>
__device__ __forceinline__ void tk_gemv(const TokenArgs& a, int nph, int p, bool barrier, unsigned target,
                                        const float* x, const float* gamma, const float* rsrc, int& T, int& icur)
{
    constexpr int RP = tk_rpt(KIND);  // rows per thread and matrix
    constexpr int R = TK_RG * RP;     // rows per tile and matrix
    constexpr int NCH = 2 * UL;       // 4-element activation chunks per thread: K <= 4096 UL
    static_assert(RP * NMAT <= TK_RED_STRIDE, "partial sums per warp");
    const KindEnt& ke = tk_ktab()[KIND];
    const int K = ke.K;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const PhaseEnt* ptab = tk_ptab<ULF>();
    const int T0 = ptab[p].T0, ntiles = ptab[p + 1].T0 - T0;
    const int r0 = tk_row0(ke.rows), r1 = tk_row1(ke.rows);
    TkMisc& m = tk_misc();

    tk_trace(a, nph, p, 0);
    float4 gv[NCH];
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
        const int ch = tid + NCONS * i;
        gv[i] = make_float4(1.f, 1.f, 1.f, 1.f);
        if (NORM && ch < K / 4)
            gv[i] = __ldg(reinterpret_cast<const float4*>(gamma) + ch);
    }
    if (barrier ? !tk_sync(a, target) : m.dead != 0)
        return;
    tk_trace(a, nph, p, 1);

    float4 xv[NCH];
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
        const int ch = tid + NCONS * i;
        xv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (ch < K / 4)
            xv[i] = __ldcg(reinterpret_cast<const float4*>(x) + ch);
    }
    if (EPI == EPI_RESID)
        for (int r = tid; r < r1 - r0; r += NCONS)
            tk_resid()[r] = __ldcg(rsrc + r0 + r);
    float ss = quantise_block<FMT, PL, NCH>(xv, gv, NORM, tk_xq(), K, tid);
    if (NORM) {
        ss = warp_sum(ss);
        if (lane == 0)
            m.gred[warp] = ss;
    }
    __syncthreads();  // quantised activation, residual rows and norm partials complete
    float rstd = 1.f;
    if (NORM) {
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < NCONS_WARPS; ++w)
            tot += m.gred[w];
        rstd = 1.0f / sqrtf(tot / static_cast<float>(K) + a.eps);
    }
    const int g = tid / TK_P, pp = tid % TK_P;
    UnitState<FMT, PL> us[UL];
    bool have[UL];
#pragma unroll
    for (int k = 0; k < UL; ++k)
        have[k] = (pp + TK_P * k) < K / 32;
    load_units<FMT, PL, UL>(us, have, tk_xq(), pp, TK_P, rstd);
    tk_trace(a, nph, p, 2);

    // Complete tile tc (token tile Tc): wait until every warp released it,
    // refill its slot with tile Tc + TK_NSTAGE, run the epilogue of its rows.
    auto complete = [&](int tc, int Tc) -> bool {
        const int sc = Tc & (TK_NSTAGE - 1);
        if (!mbar_wait(&m.empty[sc], (Tc / TK_NSTAGE) & 1)) {
            set_error(a.err, DEVERR_TIMEOUT_EMPTY);
            return false;
        }
        if (lane == 0 && Tc + TK_NSTAGE < m.ttotal)
            tk_issue<ULF>(Tc + TK_NSTAGE, icur);
        const float* rb = tk_red() + (Tc & (2 * TK_NSTAGE - 1)) * NCONS_WARPS * TK_RED_STRIDE;
        const int row0 = r0 + tc * R;
        const int nr = min(R, r1 - row0);
        for (int row = lane; row < nr; row += 32) {
            const int rg = row % TK_RG, i = row / TK_RG;
            const float* wb = rb + rg * (TK_P / 32) * TK_RED_STRIDE;
            float v0 = 0.f, v1 = 0.f;
#pragma unroll
            for (int w = 0; w < TK_P / 32; ++w) {
                v0 += wb[w * TK_RED_STRIDE + i];
                if (NMAT == 2)
                    v1 += wb[w * TK_RED_STRIDE + RP + i];
            }
            tk_epilogue<EPI>(a, p & 1, row0 + row, r0, v0, v1);
        }
        return true;
    };

    bool ok = true;
    for (int t = 0; t < ntiles; ++t, ++T) {
        const int s = T & (TK_NSTAGE - 1);
        if (!mbar_wait(&m.full[s], (T / TK_NSTAGE) & 1)) {
            set_error(a.err, DEVERR_TIMEOUT_FULL);
            ok = false;
            break;
        }
        const int nr = min(R, r1 - (r0 + t * R));
        consume_tile<FMT, PL, UL, RP, NMAT>(
            tk_smem + s * TK_SLOT, nr, R, TK_RG, g, pp, TK_P, ke.row_bytes, us, have,
            tk_red() + ((T & (2 * TK_NSTAGE - 1)) * NCONS_WARPS + warp) * TK_RED_STRIDE, lane);
        if (lane == 0)
            mbar_arrive(&m.empty[s]);
        if (t >= TK_DEFER && ((T - TK_DEFER) & (NCONS_WARPS - 1)) == warp && !complete(t - TK_DEFER, T - TK_DEFER)) {
            ok = false;
            break;
        }
    }
    if (ok)
        for (int tc = max(0, ntiles - TK_DEFER); tc < ntiles; ++tc)
            if (((T0 + tc) & (NCONS_WARPS - 1)) == warp && !complete(tc, T0 + tc)) {
                ok = false;
                break;
            }
    if (!ok)
        m.dead = 1;
    tk_trace(a, nph, p, 3);
}

// Attention phase: items (key chunk, KV head) spread over the blocks.
__device__ __forceinline__ void tk_attention(const TokenArgs& a, int nph, int p, int l, unsigned target)
{
    tk_trace(a, nph, p, 0);
    if (!tk_sync(a, target))
        return;
    tk_trace(a, nph, p, 1);
    const int group = a.n_q / a.n_kv;
    if ((threadIdx.x >> 5) < group) {
        const size_t plane = static_cast<size_t>(a.n_kv) * a.max_ctx * a.hd;
        AttnArgs t;
        t.q = a.q;
        t.kc = a.kv + static_cast<size_t>(l) * 2 * plane;
        t.vc = t.kc + plane;
        t.out = a.attn;
        t.part = a.part;
        t.counters = a.counters;
        t.n_q = a.n_q;
        t.n_kv = a.n_kv;
        t.max_ctx = a.max_ctx;
        t.n_keys = a.pos + 1;
        t.step = nullptr;
        t.err = a.err;
        const int n_keys = a.pos + 1;
        const int L = max((n_keys + ATT_CHUNKS - 1) / ATT_CHUNKS, ATT_MIN_CHUNK);
        const int nact = (n_keys + L - 1) / L;
        AttnSmem& sm = *reinterpret_cast<AttnSmem*>(tk_xq());
        for (int item = blockIdx.x; item < nact * a.n_kv; item += gridDim.x) {
            attn_block(t, item % nact, item / nact, group, sm, false);
            named_bar_sync(ATT_BAR, 32 * group);  // staging free before the next item
        }
    }
    tk_trace(a, nph, p, 3);
}

template <int ULF>
__global__ void __launch_bounds__(NCONS, 1) token_kernel(const __grid_constant__ TokenArgs a)
{
    const int nph = 5 * a.n_layers + 1;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = gridDim.x;
    PhaseEnt* ptab = tk_ptab<ULF>();
    KindEnt* ktab = tk_ktab();
    TkMisc& m = tk_misc();

    if (tid < PH_KINDS) {
        const int qdim = a.n_q * a.hd, kvdim = a.n_kv * a.hd;
        const int q4h = a.hidden / 256 * Q4K_BYTES;
        KindEnt k{};
        k.nmat = 1;
        k.R = TK_RG * tk_rpt(tid);
        switch (tid) {
        case PH_QKV: k.rows = qdim + 2 * kvdim; k.K = a.hidden; k.row_bytes = q4h; break;
        case PH_ATTN: k.R = 1; break;
        case PH_O: k.rows = a.hidden; k.K = qdim; k.row_bytes = qdim / 256 * Q4K_BYTES; break;
        case PH_GATEUP: k.rows = a.ffn; k.K = a.hidden; k.row_bytes = q4h; k.nmat = 2; break;
        case PH_DOWN_Q4: k.rows = a.hidden; k.K = a.ffn; k.row_bytes = a.ffn / 256 * Q4K_BYTES; break;
        case PH_DOWN_Q6: k.rows = a.hidden; k.K = a.ffn; k.row_bytes = a.ffn / 256 * Q6K_BYTES; break;
        default: k.rows = a.vocab; k.K = a.hidden; k.row_bytes = a.hidden / 256 * Q6K_BYTES; break;
        }
        ktab[tid] = k;
    }
    __syncthreads();
    // phase table: kind, weights and this block's tile count, then a prefix sum
    for (int p = tid; p < nph; p += NCONS) {
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
        e.T0 = (tk_row1(k.rows) - tk_row0(k.rows) + k.R - 1) / k.R;
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
            mbar_init(&m.empty[s], NCONS_WARPS);
        }
        fence_mbar_init();
        m.dead = 0;
        m.issued_hi = 0;
        for (int T = 0; T < min(TK_NSTAGE, m.ttotal); ++T)
            tk_issue<ULF>(T, icur);
        if (blockIdx.x == 0) {
            a.step->pos = a.pos;
            a.step->logits = a.logits;
        }
    }
    __syncthreads();

    int T = 0;
    unsigned target = a.bar_base;
    const size_t plane = static_cast<size_t>(a.n_kv) * a.max_ctx * a.hd;
    for (int p = 0; p < nph; ++p) {
        const int l = p / 5;
        const bool barrier = p > 0;
        if (barrier)
            target += static_cast<unsigned>(G);
        const int kind = ptab[p].kind;
        // the epilogue's pointers: written before the phase's barrier, read after it
        if (tid == 0) {
            m.y[p & 1] = kind == PH_QKV ? a.q : kind == PH_GATEUP ? a.act : kind == PH_VOCAB ? a.logits : a.x;
            m.kc[p & 1] = a.kv + static_cast<size_t>(l) * 2 * plane;
            m.vc[p & 1] = m.kc[p & 1] + plane;
        }
        const float* x0 = l == 0 ? a.x_in : a.x;  // the residual stream entering layer l
        switch (kind) {
        case PH_QKV:
            tk_gemv<ULF, PH_QKV, FMT_Q4K, 2, 1, 1, EPI_QKV, true>(a, nph, p, barrier, target, x0,
                                                                  a.layers[l].attn_norm, nullptr, T, icur);
            break;
        case PH_ATTN:
            tk_attention(a, nph, p, l, target);
            break;
        case PH_O:
            tk_gemv<ULF, PH_O, FMT_Q4K, 2, 1, 1, EPI_RESID, false>(a, nph, p, barrier, target, a.attn, nullptr, x0, T,
                                                                   icur);
            break;
        case PH_GATEUP:
            tk_gemv<ULF, PH_GATEUP, FMT_Q4K, 1, 1, 2, EPI_SWIGLU, true>(a, nph, p, barrier, target, a.x,
                                                                        a.layers[l].ffn_norm, nullptr, T, icur);
            break;
        case PH_DOWN_Q4:
            tk_gemv<ULF, PH_DOWN_Q4, FMT_Q4K, 1, ULF, 1, EPI_RESID, false>(a, nph, p, barrier, target, a.act, nullptr,
                                                                           a.x, T, icur);
            break;
        case PH_DOWN_Q6:
            tk_gemv<ULF, PH_DOWN_Q6, FMT_Q6K, 1, ULF, 1, EPI_RESID, false>(a, nph, p, barrier, target, a.act, nullptr,
                                                                           a.x, T, icur);
            break;
        default:
            tk_gemv<ULF, PH_VOCAB, FMT_Q6K, 1, 1, 1, EPI_STORE, true>(a, nph, p, barrier, target, a.x, a.out_norm,
                                                                      nullptr, T, icur);
            break;
        }
    }
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
}

}  // namespace dq

namespace dqhost {

static TokenKernel token_kernel_for(int ulf)
{
    switch (ulf) {
    case 1: return dq::token_kernel<1>;
    case 3: return dq::token_kernel<3>;
    default: return nullptr;
    }
}

int plan_token(int n_layers, int hidden, int ffn, int n_q, int n_kv, int hd, bool any_q6_down, TokenPlan* plan)
{
    using namespace dq;
    const int qdim = n_q * hd;
    if (hidden > TK_P * 32 || qdim > TK_P * 32 || hidden % 2048 || qdim % 256 || ffn % 256 || hd != ATT_HD ||
        n_q % n_kv || n_q / n_kv > 8)
        return DQ_ERR_UNSUPPORTED;
    if (any_q6_down && ffn % 2048)
        return DQ_ERR_UNSUPPORTED;
    const int ulf = (ffn + TK_P * 32 - 1) / (TK_P * 32);
    TokenKernel k = token_kernel_for(ulf);
    if (!k)
        return DQ_ERR_UNSUPPORTED;
    // tiles fit a ring slot
    const int q4h = hidden / 256 * Q4K_BYTES, q4q = qdim / 256 * Q4K_BYTES;
    const int down_rb = ffn / 256 * (any_q6_down ? Q6K_BYTES : Q4K_BYTES);
    if (TK_RG * tk_rpt(PH_QKV) * q4h > TK_SLOT || TK_RG * tk_rpt(PH_O) * q4q > TK_SLOT ||
        2 * TK_RG * tk_rpt(PH_GATEUP) * q4h > TK_SLOT || TK_RG * tk_rpt(PH_DOWN_Q6) * down_rb > TK_SLOT ||
        TK_RG * tk_rpt(PH_VOCAB) * (hidden / 256 * Q6K_BYTES) > TK_SLOT)
        return DQ_ERR_UNSUPPORTED;
    const int grid = sm_count();
    if ((hidden + grid - 1) / grid + 1 > TK_RESID_MAX)
        return DQ_ERR_UNSUPPORTED;
    const int nph = 5 * n_layers + 1;
    const int smem = tk_smem_bytes(ulf, nph);
    if (smem > 227 * 1024)
        return DQ_ERR_UNSUPPORTED;
    cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(k), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return DQ_ERR_UNSUPPORTED;
    }
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reinterpret_cast<const void*>(k), NCONS, smem);
    if (e != cudaSuccess || per_sm < 1) {
        cudaGetLastError();
        return DQ_ERR_UNSUPPORTED;
    }
    plan->ulf = ulf;
    plan->nph = nph;
    plan->grid = grid;
    plan->smem_bytes = smem;
    plan->kernel = k;
    return DQ_OK;
}

cudaError_t launch_token(const TokenPlan& plan, const dq::TokenArgs& a, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(dq::NCONS);
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
