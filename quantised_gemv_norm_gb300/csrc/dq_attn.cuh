// dq_attn.cuh -- arguments and launcher of the grouped-query decode attention.
#pragma once

#include "dq_gemv.cuh"

namespace dq {

constexpr int ATT_HD = 128;      // head dimension the kernel is written for (4 dims per lane)
constexpr int ATT_CHUNKS = 32;   // key chunks per KV head at most (thread blocks per KV head)
constexpr int ATT_BATCH = 32;    // keys staged in shared memory at a time (one per lane)
constexpr int ATT_MIN_CHUNK = 32; // fewest keys per block (one staging batch)
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
    // Qwen3 attention (k_new not null): q and this token's key are normalised
    // per head and rotated before use; the key is written to kc at n_keys - 1.
    const float* k_new;    // [n_kv][128] the token's keys as projected (fp32)
    const float* q_norm;   // [128] RMSNorm weight shared by the query heads
    const float* k_norm;   // [128] RMSNorm weight shared by the key heads
    const float2* rope;    // [max_ctx][64] (cos, sin) of pos / theta^(2i / 128)
    float eps;
    // Tagged mode (the fused token kernel; tag = 1 + parity): q, k_new and v_new carry
    // the write parity in their lowest mantissa bit and are re-read until they do;
    // the block whose chunk holds the token's position writes that position's fp16
    // key and value rows into the cache from k_new (the Qwen3 key, or the key's fp16
    // value) and v_new (the value's fp16 value); the output is stored with the same
    // tag; the chunks meet through `stamps`, not the merge counters.  tag = 0 (a
    // zero-initialised AttnArgs): the plain mode.
    int tag;
    const float* v_new;            // [n_kv][128] tagged mode
    unsigned long long wait_ns;    // tagged mode: bound on the tag waits
    // Tagged mode with more than one chunk: every chunk but the last stores its
    // partial and then, with release semantics, `seq` into stamps[g][c]; the
    // block of the last chunk (the one holding the token's position) merges once
    // it has acquired every other chunk's stamp.  seq is unique per layer and token
    // (a stale stamp never matches), so nothing is reset between calls.
    unsigned* stamps;              // [n_kv][ATT_CHUNKS]
    unsigned seq;
    // diagnostics (the fused token kernel's trace): when not null, the item's first
    // thread records global-timer ns at [1] q ready, [3] keys staged, [5] partial
    // computed, [6] merge decided, [7] output stored
    unsigned long long* trace;
};

#ifndef ATT_KV_EF
#define ATT_KV_EF 1
#endif
// The cache rows are read once a token: as L2 evict-first, so they do not push the
// vectors the phases hand on out of L2 (512 keys in the fused token: 677.4 -> 680.9
// tokens/s).
__device__ __forceinline__ void att_cp_kv16(void* dst, const void* src, uint64_t pol)
{
    if (ATT_KV_EF)
        asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
                     "l"(pol)
                     : "memory");
    else
        cp_async16(dst, src);
}
__device__ __forceinline__ uint4 att_ld_kv16(const void* src, uint64_t pol)
{
    if (!ATT_KV_EF)
        return __ldcg(reinterpret_cast<const uint4*>(src));
    uint4 v;
    asm volatile("ld.global.cg.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(src), "l"(pol));
    return v;
}

__device__ __forceinline__ void att_st_release(unsigned* p, unsigned v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned att_ld_acquire(const unsigned* p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void att_stamp(const AttnArgs& a, int i, int tid)
{
    if (a.trace && tid == 0)
        a.trace[i] = globaltimer_ns();
}

__device__ __forceinline__ float4 att_ld_relaxed_f4(const float* p)
{
    float4 v;
    asm volatile("ld.relaxed.gpu.global.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

__device__ __forceinline__ bool att_tags_ok(float4 v, uint32_t par)
{
    const uint32_t x = __float_as_uint(v.x) ^ par, y = __float_as_uint(v.y) ^ par, z = __float_as_uint(v.z) ^ par,
                   w = __float_as_uint(v.w) ^ par;
    return ((x | y | z | w) & 1u) == 0u;
}

// Load a float4 of a tagged vector, re-reading until its tags show `par`; the
// loop is warp-uniform.  False when `limit_ns` ran out.
__device__ __forceinline__ bool att_load_tagged(float4& v, const float* p, uint32_t par, unsigned long long limit_ns)
{
    v = att_ld_relaxed_f4(p);
    unsigned long long t0 = 0;
    while (!__all_sync(0xffffffffu, att_tags_ok(v, par))) {
        const unsigned long long now = globaltimer_ns();
        if (t0 == 0)
            t0 = now;
        else if (__any_sync(0xffffffffu, now - t0 > limit_ns))
            return false;
        if (!att_tags_ok(v, par))
            v = att_ld_relaxed_f4(p);
    }
    return true;
}

__device__ __forceinline__ float att_tagged(float v, uint32_t par)
{
    return __uint_as_float((__float_as_uint(v) & ~1u) | par);
}

__device__ __forceinline__ void att_st_out(float* p, float4 v, int tag)
{
    if (tag == 0) {
        *reinterpret_cast<float4*>(p) = v;
    } else {
        const uint32_t par = static_cast<uint32_t>(tag - 1) & 1u;
        asm volatile("st.relaxed.gpu.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(att_tagged(v.x, par)),
                     "f"(att_tagged(v.y, par)), "f"(att_tagged(v.z, par)), "f"(att_tagged(v.w, par))
                     : "memory");
    }
}

constexpr int ATT_BAR = 15;  // named barrier id of the attention warps

struct AttnSmem {
    __half ks[ATT_BATCH][ATT_HD + 8];  // rows padded by 16 bytes: lane j reads key j conflict-free
    __half vs[ATT_BATCH][ATT_HD];
    float qs[8][ATT_HD];
    int last;
};

// RMSNorm of one 128-dim head (4 dims per lane, weight w) followed by the
// rotate-half rotary embedding: dims i and i + 64 turn by the angle whose
// (cos, sin) is cs[i].  These are the Qwen3 family's attention inputs (the
// decode census of "The roofline holds on a second GPU" names the model, not
// these transforms): one weight vector for all query heads, one for all key
// heads, rotary base 1e6.
// The per-lane operands of head_norm_rope, loaded together ahead of use: the
// weight's 4 dims and the (cos, sin) of the lane's 4 rotation pairs.
struct NormRope {
    float4 w, c01, c23;
};

__device__ __forceinline__ NormRope load_norm_rope(const float* __restrict__ w, const float2* __restrict__ cs, int lane)
{
    const int i0 = (4 * lane) & (ATT_HD / 2 - 1);
    NormRope r;
    r.w = __ldg(reinterpret_cast<const float4*>(w) + lane);
    r.c01 = __ldg(reinterpret_cast<const float4*>(cs + i0));
    r.c23 = __ldg(reinterpret_cast<const float4*>(cs + i0 + 2));
    return r;
}

__device__ __forceinline__ float4 head_norm_rope(float4 v, const NormRope& nr, float eps, int lane)
{
    const float ss = warp_sum(v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w);
    const float r = rsqrtf(ss * (1.0f / ATT_HD) + eps);
    const float4 g = nr.w;
    v = make_float4(v.x * r * g.x, v.y * r * g.y, v.z * r * g.z, v.w * r * g.w);
    // the partner dims (i + 64 for the first half, i - 64 for the second) sit 16 lanes away
    float4 o;
    o.x = __shfl_xor_sync(0xffffffffu, v.x, 16);
    o.y = __shfl_xor_sync(0xffffffffu, v.y, 16);
    o.z = __shfl_xor_sync(0xffffffffu, v.z, 16);
    o.w = __shfl_xor_sync(0xffffffffu, v.w, 16);
    const float4 c01 = nr.c01, c23 = nr.c23;
    const float sg = lane < 16 ? -1.0f : 1.0f;  // first half: a cos - b sin; second: b cos + a sin
    return make_float4(fmaf(v.x, c01.x, sg * o.x * c01.y), fmaf(v.y, c01.z, sg * o.y * c01.w),
                       fmaf(v.z, c23.x, sg * o.z * c23.y), fmaf(v.w, c23.z, sg * o.w * c23.w));
}

// Block (c, g) of the decode attention, run by `group` warps of the calling
// block (threads tbase .. tbase + 32 group - 1, synchronised by named barrier
// bar), with `sm` (AttnSmem) as shared staging.  Used by the standalone kernel
// and by the fused token kernel (two items at a time there, tagged mode).
// Returns false when a tagged-mode wait ran out (nothing further is written).
__device__ __forceinline__ bool attn_block(const AttnArgs& a, int c, int g, int group, AttnSmem& sm, bool pdl,
                                           int bar = ATT_BAR, int tbase = 0)
{
    auto& ks = sm.ks;
    auto& vs = sm.vs;
    auto& qs = sm.qs;
    const int tid = threadIdx.x - tbase, warp = tid >> 5, lane = tid & 31;
    const int nthr = 32 * group;
    // step->pos was written before the token's first kernel: safe before the wait
    const int n_keys = a.step ? a.step->pos + 1 : a.n_keys;
    // chunks of at least ATT_MIN_CHUNK keys: short contexts take one block per KV head
    const int L = max((n_keys + ATT_CHUNKS - 1) / ATT_CHUNKS, ATT_MIN_CHUNK);
    const int j0 = c * L, j1 = min(n_keys, j0 + L);
    const int nact = (n_keys + L - 1) / L;
    if (pdl)
        pdl_wait();
    if (n_keys < 1 || n_keys > a.max_ctx) {
        if (tid == 0 && c == 0)
            set_error(a.err, DEVERR_BAD_ARG);
        return true;
    }
    if (j0 >= n_keys)
        return true;

    const int h = g * group + warp;
    const bool tagged = a.tag != 0;
    const uint32_t par = static_cast<uint32_t>(a.tag - 1) & 1u;
    const __half* kbase = a.kc + static_cast<size_t>(g) * a.max_ctx * ATT_HD;
    const __half* vbase = a.vc + static_cast<size_t>(g) * a.max_ctx * ATT_HD;
    const int pos = n_keys - 1;
    const uint64_t kvpol = ATT_KV_EF ? l2_evict_first_policy() : 0ull;
    bool ok = true;  // tagged mode: every wait of this thread ended in time
    if (tagged) {
        // the first batch's cache rows of earlier positions (earlier tokens wrote them)
        // go to shared memory while q is awaited; the position's own row comes from
        // the tagged key and value below
        const int nb = min(ATT_BATCH, j1 - j0);
        for (int idx = tid; idx < nb * (ATT_HD / 8); idx += nthr) {
            const int j = idx >> 4, ch = idx & 15;
            if (j0 + j == pos)
                continue;
            att_cp_kv16(&ks[j][8 * ch], kbase + static_cast<size_t>(j0 + j) * ATT_HD + 8 * ch, kvpol);
            att_cp_kv16(&vs[j][8 * ch], vbase + static_cast<size_t>(j0 + j) * ATT_HD + 8 * ch, kvpol);
        }
        cp_async_commit();
    }
    {
        float4 v;
        if (tagged)
            ok = att_load_tagged(v, a.q + static_cast<size_t>(h) * ATT_HD + 4 * lane, par, a.wait_ns);
        else
            v = __ldcg(reinterpret_cast<const float4*>(a.q + static_cast<size_t>(h) * ATT_HD) + lane);
        const float2* cs = a.rope + static_cast<size_t>(pos) * (ATT_HD / 2);
        if (c == nact - 1 && warp == 0 && (a.k_new || tagged)) {
            // the block whose chunk holds pos writes that position's key (the Qwen3 key
            // normalised and rotated) -- and in tagged mode its value -- before staging
            // them (the batch loop's first barrier orders the stores)
            float4 k = make_float4(0.f, 0.f, 0.f, 0.f), vv = k;
            if (tagged) {
                ok = att_load_tagged(k, a.k_new + static_cast<size_t>(g) * ATT_HD + 4 * lane, par, a.wait_ns) && ok;
                ok = att_load_tagged(vv, a.v_new + static_cast<size_t>(g) * ATT_HD + 4 * lane, par, a.wait_ns) && ok;
            } else {
                k = __ldcg(reinterpret_cast<const float4*>(a.k_new + static_cast<size_t>(g) * ATT_HD) + lane);
            }
            if (a.q_norm)  // Qwen3 inputs
                k = head_norm_rope(k, load_norm_rope(a.k_norm, cs, lane), a.eps, lane);
            const __half2 k01 = __floats2half2_rn(k.x, k.y), k23 = __floats2half2_rn(k.z, k.w);
            uint2 u;
            u.x = *reinterpret_cast<const uint32_t*>(&k01);
            u.y = *reinterpret_cast<const uint32_t*>(&k23);
            *reinterpret_cast<uint2*>(const_cast<__half*>(kbase) + static_cast<size_t>(pos) * ATT_HD + 4 * lane) = u;
            if (tagged) {
                const __half2 v01 = __floats2half2_rn(vv.x, vv.y), v23 = __floats2half2_rn(vv.z, vv.w);
                uint2 w;
                w.x = *reinterpret_cast<const uint32_t*>(&v01);
                w.y = *reinterpret_cast<const uint32_t*>(&v23);
                *reinterpret_cast<uint2*>(const_cast<__half*>(vbase) + static_cast<size_t>(pos) * ATT_HD + 4 * lane) = w;
                if (pos - j0 < ATT_BATCH) {  // the row is in the first batch: stage it from here
                    *reinterpret_cast<uint2*>(&ks[pos - j0][4 * lane]) = u;
                    *reinterpret_cast<uint2*>(&vs[pos - j0][4 * lane]) = w;
                }
            }
            __threadfence_block();
        }
        if (a.q_norm)
            v = head_norm_rope(v, load_norm_rope(a.q_norm, cs, lane), a.eps, lane);
        *reinterpret_cast<float4*>(&qs[warp][4 * lane]) = v;
    }
    att_stamp(a, 1, tid);
    const float scale = 0.08838834764831845f;  // 1 / sqrt(128)

    float m = -INFINITY, l = 0.f;
    float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
    for (int jb = j0; jb < j1; jb += ATT_BATCH) {
        const int nb = min(ATT_BATCH, j1 - jb);
        // previous batch fully consumed (and qs written on the first); on the first, in
        // tagged mode, the item's warps also learn together whether any wait ran out
        if (tagged && jb == j0) {
            cp_async_wait_all();  // this thread's staged rows landed
            if (named_bar_red_or(bar, nthr, !ok))
                return false;
        } else {
            named_bar_sync(bar, nthr);
        }
        for (int idx = tid; idx < nb * (ATT_HD / 8) && !(tagged && jb == j0); idx += nthr) {
            const int j = idx >> 4, ch = idx & 15;
            const uint4 kv = att_ld_kv16(kbase + static_cast<size_t>(jb + j) * ATT_HD + 8 * ch, kvpol);
            const uint4 vv = att_ld_kv16(vbase + static_cast<size_t>(jb + j) * ATT_HD + 8 * ch, kvpol);
            *reinterpret_cast<uint4*>(&ks[j][8 * ch]) = kv;
            *reinterpret_cast<uint4*>(&vs[j][8 * ch]) = vv;
        }
        named_bar_sync(bar, nthr);
        if (jb == j0)
            att_stamp(a, 3, tid);
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

    att_stamp(a, 5, tid);
    if (nact == 1) {  // the only block of this KV head: normalise and write directly
        const float inv = 1.0f / l;
        att_st_out(a.out + static_cast<size_t>(h) * ATT_HD + 4 * lane, make_float4(o0 * inv, o1 * inv, o2 * inv, o3 * inv),
                   a.tag);
        return true;
    }
    float* pp = a.part + (static_cast<size_t>(h) * ATT_CHUNKS + c) * ATT_PART;
    const float* hp = a.part + static_cast<size_t>(h) * ATT_CHUNKS * ATT_PART;
    // the chunks whose partials the merge loads: all of them, or in tagged mode all
    // but the merging (last) chunk, whose partial stays in registers
    int nload = nact;
    if (tagged) {
        if (c != nact - 1) {
            if (lane == 0) {
                pp[0] = m;
                pp[1] = l;
            }
            *reinterpret_cast<float4*>(pp + 4 + 4 * lane) = make_float4(o0, o1, o2, o3);
            named_bar_sync(bar, nthr);  // the item's partial stores come before the stamp
            if (tid == 0)
                att_st_release(a.stamps + g * ATT_CHUNKS + c, a.seq);
            att_stamp(a, 6, tid);
            return true;
        }
        nload = nact - 1;
        // wait for the other chunks' stamps (lane cc takes chunk cc); the warp
        // barrier passes each lane's acquire on to the loads of all lanes
        const unsigned* st = a.stamps + g * ATT_CHUNKS;
        bool mine = lane >= nload || att_ld_acquire(st + lane) == a.seq;
        unsigned long long t0 = 0;
        while (!__all_sync(0xffffffffu, mine)) {
            const unsigned long long now = globaltimer_ns();
            if (t0 == 0)
                t0 = now;
            else if (__any_sync(0xffffffffu, now - t0 > a.wait_ns))
                return false;
            if (!mine)
                mine = att_ld_acquire(st + lane) == a.seq;
        }
        __syncwarp();
        att_stamp(a, 6, tid);
    } else {
        if (lane == 0) {
            pp[0] = m;
            pp[1] = l;
        }
        *reinterpret_cast<float4*>(pp + 4 + 4 * lane) = make_float4(o0, o1, o2, o3);
        __threadfence();
        named_bar_sync(bar, nthr);
        if (tid == 0)
            sm.last = (atomicAdd(&a.counters[g], 1) == nact - 1);
        named_bar_sync(bar, nthr);
        att_stamp(a, 6, tid);
        if (!sm.last)
            return true;
        __threadfence();
    }
    // merge the chunk partials of this warp's head: lane cc holds chunk cc's (m, l)
    // and weight (nact <= 32), the output rows come 8 chunks at a time; the first 8
    // rows are loaded together with (m, l), so up to 8 chunks cost one round trip
    // and up to 16 two
    auto load_rows = [&](float4 (&ov)[8], int c0) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            ov[i] = c0 + i < nload ? __ldcg(reinterpret_cast<const float4*>(hp + (c0 + i) * ATT_PART + 4) + lane)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    float mc = -INFINITY, lc = 0.f;
    if (lane < nload) {
        const float2 ml = __ldcg(reinterpret_cast<const float2*>(hp + lane * ATT_PART));
        mc = ml.x;
        lc = ml.y;
    }
    float4 ov[8];
    load_rows(ov, 0);
    const float mown = nload < nact ? m : -INFINITY;  // tagged mode: this item's own chunk
    const float M = fmaxf(warp_max(mc), mown);
    const float wc = lane < nload ? expf(mc - M) : 0.f;
    const float wown = nload < nact ? expf(mown - M) : 0.f;
    const float Ls = warp_sum(lc * wc) + (nload < nact ? l * wown : 0.f);
    float r0 = o0 * wown, r1 = o1 * wown, r2 = o2 * wown, r3 = o3 * wown;
    for (int c0 = 0; c0 < nload; c0 += 8) {
        if (c0 > 0)
            load_rows(ov, c0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float w = __shfl_sync(0xffffffffu, wc, (c0 + i) & 31);  // 0 past nload
            r0 = fmaf(ov[i].x, w, r0); r1 = fmaf(ov[i].y, w, r1);
            r2 = fmaf(ov[i].z, w, r2); r3 = fmaf(ov[i].w, w, r3);
        }
    }
    const float inv = 1.0f / Ls;
    att_st_out(a.out + static_cast<size_t>(h) * ATT_HD + 4 * lane, make_float4(r0 * inv, r1 * inv, r2 * inv, r3 * inv),
               a.tag);
    att_stamp(a, 7, tid);
    if (!tagged) {  // the counter goes back to zero for the next call (tagged mode uses stamps)
        named_bar_sync(bar, nthr);
        if (tid == 0)
            a.counters[g] = 0;
    }
    return true;
}


}  // namespace dq

namespace dqhost {

size_t attention_workspace_bytes(int n_q, int n_kv);
// Fills tab [max_ctx][hd / 2] with (cos, sin) of p / theta^(2i / hd), computed
// in double precision and rounded once.
cudaError_t launch_rope_table(float2* tab, int max_ctx, int hd, double theta, cudaStream_t stream);
// Splits a workspace into the counters and the partials.
void attention_bind_workspace(dq::AttnArgs& a, void* ws);
cudaError_t launch_attention(const dq::AttnArgs& a, cudaStream_t stream, bool pdl);

}  // namespace dqhost
