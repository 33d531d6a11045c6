// dq_gemv.cuh -- the weight-streaming matrix-vector kernel (sm_103a).
//
// y[r] = sum_k W[r][k] x[k] for bf16, Q4_K and Q6_K rows ("The Mountain Runs",
// section 3: one output per weight row, the weights read in wide consecutive
// chunks; "The roofline holds on a second GPU", section "Hiding, fusing...":
// packed weights unpacked in registers, 32-bit accumulation, enough bytes in
// flight to cover the memory latency).
//
// Structure of one thread block (1 per SM, 512 threads, 16 warps):
//   * the block's rows stream, R rows per stage, into a ring of shared-memory
//     stages with 1-D bulk (TMA) copies that complete on an mbarrier (L2
//     evict-first: weights are read once).  The first ring-full is issued
//     right after the set-up barrier, one stage per lane of warp 0;
//   * all 16 warps consume every stage.  They are split into RG row groups of
//     P threads; within a group each thread owns UL fixed 32-weight units of
//     the K axis (16-byte units for bf16), so its slice of the activation is
//     held in registers, quantised once per block;
//   * per stage each thread forms its unit dot products for RPT rows of its
//     group, the warp reduces them (transpose-reduce) into shared memory and
//     releases the stage with an mbarrier arrive (no waiting);
//   * stage t is completed by warp t % 16 a couple of stages later: it waits
//     for the stage's release phase (normally already complete), refills the
//     slot with stage t + nstage and runs the epilogue of the stage's rows
//     from the warps' partial sums.  No warp waits for another on the common
//     path, and the extra work rotates over the warps.
// The first ring-full is issued before griddepcontrol.wait: weights never depend
// on the previous kernel, so under programmatic dependent launch the ring fills
// while the previous kernel drains.  Activations are read only after the wait.
#pragma once

#include "dq_common.cuh"

namespace dq {

constexpr int NCONS = 512;
constexpr int NCONS_WARPS = NCONS / 32;
constexpr int GEMV_THREADS = NCONS;
constexpr int MAX_STAGES = 8;
constexpr int MAX_RPT = 4;
constexpr int MAX_RG = 8;  // row groups of >= 64 threads use named barriers 1..8

enum { PRO_F32 = 0, PRO_RMS = 1, PRO_BF16 = 2 };
enum { EPI_STORE = 0, EPI_RESID = 1, EPI_QKV = 2, EPI_SWIGLU = 3 };

// Per-token arguments of the decode graph, in device memory.
struct StepArgs {
    int pos;
    int pad;
    float* logits;
};

struct GemvArgs {
    const uint8_t* W;   // matrix 0, row-major rows of row_bytes
    const uint8_t* W2;  // matrix 1 (EPI_SWIGLU: the up table), else null
    int rows;           // rows of each matrix
    int K;
    int row_bytes;
    int P;              // consumer threads per row group
    int RG;             // row groups (NCONS / P)
    int nstage;
    int stage_bytes;    // RG * RPT * row_bytes * NMAT
    int pro;            // PRO_*
    int epi;            // EPI_*
    const float* x;     // fp32 activation [K] (PRO_F32, PRO_RMS)
    const uint16_t* xb; // bf16 activation [K] (PRO_BF16)
    const float* gamma; // RMSNorm weight [K] (PRO_RMS)
    float eps;
    float* y;           // output [rows] (EPI_STORE/RESID/SWIGLU), q output (EPI_QKV)
    int y_from_step;    // EPI_STORE: write to step->logits instead of y
    const StepArgs* step;
    __half* kv_k;       // EPI_QKV: this layer's K plane [n_kv][max_ctx][hd]
    __half* kv_v;
    float* k_new;       // EPI_QKV: when not null, k rows go here (fp32 [kvdim]) for the attention to finish
    int qdim, kvdim, hd, max_ctx;
    int resid_rows;             // EPI_RESID: shared-memory slots for the block's residual rows
    int w_late;                 // 1: the weights may be the previous kernel's output -- before the
                                // dependency wait only L2 prefetches of them, the copies after it
    int* err;
    unsigned long long* trace;  // diagnostics: per-block timestamps when not null
};

// ---------------------------------------------------------- activation units

// One 32-element slice of the activation as fixed point: x ~= s * xi with 15-bit
// integers xi (PL = 1), or x ~= s * (xi + xl / 2^15) with a second 16-bit plane of
// the remainder (PL = 2, about 30 bits, fp32-level) for the inputs whose errors
// the attention amplifies.
template <int PL>
struct XQ {
    uint32_t q[16];               // q[p] = xi[2p] (low 16 bits) | xi[2p+1] << 16, |xi| <= 16383
    uint32_t l[PL == 2 ? 16 : 1]; // PL = 2: the remainder plane, same packing, |xl| <= 16384
    float s;                      // group scale
    float f;                      // Q4_K: s / 16
    float hsum;                   // Q4_K: s * (sum of the rounded values): the min term
    int s32a, s32b;               // Q6_K: 32 * sum xi[0..15], 32 * sum xi[16..31]
};

constexpr float XQ_MAX = 16383.0f;

// Natural unit index -> first k of the unit.  Q6_K units are permuted within
// spans of 8 blocks so that the 4 blocks a warp touches have distinct
// shared-memory bank phases (block stride 210 B).
template <int FMT>
__device__ __forceinline__ int unit_k0(int n)
{
    if (FMT == FMT_Q6K) {
        const int B = n >> 3, i = B & 7;
        const int Bp = (B & ~7) + (i < 4 ? 2 * i : 2 * (i - 4) + 1);
        return 256 * Bp + 32 * (n & 7);
    }
    return 32 * n;
}

// Round to the nearest integer, ties to even, for |t| < 2^22: adding 1.5 * 2^23
// leaves the rounded integer in the low mantissa bits (one FADD and one IADD
// instead of a conversion, whose pipe is a quarter as wide).
__device__ __forceinline__ int round_small(float t)
{
    return __float_as_int(__fadd_rn(t, 12582912.0f)) - 0x4B400000;
}

__device__ __forceinline__ uint32_t pack16x2(int a, int b)
{
    return (static_cast<uint32_t>(a) & 0xffffu) | (static_cast<uint32_t>(b) << 16);
}

// ------------------------------------------------------------- unit products

// Q4_K unit n of a row: 32 weights of sub-block j = n & 7 of block n >> 3.
// What a unit product needs of the stage: the sub-block's 16 code bytes, the
// block's d and dmin (fp16 pair), and the sub-block's 6-bit scale and min
// (bits 0-5 and 8-13 of smn) taken out of the header as it is read.
struct Q4KW {
    uint4 c;
    uint32_t dd, smn;
};

__device__ __forceinline__ Q4KW q4k_load(const uint8_t* rp, int n)
{
    const int j = n & 7;
    const uint8_t* bp = rp + Q4K_BYTES * (n >> 3);
    const uint4 hd = lds128(bp);
    // scale j: bits 6j.. of the 96-bit string (hd.y, hd.z, hd.w); min j: bits 48+6j..
    const uint32_t s_lo = j < 6 ? hd.y : hd.z, s_hi = j < 6 ? hd.z : hd.w;
    const uint32_t m_lo = j < 3 ? hd.z : hd.w, m_hi = j < 3 ? hd.w : 0u;
    const uint32_t sc = __funnelshift_r(s_lo, s_hi, (6 * j) & 31) & 63u;
    const uint32_t mn = __funnelshift_r(m_lo, m_hi, (48 + 6 * j) & 31) & 63u;
    return Q4KW{lds128(bp + 16 + 16 * j), hd.x, sc | (mn << 8)};
}

template <int PL>
__device__ __forceinline__ float q4k_dot(const Q4KW& w, int n, const XQ<PL>& u)
{
    (void)n;
    const uint32_t cw[4] = {w.c.x, w.c.y, w.c.z, w.c.w};
    // four independent accumulators per plane keep the dependent chains short
    int la = 0, lb = 0, ha = 0, hb = 0, la2 = 0, lb2 = 0, ha2 = 0, hb2 = 0;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const uint32_t l = cw[t] & 0x0F0F0F0Fu;  // codes of weights 4t .. 4t+3
        const uint32_t h = cw[t] & 0xF0F0F0F0u;  // 16 x codes of weights 16+4t .. 16+4t+3
        la = dp2a_lo(u.q[2 * t], l, la);
        lb = dp2a_hi(u.q[2 * t + 1], l, lb);
        ha = dp2a_lo(u.q[8 + 2 * t], h, ha);
        hb = dp2a_hi(u.q[8 + 2 * t + 1], h, hb);
        if (PL == 2) {
            la2 = dp2a_lo(u.l[2 * t], l, la2);
            lb2 = dp2a_hi(u.l[2 * t + 1], l, lb2);
            ha2 = dp2a_lo(u.l[8 + 2 * t], h, ha2);
            hb2 = dp2a_hi(u.l[8 + 2 * t + 1], h, hb2);
        }
    }
    float dot16 = static_cast<float>((la + lb) * 16 + (ha + hb));  // 16 * sum q * xi
    if (PL == 2)
        dot16 += static_cast<float>((la2 + lb2) * 16 + (ha2 + hb2)) * (1.0f / 32768.0f);
    const int sc = static_cast<int>(w.smn & 63u), mn = static_cast<int>(w.smn >> 8);
    const float d = half_bits_to_float(w.dd), dmin = half_bits_to_float(w.dd >> 16);
    return (d * static_cast<float>(sc)) * (u.f * dot16) - (dmin * static_cast<float>(mn)) * u.hsum;
}

template <int PL>
__device__ __forceinline__ float q4k_unit(const uint8_t* rp, int n, const XQ<PL>& u)
{
    return q4k_dot<PL>(q4k_load(rp, n), n, u);
}

// Q6_K unit: 32 weights of group g of (permuted) block Bp; fields start at
// even byte offsets, so they are read as aligned words and re-aligned as they
// are read: the 16 low-bit bytes, the 8 high-bit bytes, the two scales (bits
// 0-15 of sd) and the block's d (bits 16-31).
struct Q6KW {
    uint32_t ql[4], H0, H1, sd;
};

__device__ __forceinline__ int q6k_block(int n)
{
    const int B = n >> 3, i = B & 7;
    return (B & ~7) + (i < 4 ? 2 * i : 2 * (i - 4) + 1);
}

__device__ __forceinline__ Q6KW q6k_load(const uint8_t* rp, int n)
{
    const int Bp = q6k_block(n);
    const int g = n & 7;
    const uint8_t* bp = rp + Q6K_BYTES * Bp;
    const uint32_t sh = (Bp & 1) ? 16u : 0u;       // rows are 16-byte aligned
    const uint8_t* pl = bp + 16 * g - (sh >> 3);    // aligned word at or before ql
    const uint8_t* ph = bp + 128 + 8 * g - (sh >> 3);
    const uint32_t w0 = lds32(pl), w1 = lds32(pl + 4), w2 = lds32(pl + 8), w3 = lds32(pl + 12),
                   w4 = lds32(pl + 16);
    const uint32_t h0 = lds32(ph), h1 = lds32(ph + 4), h2 = lds32(ph + 8);
    Q6KW w;
    w.ql[0] = __funnelshift_r(w0, w1, sh);
    w.ql[1] = __funnelshift_r(w1, w2, sh);
    w.ql[2] = __funnelshift_r(w2, w3, sh);
    w.ql[3] = __funnelshift_r(w3, w4, sh);
    w.H0 = __funnelshift_r(h0, h1, sh);
    w.H1 = __funnelshift_r(h1, h2, sh);
    w.sd = *reinterpret_cast<const uint16_t*>(bp + 192 + 2 * g) |
           (static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(bp + 208)) << 16);
    return w;
}

__device__ __forceinline__ float q6k_dot(const Q6KW& w, int n, const XQ<1>& u)
{
    (void)n;
    int da = 0, db = 0, da2 = 0, db2 = 0;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        // high two bits of weights 4t+e sit at bits 2t of byte e: move them to bits 4-5
        const uint32_t ha = (t < 2 ? (w.H0 << (4 - 2 * t)) : (w.H0 >> (2 * t - 4))) & 0x30303030u;
        const uint32_t hb = (t < 2 ? (w.H1 << (4 - 2 * t)) : (w.H1 >> (2 * t - 4))) & 0x30303030u;
        const uint32_t qa = (w.ql[t] & 0x0F0F0F0Fu) | ha;         // q of weights 4t+e
        const uint32_t qb = ((w.ql[t] >> 4) & 0x0F0F0F0Fu) | hb;  // q of weights 16+4t+e
        da = dp2a_lo(u.q[2 * t], qa, da);
        da2 = dp2a_hi(u.q[2 * t + 1], qa, da2);
        db = dp2a_lo(u.q[8 + 2 * t], qb, db);
        db2 = dp2a_hi(u.q[8 + 2 * t + 1], qb, db2);
    }
    da += da2;
    db += db2;
    const int sca = static_cast<int>(static_cast<int8_t>(w.sd & 0xffu));
    const int scb = static_cast<int>(static_cast<int8_t>((w.sd >> 8) & 0xffu));
    const int v = sca * (da - u.s32a) + scb * (db - u.s32b);  // sum sc (q - 32) xi, |v| < 2^31
    return (half_bits_to_float(w.sd >> 16) * u.s) * static_cast<float>(v);
}

__device__ __forceinline__ float q6k_unit(const uint8_t* rp, int n, const XQ<1>& u)
{
    return q6k_dot(q6k_load(rp, n), n, u);
}

// Q2_K unit n of a row: sub-blocks 2(n & 7) and 2(n & 7) + 1 of block n >> 3
// (32 weights).  Each sub-block's 16 codes are one 32-bit word: shifting it by
// 2k and masking leaves weights 4k..4k+3 in the four bytes, in activation order.
__device__ __forceinline__ float q2k_unit(const uint8_t* rp, int n, const XQ<1>& u)
{
    const uint8_t* bp = rp + Q2K_BYTES * (n >> 3);  // 4-byte aligned (84 = 4 * 21)
    const int ja = 2 * (n & 7);
    const uint32_t hd = lds32(bp);
    const uint32_t scm = *reinterpret_cast<const uint16_t*>(bp + 4 + ja);  // sc|m of sub-blocks ja, ja + 1
    const uint32_t wa = lds32(bp + 20 + 4 * ja), wb = lds32(bp + 24 + 4 * ja);
    int da = 0, da2 = 0, db = 0, db2 = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t ca = (wa >> (2 * k)) & 0x03030303u;
        const uint32_t cb = (wb >> (2 * k)) & 0x03030303u;
        da = dp2a_lo(u.q[2 * k], ca, da);
        da2 = dp2a_hi(u.q[2 * k + 1], ca, da2);
        db = dp2a_lo(u.q[8 + 2 * k], cb, db);
        db2 = dp2a_hi(u.q[8 + 2 * k + 1], cb, db2);
    }
    const int sca = static_cast<int>(scm & 15u), ma = static_cast<int>((scm >> 4) & 15u);
    const int scb = static_cast<int>((scm >> 8) & 15u), mb = static_cast<int>(scm >> 12);
    const int v = sca * (da + da2) + scb * (db + db2);  // |v| < 2 * 15 * 16 * 3 * 16383
    const int mn32 = ma * u.s32a + mb * u.s32b;        // 32 * sum_j m_j * (sum of that half's xi)
    const float d = half_bits_to_float(hd), dmin = half_bits_to_float(hd >> 16);
    return (d * u.s) * static_cast<float>(v) - (dmin * u.s * (1.0f / 32.0f)) * static_cast<float>(mn32);
}

// Q2_K units n and n + 1 (n even: one block, sub-blocks 2(n & 7) .. + 3) of a row
// at once: the block header, the four scale/min bytes (one word) and the fp16
// conversions are shared.
__device__ __forceinline__ float q2k_unit_pair(const uint8_t* rp, int n, const XQ<1>& u0, const XQ<1>& u1)
{
    const uint8_t* bp = rp + Q2K_BYTES * (n >> 3);
    const int ja = 2 * (n & 7);
    const uint32_t hd = lds32(bp);
    const uint32_t scm = lds32(bp + 4 + ja);  // sc|m bytes of sub-blocks ja .. ja + 3 (4-byte aligned: ja % 4 == 0)
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
        w[q] = lds32(bp + 20 + 4 * (ja + q));
    int d0[4] = {0, 0, 0, 0}, d1[4] = {0, 0, 0, 0};  // per sub-block: lo and hi dp2a chains
#pragma unroll
    for (int k = 0; k < 4; ++k) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const XQ<1>& u = q < 2 ? u0 : u1;
            const int o = (q & 1) * 8;  // sub-block q & 1 of its unit: activation words 0..7 or 8..15
            const uint32_t c = (w[q] >> (2 * k)) & 0x03030303u;
            d0[q] = dp2a_lo(u.q[o + 2 * k], c, d0[q]);
            d1[q] = dp2a_hi(u.q[o + 2 * k + 1], c, d1[q]);
        }
    }
    int v[2], mn[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t sa = (scm >> (16 * h)) & 0xffu, sb = (scm >> (16 * h + 8)) & 0xffu;
        const XQ<1>& u = h ? u1 : u0;
        v[h] = static_cast<int>(sa & 15u) * (d0[2 * h] + d1[2 * h]) +
               static_cast<int>(sb & 15u) * (d0[2 * h + 1] + d1[2 * h + 1]);
        mn[h] = static_cast<int>(sa >> 4) * u.s32a + static_cast<int>(sb >> 4) * u.s32b;
    }
    const float d = half_bits_to_float(hd), dmin = half_bits_to_float(hd >> 16) * (1.0f / 32.0f);
    return (d * u0.s) * static_cast<float>(v[0]) - (dmin * u0.s) * static_cast<float>(mn[0]) +
           (d * u1.s) * static_cast<float>(v[1]) - (dmin * u1.s) * static_cast<float>(mn[1]);
}

// bf16 unit n: 8 weights at byte 16n of the row; xb holds the 8 bf16 activations.
__device__ __forceinline__ float bf16_unit(const uint8_t* rp, int n, const uint32_t (&xb)[4])
{
    const uint4 w = lds128(rp + 16 * n);
    float a0 = bf16lo(w.x) * bf16lo(xb[0]);
    float a1 = bf16hi(w.x) * bf16hi(xb[0]);
    a0 = fmaf(bf16lo(w.y), bf16lo(xb[1]), a0);
    a1 = fmaf(bf16hi(w.y), bf16hi(xb[1]), a1);
    a0 = fmaf(bf16lo(w.z), bf16lo(xb[2]), a0);
    a1 = fmaf(bf16hi(w.z), bf16hi(xb[2]), a1);
    a0 = fmaf(bf16lo(w.w), bf16lo(xb[3]), a0);
    a1 = fmaf(bf16hi(w.w), bf16hi(xb[3]), a1);
    return a0 + a1;
}

// -------------------------------------------------------- warp reductions

// Reduce NV values per lane across the warp.  Afterwards the lanes with
// (lane % (32 / NV)) == 0 hold the total of value index
// sum_s bit(lane, 16 >> s) * (NV >> (s + 1)), i.e. lane 32/NV * v holds value v.
template <int NV>
__device__ __forceinline__ void warp_transpose_reduce(float (&v)[NV], int lane)
{
    int n = NV;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        if (n > 1) {
            const bool up = (lane & o) != 0;
#pragma unroll
            for (int k = 0; k < NV / 2; ++k) {
                if (k < n / 2) {
                    const float send = up ? v[k] : v[k + n / 2];
                    const float keep = up ? v[k + n / 2] : v[k];
                    v[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            n >>= 1;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
        }
    }
}

// ------------------------------------------------------------------ kernel

template <int FMT, int PL>
struct UnitState {
    XQ<PL> x;
};
template <int PL>
struct UnitState<FMT_BF16, PL> {
    uint32_t xb[4];
};

// The k-th activation unit of thread p of a P-thread row group holding UL units:
// p + P k, or, for Q2_K with an even UL, adjacent pairs UL p + k (a pair shares one
// block of the weight row, see q2k_unit_pair).
template <int FMT, int UL>
__host__ __device__ constexpr bool q2k_pairs() { return FMT == FMT_Q2K && UL % 2 == 0; }
template <int FMT, int UL>
__device__ __forceinline__ int unit_of(int p, int P, int k)
{
    return q2k_pairs<FMT, UL>() ? UL * p + k : p + P * k;
}

// ------------------------------------------------------- shared-memory layout

// Entry strides are odd multiples of 16 bytes so that 8 lanes reading 8
// consecutive entries with 16-byte loads hit distinct banks.
constexpr int XQ_WORDS_PL1 = 28;  // q[16], s, f, hsum, s32a, s32b, pad: 112 bytes
constexpr int XQ_WORDS_PL2 = 44;  // q[16], l[16], s, f, hsum, s32a, s32b, pad: 176 bytes
constexpr int GEMV_MISC_BYTES = 256;

__host__ __device__ constexpr int xq_words(int pl) { return pl == 2 ? XQ_WORDS_PL2 : XQ_WORDS_PL1; }

// Offsets of the block's shared-memory regions: the weight ring, the quantised
// activation (one entry per 32-element unit), the block's residual rows, the
// per-warp partial sums and the barriers.
struct GemvSmem {
    int xq, resid, red, misc, total;
};

__host__ __device__ inline GemvSmem gemv_smem_layout(int fmt, int K, int nstage, int stage_bytes, int rpt, int nmat,
                                                     int pl, int resid_rows)
{
    GemvSmem L;
    int o = nstage * stage_bytes;
    L.xq = o;
    if (fmt != FMT_BF16)
        o += (K / 32) * xq_words(pl) * 4;
    L.resid = o;
    o += ((resid_rows * 4 + 15) / 16) * 16;
    L.red = o;
    o += 2 * nstage * NCONS_WARPS * rpt * nmat * 4;
    L.misc = o;
    o += GEMV_MISC_BYTES;
    L.total = o;
    return L;
}

// Largest number of 4-element activation chunks one thread quantises (K <= 16384).
constexpr int GEMV_MAX_K = 16384;
constexpr int QCHUNKS = GEMV_MAX_K / 4 / NCONS;

// ------------------------------------------------------------------ kernel

// Stream tile t (rows r0 + t R .. ) of the block's rows into its ring slot.
template <int NMAT>
__device__ __forceinline__ void issue_tile(const uint8_t* W, const uint8_t* W2, int row_bytes, int nstage,
                                           int stage_bytes, uint8_t* smem, uint64_t* full, int t, int r0, int r1,
                                           int R, uint64_t pol)
{
    const int s = t % nstage;
    const int row = r0 + t * R;
    const int nr = min(R, r1 - row);
    const uint32_t bytes = static_cast<uint32_t>(nr * row_bytes);
    uint8_t* dst = smem + static_cast<size_t>(s) * stage_bytes;
    mbar_arrive_expect_tx(&full[s], bytes * NMAT);
    bulk_g2s(dst, W + static_cast<size_t>(row) * row_bytes, bytes, &full[s], pol);
    if (NMAT == 2)
        bulk_g2s(dst + static_cast<size_t>(R) * row_bytes, W2 + static_cast<size_t>(row) * row_bytes, bytes,
                 &full[s], pol);
}

// Ask L2 for tile t of the block's rows (a hint: nothing is written and nothing
// waits for it).
template <int NMAT>
__device__ __forceinline__ void prefetch_tile(const uint8_t* W, const uint8_t* W2, int row_bytes, int t, int r0,
                                              int r1, int R)
{
    const int row = r0 + t * R;
    const uint32_t bytes = static_cast<uint32_t>(min(R, r1 - row) * row_bytes);
    prefetch_l2_bulk(W + static_cast<size_t>(row) * row_bytes, bytes);
    if (NMAT == 2)
        prefetch_l2_bulk(W2 + static_cast<size_t>(row) * row_bytes, bytes);
}

// Quantise one 4-element chunk c of the activation into the unit table xq: the
// 8 lanes c & ~7 .. c | 7 of the calling warp hold one 32-element unit (and all
// take part), four elements each.
template <int FMT, int PL>
__device__ __forceinline__ void quantise_chunk(float4 h, int c, uint32_t* xq)
{
    float amax = fmaxf(fmaxf(fabsf(h.x), fabsf(h.y)), fmaxf(fabsf(h.z), fabsf(h.w)));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float inv = amax > 0.f ? XQ_MAX / amax : 0.f;
    const float t0 = h.x * inv, t1 = h.y * inv, t2 = h.z * inv, t3 = h.w * inv;
    const int a0 = round_small(t0), a1 = round_small(t1), a2 = round_small(t2), a3 = round_small(t3);
    const int e = c & 7;
    uint32_t* q = xq + (c >> 3) * xq_words(PL);
    *reinterpret_cast<uint2*>(q + 2 * e) = make_uint2(pack16x2(a0, a1), pack16x2(a2, a3));
    int lsum = 0;
    if (PL == 2) {  // remainders: t - a is exact in fp32
        const int b0 = round_small((t0 - static_cast<float>(a0)) * 32768.0f);
        const int b1 = round_small((t1 - static_cast<float>(a1)) * 32768.0f);
        const int b2 = round_small((t2 - static_cast<float>(a2)) * 32768.0f);
        const int b3 = round_small((t3 - static_cast<float>(a3)) * 32768.0f);
        *reinterpret_cast<uint2*>(q + 16 + 2 * e) = make_uint2(pack16x2(b0, b1), pack16x2(b2, b3));
        lsum = (b0 + b1) + (b2 + b3);
    }
    // Integer sums of the rounded values: per 16-element half (Q6_K's -32 offset,
    // Q2_K's mins) and over the unit (Q4_K's min term).  Taking the min term from
    // the same rounded values keeps the product exactly sum_k W_k x^_k, so the
    // rounding error meets the full (zero-mean) weights, not only their positive part.
    int isum = (a0 + a1) + (a2 + a3);
    isum += __shfl_xor_sync(0xffffffffu, isum, 1);
    isum += __shfl_xor_sync(0xffffffffu, isum, 2);
    const int ihalf = isum;  // this 16-element half
    isum += __shfl_xor_sync(0xffffffffu, isum, 4);
    if (PL == 2) {
#pragma unroll
        for (int o = 1; o < 8; o <<= 1)
            lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    }
    float* meta = reinterpret_cast<float*>(q + 16 * PL);
    if (e == 0 || e == 4) {
        const float sc = amax / XQ_MAX;
        if (e == 0) {
            meta[0] = sc;
            meta[1] = sc * 0.0625f;
            meta[2] = sc * (static_cast<float>(isum) + static_cast<float>(lsum) * (1.0f / 32768.0f));
            reinterpret_cast<int*>(meta)[3] = 32 * ihalf;
        } else {
            reinterpret_cast<int*>(meta)[4] = 32 * ihalf;
        }
    }
}

// Quantise the activation (times gamma under RMSNorm) once per block of NT
// threads: eight lanes share one 32-element unit, four elements each; chunk
// c = tid + NT i of the vector is v[i].  Returns this thread's partial sum of x^2.
template <int FMT, int PL, int NCH, int NT = NCONS>
__device__ __forceinline__ float quantise_block(float4 (&v)[NCH], const float4 (&gv)[NCH], bool norm, uint32_t* xq,
                                                int K, int tid)
{
    float ss = 0.f;
    const int nchunks = K / 4;  // a multiple of 32: whole warps take part in each pass
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
        const int c = tid + NT * i;
        if (c >= nchunks)
            break;
        float4 h = v[i];
        if (norm) {
            ss = fmaf(h.x, h.x, ss); ss = fmaf(h.y, h.y, ss); ss = fmaf(h.z, h.z, ss); ss = fmaf(h.w, h.w, ss);
            h.x *= gv[i].x; h.y *= gv[i].y; h.z *= gv[i].z; h.w *= gv[i].w;
        }
        quantise_chunk<FMT, PL>(h, c, xq);
    }
    return ss;
}

// quantise_block with every chunk's steps interleaved (the shuffles of all
// chunks in flight together, no early exit) and the scale reciprocal taken by
// the fast divide (the group's largest element still maps to exactly +-16383;
// the other values move by at most a few ulp of fp32, far below the rounding
// step): the chain from the activation load to the stored units is one
// shuffle-and-round latency, not NCH of them.
template <int FMT, int PL, int NCH, int NT = NCONS>
__device__ __forceinline__ float quantise_block_il(float4 (&v)[NCH], const float4 (&gv)[NCH], bool norm,
                                                   uint32_t* xq, int K, int tid)
{
    float ss = 0.f;
    const int nchunks = K / 4;
    float am[NCH];
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
        float4 h = v[i];
        if (norm) {
            ss = fmaf(h.x, h.x, ss); ss = fmaf(h.y, h.y, ss); ss = fmaf(h.z, h.z, ss); ss = fmaf(h.w, h.w, ss);
            h.x *= gv[i].x; h.y *= gv[i].y; h.z *= gv[i].z; h.w *= gv[i].w;
            v[i] = h;
        }
        am[i] = fmaxf(fmaxf(fabsf(h.x), fabsf(h.y)), fmaxf(fabsf(h.z), fabsf(h.w)));
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1)
#pragma unroll
        for (int i = 0; i < NCH; ++i)
            am[i] = fmaxf(am[i], __shfl_xor_sync(0xffffffffu, am[i], o));
    uint2 pk[NCH], pl[NCH];
    int hs[NCH], hh[NCH], ls[NCH];
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
        const float inv = am[i] > 0.f ? __fdividef(XQ_MAX, am[i]) : 0.f;
        const float t0 = v[i].x * inv, t1 = v[i].y * inv, t2 = v[i].z * inv, t3 = v[i].w * inv;
        const int a0 = round_small(t0), a1 = round_small(t1), a2 = round_small(t2), a3 = round_small(t3);
        pk[i] = make_uint2(pack16x2(a0, a1), pack16x2(a2, a3));
        hs[i] = (a0 + a1) + (a2 + a3);
        ls[i] = 0;
        if (PL == 2) {
            const int b0 = round_small((t0 - static_cast<float>(a0)) * 32768.0f);
            const int b1 = round_small((t1 - static_cast<float>(a1)) * 32768.0f);
            const int b2 = round_small((t2 - static_cast<float>(a2)) * 32768.0f);
            const int b3 = round_small((t3 - static_cast<float>(a3)) * 32768.0f);
            pl[i] = make_uint2(pack16x2(b0, b1), pack16x2(b2, b3));
            ls[i] = (b0 + b1) + (b2 + b3);
        }
    }
#pragma unroll
    for (int o = 1; o < 4; o <<= 1)
#pragma unroll
        for (int i = 0; i < NCH; ++i)
            hs[i] += __shfl_xor_sync(0xffffffffu, hs[i], o);
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
        hh[i] = hs[i];  // this 16-element half
        hs[i] += __shfl_xor_sync(0xffffffffu, hs[i], 4);
    }
    if (PL == 2) {
#pragma unroll
        for (int o = 1; o < 8; o <<= 1)
#pragma unroll
            for (int i = 0; i < NCH; ++i)
                ls[i] += __shfl_xor_sync(0xffffffffu, ls[i], o);
    }
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
        const int c = tid + NT * i;
        if (c < nchunks) {
            const int e = c & 7;
            uint32_t* q = xq + (c >> 3) * xq_words(PL);
            *reinterpret_cast<uint2*>(q + 2 * e) = pk[i];
            if (PL == 2)
                *reinterpret_cast<uint2*>(q + 16 + 2 * e) = pl[i];
            float* meta = reinterpret_cast<float*>(q + 16 * PL);
            const float sc = am[i] * (1.0f / XQ_MAX);
            if (e == 0) {
                meta[0] = sc;
                meta[1] = sc * 0.0625f;
                meta[2] = sc * (static_cast<float>(hs[i]) + static_cast<float>(ls[i]) * (1.0f / 32768.0f));
                reinterpret_cast<int*>(meta)[3] = 32 * hh[i];
            } else if (e == 4) {
                reinterpret_cast<int*>(meta)[4] = 32 * hh[i];
            }
        }
    }
    return ss;
}

#ifndef GEMV_QIL
#define GEMV_QIL 1
#endif

// The standalone kernel's activation quantiser: the interleaved form for the
// chunk count K needs (2, 4, 6 or 8 chunks a thread; the chunks past K hold
// zeros and store nothing).
template <int FMT, int PL>
__device__ __forceinline__ float quantise_activation(float4 (&xv)[QCHUNKS], const float4 (&gv)[QCHUNKS], bool norm,
                                                     uint32_t* xq, int K, int tid)
{
    static_assert(QCHUNKS == 8, "chunk counts below");
    if (!GEMV_QIL)
        return quantise_block<FMT, PL, QCHUNKS>(xv, gv, norm, xq, K, tid);
    const int nch = (K / 4 + NCONS - 1) / NCONS;
    if (nch <= 2)
        return quantise_block_il<FMT, PL, 2>(*reinterpret_cast<float4(*)[2]>(&xv),
                                             *reinterpret_cast<const float4(*)[2]>(&gv), norm, xq, K, tid);
    if (nch <= 4)
        return quantise_block_il<FMT, PL, 4>(*reinterpret_cast<float4(*)[4]>(&xv),
                                             *reinterpret_cast<const float4(*)[4]>(&gv), norm, xq, K, tid);
    if (nch <= 6)
        return quantise_block_il<FMT, PL, 6>(*reinterpret_cast<float4(*)[6]>(&xv),
                                             *reinterpret_cast<const float4(*)[6]>(&gv), norm, xq, K, tid);
    return quantise_block_il<FMT, PL, 8>(xv, gv, norm, xq, K, tid);
}

// One stage of the consumers: this thread's unit products for rows g, g + RG,
// ... (RPT of them, each of NMAT matrices) of the tile, reduced over the warp
// into wred[0 .. RPT NMAT) (the warp's partial sums; matrix m, row i at m RPT + i;
// three sums are reduced as four, so wred then holds a fourth, zero entry).
// nidx[k] is the unit thread k-slot k reads: its own unit, or a valid stand-in
// whose activation is zero (load_units) when the thread has none.  Rows past
// the tile's last (a partial last tile) are computed from stale stage bytes and
// never stored, so the loop has no branches.
template <int FMT, int PL, int UL, int RPT, int NMAT>
__device__ __forceinline__ void consume_tile(const uint8_t* tile, int R, int RG, int g, int row_bytes,
                                             const UnitState<FMT, PL> (&us)[UL], const int (&nidx)[UL], float* wred,
                                             int lane)
{
    constexpr int NV = RPT * NMAT == 3 ? 4 : RPT * NMAT;  // the transpose-reduce takes powers of two
    float acc[NV];
    if (NV != RPT * NMAT)
        acc[NV - 1] = 0.f;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int row = g + RG * i;
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
            const uint8_t* rp = tile + static_cast<size_t>(m * R + row) * row_bytes;
            float sum = 0.f;
            if (FMT == FMT_Q2K && UL % 2 == 0) {  // adjacent unit pairs (q2k_pairs)
#pragma unroll
                for (int k = 0; k < UL; k += 2)
                    sum += q2k_unit_pair(rp, nidx[k], reinterpret_cast<const XQ<1>&>(us[k]),
                                         reinterpret_cast<const XQ<1>&>(us[k + 1]));
                acc[m * RPT + i] = sum;
                continue;
            }
#pragma unroll
            for (int k = 0; k < UL; ++k) {
                if (FMT == FMT_Q4K)
                    sum += q4k_unit<PL>(rp, nidx[k], reinterpret_cast<const XQ<PL>&>(us[k]));
                else if (FMT == FMT_Q6K)
                    sum += q6k_unit(rp, nidx[k], reinterpret_cast<const XQ<1>&>(us[k]));
                else if (FMT == FMT_Q2K)
                    sum += q2k_unit(rp, nidx[k], reinterpret_cast<const XQ<1>&>(us[k]));
                else
                    sum += bf16_unit(rp, nidx[k], reinterpret_cast<const uint32_t(&)[4]>(us[k]));
            }
            acc[m * RPT + i] = sum;
        }
    }
    warp_transpose_reduce<NV>(acc, lane);
    if ((lane & (32 / NV - 1)) == 0)
        wred[lane / (32 / NV)] = acc[0];
    __syncwarp();
}

// Load this thread's activation units (unit p + P k of the K axis) from the
// quantised table into registers, folding the RMS factor into the scales.
template <int FMT, int PL, int UL>
__device__ __forceinline__ void load_units(UnitState<FMT, PL> (&us)[UL], const bool (&have)[UL], const uint32_t* xq,
                                           int p, int P, float rstd)
{
#pragma unroll
    for (int k = 0; k < UL; ++k) {
        XQ<PL>& u = reinterpret_cast<XQ<PL>&>(us[k]);
        if (!have[k]) {  // no unit: a zero activation (its products vanish)
#pragma unroll
            for (int w = 0; w < 16; ++w)
                u.q[w] = 0u;
            if (PL == 2)
#pragma unroll
                for (int w = 0; w < 16; ++w)
                    u.l[w] = 0u;
            u.s = u.f = u.hsum = 0.f;
            u.s32a = u.s32b = 0;
        } else {
            const uint32_t* src = xq + (unit_k0<FMT>(unit_of<FMT, UL>(p, P, k)) >> 5) * xq_words(PL);
#pragma unroll
            for (int w = 0; w < 16; w += 4) {
                const uint4 v = *reinterpret_cast<const uint4*>(src + w);
                u.q[w] = v.x; u.q[w + 1] = v.y; u.q[w + 2] = v.z; u.q[w + 3] = v.w;
            }
            if (PL == 2) {
#pragma unroll
                for (int w = 0; w < 16; w += 4) {
                    const uint4 v = *reinterpret_cast<const uint4*>(src + 16 + w);
                    u.l[w] = v.x; u.l[w + 1] = v.y; u.l[w + 2] = v.z; u.l[w + 3] = v.w;
                }
            }
            const float* meta = reinterpret_cast<const float*>(src + 16 * PL);
            u.s = meta[0] * rstd;
            u.f = meta[1] * rstd;
            u.hsum = meta[2] * rstd;
            u.s32a = reinterpret_cast<const int*>(meta)[3];
            u.s32b = reinterpret_cast<const int*>(meta)[4];
        }
    }
}

template <int FMT, int UL, int RPT, int NMAT, int PL>
__global__ void __maxnreg__(128) gemv_stream_kernel(const __grid_constant__ GemvArgs args)
{
    // A private copy: its fields live in registers.  (Taking the address of the
    // parameter would turn every field access into a memory load.)
    const GemvArgs a = args;
    constexpr int NV = RPT * NMAT;
    extern __shared__ __align__(128) uint8_t smem[];
    const bool norm = a.pro == PRO_RMS;
    const GemvSmem L = gemv_smem_layout(FMT, a.K, a.nstage, a.stage_bytes, RPT, NMAT, PL, a.resid_rows);
    uint32_t* xq = reinterpret_cast<uint32_t*>(smem + L.xq);
    float* resid = reinterpret_cast<float*>(smem + L.resid);
    float* red = reinterpret_cast<float*>(smem + L.red);            // [2 nstage][16 warps][NV]
    float* gred = reinterpret_cast<float*>(smem + L.misc + 48);     // [16] (48 bytes reserved)
    uint64_t* full = reinterpret_cast<uint64_t*>(gred + NCONS_WARPS);  // [MAX_STAGES]
    uint64_t* empty = full + MAX_STAGES;                            // [MAX_STAGES]
    float** step_logits = reinterpret_cast<float**>(empty + MAX_STAGES);
    int* step_pos = reinterpret_cast<int*>(step_logits + 1);

    pdl_trigger();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    unsigned long long* trace = a.trace ? a.trace + 8 * blockIdx.x : nullptr;
    // block 0 also records SM clocks per stage: [2t] stage t ready (thread 0), [2t + 1]
    // thread 0 done with it, [128 + t] stage t issued (t < 64)
    unsigned long long* ttile = (a.trace && blockIdx.x == 0) ? a.trace + 8 * gridDim.x : nullptr;
    if (trace && tid == 0)
        trace[0] = globaltimer_ns();
    const int r0 = static_cast<int>(static_cast<long long>(blockIdx.x) * a.rows / gridDim.x);
    const int r1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * a.rows / gridDim.x);
    const int R = a.RG * RPT;
    const int ntiles = (r1 - r0 + R - 1) / R;
    const uint64_t pol = l2_evict_first_policy();
    const bool quant = FMT != FMT_BF16;

    if (tid == 0) {
        for (int s = 0; s < a.nstage; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NCONS_WARPS);
        }
        fence_mbar_init();
    }
    // the norm weight never depends on the previous kernel either
    float4 gv[QCHUNKS], xv[QCHUNKS];
    if (quant) {
#pragma unroll
        for (int i = 0; i < QCHUNKS; ++i) {
            const int c = tid + NCONS * i;
            gv[i] = make_float4(1.f, 1.f, 1.f, 1.f);
            if (norm && c < a.K / 4)
                gv[i] = __ldg(reinterpret_cast<const float4*>(a.gamma) + c);
        }
    }
    __syncthreads();
    // The first ring-full, one stage per lane of warp 0 (the copies start in
    // parallel).  Weights that never depend on the previous kernel (a model's
    // tables) are copied before the dependency wait; otherwise only L2 prefetches
    // go out before it (L2 is where the previous kernel's writes land, so a
    // prefetch can never leave a stale copy) and the copies follow the wait.
    const bool first = tid < min(a.nstage, ntiles);
    if (first) {
        if (a.w_late)
            prefetch_tile<NMAT>(a.W, a.W2, a.row_bytes, tid, r0, r1, R);
        else
            issue_tile<NMAT>(a.W, a.W2, a.row_bytes, a.nstage, a.stage_bytes, smem, full, tid, r0, r1, R, pol);
    }
    if (trace && tid == 0)
        trace[1] = globaltimer_ns();
    pdl_wait();  // the activation is the previous kernel's output
    if (first && a.w_late)
        issue_tile<NMAT>(a.W, a.W2, a.row_bytes, a.nstage, a.stage_bytes, smem, full, tid, r0, r1, R, pol);
    if (first && ttile)
        ttile[128 + tid] = clock64();
    if (trace && tid == 0)
        trace[2] = globaltimer_ns();

    // everything the epilogue needs from global memory, loaded once
    if (tid == 0) {
        *step_logits = a.y_from_step ? a.step->logits : a.y;
        *step_pos = a.epi == EPI_QKV ? a.step->pos : 0;
    }

    const int P = a.P;
    const int g = tid / P;
    const int p = tid - g * P;
    const int gw0 = (g * P) >> 5, nwg = P >> 5;  // the group's first warp and warp count
    const int U = (FMT == FMT_BF16) ? a.K / 8 : a.K / 32;

    UnitState<FMT, PL> us[UL];
    bool have[UL];
    int nidx[UL];
#pragma unroll
    for (int k = 0; k < UL; ++k) {
        have[k] = unit_of<FMT, UL>(p, P, k) < U;
        // a stand-in for a missing unit (zero activation); pairs keep their even start
        nidx[k] = have[k] ? unit_of<FMT, UL>(p, P, k) : (q2k_pairs<FMT, UL>() ? (U - 2 + (k & 1)) : U - 1);
    }

    if (FMT == FMT_BF16) {
#pragma unroll
        for (int k = 0; k < UL; ++k) {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (have[k])
                v = __ldcg(reinterpret_cast<const uint4*>(a.xb) + (p + P * k));
            uint32_t* xb = reinterpret_cast<uint32_t*>(&us[k]);
            xb[0] = v.x; xb[1] = v.y; xb[2] = v.z; xb[3] = v.w;
        }
        if (a.epi == EPI_RESID)
            for (int r = tid; r < r1 - r0; r += NCONS)
                resid[r] = __ldcg(a.y + r0 + r);
        __syncthreads();  // step fields and residual rows
    } else {
#pragma unroll
        for (int i = 0; i < QCHUNKS; ++i) {
            const int c = tid + NCONS * i;
            xv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (c < a.K / 4)
                xv[i] = __ldcg(reinterpret_cast<const float4*>(a.x) + c);
        }
        // the residual rows after the activation's loads are out: the round trips overlap
        if (a.epi == EPI_RESID)
            for (int r = tid; r < r1 - r0; r += NCONS)
                resid[r] = __ldcg(a.y + r0 + r);
        if (trace && tid == 0)
            trace[3] = globaltimer_ns();
        float ss = quantise_activation<FMT, PL>(xv, gv, norm, xq, a.K, tid);
        float rstd = 1.f;
        if (norm) {
            ss = warp_sum(ss);
            if (lane == 0)
                gred[warp] = ss;
        }
        __syncthreads();  // xq and gred complete
        if (trace && tid == 0)
            trace[4] = globaltimer_ns();
        if (norm) {
            float tot = 0.f;
            for (int w = 0; w < NCONS_WARPS; ++w)
                tot += gred[w];
            rstd = rsqrtf(tot / static_cast<float>(a.K) + a.eps);
        }
        load_units<FMT, PL, UL>(us, have, xq, p, P, rstd);
    }

    // Tile t is completed (its slot refilled, its rows' epilogue run) by warp
    // t % 16 as soon as that warp sees every warp release it: it tests the
    // slot's `empty` barrier after each of its stages and keeps testing while it
    // waits for its next stage, so the refill leaves without a fixed delay and a
    // warp only ever waits on another when its next stage needs that refill.
    const int rg_shift = 31 - __clz(a.RG);  // RG is a power of two
    auto complete = [&](int tc, int rslot) {
        if (lane == 0 && tc + a.nstage < ntiles) {
            issue_tile<NMAT>(a.W, a.W2, a.row_bytes, a.nstage, a.stage_bytes, smem, full, tc + a.nstage, r0, r1, R,
                             pol);
            if (ttile && tc + a.nstage < 64)
                ttile[128 + tc + a.nstage] = clock64();
        }
        const float* rb = red + rslot * NCONS_WARPS * NV;
        const int row0 = r0 + tc * R;
        const int nr = min(R, r1 - row0);
        for (int row = lane; row < nr; row += 32) {
            const int rg = row & (a.RG - 1), i = row >> rg_shift;
            const int w0 = (rg * P) >> 5;
            float v0 = 0.f, v1 = 0.f;
            for (int w = 0; w < nwg; ++w) {
                v0 += rb[(w0 + w) * NV + i];
                if (NMAT == 2)
                    v1 += rb[(w0 + w) * NV + RPT + i];
            }
            const int r = row0 + row;
            if (a.epi == EPI_STORE) {
                (*step_logits)[r] = v0;
            } else if (a.epi == EPI_RESID) {
                a.y[r] = resid[r - r0] + v0;
            } else if (a.epi == EPI_SWIGLU) {
                a.y[r] = v0 / (1.0f + expf(-v0)) * v1;
            } else {  // EPI_QKV
                if (r < a.qdim) {
                    a.y[r] = v0;
                } else {
                    const int idx = r - a.qdim;
                    const int which = idx / a.kvdim, rem = idx - which * a.kvdim;
                    const int kvh = rem / a.hd, dd = rem - kvh * a.hd;
                    __half* plane = which ? a.kv_v : a.kv_k;
                    const int pos = *step_pos;
                    if (!which && a.k_new)
                        a.k_new[rem] = v0;
                    else if (pos >= 0 && pos < a.max_ctx)
                        plane[(static_cast<size_t>(kvh) * a.max_ctx + pos) * a.hd + dd] = __float2half_rn(v0);
                    else
                        set_error(a.err, DEVERR_BAD_ARG);
                }
            }
        }
    };

    // Counters instead of divisions by the runtime stage count: stage t uses ring
    // slot t % nstage with phase (t / nstage) & 1 and partial-sum slot t % (2 nstage).
    int pend = -1, pend_s = 0, pend_r = 0;  // the tile this warp completes next (-1: none)
    uint32_t pend_ph = 0;
    bool ok = true;
    int t = 0, s = 0, rslot = 0;
    uint32_t phase = 0;
    for (; t < ntiles && ok; ++t) {
        if (pend < 0) {
            if (!mbar_wait(&full[s], phase)) {
                set_error(a.err, DEVERR_TIMEOUT_FULL);
                ok = false;
                break;
            }
        } else if (!mbar_test_wait(&full[s], phase)) {  // wait for the stage, completing the pending tile meanwhile
            const unsigned long long t0 = globaltimer_ns();
            bool got = false;
            while (pend >= 0) {
                if (mbar_test_wait(&empty[pend_s], pend_ph)) {
                    complete(pend, pend_r);
                    pend = -1;
                } else if (mbar_test_wait(&full[s], phase)) {
                    got = true;
                    break;
                } else if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
                    set_error(a.err, DEVERR_TIMEOUT_EMPTY);
                    ok = false;
                    break;
                }
            }
            if (!ok)
                break;
            if (!got && !mbar_wait(&full[s], phase)) {
                set_error(a.err, DEVERR_TIMEOUT_FULL);
                ok = false;
                break;
            }
        }
        if (trace && t == 0 && tid == 0)
            trace[5] = globaltimer_ns();
        if (ttile && tid == 0 && t < 64)
            ttile[2 * t] = clock64();
        const uint8_t* tile = smem + static_cast<size_t>(s) * a.stage_bytes;
        consume_tile<FMT, PL, UL, RPT, NMAT>(tile, R, a.RG, g, a.row_bytes, us, nidx,
                                             red + rslot * NCONS_WARPS * NV + warp * NV, lane);
        if (lane == 0)
            mbar_arrive(&empty[s]);  // release semantics: the partial sums are visible to the completer
        if (ttile && tid == 0 && t < 64)
            ttile[2 * t + 1] = clock64();
        if ((t & (NCONS_WARPS - 1)) == warp) {  // this warp's tile (a previous one was completed before
            pend = t;                           // its stage t - 16 + nstage < t could be waited for)
            pend_s = s;
            pend_ph = phase;
            pend_r = rslot;
        }
        if (pend >= 0 && mbar_test_wait(&empty[pend_s], pend_ph)) {
            complete(pend, pend_r);
            pend = -1;
        }
        if (++s == a.nstage) {
            s = 0;
            phase ^= 1u;
        }
        if (++rslot == 2 * a.nstage)
            rslot = 0;
    }
    // the tile still pending (after a timeout nothing is: no refill is owed then)
    if (ok && pend >= 0) {
        if (mbar_wait(&empty[pend_s], pend_ph))
            complete(pend, pend_r);
        else
            set_error(a.err, DEVERR_TIMEOUT_EMPTY);
    }
    (void)gw0;
    if (trace && lane == 0) {  // the last warp of the block to finish records the end
        atomicMax(trace + 6, globaltimer_ns());
        atomicAdd(trace + 7, 1ull);
    }
}

}  // namespace dq
