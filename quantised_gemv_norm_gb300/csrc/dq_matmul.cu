// dq_matmul.cu -- Y[m] = W X[m] for M token vectors over one Q4_K matrix.
//
// "The roofline holds on a second GPU", section "The Math": M tokens processed
// together share one read of the weights until the arithmetic catches up, at
// M* = (w / 16) (R / BW).  Two paths:
//
//   * CUDA cores: the single-vector streaming GEMV once per token (reads the
//     weights M times; the M = 1 path and the comparison point);
//   * tensor cores (M >= 2): every weight is read once for all M tokens.  Each
//     block takes a contiguous range of rows (at most 128 per tile: one row
//     per tensor-memory lane) and walks K in Q4_K block columns.  Each block
//     column of the tile's rows (one 144-byte block per row, rows row_bytes
//     apart) streams into a shared-memory ring with one 2-D tensor (TMA) copy.
//     Per block column (256 K) every thread dequantises 64 weights of one row to
//     fp16 in registers and stores them straight into an A buffer in tensor
//     memory (tcgen05.st); the tokens' activations are staged in shared memory
//     as fp16 in the UMMA K-major core-matrix layout.  Four control warps, one per
//     scheduler, issue the stage's sixteen tcgen05.mma (M = 128, N = tokens
//     rounded up to 16, K = 16, A from tensor memory), control warp q those of
//     fp32 accumulator q in tensor memory: one thread took about 125 cycles an MMA.  Two A/B buffers: the
//     next block column is dequantised while the MMAs run; their commit releases
//     a buffer.  The epilogue reads the accumulator with tcgen05.ld.
//     A in tensor memory keeps the dequantised weights out of shared memory,
//     whose bandwidth the MMAs would otherwise share with the dequantisation.
//
// fp16 and not bf16 operands: a dequantised Q4_K weight d sc q - dmin m has up
// to 21 significant bits; fp16 keeps 11 (relative error 2^-12 per weight,
// about 1e-4 normwise on a row), bf16 only 8 (about 1e-3, half the tolerance).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "dq_gemv_host.h"
#include "dq_tc.cuh"

namespace dq {

constexpr int MM_DQ_WARPS = 16;                // dequantisation / staging / epilogue warps
constexpr int MM_CTRL = MM_DQ_WARPS;           // the first control warp (copies and MMAs)
#ifndef MM_NCTRL_DEF
#define MM_NCTRL_DEF 4
#endif
// control warps, one per scheduler: control warp q issues the MMAs of accumulator q
constexpr int MM_NCTRL = MM_NCTRL_DEF;
constexpr int MM_THREADS = 32 * (MM_DQ_WARPS + MM_NCTRL);
constexpr int MM_ROWS = 128;                   // rows per tile = UMMA M
constexpr int MM_KC = 256;                     // K per MMA stage: one Q4_K block column
constexpr int MM_BPS = 4;                      // Q4_K block columns per ring slot
constexpr int MM_ROWB = MM_BPS * Q4K_BYTES + 16;  // 592: a slot row (4 blocks and 16 bytes of the next;
                                                  // the odd 16-byte stride keeps 8 rows on distinct banks)
constexpr int MM_NS_MAX = 4;
// operand (A in tensor memory, B in shared) buffers at most, where tensor memory
// holds them (3 measured no faster than 2: the dequantising warps set the pace)
#ifndef MM_NAB_MAX_DEF
#define MM_NAB_MAX_DEF 3
#endif
constexpr int MM_NAB_MAX = MM_NAB_MAX_DEF;
constexpr int MM_ACC = 4;                      // independent accumulators (MMA s of a stage adds into s % 4)
// every accumulator's MMAs come from one thread (one thread's MMAs run in order)
static_assert(MM_ACC % MM_NCTRL == 0, "control warps per accumulator");
constexpr int MM_TA_COLS = MM_KC / 2;          // columns of one A buffer (two fp16 per column)
// Tensor memory: accumulator i in columns [i NT, (i + 1) NT), then the nab A buffers.
__host__ __device__ constexpr int mm_ta_col(int nt) { return MM_ACC * nt; }
__host__ __device__ constexpr uint32_t mm_tmem_cols(int nt, int nab)
{
    return MM_ACC * nt + nab * MM_TA_COLS <= 256 ? 256u : 512u;
}
constexpr int MM_LBO = 128;                    // bytes between core matrices adjacent along K
constexpr int MM_SBO = (MM_KC / 8) * 128;      // bytes between 8-row (8-token) groups
constexpr int DEVERR_TIMEOUT_MMA = 32;

__host__ __device__ constexpr int mm_b_bytes(int nt) { return nt * MM_KC * 2; }
// A ring slot: box_rows rows of MM_ROWB bytes, the slot start 128-byte aligned (tensor copy destination).
__host__ __device__ constexpr int mm_slot_bytes(int box_rows) { return (box_rows * MM_ROWB + 127) / 128 * 128; }
__host__ __device__ constexpr int mm_smem_bytes(int nt, int ns, int nab, int box_rows)
{
    return ns * mm_slot_bytes(box_rows) + nab * mm_b_bytes(nt) + 128;
}

struct MmArgs {
    CUtensorMap tmap;  // W as a 2-D array of 8-byte words [rows][row_bytes / 8], box MM_ROWB bytes x box_rows
    const float* X;    // [M][K]
    float* Y;          // [M][rows]
    int M, rows, K;
    int box_rows;      // rows one tensor copy brings (>= the rows of any tile of a block)
    int ns;            // ring slots (2 .. 4)
    int nab;           // operand buffers (2 .. 4): stages whose operands may be written ahead of the MMAs
    unsigned long long* trace;  // diagnostics: block 0's per-stage cycle stamps when not null
    int* err;
};

// 2-D tensor copy global -> shared of the box at (x bytes, y rows), completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                            uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}

// Byte offset of element (r, k) in a K-major core-matrix tile with MM_KC columns.
__device__ __forceinline__ int mm_off(int r, int k)
{
    return (r >> 3) * MM_SBO + (k >> 3) * MM_LBO + (r & 7) * 16 + (k & 7) * 2;
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// Four fp16 pairs from one word of codes t (bytes b0 b1 b2 b3, already permuted
// to b0 b2 b1 b3): weights from the low nibbles (b0, b1), (b2, b3) and the high
// nibbles (b0, b1), (b2, b3), each w = A q - B.
__device__ __forceinline__ void mm_dequant_word(uint32_t t, __half2 A, __half2 B, uint32_t& lo01, uint32_t& lo23,
                                                uint32_t& hi01, uint32_t& hi23)
{
    const __half2 k1024 = __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));
    const __half2 nb = __hneg2(B);
    // 0x6400 | q is the fp16 value 1024 + q: subtracting 1024 is exact
    const uint32_t q0 = (t & 0x000F000Fu) | 0x64006400u;
    const uint32_t q1 = ((t >> 8) & 0x000F000Fu) | 0x64006400u;
    const uint32_t q2 = ((t >> 4) & 0x000F000Fu) | 0x64006400u;
    const uint32_t q3 = ((t >> 12) & 0x000F000Fu) | 0x64006400u;
    lo01 = h2_bits(__hfma2(__hsub2(*reinterpret_cast<const __half2*>(&q0), k1024), A, nb));
    lo23 = h2_bits(__hfma2(__hsub2(*reinterpret_cast<const __half2*>(&q1), k1024), A, nb));
    hi01 = h2_bits(__hfma2(__hsub2(*reinterpret_cast<const __half2*>(&q2), k1024), A, nb));
    hi23 = h2_bits(__hfma2(__hsub2(*reinterpret_cast<const __half2*>(&q3), k1024), A, nb));
}

template <int NT>
__global__ void __launch_bounds__(MM_THREADS, 1) matmul_q4k_tc_kernel(const __grid_constant__ MmArgs a)
{
    extern __shared__ __align__(1024) uint8_t sm[];
    const int slot_bytes = mm_slot_bytes(a.box_rows);
    uint8_t* ring = sm;
    uint8_t* Bbuf = sm + a.ns * slot_bytes;
    const int nab = a.nab;
    uint64_t* full = reinterpret_cast<uint64_t*>(Bbuf + nab * mm_b_bytes(NT));  // [MM_NS_MAX] slot landed
    uint64_t* opready = full + MM_NS_MAX;                                       // [nab] operands of a stage written
    uint64_t* opfree = opready + MM_NAB_MAX;                                    // [nab] a stage's MMAs done
    uint32_t* tslot = reinterpret_cast<uint32_t*>(opfree + MM_NAB_MAX);
    volatile int* fail = reinterpret_cast<volatile int*>(tslot + 1);
    int* issued = const_cast<int*>(fail) + 1;   // one past the last block column issued (over the block's tiles)
    int* committed = issued + 1;                // one past the last stage committed

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, b = blockIdx.x;
    const int r0b = static_cast<int>(static_cast<long long>(b) * a.rows / G);
    const int r1b = static_cast<int>(static_cast<long long>(b + 1) * a.rows / G);
    if (r1b <= r0b)
        return;
    const int nblk = a.K / 256;

    if (warp == 0)
        tmem_alloc(tslot, mm_tmem_cols(NT, nab));
    if (tid == 0) {
        for (int s = 0; s < a.ns; ++s)
            mbar_init(&full[s], 1);
        for (int i = 0; i < nab; ++i) {
            mbar_init(&opready[i], MM_DQ_WARPS);
            mbar_init(&opfree[i], MM_NCTRL);
        }
        fence_mbar_init();
        *fail = 0;
        *issued = 0;
        *committed = 0;
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tbase = *tslot;

    // a bounded wait; false once this block has given up
    auto wait = [&](uint64_t* bar, uint32_t parity, int code) -> bool {
        if (*fail)
            return false;
        if (!mbar_wait(bar, parity)) {
            *fail = 1;
            set_error(a.err, code);
            return false;
        }
        return true;
    };
    // the same by a whole warp, with one outcome for all its lanes (tcgen05.ld/st are warp-collective)
    auto warp_wait = [&](uint64_t* bar, uint32_t parity, int code) -> bool {
        return __all_sync(0xffffffffu, wait(bar, parity, code)) != 0;
    };

    if (warp >= MM_CTRL) {
        // ---- control: the ring's copies (control warp 0) and the MMAs (one thread
        // of each control warp: the MMAs of accumulator cq)
        const int cq = warp - MM_CTRL;
        if (lane == 0) {
            constexpr uint32_t idesc = umma_idesc_f16_f32(MM_ROWS, NT);
            const uint64_t pol = l2_evict_first_policy();
            const int ngrp = (nblk + MM_BPS - 1) / MM_BPS;  // slot loads per tile
            int bg0 = 0, g0 = 0;
            bool ok = true;
            for (int rt0 = r0b; rt0 < r1b && ok; rt0 += MM_ROWS) {
                // block columns [4 q, 4 q + 4) of the tile's rows into a ring slot (box_rows >=
                // the tile's rows: extra rows are the next block's or zero fill, as are the
                // bytes past the end of a row)
                auto issue = [&](int q) {
                    const int bg = bg0 + q;
                    const int s = bg % a.ns;
                    mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(a.box_rows * MM_ROWB));
                    tma_load_2d(ring + s * slot_bytes, &a.tmap, q * (MM_BPS * Q4K_BYTES / 8), rt0, &full[s], pol);
                    *issued = bg + 1;
                };
                if (cq == 0)
                    for (int q = 0; q < min(a.ns, ngrp); ++q)
                        issue(q);
                for (int hc = 0; hc < nblk; ++hc) {
                    const int g = g0 + hc, buf = g % nab, c = hc;
                    if (!(ok = wait(&opready[buf], (g / nab) & 1, DEVERR_TIMEOUT_FULL)))
                        break;
                    unsigned long long* tr = (a.trace && b == 0 && cq == 0 && hc < 32) ? a.trace + 8 * hc : nullptr;
                    if (tr)
                        tr[0] = clock64();
                    tc_fence_after_sync();
                    const uint32_t ta = tbase + mm_ta_col(NT) + MM_TA_COLS * buf;
                    const uint64_t bd = umma_desc_kmajor(Bbuf + buf * mm_b_bytes(NT), MM_LBO, MM_SBO);
                    // K = 16 per MMA: 8 columns of A, two core matrices of B.  MMA s adds
                    // into accumulator s % MM_ACC, so consecutive MMAs do not wait on each other.
#pragma unroll
                    for (int s = 0; s < MM_KC / 16; ++s)
                        if (s % MM_NCTRL == cq)
                            umma_f16_ta(tbase + NT * (s % MM_ACC), ta + 8 * s,
                                        bd + static_cast<uint64_t>((2 * MM_LBO * s) >> 4), idesc,
                                        (hc > 0 || s >= MM_ACC) ? 1u : 0u);
                    umma_commit(&opfree[buf]);
                    if (cq == 0)
                        *committed = g + 1;
                    if (tr)
                        tr[1] = clock64();
                    // the last stage of a slot's block columns is dequantised: refill the slot
                    const int q = c / MM_BPS;
                    if (cq == 0 && (hc + 1 == nblk || (hc + 1) % MM_BPS == 0) && q + a.ns < ngrp)
                        issue(q + a.ns);
                }
                bg0 += ngrp;
                g0 += nblk;
            }
        }
        __syncwarp();  // the warp reconverges before the block-wide barrier below
    } else {
        // ---- dequantisation, activation staging and the epilogue (8 warps)
        constexpr int NDQ = 32 * MM_DQ_WARPS;
        constexpr int NXI = (NT * (MM_KC / 8) + NDQ - 1) / NDQ;  // activation items a thread stages
        const int ngrp = (nblk + MM_BPS - 1) / MM_BPS;
        int bg0 = 0, g0 = 0;
        for (int rt0 = r0b; rt0 < r1b; rt0 += MM_ROWS) {
            const int nrows = min(MM_ROWS, r1b - rt0);
            // the tokens' activations of stage hc + 1 are loaded while stage hc is
            // processed (item t = tid + 256 i: token t % NT, 8-element group t / NT)
            float4 xn[NXI][2];
            auto load_x = [&](int hcn) {
                const int kb = hcn * MM_KC;
#pragma unroll
                for (int i = 0; i < NXI; ++i) {
                    const int it = tid + NDQ * i;
                    const int n = it % NT, kg = it / NT;
                    if (it < NT * (MM_KC / 8) && n < a.M && hcn < nblk) {
                        const float4* xp =
                            reinterpret_cast<const float4*>(a.X + static_cast<size_t>(n) * a.K + kb + 8 * kg);
                        xn[i][0] = __ldg(xp);
                        xn[i][1] = __ldg(xp + 1);
                    }
                }
            };
            load_x(0);
            bool ok = true;
            for (int hc = 0; hc < nblk; ++hc) {
                const int c = hc;
                const int g = g0 + hc, buf = g % nab;
                const int bg = bg0 + c / MM_BPS;
                unsigned long long* tr = (a.trace && b == 0 && tid == 0 && hc < 32) ? a.trace + 8 * hc : nullptr;
                if (tr)
                    tr[2] = clock64();
                if (hc % MM_BPS == 0 && !(ok = warp_wait(&full[bg % a.ns], (bg / a.ns) & 1, DEVERR_TIMEOUT_FULL)))
                    break;
                if (tr)
                    tr[3] = clock64();
                if (g >= nab && !(ok = warp_wait(&opfree[buf], ((g - nab) / nab) & 1, DEVERR_TIMEOUT_MMA)))
                    break;
                if (tr)
                    tr[4] = clock64();
                uint8_t* Bt = Bbuf + buf * mm_b_bytes(NT);
                const uint8_t* slot = ring + (bg % a.ns) * slot_bytes + (c % MM_BPS) * Q4K_BYTES;
                // weights: thread (warp w, lane) dequantises row 32 (w % 4) + lane,
                // sub-blocks w / 4 and w / 4 + 4 of this block column, into the A buffer
                // in tensor memory (one lane per row, two fp16 per column; the four warps
                // of a lane quarter take the eight sub-blocks, two each, sharing the header)
                {
                    const int row = 32 * (warp & 3) + lane;
                    const uint32_t tcol = tbase + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + mm_ta_col(NT) +
                                          MM_TA_COLS * buf;
                    uint32_t v0[16], v1[16];
                    if (row < nrows) {
                        const uint8_t* bp = slot + row * MM_ROWB;
                        const uint4 hd = lds128(bp);
                        const float d = half_bits_to_float(hd.x), dmin = half_bits_to_float(hd.x >> 16);
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int j = (warp >> 2) + 4 * h;
                            const uint4 cw = lds128(bp + 16 + 16 * j);
                            const uint32_t s_lo = j < 6 ? hd.y : hd.z, s_hi = j < 6 ? hd.z : hd.w;
                            const uint32_t m_lo = j < 3 ? hd.z : hd.w, m_hi = j < 3 ? hd.w : 0u;
                            const int sc = static_cast<int>(__funnelshift_r(s_lo, s_hi, (6 * j) & 31) & 63u);
                            const int mn = static_cast<int>(__funnelshift_r(m_lo, m_hi, (48 + 6 * j) & 31) & 63u);
                            const __half2 A = __float2half2_rn(d * static_cast<float>(sc));
                            const __half2 B = __float2half2_rn(dmin * static_cast<float>(mn));
                            // byte i of the 16: low nibble weight 32j + i, high nibble weight
                            // 32j + 16 + i; column c of the sub-block holds weights 2c, 2c + 1
                            const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
                            uint32_t(&v)[16] = h ? v1 : v0;
#pragma unroll
                            for (int w = 0; w < 4; ++w) {
                                const uint32_t t = __byte_perm(words[w], 0u, 0x3120);  // b0 b2 b1 b3
                                mm_dequant_word(t, A, B, v[2 * w], v[2 * w + 1], v[8 + 2 * w], v[8 + 2 * w + 1]);
                            }
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            v0[i] = v1[i] = 0u;
                    }
                    tmem_st16(tcol + 16 * (warp >> 2), v0);
                    tmem_st16(tcol + 16 * ((warp >> 2) + 4), v1);
                }
                // activations: fp32 -> fp16 into the B buffer (consecutive threads take
                // consecutive tokens), then the next stage's loads
#pragma unroll
                for (int i = 0; i < NXI; ++i) {
                    const int it = tid + NDQ * i;
                    const int n = it % NT, kg = it / NT;
                    if (it < NT * (MM_KC / 8) && n < a.M) {
                        const float4 x0 = xn[i][0], x1 = xn[i][1];
                        const uint4 v = make_uint4(
                            h2_bits(__floats2half2_rn(x0.x, x0.y)), h2_bits(__floats2half2_rn(x0.z, x0.w)),
                            h2_bits(__floats2half2_rn(x1.x, x1.y)), h2_bits(__floats2half2_rn(x1.z, x1.w)));
                        *reinterpret_cast<uint4*>(Bt + mm_off(n, 8 * kg)) = v;
                    }
                }
                load_x(hc + 1);
                tmem_st_wait();
                fence_proxy_async_smem();
                tc_fence_before_sync();
                if (tr)
                    tr[5] = clock64();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&opready[buf]);  // release: this warp's part of stage g is written
            }
            if (!ok)
                break;
            // accumulator complete -> Y (warps 0-3: one lane quarter each)
            if (warp < 4) {
                const int glast = g0 + nblk - 1;
                if (!warp_wait(&opfree[glast % nab], (glast / nab) & 1, DEVERR_TIMEOUT_MMA))
                    break;
                tc_fence_after_sync();
                const int row = 32 * warp + lane;
#pragma unroll
                for (int cc = 0; cc < NT / 16; ++cc) {
                    float y[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        y[q] = 0.f;
#pragma unroll
                    for (int i = 0; i < MM_ACC; ++i) {  // the accumulators' sum, in a fixed order
                        uint32_t v[16];
                        tmem_ld16(tbase + (static_cast<uint32_t>(32 * warp) << 16) + NT * i + 16 * cc, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int q = 0; q < 16; ++q)
                            y[q] += __uint_as_float(v[q]);
                    }
                    if (row < nrows) {
#pragma unroll
                        for (int q = 0; q < 16; ++q) {
                            const int n = 16 * cc + q;
                            if (n < a.M)
                                a.Y[static_cast<size_t>(n) * a.rows + rt0 + row] = y[q];
                        }
                    }
                }
                // The next tile's first MMAs overwrite the accumulator only after this
                // warp's arrival on that tile's first stage, which follows these reads.
                tc_fence_before_sync();
            }
            bg0 += ngrp;
            g0 += nblk;
        }
    }
    // After a failed wait: let this block's copies and MMAs in flight finish (bounded).
    __syncthreads();
    if (tid == 0 && *fail) {
        const int hi = *issued, gc = *committed;
        for (int bg = max(0, hi - a.ns); bg < hi; ++bg) {
            const unsigned long long t0 = globaltimer_ns();
            while (!mbar_try_wait(&full[bg % a.ns], (bg / a.ns) & 1) && globaltimer_ns() - t0 < 100000000ull) {
            }
        }
        for (int g = max(0, gc - nab); g < gc; ++g) {
            const unsigned long long t0 = globaltimer_ns();
            while (!mbar_try_wait(&opfree[g % nab], (g / nab) & 1) && globaltimer_ns() - t0 < 100000000ull) {
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tbase, mm_tmem_cols(NT, nab));
    }
}

}  // namespace dq

namespace dqhost {

static int mm_nt(int M) { return M <= 16 ? 16 : M <= 32 ? 32 : 64; }

using EncodeTiled = PFN_cuTensorMapEncodeTiled_v12000;

static EncodeTiled encode_tiled()
{
    static std::once_flag once;
    static EncodeTiled fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
        cudaGetLastError();
    });
    return fn;
}

static int launch_matmul_tc(const uint8_t* W, const float* X, float* Y, int M, int rows, int K, cudaStream_t s)
{
    static std::once_flag once[3];
    static cudaError_t attr_err[3];
    const int nt = mm_nt(M);
    const int idx = nt == 16 ? 0 : nt == 32 ? 1 : 2;
    void (*k)(dq::MmArgs) = nt == 16 ? dq::matmul_q4k_tc_kernel<16>
                          : nt == 32 ? dq::matmul_q4k_tc_kernel<32>
                                     : dq::matmul_q4k_tc_kernel<64>;
    std::call_once(once[idx], [&] {
        attr_err[idx] = cudaFuncSetAttribute(reinterpret_cast<const void*>(k),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    });
    if (attr_err[idx] != cudaSuccess)
        return set_cuda_error(attr_err[idx]);
    EncodeTiled enc = encode_tiled();
    if (!enc)
        return DQ_ERR_UNSUPPORTED;
    const int grid = std::min(sm_count(), rows);
    const int per_block = (rows + grid - 1) / grid;
    dq::MmArgs a{};
    a.X = X;
    a.Y = Y;
    a.M = M;
    a.rows = rows;
    a.K = K;
    a.box_rows = std::min(dq::MM_ROWS, per_block);
    a.err = device_error_flag();
    a.trace = gemv_trace();
    // the deepest operand pipeline, then as many ring slots, as shared memory holds
    a.nab = 2;
    a.ns = 2;
    for (int nab = dq::MM_NAB_MAX; nab >= 2 && a.nab == 2; --nab)
        for (int ns = dq::MM_NS_MAX; ns >= 2; --ns)
            if (dq::mm_smem_bytes(nt, ns, nab, a.box_rows) <= 227 * 1024 &&
                dq::MM_ACC * nt + nab * dq::MM_TA_COLS <= 512) {  // tensor memory holds it
                a.nab = nab;
                a.ns = ns;
                break;
            }
    if (dq::mm_smem_bytes(nt, a.ns, a.nab, a.box_rows) > 227 * 1024)
        return DQ_ERR_UNSUPPORTED;
    const int smem = dq::mm_smem_bytes(nt, a.ns, a.nab, a.box_rows);
    const cuuint64_t row_bytes = static_cast<cuuint64_t>(K / 256) * dq::Q4K_BYTES;
    const cuuint64_t dims[2] = {row_bytes / 8, static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(dq::MM_ROWB / 8), static_cast<cuuint32_t>(a.box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&a.tmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<uint8_t*>(W), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return DQ_ERR_UNSUPPORTED;
    k<<<grid, dq::MM_THREADS, smem, s>>>(a);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DQ_OK : set_cuda_error(e);
}

}  // namespace dqhost

extern "C" {

DQ_API int dq_matmul_q4k_path(const void* W_blocks, const float* X, float* Y, int M, int rows, int K, int path,
                              void* stream)
{
    if (!W_blocks || !X || !Y)
        return DQ_ERR_NULL;
    if (M < 1 || M > 64 || rows < 1 || K < 256 || K % 256 || path < DQ_MATMUL_AUTO || path > DQ_MATMUL_TENSOR)
        return DQ_ERR_SHAPE;
    if (!dqhost::aligned16(W_blocks) || !dqhost::aligned16(X))
        return DQ_ERR_ALIGN;
    // measured crossover: one GEMV per token is faster up to M = 3
    const bool tensor = path == DQ_MATMUL_TENSOR || (path == DQ_MATMUL_AUTO && M >= 4);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (tensor)
        return dqhost::launch_matmul_tc(static_cast<const uint8_t*>(W_blocks), X, Y, M, rows, K, s);
    if (K > 16384)
        return DQ_ERR_UNSUPPORTED;
    dqhost::GemvPlan plan;
    int st = dqhost::plan_gemv(DQ_FMT_Q4K, rows, K, 1, 1, false, &plan);
    if (st != DQ_OK)
        return st;
    for (int m = 0; m < M; ++m) {
        dq::GemvArgs a{};
        a.W = static_cast<const uint8_t*>(W_blocks);
        a.pro = dq::PRO_F32;
        a.x = X + static_cast<size_t>(m) * K;
        a.epi = dq::EPI_STORE;
        a.y = Y + static_cast<size_t>(m) * rows;
        // dependent launches: the first may follow a kernel that writes W (only L2
        // prefetches before its wait); the later ones follow this loop's own GEMVs,
        // which do not, so their first copies leave before the wait
        a.w_late = m == 0 ? 1 : 0;
        cudaError_t e = dqhost::launch_gemv(plan, a, s, true);
        if (e != cudaSuccess)
            return dqhost::set_cuda_error(e);
    }
    return DQ_OK;
}

DQ_API int dq_matmul_q4k(const void* W_blocks, const float* X, float* Y, int M, int rows, int K, void* stream)
{
    return dq_matmul_q4k_path(W_blocks, X, Y, M, rows, K, DQ_MATMUL_AUTO, stream);
}

}  // extern "C"
