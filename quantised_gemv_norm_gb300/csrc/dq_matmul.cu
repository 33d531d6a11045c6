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
constexpr int MM_ROWB = Q4K_BYTES;             // a slot row: one block (the 144-byte stride puts the
                                               // 16-byte header loads of 8 rows on distinct banks)
constexpr int MM_NS_MAX = 8;
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
// xs: the activations arrive staged (fp16, UMMA layout) with each slot's weights,
// so a slot holds the weights and the stage's B tile and there are no B buffers.
__host__ __device__ constexpr int mm_smem_bytes(int nt, int ns, int nab, int box_rows, bool xs)
{
    return xs ? ns * (mm_slot_bytes(box_rows) + mm_b_bytes(nt)) + 128
              : ns * mm_slot_bytes(box_rows) + nab * mm_b_bytes(nt) + 128;
}

struct MmArgs {
    CUtensorMap tmap;  // W as a 2-D array of 8-byte words [rows][row_bytes / 8], box MM_ROWB bytes x box_rows
    const float* X;    // [M][K]
    float* Y;          // [M][rows]
    int M, rows, K;
    int box_rows;      // rows one tensor copy brings (>= the rows of any tile)
    int ns;            // ring slots (2 .. MM_NS_MAX), one block column each
    int nab;           // operand buffers (2 .. 4): stages whose operands may be written ahead of the MMAs
    // K split (cnt not null): the stages (128-row tile, block column) are shared out
    // in contiguous runs; a tile's partial sums meet in `part`, summed by the block
    // that completes the tile's count in `cnt` (which it leaves at zero again)
    unsigned* cnt;     // [row tiles][4 lane quarters]
    float* part;       // [blocks][2][M][128]: a block's first and last partial tile
    // the activations already in fp16 B tiles (mm_stage_x_kernel: [K / 256][NT tokens x
    // 256] in the UMMA K-major layout), copied with the weights; null: the
    // dequantising warps stage them from X each stage
    const uint8_t* xh;
    unsigned long long* trace;  // diagnostics: block 0's per-stage cycle stamps when not null
    int* err;
};

// Segment i of block b (a tile's rows and the block columns [c0, c1) of them that
// the block takes); false past the block's last.  Without a K split a block takes
// whole rows (a contiguous share of the rows, in tiles of at most 128), with it a
// contiguous run of the stages numbered tile-major.
struct MmSeg {
    int rt, row0, nrows, c0, c1;
};
__device__ __forceinline__ bool mm_seg(const MmArgs& a, int b, int G, int i, MmSeg& sg)
{
    const int nblk = a.K / 256;
    if (!a.cnt) {
        const int r0b = static_cast<int>(static_cast<long long>(b) * a.rows / G);
        const int r1b = static_cast<int>(static_cast<long long>(b + 1) * a.rows / G);
        const int row0 = r0b + MM_ROWS * i;
        if (row0 >= r1b)
            return false;
        sg = MmSeg{i, row0, min(MM_ROWS, r1b - row0), 0, nblk};
        return true;
    }
    const long long S = static_cast<long long>((a.rows + MM_ROWS - 1) / MM_ROWS) * nblk;
    const long long s0 = S * b / G, s1 = S * (b + 1) / G;
    const long long rt = s0 / nblk + i;
    if (rt * nblk >= s1)
        return false;
    sg.rt = static_cast<int>(rt);
    sg.row0 = sg.rt * MM_ROWS;
    sg.nrows = min(MM_ROWS, a.rows - sg.row0);
    sg.c0 = static_cast<int>(max(s0, rt * nblk) - rt * nblk);
    sg.c1 = static_cast<int>(min(s1, (rt + 1) * nblk) - rt * nblk);
    return true;
}

// The block whose run of stages holds stage s (K split).
__device__ __forceinline__ int mm_block_of(long long s, long long S, int G)
{
    return static_cast<int>(((s + 1) * G - 1) / S);
}

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

__device__ __forceinline__ uint64_t l2_evict_last_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v)
{
    unsigned old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Four fp16 pairs from one word of codes t (bytes b0 b1 b2 b3, already permuted
// to b0 b2 b1 b3): weights from the low nibbles (b0, b1), (b2, b3) and the high
// nibbles (b0, b1), (b2, b3), each w = A q - B.  A low nibble q in mantissa bits
// 0-3 under 0x6400 is the fp16 value 1024 + q; a high nibble left in bits 4-7
// under 0x5400 (64.0, whose mantissa step is 1/16) is 64 + q: one mask and or
// per pair and one shift per word, and the subtractions are exact.
__device__ __forceinline__ void mm_dequant_word(uint32_t t, __half2 A, __half2 B, uint32_t& lo01, uint32_t& lo23,
                                                uint32_t& hi01, uint32_t& hi23)
{
    const __half2 k1024 = __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));
    const __half2 k64 = __halves2half2(__ushort_as_half(0x5400), __ushort_as_half(0x5400));
    const __half2 nb = __hneg2(B);
    const uint32_t t8 = t >> 8;  // b2, b3 in the low bytes of the halves (b1's bits above are masked off)
    const uint32_t q0 = (t & 0x000F000Fu) | 0x64006400u;
    const uint32_t q1 = (t8 & 0x000F000Fu) | 0x64006400u;
    const uint32_t q2 = (t & 0x00F000F0u) | 0x54005400u;
    const uint32_t q3 = (t8 & 0x00F000F0u) | 0x54005400u;
    lo01 = h2_bits(__hfma2(__hsub2(*reinterpret_cast<const __half2*>(&q0), k1024), A, nb));
    lo23 = h2_bits(__hfma2(__hsub2(*reinterpret_cast<const __half2*>(&q1), k1024), A, nb));
    hi01 = h2_bits(__hfma2(__hsub2(*reinterpret_cast<const __half2*>(&q2), k64), A, nb));
    hi23 = h2_bits(__hfma2(__hsub2(*reinterpret_cast<const __half2*>(&q3), k64), A, nb));
}

template <int NT>
__global__ void __launch_bounds__(MM_THREADS, 1) matmul_q4k_tc_kernel(const __grid_constant__ MmArgs a)
{
    extern __shared__ __align__(1024) uint8_t sm[];
    const bool xs = a.xh != nullptr;  // each slot: weights, then the stage's B tile
    const int wslot = mm_slot_bytes(a.box_rows);
    const int slot_bytes = wslot + (xs ? mm_b_bytes(NT) : 0);
    uint8_t* ring = sm;
    uint8_t* Bbuf = sm + a.ns * slot_bytes;
    const int nab = a.nab;
    uint64_t* full = reinterpret_cast<uint64_t*>(Bbuf + (xs ? 0 : nab * mm_b_bytes(NT)));  // [MM_NS_MAX] slot landed
    uint64_t* opready = full + MM_NS_MAX;                                       // [nab] operands of a stage written
    uint64_t* opfree = opready + MM_NAB_MAX;                                    // [nab] a stage's MMAs done
    uint32_t* tslot = reinterpret_cast<uint32_t*>(opfree + MM_NAB_MAX);
    volatile int* fail = reinterpret_cast<volatile int*>(tslot + 1);
    int* issued = const_cast<int*>(fail) + 1;   // one past the last stage whose copy was issued
    int* committed = issued + 1;                // one past the last stage committed

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, b = blockIdx.x;
    const int nblk = a.K / 256;
    unsigned long long* btr = a.trace ? a.trace + 256 + 4 * b : nullptr;  // this block's timeline
    if (btr && tid == 0)
        btr[0] = globaltimer_ns();
    MmSeg sg0;
    if (!mm_seg(a, b, G, 0, sg0))
        return;

    pdl_trigger();
    if (warp == 0)
        tmem_alloc(tslot, mm_tmem_cols(NT, nab));
    if (tid == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.tmap)) : "memory");
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
    // a dependent launch: the set-up above overlaps the previous kernel's tail.  The
    // first ring-full of weights is only asked into L2 before the wait (a later write
    // by the previous kernel lands in L2 as well, so no stale copy can result); every
    // other global access (the copies, activations, outputs, workspace) follows it.
    if (warp == MM_CTRL && lane == 0) {
        MmSeg q = sg0;
        int i = 0, col = sg0.c0;
        for (int gi = 0; gi < a.ns; ++gi) {
            asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                             reinterpret_cast<uint64_t>(&a.tmap)),
                         "r"(col * (Q4K_BYTES / 8)), "r"(q.row0)
                         : "memory");
            if (++col == q.c1) {
                if (!mm_seg(a, b, G, ++i, q))
                    break;
                col = q.c0;
            }
        }
    }
    pdl_wait();

    // a bounded wait; false once this block has given up
    auto wait = [&](uint64_t* bar, uint32_t parity, int code) -> bool {
        if (mbar_try_wait(bar, parity))
            return true;  // complete: the block's failure flag matters only for a wait that blocks
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
        // of each control warp: the MMAs of accumulator cq).  The block's stages are
        // numbered g = 0, 1, ... over its segments; stage g uses ring slot g % ns.
        const int cq = warp - MM_CTRL;
        if (lane == 0) {
            constexpr uint32_t idesc = umma_idesc_f16_f32(MM_ROWS, NT);
            const uint64_t pol = l2_evict_first_policy();
            int total = 0;
            MmSeg sg;
            for (int i = 0; mm_seg(a, b, G, i, sg); ++i)
                total += sg.c1 - sg.c0;
            // the next stage to copy: segment iseg, block column icol
            MmSeg isg = sg0;
            int iseg = 0, icol = sg0.c0, gnext = 0, islot = 0;  // islot = gnext % ns
            // one block column of a tile's rows into slot gnext % ns (box_rows >= the
            // tile's rows: extra rows are the next tile's or zero fill).  Stage and slot
            // indices advance by counters: a division by the run-time ring or buffer
            // count costs tens of instructions.
            const uint64_t pol_x = l2_evict_last_policy();  // every block reads the B tiles
            auto issue_next = [&]() {
                const int s = islot;
                if (++islot == a.ns)
                    islot = 0;
                mbar_arrive_expect_tx(&full[s],
                                      static_cast<uint32_t>(a.box_rows * MM_ROWB + (xs ? mm_b_bytes(NT) : 0)));
                tma_load_2d(ring + s * slot_bytes, &a.tmap, icol * (Q4K_BYTES / 8), isg.row0, &full[s], pol);
                if (xs)
                    bulk_g2s(ring + s * slot_bytes + wslot, a.xh + static_cast<size_t>(icol) * mm_b_bytes(NT),
                             mm_b_bytes(NT), &full[s], pol_x);
                *issued = ++gnext;
                if (++icol == isg.c1 && mm_seg(a, b, G, ++iseg, isg))
                    icol = isg.c0;
            };
            if (cq == 0)
                while (gnext < min(a.ns, total))
                    issue_next();
            int g = 0;
            int buf = 0, slot = 0, pbuf = nab - 1;  // g % nab, g % ns, (g - 1) % nab
            uint32_t bph = 0, pbph = 1;            // (g / nab) & 1, ((g - 1) / nab) & 1
            bool ok = true;
            for (int i = 0; ok && mm_seg(a, b, G, i, sg); ++i) {
                for (int hc = sg.c0; hc < sg.c1; ++hc, ++g) {
                    if (!(ok = wait(&opready[buf], bph, DEVERR_TIMEOUT_FULL)))
                        break;
                    unsigned long long* tr = (a.trace && b == 0 && cq == 0 && g < 32) ? a.trace + 8 * g : nullptr;
                    if (tr)
                        tr[0] = clock64();
                    tc_fence_after_sync();
                    const uint32_t ta = tbase + mm_ta_col(NT) + MM_TA_COLS * buf;
                    const uint64_t bd = umma_desc_kmajor(
                        xs ? ring + slot * slot_bytes + wslot : Bbuf + buf * mm_b_bytes(NT), MM_LBO, MM_SBO);
                    // K = 16 per MMA: 8 columns of A, two core matrices of B.  MMA s adds
                    // into accumulator s % MM_ACC, so consecutive MMAs do not wait on each
                    // other; the segment's first stage starts the accumulators afresh.
#pragma unroll
                    for (int s = 0; s < MM_KC / 16; ++s)
                        if (s % MM_NCTRL == cq)
                            umma_f16_ta(tbase + NT * (s % MM_ACC), ta + 8 * s,
                                        bd + static_cast<uint64_t>((2 * MM_LBO * s) >> 4), idesc,
                                        (hc > sg.c0 || s >= MM_ACC) ? 1u : 0u);
                    umma_commit(&opfree[buf]);
                    if (cq == 0)
                        *committed = g + 1;
                    if (tr)
                        tr[1] = clock64();
                    if (!xs) {
                        // stage g's slot is free (every dequantising warp read it before its
                        // opready arrival): the copy of stage g + ns goes into it
                        if (cq == 0 && g + a.ns < total)
                            issue_next();
                    } else if (cq == 0 && g >= 1 && g - 1 + a.ns < total) {
                        // the MMAs read the B tile from the slot: stage g - 1's slot is free
                        // once its MMAs are done (committed one stage ago)
                        if (!(ok = wait(&opfree[pbuf], pbph, DEVERR_TIMEOUT_MMA)))
                            break;
                        issue_next();
                    }
                    pbuf = buf;
                    pbph = bph;
                    if (++buf == nab) {
                        buf = 0;
                        bph ^= 1u;
                    }
                    if (++slot == a.ns)
                        slot = 0;
                }
            }
        }
        __syncwarp();  // the warp reconverges before the block-wide barrier below
    } else {
        // ---- dequantisation, activation staging and the epilogue (16 warps)
        constexpr int NDQ = 32 * MM_DQ_WARPS;
        constexpr int NXI = (NT * (MM_KC / 8) + NDQ - 1) / NDQ;  // activation items a thread stages
        // the tokens' activations of the next stage are loaded while a stage is
        // processed (item t = tid + NDQ i: token t % NT, 8-element group t / NT)
        float4 xn[NXI][2];
        auto load_x = [&](int hcn) {
            const int kb = hcn * MM_KC;
#pragma unroll
            for (int i = 0; i < NXI; ++i) {
                const int it = tid + NDQ * i;
                const int n = it % NT, kg = it / NT;
                if (it < NT * (MM_KC / 8) && n < a.M && hcn >= 0 && hcn < nblk) {
                    const float4* xp =
                        reinterpret_cast<const float4*>(a.X + static_cast<size_t>(n) * a.K + kb + 8 * kg);
                    xn[i][0] = __ldg(xp);
                    xn[i][1] = __ldg(xp + 1);
                }
            }
        };
        if (!xs)
            load_x(sg0.c0);
        int g = 0;
        int dbuf = 0, dslot = 0;      // g % nab, g % ns
        uint32_t dbph = 0, dsph = 0;  // (g / nab) & 1, (g / ns) & 1
        bool ok = true;
        MmSeg sg;
        for (int si = 0; ok && mm_seg(a, b, G, si, sg); ++si) {
            const int nrows = sg.nrows;
            MmSeg nx;
            const int next_c0 = mm_seg(a, b, G, si + 1, nx) ? nx.c0 : -1;
            for (int hc = sg.c0; hc < sg.c1; ++hc, ++g) {
                const int buf = dbuf, s = dslot;
                unsigned long long* tr = (a.trace && b == 0 && tid == 0 && g < 32) ? a.trace + 8 * g : nullptr;
                if (tr)
                    tr[2] = clock64();
                if (!(ok = warp_wait(&full[s], dsph, DEVERR_TIMEOUT_FULL)))
                    break;
                if (tr)
                    tr[3] = clock64();
                if (btr && g == 0 && tid == 0)
                    btr[1] = globaltimer_ns();
                // stage g - nab's MMAs (buffer buf, one use earlier) are done
                if (g >= nab && !(ok = warp_wait(&opfree[buf], dbph ^ 1u, DEVERR_TIMEOUT_MMA)))
                    break;
                if (tr)
                    tr[4] = clock64();
                uint8_t* Bt = Bbuf + buf * mm_b_bytes(NT);
                const uint8_t* slot = ring + s * slot_bytes;
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
                // consecutive tokens), then the next stage's loads (unless staged already)
                if (!xs) {
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
                    load_x(hc + 1 < sg.c1 ? hc + 1 : next_c0);
                }
                tmem_st_wait();
                fence_proxy_async_smem();
                tc_fence_before_sync();
                if (tr)
                    tr[5] = clock64();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&opready[buf]);  // release: this warp's part of stage g is written
                if (++dbuf == nab) {
                    dbuf = 0;
                    dbph ^= 1u;
                }
                if (++dslot == a.ns) {
                    dslot = 0;
                    dsph ^= 1u;
                }
            }
            if (!ok)
                break;
            // accumulator complete (warps 0-3: one lane quarter each) -> Y, or, for a
            // tile whose block columns other blocks share, -> this block's partial tile
            if (warp < 4) {
                const int glast = g - 1;
                if (!warp_wait(&opfree[glast % nab], (glast / nab) & 1, DEVERR_TIMEOUT_MMA))
                    break;
                tc_fence_after_sync();
                if (btr && tid == 0)
                    btr[2] = globaltimer_ns();
                const int row = 32 * warp + lane;
                const bool whole = sg.c0 == 0 && sg.c1 == nblk;
                float* dst = whole ? a.Y + sg.row0 + row
                                   : a.part + (static_cast<size_t>(2 * b + (si == 0 ? 0 : 1)) * a.M) * MM_ROWS + row;
                const size_t dstride = whole ? static_cast<size_t>(a.rows) : static_cast<size_t>(MM_ROWS);
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
                                dst[n * dstride] = y[q];
                        }
                    }
                }
                // The next segment's first MMAs overwrite the accumulator only after this
                // warp's arrival on that segment's first stage, which follows these reads.
                tc_fence_before_sync();
                if (!whole) {
                    // this warp's 32 rows of the partial tile are written: count them
                    // (one count per tile and lane quarter, so the four warps never wait
                    // on each other); the warp that completes a count sums the quarter's
                    // partials in block order (the same order whichever block comes
                    // last) and leaves the count at zero
                    const long long S = static_cast<long long>((a.rows + MM_ROWS - 1) / MM_ROWS) * nblk;
                    const long long t0 = static_cast<long long>(sg.rt) * nblk;
                    const int b_lo = mm_block_of(t0, S, G), b_hi = mm_block_of(t0 + nblk - 1, S, G);
                    const int which_lo = S * b_lo / G == t0 ? 0 : 1;
                    unsigned* cnt = a.cnt + 4 * sg.rt + warp;
                    // the warp barrier orders the lanes' stores before lane 0's release
                    // (cumulative), and lane 0's acquire before the lanes' loads
                    __syncwarp();
                    unsigned done = 0;
                    if (lane == 0)
                        done = atom_add_acq_rel_gpu(cnt, 1u) == static_cast<unsigned>(b_hi - b_lo) ? 1u : 0u;
                    done = __shfl_sync(0xffffffffu, done, 0);
                    __syncwarp();
                    if (done) {
                        if (row < nrows)
                            for (int n0 = 0; n0 < a.M; n0 += 16) {  // 16 tokens' loads in flight at once
                                float y[16];
#pragma unroll
                                for (int q = 0; q < 16; ++q)
                                    y[q] = 0.f;
                                for (int bb = b_lo; bb <= b_hi; ++bb) {
                                    // block bb's partial of this tile: the later blocks' runs start
                                    // in it (their first segment); block b_lo's run starts in it
                                    // only when it starts at its column 0
                                    const int which = bb == b_lo ? which_lo : 0;
                                    const float* pp =
                                        a.part + (static_cast<size_t>(2 * bb + which) * a.M + n0) * MM_ROWS + row;
                                    float v[16];
#pragma unroll
                                    for (int q = 0; q < 16; ++q)
                                        v[q] = n0 + q < a.M ? __ldcg(pp + q * MM_ROWS) : 0.f;
#pragma unroll
                                    for (int q = 0; q < 16; ++q)
                                        y[q] += v[q];
                                }
#pragma unroll
                                for (int q = 0; q < 16; ++q)
                                    if (n0 + q < a.M)
                                        a.Y[static_cast<size_t>(n0 + q) * a.rows + sg.row0 + row] = y[q];
                            }
                        if (lane == 0)
                            atomicExch(cnt, 0u);
                    }
                }
            }
        }
    }
    // After a failed wait: let this block's copies and MMAs in flight finish (bounded).
    __syncthreads();
    if (tid == 0 && *fail) {
        const int hi = *issued, gc = *committed;
        for (int gi = max(0, hi - a.ns); gi < hi; ++gi) {
            const unsigned long long t0 = globaltimer_ns();
            while (!mbar_try_wait(&full[gi % a.ns], (gi / a.ns) & 1) && globaltimer_ns() - t0 < 100000000ull) {
            }
        }
        for (int gi = max(0, gc - nab); gi < gc; ++gi) {
            const unsigned long long t0 = globaltimer_ns();
            while (!mbar_try_wait(&opfree[gi % nab], (gi / nab) & 1) && globaltimer_ns() - t0 < 100000000ull) {
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tbase, mm_tmem_cols(NT, nab));
    }
    if (btr && tid == 0)
        btr[3] = globaltimer_ns();
}

// The M tokens' activations as fp16 B tiles, one per block column: item (column hc,
// token n, 8-element group kg) converts X[n][256 hc + 8 kg .. + 8) and stores it at
// mm_off(n, 8 kg) of tile hc; tokens n >= M are zero.  A dependent launch: it waits
// for X's producer, and the product launched after it waits for it.
template <int NT>
__global__ void __launch_bounds__(256) mm_stage_x_kernel(const float* __restrict__ X, uint8_t* __restrict__ xh, int M,
                                                         int K)
{
    pdl_trigger();
    pdl_wait();
    const int it = blockIdx.x * 256 + threadIdx.x;
    const int nblk = K / 256;
    if (it >= nblk * NT * (MM_KC / 8))
        return;
    const int hc = it / (NT * (MM_KC / 8)), rem = it - hc * NT * (MM_KC / 8);
    const int n = rem % NT, kg = rem / NT;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (n < M) {
        const float4* xp = reinterpret_cast<const float4*>(X + static_cast<size_t>(n) * K + hc * MM_KC + 8 * kg);
        const float4 x0 = xp[0], x1 = xp[1];
        v = make_uint4(h2_bits(__floats2half2_rn(x0.x, x0.y)), h2_bits(__floats2half2_rn(x0.z, x0.w)),
                       h2_bits(__floats2half2_rn(x1.x, x1.y)), h2_bits(__floats2half2_rn(x1.z, x1.w)));
    }
    *reinterpret_cast<uint4*>(xh + static_cast<size_t>(hc) * mm_b_bytes(NT) + mm_off(n, 8 * kg)) = v;
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

// Workspace of the K-split product: the tiles' counts (zero between calls), then
// the blocks' partial tiles.
static long long split_grid(int rows, int K)
{
    const long long S = static_cast<long long>((rows + dq::MM_ROWS - 1) / dq::MM_ROWS) * (K / 256);
    return std::min<long long>(sm_count(), S);
}
// The counts take a fixed region (four per 128-row tile, room for 4096 tiles) so
// that no shape's partial tiles ever overlap another shape's counts: one workspace
// serves calls of any shapes that fit it.
constexpr size_t SPLIT_CNT_BYTES = 65536;
constexpr int SPLIT_MAX_ROWS = static_cast<int>(SPLIT_CNT_BYTES / 16) * dq::MM_ROWS;
// Above 16 tokens the activations are staged once as fp16 B tiles (after the counts)
// and copied with the weights; up to 16 the dequantising warps stage them (measured
// on 12288 x 4096: 64 tokens 36.4 -> 33.0 us, 32 tokens 29.7 -> 27.2 us).
static bool split_staged_x(int M) { return mm_nt(M) >= 32; }
static size_t split_xh_bytes(int M, int K)
{
    return split_staged_x(M) ? static_cast<size_t>(K / 256) * dq::mm_b_bytes(mm_nt(M)) : 0;
}
static size_t split_ws_bytes(int M, int rows, int K)
{
    return SPLIT_CNT_BYTES + split_xh_bytes(M, K) + static_cast<size_t>(split_grid(rows, K)) * 2 * M * dq::MM_ROWS * 4;
}

static int launch_matmul_tc(const uint8_t* W, const float* X, float* Y, int M, int rows, int K, void* ws,
                            cudaStream_t s)
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
    const int grid = ws ? static_cast<int>(split_grid(rows, K)) : std::min(sm_count(), rows);
    const int per_block = (rows + grid - 1) / grid;
    dq::MmArgs a{};
    a.X = X;
    a.Y = Y;
    a.M = M;
    a.rows = rows;
    a.K = K;
    a.box_rows = std::min(dq::MM_ROWS, ws ? rows : per_block);
    if (ws) {
        a.cnt = static_cast<unsigned*>(ws);
        if (split_staged_x(M))
            a.xh = static_cast<uint8_t*>(ws) + SPLIT_CNT_BYTES;
        a.part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + SPLIT_CNT_BYTES + split_xh_bytes(M, K));
    }
    const bool xs = a.xh != nullptr;
    a.err = device_error_flag();
    a.trace = gemv_trace();
    // the deepest operand pipeline, then as many ring slots, as shared memory holds
    a.nab = 2;
    a.ns = 2;
    for (int nab = dq::MM_NAB_MAX; nab >= 2 && a.nab == 2; --nab)
        for (int ns = dq::MM_NS_MAX; ns >= 2; --ns)
            if (dq::mm_smem_bytes(nt, ns, nab, a.box_rows, xs) <= 227 * 1024 &&
                dq::MM_ACC * nt + nab * dq::MM_TA_COLS <= 512) {  // tensor memory holds it
                a.nab = nab;
                a.ns = ns;
                break;
            }
    if (dq::mm_smem_bytes(nt, a.ns, a.nab, a.box_rows, xs) > 227 * 1024)
        return DQ_ERR_UNSUPPORTED;
    const int smem = dq::mm_smem_bytes(nt, a.ns, a.nab, a.box_rows, xs);
    const cuuint64_t row_bytes = static_cast<cuuint64_t>(K / 256) * dq::Q4K_BYTES;
    const cuuint64_t dims[2] = {row_bytes / 8, static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(dq::MM_ROWB / 8), static_cast<cuuint32_t>(a.box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&a.tmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<uint8_t*>(W), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return DQ_ERR_UNSUPPORTED;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (xs) {  // the fp16 B tiles first (a dependent launch of its own)
        const int items = (K / 256) * nt * (dq::MM_KC / 8);
        cfg.gridDim = dim3((items + 255) / 256);
        cfg.blockDim = dim3(256);
        cfg.dynamicSmemBytes = 0;
        void (*sx)(const float*, uint8_t*, int, int) = nt == 32 ? dq::mm_stage_x_kernel<32> : dq::mm_stage_x_kernel<64>;
        e = cudaLaunchKernelEx(&cfg, sx, X, const_cast<uint8_t*>(a.xh), M, K);
        if (e != cudaSuccess)
            return set_cuda_error(e);
    }
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(dq::MM_THREADS);
    cfg.dynamicSmemBytes = smem;
    e = cudaLaunchKernelEx(&cfg, k, a);
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
    // measured crossover on 12288 x 4096: one GEMV per token is faster up to M = 2
    // (9.3 / 17.7 / about 26 us for M = 1 / 2 / 3 against 21.8 on the tensor cores)
    const bool tensor = path == DQ_MATMUL_TENSOR || (path == DQ_MATMUL_AUTO && M >= 3);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (tensor)
        return dqhost::launch_matmul_tc(static_cast<const uint8_t*>(W_blocks), X, Y, M, rows, K, nullptr, s);
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

DQ_API long long dq_matmul_q4k_split_workspace_bytes(int M, int rows, int K)
{
    if (M < 1 || M > 64 || rows < 1 || K < 256 || K % 256)
        return DQ_ERR_SHAPE;
    if (rows > dqhost::SPLIT_MAX_ROWS)
        return DQ_ERR_UNSUPPORTED;
    return static_cast<long long>(dqhost::split_ws_bytes(M, rows, K));
}

DQ_API int dq_matmul_q4k_split(const void* W_blocks, const float* X, float* Y, int M, int rows, int K,
                               void* workspace, long long workspace_bytes, void* stream)
{
    if (!W_blocks || !X || !Y || !workspace)
        return DQ_ERR_NULL;
    if (M < 1 || M > 64 || rows < 1 || K < 256 || K % 256)
        return DQ_ERR_SHAPE;
    if (!dqhost::aligned16(W_blocks) || !dqhost::aligned16(X) || !dqhost::aligned16(workspace))
        return DQ_ERR_ALIGN;
    if (rows > dqhost::SPLIT_MAX_ROWS)
        return DQ_ERR_UNSUPPORTED;
    if (workspace_bytes < static_cast<long long>(dqhost::split_ws_bytes(M, rows, K)))
        return DQ_ERR_SHAPE;
    return dqhost::launch_matmul_tc(static_cast<const uint8_t*>(W_blocks), X, Y, M, rows, K, workspace,
                                    static_cast<cudaStream_t>(stream));
}

}  // extern "C"
