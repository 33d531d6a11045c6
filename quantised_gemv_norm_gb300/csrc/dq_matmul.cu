// dq_matmul.cu -- Y[m] = W X[m] for M token vectors over one Q4_K matrix.
//
// "The roofline holds on a second GPU", section "The Math": M tokens processed
// together share one read of the weights until the arithmetic catches up, at
// M* = (w / 16) (R / BW).  Two paths:
//
//   * CUDA cores: the single-vector streaming GEMV once per token (reads the
//     weights M times; the M = 1 path and the comparison point);
//   * tensor cores (M >= 2): every weight is read once for all M tokens.  Each
//     block takes a contiguous range of rows (at most 128 per tile) and walks
//     K in Q4_K block columns: the blocks' bytes stream into a shared-memory
//     ring with 1-D bulk copies, all threads dequantise one half block (128 K)
//     at a time to fp16 in the UMMA K-major core-matrix layout, the tokens'
//     activations are staged beside it as fp16, and one thread issues eight
//     tcgen05.mma (M = 128, N = tokens rounded up to 16, K = 16) accumulating
//     in fp32 in tensor memory.  Dequantisation of the next half block
//     overlaps the MMAs of the current one (double-buffered operands; the
//     MMAs' commit releases a buffer).  The epilogue reads the accumulator
//     with tcgen05.ld and writes Y.
//
// fp16 and not bf16 operands: a dequantised Q4_K weight d sc q - dmin m has up
// to 21 significant bits; fp16 keeps 11 (relative error 2^-12 per weight,
// about 1e-4 normwise on a row), bf16 only 8 (about 1e-3, half the tolerance).
#include <mutex>

#include "dq_gemv_host.h"
#include "dq_tc.cuh"

namespace dq {

constexpr int MM_THREADS = 256;
constexpr int MM_ROWS = 128;                   // rows per tile = UMMA M
constexpr int MM_KC = 128;                     // K per MMA stage: half a Q4_K block
constexpr int MM_NS = 4;                       // ring slots, one Q4_K block column of the tile's rows each
constexpr int MM_SLOT = MM_ROWS * Q4K_BYTES;   // 18432 bytes
constexpr int MM_A_BYTES = MM_ROWS * MM_KC * 2;
constexpr int MM_LBO = 128;                    // bytes between core matrices adjacent along K
constexpr int MM_SBO = (MM_KC / 8) * 128;      // bytes between 8-row (8-token) groups
constexpr int DEVERR_TIMEOUT_MMA = 32;

__host__ __device__ constexpr int mm_b_bytes(int nt) { return nt * MM_KC * 2; }
__host__ __device__ constexpr int mm_smem_bytes(int nt) { return MM_NS * MM_SLOT + 2 * MM_A_BYTES + 2 * mm_b_bytes(nt) + 128; }

struct MmArgs {
    const uint8_t* W;  // Q4_K rows of row_bytes
    const float* X;    // [M][K]
    float* Y;          // [M][rows]
    int M, rows, K;
    int* err;
};

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
    uint8_t* ring = sm;
    uint8_t* Abuf = sm + MM_NS * MM_SLOT;
    uint8_t* Bbuf = Abuf + 2 * MM_A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(Bbuf + 2 * mm_b_bytes(NT));  // [MM_NS]
    uint64_t* mmad = full + MM_NS;                                            // [2]: buffer's MMAs done
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mmad + 2);
    volatile int* fail = reinterpret_cast<volatile int*>(tslot + 1);
    int* issued = const_cast<int*>(fail) + 1;   // one past the last block column issued (over the block's tiles)
    int* committed = issued + 1;                // one past the last half-chunk committed

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, b = blockIdx.x;
    const int r0b = static_cast<int>(static_cast<long long>(b) * a.rows / G);
    const int r1b = static_cast<int>(static_cast<long long>(b + 1) * a.rows / G);
    if (r1b <= r0b)
        return;
    const int nblk = a.K / 256;
    const size_t row_bytes = static_cast<size_t>(nblk) * Q4K_BYTES;
    constexpr uint32_t NCOLS = NT < 32 ? 32 : NT;
    const uint64_t pol = l2_evict_first_policy();

    if (warp == 0)
        tmem_alloc(tslot, NCOLS);
    if (tid == 0) {
        for (int s = 0; s < MM_NS; ++s)
            mbar_init(&full[s], 1);
        mbar_init(&mmad[0], 1);
        mbar_init(&mmad[1], 1);
        fence_mbar_init();
        *fail = 0;
        *issued = 0;
        *committed = 0;
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tbase = *tslot;
    constexpr uint32_t idesc = umma_idesc_f16_f32(MM_ROWS, NT);

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

    int bg0 = 0;  // block columns of earlier tiles (ring slot and phase continue)
    int g0 = 0;   // half-chunks of earlier tiles (operand buffer and phase continue)
    for (int rt0 = r0b; rt0 < r1b && !*fail; rt0 += MM_ROWS) {
        const int nrows = min(MM_ROWS, r1b - rt0);
        const uint8_t* Wt = a.W + static_cast<size_t>(rt0) * row_bytes;
        // warp 0 streams block column c of the tile's rows into its ring slot
        auto issue = [&](int c) {
            const int bg = bg0 + c;
            const int s = bg % MM_NS;
            if (lane == 0)
                mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(nrows * Q4K_BYTES));
            __syncwarp();
            for (int r = lane; r < nrows; r += 32)
                bulk_g2s(ring + s * MM_SLOT + r * Q4K_BYTES, Wt + r * row_bytes + static_cast<size_t>(c) * Q4K_BYTES,
                         Q4K_BYTES, &full[s], pol);
            if (lane == 0)
                *issued = bg + 1;
        };
        if (warp == 0)
            for (int c = 0; c < min(MM_NS, nblk); ++c)
                issue(c);

        for (int hc = 0; hc < 2 * nblk; ++hc) {
            const int c = hc >> 1, half = hc & 1;
            const int g = g0 + hc, buf = g & 1;
            const int bg = bg0 + c;
            if (half == 0 && !wait(&full[bg % MM_NS], (bg / MM_NS) & 1, DEVERR_TIMEOUT_FULL))
                break;
            if (g >= 2 && !wait(&mmad[buf], ((g - 2) >> 1) & 1, DEVERR_TIMEOUT_MMA))
                break;
            uint8_t* At = Abuf + buf * MM_A_BYTES;
            uint8_t* Bt = Bbuf + buf * mm_b_bytes(NT);
            const uint8_t* slot = ring + (bg % MM_NS) * MM_SLOT;
            // weights: 128 rows x 4 sub-blocks of 32 of this half block, two units a thread
#pragma unroll
            for (int i = 0; i < (MM_ROWS * 4) / MM_THREADS; ++i) {
                const int u = tid + MM_THREADS * i;
                const int row = u >> 2, jj = u & 3, j = 4 * half + jj;
                if (row < nrows) {
                    const uint8_t* bp = slot + row * Q4K_BYTES;
                    const uint4 hd = lds128(bp);
                    const uint4 cw = lds128(bp + 16 + 16 * j);
                    const uint32_t s_lo = j < 6 ? hd.y : hd.z, s_hi = j < 6 ? hd.z : hd.w;
                    const uint32_t m_lo = j < 3 ? hd.z : hd.w, m_hi = j < 3 ? hd.w : 0u;
                    const int sc = static_cast<int>(__funnelshift_r(s_lo, s_hi, (6 * j) & 31) & 63u);
                    const int mn = static_cast<int>(__funnelshift_r(m_lo, m_hi, (48 + 6 * j) & 31) & 63u);
                    const float d = half_bits_to_float(hd.x), dmin = half_bits_to_float(hd.x >> 16);
                    const __half2 A = __float2half2_rn(d * static_cast<float>(sc));
                    const __half2 B = __float2half2_rn(dmin * static_cast<float>(mn));
                    // byte i of the 16: low nibble weight 32j + i, high nibble weight 32j + 16 + i
                    uint32_t lo[8], hi[8];
                    const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const uint32_t t = __byte_perm(words[w], 0u, 0x3120);  // b0 b2 b1 b3
                        mm_dequant_word(t, A, B, lo[2 * w], lo[2 * w + 1], hi[2 * w], hi[2 * w + 1]);
                    }
                    const int k0 = 32 * jj;  // within the 128-wide stage
                    *reinterpret_cast<uint4*>(At + mm_off(row, k0)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    *reinterpret_cast<uint4*>(At + mm_off(row, k0 + 8)) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
                    *reinterpret_cast<uint4*>(At + mm_off(row, k0 + 16)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4*>(At + mm_off(row, k0 + 24)) = make_uint4(hi[4], hi[5], hi[6], hi[7]);
                }
            }
            // activations: tokens x 16 groups of 8 K, fp32 -> fp16
            const int kbase = c * 256 + half * MM_KC;
            for (int it = tid; it < a.M * (MM_KC / 8); it += MM_THREADS) {
                const int n = it >> 4, kg = it & 15;
                const float4* xp = reinterpret_cast<const float4*>(a.X + static_cast<size_t>(n) * a.K + kbase + 8 * kg);
                const float4 x0 = __ldg(xp), x1 = __ldg(xp + 1);
                const uint4 v = make_uint4(h2_bits(__floats2half2_rn(x0.x, x0.y)), h2_bits(__floats2half2_rn(x0.z, x0.w)),
                                           h2_bits(__floats2half2_rn(x1.x, x1.y)), h2_bits(__floats2half2_rn(x1.z, x1.w)));
                *reinterpret_cast<uint4*>(Bt + mm_off(n, 8 * kg)) = v;
            }
            fence_proxy_async_smem();
            __syncthreads();
            if (*fail)
                break;
            if (warp == 0) {
                if (lane == 0) {
                    tc_fence_after_sync();
#pragma unroll
                    for (int s = 0; s < MM_KC / 16; ++s)
                        umma_f16(tbase, umma_desc_kmajor(At + s * 2 * MM_LBO, MM_LBO, MM_SBO),
                                 umma_desc_kmajor(Bt + s * 2 * MM_LBO, MM_LBO, MM_SBO), idesc, (hc > 0 || s > 0) ? 1u : 0u);
                    umma_commit(&mmad[buf]);
                    *committed = g + 1;
                }
                __syncwarp();
                // the slot's block column is dequantised: refill it
                if (half == 1 && c + MM_NS < nblk)
                    issue(c + MM_NS);
            }
        }
        if (*fail)
            break;
        // accumulator complete -> Y
        const int glast = g0 + 2 * nblk - 1;
        wait(&mmad[glast & 1], (glast >> 1) & 1, DEVERR_TIMEOUT_MMA);
        __syncthreads();  // the flag is read uniformly: tcgen05.ld is warp-collective
        tc_fence_after_sync();
        const bool ok = !*fail;
        if (warp < 4 && ok) {
            const int row = 32 * warp + lane;
#pragma unroll
            for (int cc = 0; cc < NT / 16; ++cc) {
                uint32_t v[16];
                tmem_ld16(tbase + (static_cast<uint32_t>(32 * warp) << 16) + 16 * cc, v);
                tmem_ld_wait();
                if (row < nrows) {
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int n = 16 * cc + q;
                        if (n < a.M)
                            a.Y[static_cast<size_t>(n) * a.rows + rt0 + row] = __uint_as_float(v[q]);
                    }
                }
            }
        }
        tc_fence_before_sync();
        __syncthreads();  // accumulator read before the next tile's MMAs overwrite it
        bg0 += nblk;
        g0 += 2 * nblk;
    }
    // After a failed wait: let this block's copies and MMAs in flight finish (bounded).
    __syncthreads();
    if (tid == 0 && *fail) {
        const int hi = *issued, gc = *committed;
        for (int bg = max(0, hi - MM_NS); bg < hi; ++bg) {
            const unsigned long long t0 = globaltimer_ns();
            while (!mbar_try_wait(&full[bg % MM_NS], (bg / MM_NS) & 1) && globaltimer_ns() - t0 < 100000000ull) {
            }
        }
        for (int g = max(0, gc - 2); g < gc; ++g) {
            const unsigned long long t0 = globaltimer_ns();
            while (!mbar_try_wait(&mmad[g & 1], (g >> 1) & 1) && globaltimer_ns() - t0 < 100000000ull) {
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tbase, NCOLS);
    }
}

}  // namespace dq

namespace dqhost {

static int mm_nt(int M) { return M <= 16 ? 16 : M <= 32 ? 32 : 64; }

static int launch_matmul_tc(const uint8_t* W, const float* X, float* Y, int M, int rows, int K, cudaStream_t s)
{
    static std::once_flag once[3];
    static cudaError_t attr_err[3];
    const int nt = mm_nt(M);
    const int idx = nt == 16 ? 0 : nt == 32 ? 1 : 2;
    void (*k)(dq::MmArgs) = nt == 16 ? dq::matmul_q4k_tc_kernel<16>
                          : nt == 32 ? dq::matmul_q4k_tc_kernel<32>
                                     : dq::matmul_q4k_tc_kernel<64>;
    const int smem = dq::mm_smem_bytes(nt);
    std::call_once(once[idx], [&] {
        attr_err[idx] = cudaFuncSetAttribute(reinterpret_cast<const void*>(k),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (attr_err[idx] != cudaSuccess)
        return set_cuda_error(attr_err[idx]);
    dq::MmArgs a{W, X, Y, M, rows, K, device_error_flag()};
    const int grid = std::min(sm_count(), rows);
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
    const bool tensor = path == DQ_MATMUL_TENSOR || (path == DQ_MATMUL_AUTO && M >= 2);
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
        cudaError_t e = dqhost::launch_gemv(plan, a, s, false);
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
