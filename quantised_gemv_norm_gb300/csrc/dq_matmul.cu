// dq_matmul.cu -- Y[m] = W X[m] for M token vectors over one Q4_K matrix.
//
// "The roofline holds on a second GPU", section "The Math": M tokens processed
// together share one read of the weights until the arithmetic catches up, at
// M* = (w / 16) (R / BW).  This entry point is the measured side of that
// crossover.  This version runs the single-vector streaming kernel once per
// token, so it reads the weights M times; it is the reference point the
// shared-read kernels are compared with.
#include "dq_gemv_host.h"

extern "C" {

DQ_API int dq_matmul_q4k(const void* W_blocks, const float* X, float* Y, int M, int rows, int K, void* stream)
{
    if (!W_blocks || !X || !Y)
        return DQ_ERR_NULL;
    if (M < 1 || M > 64 || rows < 1)
        return DQ_ERR_SHAPE;
    if (K > 16384)
        return DQ_ERR_UNSUPPORTED;
    if (!dqhost::aligned16(W_blocks) || !dqhost::aligned16(X) || (K % 4))
        return DQ_ERR_ALIGN;
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
        cudaError_t e = dqhost::launch_gemv(plan, a, static_cast<cudaStream_t>(stream), false);
        if (e != cudaSuccess)
            return dqhost::set_cuda_error(e);
    }
    return DQ_OK;
}

}  // extern "C"
