// dq_gemv_q2k.cu -- instantiations of the streaming GEMV kernel for q2k rows.
#include "dq_gemv_host.h"

namespace dqhost {

GemvKernel gemv_kernel_q2k(int ul, int rpt, int nmat, int pl)
{
#define DQ_K(UL, RPT, NM, PL) \
    if (ul == UL && rpt == RPT && nmat == NM && pl == PL) \
        return &dq::gemv_stream_kernel<dq::FMT_Q2K, UL, RPT, NM, PL>;
    DQ_K(1, 1, 1, 1)
    DQ_K(1, 2, 1, 1)
    DQ_K(1, 4, 1, 1)
    DQ_K(2, 1, 1, 1)
    DQ_K(2, 2, 1, 1)
    DQ_K(2, 4, 1, 1)
    DQ_K(3, 1, 1, 1)
    DQ_K(3, 2, 1, 1)
    DQ_K(3, 4, 1, 1)
    DQ_K(4, 1, 1, 1)
    DQ_K(4, 2, 1, 1)
    DQ_K(4, 4, 1, 1)
#undef DQ_K
    return nullptr;
}

}  // namespace dqhost
