// dq_gemv_bf16.cu -- instantiations of the streaming GEMV kernel for bf16 rows.
#include "dq_gemv_host.h"

namespace dqhost {

GemvKernel gemv_kernel_bf16(int ul, int rpt, int nmat, int pl)
{
#define DQ_K(UL, RPT, NM, PL) \
    if (ul == UL && rpt == RPT && nmat == NM && pl == PL) \
        return &dq::gemv_stream_kernel<dq::FMT_BF16, UL, RPT, NM, PL>;
    DQ_K(1, 1, 1, 1)
    DQ_K(1, 2, 1, 1)
    DQ_K(1, 4, 1, 1)
    DQ_K(2, 1, 1, 1)
    DQ_K(2, 2, 1, 1)
    DQ_K(2, 4, 1, 1)
    DQ_K(4, 1, 1, 1)
    DQ_K(4, 2, 1, 1)
    DQ_K(4, 4, 1, 1)
    DQ_K(8, 1, 1, 1)
    DQ_K(8, 2, 1, 1)
    DQ_K(8, 4, 1, 1)
    DQ_K(12, 1, 1, 1)
    DQ_K(12, 2, 1, 1)
    DQ_K(12, 4, 1, 1)
#undef DQ_K
    return nullptr;
}

}  // namespace dqhost
