// dq_gemv_host.h -- host-side planning and launching of the streaming GEMV kernel.
#pragma once

#include <cuda_runtime.h>

#include "dq_gemv.cuh"

namespace dqhost {

using GemvKernel = void (*)(dq::GemvArgs);

// Kernel tables, one translation unit per format (null when not instantiated).
GemvKernel gemv_kernel_q4k(int ul, int rpt, int nmat, int pl);
GemvKernel gemv_kernel_q6k(int ul, int rpt, int nmat, int pl);
GemvKernel gemv_kernel_q2k(int ul, int rpt, int nmat, int pl);
GemvKernel gemv_kernel_bf16(int ul, int rpt, int nmat, int pl);

struct GemvPlan {
    int fmt, rows, K, nmat;
    int row_bytes;
    int P, RG, UL, RPT;
    int planes;      // activation planes: 1 (15-bit) or 2 (about 30-bit, Q4_K with UL <= 2)
    int nstage, stage_bytes;
    int smem_bytes;
    int grid;
    int resid_rows;  // shared-memory slots for residual rows (EPI_RESID), else 0
    GemvKernel kernel;
};

#ifndef GEMV_STAGE_TARGET_KB
#define GEMV_STAGE_TARGET_KB 48
#endif
constexpr int GEMV_STAGE_TARGET = GEMV_STAGE_TARGET_KB * 1024;  // bytes per ring stage (upper target)
constexpr int GEMV_STAGE_MAX = 64 * 1024;      // largest stage accepted
constexpr int GEMV_RING_MAX = 176 * 1024;      // ring bytes at most (one block per SM)
constexpr int GEMV_SMEM_MAX = 227 * 1024;      // shared memory one block may use

// Chooses the thread layout, tile and ring for one matrix shape.  `planes` = 2
// asks for the two-plane activation where the format and layout allow it (else
// one plane); `resid` reserves room for the block's residual rows (the
// EPI_RESID epilogue).  Returns DQ_OK, DQ_ERR_SHAPE or DQ_ERR_UNSUPPORTED.
// Sets the kernel's shared-memory attribute (host call, not a stream operation).
int plan_gemv(int fmt, int rows, int K, int nmat, int planes, bool resid, GemvPlan* plan);

// Fills the layout fields of `a` from the plan and launches on `stream`;
// `pdl` adds the programmatic-stream-serialisation launch attribute.
cudaError_t launch_gemv(const GemvPlan& plan, dq::GemvArgs a, cudaStream_t stream, bool pdl);

// Diagnostics: GEMV launches record per-block timestamps into `buf` (8 x 64-bit
// per block: start, set-up done, dependency released, activation staged,
// activation quantised, first stage ready, end, blocks finished); NULL stops.
void set_gemv_trace(void* buf);
unsigned long long* gemv_trace();  // the buffer set by set_gemv_trace (null when off)

}  // namespace dqhost
