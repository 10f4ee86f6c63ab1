// qk_kernel_table.cuh -- the compiled kernel configurations of one (op, dtype).
//
// Include with QK_OP (an Op) and QK_T (float or __nv_bfloat16) defined.
// Ring kernels: (threads, row_threads, vec_per_thread, clustered); a row of up
// to row_threads * vec_per_thread 16-byte vectors fits one CTA, and a cluster
// of up to 16 CTAs multiplies that.  Direct kernels: (threads, elems/thread).
#pragma once

#include "qk_kernels.cuh"
#include "qk_shifted_kernels.cuh"

#define QK_RING(TH, TPR, VPT, CL) \
  {1, TH, TPR, VPT, CL, reinterpret_cast<const void*>(&row_kernel<QK_OP, QK_T, TH, TPR, VPT, CL>)}
#define QK_RING2(TH, TPR, VPT, CL)                                                    \
  {4, TH, TPR, VPT, CL,                                                               \
   reinterpret_cast<const void*>(&row_kernel<QK_OP, QK_T, TH, TPR, VPT, CL, true>)}
// Rows that do not start on a 16-byte boundary (path 6): aligned superset copies.
#define QK_SHIFT(TH, TPR, VPT, CL) \
  {6, TH, TPR, VPT, CL, reinterpret_cast<const void*>(&shifted_kernel<QK_OP, QK_T, TH, TPR, VPT, CL>)}
#define QK_DIRECT(TH, EPT, CL) \
  {2, TH, TH, EPT, CL, reinterpret_cast<const void*>(&direct_kernel<QK_OP, QK_T, TH, EPT, CL>)}

namespace qk {
namespace {
const KernelEntry kTable[] = {
    QK_RING(256, 8, 4, false),
    QK_RING(256, 8, 8, false),
    QK_RING(256, 16, 4, false),
    QK_RING(256, 16, 8, false),
    QK_RING(256, 32, 8, false),
    QK_RING(256, 32, 16, false),
    QK_RING(256, 64, 8, false),
    QK_RING(256, 128, 8, false),
    QK_RING(256, 32, 1, false),
    QK_RING(256, 32, 2, false),
    QK_RING(256, 32, 4, false),
    QK_RING(256, 64, 2, false),
    QK_RING(256, 64, 4, false),
    QK_RING(256, 128, 2, false),
    QK_RING(256, 128, 4, false),
    QK_RING(128, 128, 4, false),
    QK_RING(128, 128, 8, false),
    QK_RING(256, 256, 2, false),
    QK_RING(256, 256, 4, false),
    QK_RING(256, 256, 8, false),
    QK_RING(512, 512, 2, false),
    QK_RING(512, 512, 4, false),
    QK_RING(512, 512, 8, false),
#if QK_OP == 2  // cross-entropy: 128-thread CTAs of two 64-thread rows (finer items for short launches)
    QK_RING(128, 64, 8, false),
    QK_RING(128, 32, 16, false),
#endif
#if QK_OP != 2  // cross-entropy streams long rows instead of splitting them
    QK_RING(256, 256, 4, true),
    QK_RING(256, 256, 8, true),
    QK_RING(512, 512, 4, true),
    QK_RING(512, 512, 8, true),
    QK_RING(256, 256, 16, true),
#if QK_OP != 2
    // rows longer than a cluster holds: streamed twice in 32 KB chunks
    QK_RING2(256, 256, 8, false),
    QK_RING2(256, 256, 8, true),
#endif
#endif
    // one vector more than a power of two: a misaligned row of 2^k vectors spans 2^k + 1
    QK_SHIFT(256, 8, 5, false),
    QK_SHIFT(256, 16, 5, false),
    QK_SHIFT(256, 32, 5, false),
    QK_SHIFT(256, 64, 5, false),
    QK_SHIFT(256, 128, 5, false),
    QK_SHIFT(256, 256, 5, false),
#if QK_OP != 3  // LayerNorm at 9 vectors keeps two CTAs per SM: its narrow groups stay at 5
    QK_SHIFT(256, 16, 9, false),
    QK_SHIFT(256, 32, 9, false),
    QK_SHIFT(256, 64, 9, false),
    QK_SHIFT(256, 128, 9, false),
#endif
    QK_SHIFT(256, 256, 9, false),
#if QK_OP != 2
    QK_SHIFT(256, 256, 8, true),
    QK_SHIFT(256, 256, 9, true),
#endif
    QK_DIRECT(128, 4, false),
    QK_DIRECT(256, 16, false),
    QK_DIRECT(512, 32, false),
#if QK_OP != 2
    QK_DIRECT(512, 64, true),
#endif
};
}  // namespace
}  // namespace qk
