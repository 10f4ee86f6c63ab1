// qk_bwd_table.cuh -- compiled configurations of one backward (op, dtype).
// Include with QK_BOP (a BwdOp) and QK_T defined.
#pragma once

#include "qk_bwd_kernels.cuh"
#include "qk_shifted_kernels.cuh"

#define QK_BWD(TH, TPR, VPT, CL) \
  {3, TH, TPR, VPT, CL, reinterpret_cast<const void*>(&bwd_kernel<QK_BOP, QK_T, TH, TPR, VPT, CL>)}
// Masked path (path 5): (threads, elements per thread, clustered).
#define QK_SHIFT_GRAD(TH, TPR, VPT) \
  {6, TH, TPR, VPT, false,                 \
   reinterpret_cast<const void*>(&shifted_kernel<kXentGrad, QK_T, TH, TPR, VPT, false>)}
#define QK_SHIFT_SGRAD(TH, TPR, VPT, CL) \
  {6, TH, TPR, VPT, CL,                     \
   reinterpret_cast<const void*>(&shifted_kernel<kSoftmaxGrad, QK_T, TH, TPR, VPT, CL>)}
#define QK_BWD_DIRECT(TH, EPT, CL) \
  {5, TH, TH, EPT, CL, reinterpret_cast<const void*>(&bwd_direct_kernel<QK_BOP, QK_T, TH, EPT, CL>)}

namespace qk {
namespace {
const KernelEntry kBwdTable[] = {
    QK_BWD(256, 8, 4, false),   QK_BWD(256, 16, 4, false),  QK_BWD(256, 32, 4, false),
    QK_BWD(256, 64, 4, false),  QK_BWD(256, 128, 4, false), QK_BWD(256, 256, 4, false),
    QK_BWD(128, 128, 4, false),
#if QK_BOP == 12  // cross-entropy: wider per-thread rows, streamed long rows
    QK_BWD(256, 8, 8, false),   QK_BWD(256, 16, 8, false),  QK_BWD(256, 32, 8, false),
    QK_BWD(256, 64, 8, false),  QK_BWD(256, 128, 8, false), QK_BWD(256, 256, 8, false),
#elif QK_BOP == 10  // softmax: 8 vectors a thread, clusters for long rows
    QK_BWD(256, 256, 8, false), QK_BWD(256, 256, 8, true),
#else  // RMSNorm: 2-4 vectors a thread (x, dy, w and the dw partials live in registers)
    QK_BWD(256, 16, 2, false),  QK_BWD(256, 32, 2, false),  QK_BWD(256, 64, 2, false),
    QK_BWD(256, 128, 2, false), QK_BWD(256, 256, 2, false), QK_BWD(512, 512, 2, false),
    QK_BWD(256, 256, 2, true),  QK_BWD(512, 512, 2, true),
    QK_BWD(256, 256, 4, true),  QK_BWD(512, 512, 4, true),
#endif
#if QK_BOP == 12
    QK_BWD_DIRECT(256, 8, false),
    // unaligned rows whose dlogits share the logits' alignment (path 6)
    QK_SHIFT_GRAD(256, 8, 5),   QK_SHIFT_GRAD(256, 16, 5),  QK_SHIFT_GRAD(256, 32, 5),
    QK_SHIFT_GRAD(256, 64, 5),  QK_SHIFT_GRAD(256, 128, 5), QK_SHIFT_GRAD(256, 256, 5),
    QK_SHIFT_GRAD(256, 16, 9),  QK_SHIFT_GRAD(256, 32, 9),  QK_SHIFT_GRAD(256, 64, 9),
    QK_SHIFT_GRAD(256, 128, 9), QK_SHIFT_GRAD(256, 256, 9),
#else
    QK_BWD_DIRECT(128, 4, false),  QK_BWD_DIRECT(256, 8, false),  QK_BWD_DIRECT(512, 16, false),
    QK_BWD_DIRECT(512, 16, true),
#endif
#if QK_BOP == 10  // softmax: unaligned rows with y, dy and dx aligned alike (path 6)
    QK_SHIFT_SGRAD(256, 8, 5, false),   QK_SHIFT_SGRAD(256, 16, 5, false),
    QK_SHIFT_SGRAD(256, 32, 5, false),  QK_SHIFT_SGRAD(256, 64, 5, false),
    QK_SHIFT_SGRAD(256, 128, 5, false), QK_SHIFT_SGRAD(256, 256, 5, false),
    QK_SHIFT_SGRAD(256, 256, 9, false), QK_SHIFT_SGRAD(256, 256, 8, true),
    QK_SHIFT_SGRAD(256, 256, 9, true),
#endif
};
}  // namespace
}  // namespace qk
