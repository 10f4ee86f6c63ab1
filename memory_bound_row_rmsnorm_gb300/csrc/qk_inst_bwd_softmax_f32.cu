// Kernel instances for softmax backward, f32 rows.
#define QK_BOP 10
#define QK_T float
#include "qk_bwd_table.cuh"

namespace qk {
KernelTable bwd_kernels_softmax_f32() { return {kBwdTable, int(sizeof(kBwdTable) / sizeof(kBwdTable[0]))}; }
}  // namespace qk
