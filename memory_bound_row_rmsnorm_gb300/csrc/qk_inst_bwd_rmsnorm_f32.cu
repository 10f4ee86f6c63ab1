// Kernel instances for rmsnorm backward, f32 rows.
#define QK_BOP 11
#define QK_T float
#include "qk_bwd_table.cuh"

namespace qk {
KernelTable bwd_kernels_rmsnorm_f32() { return {kBwdTable, int(sizeof(kBwdTable) / sizeof(kBwdTable[0]))}; }
}  // namespace qk
