// Kernel instances for xent backward, bf16 rows.
#define QK_BOP 12
#define QK_T __nv_bfloat16
#include "qk_bwd_table.cuh"

namespace qk {
KernelTable bwd_kernels_xent_bf16() { return {kBwdTable, int(sizeof(kBwdTable) / sizeof(kBwdTable[0]))}; }
}  // namespace qk
