// Kernel instances for layernorm forward, f32 rows.
#define QK_OP 3
#define QK_T float
#define QK_ELEM_BYTES 4
#include "qk_kernel_table.cuh"

namespace qk {
KernelTable kernels_layernorm_f32() { return {kTable, int(sizeof(kTable) / sizeof(kTable[0]))}; }
}  // namespace qk
