// Kernel instances for layernorm forward, bf16 rows.
#define QK_OP 3
#define QK_T __nv_bfloat16
#define QK_ELEM_BYTES 2
#include "qk_kernel_table.cuh"

namespace qk {
KernelTable kernels_layernorm_bf16() { return {kTable, int(sizeof(kTable) / sizeof(kTable[0]))}; }
}  // namespace qk
