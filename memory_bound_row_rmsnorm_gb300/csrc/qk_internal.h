// qk_internal.h -- types shared by the kernel translation units and the C ABI.
#pragma once

#include <stdint.h>

namespace qk {

// Kernel-side operator codes (the ABI numbers LayerNorm 6; see qk_api.cu).
// kXentGrad, kSoftmaxGrad: cross-entropy and softmax backward on the shifted
// kernel (unaligned rows).
enum Op : int { kSoftmax = 0, kRmsNorm = 1, kXent = 2, kLayerNorm = 3, kXentGrad = 4, kSoftmaxGrad = 5 };
enum Dtype : int { kF32 = 0, kBF16 = 1 };

// Everything a row kernel needs, passed by value as its only parameter.
struct RowArgs {
  const void* x;          // [M, N] input rows (logits for cross-entropy)
  void* y;                // [M, N] output rows (softmax, RMSNorm)
  const void* w;          // [N] RMSNorm / LayerNorm weight
  const void* bias;       // [N] LayerNorm bias, may be null
  float* rstd;            // [M] RMSNorm 1/rms or LayerNorm 1/std, may be null
  float* mean;            // [M] LayerNorm row mean, may be null
  const int64_t* target;  // [M] cross-entropy targets
  float* loss;            // [M] cross-entropy loss
  float* lse;             // [M] cross-entropy log-sum-exp, may be null (kXentGrad: input)
  const float* dloss;     // [M] kXentGrad: upstream gradient, null for 1
  const void* x2;         // [M, N] kSoftmaxGrad: dy (x holds y), with x's alignment modulo 16
  int64_t M;
  int64_t N;
  float eps;
  float inv_n;          // 1 / N, rounded once on the host (RMSNorm mean)
  float z_loss;         // cross-entropy: coefficient of z * lse^2 added to the loss (0: none)
  int64_t ignore_index; // cross-entropy: rows with this target give loss 0 (when has_ignore)
  int32_t has_ignore;   // cross-entropy: nonzero when ignore_index is in use (no target value means "none")
  int32_t chunks;       // ring slots one row slice spans (streamed rows), else 1
  int64_t chunk_elems;  // shifted kernel, streamed rows: elements of one chunk, ceil(N / chunks)
  int32_t slots;        // ring slots per CTA
  uint32_t slot_bytes;  // bytes per ring slot (multiple of 128)
  int64_t num_items;    // work items: row blocks of threads/row_threads rows, or rows
  uint64_t timeout_ns;  // bound on every wait inside the kernel
  int* status;          // device status word (first failure code)
};

// Size of the fixed shared-memory header in front of the TMA ring: mbarriers,
// the block-reduction buffer and the cluster exchange buffer.
constexpr int kSmemHeader = 1024;
constexpr int kMaxSlots = 32;
// Per-column parameters of the ring kernels: RMSNorm / LayerNorm keep their
// share of w in registers up to kAffineRegsMaxVpt vectors a thread, LayerNorm
// its share of b up to kLnBiasRegsMaxVpt.  Beyond that LayerNorm stages the
// CTA's slice of the parameter in shared memory once, after the ring slots
// (w first, then b, each param_slice_bytes long); the planner sizes the
// shared memory with the same rule.
constexpr int kAffineRegsMaxVpt = 8;
constexpr int kLnBiasRegsMaxVpt = 4;
__host__ __device__ constexpr int64_t param_slice_bytes(int64_t slice_vectors) {
  return (slice_vectors * 16 + 127) / 128 * 128;
}
constexpr int kMaxCluster = 16;

// One compiled kernel.  `path` 1: TMA ring kernel (threads, row_threads,
// vec_per_thread); path 2: masked direct kernel (threads, elems_per_thread);
// path 3: backward ring kernel (as path 1); path 4: two-pass ring kernel for
// rows longer than a cluster holds (as path 1); path 5: masked backward
// kernel; path 6: shifted ring kernel (unaligned rows).
struct KernelEntry {
  int path;
  int threads;
  int row_threads;
  int vec_per_thread;
  bool clustered;
  const void* func;
};

struct KernelTable {
  const KernelEntry* entries;
  int count;
};

// Defined by the instantiation translation units, one per (op, dtype).
KernelTable kernels_softmax_f32();
KernelTable kernels_softmax_bf16();
KernelTable kernels_rmsnorm_f32();
KernelTable kernels_rmsnorm_bf16();
KernelTable kernels_xent_f32();
KernelTable kernels_xent_bf16();
KernelTable kernels_layernorm_f32();
KernelTable kernels_layernorm_bf16();
KernelTable bwd_kernels_softmax_f32();
KernelTable bwd_kernels_softmax_bf16();
KernelTable bwd_kernels_rmsnorm_f32();
KernelTable bwd_kernels_rmsnorm_bf16();
KernelTable bwd_kernels_xent_f32();
KernelTable bwd_kernels_xent_bf16();

}  // namespace qk
