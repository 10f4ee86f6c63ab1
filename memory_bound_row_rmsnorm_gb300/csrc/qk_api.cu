// qk_api.cu -- the C ABI of libqk.so: argument checks, launch plans, launches.
//
// Host side only: every element of every row is processed by the kernels in
// qk_kernels.cuh, qk_shifted_kernels.cuh and qk_bwd_kernels.cuh; nothing here
// touches row data.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <initializer_list>
#include <map>
#include <mutex>
#include <tuple>

#include "../../include/qk.h"
#include "qk_bwd_kernels.cuh"
#include "qk_device.cuh"
#include "qk_internal.h"

namespace qk {

// Device status word: the first failure code a kernel reports (0 = none).
__device__ int g_status_word;

__global__ void wait_timeout_kernel(uint64_t timeout_ns, int* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_addr(&bar);
  mbar_init(b, 1);
  fence_mbar_init();
  // Nobody arrives on `bar`, so phase 0 never completes.
  if (!mbar_wait<false>(b, 0u, timeout_ns)) report_status(status, QK_ERR_TIMEOUT);
}

namespace {

constexpr uint64_t kWaitTimeoutNs = 1000000000ull;  // 1 s bound on any in-kernel wait
constexpr int kMaxDevices = 64;
constexpr int kRingMaxVectorsPerCta = 4096;  // 256 threads x 16 vectors, or 512 x 8
constexpr int64_t kMaxRowBytes = int64_t(kMaxCluster) * kRingMaxVectorsPerCta * 16;  // 1 MiB
// Masked forward kernel (unaligned rows beyond the shifted kernel): 16
// clusters of 512 threads x 64 elements.
constexpr int64_t kMaskedMaxRow = int64_t(kMaxCluster) * 512 * 64;  // 524,288 elements
// Masked backward softmax / RMSNorm: 16 clusters of 512 threads x 16 elements.
constexpr int64_t kMaskedBwdMaxRow = int64_t(kMaxCluster) * 512 * 16;  // 131,072 elements

struct DeviceInfo {
  std::atomic<bool> ready{false};  // set once, after the fields below
  qk_status error = QK_OK;
  int sms = 0;
  int smem_optin = 0;
  int* status = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
std::map<std::tuple<int, const void*>, bool> g_attr_done;
std::map<std::tuple<int, const void*, int, int>, int> g_occ;  // (dev, func, smem, C) -> CTAs/SM or clusters

struct Override {
  bool on = false;
  qk_plan plan{};
};
constexpr int kNumOps = 7;  // softmax, RMSNorm, x-entropy; their backward passes; LayerNorm
Override g_override[kNumOps][2];
std::atomic<uint64_t> g_override_gen{1};  // bumped by every qk_set_plan_override

// Operator codes of the ABI (qk_op): the forward passes 0-2 match the kernels'
// Op values; the backward passes are 3-5 and LayerNorm (kernel Op kLayerNorm)
// is 6.
constexpr int kOpSoftmaxBwd = 3, kOpRmsNormBwd = 4, kOpXentBwd = 5, kOpLayerNorm = 6;
bool is_bwd(int op) { return op >= kOpSoftmaxBwd && op <= kOpXentBwd; }
// Input matrices one work item loads (both y/x and dy for two backward passes).
int inputs_per_item(int op) { return (op == kOpSoftmaxBwd || op == kOpRmsNormBwd) ? 2 : 1; }
bool streams_rows(int op) { return op == kXent || op == kOpXentBwd; }

KernelTable table_for(int op, int dt) {
  switch (op * 2 + dt) {
    case 0: return kernels_softmax_f32();
    case 1: return kernels_softmax_bf16();
    case 2: return kernels_rmsnorm_f32();
    case 3: return kernels_rmsnorm_bf16();
    case 4: return kernels_xent_f32();
    case 5: return kernels_xent_bf16();
    case 6: return bwd_kernels_softmax_f32();
    case 7: return bwd_kernels_softmax_bf16();
    case 8: return bwd_kernels_rmsnorm_f32();
    case 9: return bwd_kernels_rmsnorm_bf16();
    case 10: return bwd_kernels_xent_f32();
    case 11: return bwd_kernels_xent_bf16();
    case 12: return kernels_layernorm_f32();
    default: return kernels_layernorm_bf16();
  }
}

const KernelEntry* find_kernel(int op, int dt, int path, int threads, int tpr, int vpt,
                               bool clustered) {
  const KernelTable t = table_for(op, dt);
  for (int i = 0; i < t.count; ++i) {
    const KernelEntry& e = t.entries[i];
    if (e.path == path && e.threads == threads && e.row_threads == tpr &&
        e.vec_per_thread == vpt && e.clustered == clustered)
      return &e;
  }
  return nullptr;
}

// Per-device facts, read once under the lock.
qk_status device_info(int* dev_out, DeviceInfo** info) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return QK_ERR_NO_DEVICE;
  }
  DeviceInfo& d = g_dev[dev];
  if (d.ready.load(std::memory_order_acquire)) {  // fast path: no lock after the first call
    *dev_out = dev;
    *info = &d;
    return d.error;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!d.ready.load(std::memory_order_relaxed)) {
    cudaDeviceProp p;
    if (cudaGetDeviceProperties(&p, dev) != cudaSuccess) {
      cudaGetLastError();
      d.error = QK_ERR_NO_DEVICE;
    } else if (!(p.major == 10 && p.minor == 3)) {
      d.error = QK_ERR_NO_DEVICE;  // the kernels are built for sm_103a only
    } else {
      d.sms = p.multiProcessorCount;
      d.smem_optin = int(p.sharedMemPerBlockOptin);
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_status_word) != cudaSuccess) {
        cudaGetLastError();
        d.error = QK_ERR_LAUNCH;
      } else {
        d.status = static_cast<int*>(ptr);
      }
    }
    d.ready.store(true, std::memory_order_release);
  }
  *dev_out = dev;
  *info = &d;
  return d.error;
}

// Opt a kernel into the device's full shared memory (and non-portable
// clusters) once per device.
qk_status prepare_kernel(int dev, const DeviceInfo& d, const KernelEntry& k) {
  std::lock_guard<std::mutex> lock(g_mu);
  auto key = std::make_tuple(dev, k.func);
  if (g_attr_done.count(key)) return QK_OK;
  if ((k.path == 1 || k.path == 3 || k.path == 4 || k.path == 6) &&  // ring kernels: dynamic smem
      cudaFuncSetAttribute(k.func, cudaFuncAttributeMaxDynamicSharedMemorySize, d.smem_optin) !=
          cudaSuccess) {
    cudaGetLastError();
    return QK_ERR_LAUNCH;
  }
  if (k.clustered &&
      cudaFuncSetAttribute(k.func, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
          cudaSuccess) {
    cudaGetLastError();
    return QK_ERR_LAUNCH;
  }
  g_attr_done[key] = true;
  return QK_OK;
}

// Resident CTAs per SM (cluster == 0) or resident clusters on the device.
qk_status occupancy(int dev, const KernelEntry& k, int smem, int cluster, int* out) {
  {
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_occ.find(std::make_tuple(dev, k.func, smem, cluster));
    if (it != g_occ.end()) {
      *out = it->second;
      return QK_OK;
    }
  }
  int n = 0;
  cudaError_t err;
  if (cluster == 0) {
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k.func, k.threads, size_t(smem));
  } else {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(unsigned(cluster), 1, 1);
    cfg.blockDim = dim3(unsigned(k.threads), 1, 1);
    cfg.dynamicSmemBytes = size_t(smem);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaOccupancyMaxActiveClusters(&n, k.func, &cfg);
  }
  if (err != cudaSuccess) {
    cudaGetLastError();
    return QK_ERR_LAUNCH;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  g_occ[std::make_tuple(dev, k.func, smem, cluster)] = n;
  *out = n;
  return QK_OK;
}

int elem_size(int dt) { return dt == QK_F32 ? 4 : 2; }

int next_pow2(int64_t v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

struct Plan {
  const KernelEntry* kernel = nullptr;
  int cluster = 1;
  int slots = 0;
  int chunks = 1;
  int64_t num_items = 0;
  uint32_t slot_bytes = 0;
  int smem = 0;
  int ctas_per_sm = 0;
  int64_t grid = 0;
};

// The fast path's plan table: for rows of at most max_nv 16-byte vectors,
// (threads, row_threads, vec_per_thread, cluster, slots).  Chosen from sweeps
// of every compiled configuration on GB300 (M = 16384 rows, N = 256 ... 262144,
// fp32 and bf16): short rows share a warp (sub-warp row groups), mid rows
// give each thread 32-64 elements so the per-row reduction is amortised, long
// rows are split over a thread-block cluster of 256-thread CTAs (small CTAs
// pack the GPCs better than 512-thread ones).  A one-slot ring is enough when
// the slice is held in registers: the slot is refilled as soon as it has been
// read, while the previous row is still being reduced and stored.
struct Choice {
  int64_t max_nv;
  int threads, row_threads, vec_per_thread, cluster, slots;
};
constexpr int64_t kStream = INT64_MAX;  // cross-entropy: any longer row is streamed
const Choice kRmsNormTable[] = {
    {32, 256, 8, 4, 1, 2},       {64, 256, 16, 4, 1, 3},       {128, 256, 32, 4, 1, 2},
    {256, 256, 64, 4, 1, 2},     {512, 128, 128, 4, 1, 1},     {1024, 128, 128, 8, 1, 1},
    {2048, 256, 256, 8, 1, 1},   {4096, 256, 256, 8, 2, 1},    {8192, 256, 256, 8, 4, 1},
    {16384, 256, 256, 8, 8, 3},  {32768, 256, 256, 8, 16, 2},  {65536, 512, 512, 8, 16, 2},
};
// LayerNorm: from a sweep of every compiled configuration on GB300 (M = 16384,
// N = 256 ... 262144, fp32 and bf16; rows of 512 and 2048 vectors again at
// 8192-32768 rows).  Its parameters not held in registers take shared memory,
// so long rows keep fewer ring slots than RMSNorm.  This table is bf16's;
// later sweeps at 4096-32768 rows deepened its rows of 16384 elements to
// three slots (94-97 % -> 97-98 %), moved its rows of 8192 to 256-thread CTAs
// of 4 vectors a thread with two slots (88-92 % -> 91-97 % from 6144 rows on),
// its rows of 2048 to four 64-thread rows per CTA with three slots
// (64-91 % -> 63-93 %, +7 at 6144-8192 rows), and its rows of 4096 to one
// 128-thread row per CTA, four CTAs per SM where two 128-thread rows per CTA
// held two (+1 to +3 points at 2048-32768 rows); its rows of 1024 keep the
// three slots that short launches get at every length (24576 x 1024:
// 86 % -> 89 %, 32768 x 1024 87 % -> 91 %, 65536 x 1024 93 % -> 91 %).
const Choice kLayerNormTable[] = {
    {32, 256, 8, 4, 1, 2},       {64, 256, 16, 4, 1, 2},       {128, 256, 32, 4, 1, 3},
    {256, 256, 64, 4, 1, 3},     {512, 128, 128, 4, 1, 2},     {1024, 256, 256, 4, 1, 2},
    {2048, 512, 512, 4, 1, 3},   {4096, 256, 256, 8, 2, 1},    {8192, 256, 256, 8, 4, 2},
    {16384, 256, 256, 8, 8, 2},  {32768, 512, 512, 8, 8, 1},   {65536, 512, 512, 8, 16, 2},
};
// fp32 LayerNorm rows of 131072 elements (32768 vectors): clusters of 16
// 256-thread CTAs with two ring slots, 83 % -> 93 % at 8192-16384 rows; bf16
// rows of the same bytes measured 2 points slower that way and keep 512 x 8.
const Choice kLayerNormF32Table[] = {
    {32, 256, 8, 4, 1, 2},       {64, 256, 16, 4, 1, 2},       {128, 256, 32, 4, 1, 2},
    {256, 256, 32, 8, 1, 3},     {512, 256, 128, 4, 1, 2},     {1024, 128, 128, 8, 1, 1},
    {2048, 512, 512, 4, 1, 2},   {4096, 256, 256, 8, 2, 1},    {8192, 256, 256, 8, 4, 2},
    {16384, 256, 256, 8, 8, 2},  {32768, 256, 256, 8, 16, 2},  {65536, 512, 512, 8, 16, 2},
};
// Rows of 64 vectors (fp32 256, bf16 512 elements), RMSNorm and softmax:
// sixteen 16-thread rows of 4 vectors a thread per CTA, three slots
// (89-91 % -> 96-101 % at 24576-32768 rows, against eight 32-thread rows).
const Choice kSoftmaxTable[] = {
    {32, 256, 8, 4, 1, 2},       {64, 256, 16, 4, 1, 3},       {128, 256, 32, 4, 1, 3},
    {256, 256, 64, 4, 1, 2},     {512, 128, 128, 4, 1, 1},     {1024, 256, 256, 4, 1, 1},
    {2048, 512, 512, 4, 1, 3},   {4096, 256, 256, 8, 2, 1},    {8192, 256, 256, 8, 4, 2},
    {16384, 256, 256, 16, 4, 2},  {32768, 256, 256, 16, 8, 1},  {65536, 256, 256, 16, 16, 1},
};
// bf16 softmax: rows of 8192 elements (1024 vectors) in 128-thread CTAs of
// 8 vectors a thread, which keep four CTAs per SM where 256 x 4 keeps three
// (85-98 % of peak against 80-90 % at 2048-32768 rows).
const Choice kSoftmaxBf16Table[] = {
    {32, 256, 8, 4, 1, 2},       {64, 256, 16, 4, 1, 3},       {128, 256, 32, 4, 1, 3},
    {256, 256, 64, 4, 1, 2},     {512, 128, 128, 4, 1, 1},     {1024, 128, 128, 8, 1, 1},
    {2048, 512, 512, 4, 1, 3},   {4096, 256, 256, 8, 2, 1},    {8192, 256, 256, 8, 4, 2},
    {16384, 256, 256, 16, 4, 2},  {32768, 256, 256, 16, 8, 1},  {65536, 256, 256, 16, 16, 1},
};
// Cross-entropy rows of 1024 vectors stream from two slots (fp32 4096 and
// bf16 8192 elements: +3 to +10 points over one slot at 4096-32768 rows).
// Rows of 512 vectors (bf16 4096, fp32 2048 elements) take one warp a row,
// 16 vectors a lane, in 128-thread CTAs: bf16 16384 x 4096 90 % -> 100 %,
// 32768 x 4096 97 % -> 103 %; fp32 8192 x 2048 89 % -> 93 %.
const Choice kXentTable[] = {
    {32, 256, 8, 4, 1, 1},       {64, 256, 8, 8, 1, 2},        {128, 256, 16, 8, 1, 2},
    {256, 256, 32, 8, 1, 2},     {512, 128, 32, 16, 1, 2},     {1024, 128, 128, 8, 1, 2},
    {2048, 256, 256, 8, 1, 2},   {kStream, 256, 256, 4, 1, 2},  // 16 KB chunks
};

// Backward passes load two matrices per item (softmax, RMSNorm), so they hold
// at most 4-8 vectors of each per thread; cross-entropy's backward streams.
const Choice kSoftmaxBwdTable[] = {
    {32, 256, 8, 4, 1, 2},     {64, 256, 16, 4, 1, 2},    {128, 256, 64, 4, 1, 2},
    {256, 256, 128, 4, 1, 2},  {512, 128, 128, 4, 1, 1},  {1024, 256, 256, 4, 1, 1},
    {2048, 256, 256, 8, 1, 2}, {4096, 256, 256, 8, 2, 1}, {8192, 256, 256, 8, 4, 1},
    {16384, 256, 256, 8, 8, 1}, {32768, 256, 256, 8, 16, 1},
};
// RMSNorm backward: a ring depth per dtype from a sweep of 1-4 slots at
// 8192-32768 rows.  fp32 rows of 2048 take four slots (three CTAs per SM
// instead of five: 76 % -> 88 %, 86 % -> 95 %, 92 % -> 98 %; fewer CTAs also
// means fewer dw partial rows to sum), bf16 rows of 8192 three (82 % -> 88 %,
// 86 % -> 93 %, 90 % -> 97 %); the other rows measured best at two, except
// bf16 rows of 2048, which a later search on the streaming-store kernels gave
// three (+2 to +6 points from 8192 rows on, level below).
const Choice kRmsNormBwdTable[] = {
    {32, 256, 32, 2, 1, 2},    {64, 256, 64, 2, 1, 2},    {128, 256, 64, 2, 1, 2},
    {256, 256, 128, 2, 1, 2},  {512, 128, 128, 4, 1, 4},  {1024, 256, 256, 4, 1, 2},
    {2048, 256, 256, 4, 2, 2}, {4096, 512, 512, 4, 2, 2}, {8192, 512, 512, 4, 4, 2},
    {16384, 512, 512, 4, 8, 2}, {32768, 512, 512, 4, 16, 2},
};
const Choice kRmsNormBwdBf16Table[] = {
    {32, 256, 32, 2, 1, 2},    {64, 256, 64, 2, 1, 2},    {128, 256, 64, 2, 1, 2},
    {256, 256, 128, 2, 1, 3},  {512, 128, 128, 4, 1, 2},  {1024, 256, 256, 4, 1, 3},
    {2048, 256, 256, 4, 2, 2}, {4096, 512, 512, 4, 2, 2}, {8192, 512, 512, 4, 4, 2},
    {16384, 512, 512, 4, 8, 2}, {32768, 512, 512, 4, 16, 2},
};
// Cross-entropy backward rows of 256 vectors (fp32 1024, bf16 2048 elements):
// eight 32-thread rows of 8 vectors a thread per CTA, three slots (a row group
// of 128 threads held twice the row: +4 to +18 points at 2048-16384 rows,
// within a point from 24576 on).
const Choice kXentBwdTable[] = {
    {32, 256, 8, 4, 1, 1},     {64, 256, 16, 4, 1, 2},    {128, 256, 32, 4, 1, 2},
    {256, 256, 32, 8, 1, 3},   {512, 128, 128, 4, 1, 1},  {1024, 256, 256, 4, 1, 1},
    {2048, 256, 256, 8, 1, 1}, {kStream, 256, 256, 8, 1, 1},  // 32 KB chunks
};

// Chooses the ring kernel (fast path) for a row of NV 16-byte vectors.
qk_status choose_ring(int op, int dt, int64_t NV, int* th, int* tpr, int* vpt, int* cl, int* k,
                      int* slots) {
#define QK_TABLE(T) t = T, n = int(sizeof(T) / sizeof(Choice))
  const Choice* t;
  int n;
  switch (op) {
    case kSoftmax:
      if (dt == QK_BF16) {
        QK_TABLE(kSoftmaxBf16Table);
      } else {
        QK_TABLE(kSoftmaxTable);
      }
      break;
    case kRmsNorm: QK_TABLE(kRmsNormTable); break;
    case kXent: QK_TABLE(kXentTable); break;
    case kOpSoftmaxBwd: QK_TABLE(kSoftmaxBwdTable); break;
    case kOpRmsNormBwd:
      if (dt == QK_BF16) {
        QK_TABLE(kRmsNormBwdBf16Table);
      } else {
        QK_TABLE(kRmsNormBwdTable);
      }
      break;
    case kOpLayerNorm:
      if (dt == QK_F32) {
        QK_TABLE(kLayerNormF32Table);
      } else {
        QK_TABLE(kLayerNormTable);
      }
      break;
    default: QK_TABLE(kXentBwdTable); break;
  }
#undef QK_TABLE
  for (int i = 0; i < n; ++i) {
    if (NV > t[i].max_nv) continue;
    *th = t[i].threads, *tpr = t[i].row_threads, *vpt = t[i].vec_per_thread;
    *cl = t[i].cluster, *slots = t[i].slots;
    const int64_t per_cta = int64_t(*tpr) * *vpt;
    *k = (t[i].max_nv == kStream) ? int((NV + per_cta - 1) / per_cta) : 1;
    return QK_OK;
  }
  return QK_ERR_UNSUPPORTED;
}

// Rows of the forward softmax / RMSNorm / LayerNorm longer than the largest cluster plan
// (64K vectors, 1 MiB) are streamed twice.  A cluster splits each row when
// there are too few rows to occupy the GPU.
constexpr int64_t kTwoPassChunkVectors = 256 * 8;  // 32 KB chunks
bool wants_two_pass(int op, int64_t NV) {
  return (op == kSoftmax || op == kRmsNorm || op == kOpLayerNorm) &&
         NV > int64_t(kMaxCluster) * kRingMaxVectorsPerCta;
}

// Short launches: items per resident CTA below which the planner raises a
// one-row-per-slot launch to 3 ring slots (t3) or 2 (t2), when that costs no
// resident CTA.  From sweeps of 1-3 slots over 1024-32768 rows and rows of
// 256-16384 elements: a launch of few items per CTA waits mostly on its
// first loads, one of many items streams best from the table's slots.
struct SlotBands {
  int t3, t2;
};
SlotBands slot_bands(int op) {
  if (op == kRmsNorm || op == kOpLayerNorm) return {8, 0};
  if (op == kSoftmax) return {4, 8};
  return {4, 0};
}
// Backward launches below this many items per resident CTA take a ring of
// three slots when that costs no resident CTA, else two when that costs at
// most one CTA per SM, and keep the full grid.  A one-slot ring makes each CTA
// load, reduce and write its items one after another, which a short launch
// cannot hide (same-GPU A/B from graphs of 20-400 calls: softmax backward
// fp32 1024 x 4096 82 % -> 95 %, 2048 x 4096 85 % -> 93 %, bf16 2048 x 4096
// 85 % -> 98 %; cross-entropy backward fp32 4096 x 4096 85 % -> 97 %).
// Three slots at the cost of a CTA measured worse (up to 6 points), and so
// did the balanced short grid below for the two-input passes (softmax
// backward bf16 1024 x 4096: 81 % on the full grid, 67 % balanced); at 9
// items per CTA and more the table's ring was as good or better.
constexpr int kBwdDeepRingItems = 8;
// Forward launches of fewer than this many items per resident CTA (after the
// rules above) take a third ring slot even when that costs up to a third of
// the resident CTAs: with so few items every CTA's loads are in flight at once
// anyway, and the deeper ring keeps all of them in flight.
constexpr int kVeryShortItems = 2;

// Alternative kernels by the length of the launch, in items per resident CTA
// of the table's plan (ipc).  The tables were tuned at 16384 rows; these rows
// hold what measured better on shorter (and, twice, longer) launches:
//  * fp32 softmax rows of 4096 elements below 8: 128-thread CTAs of 8 vectors
//    a thread, with 3 ring slots below 4 and 2 above (1024 x 4096: 86 % ->
//    88 %; 4096 x 4096: 90 % -> 92 %); the 256 x 4 plan beats it by 1-2
//    points from 8192 rows on;
//  * cross-entropy rows of 512 vectors below 4: two 64-thread rows of 8
//    vectors a thread per 128-thread CTA, six CTAs per SM (bf16 2048 x 4096:
//    36 % -> 53 %, 4096 x 4096 64 % -> 68 %; fp32 2048 x 2048 40 % -> 56 %);
//  * backward passes (table plans tuned at 16384 rows and more): softmax
//    rows of 256 vectors below 20, four 64-thread rows of 4 vectors a thread
//    per CTA (+1 to +7 points at 2048-16384 rows); cross-entropy rows of 512
//    vectors from 4 to 10, four 64-thread rows of 8 vectors a thread, three
//    slots (+1 to +8 points at 6144-12288 rows);
//  * RMSNorm (softmax) rows of 512 vectors (bf16 4096, fp32 2048 elements)
//    from 4 to 12 (bf16 softmax 10, fp32 softmax 8): four 64-thread rows of 8
//    vectors a thread per 256-thread CTA, three slots, two CTAs per SM
//    (RMSNorm bf16 8192 x 4096: 89 % -> 95 %, fp32 10240 x 2048 89 % -> 96 %;
//    softmax fp32 6144 x 2048 91 % -> 101 %, bf16 8192 x 4096 89 % -> 94 %);
//    below 4 and from about 16 on the table's 128-thread plan measured as
//    good or better, except for fp32 softmax, whose rows of 2048 elements
//    take one 256-thread row of 2 vectors a thread with two slots from 8 on
//    (16384 x 2048: 91 % -> 96 %, 32768 x 2048 91 % -> 95 %);
//  * RMSNorm and softmax rows of 64 vectors (fp32 256, bf16 512 elements)
//    below 1.5: eight 32-thread rows per CTA, three slots.  The table's
//    sixteen-row CTAs halve the items, so in so short a launch the SMs' shares
//    of the grid come out uneven (RMSNorm fp32 8192 x 256: 66 % eight-row,
//    61 % sixteen-row); from 12288 rows on the sixteen-row plan is ahead
//    (RMSNorm bf16 12288 x 512: 65 % -> 80 %, fp32 24576 x 256: 90 % -> 97 %);
//  * fp32 LayerNorm rows of 128 vectors (512 elements) from 2 to 16: sixteen
//    16-thread rows of 8 vectors a thread per CTA, three slots (8192 x 512:
//    69 % -> 76 %, 24576 x 512: 87 % -> 100 %); at 65536 rows the table's
//    plan measured 4 points ahead;
//  * RMSNorm rows of 2048 vectors (fp32 8192, bf16 16384 elements) from 10
//    on: one 512-thread row of 4 vectors a thread per CTA, two slots, one CTA
//    per SM, where the table's 256 x 8 plan holds two (fp32 16384 x 8192:
//    98 % -> 100 %, 4096 x 8192 93 % -> 96 %; bf16 +1 point); the table's
//    plan stays ahead on shorter launches (2048 rows: 97-98 % against 88-90 %);
//  * fp32 RMSNorm backward rows of 512 vectors (2048 elements) from 32 on:
//    two 128-thread rows per 256-thread CTA, two slots, where the table's
//    plan runs one row per CTA with four (16384 x 2048 90 % -> 92 %, 65536 x
//    2048 96 % -> 100 %; the table's plan 3-7 points ahead at 1024-4096 rows);
//  * fp32 softmax rows of 256 vectors (1024 elements) from 10 on: two
//    128-thread rows of 2 vectors a thread per CTA, two slots (32768 x 1024
//    90 % -> 96 %, 65536 x 1024 91 % -> 94 %; 1-14 points behind below 16384
//    rows);
//  * fp32 LayerNorm rows of 64 vectors (256 elements) from 3 on: thirty-two
//    8-thread rows of 8 vectors a thread per CTA, three slots (16384 x 256
//    72 % -> 78 %, 32768 x 256 87 % -> 93 %; 2-5 points behind below).
// One row of those rules: operator, dtype (-1: both), rows of (nv_lo, nv_hi]
// vectors, a window [ipc_lo2, ipc_hi2) on 2 * ipc (kOpenEnd: no upper end),
// the plan, and 2 * ipc below which it takes three ring slots instead of its
// own count (0: never).
constexpr int kOpenEnd = 1 << 30;
struct LaunchAlt {
  int op, dt;
  int64_t nv_lo, nv_hi;
  int ipc_lo2, ipc_hi2, deep_below2;
  Choice c;
};
const LaunchAlt kLaunchAlts[] = {
    {kSoftmax, QK_F32, 512, 1024, 0, 16, 8, {1024, 128, 128, 8, 1, 2}},
    {kXent, -1, 256, 512, 0, 8, 0, {512, 128, 64, 8, 1, 2}},
    {kOpSoftmaxBwd, -1, 128, 256, 0, 40, 16, {256, 256, 64, 4, 1, 2}},
    {kOpXentBwd, -1, 256, 512, 8, 20, 0, {512, 256, 64, 8, 1, 3}},
    {kRmsNorm, -1, 256, 512, 8, 24, 0, {512, 256, 64, 8, 1, 3}},
    {kSoftmax, QK_BF16, 256, 512, 8, 20, 0, {512, 256, 64, 8, 1, 3}},
    {kSoftmax, QK_F32, 256, 512, 8, 16, 0, {512, 256, 64, 8, 1, 3}},
    {kSoftmax, QK_F32, 256, 512, 16, kOpenEnd, 0, {512, 256, 256, 2, 1, 2}},
    {kRmsNorm, -1, 32, 64, 0, 3, 0, {64, 256, 32, 2, 1, 3}},
    {kSoftmax, -1, 32, 64, 0, 3, 0, {64, 256, 32, 2, 1, 3}},
    {kOpLayerNorm, QK_F32, 64, 128, 4, 32, 0, {128, 256, 16, 8, 1, 3}},
    {kRmsNorm, -1, 1024, 2048, 20, kOpenEnd, 0, {2048, 512, 512, 4, 1, 2}},
    {kOpRmsNormBwd, QK_F32, 256, 512, 64, kOpenEnd, 0, {512, 256, 128, 4, 1, 2}},
    {kSoftmax, QK_F32, 128, 256, 20, kOpenEnd, 0, {256, 256, 128, 2, 1, 2}},
    {kOpLayerNorm, QK_F32, 32, 64, 6, kOpenEnd, 0, {64, 256, 8, 8, 1, 3}},
};
bool launch_alternative(int op, int dt, int64_t NV, int64_t items, int64_t resident, Choice* c) {
  for (const LaunchAlt& a : kLaunchAlts) {
    if (a.op != op || (a.dt >= 0 && a.dt != dt) || NV <= a.nv_lo || NV > a.nv_hi) continue;
    if (2 * items < a.ipc_lo2 * resident || 2 * items >= a.ipc_hi2 * resident) continue;
    *c = a.c;
    if (2 * items < a.deep_below2 * resident) c->slots = 3;
    return true;
  }
  return false;
}

qk_status plan_ring(int dev, const DeviceInfo& d, int op, int dt, int64_t M, int64_t N, Plan* p,
                    const Choice* alt = nullptr) {
  const int E = 16 / elem_size(dt);
  const int64_t NV = N / E;
  int th, tpr, vpt, cl, k;
  int slots = 0;
  bool two_pass = false;
  const Override& ov = g_override[op][dt];
  if (ov.on && ov.plan.path == 4) {  // forced two-pass plan (tuning, tests)
    if (!(op == kSoftmax || op == kRmsNorm || op == kOpLayerNorm)) return QK_ERR_UNSUPPORTED;
    th = ov.plan.threads, tpr = ov.plan.row_threads, vpt = ov.plan.vec_per_thread;
    cl = std::max(1, int(ov.plan.cluster));
    slots = ov.plan.slots;
    if (cl > kMaxCluster || tpr != th) return QK_ERR_UNSUPPORTED;
    const int64_t per_cta = int64_t(tpr) * vpt;
    k = int(((NV + cl - 1) / cl + per_cta - 1) / per_cta);
    two_pass = true;
  } else if (!ov.on && wants_two_pass(op, NV)) {
    th = 256, tpr = 256, vpt = 8, slots = 3;
    const int64_t want = 2 * int64_t(d.sms);  // row slices in flight
    cl = 1;
    while (cl < kMaxCluster && M * cl < want) cl <<= 1;
    k = int(((NV + cl - 1) / cl + kTwoPassChunkVectors - 1) / kTwoPassChunkVectors);
    two_pass = true;
  } else if (ov.on) {
    th = ov.plan.threads, tpr = ov.plan.row_threads, vpt = ov.plan.vec_per_thread;
    cl = std::max(1, int(ov.plan.cluster));
    slots = ov.plan.slots;
    const int64_t per_cta = int64_t(tpr) * vpt;
    const int64_t slice = (NV + cl - 1) / cl;
    if (cl > kMaxCluster || (cl > 1 && tpr != th)) return QK_ERR_UNSUPPORTED;
    if (slice <= per_cta) {
      k = 1;
    } else if (streams_rows(op) && cl == 1 && tpr == th) {
      k = int((NV + per_cta - 1) / per_cta);
    } else {
      return QK_ERR_UNSUPPORTED;
    }
  } else if (alt != nullptr) {
    th = alt->threads, tpr = alt->row_threads, vpt = alt->vec_per_thread;
    cl = alt->cluster, slots = alt->slots, k = 1;
  } else {
    qk_status st = choose_ring(op, dt, NV, &th, &tpr, &vpt, &cl, &k, &slots);
    if (st != QK_OK) return st;
  }
  const KernelEntry* ke =
      find_kernel(op, dt, two_pass ? 4 : (is_bwd(op) ? 3 : 1), th, tpr, vpt, cl > 1);
  if (ke == nullptr) return QK_ERR_UNSUPPORTED;
  const int nin = inputs_per_item(op);

  int64_t item_bytes;
  if (two_pass) {
    item_bytes = int64_t(tpr) * vpt * 16;
    p->num_items = M;
  } else if (k > 1) {
    item_bytes = int64_t(tpr) * vpt * 16;
    p->num_items = M;
  } else if (cl > 1) {
    item_bytes = (NV + cl - 1) / cl * 16;
    p->num_items = M;
  } else {
    const int R = th / tpr;
    item_bytes = int64_t(R) * NV * 16;
    p->num_items = (M + R - 1) / R;
  }
  const uint32_t slot_bytes = uint32_t((item_bytes + 127) / 128 * 128);
  // LayerNorm parameters not held in registers sit after the ring slots.
  int64_t param_bytes = 0;
  if (op == kOpLayerNorm && !two_pass) {  // streamed rows read w and b through L1
    const int64_t slice = cl > 1 ? (NV + cl - 1) / cl : NV;
    if (vpt > kAffineRegsMaxVpt) param_bytes += param_slice_bytes(slice);
    if (vpt > kLnBiasRegsMaxVpt) param_bytes += param_slice_bytes(slice);
  }
  if (slots <= 0) slots = 2;  // an override without a slot count
  slots = std::min(slots, kMaxSlots);
  while (slots > 1 && kSmemHeader + int64_t(slots) * nin * slot_bytes + param_bytes > d.smem_optin)
    --slots;
  const int64_t smem = kSmemHeader + int64_t(slots) * nin * slot_bytes + param_bytes;
  if (smem > d.smem_optin) return QK_ERR_UNSUPPORTED;

  qk_status st = prepare_kernel(dev, d, *ke);
  if (st != QK_OK) return st;
  int occ = 0;
  st = occupancy(dev, *ke, int(smem), cl > 1 ? cl : 0, &occ);
  if (st != QK_OK) return st;
  if (occ <= 0) return QK_ERR_UNSUPPORTED;
  // CTAs per SM the launch can hold (clusters: resident clusters' CTAs over the SMs)
  int64_t ctas_per_sm = cl > 1 ? std::max<int64_t>(1, int64_t(occ) * cl / std::max(1, d.sms)) : occ;

  // Short launches spend most of their time waiting for their first loads:
  // below the operator's bands of items per resident CTA, give each CTA a
  // ring of three (or two) slots, if that costs no resident CTA (backward
  // launches: two slots may cost one, see kBwdDeepRingItems).  (Softmax
  // fp32 1024 x 4096: 70 % -> 75 %; 2048 x 4096: 76 % -> 97 %; RMSNorm bf16
  // 16384 x 1024: 90 % -> 98 %.)
  const bool short_ok = !ov.on && !two_pass && k == 1 && cl == 1;
  const int64_t resident = ctas_per_sm * d.sms;
  if (short_ok && alt == nullptr) {
    Choice c;
    if (launch_alternative(op, dt, NV, p->num_items, resident, &c) &&
        !(c.threads == th && c.row_threads == tpr && c.vec_per_thread == vpt))
      return plan_ring(dev, d, op, dt, M, N, p, &c);  // its slots as given
  }
  int64_t smem_used = smem;
  const SlotBands band = slot_bands(op);
  const bool bwd = is_bwd(op);
  const int want = !short_ok || alt != nullptr                               ? 0
                   : bwd ? (p->num_items < kBwdDeepRingItems * resident ? 3 : 0)
                   : p->num_items < band.t3 * resident                      ? 3
                   : p->num_items < band.t2 * resident                      ? 2
                                                                             : 0;
  for (int s = want; s > slots; --s) {
    const int64_t smem_s = kSmemHeader + int64_t(s) * nin * slot_bytes + param_bytes;
    const int min_occ = (bwd && s == 2) ? std::max(1, occ - 1) : occ;  // see kBwdDeepRingItems
    int occ_s = 0;
    if (smem_s <= d.smem_optin && occupancy(dev, *ke, int(smem_s), 0, &occ_s) == QK_OK &&
        occ_s >= min_occ) {
      slots = s;
      smem_used = smem_s;
      occ = occ_s;  // unclustered here: the grid below follows the new residency
      ctas_per_sm = occ_s;
      break;
    }
  }
  // A forward launch of fewer than two items per resident CTA: a third slot
  // even at the cost of up to a third of the resident CTAs (see kVeryShortItems).
  if (short_ok && !bwd && slots < 3 && p->num_items < kVeryShortItems * int64_t(occ) * d.sms) {
    const int64_t smem_s = kSmemHeader + int64_t(3) * nin * slot_bytes + param_bytes;
    int occ_s = 0;
    if (smem_s <= d.smem_optin && occupancy(dev, *ke, int(smem_s), 0, &occ_s) == QK_OK &&
        3 * occ_s >= 2 * occ && occ_s > 0) {
      slots = 3;
      smem_used = smem_s;
      occ = occ_s;
      ctas_per_sm = occ_s;
    }
  }

  p->kernel = ke;
  p->cluster = cl;
  p->slots = slots;
  p->chunks = k;
  p->slot_bytes = slot_bytes;
  p->smem = int(smem_used);
  // Persistent grid: every resident CTA (or cluster) once, at most one per item.
  int64_t units = cl > 1 ? int64_t(occ) : int64_t(occ) * d.sms;
  if (ov.on && ov.plan.grid > 0) units = std::min<int64_t>(units, std::max(1, ov.plan.grid / cl));
  units = std::min<int64_t>(units, p->num_items);
  // A launch of fewer than two items per CTA lasts as long as its busiest
  // CTA: give every CTA the same number (softmax fp32 1024 x 4096: 512 CTAs of
  // two rows rather than 608 of one or two, 86 % -> 87 %; cross-entropy
  // backward fp32 1024 x 4096 +2 points).  At three or more items per CTA the
  // full grid measured better, and so it did for the backward passes that
  // load two matrices per item (softmax, RMSNorm; see kBwdDeepRingItems) and
  // for softmax, RMSNorm and LayerNorm CTAs of several rows, whose shrunken
  // grid leaves some SMs one CTA and others two (same-GPU A/B: +4 to +11
  // points, softmax bf16 4096 x 1024 52 % -> 63 %; cross-entropy, forward and
  // backward, measured 1-3 points better with even shares).
  const bool rows_per_cta = th > tpr && (op == kSoftmax || op == kRmsNorm || op == kOpLayerNorm);
  if (short_ok && nin == 1 && !rows_per_cta && p->num_items < 2 * units) {
    const int64_t per = (p->num_items + units - 1) / units;
    units = (p->num_items + per - 1) / per;
  }
  p->ctas_per_sm = int(ctas_per_sm);
  p->grid = units * cl;
  return QK_OK;
}

// Rows that do not start on a 16-byte boundary (shifted ring kernel): each
// step copies the aligned range around its elements, so a row group must hold
// ceil((15 + slice bytes) / 16) vectors: one more than the aligned row when
// it is misaligned, hence row groups of 5 (or 9) vectors a thread.  Row groups
// from 8 to 256 threads of 5 or 9 vectors (the smallest that holds the row),
// then the smallest cluster
// of 256 x 9 CTAs (256 x 8 when the slice fits: fewer registers) for softmax / RMSNorm /
// LayerNorm; cross-entropy streams longer rows in equal chunks of at most 2303
// vectors.
struct ShiftChoice {
  int threads, row_threads, vec_per_thread, slots;
};
// In order of capacity (row_threads x vec_per_thread vectors): the first that
// holds the row is the one with the least padding.
constexpr ShiftChoice kShiftTable[] = {
    {256, 8, 5, 2},   {256, 16, 5, 2},  {256, 16, 9, 2},  {256, 32, 5, 2},
    {256, 32, 9, 2},  {256, 64, 5, 2},  {256, 64, 9, 2},  {256, 128, 5, 2},
    {256, 128, 9, 2}, {256, 256, 5, 2}, {256, 256, 9, 1},
};
int64_t span_vectors(int64_t elems, int es) { return (15 + elems * es + 15) / 16; }

qk_status plan_shifted(int dev, const DeviceInfo& d, int op, int dt, int64_t M, int64_t N, Plan* p) {
  const int es = elem_size(dt);
  const int kinds = int(sizeof(kShiftTable) / sizeof(ShiftChoice));
  const int last = kinds - 1;
  const bool streams = (op == kXent || op == kOpXentBwd);  // no row reduction to keep
  int pick = -1, cl = 1, k = 1;
  // LayerNorm and softmax backward hold two CTAs per SM at 9 vectors a thread
  // (counts, or a second input): their narrow row groups stay at 5 vectors.
  const bool narrow9 = !(op == kOpLayerNorm || op == kOpSoftmaxBwd);
  for (int i = 0; i <= last && pick < 0; ++i) {
    const ShiftChoice& c = kShiftTable[i];
    if (c.vec_per_thread == 9 && c.row_threads < 256 && !narrow9) continue;
    if (span_vectors(N, es) <= int64_t(c.row_threads) * c.vec_per_thread) pick = i;
  }
  if (pick < 0 && streams) {  // stream the row in chunks of (cap - 1) vectors
    pick = last;
    const int64_t che = (int64_t(kShiftTable[pick].row_threads) * kShiftTable[pick].vec_per_thread - 1) *
                        (16 / es);
    k = int((N + che - 1) / che);
  }
  ShiftChoice c = pick >= 0 ? kShiftTable[pick] : ShiftChoice{256, 256, 8, 1};
  if (pick < 0) {  // the smallest cluster of 256 x 9 CTAs, as 256 x 8 when that fits too
    cl = 2;
    while (cl <= kMaxCluster && span_vectors((N + cl - 1) / cl, es) > 256 * 9) cl <<= 1;
    if (cl > kMaxCluster) return QK_ERR_UNSUPPORTED;
    c.vec_per_thread = span_vectors((N + cl - 1) / cl, es) <= 256 * 8 ? 8 : 9;
  }
  const KernelEntry* ke = find_kernel(op, dt, 6, c.threads, c.row_threads, c.vec_per_thread, cl > 1);
  if (ke == nullptr) return QK_ERR_UNSUPPORTED;
  const int R = c.threads / c.row_threads;
  int64_t item_bytes;
  if (k > 1) {
    item_bytes = int64_t(c.row_threads) * c.vec_per_thread * 16;
    p->num_items = M;
  } else if (cl > 1) {
    item_bytes = span_vectors((N + cl - 1) / cl, es) * 16;
    p->num_items = M;
  } else {
    item_bytes = span_vectors(int64_t(R) * N, es) * 16;
    p->num_items = (M + R - 1) / R;
  }
  const uint32_t slot_bytes = uint32_t((item_bytes + 127) / 128 * 128);
  int64_t param_bytes = 0;  // staged w (and b), element slices of the CTA
  if (op == kRmsNorm || op == kOpLayerNorm) {
    const int64_t slice = ((N + cl - 1) / cl * es + 15) / 16;
    param_bytes = param_slice_bytes(slice) * (op == kOpLayerNorm ? 2 : 1);
  }
  const int nin = op == kOpSoftmaxBwd ? 2 : 1;  // y and dy share each slot
  // Forward cross-entropy keeps nothing of a row but its running pair, so the
  // 256 x 9 groups take a second slot to overlap the next chunk's copy with
  // this one (16384 x 50257 bf16: 80 % -> 95 %); the operators that hold the
  // row in registers measured slower with it (softmax, RMSNorm, and the
  // backward, whose stores share the SM's bandwidth).
  int slots = op == kXent ? std::max(c.slots, 2) : c.slots;
  while (slots > 1 && kSmemHeader + int64_t(slots) * nin * slot_bytes + param_bytes > d.smem_optin)
    --slots;
  const int64_t smem = kSmemHeader + int64_t(slots) * nin * slot_bytes + param_bytes;
  if (smem > d.smem_optin) return QK_ERR_UNSUPPORTED;
  qk_status st = prepare_kernel(dev, d, *ke);
  if (st != QK_OK) return st;
  int occ = 0;
  st = occupancy(dev, *ke, int(smem), cl > 1 ? cl : 0, &occ);
  if (st != QK_OK) return st;
  if (occ <= 0) return QK_ERR_UNSUPPORTED;
  p->kernel = ke;
  p->cluster = cl;
  p->slots = slots;
  p->chunks = k;
  p->slot_bytes = slot_bytes;
  p->smem = int(smem);
  int64_t units = cl > 1 ? int64_t(occ) : int64_t(occ) * d.sms;
  units = std::min<int64_t>(units, p->num_items);
  p->ctas_per_sm = cl > 1 ? std::max(1, occ * cl / std::max(1, d.sms)) : occ;
  p->grid = units * cl;
  return QK_OK;
}

// Masked direct path: one row per CTA, or per cluster for long rows.
qk_status plan_direct(int dev, const DeviceInfo& d, int op, int dt, int64_t M, int64_t N, Plan* p) {
  int th, ept, cl = 1;
  bool clustered = false;
  if (N <= 512) th = 128, ept = 4;
  else if (N <= 4096) th = 256, ept = 16;
  else if (N <= 16384 || op == kXent) th = 512, ept = 32;
  else {
    th = 512, ept = 64;
    clustered = true;
    const int64_t c = (N + 32767) / 32768;
    if (c > kMaxCluster) return QK_ERR_UNSUPPORTED;
    cl = next_pow2(c);
  }
  const KernelEntry* ke = find_kernel(op, dt, 2, th, th, ept, clustered);
  if (ke == nullptr) return QK_ERR_UNSUPPORTED;
  if (M * cl > int64_t(INT32_MAX)) return QK_ERR_UNSUPPORTED;
  qk_status st = prepare_kernel(dev, d, *ke);
  if (st != QK_OK) return st;
  p->kernel = ke;
  p->cluster = cl;
  p->slots = 0;
  p->chunks = op == kXent ? int((N + int64_t(th) * ept - 1) / (int64_t(th) * ept)) : 1;
  p->num_items = M;
  p->slot_bytes = 0;
  p->smem = 0;
  p->ctas_per_sm = 0;
  p->grid = M * cl;
  return QK_OK;
}

int64_t max_row_elements(int op, int dt) {
  if (streams_rows(op) || op == kSoftmax || op == kRmsNorm || op == kOpLayerNorm)
    return INT64_MAX;  // streamed rows
  if (is_bwd(op)) return kMaxRowBytes / 2 / elem_size(dt);  // 512 KiB rows (two inputs)
  return kMaxRowBytes / elem_size(dt);
}

qk_status launch(const Plan& p, void* args, void* stream) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.gridDim = dim3(unsigned(p.grid), 1, 1);
  cfg.blockDim = dim3(unsigned(p.kernel->threads), 1, 1);
  cfg.dynamicSmemBytes = size_t(p.smem);
  cfg.stream = static_cast<cudaStream_t>(stream);
  // The kernels wait for the previous grid (griddepcontrol.wait) before their
  // first global access, so they may be launched before it finishes.
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.kernel->clustered) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = unsigned(p.cluster);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  void* params[] = {args};
  if (cudaLaunchKernelExC(&cfg, p.kernel->func, params) != cudaSuccess) {
    cudaGetLastError();
    return QK_ERR_LAUNCH;
  }
  return QK_OK;
}

// Forward kernels: the ring (16-byte aligned rows), the shifted ring (rows
// that start anywhere, x and y with the same alignment modulo 16), the masked
// direct kernel (everything else, and shifted rows beyond its capacity).
enum RowPath : int { kPathDirect = 0, kPathRing = 1, kPathShifted = 2 };

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }
bool same_mod16(const void* a, const void* b) {
  return ((reinterpret_cast<uintptr_t>(a) ^ reinterpret_cast<uintptr_t>(b)) & 15u) == 0;
}
int row_path(bool fast, bool same_alignment) {
  return fast ? kPathRing : same_alignment ? kPathShifted : kPathDirect;
}
bool aligned_to(const void* ptr, size_t n) { return (reinterpret_cast<uintptr_t>(ptr) % n) == 0; }

// [a, a+na) and [b, b+nb) share a byte.
bool overlap(const void* a, int64_t na, const void* b, int64_t nb) {
  if (a == nullptr || b == nullptr || na <= 0 || nb <= 0) return false;
  const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
  return pa < pb + uintptr_t(nb) && pb < pa + uintptr_t(na);
}

qk_status check_sizes(int op, int dt, int64_t M, int64_t N) {
  if (dt != QK_F32 && dt != QK_BF16) return QK_ERR_INVALID_ARG;
  if (M < 0 || N <= 0) return QK_ERR_INVALID_ARG;
  if (M > 0 && N > INT64_MAX / 16 / M) return QK_ERR_INVALID_ARG;  // byte offsets fit int64
  if (N > max_row_elements(op, dt)) return QK_ERR_UNSUPPORTED;
  return QK_OK;
}

// Shared tail of the three entry points: plan, fill args, launch.
qk_status run(int op, int dt, RowArgs a, int path, void* stream) {
  int dev;
  DeviceInfo* d;
  qk_status st = device_info(&dev, &d);
  if (st != QK_OK) return st;
  // Per-thread cache of the last plan of each (op, dtype, path): repeated
  // calls with the same shape skip the table walk and the occupancy queries.
  struct Cached {
    int dev = -1;
    int64_t M = -1, N = -1;
    uint64_t gen = 0;
    Plan plan;
  };
  // (softmax, RMSNorm, x-entropy, LayerNorm, x-entropy and softmax backward) x dtype x path
  thread_local Cached cache[6][2][3];
  const int oi = op == kOpLayerNorm ? 3 : op == kOpXentBwd ? 4 : op == kOpSoftmaxBwd ? 5 : op;
  Cached& c = cache[oi][dt][path];
  const uint64_t gen = g_override_gen.load(std::memory_order_acquire);
  if (!(c.dev == dev && c.M == a.M && c.N == a.N && c.gen == gen)) {
    Plan np;
    if (path == kPathRing) {
      st = plan_ring(dev, *d, op, dt, a.M, a.N, &np);
    } else if (path == kPathShifted) {
      st = plan_shifted(dev, *d, op, dt, a.M, a.N, &np);
      if (st == QK_ERR_UNSUPPORTED && !is_bwd(op)) st = plan_direct(dev, *d, op, dt, a.M, a.N, &np);
    } else {
      st = plan_direct(dev, *d, op, dt, a.M, a.N, &np);
    }
    if (st != QK_OK) return st;
    c.dev = dev, c.M = a.M, c.N = a.N, c.gen = gen, c.plan = np;
  }
  const Plan& p = c.plan;
  a.chunks = p.chunks;
  a.chunk_elems = (a.N + p.chunks - 1) / p.chunks;
  a.slots = p.slots;
  a.slot_bytes = p.slot_bytes;
  a.num_items = p.num_items;
  a.timeout_ns = kWaitTimeoutNs;
  a.inv_n = float(1.0 / double(a.N));
  a.status = d->status;
  return launch(p, &a, stream);
}

// Rows of fp32 dw partials a backward RMSNorm launch writes (one per CTA, or
// per cluster), hence its workspace: rows * N * 4 bytes.
int64_t dw_partial_rows(const Plan& p) { return p.grid / std::max(1, p.cluster); }

// Masked backward path: a persistent grid of one-row CTAs (or clusters for
// rows beyond 8192 elements), each thread holding up to 16 elements of each
// input in registers, so rows are limited to kMaskedBwdMaxRow elements.
// Cross-entropy streams any row in chunks.
qk_status plan_direct_bwd(int dev, const DeviceInfo& d, int op, int dt, int64_t M, int64_t N,
                          Plan* p) {
  int th, ept, cl = 1;
  if (op == kOpXentBwd) {
    th = 256, ept = 8;
  } else if (N <= 512) {
    th = 128, ept = 4;
  } else if (N <= 2048) {
    th = 256, ept = 8;
  } else if (N <= 8192) {
    th = 512, ept = 16;
  } else {
    if (N > kMaskedBwdMaxRow) return QK_ERR_UNSUPPORTED;
    th = 512, ept = 16;
    cl = next_pow2((N + 8191) / 8192);
  }
  const KernelEntry* ke = find_kernel(op, dt, 5, th, th, ept, cl > 1);
  if (ke == nullptr) return QK_ERR_UNSUPPORTED;
  qk_status st = prepare_kernel(dev, d, *ke);
  if (st != QK_OK) return st;
  int occ = 0;
  st = occupancy(dev, *ke, 0, cl > 1 ? cl : 0, &occ);
  if (st != QK_OK) return st;
  if (occ <= 0) return QK_ERR_UNSUPPORTED;
  const int64_t units = std::min<int64_t>(M, cl > 1 ? int64_t(occ) : int64_t(occ) * d.sms);
  p->kernel = ke;
  p->cluster = cl;
  p->slots = 0;
  p->chunks = 1;
  p->num_items = M;
  p->slot_bytes = 0;
  p->smem = 0;
  p->ctas_per_sm = cl > 1 ? std::max(1, occ * cl / std::max(1, d.sms)) : occ;
  p->grid = units * cl;
  return QK_OK;
}

qk_status plan_bwd_cached(int op, int dt, int64_t M, int64_t N, bool fast, int* dev,
                          DeviceInfo** d, const Plan** out) {
  qk_status st = device_info(dev, d);
  if (st != QK_OK) return st;
  struct Cached {
    int dev = -1;
    int64_t M = -1, N = -1;
    uint64_t gen = 0;
    Plan plan;
  };
  thread_local Cached cache[3][2][2];  // (op, dtype, ring or masked)
  Cached& c = cache[op - kOpSoftmaxBwd][dt][fast ? 1 : 0];
  const uint64_t gen = g_override_gen.load(std::memory_order_acquire);
  if (!(c.dev == *dev && c.M == M && c.N == N && c.gen == gen)) {
    Plan np;
    st = fast ? plan_ring(*dev, **d, op, dt, M, N, &np) : plan_direct_bwd(*dev, **d, op, dt, M, N, &np);
    if (st != QK_OK) return st;
    c.dev = *dev, c.M = M, c.N = N, c.gen = gen, c.plan = np;
  }
  *out = &c.plan;
  return QK_OK;
}

// Backward launch: the ring kernel (or the masked one), then (RMSNorm) the
// fixed-order dw sum.
qk_status run_bwd(int op, int dt, BwdArgs a, float* dw, size_t workspace_bytes, bool fast,
                  void* stream) {
  int dev;
  DeviceInfo* d;
  const Plan* pp;
  qk_status st = plan_bwd_cached(op, dt, a.M, a.N, fast, &dev, &d, &pp);
  if (st != QK_OK) return st;
  const Plan& p = *pp;
  const int64_t rows = dw_partial_rows(p);
  if (op == kOpRmsNormBwd && workspace_bytes < size_t(rows) * size_t(a.N) * 4)
    return QK_ERR_INVALID_ARG;
  a.chunks = p.chunks;
  a.slots = p.slots;
  a.slot_bytes = p.slot_bytes;
  a.num_items = p.num_items;
  a.timeout_ns = kWaitTimeoutNs;
  a.inv_n = float(1.0 / double(a.N));
  a.status = d->status;
  st = launch(p, &a, stream);
  if (st != QK_OK || op != kOpRmsNormBwd) return st;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(unsigned((a.N + 31) / 32), 1, 1);
  cfg.blockDim = dim3(kDwReduceThreads, 1, 1);
  cfg.stream = static_cast<cudaStream_t>(stream);
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const float* part = a.dw_partial;
  int64_t n = a.N;
  if (cudaLaunchKernelEx(&cfg, dw_reduce_kernel<0>, part, dw, rows, n) != cudaSuccess) {
    cudaGetLastError();
    return QK_ERR_LAUNCH;
  }
  return QK_OK;
}

}  // namespace
}  // namespace qk

using namespace qk;

extern "C" {

const char* qk_status_string(qk_status s) {
  switch (s) {
    case QK_OK: return "ok";
    case QK_ERR_INVALID_ARG: return "invalid argument";
    case QK_ERR_UNSUPPORTED: return "unsupported size or plan";
    case QK_ERR_MISALIGNED: return "pointer not aligned to its element size";
    case QK_ERR_LAUNCH: return "CUDA launch or query failed";
    case QK_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out";
    case QK_ERR_NO_DEVICE: return "no usable sm_103 CUDA device";
  }
  return "unknown status";
}

int64_t qk_max_row_elements(qk_op op, qk_dtype dtype) {
  if (op < 0 || op >= kNumOps || (dtype != QK_F32 && dtype != QK_BF16)) return 0;
  return max_row_elements(op, dtype);
}

qk_status qk_softmax_fwd(const void* x, void* y, int64_t M, int64_t N, qk_dtype dtype,
                         void* stream) {
  qk_status st = check_sizes(kSoftmax, dtype, M, N);
  if (st != QK_OK) return st;
  if (M == 0) return QK_OK;
  if (x == nullptr || y == nullptr) return QK_ERR_INVALID_ARG;
  const size_t es = size_t(elem_size(dtype));
  if (!aligned_to(x, es) || !aligned_to(y, es)) return QK_ERR_MISALIGNED;
  const int64_t bytes = M * N * int64_t(es);
  if (x != y && overlap(x, bytes, y, bytes)) return QK_ERR_INVALID_ARG;
  RowArgs a = {};
  a.x = x;
  a.y = y;
  a.M = M;
  a.N = N;
  const bool fast = aligned16(x) && aligned16(y) && (N * int64_t(es)) % 16 == 0;
  if (!fast && N > kMaskedMaxRow) return QK_ERR_UNSUPPORTED;
  return run(kSoftmax, dtype, a, row_path(fast, same_mod16(x, y)), stream);
}

qk_status qk_rmsnorm_fwd(const void* x, const void* w, void* y, float* rstd, int64_t M,
                         int64_t N, float eps, qk_dtype dtype, void* stream) {
  qk_status st = check_sizes(kRmsNorm, dtype, M, N);
  if (st != QK_OK) return st;
  if (!(std::isfinite(eps) && eps >= 0.f)) return QK_ERR_INVALID_ARG;
  if (M == 0) return QK_OK;
  if (x == nullptr || w == nullptr || y == nullptr) return QK_ERR_INVALID_ARG;
  const size_t es = size_t(elem_size(dtype));
  if (!aligned_to(x, es) || !aligned_to(y, es) || !aligned_to(w, es) || !aligned_to(rstd, 4))
    return QK_ERR_MISALIGNED;
  const int64_t bytes = M * N * int64_t(es), wbytes = N * int64_t(es), rbytes = M * 4;
  if ((x != y && overlap(x, bytes, y, bytes)) || overlap(y, bytes, w, wbytes) ||
      overlap(rstd, rbytes, x, bytes) || overlap(rstd, rbytes, y, bytes) ||
      overlap(rstd, rbytes, w, wbytes))
    return QK_ERR_INVALID_ARG;
  RowArgs a = {};
  a.x = x;
  a.w = w;
  a.y = y;
  a.rstd = rstd;
  a.M = M;
  a.N = N;
  a.eps = eps;
  const bool fast =
      aligned16(x) && aligned16(y) && aligned16(w) && (N * int64_t(es)) % 16 == 0;
  if (!fast && N > kMaskedMaxRow) return QK_ERR_UNSUPPORTED;
  return run(kRmsNorm, dtype, a, row_path(fast, same_mod16(x, y)), stream);
}

qk_status qk_layernorm_fwd(const void* x, const void* w, const void* b, void* y, float* mean,
                           float* rstd, int64_t M, int64_t N, float eps, qk_dtype dtype,
                           void* stream) {
  qk_status st = check_sizes(kOpLayerNorm, dtype, M, N);
  if (st != QK_OK) return st;
  if (!(std::isfinite(eps) && eps >= 0.f)) return QK_ERR_INVALID_ARG;
  if (M == 0) return QK_OK;
  if (x == nullptr || w == nullptr || y == nullptr) return QK_ERR_INVALID_ARG;
  const size_t es = size_t(elem_size(dtype));
  if (!aligned_to(x, es) || !aligned_to(y, es) || !aligned_to(w, es) || !aligned_to(b, es) ||
      !aligned_to(mean, 4) || !aligned_to(rstd, 4))
    return QK_ERR_MISALIGNED;
  const int64_t bytes = M * N * int64_t(es), wbytes = N * int64_t(es), rbytes = M * 4;
  if ((x != y && overlap(x, bytes, y, bytes)) || overlap(y, bytes, w, wbytes) ||
      overlap(y, bytes, b, wbytes))
    return QK_ERR_INVALID_ARG;
  for (const float* o : {mean, rstd}) {  // the per-row outputs overlap nothing
    if (overlap(o, rbytes, x, bytes) || overlap(o, rbytes, y, bytes) ||
        overlap(o, rbytes, w, wbytes) || overlap(o, rbytes, b, wbytes))
      return QK_ERR_INVALID_ARG;
  }
  if (overlap(mean, rbytes, rstd, rbytes)) return QK_ERR_INVALID_ARG;
  RowArgs a = {};
  a.x = x;
  a.w = w;
  a.bias = b;
  a.y = y;
  a.mean = mean;
  a.rstd = rstd;
  a.M = M;
  a.N = N;
  a.eps = eps;
  const bool fast = aligned16(x) && aligned16(y) && aligned16(w) && aligned16(b) &&
                    (N * int64_t(es)) % 16 == 0;
  if (!fast && N > kMaskedMaxRow) return QK_ERR_UNSUPPORTED;
  return run(kOpLayerNorm, dtype, a, row_path(fast, same_mod16(x, y)), stream);
}

qk_status qk_xent_fwd_ex(const void* logits, const int64_t* targets, float* loss, float* lse,
                         float* mean_loss, int64_t M, int64_t N, qk_dtype dtype,
                         const qk_xent_options* options, void* stream) {
  const int has_ignore = options != nullptr && options->has_ignore_index != 0;
  const int64_t ignore = has_ignore ? options->ignore_index : 0;
  const float z = options != nullptr ? options->z_loss : 0.f;
  qk_status st = check_sizes(kXent, dtype, M, N);
  if (st != QK_OK) return st;
  if (!std::isfinite(z)) return QK_ERR_INVALID_ARG;
  if (M == 0) return QK_OK;
  if (logits == nullptr || targets == nullptr || loss == nullptr) return QK_ERR_INVALID_ARG;
  const size_t es = size_t(elem_size(dtype));
  if (!aligned_to(logits, es) || !aligned_to(targets, 8) || !aligned_to(loss, 4) ||
      !aligned_to(lse, 4) || !aligned_to(mean_loss, 4))
    return QK_ERR_MISALIGNED;
  const int64_t bytes = M * N * int64_t(es), tbytes = M * 8, obytes = M * 4;
  if (overlap(loss, obytes, logits, bytes) || overlap(loss, obytes, targets, tbytes) ||
      overlap(loss, obytes, lse, obytes) || overlap(lse, obytes, logits, bytes) ||
      overlap(lse, obytes, targets, tbytes) || overlap(mean_loss, 4, logits, bytes) ||
      overlap(mean_loss, 4, targets, tbytes) || overlap(mean_loss, 4, loss, obytes) ||
      overlap(mean_loss, 4, lse, obytes))
    return QK_ERR_INVALID_ARG;
  RowArgs a = {};
  a.x = logits;
  a.target = targets;
  a.loss = loss;
  a.lse = lse;
  a.M = M;
  a.N = N;
  a.ignore_index = ignore;
  a.has_ignore = has_ignore;
  a.z_loss = z;
  const bool fast = aligned16(logits) && (N * int64_t(es)) % 16 == 0;
  st = run(kXent, dtype, a, row_path(fast, true), stream);
  if (st != QK_OK || mean_loss == nullptr) return st;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(1, 1, 1);
  cfg.blockDim = dim3(1024, 1, 1);
  cfg.stream = static_cast<cudaStream_t>(stream);
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const float* lp = loss;
  if (cudaLaunchKernelEx(&cfg, xent_mean_kernel<0>, lp, targets, M, has_ignore, ignore, mean_loss) !=
      cudaSuccess) {
    cudaGetLastError();
    return QK_ERR_LAUNCH;
  }
  return QK_OK;
}

qk_status qk_xent_fwd(const void* logits, const int64_t* targets, float* loss, float* lse,
                      int64_t M, int64_t N, qk_dtype dtype, void* stream) {
  return qk_xent_fwd_ex(logits, targets, loss, lse, nullptr, M, N, dtype, nullptr, stream);
}

// Fast-path requirements of the backward passes: 16-byte aligned rows.
static bool bwd_aligned(int dt, int64_t N, std::initializer_list<const void*> ptrs) {
  if ((N * int64_t(elem_size(dt))) % 16 != 0) return false;
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return false;
  return true;
}

qk_status qk_softmax_bwd(const void* y, const void* dy, void* dx, int64_t M, int64_t N,
                         qk_dtype dtype, void* stream) {
  qk_status st = check_sizes(kOpSoftmaxBwd, dtype, M, N);
  if (st != QK_OK) return st;
  if (M == 0) return QK_OK;
  if (y == nullptr || dy == nullptr || dx == nullptr) return QK_ERR_INVALID_ARG;
  const size_t es = size_t(elem_size(dtype));
  if (!aligned_to(y, es) || !aligned_to(dy, es) || !aligned_to(dx, es)) return QK_ERR_MISALIGNED;
  const int64_t bytes = M * N * int64_t(es);
  if ((dx != y && overlap(dx, bytes, y, bytes)) || (dx != dy && overlap(dx, bytes, dy, bytes)))
    return QK_ERR_INVALID_ARG;
  const bool fast = bwd_aligned(dtype, N, {y, dy, dx});
  if (!fast && N > kMaskedBwdMaxRow) return QK_ERR_UNSUPPORTED;
  if (!fast && same_mod16(y, dy) && same_mod16(y, dx)) {  // the shifted ring kernel
    RowArgs r = {};
    r.x = y;
    r.x2 = dy;
    r.y = dx;
    r.M = M;
    r.N = N;
    st = run(kOpSoftmaxBwd, dtype, r, kPathShifted, stream);
    if (st != QK_ERR_UNSUPPORTED) return st;
  }
  BwdArgs a = {};
  a.in0 = y;
  a.in1 = dy;
  a.out = dx;
  a.M = M;
  a.N = N;
  return run_bwd(kOpSoftmaxBwd, dtype, a, nullptr, 0, fast, stream);
}

qk_status qk_rmsnorm_bwd_workspace_size(int64_t M, int64_t N, qk_dtype dtype, size_t* bytes) {
  if (bytes == nullptr) return QK_ERR_INVALID_ARG;
  *bytes = 0;
  qk_status st = check_sizes(kOpRmsNormBwd, dtype, M, N);
  if (st != QK_OK || M == 0) return st;
  // The path depends on the pointers, which are not known here: enough for
  // either path that these sizes may take.
  int dev;
  DeviceInfo* d;
  const Plan* p;
  int64_t rows = 0;
  const bool may_be_fast = (N * int64_t(elem_size(dtype))) % 16 == 0;
  if (may_be_fast) {
    st = plan_bwd_cached(kOpRmsNormBwd, dtype, M, N, true, &dev, &d, &p);
    if (st != QK_OK) return st;
    rows = dw_partial_rows(*p);
  }
  st = plan_bwd_cached(kOpRmsNormBwd, dtype, M, N, false, &dev, &d, &p);
  if (st == QK_OK) {
    rows = std::max(rows, dw_partial_rows(*p));
  } else if (!(may_be_fast && st == QK_ERR_UNSUPPORTED)) {
    return st;  // a masked row too long is only an error when the row cannot be aligned
  }
  *bytes = size_t(rows) * size_t(N) * 4;
  return QK_OK;
}

qk_status qk_rmsnorm_bwd(const void* x, const void* w, const float* rstd, const void* dy, void* dx,
                         float* dw, void* workspace, size_t workspace_bytes, int64_t M, int64_t N,
                         qk_dtype dtype, void* stream) {
  qk_status st = check_sizes(kOpRmsNormBwd, dtype, M, N);
  if (st != QK_OK) return st;
  if (M == 0) return QK_OK;
  if (x == nullptr || w == nullptr || rstd == nullptr || dy == nullptr || dx == nullptr ||
      dw == nullptr || workspace == nullptr)
    return QK_ERR_INVALID_ARG;
  const size_t es = size_t(elem_size(dtype));
  if (!aligned_to(x, es) || !aligned_to(w, es) || !aligned_to(dy, es) || !aligned_to(dx, es) ||
      !aligned_to(rstd, 4) || !aligned_to(dw, 4) || !aligned_to(workspace, 16))
    return QK_ERR_MISALIGNED;
  const int64_t bytes = M * N * int64_t(es), wb = N * int64_t(es);
  const int64_t wsb = int64_t(std::min<size_t>(workspace_bytes, size_t(INT64_MAX)));
  if ((dx != x && overlap(dx, bytes, x, bytes)) || (dx != dy && overlap(dx, bytes, dy, bytes)) ||
      overlap(dx, bytes, w, wb) || overlap(dx, bytes, rstd, M * 4) || overlap(dw, N * 4, x, bytes) ||
      overlap(dw, N * 4, dy, bytes) || overlap(dw, N * 4, dx, bytes) || overlap(dw, N * 4, w, wb) ||
      overlap(dw, N * 4, rstd, M * 4) || overlap(workspace, wsb, x, bytes) ||
      overlap(workspace, wsb, dy, bytes) || overlap(workspace, wsb, dx, bytes) ||
      overlap(workspace, wsb, dw, N * 4))
    return QK_ERR_INVALID_ARG;
  const bool fast = bwd_aligned(dtype, N, {x, w, dy, dx});
  if (!fast && N > kMaskedBwdMaxRow) return QK_ERR_UNSUPPORTED;
  BwdArgs a = {};
  a.in0 = x;
  a.in1 = dy;
  a.w = w;
  a.rstd = rstd;
  a.out = dx;
  a.dw_partial = static_cast<float*>(workspace);
  a.M = M;
  a.N = N;
  return run_bwd(kOpRmsNormBwd, dtype, a, dw, workspace_bytes, fast, stream);
}

qk_status qk_xent_bwd_ex(const void* logits, const int64_t* targets, const float* lse,
                         const float* dloss, void* dlogits, int64_t M, int64_t N, qk_dtype dtype,
                         const qk_xent_options* options, void* stream) {
  const int has_ignore = options != nullptr && options->has_ignore_index != 0;
  const int64_t ignore = has_ignore ? options->ignore_index : 0;
  const float z = options != nullptr ? options->z_loss : 0.f;
  qk_status st = check_sizes(kOpXentBwd, dtype, M, N);
  if (st != QK_OK) return st;
  if (!std::isfinite(z)) return QK_ERR_INVALID_ARG;
  if (M == 0) return QK_OK;
  if (logits == nullptr || targets == nullptr || lse == nullptr || dlogits == nullptr)
    return QK_ERR_INVALID_ARG;
  const size_t es = size_t(elem_size(dtype));
  if (!aligned_to(logits, es) || !aligned_to(dlogits, es) || !aligned_to(targets, 8) ||
      !aligned_to(lse, 4) || !aligned_to(dloss, 4))
    return QK_ERR_MISALIGNED;
  const int64_t bytes = M * N * int64_t(es);
  if ((dlogits != logits && overlap(dlogits, bytes, logits, bytes)) ||
      overlap(dlogits, bytes, targets, M * 8) || overlap(dlogits, bytes, lse, M * 4) ||
      overlap(dlogits, bytes, dloss, M * 4))
    return QK_ERR_INVALID_ARG;
  const bool fast = bwd_aligned(dtype, N, {logits, dlogits});
  if (!fast && same_mod16(logits, dlogits)) {  // the shifted ring kernel, as in the forward pass
    RowArgs r = {};
    r.x = logits;
    r.y = dlogits;
    r.lse = const_cast<float*>(lse);  // read only
    r.dloss = dloss;
    r.target = targets;
    r.M = M;
    r.N = N;
    r.ignore_index = ignore;
    r.has_ignore = has_ignore;
    r.z_loss = z;
    st = run(kOpXentBwd, dtype, r, kPathShifted, stream);
    if (st != QK_ERR_UNSUPPORTED) return st;
  }
  BwdArgs a = {};
  a.in0 = logits;
  a.target = targets;
  a.lse = lse;
  a.dloss = dloss;
  a.out = dlogits;
  a.M = M;
  a.N = N;
  a.ignore_index = ignore;
  a.has_ignore = has_ignore;
  a.z_loss = z;
  return run_bwd(kOpXentBwd, dtype, a, nullptr, 0, fast, stream);
}

qk_status qk_xent_bwd(const void* logits, const int64_t* targets, const float* lse,
                      const float* dloss, void* dlogits, int64_t M, int64_t N, qk_dtype dtype,
                      void* stream) {
  return qk_xent_bwd_ex(logits, targets, lse, dloss, dlogits, M, N, dtype, nullptr, stream);
}

qk_status qk_get_device_status(void* stream) {
  int dev;
  DeviceInfo* d;
  qk_status st = device_info(&dev, &d);
  if (st != QK_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return QK_ERR_LAUNCH;
  }
  int v = 0;
  if (cudaMemcpy(&v, d->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return QK_ERR_LAUNCH;
  }
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(d->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) {
      cudaGetLastError();
      return QK_ERR_LAUNCH;
    }
  }
  return static_cast<qk_status>(v);
}

qk_status qk_get_plan(qk_op op, qk_dtype dtype, int64_t M, int64_t N, qk_plan* plan) {
  if (plan == nullptr || op < 0 || op >= kNumOps) return QK_ERR_INVALID_ARG;
  qk_status st = check_sizes(op, dtype, M, N);
  if (st != QK_OK) return st;
  int dev;
  DeviceInfo* d;
  st = device_info(&dev, &d);
  if (st != QK_OK) return st;
  const bool fast = (N * int64_t(elem_size(dtype))) % 16 == 0;
  const int64_t m = std::max<int64_t>(M, 1);
  Plan p;
  if (fast) {
    st = plan_ring(dev, *d, op, dtype, m, N, &p);
  } else if (is_bwd(op)) {  // softmax, x-entropy: the shifted kernel when it fits, else the masked one
    st = (op == kOpXentBwd || op == kOpSoftmaxBwd) ? plan_shifted(dev, *d, op, dtype, m, N, &p)
                                                   : QK_ERR_UNSUPPORTED;
    if (st == QK_ERR_UNSUPPORTED) st = plan_direct_bwd(dev, *d, op, dtype, m, N, &p);
  } else {  // x and y 16-byte aligned, N not: the shifted ring, else the masked kernel
    st = plan_shifted(dev, *d, op, dtype, m, N, &p);
    if (st == QK_ERR_UNSUPPORTED) st = plan_direct(dev, *d, op, dtype, m, N, &p);
  }
  if (st != QK_OK) return st;
  plan->path = p.kernel->path;
  plan->threads = p.kernel->threads;
  plan->row_threads = p.kernel->row_threads;
  plan->vec_per_thread = p.kernel->vec_per_thread;
  plan->cluster = p.cluster;
  plan->slots = p.slots;
  plan->chunks = p.chunks;
  plan->ctas_per_sm = p.ctas_per_sm;
  plan->grid = int32_t(std::min<int64_t>(p.grid, INT32_MAX));
  plan->smem_bytes = p.smem;
  return QK_OK;
}

qk_status qk_set_plan_override(qk_op op, qk_dtype dtype, const qk_plan* plan) {
  if (op < 0 || op >= kNumOps || (dtype != QK_F32 && dtype != QK_BF16)) return QK_ERR_INVALID_ARG;
  if (plan == nullptr) {
    g_override[op][dtype].on = false;
    g_override_gen.fetch_add(1, std::memory_order_acq_rel);
    return QK_OK;
  }
  if (plan->cluster < 0 || plan->cluster > kMaxCluster || plan->slots < 0 ||
      plan->slots > kMaxSlots)
    return QK_ERR_INVALID_ARG;
  const bool clustered = plan->cluster > 1;
  if (find_kernel(op, dtype, is_bwd(op) ? 3 : 1, plan->threads, plan->row_threads,
                  plan->vec_per_thread, clustered) == nullptr)
    return QK_ERR_UNSUPPORTED;
  g_override[op][dtype].plan = *plan;
  g_override[op][dtype].on = true;
  g_override_gen.fetch_add(1, std::memory_order_acq_rel);
  return QK_OK;
}

qk_status qk_test_wait_timeout(uint64_t timeout_ns, void* stream) {
  if (timeout_ns == 0 || timeout_ns > 10000000000ull) return QK_ERR_INVALID_ARG;
  int dev;
  DeviceInfo* d;
  qk_status st = device_info(&dev, &d);
  if (st != QK_OK) return st;
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(timeout_ns, d->status);
  if (cudaGetLastError() != cudaSuccess) return QK_ERR_LAUNCH;
  return QK_OK;
}

}  // extern "C"
