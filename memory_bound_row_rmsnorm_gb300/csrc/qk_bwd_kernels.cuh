// qk_bwd_kernels.cuh -- backward passes of the three row operators, sm_103a.
//
// Same structure as the forward ring kernel (qk_kernels.cuh): a persistent
// grid, one thread streaming whole work items into a shared-memory ring with
// cp.async.bulk under mbarriers, rows reduced from registers through warp,
// block and (for long rows) cluster DSMEM, every output stored once.  A ring
// slot holds one item of each input matrix:
//   softmax  dx = y * (dy - sum_k dy_k y_k)                  inputs y, dy
//   RMSNorm  dx = r dy w - x r^3 (1/N) sum_k dy_k w_k x_k     inputs x, dy (+ rstd, w)
//            dw_j = sum_i dy_ij x_ij r_i                        column sums over all rows
//   x-ent    dx = dloss * (exp(x - lse) - onehot(t))           input logits (+ lse, t, dloss)
// Cross-entropy needs no reduction over the row, so long rows are streamed in
// chunks.  RMSNorm's dw: each thread accumulates fp32 partials for the fixed
// columns it owns; at the end the row groups of a CTA are summed in shared
// memory and the CTA writes one partial row to the caller's workspace, which
// dw_reduce_kernel sums over CTAs in a fixed order (deterministic).
#pragma once

#include "qk_device.cuh"
#include "qk_internal.h"
#include "qk_kernels.cuh"  // warp_reduce, merge_partials

namespace qk {

enum BwdOp : int { kSoftmaxBwd = 10, kRmsNormBwd = 11, kXentBwd = 12 };

struct BwdArgs {
  const void* in0;      // [M, N] y (softmax), x (RMSNorm), logits (x-entropy)
  const void* in1;      // [M, N] dy (softmax, RMSNorm); unused for x-entropy
  const void* w;        // [N] RMSNorm weight
  const float* rstd;    // [M] RMSNorm forward rstd
  const float* lse;     // [M] x-entropy forward log-sum-exp
  const float* dloss;   // [M] x-entropy upstream gradient (null: 1 for every row)
  const int64_t* target;  // [M] x-entropy targets
  void* out;            // [M, N] dx / dlogits
  float* dw_partial;    // RMSNorm: [partial_rows, N] fp32 workspace
  int64_t M;
  int64_t N;
  float inv_n;          // 1 / N
  float z_loss;         // x-entropy: z-loss coefficient (gradient factor 1 + 2 z lse)
  int64_t ignore_index; // x-entropy: rows with this target get zero gradient (when has_ignore)
  int32_t has_ignore;   // x-entropy: nonzero when ignore_index is in use
  int32_t chunks;       // ring steps per row (streamed x-entropy rows), else 1
  int32_t slots;        // ring slots per CTA
  uint32_t slot_bytes;  // bytes of ONE input's item in a slot (multiple of 128)
  int64_t num_items;
  uint64_t timeout_ns;
  int* status;
};

// Residency requests for the launch bounds (0: none): cross-entropy's
// 8-vector plans hold three CTAs per SM.
template <int OP, int THREADS, int VPT>
constexpr int bwd_min_blocks() {
  return (OP == kXentBwd && THREADS == 256 && VPT == 8) ? 3 : 0;
}

template <int OP, typename T, int THREADS, int TPR, int VPT, bool CLUSTER>
__global__ void __launch_bounds__(THREADS, (bwd_min_blocks<OP, THREADS, VPT>())) bwd_kernel(const BwdArgs a) {
  using V = Vec16<T>;
  constexpr int E = V::kElems;
  constexpr int NIN = (OP == kXentBwd) ? 1 : 2;  // input matrices per item
  constexpr int NW = THREADS / 32;
  constexpr int WPG = TPR / 32;
  constexpr int GW = TPR < 32 ? TPR : 32;
  constexpr int R = THREADS / TPR;
  constexpr int64_t CH = int64_t(TPR) * VPT;
  static_assert((TPR % 32 == 0 || 32 % TPR == 0) && THREADS % TPR == 0 && TPR >= 4, "row groups");
  static_assert(!CLUSTER || TPR == THREADS, "a clustered row spans the whole CTA");
  static_assert(NW <= 16, "block-reduction buffer holds 16 warps");
  static_assert(!(CLUSTER && OP == kXentBwd), "x-entropy rows are streamed, not split");

  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* xbar = reinterpret_cast<uint64_t*>(smem + 8 * kMaxSlots);
  float2* red = reinterpret_cast<float2*>(smem + 512);
  float2* xbuf = reinterpret_cast<float2*>(smem + 768);
  unsigned char* ring = smem + kSmemHeader;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = tid / TPR, l = tid % TPR;
  const int64_t M = a.M, N = a.N, NV = N / E;
  const int S = a.slots;
  const int64_t K = a.chunks;
  const uint32_t item_stride = uint32_t(NIN) * a.slot_bytes;  // bytes of one ring slot

  uint32_t C = 1, rank = 0, cid = blockIdx.x, ncl = gridDim.x;
  if constexpr (CLUSTER) {
    C = cluster_nctarank();
    rank = cluster_ctarank();
    cid = cluster_id_x();
    ncl = num_clusters_x();
  }
  const int64_t SV = (NV + C - 1) / C;
  const int64_t v0 = min(NV, int64_t(rank) * SV);
  const int64_t nv = min(NV, v0 + SV) - v0;
  const int64_t n_local = a.num_items > int64_t(cid) ? (a.num_items - 1 - cid) / ncl + 1 : 0;
  const int64_t q_total = n_local * K;
  const uint32_t full0 = smem_addr(full), xbar0 = smem_addr(xbar), ring0 = smem_addr(ring);

  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(full0 + 8 * s, 1);
    mbar_init(xbar0, 1);
    mbar_init(xbar0 + 8, 1);
    fence_mbar_init();
  }
  if constexpr (CLUSTER) {
    cluster_sync_all();
  } else {
    __syncthreads();
  }
  // The first item of every input into L2 while the previous kernel in the
  // stream finishes (a hint; the copies into shared memory follow the wait).
  if (!CLUSTER && tid == 0 && q_total > 0) {
    int64_t off, bytes;
    if (K > 1) {
      off = int64_t(cid) * NV * 16;
      bytes = min(int64_t(S) * CH, NV) * 16;
    } else {
      const int64_t r0 = int64_t(cid) * R;
      off = r0 * NV * 16;
      bytes = min(int64_t(R), M - r0) * NV * 16;
    }
    const void* in[2] = {a.in0, a.in1};
#pragma unroll
    for (int i = 0; i < NIN; ++i)
      for (int64_t o = 0; o < bytes; o += 32768)
        bulk_prefetch_l2(static_cast<const unsigned char*>(in[i]) + off + o,
                         uint32_t(min(int64_t(32768), bytes - o)));
  }
  grid_dependency_wait();
  allow_dependent_launch();

  // ---- producer (thread 0): one item of every input per ring slot ----
  uint64_t policy = 0;
  int64_t p_item = cid, p_left = q_total;
  int p_chunk = 0, p_slot = 0;
  const unsigned char* src[2] = {static_cast<const unsigned char*>(a.in0),
                                 static_cast<const unsigned char*>(a.in1)};
  auto issue_next = [&]() {
    int64_t off, bytes;
    if (K > 1) {
      const int64_t c0 = int64_t(p_chunk) * CH;
      off = (p_item * NV + c0) * 16;
      bytes = min(CH, NV - c0) * 16;
    } else if (CLUSTER) {
      off = (p_item * NV + v0) * 16;
      bytes = nv * 16;
    } else {
      const int64_t r0 = p_item * R;
      off = r0 * NV * 16;
      bytes = min(int64_t(R), M - r0) * NV * 16;
    }
    const uint32_t bar = full0 + 8u * uint32_t(p_slot);
    const uint32_t dst = ring0 + uint32_t(p_slot) * item_stride;
    mbar_arrive_expect_tx(bar, uint32_t(bytes) * NIN);
#pragma unroll
    for (int in = 0; in < NIN; ++in)
      for (int64_t o = 0; o < bytes; o += 32768)
        bulk_copy_g2s(dst + uint32_t(in) * a.slot_bytes + uint32_t(o), src[in] + off + o,
                      uint32_t(min(int64_t(32768), bytes - o)), bar, policy);
    if (++p_slot == S) p_slot = 0;
    if (++p_chunk == K) {
      p_chunk = 0;
      p_item += ncl;
    }
    --p_left;
  };
  if (tid == 0) {
    policy = l2_evict_first_policy();
    for (int s = 0; s < S && p_left > 0; ++s) issue_next();
  }

  // RMSNorm: weight in registers (its columns never change), fp32 dw partials.
  constexpr bool kWeightInRegs = VPT <= 8;
  const uint4* wg = static_cast<const uint4*>(a.w) + v0;
  uint4 wv[(OP == kRmsNormBwd && kWeightInRegs) ? VPT : 1];
  float dwacc[OP == kRmsNormBwd ? VPT * E : 1];
  if constexpr (OP == kRmsNormBwd) {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int64_t lv = l + int64_t(k) * TPR;
      if constexpr (kWeightInRegs) wv[k] = lv < nv ? __ldg(wg + lv) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int e = 0; e < VPT * E; ++e) dwacc[e] = 0.f;
  }

  // Per-row scalars of the next item, loaded one item ahead.
  auto row_of = [&](int64_t it) -> int64_t { return (K > 1 || CLUSTER) ? it : it * R + g; };
  float s_next = 0.f, g_next = 1.f;  // rstd or lse; upstream gradient
  int64_t t_next = -1;
  auto prefetch = [&](int64_t it) {
    const int64_t rw = row_of(it);
    if (it < a.num_items && rw < M) {
      if constexpr (OP == kRmsNormBwd) s_next = __ldg(a.rstd + rw);
      if constexpr (OP == kXentBwd) {
        s_next = __ldg(a.lse + rw);
        g_next = a.dloss != nullptr ? __ldg(a.dloss + rw) : 1.f;
        t_next = __ldg(a.target + rw);
      }
    }
  };
  if constexpr (OP != kSoftmaxBwd) prefetch(cid);

  uint4 xa[VPT], xb[NIN == 2 ? VPT : 1];  // raw vectors of input 0 and input 1
  float rs = 0.f, gs = 1.f;               // current row's rstd / lse, upstream gradient
  int64_t trow = -1;
  bool failed = false, abort = false;
  int64_t q = 0, item = cid;
  int j = 0, slot = 0;
  uint32_t phase = 0, ibit = 0, xphase = 0;

  for (; q < q_total; ++q) {
    if (!mbar_wait<false>(full0 + 8u * uint32_t(slot), phase, a.timeout_ns)) {
      report_status(a.status, 5);
      failed = true;
    }
    const bool single = (K > 1) || CLUSTER;
    const int64_t row = row_of(item);
    const bool row_ok = row < M;
    const int cn = int((K > 1) ? min(CH, NV - int64_t(j) * CH) : nv);
    const int64_t cbase = (K > 1) ? int64_t(j) * CH : v0;
    const unsigned char* sb = ring + size_t(slot) * item_stride +
                              (single ? size_t(0) : size_t(g) * size_t(NV) * 16);
    if (j == 0 && OP != kSoftmaxBwd) {
      rs = s_next, gs = g_next, trow = t_next;
      prefetch(item + ncl);
    }
    // Cross-entropy: the thread holding x[target] in this slot reads it once
    // here (the slot is refilled after the barrier below) and rewrites that
    // one output element after its vector store.
    int64_t tl = -1;       // target vector, relative to the slot
    bool own_t = false;
    float xt = 0.f;
    if constexpr (OP == kXentBwd) {
      if (row_ok && !failed && trow >= 0 && trow < N) {
        tl = trow / E - cbase;
        own_t = tl >= 0 && tl < cn && int(tl) % TPR == l;
        if (own_t) xt = V::load1(sb + tl * 16 + (trow % E) * int64_t(sizeof(T)));
      }
    }
    bool valid[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int lv = l + k * TPR;
      valid[k] = row_ok && lv < cn && !failed;
      xa[k] = valid[k] ? *reinterpret_cast<const uint4*>(sb + lv * 16) : make_uint4(0u, 0u, 0u, 0u);
      if constexpr (NIN == 2)
        xb[k] = valid[k] ? *reinterpret_cast<const uint4*>(sb + a.slot_bytes + lv * 16)
                         : make_uint4(0u, 0u, 0u, 0u);
    }

    // ---- thread-level dot product (padding vectors are zero) ----
    float ps = 0.f;
    if constexpr (OP != kXentBwd) {
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        float fa[E], fb[E];
        V::unpack(xa[k], fa);
        V::unpack(xb[k], fb);
        if constexpr (OP == kSoftmaxBwd) {  // sum dy * y
#pragma unroll
          for (int e = 0; e < E; e += 2)
            acc = fma2(make_float2(fa[e], fa[e + 1]), make_float2(fb[e], fb[e + 1]), acc);
        } else {  // sum dy * w * x
          float fw[E];
          if constexpr (kWeightInRegs) {
            V::unpack_fresh(wv[k], fw);  // not hoisted: keep w packed across the loop
          } else {
            V::unpack(valid[k] ? __ldg(wg + l + k * TPR) : make_uint4(0u, 0u, 0u, 0u), fw);
          }
#pragma unroll
          for (int e = 0; e < E; e += 2)
            acc = fma2(mul2(make_float2(fb[e], fb[e + 1]), make_float2(fw[e], fw[e + 1])),
                       make_float2(fa[e], fa[e + 1]), acc);
        }
      }
      ps = acc.x + acc.y;
      warp_reduce<kRmsNorm, GW>(ps, ps);  // a plain sum over the row group's lanes
      if (WPG > 1 && lane == 0) red[ibit * 16 + warp] = make_float2(0.f, ps);
    }
    if (__syncthreads_or(failed)) {
      abort = true;
      break;
    }
    if (tid == 0 && p_left > 0) issue_next();
    const uint32_t row_ibit = ibit, row_xphase = xphase;
    if (++slot == S) {
      slot = 0;
      phase ^= 1u;
    }
    const bool row_end = (j == K - 1);
    if (row_end) {
      j = 0;
      item += ncl;
      xphase ^= ibit;
      ibit ^= 1u;
    } else {
      ++j;
    }

    float dot = 0.f;
    if constexpr (OP != kXentBwd) {
      float unused = 0.f;
      dot = ps;
      if constexpr (WPG > 1) merge_partials<kRmsNorm>(red + row_ibit * 16 + g * WPG, WPG, unused, dot);
      if constexpr (CLUSTER) {
        const uint32_t xb_ = xbar0 + 8u * row_ibit;
        if (tid == 0) {
          mbar_arrive_expect_tx(xb_, C * 8u);
          const uint32_t mine = smem_addr(xbuf + row_ibit * kMaxCluster + rank);
          for (uint32_t r = 0; r < C; ++r)
            st_async_f2(map_to_rank(mine, r), 0.f, dot, map_to_rank(xb_, r));
        }
        if (!mbar_wait<true>(xb_, row_xphase, a.timeout_ns)) {
          report_status(a.status, 5);
          failed = true;
        }
        merge_partials<kRmsNorm>(xbuf + row_ibit * kMaxCluster, int(C), unused, dot);
      }
    }
    if (!row_ok) continue;

    // ---- finish: every output vector once ----
    uint4* og = static_cast<uint4*>(a.out) + row * NV + cbase;
    if constexpr (OP == kSoftmaxBwd) {
      const float2 nd = make_float2(-dot, -dot);
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        if (!valid[k]) continue;
        float fa[E], fb[E], o[E];
        V::unpack_fresh(xa[k], fa);
        V::unpack_fresh(xb[k], fb);
#pragma unroll
        for (int e = 0; e < E; e += 2) {  // y * (dy - dot)
          const float2 v = mul2(make_float2(fa[e], fa[e + 1]), add2(make_float2(fb[e], fb[e + 1]), nd));
          o[e] = v.x;
          o[e + 1] = v.y;
        }
        __stcs(og + l + k * TPR, V::pack(o));
      }
    } else if constexpr (OP == kRmsNormBwd) {
      const float c = rs * rs * rs * dot * a.inv_n;
      const float2 r2 = make_float2(rs, rs), nc = make_float2(-c, -c);
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        if (!valid[k]) continue;
        float fx[E], fd[E], fw[E], o[E];
        V::unpack_fresh(xa[k], fx);
        V::unpack_fresh(xb[k], fd);
        if constexpr (kWeightInRegs) {
          V::unpack_fresh(wv[k], fw);
        } else {
          V::unpack(__ldg(wg + l + k * TPR), fw);
        }
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          const float2 x2 = make_float2(fx[e], fx[e + 1]), d2 = make_float2(fd[e], fd[e + 1]);
          // dx = (r * dy) * w - x * c
          const float2 v = fma2(x2, nc, mul2(mul2(r2, d2), make_float2(fw[e], fw[e + 1])));
          o[e] = v.x;
          o[e + 1] = v.y;
          // dw partial: (dy * x) * r
          const float2 pw = mul2(mul2(d2, x2), r2);
          dwacc[k * E + e] += pw.x;
          dwacc[k * E + e + 1] += pw.y;
        }
        __stcs(og + l + k * TPR, V::pack(o));
      }
    } else {  // cross-entropy: dloss * (exp(x - lse) - onehot)
      const bool ignored = a.has_ignore && trow == a.ignore_index;
      const bool tok = trow >= 0 && trow < N;
      // zero row if ignored, NaN row for a bad target; the z-loss term scales
      // the softmax part by 1 + 2 z lse
      const float gv = ignored ? 0.f : (tok ? gs : __int_as_float(0x7fc00000));
      const float zf = fmaf(2.f * a.z_loss, rs, 1.f);
      const float lb = rs * kLog2e;
      const float2 zf2 = make_float2(zf, zf), gv2 = make_float2(gv, gv);
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        if (!valid[k]) continue;
        float f[E], o[E];
        V::unpack_fresh(xa[k], f);
#pragma unroll
        for (int e = 0; e < E; e += 2) {  // (exp(x - lse) (1 + 2 z lse)) dloss
          const float2 t = fma2(make_float2(f[e], f[e + 1]), make_float2(kLog2e, kLog2e),
                                make_float2(-lb, -lb));
          const float2 v =
              mul2(mul2(make_float2(exp2_approx(t.x), exp2_approx(t.y)), zf2), gv2);
          o[e] = v.x;
          o[e + 1] = v.y;
        }
        // A plain store: the target element below rewrites part of one of
        // these vectors, and a streaming store (which the softmax and RMSNorm
        // gradients use) measured 1-3 points slower here for bf16.
        og[l + k * TPR] = V::pack(o);
      }
      if (own_t) {  // the target element: the same terms, minus the one-hot 1
        const float p = exp2_approx(fmaf(xt, kLog2e, -lb)) * zf - 1.f;
        V::store1(reinterpret_cast<T*>(og + tl) + (trow % E), p * gv);
      }
    }
  }

  if (abort) {
    if (tid == 0) {
      const int64_t outstanding = (q_total - q) - p_left;
      for (int64_t n = 0; n < outstanding; ++n) {
        mbar_wait<false>(full0 + 8u * uint32_t(slot), phase, a.timeout_ns);
        if (++slot == S) {
          slot = 0;
          phase ^= 1u;
        }
      }
    }
    __syncthreads();
  }

  // ---- RMSNorm dw: sum the row groups of this CTA, write one partial row ----
  if constexpr (OP == kRmsNormBwd && R == 1 && E == 8) {
    // One row group: each thread's partials are already the CTA's for its
    // columns, E consecutive floats per vector, stored as 16-byte vectors
    // (the row's byte offset N * 4 and the slice's v0 * E * 4 are multiples
    // of 16 on this path).  bf16 only: against the staged sum below it
    // measured +1 point for bf16 and -2 for fp32 rows of 4096 (the fp32 kernel
    // took 10 more registers), on the same GPU.
    float4* dst = reinterpret_cast<float4*>(a.dw_partial + int64_t(cid) * N + v0 * E);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int64_t lv = l + int64_t(k) * TPR;
      if (lv < nv) {
#pragma unroll
        for (int q = 0; q < E / 4; ++q)
          dst[lv * (E / 4) + q] = make_float4(dwacc[k * E + 4 * q], dwacc[k * E + 4 * q + 1],
                                              dwacc[k * E + 4 * q + 2], dwacc[k * E + 4 * q + 3]);
      }
    }
  } else if constexpr (OP == kRmsNormBwd) {
    // The ring is idle now (every load was consumed or drained): reuse it.
    float* sd = reinterpret_cast<float*>(ring);
    const int64_t prow = int64_t(cid);  // one partial row per CTA (clusters: per cluster, own slice)
    for (int gg = 0; gg < R; ++gg) {
      if (g == gg) {
#pragma unroll
        for (int k = 0; k < VPT; ++k)
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const int col = (l + k * TPR) * E + e;  // column inside this CTA's slice
            if (col < nv * E) sd[col] = (gg == 0 ? 0.f : sd[col]) + dwacc[k * E + e];
          }
      }
      __syncthreads();
    }
    float* dst = a.dw_partial + prow * N + v0 * E;
    for (int64_t col = tid; col < nv * E; col += THREADS) dst[col] = sd[col];
  }
  if constexpr (CLUSTER) cluster_sync_all();
}

// ---------------------------------------------------------------------------
// Masked backward path: rows whose start or length is not a multiple of 16
// bytes.  A persistent grid of CTAs (or of clusters, for long rows) walks the
// rows; each thread holds EPT elements of each input of its slice in
// registers (element loads), the row's dot product goes through the warp,
// block and cluster levels as in bwd_kernel, and every output element is
// stored once.  RMSNorm's dw partials stay in registers for the columns a
// thread owns and are written as one partial row per CTA (or per cluster,
// its own slice).  Cross-entropy has no row reduction: any N is streamed in
// chunks of THREADS * EPT elements.
// ---------------------------------------------------------------------------
template <int OP, typename T, int THREADS, int EPT, bool CLUSTER>
__global__ void __launch_bounds__(THREADS) bwd_direct_kernel(const BwdArgs a) {
  using V = Vec16<T>;
  constexpr int NW = THREADS / 32;
  constexpr int64_t CH = int64_t(THREADS) * EPT;
  static_assert(!(CLUSTER && OP == kXentBwd), "x-entropy rows are streamed, not split");
  __shared__ float red[2][NW];
  __shared__ float2 xbuf[2][kMaxCluster];
  __shared__ __align__(8) uint64_t xbar[2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t C = 1, rank = 0;
  int64_t cid = blockIdx.x, ncl = gridDim.x;
  if constexpr (CLUSTER) {
    C = cluster_nctarank();
    rank = cluster_ctarank();
    cid = cluster_id_x();
    ncl = num_clusters_x();
  }
  const int64_t M = a.M, N = a.N;
  const int64_t SE = (N + C - 1) / C;
  const int64_t e0 = min(N, int64_t(rank) * SE);
  const int64_t ne = min(N, e0 + SE) - e0;
  const uint32_t xb0 = smem_addr(&xbar[0]);
  if constexpr (CLUSTER) {
    if (tid == 0) {
      mbar_init(xb0, 1);
      mbar_init(xb0 + 8, 1);
      fence_mbar_init();
    }
    cluster_sync_all();  // peers' barriers exist before anyone stores into them
  }
  grid_dependency_wait();
  allow_dependent_launch();

  const T* in0 = static_cast<const T*>(a.in0);
  const T* in1 = static_cast<const T*>(a.in1);
  T* out = static_cast<T*>(a.out);

  if constexpr (OP == kXentBwd) {  // dloss * ((1 + 2 z lse) exp(x - lse) - onehot(t))
    for (int64_t row = cid; row < M; row += ncl) {
      const float lse = __ldg(a.lse + row);
      const float gr = a.dloss != nullptr ? __ldg(a.dloss + row) : 1.f;
      const int64_t t = __ldg(a.target + row);
      const bool ignored = a.has_ignore && t == a.ignore_index, tok = t >= 0 && t < N;
      const float gv = ignored ? 0.f : (tok ? gr : __int_as_float(0x7fc00000));
      const float zf = fmaf(2.f * a.z_loss, lse, 1.f);
      const float lb = lse * kLog2e;
      const T* xr = in0 + row * N;
      T* orow = out + row * N;
      for (int64_t c0 = 0; c0 < N; c0 += CH) {
        float f[EPT];
#pragma unroll
        for (int k = 0; k < EPT; ++k) {  // all loads first, then the math and stores
          const int64_t e = c0 + tid + int64_t(k) * THREADS;
          f[k] = e < N ? V::load1(xr + e) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < EPT; ++k) {
          const int64_t e = c0 + tid + int64_t(k) * THREADS;
          if (e >= N) continue;
          float p = exp2_approx(fmaf(f[k], kLog2e, -lb)) * zf;
          if (e == t) p -= 1.f;
          V::store1(orow + e, p * gv);
        }
      }
    }
    return;
  } else {
    // RMSNorm: the weight of the columns this thread owns, and their dw partials.
    float wf[OP == kRmsNormBwd ? EPT : 1];
    float dwacc[OP == kRmsNormBwd ? EPT : 1];
    if constexpr (OP == kRmsNormBwd) {
      const T* wr = static_cast<const T*>(a.w) + e0;
#pragma unroll
      for (int k = 0; k < EPT; ++k) {
        const int64_t e = tid + int64_t(k) * THREADS;
        wf[k] = e < ne ? V::load1(wr + e) : 0.f;
        dwacc[k] = 0.f;
      }
    }
    uint32_t ib = 0, xph = 0;  // row parity: buffers; phase of the cluster barrier
    bool failed = false;
    for (int64_t row = cid; row < M; row += ncl) {
      const T* ra = in0 + row * N + e0;  // y (softmax) or x (RMSNorm)
      const T* rb = in1 + row * N + e0;  // dy
      float fa[EPT], fb[EPT];
#pragma unroll
      for (int k = 0; k < EPT; ++k) {
        const int64_t e = tid + int64_t(k) * THREADS;
        fa[k] = e < ne ? V::load1(ra + e) : 0.f;
        fb[k] = e < ne ? V::load1(rb + e) : 0.f;
      }
      const float rs = (OP == kRmsNormBwd) ? __ldg(a.rstd + row) : 0.f;
      float ps = 0.f;  // sum dy * y, or sum dy * w * x (padding is zero)
#pragma unroll
      for (int k = 0; k < EPT; ++k)
        ps = (OP == kSoftmaxBwd) ? fmaf(fb[k], fa[k], ps) : fmaf(fb[k] * wf[k], fa[k], ps);
      ps = group_sum<32>(ps);
      if (lane == 0) red[ib][warp] = ps;
      __syncthreads();
      float dot = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) dot += red[ib][w];  // index order
      if constexpr (CLUSTER) {
        const uint32_t xb = xb0 + 8u * ib;
        if (tid == 0) {
          mbar_arrive_expect_tx(xb, C * 8u);
          const uint32_t mine = smem_addr(&xbuf[ib][rank]);
          for (uint32_t r = 0; r < C; ++r) st_async_f2(map_to_rank(mine, r), 0.f, dot, map_to_rank(xb, r));
        }
        if (!mbar_wait<true>(xb, xph, a.timeout_ns)) {
          report_status(a.status, 5);
          failed = true;
        }
        if (__syncthreads_or(failed)) break;  // leave together; peers time out the same way
        dot = 0.f;
        for (uint32_t r = 0; r < C; ++r) dot += xbuf[ib][r].y;  // rank order
        xph ^= ib;  // buffer b's barrier completes every second row
      }
      ib ^= 1u;
      T* orow = out + row * N + e0;
      if constexpr (OP == kSoftmaxBwd) {  // y * (dy - dot)
#pragma unroll
        for (int k = 0; k < EPT; ++k) {
          const int64_t e = tid + int64_t(k) * THREADS;
          if (e < ne) V::store1(orow + e, fa[k] * (fb[k] - dot));
        }
      } else {  // (r dy) w - x (r^3 dot / N); dw partial (dy x) r
        const float c = rs * rs * rs * dot * a.inv_n;
#pragma unroll
        for (int k = 0; k < EPT; ++k) {
          const int64_t e = tid + int64_t(k) * THREADS;
          if (e >= ne) continue;
          V::store1(orow + e, fmaf(fa[k], -c, (rs * fb[k]) * wf[k]));
          dwacc[k] += (fb[k] * fa[k]) * rs;
        }
      }
    }
    if constexpr (OP == kRmsNormBwd) {  // one partial row per CTA (per cluster: this slice)
      float* dst = a.dw_partial + cid * N + e0;
#pragma unroll
      for (int k = 0; k < EPT; ++k) {
        const int64_t e = tid + int64_t(k) * THREADS;
        if (e < ne) dst[e] = dwacc[k];
      }
    }
    if constexpr (CLUSTER) cluster_sync_all();  // no CTA leaves while peers may write to it
  }
}

// dw[j] = sum over the partial rows p of partial[p][j], in a fixed order:
// 32 columns per CTA (one per lane, a 128-byte line per warp and row), 32
// warps each summing every 32nd row in row order, then the 32 warp sums in
// index order.  The partial rows were just written by the ring kernel and sit
// in L2; what bounds this kernel is how many of those lines are in flight, so
// each warp issues the loads of up to 16 of its rows before it adds them (a
// few hundred partial rows: every load of a warp in one round trip).  The sum
// keeps the plain row order: the same bits as a one-row-at-a-time loop.
// (A template so that every translation unit may include this header.)
constexpr int kDwReduceThreads = 1024;
template <int kUnused = 0>
__global__ void __launch_bounds__(kDwReduceThreads) dw_reduce_kernel(const float* __restrict__ partial,
                                                                     float* __restrict__ dw, int64_t rows,
                                                                     int64_t N) {
  constexpr int NW = kDwReduceThreads / 32;
  __shared__ float part[NW][33];
  grid_dependency_wait();
  allow_dependent_launch();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t col = int64_t(blockIdx.x) * 32 + lane;
  float acc = 0.f;
  if (col < N) {
    constexpr int kDepth = 16;  // rows of one warp whose loads are in flight together
    const float* p = partial + col;
    for (int64_t base = warp; base < rows; base += int64_t(kDepth) * NW) {
      float v[kDepth];
#pragma unroll
      for (int u = 0; u < kDepth; ++u) {
        const int64_t r = base + int64_t(u) * NW;
        v[u] = r < rows ? __ldcg(p + r * N) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kDepth; ++u)
        if (base + int64_t(u) * NW < rows) acc += v[u];
    }
  }
  part[warp][lane] = acc;
  __syncthreads();
  if (warp == 0 && col < N) {
    float s = part[0][lane];
#pragma unroll
    for (int w = 1; w < NW; ++w) s += part[w][lane];
    dw[col] = s;
  }
}

}  // namespace qk
