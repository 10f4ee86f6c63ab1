// qk_shifted_kernels.cuh -- the forward ring kernel for rows that do not start
// on a 16-byte boundary (N * sizeof(T) not a multiple of 16, or x offset by
// some elements), sm_103a.
//
// shifted_kernel keeps the structure of row_kernel (qk_kernels.cuh): a
// persistent grid, one thread streaming work items into a shared-memory ring
// with cp.async.bulk under mbarriers, reductions through warp, block and
// cluster (DSMEM) levels, every output stored once.  What differs:
//   * A work item is a range [L, H) of the flattened M x N matrix: R whole
//     rows, one CTA's slice of a row, or one chunk of a streamed row.  The
//     bulk copy moves the 16-byte aligned range that contains it, so the
//     slot's element 0 is flat element F0 <= L.  The extra bytes at the two
//     ends belong to neighbouring rows (or lie before x / after its end, but
//     inside the same aligned 16-byte block as a byte of x, hence inside the
//     same page); they are read, never used.
//   * Each row group works on the slot vectors that overlap its row's window
//     of elements.  The first and last of them are partial: their outside
//     elements are replaced by the reduction's neutral element when read, and
//     they are stored element by element.  Whole vectors are stored with one
//     16-byte store, which needs y to have x's alignment modulo 16 (the host
//     checks this before choosing the kernel).
//   * RMSNorm / LayerNorm parameters: the columns a thread meets change from
//     row to row, so each CTA stages its slice of w (and b) in shared memory
//     once and the finish reads them element by element.
//   * LayerNorm rows held by one CTA take two passes over the registers: the
//     row sum, then the squared deviations from the row mean, each a plain sum
//     through the warp and block levels (a second barrier).  Rows split over a
//     cluster merge (count, mean, M2) partials instead, their counts carried
//     through the block level in a second small buffer.
// Cited: QbitAI article on QuACK, section "硬件感知的加载与存储策略" (asynchronous
// GMEM->SMEM staging of the row, vectorised SMEM->register loads) and section
// "硬件感知的归约策略" (thread, warp, block and cluster reduction).
#pragma once

#include "qk_device.cuh"
#include "qk_internal.h"
#include "qk_kernels.cuh"  // warp_reduce, merge_partials, kCopyBytes, kStatusTimeout

namespace qk {

// Resident CTAs per SM asked of the register allocator (256-thread CTAs):
// left alone it gave some configurations 110-118 registers and others 74-80
// for the same code, i.e. two CTAs per SM instead of three.  These requests
// compile without spilling: 4 (5 vectors a thread) and 3 (8-9 vectors), and
// 3 and 2 for LayerNorm (counts and a bias) and softmax backward (two inputs).
template <int OP, int VPT>
constexpr int shifted_min_blocks() {
  return (OP == kLayerNorm || OP == kSoftmaxGrad) ? (VPT >= 8 ? 2 : 3) : (VPT >= 8 ? 3 : 4);
}

// bf16 elements sh .. sh + 7 of the 16 held by the 16-byte vectors a, b (a
// first): a shift by whole words in two select stages, then by half a word
// with one byte permute.  sh is the same for every vector of a row, so the
// selects do not diverge.
__device__ __forceinline__ uint4 bf16_window(uint4 a, uint4 b, int sh) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t s[6], t[5];
#pragma unroll
  for (int i = 0; i < 6; ++i) s[i] = (sh & 4) ? w[i + 2] : w[i];
#pragma unroll
  for (int i = 0; i < 5; ++i) t[i] = (sh & 2) ? s[i + 1] : s[i];
  const uint32_t sel = (sh & 1) ? 0x5432u : 0x3210u;  // high half of t[j], low half of t[j + 1]
  return make_uint4(__byte_perm(t[0], t[1], sel), __byte_perm(t[1], t[2], sel),
                    __byte_perm(t[2], t[3], sel), __byte_perm(t[3], t[4], sel));
}

template <int OP, typename T, int THREADS, int TPR, int VPT, bool CLUSTER>
__global__ void __launch_bounds__(THREADS, (shifted_min_blocks<OP, VPT>()))
    shifted_kernel(const RowArgs a) {
  using V = Vec16<T>;
  constexpr int E = V::kElems;
  constexpr int ES = int(sizeof(T));
  constexpr int NW = THREADS / 32;
  constexpr int WPG = TPR / 32;
  constexpr int GW = TPR < 32 ? TPR : 32;
  constexpr int R = THREADS / TPR;
  constexpr int NIN = (OP == kSoftmaxGrad) ? 2 : 1;  // input matrices per slot (y and dy)
  constexpr int RED = (OP == kSoftmaxGrad) ? kRmsNorm : OP;  // softmax backward reduces a plain sum
  static_assert((TPR % 32 == 0 || 32 % TPR == 0) && THREADS % TPR == 0 && TPR >= 4, "row groups");
  static_assert(!CLUSTER || TPR == THREADS, "a clustered row spans the whole CTA");
  static_assert(NW <= 16, "block-reduction buffer holds 16 warps");
  static_assert(!(CLUSTER && (OP == kXent || OP == kXentGrad)), "cross-entropy rows are streamed, not split");

  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* xbar = reinterpret_cast<uint64_t*>(smem + 8 * kMaxSlots);
  float* cnt_red = reinterpret_cast<float*>(smem + 384);   // [2][16] LayerNorm warp counts or M2 partials
  float2* red = reinterpret_cast<float2*>(smem + 512);
  float2* xbuf = reinterpret_cast<float2*>(smem + 768);
  unsigned char* ring = smem + kSmemHeader;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = tid / TPR, l = tid % TPR;
  const int64_t M = a.M, N = a.N;
  const int S = a.slots;
  const int64_t K = a.chunks;  // chunks per row slice (cross-entropy streaming), else 1
  // Elements of one chunk of a streamed row (a.chunk_elems): the row in K
  // equal parts, each at most (TPR * VPT - 1) * E elements so that its
  // aligned copy fits the TPR * VPT vectors of a row group.

  uint32_t C = 1, rank = 0, cid = blockIdx.x, ncl = gridDim.x;
  if constexpr (CLUSTER) {
    C = cluster_nctarank();
    rank = cluster_ctarank();
    cid = cluster_id_x();
    ncl = num_clusters_x();
  }
  // Column slice of this CTA, in elements (the whole row unless clustered).
  const int64_t SE = (N + C - 1) / C;
  const int64_t e0 = min(N, int64_t(rank) * SE);
  const int64_t ne = min(N, e0 + SE) - e0;
  const int64_t CHE = a.chunk_elems;  // streamed rows never span a cluster: ne = N

  const int64_t n_local = a.num_items > int64_t(cid) ? (a.num_items - 1 - cid) / ncl + 1 : 0;
  const int64_t q_total = n_local * K;
  const uint32_t full0 = smem_addr(full), xbar0 = smem_addr(xbar), ring0 = smem_addr(ring);
  const uintptr_t xaddr = reinterpret_cast<uintptr_t>(a.x);

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
  // The aligned range of the first step into L2 while the previous kernel in
  // the stream finishes (a hint; the copies into shared memory follow the wait).
  if (!CLUSTER && tid == 0 && q_total > 0) {
    const int64_t L = (K > 1) ? int64_t(cid) * N : int64_t(cid) * R * N;
    const int64_t H = (K > 1) ? min(L + N, L + CHE) : min(M, (int64_t(cid) + 1) * R) * N;
    const uintptr_t lo = (xaddr + uintptr_t(L * ES)) & ~uintptr_t(15);
    const uintptr_t hi = (xaddr + uintptr_t(H * ES) + 15) & ~uintptr_t(15);
    const int64_t bytes = H > L ? int64_t(hi - lo) : 0;
#pragma unroll
    for (int in = 0; in < NIN; ++in) {
      const uintptr_t s_in = in == 0 ? lo : lo - xaddr + reinterpret_cast<uintptr_t>(a.x2);
      for (int64_t o = 0; o < bytes; o += kCopyBytes)
        bulk_prefetch_l2(reinterpret_cast<const void*>(s_in + uintptr_t(o)),
                         uint32_t(min(kCopyBytes, bytes - o)));
    }
  }
  grid_dependency_wait();
  allow_dependent_launch();

  // The flat element range [L, H) of step (item, chunk) and the flat index F0
  // of its slot's first element (the aligned start of the copy).
  auto step_range = [&](int64_t it, int64_t c, int64_t& L, int64_t& H) {
    if (K > 1) {
      L = it * N + e0 + c * CHE;
      H = min(it * N + e0 + ne, L + CHE);
    } else if (CLUSTER) {
      L = it * N + e0;
      H = L + ne;
    } else {
      L = it * R * N;
      H = min(M, (it + 1) * R) * N;
    }
    if (H < L) H = L;  // an empty trailing chunk of a short slice
  };
  auto slot_origin = [&](int64_t L) -> int64_t {  // F0, in elements relative to x
    const uintptr_t a0 = (xaddr + uintptr_t(L * ES)) & ~uintptr_t(15);
    return (int64_t(a0) - int64_t(xaddr)) / ES;
  };

  // ---- producer (thread 0) ----
  uint64_t policy = 0;
  int64_t p_item = cid, p_left = q_total;
  int p_chunk = 0, p_slot = 0;
  auto issue_next = [&]() {
    int64_t L, H;
    step_range(p_item, p_chunk, L, H);
    int64_t bytes = 0;
    uintptr_t src = 0;
    if (H > L) {
      src = (xaddr + uintptr_t(L * ES)) & ~uintptr_t(15);
      const uintptr_t end = (xaddr + uintptr_t(H * ES) + 15) & ~uintptr_t(15);
      bytes = int64_t(end - src);
    }
    const uint32_t dst = ring0 + uint32_t(p_slot) * uint32_t(NIN) * a.slot_bytes;
    const uint32_t bar = full0 + 8u * uint32_t(p_slot);
    mbar_arrive_expect_tx(bar, uint32_t(bytes) * NIN);
#pragma unroll
    for (int in = 0; in < NIN; ++in) {
      // the second input (dy) has x's alignment modulo 16, so the same element range
      const uintptr_t s_in = in == 0 ? src : src - xaddr + reinterpret_cast<uintptr_t>(a.x2);
      for (int64_t o = 0; o < bytes; o += kCopyBytes)
        bulk_copy_g2s(dst + uint32_t(in) * a.slot_bytes + uint32_t(o),
                      reinterpret_cast<const void*>(s_in + uintptr_t(o)),
                      uint32_t(min(kCopyBytes, bytes - o)), bar, policy);
    }
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

  // ---- per-column parameters, staged once (RMSNorm w; LayerNorm w and b) ----
  constexpr bool kAffine = (OP == kRmsNorm || OP == kLayerNorm);
  T* wsm = reinterpret_cast<T*>(ring + size_t(S) * NIN * a.slot_bytes);
  T* bsm = wsm + param_slice_bytes((SE * ES + 15) / 16) / ES;
  if constexpr (kAffine) {
    const T* wg = static_cast<const T*>(a.w) + e0;
    const T* bg = static_cast<const T*>(a.bias) + e0;  // unused when null
    for (int64_t c = tid; c < ne; c += THREADS) {
      wsm[c] = wg[c];
      if constexpr (OP == kLayerNorm) bsm[c] = a.bias != nullptr ? bg[c] : T(0.f);
    }
    __syncthreads();
  }

  constexpr uint32_t kFill =
      (OP == kRmsNorm || OP == kLayerNorm || OP == kSoftmaxGrad) ? 0u : V::kNegInfBits;
  uint4 xr[VPT];
  uint4 xr2[NIN == 2 ? VPT : 1];  // softmax backward: dy
  float run_m = kNegInf, run_s = 0.f;  // cross-entropy: running pair of a streamed row
  float xt = 0.f;                      // cross-entropy: x[target] if this thread holds it
  bool own_t = false;
  int64_t trow = -1, t_next = -1;
  if constexpr (OP == kXent) {
    const int64_t row0 = (K > 1) ? int64_t(cid) : int64_t(cid) * R + g;
    if (q_total > 0 && row0 < M) t_next = __ldg(a.target + row0);
  }
  float g_lb = 0.f, g_zf = 1.f, g_gv = 1.f;  // kXentGrad: lse log2 e, 1 + 2 z lse, upstream factor
  int64_t g_t = -1;                          // kXentGrad: the row's target
  float ln_cc = 0.f;  // LayerNorm: elements of cluster rank (lane % 16)
  if constexpr (OP == kLayerNorm && CLUSTER) {
    const uint32_t r = uint32_t(lane) & 15u;
    const int64_t s0 = min(N, int64_t(r) * SE);
    ln_cc = r < C ? float(min(N, s0 + SE) - s0) : 0.f;
  }
  bool failed = false, abort = false;
  int64_t q = 0, item = cid;
  int j = 0, slot = 0;
  uint32_t phase = 0, ibit = 0, xphase = 0;

  for (; q < q_total; ++q) {
    if (!mbar_wait<false>(full0 + 8u * uint32_t(slot), phase, a.timeout_ns)) {
      report_status(a.status, kStatusTimeout);
      failed = true;
    }
    const bool single = (K > 1) || CLUSTER;  // one row per step
    int64_t L, H;
    step_range(item, j, L, H);
    const int64_t F0 = slot_origin(L);
    const int64_t row = single ? item : item * R + g;
    const bool row_ok = row < M;
    // This row group's window of slot elements [s_lo, s_hi), the slot vectors
    // over it [vb, vb + cn), and the column of element s_lo.
    const int64_t Lg = single ? L : row * N, Hg = single ? H : row * N + N;
    const int s_lo = int(Lg - F0), s_hi = int(Hg - F0);
    const int vb = s_lo / E;
    const int cn = (row_ok && Hg > Lg) ? (s_hi + E - 1) / E - vb : 0;
    const int64_t col0 = single ? L - item * N : 0;  // column of element s_lo
    const unsigned char* sb = ring + size_t(slot) * NIN * a.slot_bytes + size_t(vb) * 16;

    bool valid[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int lv = l + k * TPR;
      valid[k] = lv < cn && !failed;
      xr[k] = valid[k] ? *reinterpret_cast<const uint4*>(sb + lv * 16)
                       : make_uint4(kFill, kFill, kFill, kFill);
      if (valid[k] && (lv == 0 || lv == cn - 1)) {  // a partial vector at an end of the window
        const int i0 = (vb + lv) * E;
        xr[k] = V::keep(xr[k], s_lo - i0, s_hi - i0, kFill);
      }
      if constexpr (NIN == 2) {  // dy, masked the same way (zero: its products vanish)
        xr2[k] = valid[k] ? *reinterpret_cast<const uint4*>(sb + a.slot_bytes + lv * 16)
                          : make_uint4(0u, 0u, 0u, 0u);
        if (valid[k] && (lv == 0 || lv == cn - 1)) {
          const int i0 = (vb + lv) * E;
          xr2[k] = V::keep(xr2[k], s_lo - i0, s_hi - i0, 0u);
        }
      }
    }

    // ---- cross-entropy backward: no reduction, every step writes its chunk ----
    // dlogits = dloss * ((1 + 2 z lse) exp(x - lse) - onehot(t)); a row whose
    // target is the ignore index (if any) gets 0, one with a target outside [0, N) NaN.
    if constexpr (OP == kXentGrad) {
      if (j == 0 && row_ok) {
        const float lse = __ldg(a.lse + row);
        g_t = __ldg(a.target + row);
        const float gr = a.dloss != nullptr ? __ldg(a.dloss + row) : 1.f;
        const bool ignored = a.has_ignore && g_t == a.ignore_index, tok = g_t >= 0 && g_t < N;
        g_gv = ignored ? 0.f : (tok ? gr : __int_as_float(0x7fc00000));
        g_zf = fmaf(2.f * a.z_loss, lse, 1.f);
        g_lb = lse * kLog2e;
      }
      // The thread holding x[target] reads it from the slot before it is
      // refilled, and rewrites that one output element after its vector.
      int64_t it_t = -1;  // slot element of the target
      bool own_t = false;
      float xt = 0.f;
      if (row_ok && !failed && g_t >= 0 && g_t < N) {
        it_t = row * N + g_t - F0;
        if (it_t >= s_lo && it_t < s_hi) {
          const int vi = int(it_t / E) - vb;
          own_t = vi % TPR == l;
          if (own_t) xt = V::load1(sb + vi * 16 + int(it_t % E) * ES);
        }
      }
      if (__syncthreads_or(failed)) {  // the slot is free: every thread holds its vectors
        abort = true;
        break;
      }
      if (tid == 0 && p_left > 0) issue_next();
      if (++slot == S) {
        slot = 0;
        phase ^= 1u;
      }
      if (j == K - 1) {
        j = 0;
        item += ncl;
      } else {
        ++j;
      }
      unsigned char* yb = static_cast<unsigned char*>(a.y);
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        if (!valid[k]) continue;
        const int i0 = (vb + l + k * TPR) * E;
        const int lo = max(0, s_lo - i0), hi = min(E, s_hi - i0);
        float f[E], o[E];
        V::unpack_fresh(xr[k], f);
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = (exp2_approx(fmaf(f[e], kLog2e, -g_lb)) * g_zf) * g_gv;
        unsigned char* dst = yb + (F0 + i0) * ES;  // 16-byte aligned: dlogits has the logits' alignment
        if (lo == 0 && hi == E) {
          __stcs(reinterpret_cast<uint4*>(dst), V::pack(o));
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e)
            if (e >= lo && e < hi) V::store1(dst + e * ES, o[e]);
        }
      }
      if (own_t) {  // the target element, minus the one-hot 1
        const float p = exp2_approx(fmaf(xt, kLog2e, -g_lb)) * g_zf - 1.f;
        V::store1(yb + (F0 + it_t) * ES, p * g_gv);
      }
      continue;
    }

    // ---- thread-level reduction ----
    float pm = kNegInf, ps = 0.f, pn = 0.f, tm = kNegInf;
    if constexpr (OP == kSoftmaxGrad) {  // sum dy * y
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        float f[E], d[E];
        V::unpack(xr[k], f);
        V::unpack(xr2[k], d);
#pragma unroll
        for (int e = 0; e < E; e += 2)
          acc = fma2(make_float2(f[e], f[e + 1]), make_float2(d[e], d[e + 1]), acc);
      }
      ps = acc.x + acc.y;
    } else if constexpr (OP == kRmsNorm) {
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        float f[E];
        V::unpack(xr[k], f);
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          const float2 v = make_float2(f[e], f[e + 1]);
          acc = fma2(v, v, acc);
        }
      }
      ps = acc.x + acc.y;
    } else if constexpr (OP == kLayerNorm && !CLUSTER) {
      // First of two passes over the registers: the row sum (padding is 0).
      // The squared deviations from the row mean follow the block reduction.
      float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        if (!valid[k]) continue;
        float f[E];
        V::unpack(xr[k], f);
#pragma unroll
        for (int e = 0; e < E; e += 2) s2 = add2(s2, make_float2(f[e], f[e + 1]));
      }
      ps = s2.x + s2.y;
    } else if constexpr (OP == kLayerNorm) {
      float2 s2 = make_float2(0.f, 0.f);
      int cnt = 0;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        if (!valid[k]) continue;
        const int i0 = (vb + l + k * TPR) * E;
        cnt += min(E, s_hi - i0) - max(0, s_lo - i0);
        float f[E];
        V::unpack(xr[k], f);
#pragma unroll
        for (int e = 0; e < E; e += 2) s2 = add2(s2, make_float2(f[e], f[e + 1]));  // padding is 0
      }
      const float sum = s2.x + s2.y;
      const float mu = cnt > 0 ? __fdiv_rn(sum, float(cnt)) : 0.f;
      float qd = 0.f;
      float2 q2 = make_float2(0.f, 0.f);
      const float2 nmu = make_float2(-mu, -mu);
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        if (!valid[k]) continue;
        const int i0 = (vb + l + k * TPR) * E;
        const int lo = max(0, s_lo - i0), hi = min(E, s_hi - i0);
        float f[E];
        V::unpack(xr[k], f);
        if (lo == 0 && hi == E) {  // a whole vector: packed
#pragma unroll
          for (int e = 0; e < E; e += 2) {
            const float2 d = add2(make_float2(f[e], f[e + 1]), nmu);
            q2 = fma2(d, d, q2);
          }
        } else {  // a partial vector at an end of the window
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const float d = f[e] - mu;
            if (e >= lo && e < hi) qd = fmaf(d, d, qd);
          }
        }
      }
      pn = float(cnt);
      pm = mu;
      ps = qd + (q2.x + q2.y);
    } else {
      if constexpr (OP == kXent) {
        if (j == 0) {
          run_m = kNegInf;
          run_s = 0.f;
          own_t = false;
          trow = t_next;
          const int64_t nrow = single ? item + ncl : (item + ncl) * R + g;
          t_next = nrow < M ? __ldg(a.target + nrow) : -1;
        }
        if (row_ok && trow >= 0 && trow < N) {  // x[target] if it lies in this thread's vectors
          const int64_t it = row * N + trow - F0;  // slot element of the target
          if (it >= s_lo && it < s_hi) {
            const int vi = int(it / E) - vb;
            if (vi % TPR == l) {  // one element read from the slot
              xt = V::load1(sb + vi * 16 + int(it % E) * int(sizeof(T)));
              own_t = true;
            }
          }
        }
      }
      float m = (OP == kXent) ? run_m : kNegInf;
      // Cross-entropy: the maximum as a tree and four accumulator pairs
      // (short dependency chains); softmax keeps one chain of each.
      constexpr bool kShortChains = (OP == kXent);
      if constexpr (kShortChains) {
        m = fmaxf(m, V::template max_all<VPT>(xr));
      } else {
#pragma unroll
        for (int k = 0; k < VPT; ++k) m = V::max_into(m, xr[k]);
      }
      const float mb = (m == kNegInf) ? 0.f : m * kLog2e;
      const float2 l2e = make_float2(kLog2e, kLog2e), nmb = make_float2(-mb, -mb);
      float2 a4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                      make_float2(0.f, 0.f)};
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        float f[E];
        V::unpack(xr[k], f);
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          const float2 t = fma2(make_float2(f[e], f[e + 1]), l2e, nmb);
          const int c = kShortChains ? ((k * E + e) / 2) & 3 : 0;
          a4[c] = add2(a4[c], make_float2(exp2_approx(t.x), exp2_approx(t.y)));  // padding: 2^-inf = 0
        }
      }
      const float2 acc =
          kShortChains ? add2(add2(a4[0], a4[1]), add2(a4[2], a4[3])) : a4[0];
      if constexpr (OP == kSoftmax) {
        tm = m;
        pm = m;
        ps = acc.x + acc.y;
      } else {  // fold the chunk into the running pair of the row
        if (m != kNegInf) run_s = run_s * exp2_approx((run_m - m) * kLog2e) + (acc.x + acc.y);
        run_m = m;
        pm = run_m;
        ps = run_s;
      }
    }

    // ---- warp butterfly; warp partials to the block buffer ----
    const bool row_end = (j == K - 1);
    if (row_end) {
      if constexpr (OP == kLayerNorm && !CLUSTER) {
        ps = group_sum<GW>(ps);  // the row group's sum, through the barrier below
      } else if constexpr (OP == kLayerNorm) {
        group_welford<GW>(pn, pm, ps);
        if (WPG > 1 && lane == 0) cnt_red[ibit * 16 + warp] = pn;
      } else {
        warp_reduce<RED, GW>(pm, ps);
      }
      if (WPG > 1 && lane == 0) red[ibit * 16 + warp] = make_float2(pm, ps);
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
    if (row_end) {
      xphase ^= ibit;
      ibit ^= 1u;
    }
    if (j == K - 1) {
      j = 0;
      item += ncl;
    } else {
      ++j;
    }
    if (!row_end) continue;

    // ---- block reduction over the warps of this row group ----
    if constexpr (OP == kLayerNorm && !CLUSTER) {
      // The mean from the row sum (warp partials added in a fixed order), then
      // the second pass: squared deviations from it, summed the same way.
      float tot = ps;
      if constexpr (WPG > 1) {
        tot = 0.f;
#pragma unroll
        for (int w = 0; w < WPG; ++w) tot += red[row_ibit * 16 + g * WPG + w].y;
      }
      const float mu = tot * a.inv_n;
      const float2 nmu = make_float2(-mu, -mu);
      float qd = 0.f;
      float2 q2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        if (!valid[k]) continue;
        const int i0 = (vb + l + k * TPR) * E;
        const int lo = max(0, s_lo - i0), hi = min(E, s_hi - i0);
        float f[E];
        V::unpack(xr[k], f);
        if (lo == 0 && hi == E) {  // a whole vector: packed
#pragma unroll
          for (int e = 0; e < E; e += 2) {
            const float2 d = add2(make_float2(f[e], f[e + 1]), nmu);
            q2 = fma2(d, d, q2);
          }
        } else {  // a partial vector at an end of the window
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const float d = f[e] - mu;
            if (e >= lo && e < hi) qd = fmaf(d, d, qd);
          }
        }
      }
      float m2 = group_sum<GW>(qd + (q2.x + q2.y));
      if constexpr (WPG > 1) {
        if (lane == 0) cnt_red[row_ibit * 16 + warp] = m2;
        __syncthreads();
        m2 = 0.f;
#pragma unroll
        for (int w = 0; w < WPG; ++w) m2 += cnt_red[row_ibit * 16 + g * WPG + w];
      }
      pm = mu;
      ps = m2;
    } else if constexpr (WPG > 1) {
      if constexpr (OP == kLayerNorm) {  // butterfly of width WPG; lane l takes warp l % WPG
        const int w = row_ibit * 16 + g * WPG + lane % WPG;
        pm = red[w].x;
        ps = red[w].y;
        pn = cnt_red[w];
        group_welford<WPG>(pn, pm, ps);
      } else {
        merge_partials<RED>(red + row_ibit * 16 + g * WPG, WPG, pm, ps);
      }
    }

    // ---- cluster reduction (DSMEM) ----
    if constexpr (CLUSTER) {
      const uint32_t b = row_ibit;
      const uint32_t xb = xbar0 + 8u * b;
      if (tid == 0) {
        mbar_arrive_expect_tx(xb, C * 8u);
        const uint32_t mine = smem_addr(xbuf + b * kMaxCluster + rank);
        for (uint32_t r = 0; r < C; ++r) st_async_f2(map_to_rank(mine, r), pm, ps, map_to_rank(xb, r));
      }
      if (!mbar_wait<true>(xb, row_xphase, a.timeout_ns)) {
        report_status(a.status, kStatusTimeout);
        failed = true;
      }
      if constexpr (OP == kLayerNorm) {  // width 16; ranks beyond C hold count 0
        const uint32_t r = uint32_t(lane) & 15u;
        const float2 v = r < C ? xbuf[b * kMaxCluster + r] : make_float2(0.f, 0.f);
        pn = ln_cc;
        pm = v.x;
        ps = v.y;
        group_welford<16>(pn, pm, ps);
      } else {
        merge_partials<RED>(xbuf + b * kMaxCluster, int(C), pm, ps);
      }
    }

    // ---- finish: whole vectors with one 16-byte store, partial ones by element ----
    if (!row_ok) continue;
    unsigned char* yb = static_cast<unsigned char*>(a.y);
    if constexpr (OP == kXent) {
      const bool leader = (l == 0 && rank == 0);
      const bool ignored = a.has_ignore && trow == a.ignore_index;
      if (leader || own_t) {
        const float lse = pm + logf(ps);
        if (leader) {
          if (a.lse != nullptr) a.lse[row] = lse;
          if (ignored) {
            a.loss[row] = 0.f;
          } else if (!(trow >= 0 && trow < N)) {
            a.loss[row] = __int_as_float(0x7fc00000);  // NaN
          }
        }
        if (own_t && !ignored) a.loss[row] = fmaf(a.z_loss * lse, lse, lse - xt);  // + z lse^2
      }
    } else {
      float sa = 0.f, sb2 = 0.f;  // per-row factors of the finish
      if constexpr (OP == kSoftmax) {
        sa = softmax_scale(tm, pm, ps);                                               // scale
        sb2 = (tm == kNegInf) ? 0.f : tm * kLog2e;                                    // m_t log2 e
      } else if constexpr (OP == kRmsNorm) {
        sa = rsqrtf(fmaf(ps, a.inv_n, a.eps));
        if (l == 0 && rank == 0 && a.rstd != nullptr) a.rstd[row] = sa;
      } else if constexpr (OP == kSoftmaxGrad) {
        sb2 = -ps;  // -sum dy * y
      } else {  // LayerNorm
        sa = rsqrtf(fmaf(ps, a.inv_n, a.eps));
        sb2 = -pm * sa;
        if (l == 0 && rank == 0) {
          if (a.rstd != nullptr) a.rstd[row] = sa;
          if (a.mean != nullptr) a.mean[row] = pm;
        }
      }
      const int64_t cbase = col0 - e0 - s_lo;  // staged column of slot element i: cbase + i
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        if (!valid[k]) continue;
        const int i0 = (vb + l + k * TPR) * E;
        const int lo = max(0, s_lo - i0), hi = min(E, s_hi - i0);
        float f[E], o[E], w[E], bb[E], d[E];
        V::unpack_fresh(xr[k], f);
        if constexpr (NIN == 2) V::unpack_fresh(xr2[k], d);
        if constexpr (kAffine) {  // the columns of this vector, from the staged slice
          if (OP == kLayerNorm && E == 8 && lo == 0 && hi == E) {
            // A whole bf16 vector of LayerNorm: its 8 columns of w and of b
            // start sh elements into an aligned vector of the slice (all 8
            // lie inside the slice, so the second vector, read only when
            // sh > 0, does too).  For RMSNorm's single parameter the element
            // loads below measured faster (16384 x 4097: 72 % against 71 %;
            // LayerNorm 42 % -> 46 % with this).
            const int64_t c0 = cbase + i0;
            const int sh = int(c0 & 7);
            // (With sh = 0 the window is the first vector alone; the index
            // below then reads it twice rather than a vector past the slice.)
            const uint4* wv = reinterpret_cast<const uint4*>(wsm) + (c0 >> 3);
            V::unpack(bf16_window(wv[0], wv[sh ? 1 : 0], sh), w);
            if constexpr (OP == kLayerNorm) {
              const uint4* bv = reinterpret_cast<const uint4*>(bsm) + (c0 >> 3);
              V::unpack(bf16_window(bv[0], bv[sh ? 1 : 0], sh), bb);
            }
          } else {
#pragma unroll
            for (int e = 0; e < E; ++e) {
              const bool in = (e >= lo && e < hi);
              w[e] = in ? V::load1(wsm + (cbase + i0 + e)) : 0.f;
              if constexpr (OP == kLayerNorm) bb[e] = in ? V::load1(bsm + (cbase + i0 + e)) : 0.f;
            }
          }
        }
        const float2 a2 = make_float2(sa, sa), b2 = make_float2(sb2, sb2);
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          const float2 x2 = make_float2(f[e], f[e + 1]);
          float2 v;
          if constexpr (OP == kSoftmax) {  // exp(x - m_t) * scale (scalar: fewer live registers)
            v = make_float2(exp2_approx(fmaf(x2.x, kLog2e, -sb2)) * sa,
                            exp2_approx(fmaf(x2.y, kLog2e, -sb2)) * sa);
          } else if constexpr (OP == kSoftmaxGrad) {  // y * (dy - sum dy * y)
            v = mul2(x2, add2(make_float2(d[e], d[e + 1]), b2));
          } else if constexpr (OP == kRmsNorm) {  // (x * rstd) * w
            v = mul2(mul2(x2, a2), make_float2(w[e], w[e + 1]));
          } else {  // (x * rstd - mean * rstd) * w + b
            v = fma2(fma2(x2, a2, b2), make_float2(w[e], w[e + 1]), make_float2(bb[e], bb[e + 1]));
          }
          o[e] = v.x;
          o[e + 1] = v.y;
        }
        unsigned char* dst = yb + (F0 + i0) * ES;  // 16-byte aligned: y has x's alignment
        if (lo == 0 && hi == E) {
          __stcs(reinterpret_cast<uint4*>(dst), V::pack(o));
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e)
            if (e >= lo && e < hi) V::store1(dst + e * ES, o[e]);
        }
      }
    }
  }

  if (abort) {  // leave no bulk copy in flight into this CTA's shared memory
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
  if constexpr (CLUSTER) cluster_sync_all();
}

}  // namespace qk
