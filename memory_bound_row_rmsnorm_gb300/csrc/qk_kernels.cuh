// qk_kernels.cuh -- the row-reduction kernels for sm_103a (GB300).
//
// row_kernel: the fast path (16-byte aligned rows).  The row reduction is a
// (max, sum of exponentials) pair for softmax and cross-entropy, a sum of
// squares for RMSNorm, and a (count, mean, M2) triple for LayerNorm.
//   * Persistent grid: each CTA (or each cluster of CTAs) walks a strided list
//     of work items.  An item is a block of `threads / row_threads` consecutive
//     rows (contiguous in memory), one row slice of a cluster, or one chunk of
//     a streamed row.
//   * One thread issues bulk TMA copies (cp.async.bulk) of whole items into a
//     ring of shared-memory slots; each slot has an mbarrier that completes
//     when its bytes land.  The ring keeps `slots - 1` items in flight while
//     one is being reduced, so HBM reads are overlapped with the reduction and
//     the stores of earlier rows.  Every input byte crosses HBM once.
//   * Consumers read 16-byte vectors from shared memory (consecutive threads
//     take consecutive vectors: no bank conflicts) into registers, reduce per
//     thread, then warp butterfly, then across the warps of a row through a
//     shared buffer, then -- for rows split over a cluster -- across CTAs by
//     st.async into every peer's shared memory, counted by an mbarrier.
//   * The finish works from registers and stores each output vector once with
//     a 16-byte store.
//   Cited: QbitAI article on QuACK, section "硬件感知的加载与存储策略" (TV layout,
//   128-bit coalesced accesses, asynchronous GMEM->SMEM staging, store straight
//   back to GMEM after the reduction) and section "硬件感知的归约策略" (thread,
//   warp, block and cluster reduction; the arrival-counting barrier that keeps
//   a CTA from reading its buffer before every peer has written it).
//
// direct_kernel: the masked path for rows whose start or length is not a
//   multiple of 16 bytes.  Plain element loads into registers, the same
//   reduction hierarchy, element stores.  Slower but exact on any N.
#pragma once

#include "qk_device.cuh"
#include "qk_internal.h"

#include <type_traits>

namespace qk {

constexpr int64_t kCopyBytes = 32768;  // largest single bulk copy issued
constexpr int kStatusTimeout = 5;      // QK_ERR_TIMEOUT

// Reduces the pair (m, s) (or the sum s for RMSNorm) over WIDTH lanes.
template <int OP, int WIDTH = 32>
__device__ __forceinline__ void warp_reduce(float& m, float& s) {
  if constexpr (OP == kRmsNorm) {
    s = group_sum<WIDTH>(s);
  } else {
    group_ms<WIDTH>(m, s);
  }
}

// Merges n partial pairs (or sums) p[0..n) in index order: the maximum first,
// then each partial rescaled to it once.  Every thread that calls this with
// the same partials gets the same bits.
template <int OP>
__device__ __forceinline__ void merge_partials(const float2* p, int n, float& m, float& s) {
  if constexpr (OP == kRmsNorm) {
    float acc = p[0].y;
    for (int w = 1; w < n; ++w) acc += p[w].y;
    s = acc;
  } else {
    float mx = p[0].x;
    for (int w = 1; w < n; ++w) mx = fmaxf(mx, p[w].x);
    float acc = 0.f;
    if (mx != kNegInf)
      for (int w = 0; w < n; ++w)
        if (p[w].x != kNegInf) acc += p[w].y * exp2_approx((p[w].x - mx) * kLog2e);
    m = mx;
    s = acc;
  }
}

// The softmax finish factor exp(m_t - M) / S of a thread whose own entries
// have maximum m_t, in a row of maximum M and sum S = sum exp(x - M): 0 when
// the thread holds only -inf entries (their probabilities are 0), NaN when the
// whole row is -inf (S = 0: there is no distribution to normalise, and the
// plain definition gives 0/0).
__device__ __forceinline__ float softmax_scale(float tm, float pm, float ps) {
  if (pm == kNegInf) return __int_as_float(0x7fc00000);
  return (tm == kNegInf) ? 0.f : __fdividef(exp2_approx((tm - pm) * kLog2e), ps);
}

// TWO_PASS (softmax, RMSNorm, LayerNorm rows longer than a cluster holds): every row
// slice is streamed through the ring twice in chunks -- the first pass
// accumulates the reduction, the second re-reads each chunk and writes its
// outputs with the row's totals (three HBM passes instead of two).
// Residency requests for the launch bounds (0: none).  A few 128-thread plans
// sit just under an occupancy step; these keep the register allocator there.
template <int OP, typename T, int THREADS, int VPT, bool CLUSTER, bool TWO_PASS>
constexpr int row_min_blocks() {
  if (THREADS != 128 || VPT != 4 || CLUSTER || TWO_PASS) return 0;
  if (OP == kSoftmax) return std::is_same<T, float>::value ? 10 : 8;
  if (OP == kRmsNorm) return std::is_same<T, float>::value ? 8 : 0;
  return 0;
}

template <int OP, typename T, int THREADS, int TPR, int VPT, bool CLUSTER, bool TWO_PASS = false>
__global__ void __launch_bounds__(THREADS, (row_min_blocks<OP, T, THREADS, VPT, CLUSTER, TWO_PASS>()))
    row_kernel(const RowArgs a) {
  using V = Vec16<T>;
  constexpr int E = V::kElems;       // elements per 16-byte vector
  constexpr int NW = THREADS / 32;   // warps per CTA
  constexpr int WPG = TPR / 32;      // warps per row group (0: a group is part of a warp)
  constexpr int GW = TPR < 32 ? TPR : 32;  // lanes of a warp that share a row
  constexpr int R = THREADS / TPR;   // rows per item (unclustered, unchunked)
  constexpr int64_t CH = int64_t(TPR) * VPT;  // vectors per row-slice chunk
  static_assert((TPR % 32 == 0 || 32 % TPR == 0) && THREADS % TPR == 0 && TPR >= 4,
                "a row group is whole warps or a power-of-two part of one");
  static_assert(!CLUSTER || TPR == THREADS, "a clustered row spans the whole CTA");
  static_assert(NW <= 16, "block-reduction buffer holds 16 warps");
  static_assert(!TWO_PASS || (TPR == THREADS && OP != kXent),
                "two passes: softmax, RMSNorm and LayerNorm, one row per CTA");

  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);                  // [kMaxSlots]
  uint64_t* xbar = reinterpret_cast<uint64_t*>(smem + 8 * kMaxSlots);  // [2]
  float* cnt_red = reinterpret_cast<float*>(smem + 384);               // [2][16] LayerNorm counts
  float2* red = reinterpret_cast<float2*>(smem + 512);                 // [2][16]
  float2* xbuf = reinterpret_cast<float2*>(smem + 768);                // [2][kMaxCluster]
  unsigned char* ring = smem + kSmemHeader;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int g = tid / TPR;  // row group inside an item
  const int l = tid % TPR;  // thread inside its row group
  const int64_t M = a.M, N = a.N;
  const int64_t NV = N / E;  // vectors per row
  const int S = a.slots;
  const int64_t K = a.chunks;              // chunks per row slice
  const int64_t KK = TWO_PASS ? 2 * K : K;  // ring steps per work item
  constexpr bool kChunked = TWO_PASS;        // slices stream in chunks (also when K > 1)

  uint32_t C = 1, rank = 0, cid = blockIdx.x, ncl = gridDim.x;
  if constexpr (CLUSTER) {
    C = cluster_nctarank();
    rank = cluster_ctarank();
    cid = cluster_id_x();
    ncl = num_clusters_x();
  }
  // Column slice of this CTA, in vectors (the whole row unless clustered).
  const int64_t SV = (NV + C - 1) / C;
  const int64_t v0 = min(NV, int64_t(rank) * SV);
  const int64_t nv = min(NV, v0 + SV) - v0;

  // Local steps: item i of this cluster is cid + i * ncl; each item has K chunks.
  const int64_t n_local = a.num_items > int64_t(cid) ? (a.num_items - 1 - cid) / ncl + 1 : 0;
  const int64_t q_total = n_local * KK;

  const uint32_t full0 = smem_addr(full), xbar0 = smem_addr(xbar), ring0 = smem_addr(ring);
  const unsigned char* xg = static_cast<const unsigned char*>(a.x);

  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(full0 + 8 * s, 1);
    mbar_init(xbar0, 1);
    mbar_init(xbar0 + 8, 1);
    fence_mbar_init();
  }
  if constexpr (CLUSTER) {
    cluster_sync_all();  // peers' barriers exist before anyone stores into them
  } else {
    __syncthreads();
  }
  // While the previous kernel in the stream finishes, bring this CTA's first
  // item (the slots of its first ring fill) into L2, so that HBM is not idle
  // between the two kernels.  (Not for clusters: their launches are long and
  // measured a point or two slower with it.)
  if (!CLUSTER && tid == 0 && q_total > 0) {
    int64_t off, bytes;
    if (K > 1 || kChunked) {  // the first chunks of the row
      off = int64_t(cid) * NV * 16;
      bytes = min(int64_t(S) * CH, nv) * 16;
    } else {
      const int64_t r0 = int64_t(cid) * R;
      off = r0 * NV * 16;
      bytes = min(int64_t(R), M - r0) * NV * 16;
    }
    for (int64_t o = 0; o < bytes; o += kCopyBytes)
      bulk_prefetch_l2(xg + off + o, uint32_t(min(kCopyBytes, bytes - o)));
  }
  // Everything above touched only shared memory (and L2, by hint); from here
  // on global memory is read, which the previous kernel may still be writing.
  grid_dependency_wait();
  allow_dependent_launch();

  // Producer state (thread 0 only): the next step to load, as (item, chunk)
  // and its ring slot.  Steps are issued in order, so everything advances by
  // increments -- no 64-bit division in the loop.
  uint64_t policy = 0;
  int64_t p_item = cid, p_left = q_total;
  int p_chunk = 0, p_slot = 0;
  auto issue_next = [&]() {
    int64_t off, bytes;
    if (K > 1 || kChunked) {  // one chunk of this CTA's slice of a streamed row
      const int64_t c0 = int64_t(p_chunk >= K ? p_chunk - K : p_chunk) * CH;  // 2nd pass: same chunks
      off = (p_item * NV + v0 + c0) * 16;
      // K is sized for the longest slice; the last CTA's slice may be shorter,
      // so its last chunks can be empty (then the barrier just completes).
      bytes = max(int64_t(0), min(CH, nv - c0)) * 16;
    } else if (CLUSTER) {  // this CTA's slice of one row
      off = (p_item * NV + v0) * 16;
      bytes = nv * 16;
    } else {  // R consecutive rows
      const int64_t r0 = p_item * R;
      off = r0 * NV * 16;
      bytes = min(int64_t(R), M - r0) * NV * 16;
    }
    const uint32_t dst = ring0 + uint32_t(p_slot) * a.slot_bytes;
    const uint32_t bar = full0 + 8u * uint32_t(p_slot);
    mbar_arrive_expect_tx(bar, uint32_t(bytes));
    for (int64_t o = 0; o < bytes; o += kCopyBytes)
      bulk_copy_g2s(dst + uint32_t(o), xg + off + o, uint32_t(min(kCopyBytes, bytes - o)), bar,
                    policy);
    if (++p_slot == S) p_slot = 0;
    if (++p_chunk == KK) {
      p_chunk = 0;
      p_item += ncl;
    }
    --p_left;
  };
  if (tid == 0) {
    policy = l2_evict_first_policy();
    for (int s = 0; s < S && p_left > 0; ++s) issue_next();
  }

  // RMSNorm weight: the columns a thread touches never change, so its share
  // of w is loaded once into registers -- unless that would take more than
  // 8 vectors of registers, in which case the finish re-reads it through L1
  // (the slice a CTA needs stays cached there; HBM sees w once).
  // two passes: columns change per chunk
  constexpr bool kWeightInRegs = VPT <= kAffineRegsMaxVpt && !TWO_PASS;
  constexpr bool kAffine = (OP == kRmsNorm || OP == kLayerNorm);
  // LayerNorm's bias likewise, but only up to 4 vectors: with 8, w and b
  // together would cost a second CTA per SM.  What LayerNorm does not hold in
  // registers it stages in shared memory, so that the finish never waits on
  // a global load.
  constexpr bool kBiasInRegs = OP == kLayerNorm && VPT <= kLnBiasRegsMaxVpt && !TWO_PASS;
  constexpr bool kWeightInSmem = OP == kLayerNorm && !kWeightInRegs && !TWO_PASS;
  constexpr bool kBiasInSmem = OP == kLayerNorm && !kBiasInRegs && !TWO_PASS;
  uint4 wv[kWeightInRegs ? VPT : 1];
  uint4 bv[kBiasInRegs ? VPT : 1];
  uint4* wsm = reinterpret_cast<uint4*>(ring + size_t(S) * a.slot_bytes);
  uint4* bsm = wsm + (kWeightInSmem ? param_slice_bytes(SV) / 16 : 0);
  const uint4* wg = static_cast<const uint4*>(a.w) + v0;
  const uint4* bg = static_cast<const uint4*>(a.bias) + v0;  // unused when bias is null
  if constexpr (kAffine && kWeightInRegs) {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int64_t lv = l + int64_t(k) * TPR;
      wv[k] = lv < nv ? __ldg(wg + lv) : make_uint4(0u, 0u, 0u, 0u);
      if constexpr (kBiasInRegs)
        bv[k] = (lv < nv && a.bias != nullptr) ? __ldg(bg + lv) : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  if constexpr (kWeightInSmem || kBiasInSmem) {
    for (int64_t v = tid; v < nv; v += THREADS) {
      if constexpr (kWeightInSmem) wsm[v] = __ldg(wg + v);
      if constexpr (kBiasInSmem) bsm[v] = a.bias != nullptr ? __ldg(bg + v) : make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
  }

  // Softmax keeps exp(x - thread max) in registers for the finish, unless
  // that would take too many registers (bf16 with 16 vectors a thread, or 8 in
  // a clustered kernel, where occupancy hides the DSMEM exchange): then the finish
  // recomputes it from the packed input, trading one more SFU op per element
  // for half the registers (more CTAs per SM).
  constexpr bool kKeepExp = !(E == 8 && (VPT >= 16 || (CLUSTER && VPT >= 8)));
  uint4 xr[VPT];                       // raw input vectors of the current row (chunk)
  float ef[kKeepExp ? VPT * E : 1];    // softmax: exp(x - thread max)
  float run_m = kNegInf, run_s = 0.f;  // cross-entropy, two-pass softmax: running pair
  float run_ss = 0.f;                  // two-pass RMSNorm: running sum of squares (LayerNorm: M2)
  float run_n = 0.f;                   // two-pass LayerNorm: running count (mean in run_m)
  float tot_a = 0.f, tot_b = 0.f;      // two-pass: the row's totals for the second pass
  float xt = 0.f;                      // cross-entropy: x[target] if this thread holds it
  bool own_t = false;
  int64_t trow = -1;
  int64_t t_next = -1;  // cross-entropy: target of the next item's row
  if constexpr (OP == kXent) {
    const int64_t row0 = (K > 1 || CLUSTER) ? int64_t(cid) : int64_t(cid) * R + g;
    if (q_total > 0 && row0 < M) t_next = __ldg(a.target + row0);
  }
  // LayerNorm merges (count, mean, M2) partials; the counts follow from the
  // slice geometry (a LayerNorm slice is never chunked), so they are fixed
  // for the launch: `ln_full` when every thread holds VPT vectors, the count
  // of warp (lane % WPG) of this row group, and that of cluster rank (lane % 16).
  bool ln_full = false;
  float ln_wc = 0.f, ln_cc = 0.f;
  if constexpr (OP == kLayerNorm) {
    ln_full = !TWO_PASS && (nv == int64_t(TPR) * VPT);
    if constexpr (WPG > 1) {
      const int w = lane % WPG;
      int c = 0;
#pragma unroll
      for (int k = 0; k < VPT; ++k) c += max(0, min(32, int(nv) - k * TPR - w * 32));
      ln_wc = float(c * E);
    }
    if constexpr (CLUSTER) {
      const uint32_t r = uint32_t(lane) & 15u;
      const int64_t s0 = min(NV, int64_t(r) * SV);
      ln_cc = r < C ? float((min(NV, s0 + SV) - s0) * E) : 0.f;
    }
  }
  bool failed = false;  // a wait of this thread ran out
  bool abort = false;   // block-uniform: some thread's wait ran out
  // Consumer position: step q is chunk j of local item i (item = cid + i*ncl),
  // held in ring slot `slot` whose barrier phase parity is `phase`.
  int64_t q = 0, item = cid;
  int j = 0, slot = 0;
  uint32_t phase = 0, ibit = 0, xphase = 0;  // parities: ring, item (red/xbuf), cluster barrier

  for (; q < q_total; ++q) {
    if (!mbar_wait<false>(full0 + 8u * uint32_t(slot), phase, a.timeout_ns)) {
      report_status(a.status, kStatusTimeout);
      failed = true;
    }

    const bool single = (K > 1) || CLUSTER || kChunked;  // one row per item
    const int64_t row = single ? item : item * R + g;
    const bool row_ok = row < M;
    const bool second = TWO_PASS && j >= K;  // second pass over the row: write outputs
    const int64_t chunk = second ? j - K : j;
    const bool chunked = (K > 1) || kChunked;
    // vectors of this row in the slot (0 for an empty trailing chunk of a short slice)
    const int cn = int(chunked ? max(int64_t(0), min(CH, nv - chunk * CH)) : nv);
    const int64_t cbase = chunked ? v0 + chunk * CH : v0;  // first column vector in the slot
    const unsigned char* sb =
        ring + size_t(slot) * a.slot_bytes + (single ? size_t(0) : size_t(g) * size_t(NV) * 16);

    // Padding lanes get the reduction's neutral element (0 for a sum of
    // squares, -inf for a maximum / sum of exponentials), so the arithmetic
    // below needs no per-element masking.
    constexpr uint32_t kFill = (OP == kRmsNorm || OP == kLayerNorm) ? 0u : V::kNegInfBits;
    bool valid[VPT];
    // Cross-entropy: when every vector of the group is data, plain loads
    // without the per-vector selects (the other operators measured no gain
    // and, for some plans, a register more than a resident CTA allows).
    if (OP == kXent && row_ok && !failed && cn == TPR * VPT) {
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        valid[k] = true;
        xr[k] = *reinterpret_cast<const uint4*>(sb + (l + k * TPR) * 16);
      }
    } else {
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int lv = l + k * TPR;
        valid[k] = row_ok && lv < cn && !failed;
        xr[k] = valid[k] ? *reinterpret_cast<const uint4*>(sb + lv * 16)
                         : make_uint4(kFill, kFill, kFill, kFill);
      }
    }

    // ---- thread-level reduction (registers) ----
    float pm = kNegInf, ps = 0.f;  // partial (max, sum-exp), or (-, sum of squares)
    float pn = 0.f;                // LayerNorm: element count of the partial (mean pm, M2 ps)
    float tm = kNegInf;            // softmax: this thread's own maximum
    if (second) {
      // two-pass, second pass: nothing to reduce
    } else if constexpr (OP == kRmsNorm && TWO_PASS) {
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
      run_ss = (j == 0 ? 0.f : run_ss) + (acc.x + acc.y);
      ps = run_ss;
    } else if constexpr (OP == kLayerNorm) {
      // (count, mean, M2) of this thread's elements: the mean first, then the
      // squared deviations from it, both over the registers.  Padding is 0,
      // so it adds nothing to the sum; it is left out of the count and of M2.
      // (Four independent accumulator pairs: short dependency chains.)
      constexpr float kInvFull = 1.f / float(E * VPT);  // a power of two: exact
      float2 s4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                      make_float2(0.f, 0.f)};
      float cnt = 0.f;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        float f[E];
        V::unpack(xr[k], f);
        cnt += valid[k] ? float(E) : 0.f;
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          const int c = ((k * E + e) / 2) & 3;
          s4[c] = add2(s4[c], make_float2(f[e], f[e + 1]));
        }
      }
      const float2 s2 = add2(add2(s4[0], s4[1]), add2(s4[2], s4[3]));
      const float sum = s2.x + s2.y;
      // Full rows: every thread holds VPT vectors (a padded thread of a row
      // that is not written has sum 0 and M2 0, which harms nothing).
      const float mu = ln_full ? sum * kInvFull : (cnt > 0.f ? __fdiv_rn(sum, cnt) : 0.f);
      const float2 nmu = make_float2(-mu, -mu);
      float2 q4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                      make_float2(0.f, 0.f)};
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        if (!ln_full && !valid[k]) continue;
        float f[E];
        V::unpack(xr[k], f);
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          const int c = ((k * E + e) / 2) & 3;
          const float2 d = add2(make_float2(f[e], f[e + 1]), nmu);
          q4[c] = fma2(d, d, q4[c]);
        }
      }
      const float2 q2 = add2(add2(q4[0], q4[1]), add2(q4[2], q4[3]));
      pn = cnt;
      pm = ln_full ? sum : mu;  // full rows reduce in sum form (below)
      ps = q2.x + q2.y;
      if constexpr (TWO_PASS) {  // fold the chunk into the thread's running (count, mean, M2)
        if (j == 0) {
          run_n = pn, run_m = pm, run_ss = ps;
        } else {
          welford_merge(run_n, run_m, run_ss, pn, pm, ps);
        }
        pn = run_n, pm = run_m, ps = run_ss;
      }
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
    } else {
      if constexpr (TWO_PASS) {
        if (j == 0) {
          run_m = kNegInf;
          run_s = 0.f;
        }
      }
      if constexpr (OP == kXent) {
        if (j == 0) {
          run_m = kNegInf;
          run_s = 0.f;
          own_t = false;
          trow = t_next;  // loaded one item ahead, so its latency is hidden
          const int64_t nrow = single ? item + ncl : (item + ncl) * R + g;
          t_next = nrow < M ? __ldg(a.target + nrow) : -1;
        }
        if (trow >= 0 && trow < N) {  // capture x[target] if it is in this thread's vectors
          const int64_t tl = trow / E - cbase;  // target vector, relative to the slot
          if (tl >= 0 && tl < cn && int(tl) % TPR == l) {
            // One element read from the slot (still held until the barrier
            // below), rather than a select over every element in registers.
            xt = V::load1(sb + tl * 16 + (trow % E) * int64_t(sizeof(T)));
            own_t = true;
          }
        }
      }
      // Streamed pairs start from the running maximum, so a chunk with no
      // elements for this thread leaves the pair unchanged.
      float m = (OP == kXent || TWO_PASS) ? run_m : kNegInf;
      // Cross-entropy: the maximum as a tree and four independent accumulator
      // pairs (short dependency chains).  Softmax keeps one chain of each: it
      // also holds the exponentials for the finish, and the extra registers
      // would cost a resident CTA.
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
          const float2 ev = make_float2(exp2_approx(t.x), exp2_approx(t.y));  // padding: 2^-inf = 0
          if constexpr (OP == kSoftmax && kKeepExp && !TWO_PASS) {
            ef[k * E + e] = ev.x;
            ef[k * E + e + 1] = ev.y;
          }
          const int c = kShortChains ? ((k * E + e) / 2) & 3 : 0;
          a4[c] = add2(a4[c], ev);
        }
      }
      const float2 acc =
          kShortChains ? add2(add2(a4[0], a4[1]), add2(a4[2], a4[3])) : a4[0];
      if constexpr (OP == kSoftmax && !TWO_PASS) {
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
    const bool row_end = (j == K - 1);  // the row's reduction is complete (first pass)
    if (row_end) {
      if constexpr (OP == kLayerNorm) {
        if (ln_full) {  // the same for every row group of the launch
          group_welford_sum<GW, E * VPT>(pm, ps);
        } else {
          group_welford<GW>(pn, pm, ps);
        }
        // Streamed rows: the counts of the warps no longer follow from the
        // geometry of one slot, so they travel through shared memory.
        if (TWO_PASS && WPG > 1 && lane == 0) cnt_red[ibit * 16 + warp] = pn;
      } else {
        warp_reduce<OP, GW>(pm, ps);
      }
      if (WPG > 1 && lane == 0) red[ibit * 16 + warp] = make_float2(pm, ps);
    }
    // One barrier per step: the slot is free again (every thread has its data
    // in registers) and the warp partials are visible.  It also carries a
    // failed wait to the whole CTA so that everyone leaves together.
    if (__syncthreads_or(failed)) {
      abort = true;
      break;
    }
    if (tid == 0 && p_left > 0) issue_next();
    // advance the consumer position to step q + 1
    const uint32_t row_ibit = ibit, row_xphase = xphase;
    if (++slot == S) {
      slot = 0;
      phase ^= 1u;
    }
    if (row_end) {
      xphase ^= ibit;  // the cluster barrier of buffer b flips every second item
      ibit ^= 1u;
    }
    if (j == KK - 1) {
      j = 0;
      item += ncl;
    } else {
      ++j;
    }
    if (!row_end) {
      if constexpr (TWO_PASS) {
        if (second && row_ok) {  // write this chunk's outputs with the row's totals
          uint4* yg = static_cast<uint4*>(a.y) + row * NV + cbase;
          const uint4* wg2 = static_cast<const uint4*>(a.w) + cbase;
#pragma unroll
          for (int k = 0; k < VPT; ++k) {
            if (!valid[k]) continue;
            float f[E], o[E];
            V::unpack_fresh(xr[k], f);
            if constexpr (OP == kSoftmax) {  // exp(x - M) / S
#pragma unroll
              for (int e = 0; e < E; e += 2) {
                const float2 t = fma2(make_float2(f[e], f[e + 1]), make_float2(kLog2e, kLog2e),
                                      make_float2(-tot_a, -tot_a));
                const float2 v = mul2(make_float2(exp2_approx(t.x), exp2_approx(t.y)),
                                      make_float2(tot_b, tot_b));
                o[e] = v.x;
                o[e + 1] = v.y;
              }
            } else if constexpr (OP == kRmsNorm) {  // (x * rstd) * w
              float w[E];
              V::unpack(__ldg(wg2 + l + k * TPR), w);
#pragma unroll
              for (int e = 0; e < E; e += 2) {
                const float2 v = mul2(mul2(make_float2(f[e], f[e + 1]), make_float2(tot_a, tot_a)),
                                      make_float2(w[e], w[e + 1]));
                o[e] = v.x;
                o[e + 1] = v.y;
              }
            } else {  // LayerNorm: (x * rstd - mean * rstd) * w + b
              float w[E], bb[E];
              V::unpack(__ldg(wg2 + l + k * TPR), w);
              V::unpack(a.bias != nullptr ? __ldg(static_cast<const uint4*>(a.bias) + cbase + l + k * TPR)
                                          : make_uint4(0u, 0u, 0u, 0u),
                        bb);
#pragma unroll
              for (int e = 0; e < E; e += 2) {
                const float2 v = fma2(fma2(make_float2(f[e], f[e + 1]), make_float2(tot_a, tot_a),
                                           make_float2(tot_b, tot_b)),
                                      make_float2(w[e], w[e + 1]), make_float2(bb[e], bb[e + 1]));
                o[e] = v.x;
                o[e + 1] = v.y;
              }
            }
            __stcs(yg + l + k * TPR, V::pack(o));
          }
        }
      }
      continue;
    }

    // ---- block reduction over the warps of this row group ----
    if constexpr (OP == kLayerNorm) {
      // Every warp of the group merges the group's WPG warp partials with a
      // butterfly of width WPG (lane l takes partial l % WPG).
      if constexpr (WPG > 1) {
        const float2 v = red[row_ibit * 16 + g * WPG + lane % WPG];
        pm = v.x;
        ps = v.y;
        if (ln_full) {
          group_welford_sum<WPG, 32 * VPT * E>(pm, ps);
        } else {
          pn = TWO_PASS ? cnt_red[row_ibit * 16 + g * WPG + lane % WPG] : ln_wc;
          group_welford<WPG>(pn, pm, ps);
        }
      }
      if (ln_full) {  // back to (count, mean): the count is a power of two
        constexpr float kInvGroup = 1.f / float(TPR * VPT * E);
        pn = float(TPR * VPT * E);
        pm = pm * kInvGroup;
      }
    } else if constexpr (WPG > 1) {
      merge_partials<OP>(red + row_ibit * 16 + g * WPG, WPG, pm, ps);
    }

    // ---- cluster reduction: every CTA's partial into every peer (DSMEM) ----
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
      if constexpr (OP == kLayerNorm) {  // a butterfly over the C partials
        if (NV % C == 0 && (C & (C - 1)) == 0) {  // equal slices, C a power of two
          const float2 v = xbuf[b * kMaxCluster + (uint32_t(lane) & (C - 1))];
          pn = float(SV * E);
          pm = v.x;
          ps = v.y;
          switch (C) {
            case 2: group_welford_equal<2>(pn, pm, ps); break;
            case 4: group_welford_equal<4>(pn, pm, ps); break;
            case 8: group_welford_equal<8>(pn, pm, ps); break;
            case 16: group_welford_equal<16>(pn, pm, ps); break;
            default: break;  // C == 1: nothing to merge
          }
        } else {  // width 16; lanes beyond C hold count 0 and are neutral
          const uint32_t r = uint32_t(lane) & 15u;
          const float2 v = r < C ? xbuf[b * kMaxCluster + r] : make_float2(0.f, 0.f);
          pn = ln_cc;
          pm = v.x;
          ps = v.y;
          group_welford<16>(pn, pm, ps);
        }
      } else {
        merge_partials<OP>(xbuf + b * kMaxCluster, int(C), pm, ps);
      }
    }

    if constexpr (TWO_PASS) {  // keep the totals for the second pass
      if constexpr (OP == kSoftmax) {
        tot_a = (pm == kNegInf) ? 0.f : pm * kLog2e;  // M log2 e
        // 1 / S, NaN for a row with no finite entry (as softmax_scale)
        tot_b = (pm == kNegInf) ? __int_as_float(0x7fc00000) : __fdividef(1.f, ps);
      } else if constexpr (OP == kRmsNorm) {
        tot_a = rsqrtf(fmaf(ps, a.inv_n, a.eps));     // rstd
        if (l == 0 && rank == 0 && row_ok && a.rstd != nullptr) a.rstd[row] = tot_a;
      } else {                                        // LayerNorm
        tot_a = rsqrtf(fmaf(ps, a.inv_n, a.eps));     // rstd
        tot_b = -pm * tot_a;                          // -mean * rstd
        if (l == 0 && rank == 0 && row_ok) {
          if (a.rstd != nullptr) a.rstd[row] = tot_a;
          if (a.mean != nullptr) a.mean[row] = pm;
        }
      }
      continue;
    }

    // ---- finish: outputs from registers, each stored once ----
    // Output vectors go out as streaming stores (st.global.cs): nothing in the
    // launch reads them again, and lines marked evict-first leave L2 for HBM
    // ahead of the inputs still arriving (same-GPU A/B: RMSNorm bf16
    // 16384 x 4096 92.8 % -> 94.7 %, +1 to +3 points on most rows of 1024-16384
    // elements).  The backward and shifted kernels store the same way.
    if (!row_ok) continue;
    if constexpr (OP == kSoftmax) {
      const float scale = softmax_scale(tm, pm, ps);
      const float2 sc = make_float2(scale, scale);
      const float mb = (tm == kNegInf) ? 0.f : tm * kLog2e;
      uint4* yg = static_cast<uint4*>(a.y) + row * NV + cbase;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        if (!valid[k]) continue;
        float o[E];
        if constexpr (!kKeepExp) V::unpack_fresh(xr[k], o);
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          float2 ev;
          if constexpr (kKeepExp) {
            ev = make_float2(ef[k * E + e], ef[k * E + e + 1]);
          } else {  // same argument and rounding as in the reduction pass
            const float2 t = fma2(make_float2(o[e], o[e + 1]), make_float2(kLog2e, kLog2e),
                                  make_float2(-mb, -mb));
            ev = make_float2(exp2_approx(t.x), exp2_approx(t.y));
          }
          const float2 v = mul2(ev, sc);
          o[e] = v.x;
          o[e + 1] = v.y;
        }
        __stcs(yg + l + k * TPR, V::pack(o));
      }
    } else if constexpr (OP == kRmsNorm) {
      const float r = rsqrtf(fmaf(ps, a.inv_n, a.eps));  // 1/sqrt(mean of squares + eps)
      const float2 r2 = make_float2(r, r);
      uint4* yg = static_cast<uint4*>(a.y) + row * NV + cbase;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        if (!valid[k]) continue;
        float f[E], w[E], o[E];
        V::unpack_fresh(xr[k], f);
        if constexpr (kWeightInRegs) {
          V::unpack_fresh(wv[k], w);
        } else {
          V::unpack(__ldg(wg + l + k * TPR), w);
        }
#pragma unroll
        for (int e = 0; e < E; e += 2) {  // (x * rstd) * w, each product rounded once
          const float2 v = mul2(mul2(make_float2(f[e], f[e + 1]), r2), make_float2(w[e], w[e + 1]));
          o[e] = v.x;
          o[e + 1] = v.y;
        }
        __stcs(yg + l + k * TPR, V::pack(o));
      }
      if (l == 0 && rank == 0 && a.rstd != nullptr) a.rstd[row] = r;
    } else if constexpr (OP == kLayerNorm) {
      const float r = rsqrtf(fmaf(ps, a.inv_n, a.eps));  // 1/sqrt(population variance + eps)
      const float2 r2 = make_float2(r, r), c2 = make_float2(-pm * r, -pm * r);
      uint4* yg = static_cast<uint4*>(a.y) + row * NV + cbase;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        if (!valid[k]) continue;
        float f[E], w[E], bb[E], o[E];
        if constexpr (VPT <= 4) {
          V::unpack(xr[k], f);  // may reuse the unpacked values of the reduction
        } else {
          V::unpack_fresh(xr[k], f);  // only the packed input stays live across the reduction
        }
        if constexpr (kWeightInRegs) {
          V::unpack_fresh(wv[k], w);
        } else {
          V::unpack(wsm[l + k * TPR], w);
        }
        if constexpr (kBiasInRegs) {
          V::unpack_fresh(bv[k], bb);
        } else {
          V::unpack(bsm[l + k * TPR], bb);
        }
#pragma unroll
        for (int e = 0; e < E; e += 2) {  // (x * rstd - mean * rstd) * w + b
          const float2 v = fma2(fma2(make_float2(f[e], f[e + 1]), r2, c2),
                                make_float2(w[e], w[e + 1]), make_float2(bb[e], bb[e + 1]));
          o[e] = v.x;
          o[e + 1] = v.y;
        }
        __stcs(yg + l + k * TPR, V::pack(o));
      }
      if (l == 0 && rank == 0) {
        if (a.rstd != nullptr) a.rstd[row] = r;
        if (a.mean != nullptr) a.mean[row] = pm;
      }
    } else {
      const bool leader = (l == 0 && rank == 0);
      const bool ignored = a.has_ignore && trow == a.ignore_index;
      if (leader || own_t) {  // only the threads that write need the logarithm
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
    }
  }

  if (abort) {
    // Leave no bulk copy in flight into this CTA's shared memory: wait (bounded)
    // for every step issued but not consumed, from the current ring position on.
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
  if constexpr (CLUSTER) cluster_sync_all();  // no CTA leaves while peers may write to it
}

// ---------------------------------------------------------------------------
// Masked direct path: any N, any element-aligned pointers.  One row per CTA
// (or per cluster); cross-entropy streams its row through registers.
// ---------------------------------------------------------------------------
template <int OP, typename T, int THREADS, int EPT, bool CLUSTER>
__global__ void __launch_bounds__(THREADS) direct_kernel(const RowArgs a) {
  using V = Vec16<T>;
  constexpr int NW = THREADS / 32;
  constexpr int64_t CH = int64_t(THREADS) * EPT;
  __shared__ float2 red[NW];
  __shared__ float2 xbuf[kMaxCluster];
  __shared__ __align__(8) uint64_t xbar;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t C = 1, rank = 0;
  int64_t row = blockIdx.x;
  if constexpr (CLUSTER) {
    C = cluster_nctarank();
    rank = cluster_ctarank();
    row = cluster_id_x();
  }
  const int64_t N = a.N;
  const int64_t SE = (N + C - 1) / C;
  const int64_t e0 = min(N, int64_t(rank) * SE);
  const int64_t ne = min(N, e0 + SE) - e0;
  const uint32_t xb = smem_addr(&xbar);
  if constexpr (CLUSTER) {
    if (tid == 0) {
      mbar_init(xb, 1);
      fence_mbar_init();
    }
    cluster_sync_all();
  }
  grid_dependency_wait();
  allow_dependent_launch();

  const T* xrow = static_cast<const T*>(a.x) + row * N + e0;
  float f[EPT];
  float pm = kNegInf, ps = 0.f, tm = kNegInf, xt = 0.f;
  float pn = 0.f;  // LayerNorm: element count of the partial (mean pm, M2 ps)
  bool own_t = false;
  const int64_t trow = (OP == kXent) ? a.target[row] : -1;

  for (int64_t c0 = 0; c0 < ne; c0 += CH) {  // more than one pass only for cross-entropy
#pragma unroll
    for (int k = 0; k < EPT; ++k) {
      const int64_t e = c0 + tid + int64_t(k) * THREADS;
      f[k] = e < ne ? V::load1(xrow + e) : ((OP == kRmsNorm || OP == kLayerNorm) ? 0.f : kNegInf);
    }
    if constexpr (OP == kLayerNorm) {  // one chunk: the row slice fits the registers
      float sum = 0.f;
      int cnt = 0;
#pragma unroll
      for (int k = 0; k < EPT; ++k) {
        const bool in = c0 + tid + int64_t(k) * THREADS < ne;
        sum += f[k];  // padding is 0
        cnt += in ? 1 : 0;
      }
      pn = float(cnt);
      pm = cnt > 0 ? __fdiv_rn(sum, pn) : 0.f;
      ps = 0.f;
#pragma unroll
      for (int k = 0; k < EPT; ++k) {
        const float d = f[k] - pm;
        if (c0 + tid + int64_t(k) * THREADS < ne) ps = fmaf(d, d, ps);
      }
    } else if constexpr (OP == kRmsNorm) {
#pragma unroll
      for (int k = 0; k < EPT; ++k) ps = fmaf(f[k], f[k], ps);
    } else {
      float m = pm;
#pragma unroll
      for (int k = 0; k < EPT; ++k) m = fmaxf(m, f[k]);
      if (m != kNegInf) {
        ps *= exp2_approx((pm - m) * kLog2e);
        const float mb = m * kLog2e;
#pragma unroll
        for (int k = 0; k < EPT; ++k) {
          const float v = exp2_approx(fmaf(f[k], kLog2e, -mb));  // masked: exp2(-inf) = 0
          if constexpr (OP == kSoftmax) f[k] = v;
          ps += v;
        }
        pm = m;
      }
      tm = pm;
      if constexpr (OP == kXent) {
#pragma unroll
        for (int k = 0; k < EPT; ++k) {
          const int64_t e = c0 + tid + int64_t(k) * THREADS;  // padding lanes never match
          if (e < ne && e0 + e == trow) {
            xt = f[k];
            own_t = true;
          }
        }
      }
    }
  }

  if constexpr (OP == kLayerNorm) {
    group_welford<32>(pn, pm, ps);
  } else {
    warp_reduce<OP>(pm, ps);
  }
  if (lane == 0) red[warp] = make_float2(pm, ps);
  __syncthreads();
  if constexpr (OP == kLayerNorm) {  // warp w holds elements w*32 .. w*32+31 of each chunk column
    auto warp_count = [&](int w) {
      int64_t c = 0;
#pragma unroll
      for (int k = 0; k < EPT; ++k)
        c += max(int64_t(0), min(int64_t(32), ne - int64_t(k) * THREADS - int64_t(w) * 32));
      return float(c);
    };
    pn = warp_count(0);
    pm = red[0].x;
    ps = red[0].y;
    for (int w = 1; w < NW; ++w) welford_merge(pn, pm, ps, warp_count(w), red[w].x, red[w].y);
  } else {
    merge_partials<OP>(red, NW, pm, ps);
  }
  if constexpr (CLUSTER) {
    if (tid == 0) {
      mbar_arrive_expect_tx(xb, C * 8u);
      const uint32_t mine = smem_addr(&xbuf[rank]);
      for (uint32_t r = 0; r < C; ++r) st_async_f2(map_to_rank(mine, r), pm, ps, map_to_rank(xb, r));
    }
    if (!mbar_wait<true>(xb, 0u, a.timeout_ns)) report_status(a.status, kStatusTimeout);
    if constexpr (OP == kLayerNorm) {  // CTA r holds the ne_r elements of its slice
      auto cta_count = [&](uint32_t r) {
        const int64_t s0 = min(N, int64_t(r) * SE);
        return float(min(N, s0 + SE) - s0);
      };
      pn = cta_count(0);
      pm = xbuf[0].x;
      ps = xbuf[0].y;
      for (uint32_t r = 1; r < C; ++r) welford_merge(pn, pm, ps, cta_count(r), xbuf[r].x, xbuf[r].y);
    } else {
      merge_partials<OP>(xbuf, int(C), pm, ps);
    }
  }

  if constexpr (OP == kSoftmax) {
    const float scale = softmax_scale(tm, pm, ps);
    T* yrow = static_cast<T*>(a.y) + row * N + e0;
#pragma unroll
    for (int k = 0; k < EPT; ++k) {
      const int64_t e = tid + int64_t(k) * THREADS;
      if (e < ne) V::store1(yrow + e, f[k] * scale);
    }
  } else if constexpr (OP == kRmsNorm) {
    const float r = rsqrtf(fmaf(ps, a.inv_n, a.eps));  // 1/sqrt(mean of squares + eps)
    T* yrow = static_cast<T*>(a.y) + row * N + e0;
    const T* wrow = static_cast<const T*>(a.w) + e0;
#pragma unroll
    for (int k = 0; k < EPT; ++k) {
      const int64_t e = tid + int64_t(k) * THREADS;
      if (e < ne) V::store1(yrow + e, __fmul_rn(__fmul_rn(f[k], r), V::load1(wrow + e)));
    }
    if (tid == 0 && rank == 0 && a.rstd != nullptr) a.rstd[row] = r;
  } else if constexpr (OP == kLayerNorm) {
    const float r = rsqrtf(fmaf(ps, a.inv_n, a.eps));  // 1/sqrt(population variance + eps)
    T* yrow = static_cast<T*>(a.y) + row * N + e0;
    const T* wrow = static_cast<const T*>(a.w) + e0;
    const T* brow = static_cast<const T*>(a.bias) + e0;  // unused when bias is null
#pragma unroll
    for (int k = 0; k < EPT; ++k) {
      const int64_t e = tid + int64_t(k) * THREADS;
      if (e < ne) {
        const float b = a.bias != nullptr ? V::load1(brow + e) : 0.f;
        V::store1(yrow + e, fmaf(__fmul_rn(__fsub_rn(f[k], pm), r), V::load1(wrow + e), b));
      }
    }
    if (tid == 0 && rank == 0) {
      if (a.rstd != nullptr) a.rstd[row] = r;
      if (a.mean != nullptr) a.mean[row] = pm;
    }
  } else {
    const float lse = pm + logf(ps);
    const bool ignored = a.has_ignore && trow == a.ignore_index;
    if (tid == 0 && rank == 0) {
      if (a.lse != nullptr) a.lse[row] = lse;
      if (ignored) {
        a.loss[row] = 0.f;
      } else if (!(trow >= 0 && trow < N)) {
        a.loss[row] = __int_as_float(0x7fc00000);
      }
    }
    if (own_t && !ignored) a.loss[row] = fmaf(a.z_loss * lse, lse, lse - xt);
  }
  if constexpr (CLUSTER) cluster_sync_all();
}

// Mean of the per-row losses over the rows not ignored (with has_ignore, those
// whose target is not ignore_index; NaN when there are none): one CTA, each thread summing a fixed strided
// subset in order, then a fixed-shape tree -- deterministic.
template <int kUnused = 0>
__global__ void __launch_bounds__(1024) xent_mean_kernel(const float* __restrict__ loss,
                                                         const int64_t* __restrict__ target,
                                                         int64_t M, int has_ignore,
                                                         int64_t ignore_index,
                                                         float* __restrict__ mean) {
  __shared__ float ssum[1024];
  __shared__ int64_t scnt[1024];
  grid_dependency_wait();
  allow_dependent_launch();
  const int tid = threadIdx.x;
  float acc = 0.f;
  int64_t cnt = 0;
  for (int64_t i = tid; i < M; i += 1024) {
    if (!(has_ignore && target[i] == ignore_index)) {
      acc += loss[i];
      ++cnt;
    }
  }
  ssum[tid] = acc;
  scnt[tid] = cnt;
  __syncthreads();
  for (int s = 512; s > 0; s >>= 1) {
    if (tid < s) {
      ssum[tid] += ssum[tid + s];
      scnt[tid] += scnt[tid + s];
    }
    __syncthreads();
  }
  if (tid == 0) *mean = ssum[0] / float(scnt[0]);  // 0 / 0 = NaN when every row is ignored
}

}  // namespace qk
