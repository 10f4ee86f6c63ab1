// qk_device.cuh -- device primitives for the sm_103a row-reduction kernels.
//
// Hand-written inline PTX (public PTX ISA) for:
//   * mbarriers with expect-tx byte counting and bounded parity waits,
//   * bulk (non-tensor) TMA copies global -> shared, completing on an mbarrier,
//   * thread-block-cluster addressing (mapa) and st.async into a peer CTA's
//     shared memory that completes on the peer's mbarrier,
//   * 16-byte vector packing for fp32 / bf16 rows,
//   * the reduction operators: sum, and the (max, sum-of-exponentials) pair
//     of an online softmax.
//
// The reduction hierarchy (thread -> warp shuffle -> block shared memory ->
// cluster DSMEM) follows the QbitAI article on QuACK, section
// "硬件感知的归约策略" (hardware-aware reduction), parts 1-4.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace qk {

constexpr float kLog2e = 1.4426950408889634f;  // log2(e): exp(x) = 2^(x * log2 e)
constexpr float kNegInf = -__builtin_huge_valf();

// ---------------------------------------------------------------------------
// Shared-memory addressing and special registers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t num_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
// Makes initialised barriers visible to the async proxy and to peer CTAs.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
// Acquire at cluster scope: for data that peer CTAs wrote with st.async.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for the phase with the given parity to complete, giving up after
// timeout_ns nanoseconds of the global timer.  Returns false on time-out; the
// caller records the failure and leaves its loop, so no wait is unbounded.
template <bool kClusterScope>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
  auto poll = [&]() {
    return kClusterScope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
  };
  if (poll()) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (poll()) return true;
    if (global_timer_ns() - t0 > timeout_ns) return false;
  }
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialisation may start while the previous kernel in the stream is still
// running; grid_dependency_wait() blocks until that kernel has completed and
// its writes are visible, so it must precede the first global-memory access.
// allow_dependent_launch() lets the next kernel in the stream start early
// (it takes effect once every CTA of this grid has issued it or exited).
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// First error wins; later ones are dropped.
__device__ __forceinline__ void report_status(int* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------------------
// Bulk TMA copy global -> shared (non-tensor form: contiguous bytes)
// ---------------------------------------------------------------------------
// L2 policy for data read exactly once: evict it first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// dst, bar: shared addresses of this CTA; src: global, 16-byte aligned;
// bytes: a multiple of 16.  Completion adds `bytes` to bar's tx count.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Hint: pull [src, src + bytes) from HBM into L2 (both 16-byte multiples).
// It returns nothing to the SM, so it may be issued before the kernel that
// writes those bytes has finished: L2 is where every write lands, and the
// copies into shared memory that read the data later come after the wait.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------------------
// Thread-block cluster / DSMEM
// ---------------------------------------------------------------------------
// Address of the same shared-memory object in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// 8-byte store into a (possibly remote) CTA's shared memory; completes by
// adding 8 bytes to the tx count of the mbarrier `rbar` in that same CTA.
__device__ __forceinline__ void st_async_f2(uint32_t raddr, float a, float b, uint32_t rbar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(
          raddr),
      "f"(a), "f"(b), "r"(rbar)
      : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

// ---------------------------------------------------------------------------
// Arithmetic
// ---------------------------------------------------------------------------
// 2^x with the SFU's approximate base-2 exponential (PTX ex2.approx.ftz.f32).
__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed pairs of fp32 (sm_100+ f32x2 forms): two IEEE round-to-nearest
// results per instruction, bit-identical to the scalar operations.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
// Element-wise maximum of two packed bf16 pairs (exact; NaN loses to a number).
__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Butterfly (xor) reductions over groups of WIDTH consecutive lanes (WIDTH a
// power of two <= 32): after the loop every lane holds its group's result.
// Addition is commutative in IEEE arithmetic, so both lanes of each step
// compute the same value and all lanes of a group agree bit for bit.
template <int WIDTH = 32>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = WIDTH / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
template <int WIDTH = 32>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int o = WIDTH / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
// Reduces online-softmax pairs over the group: the maximum first, then each
// lane rescales its own sum to it once, then a plain sum.  One SFU op per lane
// instead of two per butterfly step.
template <int WIDTH = 32>
__device__ __forceinline__ void group_ms(float& m, float& s) {
  const float mg = group_max<WIDTH>(m);
  const float sl = (m == kNegInf) ? 0.f : s * exp2_approx((m - mg) * kLog2e);
  s = group_sum<WIDTH>(sl);
  m = mg;
}

// (count, mean, M2) of a set of values, merged pairwise (the parallel form of
// Welford's update, Chan et al.): with a the side with more values and
// d = mean_b - mean_a,
//   n = n_a + n_b,  mean = mean_a + d n_b / n,  M2 = M2_a + M2_b + d^2 n_a n_b / n.
// With equal counts this is mean = (mean_a + mean_b) / 2 and
// M2 = M2_a + M2_b + d^2 n_a / 2, which needs no division; otherwise 1/n is
// one approximate reciprocal (a relative error of an ulp or two in the update
// terms).  Both forms leave the mean exact when the two means are equal.
// Every product and sum is rounded explicitly and the result does not depend
// on the argument order, so merge(a, b) == merge(b, a) bit for bit (butterfly
// lanes agree).  An empty side leaves the other one unchanged.
__device__ __forceinline__ void welford_merge_equal(float& mean, float& m2, float n, float mean2,
                                                    float m22) {
  const float d = __fsub_rn(mean2, mean);
  mean = __fmul_rn(__fadd_rn(mean, mean2), 0.5f);
  m2 = __fadd_rn(__fadd_rn(m2, m22), __fmul_rn(__fmul_rn(d, d), __fmul_rn(n, 0.5f)));
}
__device__ __forceinline__ void welford_merge(float& n, float& mean, float& m2, float n2,
                                              float mean2, float m22) {
  if (n2 == 0.f) return;
  if (n == 0.f) {
    n = n2;
    mean = mean2;
    m2 = m22;
    return;
  }
  if (n == n2) {
    welford_merge_equal(mean, m2, n, mean2, m22);
    n = __fadd_rn(n, n);
    return;
  }
  const bool a_first = n > n2;  // the same choice from either side
  const float na = a_first ? n : n2, ma = a_first ? mean : mean2;
  const float nb = a_first ? n2 : n, mb = a_first ? mean2 : mean;
  const float nt = __fadd_rn(na, nb);
  const float rn = __fdividef(1.f, nt);
  const float d = __fsub_rn(mb, ma);
  mean = __fadd_rn(ma, __fmul_rn(d, __fmul_rn(nb, rn)));
  m2 = __fadd_rn(__fadd_rn(m2, m22), __fmul_rn(__fmul_rn(d, d), __fmul_rn(__fmul_rn(na, nb), rn)));
  n = nt;
}
// Butterfly over WIDTH lanes (a power of two): every lane ends with the merge
// of all WIDTH partials.  Lanes with n = 0 are neutral.
template <int WIDTH = 32>
__device__ __forceinline__ void group_welford(float& n, float& mean, float& m2) {
#pragma unroll
  for (int o = WIDTH / 2; o > 0; o >>= 1) {
    const float n2 = __shfl_xor_sync(0xffffffffu, n, o);
    const float mean2 = __shfl_xor_sync(0xffffffffu, mean, o);
    const float m22 = __shfl_xor_sync(0xffffffffu, m2, o);
    welford_merge(n, mean, m2, n2, mean2, m22);
  }
}
// Sum form of the equal-count butterfly, for counts that are powers of two:
// lanes carry (S = n mean, M2) and each side of a merge holds n values, so
//   S = S_a + S_b,  M2 = M2_a + M2_b + (S_b - S_a)^2 / (2 n),
// which is the equal-count merge above scaled by n (exact for a power of
// two).  N0 is every lane's count before the first level; 1/(2n) folds to a
// constant at each level.
template <int WIDTH, int N0>
__device__ __forceinline__ void group_welford_sum(float& s, float& m2) {
#pragma unroll
  for (int o = WIDTH / 2, n = N0; o > 0; o >>= 1, n *= 2) {
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const float q2 = __shfl_xor_sync(0xffffffffu, m2, o);
    const float d = __fsub_rn(s2, s);
    s = __fadd_rn(s, s2);
    m2 = __fmaf_rn(__fmul_rn(d, d), 0.5f / float(n), __fadd_rn(m2, q2));
  }
}
// The same when every lane's count is n (it doubles at each level): no
// counts travel and no branch is taken.
template <int WIDTH = 32>
__device__ __forceinline__ void group_welford_equal(float& n, float& mean, float& m2) {
#pragma unroll
  for (int o = WIDTH / 2; o > 0; o >>= 1) {
    const float mean2 = __shfl_xor_sync(0xffffffffu, mean, o);
    const float m22 = __shfl_xor_sync(0xffffffffu, m2, o);
    welford_merge_equal(mean, m2, n, mean2, m22);
    n = __fadd_rn(n, n);
  }
}

// ---------------------------------------------------------------------------
// 16-byte vectors of fp32 (4 elements) or bf16 (8 elements)
// ---------------------------------------------------------------------------
template <typename T>
struct Vec16;

template <>
struct Vec16<float> {
  static constexpr int kElems = 4;
  __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  __device__ __forceinline__ static void unpack_fresh(const uint4& v, float* f) { unpack(v, f); }
  // Bit pattern of -inf in every element: the neutral value of a maximum.
  static constexpr uint32_t kNegInfBits = 0xff800000u;
  // Running maximum over the four elements of v.
  __device__ __forceinline__ static float max_into(float m, const uint4& v) {
    return fmaxf(fmaxf(m, fmaxf(__uint_as_float(v.x), __uint_as_float(v.y))),
                 fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
  }
  // Maximum over the elements of n vectors as a pairwise tree: depth
  // log2(4n) instead of a chain of 4n comparisons.
  template <int NV>
  __device__ __forceinline__ static float max_all(const uint4* v) {
    float t[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k)
      t[k] = fmaxf(fmaxf(__uint_as_float(v[k].x), __uint_as_float(v[k].y)),
                   fmaxf(__uint_as_float(v[k].z), __uint_as_float(v[k].w)));
#pragma unroll
    for (int s = 1; s < NV; s *= 2)
#pragma unroll
      for (int k = 0; k + s < NV; k += 2 * s) t[k] = fmaxf(t[k], t[k + s]);
    return t[0];
  }
  __device__ __forceinline__ static uint4 pack(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
  __device__ __forceinline__ static float load1(const void* p) {
    return *static_cast<const float*>(p);
  }
  __device__ __forceinline__ static void store1(void* p, float v) { *static_cast<float*>(p) = v; }
  // v with the elements outside [lo, hi) replaced by the element with bits fill.
  __device__ __forceinline__ static uint4 keep(uint4 v, int lo, int hi, uint32_t fill) {
    return make_uint4(0 >= lo && 0 < hi ? v.x : fill, 1 >= lo && 1 < hi ? v.y : fill,
                      2 >= lo && 2 < hi ? v.z : fill, 3 >= lo && 3 < hi ? v.w : fill);
  }
};

template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int kElems = 8;
  // bf16 -> fp32 is exact: the 16 bits become the high half of the float.
  __device__ __forceinline__ static void unpack2(uint32_t u, float& lo, float& hi) {
    lo = __uint_as_float(u << 16);
    hi = __uint_as_float(u & 0xffff0000u);
  }
  __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
    unpack2(v.x, f[0], f[1]);
    unpack2(v.y, f[2], f[3]);
    unpack2(v.z, f[4], f[5]);
    unpack2(v.w, f[6], f[7]);
  }
  static constexpr uint32_t kNegInfBits = 0xff80ff80u;
  // Running maximum over the eight elements of v, compared as packed bf16
  // pairs (exact), widened once at the end.
  __device__ __forceinline__ static float max_into(float m, const uint4& v) {
    const uint32_t p = max_bf16x2(max_bf16x2(v.x, v.y), max_bf16x2(v.z, v.w));
    float lo, hi;
    unpack2(p, lo, hi);
    return fmaxf(m, fmaxf(lo, hi));
  }
  // Maximum over the elements of n vectors: a pairwise tree of packed bf16
  // comparisons (exact), widened once at the end.
  template <int NV>
  __device__ __forceinline__ static float max_all(const uint4* v) {
    uint32_t t[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k)
      t[k] = max_bf16x2(max_bf16x2(v[k].x, v[k].y), max_bf16x2(v[k].z, v[k].w));
#pragma unroll
    for (int s = 1; s < NV; s *= 2)
#pragma unroll
      for (int k = 0; k + s < NV; k += 2 * s) t[k] = max_bf16x2(t[k], t[k + s]);
    float lo, hi;
    unpack2(t[0], lo, hi);
    return fmaxf(lo, hi);
  }
  // Same as unpack, but opaque to the optimiser: it cannot be hoisted out of
  // a loop or merged with an earlier unpack, so the packed form (half the
  // registers) is what stays live between the reduction and the finish.
  __device__ __forceinline__ static void unpack_fresh(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t lo, hi;
      asm volatile("shl.b32 %0, %1, 16;" : "=r"(lo) : "r"(w[i]));
      asm volatile("and.b32 %0, %1, 0xffff0000;" : "=r"(hi) : "r"(w[i]));
      f[2 * i] = __uint_as_float(lo);
      f[2 * i + 1] = __uint_as_float(hi);
    }
  }
  __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // round to nearest even
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  __device__ __forceinline__ static uint4 pack(const float* f) {
    return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
  }
  __device__ __forceinline__ static float load1(const void* p) {
    const uint16_t b = *static_cast<const uint16_t*>(p);
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
  __device__ __forceinline__ static void store1(void* p, float v) {
    *static_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(v);
  }
  // v with the elements outside [lo, hi) replaced by the element with bits
  // fill (both halves of fill hold that element).
  __device__ __forceinline__ static uint32_t keep2(uint32_t u, int e, int lo, int hi, uint32_t fill) {
    const uint32_t mlo = (e >= lo && e < hi) ? 0x0000ffffu : 0u;
    const uint32_t mhi = (e + 1 >= lo && e + 1 < hi) ? 0xffff0000u : 0u;
    const uint32_t m = mlo | mhi;
    return (u & m) | (fill & ~m);
  }
  __device__ __forceinline__ static uint4 keep(uint4 v, int lo, int hi, uint32_t fill) {
    return make_uint4(keep2(v.x, 0, lo, hi, fill), keep2(v.y, 2, lo, hi, fill),
                      keep2(v.z, 4, lo, hi, fill), keep2(v.w, 6, lo, hi, fill));
  }
};

}  // namespace qk
