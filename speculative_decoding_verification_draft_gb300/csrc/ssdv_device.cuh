// ssdv_device.cuh -- device building blocks shared by the verification and
// Saguaro kernels: inline-PTX wrappers (mbarrier, bulk async copy, cluster
// barrier, distributed shared memory), the Philox4x32-10 generator, row
// staging into shared memory, the fused softmax-statistics pass, the weighted
// pass with per-warp partial sums, and the inverse-CDF search.
//
// Work decomposition: one thread-block cluster per (request, position) unit.
// CTA `rank` of the cluster owns the contiguous vocabulary slice
// [rank * slice, rank * slice + n) of the unit's rows and keeps it resident in
// its shared memory, so every logit is read from HBM exactly once; the
// second and later passes (residual, Saguaro mix, CDF search) run on-chip.
#pragma once

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "ssdv_internal.h"

namespace ssdv {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kVecPerThreadStage = 2;
constexpr int kStageBytes = kThreads * kVecPerThreadStage * 16;  // 8 KB per row per stage
constexpr int kMaxStages = 32;
constexpr uint32_t kWaitLimit = 1u << 24;  // bounded polls of an mbarrier
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// 2^x as one ex2.approx.ftz.f32 instruction (relative error about 2 ulp;
// results below 2^-126 flush to zero, which no sum here can notice).  Every
// weight and every partial sum of a row uses this same function.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// Packed pairs of fp32 (one FMA / ADD instruction for two lanes of data).
// ---------------------------------------------------------------------------
struct F2 {
  unsigned long long v;
};
__device__ __forceinline__ F2 f2_make(float lo, float hi) {
  F2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(F2 a, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a.v));
}
__device__ __forceinline__ F2 f2_fma(F2 a, F2 b, F2 c) {
  F2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
  return r;
}
__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
  F2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}

// ---------------------------------------------------------------------------
// Element types: bf16 is handled as its raw 16-bit pattern.
// ---------------------------------------------------------------------------
template <typename E>
struct Elem;
template <>
struct Elem<uint16_t> {
  static constexpr int kVec = 8;  // elements per 16-byte vector
  // exp2(x * c - mc) summed over a raw vector, as a packed pair of partial sums
  static __device__ __forceinline__ F2 exp_sum(const uint4& v, F2 c2, F2 nmc2);
  // running maximum of raw vectors, two bf16 lanes per word (max.bf16x2 is
  // exact: it only selects one of its inputs)
  static __device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
  static __device__ __forceinline__ uint4 max_init() { return make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u); }
  static __device__ __forceinline__ uint4 max_acc(uint4 acc, const uint4& v) {
    return make_uint4(bmax2(acc.x, v.x), bmax2(acc.y, v.y), bmax2(acc.z, v.z), bmax2(acc.w, v.w));
  }
  static __device__ __forceinline__ float max_final(const uint4& acc) {
    const uint32_t m = bmax2(bmax2(acc.x, acc.y), bmax2(acc.z, acc.w));
    return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
  }
  static __device__ __forceinline__ float to_float(uint16_t h) {
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
  }
  static __device__ __forceinline__ uint16_t neg_inf() { return 0xFF80u; }
  static __device__ __forceinline__ void unpack(const uint4& v, float (&f)[8]) {
    f[0] = __uint_as_float(v.x << 16);
    f[1] = __uint_as_float(v.x & 0xFFFF0000u);
    f[2] = __uint_as_float(v.y << 16);
    f[3] = __uint_as_float(v.y & 0xFFFF0000u);
    f[4] = __uint_as_float(v.z << 16);
    f[5] = __uint_as_float(v.z & 0xFFFF0000u);
    f[6] = __uint_as_float(v.w << 16);
    f[7] = __uint_as_float(v.w & 0xFFFF0000u);
  }
};
template <>
struct Elem<float> {
  static constexpr int kVec = 4;
  // exp2(x * c - mc) summed over a raw vector, as a packed pair of partial sums
  static __device__ __forceinline__ F2 exp_sum(const uint4& v, F2 c2, F2 nmc2);
  // running maximum of raw vectors (kept as four floats)
  static __device__ __forceinline__ uint4 max_init() {
    const uint32_t n = __float_as_uint(-INFINITY);
    return make_uint4(n, n, n, n);
  }
  static __device__ __forceinline__ uint4 max_acc(uint4 acc, const uint4& v) {
    return make_uint4(__float_as_uint(fmaxf(__uint_as_float(acc.x), __uint_as_float(v.x))),
                      __float_as_uint(fmaxf(__uint_as_float(acc.y), __uint_as_float(v.y))),
                      __float_as_uint(fmaxf(__uint_as_float(acc.z), __uint_as_float(v.z))),
                      __float_as_uint(fmaxf(__uint_as_float(acc.w), __uint_as_float(v.w))));
  }
  static __device__ __forceinline__ float max_final(const uint4& acc) {
    return fmaxf(fmaxf(__uint_as_float(acc.x), __uint_as_float(acc.y)),
                 fmaxf(__uint_as_float(acc.z), __uint_as_float(acc.w)));
  }
  static __device__ __forceinline__ float to_float(float x) { return x; }
  static __device__ __forceinline__ float neg_inf() { return -INFINITY; }
  static __device__ __forceinline__ void unpack(const uint4& v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
};

__device__ __forceinline__ F2 f2_exp2(F2 a) {
  float lo, hi;
  f2_split(a, lo, hi);
  return f2_make(fast_exp2(lo), fast_exp2(hi));
}
__device__ __forceinline__ F2 Elem<uint16_t>::exp_sum(const uint4& v, F2 c2, F2 nmc2) {
  const F2 a = f2_exp2(f2_fma(f2_make(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u)), c2, nmc2));
  const F2 b = f2_exp2(f2_fma(f2_make(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u)), c2, nmc2));
  const F2 d = f2_exp2(f2_fma(f2_make(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xFFFF0000u)), c2, nmc2));
  const F2 e = f2_exp2(f2_fma(f2_make(__uint_as_float(v.w << 16), __uint_as_float(v.w & 0xFFFF0000u)), c2, nmc2));
  return f2_add(f2_add(a, b), f2_add(d, e));
}
__device__ __forceinline__ F2 Elem<float>::exp_sum(const uint4& v, F2 c2, F2 nmc2) {
  const F2 a = f2_exp2(f2_fma(f2_make(__uint_as_float(v.x), __uint_as_float(v.y)), c2, nmc2));
  const F2 b = f2_exp2(f2_fma(f2_make(__uint_as_float(v.z), __uint_as_float(v.w)), c2, nmc2));
  return f2_add(a, b);
}

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait for phase `parity` of an mbarrier; false if the bound ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  for (uint32_t it = 0; it < kWaitLimit; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Bulk asynchronous copy global -> this CTA's shared memory, completing on an
// mbarrier.  dst, src 16-byte aligned; bytes a positive multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Split cluster barrier (all threads of every CTA execute both halves).
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Asynchronous stores into another CTA's shared memory that complete on that
// CTA's mbarrier (remote addresses from mapa).
__device__ __forceinline__ void st_async_v4(uint32_t remote, float4 v, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   remote),
               "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(remote_bar)
               : "memory");
}
__device__ __forceinline__ void st_async_b64(uint32_t remote, unsigned long long v, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b64 [%0], %1, [%2];" ::"r"(remote), "l"(v),
               "r"(remote_bar)
               : "memory");
}

// Wait (bounded) for phase 0 of a barrier completed by other CTAs' st.async.
__device__ __forceinline__ bool xbar_wait_bounded(uint64_t* bar) {
  for (uint32_t it = 0; it < kWaitLimit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], 0;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar))
        : "memory");
    if (done) return true;
  }
  return false;
}

// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void* local, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_addr(local)), "r"(rank));
  return out;
}
__device__ __forceinline__ float dsmem_ld_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ double dsmem_ld_f64(uint32_t a) {
  double v;
  asm volatile("ld.shared::cluster.f64 %0, [%1];" : "=d"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ int dsmem_ld_s32(uint32_t a) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}

__device__ __forceinline__ int ld_volatile(const int32_t* p) { return *reinterpret_cast<const volatile int32_t*>(p); }

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11).  Key = (seed lo, seed hi),
// counter = (request, position, 0, 0).  Word d is the uniform of draw d.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t a0 = 0xD2511F53u * c.x, h0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t a1 = 0xCD9E8D57u * c.z, h1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(h1 ^ c.y ^ k0, a1, h0 ^ c.w ^ k1, a0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

__device__ __forceinline__ float word_to_uniform(uint32_t w) { return static_cast<float>(w >> 8) * 0x1p-24f; }

struct Draws {
  float accept, resample, saguaro;
};
__device__ __forceinline__ Draws unit_draws(uint64_t seed, int b, int i) {
  const uint4 w = philox4x32_10(make_uint4(static_cast<uint32_t>(b), static_cast<uint32_t>(i), 0u, 0u),
                                static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
  return Draws{word_to_uniform(w.x), word_to_uniform(w.y), word_to_uniform(w.z)};
}

// ---------------------------------------------------------------------------
// Softmax statistics: (m, s) with s = sum exp2(x*c - fl(m*c)), c = log2(e)/T.
// Partial pairs combine exactly as the terms were formed, so the combined s
// equals sum exp2(x*c - fl(M*c)) up to rounding.
// ---------------------------------------------------------------------------
struct MaxSum {
  float m, s;
};
// fl(m * c) without contraction into a neighbouring add: every term and every
// rescale factor of a row uses this same rounded product.
__device__ __forceinline__ float scaled_max(float m, float c) { return __fmul_rn(m, c); }
// exp2(fl(m_from*c) - fl(m_to*c)): moves a partial sum from one reference max to another.
__device__ __forceinline__ float rescale(float m_from, float m_to, float c) {
  return fast_exp2(__fsub_rn(scaled_max(m_from, c), scaled_max(m_to, c)));
}
__device__ __forceinline__ MaxSum combine_ms(MaxSum a, MaxSum b, float c) {
  const float M = fmaxf(a.m, b.m);
  if (M == -INFINITY) return MaxSum{M, 0.f};
  const float sa = (a.m == -INFINITY) ? 0.f : a.s * rescale(a.m, M, c);
  const float sb = (b.m == -INFINITY) ? 0.f : b.s * rescale(b.m, M, c);
  return MaxSum{M, sa + sb};
}

struct ArgMax {
  float v;
  int i;  // -1 = empty
};
__device__ __forceinline__ ArgMax better_arg(ArgMax a, ArgMax b) {
  if (a.i < 0) return b;
  if (b.i < 0) return a;
  if (b.v > a.v || (b.v == a.v && b.i < a.i)) return b;
  return a;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Pairwise sum of a small fixed-size array.
template <int N>
__device__ __forceinline__ float pair_sum(const float (&a)[N]) {
  if constexpr (N == 8) {
    return ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
  } else {
    return (a[0] + a[1]) + (a[2] + a[3]);
  }
}

// ---------------------------------------------------------------------------
// Slice staging.  The caller owns `bars` (kMaxStages mbarriers) in shared
// memory.  Bulk path: thread 0 issues, per stage, one copy per row; every
// thread later waits on the stage's barrier.  Plain path (rows not 16-byte
// aligned): all threads copy with ordinary loads, padding the slice to a whole
// vector with -inf, then the block synchronises.
// ---------------------------------------------------------------------------
template <typename E>
struct Slice {
  const E* gt;  // global target slice start (row + lo)
  const E* gd;  // global draft slice start, or nullptr
  E* st;        // shared target slice
  E* sd;        // shared draft slice (valid when gd)
  int n;        // elements in this CTA's slice (may be 0)
  int nvec;     // ceil(n / kVec)
  int nstage;   // stages covering nvec
  bool bulk;
};

template <typename E>
__device__ __forceinline__ void stage_issue(const Slice<E>& sl, uint64_t* bars, int stage_elems) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < sl.nstage; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (sl.bulk) {
    if (threadIdx.x == 0) {
      const uint64_t pol = l2_policy_evict_first();
      for (int s = 0; s < sl.nstage; ++s) {
        const int e0 = s * stage_elems;
        const int ne = min(stage_elems, sl.n - e0);
        const uint32_t bytes = static_cast<uint32_t>(ne) * sizeof(E);
        mbar_arrive_expect_tx(&bars[s], sl.gd ? 2 * bytes : bytes);
        bulk_copy_g2s(sl.st + e0, sl.gt + e0, bytes, &bars[s], pol);
        if (sl.gd) bulk_copy_g2s(sl.sd + e0, sl.gd + e0, bytes, &bars[s], pol);
      }
    }
  } else {
    constexpr int kVec = Elem<E>::kVec;
    const int padded = sl.nvec * kVec;
    for (int e = threadIdx.x; e < padded; e += kThreads) {
      sl.st[e] = e < sl.n ? sl.gt[e] : Elem<E>::neg_inf();
      if (sl.gd) sl.sd[e] = e < sl.n ? sl.gd[e] : Elem<E>::neg_inf();
    }
    __syncthreads();
  }
}

// Wait for stage s (bulk path).  Returns false when the bounded wait ran out.
template <typename E>
__device__ __forceinline__ bool stage_wait(const Slice<E>& sl, uint64_t* bars, int s) {
  if (!sl.bulk) return true;
  return mbar_wait_bounded(&bars[s], 0);
}

// After a timeout: give the copies still in flight a bounded chance to land
// before the CTA leaves (its shared memory is their destination).
template <typename E>
__device__ __forceinline__ void stage_drain(const Slice<E>& sl, uint64_t* bars) {
  if (!sl.bulk || threadIdx.x != 0) return;
  for (int s = 0; s < sl.nstage; ++s) mbar_wait_bounded(&bars[s], 0);
}

template <typename E>
__device__ __forceinline__ void load_vec(const E* base, int v, float (&f)[Elem<E>::kVec]) {
  const uint4 raw = reinterpret_cast<const uint4*>(base)[v];
  Elem<E>::unpack(raw, f);
}

// ---------------------------------------------------------------------------
// Statistics pass over the staged slice, stage by stage as the copies land.
// Target: (m, s) at scale c (if want_exp) and the argmax (if want_arg);
// draft: (m, s) when sl.gd.  Results are per thread.
// ---------------------------------------------------------------------------
template <typename E>
struct ThreadStats {
  MaxSum t, d;
  ArgMax a;
  bool timeout;
};

template <typename E>
__device__ __forceinline__ ThreadStats<E> stats_pass(const Slice<E>& sl, uint64_t* bars, int stage_vecs, float c,
                                                     bool want_exp, bool want_arg, int lo) {
  constexpr int kVec = Elem<E>::kVec;
  ThreadStats<E> r{{-INFINITY, 0.f}, {-INFINITY, 0.f}, {-INFINITY, -1}, false};
  for (int s = 0; s < sl.nstage; ++s) {
    if (!stage_wait(sl, bars, s)) r.timeout = true;
    const int v_end = min(sl.nvec, (s + 1) * stage_vecs);
    float ft[kVecPerThreadStage][kVec], fd[kVecPerThreadStage][kVec];
    bool have[kVecPerThreadStage];
    float lmt = -INFINITY, lmd = -INFINITY;
#pragma unroll
    for (int k = 0; k < kVecPerThreadStage; ++k) {
      const int v = s * stage_vecs + k * kThreads + threadIdx.x;
      have[k] = v < v_end;
      if (have[k]) {
        load_vec(sl.st, v, ft[k]);
        if (sl.gd) load_vec(sl.sd, v, fd[k]);
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
          lmt = fmaxf(lmt, ft[k][e]);
          if (sl.gd) lmd = fmaxf(lmd, fd[k][e]);
        }
        if (want_arg) {
#pragma unroll
          for (int e = 0; e < kVec; ++e) {
            if (r.a.i < 0 || ft[k][e] > r.a.v) {
              r.a.v = ft[k][e];
              r.a.i = lo + v * kVec + e;
            }
          }
        }
      }
    }
    if (!want_exp) continue;
    if (lmt > r.t.m) {
      r.t.s = (r.t.m == -INFINITY) ? 0.f : r.t.s * rescale(r.t.m, lmt, c);
      r.t.m = lmt;
    }
    if (sl.gd && lmd > r.d.m) {
      r.d.s = (r.d.m == -INFINITY) ? 0.f : r.d.s * rescale(r.d.m, lmd, c);
      r.d.m = lmd;
    }
    const float mct = scaled_max(r.t.m, c), mcd = scaled_max(r.d.m, c);
#pragma unroll
    for (int k = 0; k < kVecPerThreadStage; ++k) {
      if (!have[k]) continue;
      float et[kVec];
#pragma unroll
      for (int e = 0; e < kVec; ++e) et[e] = fast_exp2(fmaf(ft[k][e], c, -mct));
      r.t.s += pair_sum(et);
      if (sl.gd) {
        float ed[kVec];
#pragma unroll
        for (int e = 0; e < kVec; ++e) ed[e] = fast_exp2(fmaf(fd[k][e], c, -mcd));
        r.d.s += pair_sum(ed);
      }
    }
  }
  return r;
}

// Block reduction of per-thread statistics; the result is valid in every lane
// of warp 0 (a fixed butterfly over the warps' partials).
struct BlockStats {
  MaxSum t, d;
  ArgMax a;
  int timeout;
};

__device__ __forceinline__ void butterfly_stats(MaxSum& t, MaxSum& d, ArgMax& a, int& to, float c) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    MaxSum ot{__shfl_xor_sync(0xFFFFFFFFu, t.m, o), __shfl_xor_sync(0xFFFFFFFFu, t.s, o)};
    MaxSum od{__shfl_xor_sync(0xFFFFFFFFu, d.m, o), __shfl_xor_sync(0xFFFFFFFFu, d.s, o)};
    ArgMax oa{__shfl_xor_sync(0xFFFFFFFFu, a.v, o), __shfl_xor_sync(0xFFFFFFFFu, a.i, o)};
    t = combine_ms(t, ot, c);
    d = combine_ms(d, od, c);
    a = better_arg(a, oa);
    to |= __shfl_xor_sync(0xFFFFFFFFu, to, o);
  }
}

template <typename E>
__device__ __forceinline__ BlockStats block_reduce_stats(const ThreadStats<E>& ts, float c, float* red_f,
                                                         int* red_i) {
  // red_f: 5 * kWarps floats, red_i: 2 * kWarps ints
  MaxSum t = ts.t, d = ts.d;
  ArgMax a = ts.a;
  int to = ts.timeout ? 1 : 0;
  butterfly_stats(t, d, a, to, c);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    red_f[0 * kWarps + warp] = t.m;
    red_f[1 * kWarps + warp] = t.s;
    red_f[2 * kWarps + warp] = d.m;
    red_f[3 * kWarps + warp] = d.s;
    red_f[4 * kWarps + warp] = a.v;
    red_i[0 * kWarps + warp] = a.i;
    red_i[1 * kWarps + warp] = to;
  }
  __syncthreads();
  BlockStats out{{-INFINITY, 0.f}, {-INFINITY, 0.f}, {-INFINITY, -1}, 0};
  if (warp == 0) {
    if (lane < kWarps) {
      out.t = MaxSum{red_f[0 * kWarps + lane], red_f[1 * kWarps + lane]};
      out.d = MaxSum{red_f[2 * kWarps + lane], red_f[3 * kWarps + lane]};
      out.a = ArgMax{red_f[4 * kWarps + lane], red_i[0 * kWarps + lane]};
      out.timeout = red_i[1 * kWarps + lane];
    }
    butterfly_stats(out.t, out.d, out.a, out.timeout, c);
  }
  return out;
}

// ---------------------------------------------------------------------------
// Push-based cluster exchange.  Every CTA owns an Inbox; for exchange e it
// expects one record from each CTA of the cluster, delivered by st.async and
// counted on its barrier xbar[e].  No CTA ever reads another CTA's shared
// memory, so no CTA has to wait for its peers before it exits.
// ---------------------------------------------------------------------------
constexpr int kMaxCluster = 16;
enum { kXStats = 0, kXSum0 = 1, kXSum1 = 2, kXSum2 = 3, kXTop = 4, kNumX = 5 };

struct Inbox {
  float4 stats[kMaxCluster][2];       // {t.m, t.s, d.m, d.s}, {argmax v, argmax i, timeout, 0}
  double sums[3][kMaxCluster];        // per-pass CTA sums of weights
  float4 top[kMaxCluster][4];         // top-8: 8 values, 8 indices (Saguaro, rank 0 only)
};

// Thread 0 at start-up: the exchange barriers and their expected bytes.
__device__ __forceinline__ void inbox_init(uint64_t* xbar, int csize, bool want_top) {
  for (int e = 0; e < kNumX; ++e) mbar_init(&xbar[e], 1);
  fence_mbar_init();
  mbar_arrive_expect_tx(&xbar[kXStats], static_cast<uint32_t>(csize) * 32u);
  mbar_arrive_expect_tx(&xbar[kXSum0], static_cast<uint32_t>(csize) * 8u);
  mbar_arrive_expect_tx(&xbar[kXSum1], static_cast<uint32_t>(csize) * 8u);
  mbar_arrive_expect_tx(&xbar[kXSum2], static_cast<uint32_t>(csize) * 8u);
  if (want_top) mbar_arrive_expect_tx(&xbar[kXTop], static_cast<uint32_t>(csize) * 64u);
}

// Warp 0: send this CTA's statistics (held by lane 0) to every CTA.
__device__ __forceinline__ void push_stats(Inbox* inbox, uint64_t* xbar, int csize, int my_rank,
                                           const BlockStats& bs) {
  const int lane = threadIdx.x & 31;
  float4 a = make_float4(bs.t.m, bs.t.s, bs.d.m, bs.d.s);
  float4 b = make_float4(bs.a.v, __int_as_float(bs.a.i), __int_as_float(bs.timeout), 0.f);
  a.x = __shfl_sync(0xFFFFFFFFu, a.x, 0);
  a.y = __shfl_sync(0xFFFFFFFFu, a.y, 0);
  a.z = __shfl_sync(0xFFFFFFFFu, a.z, 0);
  a.w = __shfl_sync(0xFFFFFFFFu, a.w, 0);
  b.x = __shfl_sync(0xFFFFFFFFu, b.x, 0);
  b.y = __shfl_sync(0xFFFFFFFFu, b.y, 0);
  b.z = __shfl_sync(0xFFFFFFFFu, b.z, 0);
  if (lane < csize) {
    const uint32_t bar = dsmem_addr(&xbar[kXStats], lane);
    st_async_v4(dsmem_addr(&inbox->stats[my_rank][0], lane), a, bar);
    st_async_v4(dsmem_addr(&inbox->stats[my_rank][1], lane), b, bar);
  }
}

// Warp 0: wait for every CTA's statistics and combine them.  The xor
// butterfly applies the same (commutative) combine tree in every lane and in
// every CTA, so all of them obtain bit-identical row statistics.
__device__ __forceinline__ BlockStats gather_stats(Inbox* inbox, uint64_t* xbar, int csize, float c) {
  const int lane = threadIdx.x & 31;
  const bool ok = xbar_wait_bounded(&xbar[kXStats]);
  BlockStats out{{-INFINITY, 0.f}, {-INFINITY, 0.f}, {-INFINITY, -1}, ok ? 0 : 1};
  if (lane < csize) {
    const float4 a = inbox->stats[lane][0], b = inbox->stats[lane][1];
    out.t = MaxSum{a.x, a.y};
    out.d = MaxSum{a.z, a.w};
    out.a = ArgMax{b.x, __float_as_int(b.y)};
    out.timeout |= __float_as_int(b.z);
  }
  butterfly_stats(out.t, out.d, out.a, out.timeout, c);
  return out;
}

// Warp 0: send this CTA's pass-p weight sum (held by lane 0) to every CTA.
__device__ __forceinline__ void push_sum(Inbox* inbox, uint64_t* xbar, int csize, int my_rank, int p, double v) {
  const int lane = threadIdx.x & 31;
  v = __shfl_sync(0xFFFFFFFFu, v, 0);
  if (lane < csize)
    st_async_b64(dsmem_addr(&inbox->sums[p][my_rank], lane), static_cast<unsigned long long>(__double_as_longlong(v)),
                 dsmem_addr(&xbar[kXSum0 + p], lane));
}

// Warp 0: wait for every CTA's pass-p sum; returns the cluster total and, for
// the target u * total, the owning rank (-1 if the total is not positive), the
// target minus the weight of the ranks before the owner (*local), and that
// weight (*prefix).  A target beyond every boundary (rounding) goes to the
// last rank with positive weight.  Identical in every lane and CTA.
__device__ __forceinline__ double gather_sums(Inbox* inbox, uint64_t* xbar, int csize, int p, double u, int* owner,
                                              double* local, double* prefix, int* timeout) {
  const int lane = threadIdx.x & 31;
  if (!xbar_wait_bounded(&xbar[kXSum0 + p])) *timeout = 1;
  const double mine = lane < csize ? inbox->sums[p][lane] : 0.0;
  double incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  const double tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
  *owner = -1;
  *local = 0.0;
  *prefix = 0.0;
  if (!(tot > 0.0)) return tot;
  const double target = u * tot;
  const double excl = incl - mine;
  const unsigned hit = __ballot_sync(0xFFFFFFFFu, lane < csize && mine > 0.0 && target < incl);
  const unsigned pos = __ballot_sync(0xFFFFFFFFu, lane < csize && mine > 0.0);
  const int r = hit ? __ffs(hit) - 1 : 31 - __clz(pos);
  const double pre = __shfl_sync(0xFFFFFFFFu, excl, r);
  *owner = r;
  *prefix = pre;
  *local = target - pre;
  return tot;
}

// ---------------------------------------------------------------------------
// Weighted pass: each warp owns a contiguous run of vectors of the slice (its
// lanes interleave inside the run, so the shared-memory reads are conflict
// free).  wfun(xt[], xd[], w[]) turns one vector into kVec weights.  Writes the
// per-warp sums to wsum[] and returns the CTA sum (thread 0, fp64 over warps).
// If TOPK > 0, each lane also keeps its TOPK largest (weight, token) pairs.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void warp_range(int nvec, int warp, int& v0, int& v1) {
  const int per = (nvec + kWarps - 1) / kWarps;
  v0 = min(nvec, warp * per);
  v1 = min(nvec, v0 + per);
}

template <int K>
struct TopK {
  float v[K > 0 ? K : 1];
  int i[K > 0 ? K : 1];
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int s = 0; s < (K > 0 ? K : 1); ++s) {
      v[s] = -1.f;
      i[s] = 0x7FFFFFFF;
    }
  }
  // Insert (w, idx); indices arrive in increasing order per lane, so an equal
  // weight never displaces an earlier (lower-index) entry.
  __device__ __forceinline__ void push(float w, int idx) {
    if constexpr (K > 0) {
      if (!(w > v[K - 1])) return;
#pragma unroll
      for (int s = K - 1; s >= 0; --s) {
        const float pv = (s > 0) ? v[s - 1] : INFINITY;
        const int pi = (s > 0) ? i[s - 1] : 0;
        if (w > pv) {
          v[s] = pv;
          i[s] = pi;
        } else if (w > v[s]) {
          v[s] = w;
          i[s] = idx;
        }
      }
    }
  }
  __device__ __forceinline__ void pop() {
#pragma unroll
    for (int s = 0; s < (K > 0 ? K : 1) - 1; ++s) {
      v[s] = v[s + 1];
      i[s] = i[s + 1];
    }
    v[(K > 0 ? K : 1) - 1] = -1.f;
    i[(K > 0 ? K : 1) - 1] = 0x7FFFFFFF;
  }
};

__device__ __forceinline__ bool ranks_before(float v1, int i1, float v2, int i2) {
  return v1 > v2 || (v1 == v2 && i1 < i2);
}

template <typename E, int K, typename WFun>
__device__ __forceinline__ double weighted_pass(const Slice<E>& sl, int lo, const WFun& wfun, float* wsum,
                                                TopK<K>& tk) {
  constexpr int kVec = Elem<E>::kVec;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int v0, v1;
  warp_range(sl.nvec, warp, v0, v1);
  float acc = 0.f;
  for (int v = v0 + lane; v < v1; v += 32) {
    float xt[kVec], xd[kVec], w[kVec];
    load_vec(sl.st, v, xt);
    if (sl.gd) load_vec(sl.sd, v, xd);
    wfun(xt, xd, w);
    acc += pair_sum(w);
    if constexpr (K > 0) {
#pragma unroll
      for (int e = 0; e < kVec; ++e) tk.push(w[e], lo + v * kVec + e);
    }
  }
  acc = warp_sum(acc);
  if (lane == 0) wsum[warp] = acc;
  __syncthreads();
  double cta = 0.0;
  if (threadIdx.x == 0)
    for (int w = 0; w < kWarps; ++w) cta += static_cast<double>(wsum[w]);
  return cta;
}

// Merge the lanes' top-K lists of one warp; every lane returns the warp's
// list in `out` (descending, lower index first among equals).
template <int K>
__device__ __forceinline__ void warp_merge_topk(TopK<K>& tk, float (&ov)[K], int (&oi)[K]) {
#pragma unroll
  for (int r = 0; r < K; ++r) {
    float v = tk.v[0];
    int id = tk.i[0];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xFFFFFFFFu, v, o);
      const int i2 = __shfl_xor_sync(0xFFFFFFFFu, id, o);
      if (ranks_before(v2, i2, v, id)) {
        v = v2;
        id = i2;
      }
    }
    ov[r] = v;
    oi[r] = id;
    if (tk.i[0] == id && tk.v[0] == v && id != 0x7FFFFFFF) tk.pop();
  }
}

// ---------------------------------------------------------------------------
// Inverse-CDF search.
//
// pick_warp (thread 0): given per-warp sums of a chunk and a target tl
// relative to the chunk start, the warp whose run holds tl and the weight
// before that run (a target beyond every boundary through rounding goes to
// the last warp with positive weight; -1 if none).
//
// warp_scan (one warp): scans vectors [v0, v1) with a warp prefix scan and
// fp64 carries for the smallest element whose running sum exceeds tl (tl
// relative to v0; again falling back to the last positive element).  `load`
// fills the target / draft values of vector v and `wfun` turns them into
// weights.  Returns in every lane the element index relative to the chunk
// start (-1 if no positive weight), its CDF position relative to v0 and its
// weight.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int pick_warp(const float* wsum, int nwarps, double tl, double* base) {
  double acc = 0.0;
  int pick = -1, last_pos = -1;
  double pick_base = 0.0, last_base = 0.0;
  for (int w = 0; w < nwarps; ++w) {
    const double ws = static_cast<double>(wsum[w]);
    if (ws > 0.0) {
      last_pos = w;
      last_base = acc;
    }
    if (pick < 0 && ws > 0.0 && tl < acc + ws) {
      pick = w;
      pick_base = acc;
    }
    acc += ws;
  }
  if (pick < 0) {
    pick = last_pos;
    pick_base = last_base;
  }
  *base = pick_base;
  return pick;
}

struct ScanHit {
  int elem;     // element index relative to the chunk start, -1 if none
  double edge;  // weight before the element, relative to the scan start
  float w;      // the element's weight
};

template <int kVec, typename Load, typename WFun>
__device__ __forceinline__ ScanHit warp_scan(int v0, int v1, double tl, const Load& load, const WFun& wfun) {
  const int lane = threadIdx.x & 31;
  double carry = 0.0;
  ScanHit hit{-1, NAN, 0.f};
  int last_vec = -1;  // last vector with positive weight
  for (int vb = v0; vb < v1 && hit.elem < 0; vb += 32) {
    const int v = vb + lane;
    float w[kVec];
    float vs = 0.f;
    if (v < v1) {
      float xt[kVec], xd[kVec];
      load(v, xt, xd);
      wfun(xt, xd, w);
      vs = pair_sum(w);
    } else {
#pragma unroll
      for (int e = 0; e < kVec; ++e) w[e] = 0.f;
    }
    float incl = vs;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    const float total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    const unsigned pos = __ballot_sync(0xFFFFFFFFu, vs > 0.f);
    if (pos) last_vec = vb + 31 - __clz(pos);
    const unsigned hm = __ballot_sync(0xFFFFFFFFu, (vs > 0.f) && (tl < carry + static_cast<double>(incl)));
    if (hm) {
      const int L = __ffs(hm) - 1;
      int tok = -1;
      double edge = 0.0;
      float wt = 0.f;
      if (lane == L) {
        double a = carry + static_cast<double>(incl - vs);
        int last_e = -1;
        double a_last = a;
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
          const double before = a;
          if (w[e] > 0.f) {
            last_e = e;
            a_last = before;
          }
          a += static_cast<double>(w[e]);
          if (tok < 0 && w[e] > 0.f && tl < a) {
            tok = e;
            edge = before;
          }
        }
        if (tok < 0) {
          tok = last_e;
          edge = a_last;
        }
#pragma unroll
        for (int e = 0; e < kVec; ++e)
          if (e == tok) wt = w[e];
        tok = v * kVec + tok;
      }
      hit.elem = __shfl_sync(0xFFFFFFFFu, tok, L);
      hit.edge = __shfl_sync(0xFFFFFFFFu, edge, L);
      hit.w = __shfl_sync(0xFFFFFFFFu, wt, L);
    }
    carry += static_cast<double>(total);
  }
  if (hit.elem < 0 && last_vec >= 0) {
    // rounding left the target past the run: take its last positive element
    int e_last = kVec - 1;
    float wl = 0.f;
    if (lane == 0) {
      float xt[kVec], xd[kVec], w[kVec];
      load(last_vec, xt, xd);
      wfun(xt, xd, w);
#pragma unroll
      for (int e = 0; e < kVec; ++e)
        if (w[e] > 0.f) {
          e_last = e;
          wl = w[e];
        }
    }
    hit.elem = __shfl_sync(0xFFFFFFFFu, last_vec * kVec + e_last, 0);
    hit.w = __shfl_sync(0xFFFFFFFFu, wl, 0);
    hit.edge = NAN;
  }
  return hit;
}

// The search inside a slice resident in shared memory whose per-warp sums
// (from weighted_pass) are in wsum[].  Writes the global token to *result,
// the drawn element's CDF position relative to this CTA's start (NaN after a
// rounding fallback) to *edge_lo and its weight to *edge_w (shared memory).
template <typename E, typename WFun>
__device__ __forceinline__ void cdf_search(const Slice<E>& sl, int lo, const WFun& wfun, const float* wsum, double tl,
                                           int* sh_warp, double* sh_base, int* result, double* edge_lo,
                                           float* edge_w) {
  constexpr int kVec = Elem<E>::kVec;
  if (threadIdx.x == 0) {
    *sh_warp = pick_warp(wsum, kWarps, tl, sh_base);
    *result = -1;
    *edge_lo = NAN;
    *edge_w = 0.f;
  }
  __syncthreads();
  const int pick = *sh_warp;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (pick >= 0 && warp == pick) {
    int v0, v1;
    warp_range(sl.nvec, warp, v0, v1);
    const double base = *sh_base;
    auto load = [&](int v, float(&xt)[kVec], float(&xd)[kVec]) {
      load_vec(sl.st, v, xt);
      if (sl.gd) load_vec(sl.sd, v, xd);
    };
    const ScanHit h = warp_scan<kVec>(v0, v1, tl - base, load, wfun);
    if (lane == 0) {
      *result = h.elem >= 0 ? lo + h.elem : -1;
      *edge_lo = base + h.edge;
      *edge_w = h.w;
    }
  }
  __syncthreads();
}


// ---------------------------------------------------------------------------
// Programmatic dependent launch and arrival counters.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }


// Arrival counter with acquire-release semantics: the releases of earlier
// arrivals (their published sums) are visible to the last one.
__device__ __forceinline__ int ticket_add(int32_t* p) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(p) : "memory");
  return old;
}


// ---------------------------------------------------------------------------
// Pieces: 128 vectors of a row, handled by one warp (lane L holds vectors
// 4L .. 4L+3).  Piece sums, the lane-scan search of a row's pieces and of one
// piece, used by the sampling passes of verification and Saguaro.
// ---------------------------------------------------------------------------
constexpr int kPieceVecs = 128;  // vectors per piece: 4 per lane

// A piece's vectors as raw 16-byte words, lane L holding the 4 consecutive
// vectors 4L .. 4L+3, target and, when gd is given, draft; elements past n
// read as -inf (weight 0).  One round of loads.
template <typename E>
struct PieceRows {
  uint4 rt[4], rd[4];
  __device__ __forceinline__ void load(const E* gt, const E* gd, int n, bool aligned) {
    constexpr int kVec = Elem<E>::kVec;
    const int lane = threadIdx.x & 31;
    const int nv = (n + kVec - 1) / kVec;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int v = 4 * lane + k;
      rt[k] = rd[k] = Elem<E>::max_init();  // all -inf
      if (v >= nv) continue;
      if (aligned) {
        rt[k] = __ldg(reinterpret_cast<const uint4*>(gt) + v);
        if (gd) rd[k] = __ldg(reinterpret_cast<const uint4*>(gd) + v);
      } else {
        rt[k] = gather_vec(gt, v * kVec, n);
        if (gd) rd[k] = gather_vec(gd, v * kVec, n);
      }
    }
  }
  // Elements [i0, i0 + kVec) of a row not aligned to 16 bytes, -inf past n.
  static __device__ __forceinline__ uint4 gather_vec(const E* g, int i0, int n) {
    uint32_t w[4];
    if constexpr (sizeof(E) == 2) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t lo = i0 + 2 * j < n ? static_cast<uint32_t>(g[i0 + 2 * j]) : 0xFF80u;
        const uint32_t hi = i0 + 2 * j + 1 < n ? static_cast<uint32_t>(g[i0 + 2 * j + 1]) : 0xFF80u;
        w[j] = lo | (hi << 16);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = __float_as_uint(i0 + j < n ? static_cast<float>(g[i0 + j]) : -INFINITY);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
  template <typename WFun>
  __device__ __forceinline__ void weights(int k, const WFun& wfun, float (&w)[Elem<E>::kVec]) const {
    float xt[Elem<E>::kVec], xd[Elem<E>::kVec];
    Elem<E>::unpack(rt[k], xt);
    Elem<E>::unpack(rd[k], xd);
    wfun(xt, xd, w);
  }
};

// The weight sum of a lane's 4 vectors (in vector order).
template <typename E, typename WFun>
__device__ __forceinline__ float piece_lane_sum(const PieceRows<E>& pr, const WFun& wfun) {
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float w[Elem<E>::kVec];
    pr.weights(k, wfun, w);
    s += pair_sum(w);
  }
  return s;
}

// One warp, one value per lane in index order: the exclusive prefix of every
// lane (fp64) and the first lane whose running sum passes tl, else the last
// lane with a positive value (-1 if none).
__device__ __forceinline__ int lane_locate(double v, double tl, double* before) {
  const int lane = threadIdx.x & 31;
  double incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  const unsigned hm = __ballot_sync(0xFFFFFFFFu, v > 0.0 && tl < incl);
  const unsigned pm = __ballot_sync(0xFFFFFFFFu, v > 0.0);
  const int L = hm ? __ffs(hm) - 1 : (pm ? 31 - __clz(pm) : -1);
  *before = __shfl_sync(0xFFFFFFFFu, incl - v, L >= 0 ? L : 0);
  return L;
}

// One warp: the element of a loaded piece whose running weight first exceeds
// tl (relative to the piece start), falling back to the last element with
// positive weight: a lane scan over the lanes' sums, then the found lane's 4
// vectors element by element (fp32 from the lane's start: the lane's weight is
// a small share of the row's).  Returns the element index relative to the
// piece start (-1 if none), the weight before it and its weight.
template <typename E, typename WFun>
__device__ __forceinline__ ScanHit scan_piece(const PieceRows<E>& pr, const WFun& wfun, double tl) {
  constexpr int kVec = Elem<E>::kVec;
  const int lane = threadIdx.x & 31;
  float w[4][kVec];
  float ls = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    pr.weights(k, wfun, w[k]);
    ls += pair_sum(w[k]);
  }
  double before = 0.0;
  const int L = lane_locate(static_cast<double>(ls), tl, &before);
  if (L < 0) return ScanHit{-1, NAN, 0.f};
  int el = -1;
  float edge = 0.f, we = 0.f;
  if (lane == L) {
    const float t = static_cast<float>(tl - before);
    float acc = 0.f;
    bool done = false;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
#pragma unroll
      for (int e = 0; e < kVec; ++e) {
        if (!done && w[k][e] > 0.f) {
          el = k * kVec + e;  // the hit, or the last positive element so far
          edge = acc;
          we = w[k][e];
          done = t < acc + w[k][e];
        }
        acc += w[k][e];
      }
    }
  }
  el = __shfl_sync(0xFFFFFFFFu, el, L);
  edge = __shfl_sync(0xFFFFFFFFu, edge, L);
  we = __shfl_sync(0xFFFFFFFFu, we, L);
  if (el < 0) return ScanHit{-1, NAN, 0.f};
  return ScanHit{4 * L * kVec + el, before + static_cast<double>(edge), we};
}

// One warp: a row's piece sums, copied into the warp's shared slice `v` (lane
// L's consecutive share first summed by lane L), the lane sums and the row
// total (fp64 over lanes), valid in every lane.
struct RowPieces {
  float* v;  // shared, np floats
  int per;
  float lane_sum;
  double total;
  __device__ __forceinline__ void load(const float* psum, int np, float* slice) {
    const int lane = threadIdx.x & 31;
    v = slice;
    per = (np + 31) / 32;
    for (int q = lane; q < np; q += 32) v[q] = __ldcg(psum + q);
    __syncwarp();
    lane_sum = 0.f;
    for (int k = 0; k < per; ++k) {
      const int q = lane * per + k;
      if (q < np) lane_sum += v[q];
    }
    double t = static_cast<double>(lane_sum);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
    total = t;
  }
};


// The element of a row drawn at u * total of the row's piece sums.
struct RowDraw {
  int elem;     // element index in the row, -1 if none
  double edge;  // weight before it (from the row start)
  float w;      // its weight
};

// One warp: the lane whose run of pieces holds target = u * total, the piece
// within that run, then that piece reloaded and scanned (wfun gives the
// weights; drow may be null).
template <typename E, typename WFun>
__device__ __forceinline__ RowDraw warp_locate_row(const RowPieces& rp, double u, const E* trow, const E* drow,
                                                   int V, bool aligned, const WFun& wfun) {
  constexpr int kVec = Elem<E>::kVec;
  const int lane = threadIdx.x & 31;
  const int pelems = kPieceVecs * kVec;
  const int np = (V + pelems - 1) / pelems;
  const double target = u * rp.total;
  double before = 0.0;
  const int L = lane_locate(static_cast<double>(rp.lane_sum), target, &before);
  int owner = -1;
  float obefore = 0.f;
  if (lane == L) {
    const float t = static_cast<float>(target - before);
    float acc = 0.f;
    for (int k = 0; k < rp.per; ++k) {
      const int q = L * rp.per + k;
      const float w = q < np ? rp.v[q] : 0.f;
      if (w > 0.f) {
        owner = q;  // the hit, or the last positive piece so far
        obefore = acc;
        if (t < acc + w) break;
      }
      acc += w;
    }
  }
  owner = __shfl_sync(0xFFFFFFFFu, owner, L >= 0 ? L : 0);
  const double owner_before = before + static_cast<double>(__shfl_sync(0xFFFFFFFFu, obefore, L >= 0 ? L : 0));
  RowDraw d{-1, NAN, 0.f};
  if (L >= 0 && owner >= 0) {
    const int olo = owner * pelems;
    PieceRows<E> pr;
    pr.load(trow + olo, drow ? drow + olo : nullptr, min(pelems, V - olo), aligned);
    const ScanHit h = scan_piece(pr, wfun, target - owner_before);
    if (h.elem >= 0) d = RowDraw{olo + h.elem, owner_before + h.edge, h.w};
  }
  return d;
}

}  // namespace ssdv
