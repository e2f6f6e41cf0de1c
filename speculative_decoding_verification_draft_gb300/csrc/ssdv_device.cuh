// ssdv_device.cuh -- device building blocks shared by the verification,
// Saguaro and top-p kernels: exp2 and packed fp32 pairs, the bf16 / fp32
// element types, the Philox4x32-10 generator, softmax statistics and their
// combine, warp top-k lists, float-float running sums, programmatic dependent
// launch and arrival counters, and the piece loads and lane-scan searches of
// the inverse-CDF draw.
#pragma once

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "ssdv_internal.h"

namespace ssdv {

constexpr int kThreads = 256;
// vectors of a chunk row per thread in the register form of the streaming kernel
constexpr int kRegVecs = 8;
constexpr int kWarps = kThreads / 32;
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
// A chunk of a target row (and of a draft row) and its shared-memory copy.
// ---------------------------------------------------------------------------
template <typename E>
struct Slice {
  const E* gt;  // global target slice start (row + lo)
  const E* gd;  // global draft slice start, or nullptr
  E* st;        // shared target slice
  E* sd;        // shared draft slice (valid when gd)
  int n;        // elements in this CTA's slice (may be 0)
  int nvec;     // ceil(n / kVec)
};

template <typename E>
__device__ __forceinline__ void load_vec(const E* base, int v, float (&f)[Elem<E>::kVec]) {
  const uint4 raw = reinterpret_cast<const uint4*>(base)[v];
  Elem<E>::unpack(raw, f);
}

// Warp butterfly of per-lane row statistics (target and draft (max, sum), the
// target argmax); the result is valid in every lane.
__device__ __forceinline__ void butterfly_stats(MaxSum& t, MaxSum& d, ArgMax& a, float c) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    MaxSum ot{__shfl_xor_sync(0xFFFFFFFFu, t.m, o), __shfl_xor_sync(0xFFFFFFFFu, t.s, o)};
    MaxSum od{__shfl_xor_sync(0xFFFFFFFFu, d.m, o), __shfl_xor_sync(0xFFFFFFFFu, d.s, o)};
    ArgMax oa{__shfl_xor_sync(0xFFFFFFFFu, a.v, o), __shfl_xor_sync(0xFFFFFFFFu, a.i, o)};
    t = combine_ms(t, ot, c);
    d = combine_ms(d, od, c);
    a = better_arg(a, oa);
  }
}

// ---------------------------------------------------------------------------
// Top-K: a lane's K largest (weight, index) pairs, descending, and the merge
// of a warp's lanes.
// ---------------------------------------------------------------------------
// kNegInf: keys may be -inf (logits), so an empty slot is told apart by its
// index; otherwise keys are finite and larger than the empty value -inf.
template <int K, bool kNegInf = false>
struct TopK {
  static constexpr int kEmpty = 0x7FFFFFFF;  // index of an empty slot (ranks after everything)
  float v[K > 0 ? K : 1];
  int i[K > 0 ? K : 1];
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int s = 0; s < (K > 0 ? K : 1); ++s) {
      v[s] = -INFINITY;
      i[s] = kEmpty;
    }
  }
  // Whether (w, a later index) ranks before slot s: slot s is empty or w is
  // larger.  Indices arrive in increasing order per lane, so an equal value
  // never displaces an earlier (lower-index) entry.
  __device__ __forceinline__ bool beats(float w, int s) const {
    if constexpr (kNegInf) return i[s] == kEmpty || w > v[s];
    return w > v[s];
  }
  __device__ __forceinline__ void push(float w, int idx) {
    if constexpr (K > 0) {
      if (!beats(w, K - 1)) return;
#pragma unroll
      for (int s = K - 1; s >= 0; --s) {
        if (s > 0 && beats(w, s - 1)) {
          v[s] = v[s - 1];
          i[s] = i[s - 1];
        } else if (beats(w, s)) {
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
    v[(K > 0 ? K : 1) - 1] = -INFINITY;
    i[(K > 0 ? K : 1) - 1] = kEmpty;
  }
};

__device__ __forceinline__ bool ranks_before(float v1, int i1, float v2, int i2) {
  return v1 > v2 || (v1 == v2 && i1 < i2);
}

// Merge the lanes' top-K lists of one warp; every lane returns the warp's
// list in `out` (descending, lower index first among equals).
template <int K, bool kNegInf>
__device__ __forceinline__ void warp_merge_topk(TopK<K, kNegInf>& tk, float (&ov)[K], int (&oi)[K]) {
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
// Float-float numbers: hi + lo with |lo| at most half an ulp of hi, about 48
// significant bits.  Running sums across lanes and pieces use them: a chain of
// dependent fp64 adds is slow on GB300's small fp64 units, and fp32 alone
// would put a row's CDF edges too far from the exact ones.  The error-free
// transformations are Knuth's TwoSum and the FMA form of Dekker's TwoProduct;
// every operation is an explicit round-to-nearest intrinsic, so the compiler
// neither contracts nor reorders them.
// ---------------------------------------------------------------------------
struct FF {
  float hi, lo;
};
__device__ __forceinline__ FF ff_fast_two_sum(float a, float b) {  // |a| >= |b|
  const float s = __fadd_rn(a, b);
  return FF{s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ FF ff_add(FF a, FF b) {
  const float s = __fadd_rn(a.hi, b.hi);
  const float bb = __fsub_rn(s, a.hi);
  const float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bb)), __fsub_rn(b.hi, bb));
  return ff_fast_two_sum(s, __fadd_rn(e, __fadd_rn(a.lo, b.lo)));
}
__device__ __forceinline__ FF ff_sub(FF a, FF b) { return ff_add(a, FF{-b.hi, -b.lo}); }
// a * u for a float u
__device__ __forceinline__ FF ff_mul(FF a, float u) {
  const float p = __fmul_rn(a.hi, u);
  const float e = __fmaf_rn(a.hi, u, -p);
  return ff_fast_two_sum(p, __fmaf_rn(a.lo, u, e));
}
__device__ __forceinline__ bool ff_lt(FF a, FF b) { return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo); }
__device__ __forceinline__ float ff_float(FF a) { return __fadd_rn(a.hi, a.lo); }
__device__ __forceinline__ double ff_double(FF a) { return static_cast<double>(a.hi) + static_cast<double>(a.lo); }
__device__ __forceinline__ FF ff_shfl_xor(FF a, int o) {
  return FF{__shfl_xor_sync(0xFFFFFFFFu, a.hi, o), __shfl_xor_sync(0xFFFFFFFFu, a.lo, o)};
}
// sum of one float per lane, valid in every lane
__device__ __forceinline__ FF ff_warp_sum(float v) {
  FF t{v, 0.f};
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t = ff_add(t, ff_shfl_xor(t, o));
  return t;
}

struct ScanHit {
  int elem;  // element index relative to the chunk start, -1 if none
  FF edge;   // weight before the element, relative to the scan start
  float w;   // the element's weight
};

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
  // The raw logits of vector k (target, draft).
  __device__ __forceinline__ void raw(int k, float (&xt)[Elem<E>::kVec], float (&xd)[Elem<E>::kVec]) const {
    Elem<E>::unpack(rt[k], xt);
    Elem<E>::unpack(rd[k], xd);
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
// lane (float-float) and the first lane whose running sum passes tl, else the
// last lane with a positive value (-1 if none).
__device__ __forceinline__ int lane_locate(float v, FF tl, FF* before) {
  const int lane = threadIdx.x & 31;
  FF incl{v, 0.f};
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const FF t{__shfl_up_sync(0xFFFFFFFFu, incl.hi, o), __shfl_up_sync(0xFFFFFFFFu, incl.lo, o)};
    if (lane >= o) incl = ff_add(incl, t);
  }
  const unsigned hm = __ballot_sync(0xFFFFFFFFu, v > 0.f && ff_lt(tl, incl));
  const unsigned pm = __ballot_sync(0xFFFFFFFFu, v > 0.f);
  const int L = hm ? __ffs(hm) - 1 : (pm ? 31 - __clz(pm) : -1);
  const FF ex = ff_sub(incl, FF{v, 0.f});
  *before = FF{__shfl_sync(0xFFFFFFFFu, ex.hi, L >= 0 ? L : 0), __shfl_sync(0xFFFFFFFFu, ex.lo, L >= 0 ? L : 0)};
  return L;
}

// One warp: the element of a loaded piece whose running weight first exceeds
// tl (relative to the piece start), falling back to the last element with
// positive weight: a lane scan over the lanes' sums, then the found lane's 4
// vectors element by element (fp32 from the lane's start: the lane's weight is
// a small share of the row's).  Returns the element index relative to the
// piece start (-1 if none), the weight before it and its weight.
template <typename E, typename WFun>
__device__ __forceinline__ ScanHit scan_piece(const PieceRows<E>& pr, const WFun& wfun, FF tl) {
  constexpr int kVec = Elem<E>::kVec;
  const int lane = threadIdx.x & 31;
  float w[4][kVec];
  float ls = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    pr.weights(k, wfun, w[k]);
    ls += pair_sum(w[k]);
  }
  FF before;
  const int L = lane_locate(ls, tl, &before);
  if (L < 0) return ScanHit{-1, FF{NAN, 0.f}, 0.f};
  int el = -1;
  float edge = 0.f, we = 0.f;
  if (lane == L) {
    const float t = ff_float(ff_sub(tl, before));
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
  if (el < 0) return ScanHit{-1, FF{NAN, 0.f}, 0.f};
  return ScanHit{4 * L * kVec + el, ff_add(before, FF{edge, 0.f}), we};
}

// One warp: a row's piece sums, copied into the warp's shared slice `v` (lane
// L's consecutive share first summed by lane L), the lane sums and the row
// total (fp64 over lanes), valid in every lane.
struct RowPieces {
  float* v;  // shared, np floats
  int per;
  float lane_sum;
  FF tot;        // the row total
  double total;  // the same, as one fp64 value
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
    tot = ff_warp_sum(lane_sum);
    total = ff_double(tot);
  }
};


// The element of a row drawn at u * total of the row's piece sums.
struct RowDraw {
  int elem;  // element index in the row, -1 if none
  FF edge;   // weight before it (from the row start)
  float w;   // its weight
};

// One warp: the lane whose run of pieces holds target = u * total, the piece
// within that run, then that piece reloaded and scanned (wfun gives the
// weights; drow may be null).
template <typename E, typename WFun>
__device__ __forceinline__ RowDraw warp_locate_row(const RowPieces& rp, float u, const E* trow, const E* drow,
                                                   int V, bool aligned, const WFun& wfun) {
  constexpr int kVec = Elem<E>::kVec;
  const int lane = threadIdx.x & 31;
  const int pelems = kPieceVecs * kVec;
  const int np = (V + pelems - 1) / pelems;
  const FF target = ff_mul(rp.tot, u);
  FF before;
  const int L = lane_locate(rp.lane_sum, target, &before);
  int owner = -1;
  float obefore = 0.f;
  if (lane == L) {
    const float t = ff_float(ff_sub(target, before));
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
  const FF owner_before = ff_add(before, FF{__shfl_sync(0xFFFFFFFFu, obefore, L >= 0 ? L : 0), 0.f});
  RowDraw d{-1, FF{NAN, 0.f}, 0.f};
  if (L >= 0 && owner >= 0) {
    const int olo = owner * pelems;
    PieceRows<E> pr;
    pr.load(trow + olo, drow ? drow + olo : nullptr, min(pelems, V - olo), aligned);
    const ScanHit h = scan_piece(pr, wfun, ff_sub(target, owner_before));
    if (h.elem >= 0) d = RowDraw{olo + h.elem, ff_add(owner_before, h.edge), h.w};
  }
  return d;
}

}  // namespace ssdv
