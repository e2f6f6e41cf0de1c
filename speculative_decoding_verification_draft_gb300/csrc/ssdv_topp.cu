// ssdv_topp.cu -- top-p (nucleus) thresholds for verification.
//
// Verification composes with top-p when both sides truncate the same way (the
// verification blog's closing remark and its section on matching sampling
// parameters): each target and draft row keeps the tokens whose logit is at
// least th, the largest logit value whose upper set {x >= th} holds at least
// top_p of the row's probability mass (tokens tied with the last one needed
// are kept), renormalised.
//
// th is found per row by a select over levels, each a counting pass over the
// rows' chunks followed by a select pass (one CTA per row).  Level 0 bins
// every element by its mass relative to the row maximum, an eighth of an
// octave per bin (bin = floor(8 (fl(m c) - x c)), the last bin holding the
// tail), which spreads a row's elements over many bins; the select fixes the
// bin b* in which the mass counted from the top reaches ceil(top_p * total).
// The later levels resolve th inside b* by a radix select over a monotone
// 32-bit key of the logit, high digits first (bf16: two 8-bit digits of the
// 16 bits that matter; fp32: digits of 11, 11 and 10 bits), counting only the
// elements of b* (topp_refine_kernel: so few that their masses go straight to
// global memory).  Masses exp2(x c - fl(m c)) are summed in fixed point (2^-40
// units), so the integer sums are exact and the same on every run whatever
// the order of the atomics.
#include <algorithm>

#include "ssdv_device.cuh"

namespace ssdv {

namespace {

constexpr int kHistThreads = 256;
constexpr uint32_t kRowDone = 0xFFFFFFFFu;     // bstar of a row whose th is fixed before the last level
constexpr uint32_t kDirectFlag = 0x80000000u;  // level 1's word for the select: keys counted directly

__device__ __forceinline__ bool temperature_ok_tp(float T) { return T == 0.f || (T >= 1e-6f && T <= 3.0e38f); }

// Monotone key of a logit (-0 taken as +0, as the comparisons x >= th do).
__device__ __forceinline__ uint32_t logit_key(float x) {
  const uint32_t b = __float_as_uint(x + 0.f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// round(e * 2^40) for 0 <= e < 2, from two 32-bit conversions
__device__ __forceinline__ unsigned long long mass_fixed(float e) {
  const float f = e * 256.f;
  const uint32_t hi = __float2uint_rz(f);
  const float r = f - __uint2float_rz(hi);  // exact
  return (static_cast<unsigned long long>(hi) << 32) + __float2uint_rn(r * 4294967296.f);
}

// Row slot rs = (b * W + i) * 2 + which (0 target, 1 draft): whether it is a
// row of a sampled request that verification reads.
__device__ __forceinline__ bool slot_active(const TopPArgs& a, int b, int i, int which, float* T_out) {
  const int g = a.gamma ? a.gamma[b] : a.gmax;
  const float T = a.temps ? a.temps[b] : a.temp_scalar;
  *T_out = T;
  if (g < 0 || g > a.gmax || !temperature_ok_tp(T) || T == 0.f) return false;
  return which == 0 ? i <= g : i < g;
}

}  // namespace

namespace {

// The row maximum from the row's chunk records (every lane of the calling
// warp gets it): the largest chunk maximum.
__device__ __forceinline__ float row_max_warp(const TopPArgs& a, int b, int i, int which) {
  const int lane = threadIdx.x & 31, NC = a.geo.nchunk, W = a.gmax + 1;
  float m = -INFINITY;
  for (int q = lane; q < NC; q += 32) {
    const float4 r0 = __ldcg(a.part + ((static_cast<size_t>(b) * W + i) * NC + q) * 2);
    m = fmaxf(m, which ? r0.z : r0.x);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  return m;
}

constexpr int kNVH = 6;  // 16-byte vectors per thread loaded at once

// One chunk of one row: its elements' logits handed to f, the aligned case
// from loads issued (all of a thread's at once) before the wait for the
// previous kernel, since the logits are inputs complete before the call.
template <typename E, typename F>
__device__ __forceinline__ void for_chunk(const TopPArgs& a, const E* row, int lo, int n, F&& f) {
  constexpr int kVec = Elem<E>::kVec;
  const int nvec = n / kVec;  // aligned rows: whole vectors
  const bool batched = a.geo.aligned && nvec <= kNVH * kHistThreads;
  uint4 r[kNVH];
  if (batched) {
    const uint4* rv = reinterpret_cast<const uint4*>(row + lo);
#pragma unroll
    for (int k = 0; k < kNVH; ++k) {
      const int v = threadIdx.x + k * kHistThreads;
      r[k] = v < nvec ? __ldg(rv + v) : Elem<E>::max_init();
    }
  }
  griddep_wait();  // the records (and the previous level's digits) are complete and visible
  f.begin();
  if (batched) {
#pragma unroll
    for (int k = 0; k < kNVH; ++k) {
      float x[kVec];
      Elem<E>::unpack(r[k], x);
#pragma unroll
      for (int e = 0; e < kVec; e += 2) f.pair(x[e], x[e + 1]);
    }
  } else if (a.geo.aligned) {
    const uint4* rv = reinterpret_cast<const uint4*>(row + lo);
    for (int v = threadIdx.x; v < nvec; v += kHistThreads) {
      float x[kVec];
      Elem<E>::unpack(__ldg(rv + v), x);
#pragma unroll
      for (int e = 0; e < kVec; ++e) f(x[e]);
    }
  } else {
    for (int e = threadIdx.x; e < n; e += kHistThreads) f(Elem<E>::to_float(row[lo + e]));
  }
}

template <typename E>
__device__ __forceinline__ const E* slot_row(const TopPArgs& a, int b, int i, int which) {
  const int W = a.gmax + 1, V = a.geo.V;
  return which ? static_cast<const E*>(a.draft) + (static_cast<size_t>(b) * a.gmax + i) * V
               : static_cast<const E*>(a.target) + (static_cast<size_t>(b) * W + i) * V;
}

// Level 0's counter: every element's mass into the warp's own copy of the
// 256 mass bins, as two 32-bit words a bin.  The 2^-40 fixed-point mass
// round(e 2^40) is split as hi 2^20 + lo with hi = floor(e 2^20) and
// lo = round((e 2^20 - hi) 2^20), both straight from 32-bit conversions (e
// 2^20 and its fraction are exact in fp32, so only the last step rounds, as
// round(e 2^40) does).  Each word takes at most 2^20 per element (e <= 1),
// and a warp sees at most 2048 elements of a chunk (chunks hold at most
// 16384): neither word can overflow, and no atomic needs its old value.  The
// bin's mass is (sum of hi) 2^20 + (sum of lo).
struct MassBins {
  const TopPArgs* a;
  int b, i, which;
  uint32_t* hist;  // this warp's copy
  float cc, mc;
  __device__ __forceinline__ void begin() { mc = scaled_max(row_max_warp(*a, b, i, which), cc); }
  __device__ __forceinline__ void operator()(float x) const {
    if (x == -INFINITY) return;  // no mass
    const float d = __fmaf_rn(-x, cc, mc);  // fl(m c) - x c, one rounding
    const int bin = min(255, max(0, __float2int_rd(d * 8.f)));
    const int digit = 255 - bin;  // larger digit, larger mass
    const float f = fast_exp2(-d) * 1048576.f;  // e 2^20, exact
    const uint32_t hi20 = __float2uint_rz(f);
    const uint32_t lo20 = __float2uint_rn((f - __uint2float_rz(hi20)) * 1048576.f);  // only the conversion rounds
    if (lo20) atomicAdd(&hist[digit], lo20);
    if (hi20) atomicAdd(&hist[256 + digit], hi20);
  }
  // Two elements at once: the same roundings element by element, with the
  // floating-point steps as f32x2 pairs (the multiplications are exact
  // power-of-two scalings).  A -inf element gets d = +inf, the last bin and
  // mass 0, so it adds nothing.
  __device__ __forceinline__ void pair(float x0, float x1) const {
    float d0, d1, s0, s1;
    f2_split(f2_fma(f2_make(x0, x1), f2_make(-cc, -cc), f2_make(mc, mc)), d0, d1);  // fl(m c) - x c
    f2_split(f2_fma(f2_make(d0, d1), f2_make(8.f, 8.f), f2_make(0.f, 0.f)), s0, s1);
    const int g0 = 255 - min(255, max(0, __float2int_rd(s0)));
    const int g1 = 255 - min(255, max(0, __float2int_rd(s1)));
    float f0, f1, r0, r1, t0, t1;
    f2_split(f2_fma(f2_make(fast_exp2(-d0), fast_exp2(-d1)), f2_make(1048576.f, 1048576.f), f2_make(0.f, 0.f)), f0,
             f1);  // e 2^20
    const uint32_t hi0 = __float2uint_rz(f0), hi1 = __float2uint_rz(f1);
    f2_split(f2_add(f2_make(f0, f1), f2_make(-__uint2float_rz(hi0), -__uint2float_rz(hi1))), r0, r1);  // exact
    f2_split(f2_fma(f2_make(r0, r1), f2_make(1048576.f, 1048576.f), f2_make(0.f, 0.f)), t0, t1);
    const uint32_t lo0 = __float2uint_rn(t0), lo1 = __float2uint_rn(t1);
    if (lo0) atomicAdd(&hist[g0], lo0);
    if (hi0) atomicAdd(&hist[256 + g0], hi0);
    if (lo1) atomicAdd(&hist[g1], lo1);
    if (hi1) atomicAdd(&hist[256 + g1], hi1);
  }
};

// Later levels' counter: the elements of the chosen mass bin b* whose key
// carries the digits fixed so far add their mass to the global histogram of
// this level's digit.  Almost every element is rejected by two compares
// against b*'s logit interval, so the few masses go straight to global
// memory: no shared histogram and no block barrier.
struct DigitMasses {
  const TopPArgs* a;
  int b, i, which;
  unsigned long long* hist;  // this row slot's global histogram
  float cc, mc, xlo, xhi;
  uint32_t bstar, prefix;
  int hi_shift, nb;
  bool direct;      // level 1 of bf16 rows: the digit is the whole 16-bit key, less base16
  uint32_t base16;
  __device__ __forceinline__ void begin() {
    mc = scaled_max(row_max_warp(*a, b, i, which), cc);
    // the logits whose bin can be b*: the bin's edges d = b*/8 and (b*+1)/8
    // turned into logits and widened well past the rounding of d; the few
    // candidates take the exact bin test
    const float pad = (fabsf(mc / cc) + 1.f) * 1e-5f;
    xlo = -INFINITY;
    xhi = INFINITY;
    if (bstar > 0u) xhi = (mc - static_cast<float>(bstar) * 0.125f) / cc + pad;
    if (bstar < 255u) xlo = (mc - static_cast<float>(bstar + 1u) * 0.125f) / cc - pad;
    // bf16 logits carry 16 key bits.  When b*'s interval spans at most nb of
    // them, level 1 counts every key of b* in a bin of its own, and its
    // select fixes th outright (the key is monotone in the logit, so every
    // candidate's key lies in [key(xlo), key(xhi)]).
    direct = false;
    base16 = 0u;
    if (a->level == 1 && a->nlevels == 3 && bstar > 0u && bstar < 255u) {
      const uint32_t lo16 = logit_key(xlo) >> 16, hi16 = logit_key(xhi) >> 16;
      direct = hi16 - lo16 < static_cast<uint32_t>(nb);
      base16 = lo16;
    }
  }
  // Whether x can lie in b*: not -inf (no mass) and inside b*'s logit interval.
  __device__ __forceinline__ bool candidate(float x) const { return x != -INFINITY && x >= xlo && x <= xhi; }
  __device__ __forceinline__ void operator()(float x) const {
    if (candidate(x)) process(x);
  }
  __device__ __forceinline__ void pair(float x0, float x1) const {
    (*this)(x0);
    (*this)(x1);
  }
  // A candidate: the exact bin test, then its mass into its digit's bin.
  __device__ __forceinline__ void process(float x) const {
    const float d = __fmaf_rn(-x, cc, mc);
    const int bin = min(255, max(0, __float2int_rd(d * 8.f)));
    if (static_cast<uint32_t>(bin) != bstar) return;
    const uint32_t k = logit_key(x);
    if (a->level >= 2 && (k >> hi_shift) != prefix) return;
    const int digit = direct ? static_cast<int>((k >> 16) - base16)
                             : static_cast<int>((k >> a->shift) & static_cast<uint32_t>(nb - 1));
    const unsigned long long mass = mass_fixed(fast_exp2(-d));
    if (mass) atomicAdd(&hist[digit], mass);
  }
};

}  // namespace

// Level 0 over one chunk of one row.  Grid (chunk, row slot (i, which),
// request).  Each warp bins into its own copy; the copies are summed into the
// row's global histogram at the end.
template <typename E>
__global__ void __launch_bounds__(kHistThreads, 5) topp_hist_kernel(const TopPArgs a) {
  extern __shared__ __align__(16) uint32_t s_hist[];  // [warps][2][256]
  griddep_launch_dependents();
  const int c = blockIdx.x, i = blockIdx.y >> 1, which = blockIdx.y & 1, b = blockIdx.z;
  float T;
  if (!slot_active(a, b, i, which, &T)) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t* my_hist = s_hist + warp * 512;
  for (int d = lane; d < 512; d += 32) my_hist[d] = 0u;
  __syncwarp();
  const int lo = c * a.geo.chunk;
  MassBins f{&a, b, i, which, my_hist, kLog2e / T, 0.f};
  for_chunk<E>(a, slot_row<E>(a, b, i, which), lo, min(a.geo.chunk, a.geo.V - lo), f);
  __syncthreads();
  const size_t rs = (static_cast<size_t>(b) * (a.gmax + 1) + i) * 2 + which;
  unsigned long long* h = a.hist + rs * 256;
  for (int d = threadIdx.x; d < 256; d += kHistThreads) {
    unsigned long long m = 0ull;
    for (int q = 0; q < kHistThreads / 32; ++q)
      m += (static_cast<unsigned long long>(s_hist[q * 512 + 256 + d]) << 20) + s_hist[q * 512 + d];
    if (m) atomicAdd(&h[d], m);
  }
}

// One chunk c of row slot (b, i, which) at levels 1.. (the CTA's threads).
template <typename E>
__device__ __forceinline__ void refine_chunk(const TopPArgs& a, int c, int b, int i, int which, float T) {
  const size_t rs = (static_cast<size_t>(b) * (a.gmax + 1) + i) * 2 + which;
  const int lo = c * a.geo.chunk;
  DigitMasses f;
  f.a = &a;
  f.b = b;
  f.i = i;
  f.which = which;
  f.nb = 1 << a.bits;
  f.hist = a.hist + rs * f.nb;
  f.cc = kLog2e / T;
  f.hi_shift = a.shift + a.bits;  // key bits above this level's digit (levels >= 2: all decided)
  // b* and the prefix come from the previous selects: read after the wait
  struct Late {
    DigitMasses& g;
    size_t rs;
    int c;
    __device__ __forceinline__ void begin() {
      g.bstar = __ldcg(g.a->bstar + rs);
      g.prefix = g.a->level >= 2 ? __ldcg(g.a->prefix + rs) : 0u;
      g.begin();
      // level 1 of bf16 rows: tell the select how this row was counted (every
      // CTA of the row derives the same answer)
      if (g.a->level == 1 && g.a->nlevels == 3 && c == 0 && threadIdx.x == 0)
        g.a->prefix[rs] = g.direct ? (kDirectFlag | g.base16) : 0u;
    }
    __device__ __forceinline__ void operator()(float x) const { g(x); }
    __device__ __forceinline__ void pair(float x0, float x1) const { g.pair(x0, x1); }
  } late{f, rs, c};
  const E* row = slot_row<E>(a, b, i, which);
  const int n = min(a.geo.chunk, a.geo.V - lo);
  constexpr int kVec = Elem<E>::kVec;
  const int nvec = n / kVec;  // aligned rows: whole vectors
  // bf16 rows keep the per-element test (the mask measured 0.5 % slower there)
  if (sizeof(E) == 2 || !(a.geo.aligned && nvec <= kNVH * kHistThreads)) {
    for_chunk<E>(a, row, lo, n, late);
    return;
  }
  // fp32 rows: almost every element fails the candidate test, so the test
  // runs branch-free over the thread's elements into a bit mask, and the few
  // candidates are read again (from L1) and processed one by one: 397.5 to
  // 367.5 us per fp32 top-p round at B=64, gamma 4, V=128256, top_p 0.9.
  static_assert(kNVH * kVec <= 64, "one bit per element of a thread");
  const uint4* rv = reinterpret_cast<const uint4*>(row + lo);
  uint4 r[kNVH];
#pragma unroll
  for (int k = 0; k < kNVH; ++k) {
    const int v = threadIdx.x + k * kHistThreads;
    r[k] = v < nvec ? __ldg(rv + v) : Elem<E>::max_init();
  }
  griddep_wait();  // the records and the previous levels' digits are complete and visible
  late.begin();
  unsigned long long mask = 0ull;
#pragma unroll
  for (int k = 0; k < kNVH; ++k) {
    float x[kVec];
    Elem<E>::unpack(r[k], x);
#pragma unroll
    for (int e = 0; e < kVec; ++e)
      if (f.candidate(x[e])) mask |= 1ull << (k * kVec + e);
  }
  while (mask) {
    const int bit = __ffsll(static_cast<long long>(mask)) - 1;
    mask &= mask - 1ull;
    const int v = threadIdx.x + (bit / kVec) * kHistThreads;
    f.process(Elem<E>::to_float(row[lo + v * kVec + bit % kVec]));
  }
}

// Levels 1.. over one chunk of one row.  Grid as level 0.
template <typename E>
__global__ void __launch_bounds__(kHistThreads) topp_refine_kernel(const TopPArgs a) {
  griddep_launch_dependents();
  const int c = blockIdx.x, i = blockIdx.y >> 1, which = blockIdx.y & 1, b = blockIdx.z;
  float T;
  if (!slot_active(a, b, i, which, &T)) return;
  refine_chunk<E>(a, c, b, i, which, T);
}

// Level 2 of bf16 rows: only the row slots that level 1 left open (a few per
// cent at top_p 0.9), as (slot, chunk) items over a grid of one wave, so that
// the rows level 1 finished cost no CTAs.
template <typename E>
__global__ void __launch_bounds__(kHistThreads) topp_refine_open_kernel(const TopPArgs a) {
  griddep_launch_dependents();
  griddep_wait();  // level 1's select has listed the open rows
  const int NC = a.geo.nchunk, W = a.gmax + 1;
  const int items = static_cast<int>(__ldcg(a.todo_count)) * NC;
  for (int it = blockIdx.x; it < items; it += gridDim.x) {
    const int rs = static_cast<int>(__ldcg(a.todo + it / NC));
    const int which = rs & 1, i = (rs >> 1) % W, b = (rs >> 1) / W;
    float T;
    if (!slot_active(a, b, i, which, &T)) continue;  // listed rows are active; uniform over the CTA
    refine_chunk<E>(a, it % NC, b, i, which, T);
  }
}

// Thread t* of a select: the digit among its bins (cum = the mass above its
// top bin), then the level's outputs.
__device__ __forceinline__ void select_write(const TopPArgs& a, size_t rs, const unsigned long long (&v)[8],
                                             int per, unsigned long long cum, unsigned long long goal) {
  const int t = threadIdx.x;
  int d = t * per;
  unsigned long long dmass = v[0];
  bool found = false;
#pragma unroll
  for (int k = 7; k >= 0; --k) {
    if (k < per && !found) {
      if (cum + v[k] >= goal || k == 0) {
        d = t * per + k;
        dmass = v[k];
        found = true;
      } else {
        cum += v[k];
      }
    }
  }
  const uint32_t prefix = a.level >= 2 ? __ldcg(a.prefix + rs) : 0u;
  const uint32_t np = (prefix << a.bits) | static_cast<uint32_t>(d);
  const uint32_t word = a.level == 1 && a.nlevels == 3 ? __ldcg(a.prefix + rs) : 0u;
  if (word & kDirectFlag) {
    // bf16 row counted by whole keys: digit d is key16 - base16, so th is
    // that key's logit (low bits as at the last level) and the row is done
    uint32_t k = ((word & 0xFFFFu) + static_cast<uint32_t>(d)) << 16;
    if (!(k & 0x80000000u)) k |= 0xFFFFu;
    a.th[rs] = key_logit(k);
    a.z[rs] = static_cast<float>(static_cast<double>(cum + dmass) * (1.0 / 1099511627776.0));
    a.bstar[rs] = kRowDone;
  } else if (a.level == 0) {
    a.bstar[rs] = 255u - static_cast<uint32_t>(d);
    a.above[rs] = cum;
    a.goal[rs] = goal;
  } else if (a.level + 1 < a.nlevels) {
    a.prefix[rs] = np;
    a.above[rs] = cum;
    a.goal[rs] = goal;
    // bf16 rows still open after level 1: level 2 counts only these
    if (a.level == 1 && a.nlevels == 3) a.todo[atomicAdd(a.todo_count, 1u)] = static_cast<uint32_t>(rs);
  } else {
    // the key's undecided low bits (bf16: the 16 that a bf16 logit lacks)
    // are those of the smallest logit with these digits, so th is that
    // logit exactly
    uint32_t k = np << a.shift;
    if (a.shift && !(k & 0x80000000u)) k |= (1u << a.shift) - 1u;
    a.th[rs] = key_logit(k);
    a.z[rs] = static_cast<float>(static_cast<double>(cum + dmass) * (1.0 / 1099511627776.0));
  }
}

// The select of row slot rs, by every thread of the CTA (s_w: 8 words of
// shared memory, free again when it returns).  Thread t holds bins
// [t * per, t * per + per), per = bins / 256; a block suffix scan of the bin
// masses (the mass at or above each thread's first bin) finds the last thread
// whose suffix, with the mass above the level's range, reaches the goal, and
// that thread finds the digit among its bins.  At the last level it writes the
// threshold logit and the kept mass.
__device__ __forceinline__ void select_slot(const TopPArgs& a, size_t rs, unsigned long long* s_w) {
  const int nb = 1 << a.bits, per = nb >> 8;  // 1, 4 or 8
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const unsigned long long* h = a.hist + rs * nb + static_cast<size_t>(t) * per;
  unsigned long long v[8], ls = 0ull;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    v[k] = k < per ? __ldcg(h + k) : 0ull;
    ls += v[k];
  }
  // suffix sums: within the warp, then the later warps' totals
  unsigned long long suf = ls;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long x = __shfl_down_sync(0xFFFFFFFFu, suf, o);
    if (lane + o < 32) suf += x;
  }
  if (lane == 0) s_w[warp] = suf;
  __syncthreads();
  unsigned long long tot = 0ull;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    tot += s_w[w];
    if (w > warp) suf += s_w[w];
  }
  const unsigned long long above = a.level ? __ldcg(a.above + rs) : 0ull;
  unsigned long long goal;
  if (a.level == 0) {
    goal = static_cast<unsigned long long>(ceil(static_cast<double>(a.top_p) * static_cast<double>(tot)));
    // the product rounds in fp64 (tot may exceed 2^53): keep 1 <= goal <= tot
    goal = goal < tot ? goal : tot;
    if (goal == 0ull) goal = 1ull;
  } else {
    goal = __ldcg(a.goal + rs);
  }
  // the suffix does not grow with t, so the threads that reach the goal are
  // 0 .. t*: their count locates t*
  const int tstar = max(0, __syncthreads_count(above + suf >= goal) - 1);
  if (t == tstar) select_write(a, rs, v, per, above + suf - ls, goal);
  __syncthreads();  // s_w is read by every thread before a later row reuses it
}

// Select of one level: one CTA per row slot fixes the next digit.
__global__ void __launch_bounds__(256) topp_select_kernel(const TopPArgs a) {
  __shared__ unsigned long long s_w[8];
  griddep_launch_dependents();
  const int W = a.gmax + 1;
  const size_t rs = blockIdx.x;
  const int b = static_cast<int>(rs / (2 * W)), i = static_cast<int>((rs / 2) % W), which = static_cast<int>(rs & 1);
  float T;
  if (!slot_active(a, b, i, which, &T)) return;  // uniform over the CTA
  griddep_wait();  // the level's histograms are complete and visible
  if (a.level >= 2 && __ldcg(a.bstar + rs) == kRowDone) return;  // th fixed at level 1 (uniform)
  select_slot(a, rs, s_w);
}

// Select of level 2 of bf16 rows: one wave of CTAs over the rows level 1
// left open.
__global__ void __launch_bounds__(256) topp_select_open_kernel(const TopPArgs a) {
  __shared__ unsigned long long s_w[8];
  griddep_launch_dependents();
  griddep_wait();  // the level's histograms and the open rows' list are complete and visible
  const int n = static_cast<int>(__ldcg(a.todo_count));
  for (int r = blockIdx.x; r < n; r += gridDim.x) select_slot(a, __ldcg(a.todo + r), s_w);
}

template __global__ void topp_hist_kernel<uint16_t>(const TopPArgs);
template __global__ void topp_hist_kernel<float>(const TopPArgs);
template __global__ void topp_refine_kernel<uint16_t>(const TopPArgs);
template __global__ void topp_refine_kernel<float>(const TopPArgs);
template __global__ void topp_refine_open_kernel<uint16_t>(const TopPArgs);

cudaError_t launch_topp_level(const TopPArgs& a, int esize, cudaStream_t stream) {
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.geo.nchunk, 2 * (a.gmax + 1), a.B);
  cfg.blockDim = dim3(kHistThreads, 1, 1);
  // level 0: one histogram of 256 bins (two 32-bit words each) per warp
  cfg.dynamicSmemBytes = a.level == 0 ? static_cast<size_t>(8 * 256) * (kHistThreads / 32) : 0;
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (a.level == 0) {
    e = esize == 2 ? cudaLaunchKernelEx(&cfg, topp_hist_kernel<uint16_t>, a)
                   : cudaLaunchKernelEx(&cfg, topp_hist_kernel<float>, a);
  } else if (a.level == 2 && a.nlevels == 3 && esize == 2) {
    // one wave over the rows level 1 left open
    int dev = 0, sms = 0, per_sm = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, topp_refine_open_kernel<uint16_t>, kHistThreads, 0);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(static_cast<unsigned>(std::max(1, sms * std::max(1, per_sm))), 1, 1);
    e = cudaLaunchKernelEx(&cfg, topp_refine_open_kernel<uint16_t>, a);
  } else {
    e = esize == 2 ? cudaLaunchKernelEx(&cfg, topp_refine_kernel<uint16_t>, a)
                   : cudaLaunchKernelEx(&cfg, topp_refine_kernel<float>, a);
  }
  if (e != cudaSuccess) return e;
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = 0;
  if (a.level == 2 && a.nlevels == 3 && esize == 2) {
    // one wave over the rows level 1 left open
    int dev = 0, sms = 0, per_sm = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, topp_select_open_kernel, 256, 0);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(static_cast<unsigned>(std::max(1, sms * std::max(1, per_sm))), 1, 1);
    return cudaLaunchKernelEx(&cfg, topp_select_open_kernel, a);
  }
  const size_t nslots = static_cast<size_t>(a.B) * (a.gmax + 1) * 2;
  cfg.gridDim = dim3(static_cast<unsigned>(nslots), 1, 1);
  return cudaLaunchKernelEx(&cfg, topp_select_kernel, a);
}

}  // namespace ssdv
