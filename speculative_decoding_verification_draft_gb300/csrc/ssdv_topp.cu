// ssdv_topp.cu -- top-p (nucleus) thresholds for verification.
//
// Verification composes with top-p when both sides truncate the same way (the
// verification blog's closing remark and its section on matching sampling
// parameters): each target and draft row keeps the tokens whose logit is at
// least th, the largest logit value whose upper set {x >= th} holds at least
// top_p of the row's probability mass (tokens tied with the last one needed
// are kept), renormalised.
//
// th is found per row by a radix select over a monotone 32-bit key of the
// logit, from the high digits down (bf16: two 8-bit digits of the 16 bits that
// matter; fp32: digits of 11, 11 and 10 bits).  Each level is a histogram pass
// over the rows' chunks -- the mass exp2(x c - fl(m c)) of every element whose
// key matches the digits fixed so far, in fixed point (2^-40 units) so that
// the integer sums are exact and the same on every run whatever the order of
// the atomics -- then a select pass (one warp per row) that fixes the next
// digit: the largest one whose upper mass reaches ceil(top_p * total).
#include "ssdv_device.cuh"

namespace ssdv {

namespace {

constexpr float kFix = 1099511627776.0f;  // 2^40
constexpr int kHistThreads = 256;

__device__ __forceinline__ bool temperature_ok_tp(float T) { return T == 0.f || (T >= 1e-6f && T <= 3.0e38f); }

// Monotone key of a logit (-0 taken as +0, as the comparisons x >= th do).
__device__ __forceinline__ uint32_t logit_key(float x) {
  const uint32_t b = __float_as_uint(x + 0.f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
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

// Histogram of one level over one chunk of one row.  Grid (chunk, row slot
// (i, which), request).
template <typename E>
__global__ void __launch_bounds__(kHistThreads) topp_hist_kernel(const TopPArgs a) {
  extern __shared__ __align__(16) unsigned long long s_hist[];
  __shared__ float sh_m;
  griddep_launch_dependents();
  const int W = a.gmax + 1, NC = a.geo.nchunk, V = a.geo.V;
  const int c = blockIdx.x, i = blockIdx.y >> 1, which = blockIdx.y & 1, b = blockIdx.z;
  float T;
  if (!slot_active(a, b, i, which, &T)) return;
  const int nb = 1 << a.bits;
  for (int d = threadIdx.x; d < nb; d += kHistThreads) s_hist[d] = 0ull;
  griddep_wait();  // the records (and the previous level's digits) are complete and visible
  const size_t rs = (static_cast<size_t>(b) * W + i) * 2 + which;
  if (threadIdx.x < 32) {
    // the row maximum: the largest chunk maximum of the row's records
    float m = -INFINITY;
    for (int q = threadIdx.x; q < NC; q += 32) {
      const float4 r0 = __ldcg(a.part + ((static_cast<size_t>(b) * W + i) * NC + q) * 2);
      m = fmaxf(m, which ? r0.z : r0.x);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (threadIdx.x == 0) sh_m = m;
  }
  __syncthreads();
  const float cc = kLog2e / T;
  const float nmc = -scaled_max(sh_m, cc);
  const uint32_t prefix = a.level ? __ldcg(a.prefix + rs) : 0u;
  const int hi_shift = a.shift + a.bits;  // bits above this level's digit: all decided
  const E* row = which ? static_cast<const E*>(a.draft) + (static_cast<size_t>(b) * a.gmax + i) * V
                       : static_cast<const E*>(a.target) + (static_cast<size_t>(b) * W + i) * V;
  const int lo = c * a.geo.chunk;
  const int n = min(a.geo.chunk, V - lo);
  for (int e = threadIdx.x; e < n; e += kHistThreads) {
    const float x = Elem<E>::to_float(row[lo + e]);
    if (x == -INFINITY) continue;  // no mass
    const uint32_t k = logit_key(x);
    if (hi_shift < 32 && (k >> hi_shift) != prefix) continue;
    const unsigned long long mass = __float2ull_rn(fast_exp2(fmaf(x, cc, nmc)) * kFix);
    if (mass) atomicAdd(&s_hist[(k >> a.shift) & (nb - 1)], mass);
  }
  __syncthreads();
  unsigned long long* h = a.hist + rs * nb;
  for (int d = threadIdx.x; d < nb; d += kHistThreads)
    if (s_hist[d]) atomicAdd(&h[d], s_hist[d]);
}

// Select of one level: one warp per row slot fixes the next digit.  At the
// last level it writes the threshold logit and the kept mass.
__global__ void __launch_bounds__(256) topp_select_kernel(const TopPArgs a) {
  griddep_launch_dependents();
  const int W = a.gmax + 1;
  const int lane = threadIdx.x & 31;
  const size_t rs = static_cast<size_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const size_t nslots = static_cast<size_t>(a.B) * W * 2;
  if (rs >= nslots) return;
  const int b = static_cast<int>(rs / (2 * W)), i = static_cast<int>((rs / 2) % W), which = static_cast<int>(rs & 1);
  float T;
  if (!slot_active(a, b, i, which, &T)) return;
  griddep_wait();  // the level's histograms are complete and visible
  const int nb = 1 << a.bits, per = nb / 32;
  const unsigned long long* h = a.hist + rs * nb;
  // lane L holds bins [L * per, L * per + per)
  unsigned long long ls = 0ull;
  for (int k = 0; k < per; ++k) ls += __ldcg(h + lane * per + k);
  unsigned long long above = a.level ? __ldcg(a.above + rs) : 0ull;
  unsigned long long goal;
  if (a.level == 0) {
    unsigned long long tot = ls;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xFFFFFFFFu, tot, o);
    goal = static_cast<unsigned long long>(ceil(static_cast<double>(a.top_p) * static_cast<double>(tot)));
    // the product rounds in fp64 (tot may exceed 2^53): keep 1 <= goal <= tot
    goal = goal < tot ? goal : tot;
    if (goal == 0ull) goal = 1ull;
  } else {
    goal = __ldcg(a.goal + rs);
  }
  // suffix sums over lanes: the mass of bins at or above lane L's first bin
  unsigned long long suf = ls;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_down_sync(0xFFFFFFFFu, suf, o);
    if (lane + o < 32) suf += t;
  }
  // the highest lane whose suffix (with the mass above the prefix range)
  // reaches the target holds the digit
  const unsigned hitm = __ballot_sync(0xFFFFFFFFu, above + suf >= goal);
  const int L = hitm ? 31 - __clz(hitm) : 0;
  const unsigned long long above_lane = above + __shfl_sync(0xFFFFFFFFu, suf - ls, L);
  if (lane == L) {
    // within the lane, from its top bin down
    unsigned long long cum = above_lane;
    int d = lane * per;
    unsigned long long dmass = 0ull;
    for (int k = per - 1; k >= 0; --k) {
      const unsigned long long m = __ldcg(h + lane * per + k);
      if (cum + m >= goal || k == 0) {
        d = lane * per + k;
        dmass = m;
        break;
      }
      cum += m;
    }
    const uint32_t prefix = a.level ? __ldcg(a.prefix + rs) : 0u;
    const uint32_t np = (prefix << a.bits) | static_cast<uint32_t>(d);
    if (a.level + 1 < a.nlevels) {
      a.prefix[rs] = np;
      a.above[rs] = cum;
      a.goal[rs] = goal;
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
}

template __global__ void topp_hist_kernel<uint16_t>(const TopPArgs);
template __global__ void topp_hist_kernel<float>(const TopPArgs);

cudaError_t launch_topp_level(const TopPArgs& a, int esize, cudaStream_t stream) {
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.geo.nchunk, 2 * (a.gmax + 1), a.B);
  cfg.blockDim = dim3(kHistThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(8) << a.bits;
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  cudaError_t e = esize == 2 ? cudaLaunchKernelEx(&cfg, topp_hist_kernel<uint16_t>, a)
                             : cudaLaunchKernelEx(&cfg, topp_hist_kernel<float>, a);
  if (e != cudaSuccess) return e;
  const size_t nslots = static_cast<size_t>(a.B) * (a.gmax + 1) * 2;
  cfg.gridDim = dim3(static_cast<unsigned>((nslots + 7) / 8), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, topp_select_kernel, a);
}

}  // namespace ssdv
