// ssdv_verify.cu -- batched speculative-decoding verification.
//
// Method (speculative-decoding blog "投机解码 (Speculative Decoding)", section
// 3): at draft position i of request b, accept draft token x_i iff
// u_i < min(1, q_i(x_i) / p_i(x_i)); at the first rejection n emit one token
// drawn from (q_n - p_n)+ / sum (q_n - p_n)+ and stop (rollback of the rest,
// SSD-as-async-inference blog); if every draft token is accepted emit a bonus
// token drawn from q_gamma.  Greedy requests (T = 0) accept while x_i equals
// the target argmax.
//
// Two kernels on the caller's stream:
//  1. The streaming kernel: one CTA per (request, position, vocabulary chunk)
//     reduces the target chunk (and the draft chunk of a sampled draft
//     position) to a 32-byte record: max and sum of exponentials of each row,
//     or the target argmax of a greedy row.  Rows whose starts are 16-byte
//     aligned take the register form (stream_reg_kernel: every thread's
//     16-byte loads issued at once); other rows are staged into shared memory
//     (stream_kernel).  Every logit is read from HBM exactly once, by
//     short-lived CTAs.
//  2. sample_kernel: small CTAs, each covering a few pieces (128 vectors
//     each) of one request's draw row.  Before waiting for the records it
//     reads the draft tokens, their two logits and the uniforms (inputs).
//     Every CTA combines the request's records, takes every accept decision
//     and finds the first rejection n; then each warp loads its pieces of row
//     n (partly from L2: in plain calls the streaming kernel reads the low
//     positions last) -- target and draft for a residual draw, target for the
//     bonus draw -- and
//     publishes their weight sums.  The last warp to arrive sums the pieces in
//     order, finds the piece holding u * S, reloads that piece and scans it.
//
// A call runs as segments of requests, each a streaming + sampling pair, all
// launched with programmatic dependent launch.  The first streaming kernel's
// CTAs wait (griddepcontrol.wait) for the previous kernel on the stream before
// reading anything; every sampling CTA waits for its streaming kernel before
// reading the records.  Each kernel lets its dependents launch only after its
// own wait, so a later segment's streaming kernel launches after the first
// segment's CTAs saw the call's inputs complete, and may stream while the
// previous segment's sampling kernel runs: the segments use disjoint
// workspace rows.  A plain call never overlaps the work of the previous call;
// a pipelined call's streaming kernel runs beside the previous call's sampling
// kernel (only its first CTA waits), on the other workspace half.
#include <type_traits>

#include "ssdv_device.cuh"

namespace ssdv {

namespace {

__device__ __forceinline__ bool temperature_ok(float T) { return T == 0.f || (T >= 1e-6f && T <= 3.0e38f); }

// Residual weights scaled by Z_t: w = max(e_t - (Z_t/Z_d) e_d, 0) with
// e = exp2(x*c - fl(m*c)).  Its sum is Z_t * sum (q - p)+.
template <typename E>
struct ResidualW {
  float c, mct, mcd, kr;
  __device__ __forceinline__ void operator()(const float (&xt)[Elem<E>::kVec], const float (&xd)[Elem<E>::kVec],
                                             float (&w)[Elem<E>::kVec]) const {
    constexpr int kVec = Elem<E>::kVec;
    const F2 c2 = f2_make(c, c), nt = f2_make(-mct, -mct), nd = f2_make(-mcd, -mcd), nk = f2_make(-kr, -kr);
#pragma unroll
    for (int e = 0; e < kVec; e += 2) {
      const F2 et = f2_exp2(f2_fma(f2_make(xt[e], xt[e + 1]), c2, nt));
      const F2 ad = f2_fma(f2_make(xd[e], xd[e + 1]), c2, nd);
      const F2 ed = f2_exp2(ad);
      float w0, w1;
      f2_split(f2_fma(nk, ed, et), w0, w1);
      w[e] = fmaxf(w0, 0.f);
      w[e + 1] = fmaxf(w1, 0.f);
    }
  }
};

// sqrt.approx, as the Saguaro mix pass computes the weights that Zs sums.
__device__ __forceinline__ float sqrt_fast(float x) {
  float y;
  asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Residual weights when the draft tokens came from the Saguaro distribution
// p' = sqrt(p * max(r, 1e-8)) / Zs of their position (r = (q - p)+ / S, or q
// when S = 0): w = max(q - p', 0) in probability units.
template <typename E>
struct SagDraftW {
  float c, mct, mcd, kr;  // kr = Z_t / Z_d
  float inv_zt, inv_zd;   // 1 / Z_t, 1 / Z_d
  float inv_s;            // 1 / S in weight units (1 / Z_t when S = 0: r = q)
  float inv_zs;           // 1 / Zs
  int target_only;        // S = 0
  __device__ __forceinline__ void operator()(const float (&xt)[Elem<E>::kVec], const float (&xd)[Elem<E>::kVec],
                                             float (&w)[Elem<E>::kVec]) const {
#pragma unroll
    for (int e = 0; e < Elem<E>::kVec; ++e) {
      const float et = fast_exp2(fmaf(xt[e], c, -mct));
      const float ed = fast_exp2(fmaf(xd[e], c, -mcd));
      const float wa = target_only ? et : fmaxf(fmaf(-kr, ed, et), 0.f);
      const float ps = sqrt_fast(ed * inv_zd * fmaxf(wa * inv_s, 1e-8f)) * inv_zs;
      w[e] = fmaxf(fmaf(et, inv_zt, -ps), 0.f);
    }
  }
};

// Top-p: the residual of the truncated distributions, scaled by the target's
// kept mass: w = max(e_t [x_t >= th_t] - (Zt/Zd) e_d [x_d >= th_d], 0), with
// Zt, Zd the kept masses (the nuclei: logits at or above the thresholds).
template <typename E>
struct TopPResidualW {
  float c, mct, mcd, kr;  // kr = Zt / Zd of the kept masses
  float th_t, th_d;       // nucleus thresholds (logits)
  __device__ __forceinline__ void operator()(const float (&xt)[Elem<E>::kVec], const float (&xd)[Elem<E>::kVec],
                                             float (&w)[Elem<E>::kVec]) const {
#pragma unroll
    for (int e = 0; e < Elem<E>::kVec; ++e) {
      const float et = xt[e] >= th_t ? fast_exp2(fmaf(xt[e], c, -mct)) : 0.f;
      const float ed = xd[e] >= th_d ? fast_exp2(fmaf(xd[e], c, -mcd)) : 0.f;
      w[e] = fmaxf(fmaf(-kr, ed, et), 0.f);
    }
  }
};

// Top-p target weights: w = e_t on the nucleus, 0 elsewhere.
template <typename E>
struct TopPTargetW {
  float c, mct, th_t;
  __device__ __forceinline__ void operator()(const float (&xt)[Elem<E>::kVec], const float (&)[Elem<E>::kVec],
                                             float (&w)[Elem<E>::kVec]) const {
#pragma unroll
    for (int e = 0; e < Elem<E>::kVec; ++e) w[e] = xt[e] >= th_t ? fast_exp2(fmaf(xt[e], c, -mct)) : 0.f;
  }
};

// Target weights: w = e_t (proportional to q).
template <typename E>
struct TargetW {
  float c, mct;
  __device__ __forceinline__ void operator()(const float (&xt)[Elem<E>::kVec], const float (&)[Elem<E>::kVec],
                                             float (&w)[Elem<E>::kVec]) const {
#pragma unroll
    for (int e = 0; e < Elem<E>::kVec; ++e) w[e] = fast_exp2(fmaf(xt[e], c, -mct));
  }
};

// Copy one chunk (target and optionally draft) of a row that is not 16-byte
// aligned into shared memory with plain loads, padded with -inf to a whole
// vector; visible to every thread after the block barrier.
template <typename E>
__device__ __forceinline__ void stage_chunk(const Slice<E>& sl) {
  constexpr int kVec = Elem<E>::kVec;
  const int padded = sl.nvec * kVec;
  for (int e = threadIdx.x; e < padded; e += kThreads) {
    sl.st[e] = e < sl.n ? sl.gt[e] : Elem<E>::neg_inf();
    if (sl.gd) sl.sd[e] = e < sl.n ? sl.gd[e] : Elem<E>::neg_inf();
  }
  __syncthreads();
}

// One unit's combined row statistics (sampling kernel).
struct UnitStat {
  float tm, ts, dm, ds, av;
  int ai;
};

}  // namespace

// ---------------------------------------------------------------------------
// Kernel 1: per-chunk row statistics.
// ---------------------------------------------------------------------------
template <typename E>
__global__ void __launch_bounds__(kThreads) stream_kernel(const VerifyArgs a) {
  constexpr int kVec = Elem<E>::kVec;
  extern __shared__ __align__(128) uint8_t dyn_smem[];
  __shared__ float red_f[5 * kWarps];
  __shared__ int red_i[2 * kWarps];
  // The first segment of a call waits for the previous kernel on the stream
  // before it reads or writes anything.  A later segment reads logits that
  // were complete before the first segment's CTAs passed that wait (its
  // launch follows them through the chain of launches) and writes workspace
  // rows of its own requests, so only its first CTA waits -- for the previous
  // segment's sampling kernel -- which orders the completions of the chain.
  if (a.first || (blockIdx.x | blockIdx.y | blockIdx.z) == 0) griddep_wait();
  griddep_launch_dependents();  // the sampling kernel may become resident

  const ChunkGeometry& geo = a.geo;
  const int V = geo.V, NC = geo.nchunk, W = a.gmax + 1;
  // Dispatch order, positions from the last to the first.  Position-major
  // (chunk, request, position): the rows of the low positions -- where the
  // first rejection, and with it the sampling kernel's residual pass, usually
  // falls -- are read last and are still in L2 when the sampling kernel needs
  // them.  Request-major (chunk, position, request): one request's rows after
  // another.  Measured at B=64, gamma 4, V=128256 bf16: 29.06 against 29.46
  // us per pipelined call, 42.02 against 41.84 us per plain call; the Saguaro
  // round 0.940 against 0.945 ms; a ragged round 0.241 against 0.238 ms.
  const int c = blockIdx.x;
  const int b = a.req_major ? blockIdx.z : blockIdx.y;
  const int i = W - 1 - static_cast<int>(a.req_major ? blockIdx.y : blockIdx.z);
  const int tid = threadIdx.x;
  // The first CTA of each request clears the request's arrival counters for
  // the sampling kernel (which reads them only after this grid completes).
  if (i == 0 && c == 0 && tid < W) a.ticket[b * W + tid] = 0;

  const int g = a.gamma ? a.gamma[b] : a.gmax;
  const float T = a.temps ? a.temps[b] : a.temp_scalar;
  if (g < 0 || g > a.gmax || !temperature_ok(T) || i > g) return;  // padded rows are never read
  const bool greedy = (T == 0.f);
  const bool has_draft = !greedy && i < g;

  const int lo = c * geo.chunk;
  Slice<E> sl;
  sl.n = min(geo.chunk, V - lo);
  sl.nvec = (sl.n + kVec - 1) / kVec;
  sl.gt = static_cast<const E*>(a.target) + (static_cast<size_t>(b) * W + i) * V + lo;
  sl.gd = has_draft ? static_cast<const E*>(a.draft) + (static_cast<size_t>(b) * a.gmax + i) * V + lo : nullptr;
  sl.st = reinterpret_cast<E*>(dyn_smem);
  sl.sd = reinterpret_cast<E*>(dyn_smem + geo.row_smem);
  stage_chunk(sl);
  const uint4* vt = reinterpret_cast<const uint4*>(sl.st);
  const uint4* vd = reinterpret_cast<const uint4*>(sl.sd);

  const int warp = tid >> 5, lane = tid & 31;
  float4* rec = a.part + ((static_cast<size_t>(b) * W + i) * NC + c) * 2;
  if (greedy) {
    // Target argmax: each thread scans its vectors in index order (the first
    // of equal values wins), then a warp butterfly and thread 0 over warps.
    ArgMax am{-INFINITY, -1};
    for (int v = tid; v < sl.nvec; v += kThreads) {
      float xt[kVec];
      load_vec(sl.st, v, xt);
#pragma unroll
      for (int e = 0; e < kVec; ++e) {
        if (am.i < 0 || xt[e] > am.v) {
          am.v = xt[e];
          am.i = lo + v * kVec + e;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const ArgMax oa{__shfl_xor_sync(0xFFFFFFFFu, am.v, o), __shfl_xor_sync(0xFFFFFFFFu, am.i, o)};
      am = better_arg(am, oa);
    }
    if (lane == 0) {
      red_f[warp] = am.v;
      red_i[warp] = am.i;
    }
    __syncthreads();
    if (tid == 0) {
      ArgMax best{-INFINITY, -1};
      for (int w = 0; w < kWarps; ++w) best = better_arg(best, ArgMax{red_f[w], red_i[w]});
      rec[0] = make_float4(best.v, 0.f, -INFINITY, 0.f);
      rec[1] = make_float4(best.v, __int_as_float(best.i), 0.f, 0.f);
    }
    return;
  }

  // pass 1: the chunk maxima (packed max per thread, warp butterfly, and every
  // thread folds the eight warp maxima itself)
  uint4 pt = Elem<E>::max_init(), pd = Elem<E>::max_init();
  for (int v = tid; v < sl.nvec; v += kThreads) {
    pt = Elem<E>::max_acc(pt, vt[v]);
    if (has_draft) pd = Elem<E>::max_acc(pd, vd[v]);
  }
  float mt = Elem<E>::max_final(pt), md = Elem<E>::max_final(pd);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mt = fmaxf(mt, __shfl_xor_sync(0xFFFFFFFFu, mt, o));
    md = fmaxf(md, __shfl_xor_sync(0xFFFFFFFFu, md, o));
  }
  if (lane == 0) {
    red_f[warp] = mt;
    red_f[kWarps + warp] = md;
  }
  __syncthreads();
  mt = red_f[0];
  md = red_f[kWarps];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) {
    mt = fmaxf(mt, red_f[w]);
    md = fmaxf(md, red_f[kWarps + w]);
  }

  // pass 2: sums of exp2(x*c - fl(m*c)) against the chunk maxima
  const float cc = kLog2e / T;
  const F2 c2 = f2_make(cc, cc);
  float st = 0.f, sd = 0.f;
  if (mt != -INFINITY) {
    const float nm = -scaled_max(mt, cc);
    const F2 nm2 = f2_make(nm, nm);
    F2 acc = f2_make(0.f, 0.f);
    for (int v = tid; v < sl.nvec; v += kThreads) acc = f2_add(acc, Elem<E>::exp_sum(vt[v], c2, nm2));
    float a0, a1;
    f2_split(acc, a0, a1);
    st = a0 + a1;
  }
  if (has_draft && md != -INFINITY) {
    const float nm = -scaled_max(md, cc);
    const F2 nm2 = f2_make(nm, nm);
    F2 acc = f2_make(0.f, 0.f);
    for (int v = tid; v < sl.nvec; v += kThreads) acc = f2_add(acc, Elem<E>::exp_sum(vd[v], c2, nm2));
    float a0, a1;
    f2_split(acc, a0, a1);
    sd = a0 + a1;
  }
  st = warp_sum(st);
  sd = warp_sum(sd);
  if (lane == 0) {
    red_f[2 * kWarps + warp] = st;
    red_f[3 * kWarps + warp] = sd;
  }
  __syncthreads();
  if (tid == 0) {
    float s0 = 0.f, s1 = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      s0 += red_f[2 * kWarps + w];
      s1 += red_f[3 * kWarps + w];
    }
    rec[0] = make_float4(mt, s0, has_draft ? md : -INFINITY, s1);
    rec[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// ---------------------------------------------------------------------------
// Kernel 1, register form (rows 16-byte aligned, at most kNV vectors of a
// chunk row per thread).  Every thread issues the 16-byte loads of all its
// target and draft vectors at once, so a CTA keeps its whole chunk in flight
// with no staging buffer, no mbarrier and one block barrier.  A thread whose
// k-th vector lies past the chunk re-reads the chunk's last vector instead:
// harmless for the maxima, and left out of the sums.  Each warp takes the
// maxima of its lanes' vectors, sums exp2(x*c - fl(m_w*c)) against its own
// maxima m_w, and thread 0 folds the eight warps' (max, sum) pairs into the
// chunk record (the same record as the shared-memory form).
// ---------------------------------------------------------------------------
namespace {

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Resident CTAs per SM the register form is built for (registers bound it).
constexpr int reg_min_blocks(int nv) { return nv <= 4 ? 5 : nv <= 6 ? 4 : 3; }

}  // namespace

template <typename E, int kNV>
__global__ void __launch_bounds__(kThreads, reg_min_blocks(kNV)) stream_reg_kernel(const VerifyArgs a) {
  constexpr int kVec = Elem<E>::kVec;
  __shared__ float red_f[4 * kWarps];
  __shared__ int red_i[kWarps];
  // ordering with the previous kernel: as in the shared-memory form
  if (a.first || (blockIdx.x | blockIdx.y | blockIdx.z) == 0) griddep_wait();
  griddep_launch_dependents();

  const ChunkGeometry& geo = a.geo;
  const int V = geo.V, NC = geo.nchunk, W = a.gmax + 1;
  const int c = blockIdx.x;  // dispatch order as in the shared-memory form
  const int b = a.req_major ? blockIdx.z : blockIdx.y;
  const int i = W - 1 - static_cast<int>(a.req_major ? blockIdx.y : blockIdx.z);
  const int tid = threadIdx.x;
  if (i == 0 && c == 0 && tid < W) a.ticket[b * W + tid] = 0;

  const int g = a.gamma ? a.gamma[b] : a.gmax;
  const float T = a.temps ? a.temps[b] : a.temp_scalar;
  if (g < 0 || g > a.gmax || !temperature_ok(T) || i > g) return;  // padded rows are never read
  const bool greedy = (T == 0.f);
  const bool has_draft = !greedy && i < g;

  const int lo = c * geo.chunk;
  const int nvec = min(geo.chunk, V - lo) / kVec;  // aligned rows: whole vectors, at least one
  const E* rt_e = static_cast<const E*>(a.target) + (static_cast<size_t>(b) * W + i) * V + lo;
  const E* rd_e = has_draft ? static_cast<const E*>(a.draft) + (static_cast<size_t>(b) * a.gmax + i) * V + lo : nullptr;
  const uint4* gt = reinterpret_cast<const uint4*>(rt_e);
  const uint4* gd = reinterpret_cast<const uint4*>(rd_e);

  uint4 vt[kNV], vd[kNV];
#pragma unroll
  for (int k = 0; k < kNV; ++k) vt[k] = ld_stream(gt + min(tid + k * kThreads, nvec - 1));
  if (has_draft) {
#pragma unroll
    for (int k = 0; k < kNV; ++k) vd[k] = ld_stream(gd + min(tid + k * kThreads, nvec - 1));
  } else {
#pragma unroll
    for (int k = 0; k < kNV; ++k) vd[k] = Elem<E>::max_init();
  }

  const int warp = tid >> 5, lane = tid & 31;
  float4* rec = a.part + ((static_cast<size_t>(b) * W + i) * NC + c) * 2;
  if (greedy) {
    // target argmax: each thread in index order (the first of equal values
    // wins), then the warp butterfly and thread 0 over warps
    ArgMax am{-INFINITY, -1};
#pragma unroll
    for (int k = 0; k < kNV; ++k) {
      const int v = tid + k * kThreads;
      if (v < nvec) {
        float f[kVec];
        Elem<E>::unpack(vt[k], f);
#pragma unroll
        for (int e = 0; e < kVec; ++e)
          if (am.i < 0 || f[e] > am.v) am = ArgMax{f[e], lo + v * kVec + e};
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const ArgMax oa{__shfl_xor_sync(0xFFFFFFFFu, am.v, o), __shfl_xor_sync(0xFFFFFFFFu, am.i, o)};
      am = better_arg(am, oa);
    }
    if (lane == 0) {
      red_f[warp] = am.v;
      red_i[warp] = am.i;
    }
    __syncthreads();
    if (tid == 0) {
      ArgMax best{-INFINITY, -1};
      for (int w = 0; w < kWarps; ++w) best = better_arg(best, ArgMax{red_f[w], red_i[w]});
      rec[0] = make_float4(best.v, 0.f, -INFINITY, 0.f);
      rec[1] = make_float4(best.v, __int_as_float(best.i), 0.f, 0.f);
    }
    return;
  }

  // the warp's maxima (packed per thread, then a butterfly)
  uint4 pt = Elem<E>::max_init(), pd = Elem<E>::max_init();
#pragma unroll
  for (int k = 0; k < kNV; ++k) {
    pt = Elem<E>::max_acc(pt, vt[k]);
    pd = Elem<E>::max_acc(pd, vd[k]);
  }
  float mt = Elem<E>::max_final(pt), md = Elem<E>::max_final(pd);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mt = fmaxf(mt, __shfl_xor_sync(0xFFFFFFFFu, mt, o));
    md = fmaxf(md, __shfl_xor_sync(0xFFFFFFFFu, md, o));
  }
  // sums of exp2(x*c - fl(m_w*c)) against the warp's maxima
  const float cc = kLog2e / T;
  const F2 c2 = f2_make(cc, cc);
  float st = 0.f, sd = 0.f;
  if (mt != -INFINITY) {
    const float nm = -scaled_max(mt, cc);
    const F2 nm2 = f2_make(nm, nm);
    F2 acc = f2_make(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kNV; ++k)
      if (tid + k * kThreads < nvec) acc = f2_add(acc, Elem<E>::exp_sum(vt[k], c2, nm2));
    float a0, a1;
    f2_split(acc, a0, a1);
    st = a0 + a1;
  }
  if (md != -INFINITY) {
    const float nm = -scaled_max(md, cc);
    const F2 nm2 = f2_make(nm, nm);
    F2 acc = f2_make(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kNV; ++k)
      if (tid + k * kThreads < nvec) acc = f2_add(acc, Elem<E>::exp_sum(vd[k], c2, nm2));
    float a0, a1;
    f2_split(acc, a0, a1);
    sd = a0 + a1;
  }
  st = warp_sum(st);
  sd = warp_sum(sd);
  if (lane == 0) {
    red_f[warp] = mt;
    red_f[kWarps + warp] = st;
    red_f[2 * kWarps + warp] = md;
    red_f[3 * kWarps + warp] = sd;
  }
  __syncthreads();
  if (tid == 0) {
    MaxSum t{-INFINITY, 0.f}, d{-INFINITY, 0.f};
    for (int w = 0; w < kWarps; ++w) {
      t = combine_ms(t, MaxSum{red_f[w], red_f[kWarps + w]}, cc);
      d = combine_ms(d, MaxSum{red_f[2 * kWarps + w], red_f[3 * kWarps + w]}, cc);
    }
    rec[0] = make_float4(t.m, t.s, has_draft ? d.m : -INFINITY, d.s);
    rec[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// ---------------------------------------------------------------------------
// Kernel 2: decisions and the draw.
// ---------------------------------------------------------------------------
namespace {

__device__ void write_outputs(const VerifyArgs& a, int b, int n, int last, const int* tok_x) {
  const int W = a.gmax + 1;
  int32_t* out = a.out_tokens + static_cast<size_t>(b) * W;
  for (int k = 0; k < n; ++k) out[k] = tok_x[k];
  out[n] = last;
  for (int k = n + 1; k < W; ++k) out[k] = -1;
  a.n_accepted[b] = n;
}

__device__ void write_error(const VerifyArgs& a, int b) {
  const int W = a.gmax + 1;
  int32_t* out = a.out_tokens + static_cast<size_t>(b) * W;
  for (int k = 0; k < W; ++k) out[k] = -1;
  a.n_accepted[b] = -1;
}

}  // namespace


// ---------------------------------------------------------------------------
// Kernel 2: decisions and the draw, warp by warp.  A piece is 128 vectors
// (four 32-vector blocks) of a row; a warp takes geo.ppw consecutive pieces
// of one draw row and a CTA of kT2 threads kW2 such runs.  Every CTA of
// a request combines the request's records and takes the decisions (identical
// results); then each warp loads its pieces of row n -- target and draft for a
// residual draw, target for the bonus draw -- one round of loads per piece,
// publishes their weight sums and arrives once on the row's counter.  The last
// warp to arrive sums the pieces in order, finds the piece holding u * S,
// reloads that piece and scans it.
// ---------------------------------------------------------------------------
constexpr int kT2 = 128;  // threads of a sampling CTA
constexpr int kW2 = kT2 / 32;

// One warp: the draw at u * total from a row's piece sums (warp_locate_row);
// writes request b's outputs (tok_x: its first n draft tokens) and, with
// statistics, the CDF edges of the drawn token.
template <typename E, typename WFun>
__device__ __forceinline__ void warp_draw_row(const VerifyArgs& a, int b, int n, size_t pi_idx, const RowPieces& rp,
                                           float ures, const E* trow, const E* drow, bool aligned, const WFun& wfun,
                                           const int* tok_x) {
  const int lane = threadIdx.x & 31;
  const RowDraw d = warp_locate_row<E>(rp, ures, trow, drow, a.geo.V, aligned, wfun);
  if (lane == 0) {
    if (d.elem < 0 || !(rp.total > 0.0)) {
      write_error(a, b);
      atomicOr(a.status, 1 << SSD_ERR_DRAW);
    } else {
      if (a.stats) {
        float* st = a.stats + pi_idx * SSD_NSTAT_VERIFY;
        const double edge = ff_double(d.edge);
        st[8] = static_cast<float>(static_cast<double>(ures) - edge / rp.total);
        st[9] = static_cast<float>((edge + static_cast<double>(d.w)) / rp.total - static_cast<double>(ures));
      }
      write_outputs(a, b, n, d.elem, tok_x);
    }
  }
}

// Sampling modes: plain; draft tokens from the Saguaro distribution; top-p.
enum { kModePlain = 0, kModeSag = 1, kModeTopP = 2 };

template <typename E, int kMode>
__global__ void __launch_bounds__(kT2, 8) sample_kernel(const VerifyArgs a) {
  constexpr bool kSag = kMode == kModeSag, kTopP = kMode == kModeTopP;
  __shared__ UnitStat ust[SSD_MAX_GAMMA + 1];
  __shared__ int tok_x[SSD_MAX_GAMMA];
  __shared__ float tok_t[SSD_MAX_GAMMA], tok_d[SSD_MAX_GAMMA];
  __shared__ int sh_n, sh_bad, sh_sag_bad;
  __shared__ float sh_uacc[SSD_MAX_GAMMA + 1], sh_ures[SSD_MAX_GAMMA + 1];
  // [NP]: the last warp's copy of its row's piece sums.  A CTA's warps all
  // cover one draw row, and only one warp of the grid arrives last on a row,
  // so one copy per CTA suffices (less shared memory leaves more of the
  // unified L1/shared array to L1).
  extern __shared__ float s_pieces[];

  constexpr int kVec = Elem<E>::kVec;
  const ChunkGeometry& geo = a.geo;
  const int V = geo.V, NC = geo.nchunk, W = a.gmax + 1, NP = geo.npiece;
  const int pelems = kPieceVecs * kVec;
  const int c = blockIdx.x, pi = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // The next kernel may launch now.  The first CTA of every streaming kernel
  // waits for this grid to complete before it lets its own dependents launch,
  // so the next-but-one sampling kernel still starts after this one ends, and
  // a streaming kernel launched now writes only the other workspace half
  // (the previous sampling kernel, which used that half, has completed).
  griddep_launch_dependents();
  const int g = a.gamma ? a.gamma[b] : a.gmax;
  const float T = a.temps ? a.temps[b] : a.temp_scalar;
  const bool bad_gamma = g > a.gmax, bad_temp = !temperature_ok(T);
  if (g < 0 || bad_gamma || bad_temp) {  // padded or invalid request
    if (pi == 0 && c == 0 && tid == 0) {
      write_error(a, b);
      if (bad_gamma) atomicOr(a.status, 1 << SSD_ERR_GAMMA);
      if (bad_temp && g >= 0) atomicOr(a.status, 1 << SSD_ERR_TEMPERATURE);
    }
    return;
  }
  if (pi > g) return;
  const bool greedy = (T == 0.f);

  // Inputs only (overlaps the streaming kernel's tail; the kernel that wrote
  // them completed before any streaming CTA let this grid launch): the draft
  // tokens, and every position's accept and resample uniforms.
  if (warp == 0) {
    if (lane <= g) {
      const Draws d = unit_draws(a.seed, a.req_base + b, lane);
      sh_uacc[lane] = d.accept;
      sh_ures[lane] = d.resample;
    }
    bool bad = false;
    if (lane < g) {
      const int x = a.draft_tokens[static_cast<size_t>(b) * a.gmax + lane];
      bad = x < 0 || x >= V;
      tok_x[lane] = x;
      if (!bad && !greedy) {  // the two logits of the accept test
        tok_t[lane] = Elem<E>::to_float(static_cast<const E*>(a.target)[(static_cast<size_t>(b) * W + lane) * V + x]);
        tok_d[lane] = Elem<E>::to_float(static_cast<const E*>(a.draft)[(static_cast<size_t>(b) * a.gmax + lane) * V + x]);
      }
    }
    const unsigned anybad = __ballot_sync(0xFFFFFFFFu, bad);
    if (lane == 0) sh_bad = anybad != 0;
  }
  __syncthreads();
  if (sh_bad) {
    if (pi == 0 && c == 0 && tid == 0) {
      write_error(a, b);
      atomicOr(a.status, 1 << SSD_ERR_TOKEN_RANGE);
    }
    return;
  }
  griddep_wait();  // the streaming kernel's records are complete and visible

  // Row statistics of every position of the request, combined from the chunk
  // records (the same butterfly in every CTA: identical results).
  const float cc = greedy ? 1.f : kLog2e / T;
  // A warp combines positions warp, warp + kW2, ..., two at a time: both
  // positions' records are loaded (one round), then combined.
  for (int u0 = warp; u0 <= g; u0 += 2 * kW2) {
    float4 r0[2], r1[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int u = u0 + j * kW2;
      if (u <= g && lane < NC) {
        const float4* rec = a.part + ((static_cast<size_t>(b) * W + u) * NC + lane) * 2;
        r0[j] = __ldcg(rec);
        r1[j] = __ldcg(rec + 1);
      }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int u = u0 + j * kW2;
      if (u > g) break;
      MaxSum t{-INFINITY, 0.f}, d{-INFINITY, 0.f};
      ArgMax am{-INFINITY, -1};
      if (lane < NC) {
        t = MaxSum{r0[j].x, r0[j].y};
        d = MaxSum{r0[j].z, r0[j].w};
        if (greedy) am = ArgMax{r1[j].x, __float_as_int(r1[j].y)};
      }
      butterfly_stats(t, d, am, cc);
      if (lane == 0) ust[u] = UnitStat{t.m, t.s, d.m, d.s, am.v, am.i};
    }
  }
  __syncthreads();

  // Decisions: accept tests of positions 0..g-1 and the first rejection.
  if (warp == 0) {
    const float uacc = sh_uacc[min(lane, g)];
    bool acc = true;
    float ratio_acc = 1.f;
    int sag_bad = 0;
    if (lane < g) {
      const UnitStat s = ust[lane];
      if (greedy) {
        acc = tok_x[lane] == s.ai;
      } else if constexpr (kTopP) {
        // a = min(1, q'(x)/p'(x)) on the truncated distributions: q'(x) = 0
        // outside the target's nucleus (rejected), p'(x) = 0 outside the
        // draft's (accepted)
        const size_t rt = (static_cast<size_t>(b) * W + lane) * 2;
        const float tht = __ldcg(a.tp_th + rt), thd = __ldcg(a.tp_th + rt + 1);
        const float zt = __ldcg(a.tp_z + rt), zd = __ldcg(a.tp_z + rt + 1);
        const float q = tok_t[lane] >= tht ? fast_exp2(fmaf(tok_t[lane], cc, -scaled_max(s.tm, cc))) / zt : 0.f;
        const float p = tok_d[lane] >= thd ? fast_exp2(fmaf(tok_d[lane], cc, -scaled_max(s.dm, cc))) / zd : 0.f;
        if (p > 0.f) ratio_acc = fminf(1.f, q / p);
        acc = uacc < ratio_acc;
      } else if constexpr (kSag) {
        // a = min(1, q(x)/p'(x)), p'(x) = sqrt(p(x) max(r(x), 1e-8)) / Zs
        if (tok_d[lane] != -INFINITY) {
          const size_t uu = static_cast<size_t>(b) * W + lane;
          const double Sw = __ldcg(a.sag_S + uu);
          const float zs = __ldcg(a.sag_Zs + uu);
          const float et = fast_exp2(fmaf(tok_t[lane], cc, -scaled_max(s.tm, cc)));
          const float ed = fast_exp2(fmaf(tok_d[lane], cc, -scaled_max(s.dm, cc)));
          const float q = et / s.ts;
          const float r = Sw > 0.0 ? static_cast<float>(fmaxf(fmaf(-(s.ts / s.ds), ed, et), 0.f) / Sw) : q;
          const float ps = sqrt_fast(ed / s.ds * fmaxf(r, 1e-8f)) / zs;
          if (ps > 0.f) ratio_acc = fminf(1.f, q / ps);
          if (!(zs > 0.f)) sag_bad = 1;  // no Saguaro weight: nothing to verify against
        }
        acc = uacc < ratio_acc;
      } else {
        // a = min(1, q(x)/p(x)), the ratio as one exp2 of the exponent difference
        if (tok_d[lane] != -INFINITY) {
          const float lt = fmaf(tok_t[lane], cc, -scaled_max(s.tm, cc));
          const float ld = fmaf(tok_d[lane], cc, -scaled_max(s.dm, cc));
          ratio_acc = fminf(1.f, fast_exp2(lt - ld) * (s.ds / s.ts));
        }
        acc = uacc < ratio_acc;
      }
    }
    const unsigned rej = __ballot_sync(0xFFFFFFFFu, lane < g && !acc);
    const int n = rej ? __ffs(rej) - 1 : g;
    if (lane == 0) sh_n = n;
    if constexpr (kSag) {
      const int any_bad = __any_sync(0xFFFFFFFFu, sag_bad);
      if (lane == 0) sh_sag_bad = any_bad;
    }
    if (a.stats && c == 0 && lane == pi) {
      float* st = a.stats + (static_cast<size_t>(b) * W + pi) * SSD_NSTAT_VERIFY;
      const UnitStat s = ust[pi];
      if (greedy) {
        st[0] = s.av;
      } else {
        st[0] = s.tm;
        st[1] = logf(s.ts) - fmaf(s.tm, cc, -scaled_max(s.tm, cc)) * 0.6931471805599453f;
        if (pi < g) {
          const float mct = scaled_max(s.tm, cc), mcd = scaled_max(s.dm, cc);
          st[2] = s.dm;
          st[3] = logf(s.ds) - fmaf(s.dm, cc, -mcd) * 0.6931471805599453f;
          st[4] = fast_exp2(fmaf(tok_t[pi], cc, -mct)) / s.ts;
          st[5] = fast_exp2(fmaf(tok_d[pi], cc, -mcd)) / s.ds;
          st[7] = ratio_acc;
        }
      }
    }
  }
  __syncthreads();
  const int n = sh_n;
  const bool err_any = kSag && sh_sag_bad;
  if (greedy || err_any) {
    if (pi == 0 && c == 0 && tid == 0) {
      if (err_any) {
        write_error(a, b);
        atomicOr(a.status, 1 << SSD_ERR_DRAW);
      } else {
        write_outputs(a, b, n, ust[n].ai, tok_x);
      }
    }
    return;
  }

  // The draw row: row n (pos = pi for every row below g with statistics; the
  // bonus row g only when it is drawn from).
  const int pos = a.debug ? pi : n;
  if (pos == g && n != g) return;
  const bool residual = pos < g;
  const UnitStat s = ust[pos];
  const float mct = scaled_max(s.tm, cc);
  const float mcd = residual ? scaled_max(s.dm, cc) : 0.f;
  const float kr = residual ? s.ts / s.ds : 0.f;
  // the residual weights: (q - p)+ scaled by Z_t, (q - p')+ under Saguaro
  // sampling, or the truncated residual under top-p
  using RW = std::conditional_t<kSag, SagDraftW<E>, std::conditional_t<kTopP, TopPResidualW<E>, ResidualW<E>>>;
  using TW = std::conditional_t<kTopP, TopPTargetW<E>, TargetW<E>>;
  RW rw;
  TW tw;
  if constexpr (kTopP) {
    const size_t rt = (static_cast<size_t>(b) * W + pos) * 2;
    const float tht = __ldcg(a.tp_th + rt), zt = __ldcg(a.tp_z + rt);
    const float thd = residual ? __ldcg(a.tp_th + rt + 1) : 0.f, zd = residual ? __ldcg(a.tp_z + rt + 1) : 1.f;
    rw = TopPResidualW<E>{cc, mct, mcd, zt / zd, tht, thd};
    tw = TopPTargetW<E>{cc, mct, tht};
  } else {
    tw = TW{cc, mct};
  }
  if constexpr (kSag) {
    const size_t uu = static_cast<size_t>(b) * W + pos;
    const double Sw = residual ? __ldcg(a.sag_S + uu) : 0.0;
    const float zs = residual ? __ldcg(a.sag_Zs + uu) : 1.f;
    rw = SagDraftW<E>{cc, mct, mcd, kr, 1.f / s.ts, 1.f / s.ds,
                      Sw > 0.0 ? static_cast<float>(1.0 / Sw) : 1.f / s.ts, 1.f / zs, Sw > 0.0 ? 0 : 1};
  } else if constexpr (!kTopP) {
    rw = ResidualW<E>{cc, mct, mcd, kr};
  }
  const float ures = sh_ures[pos];
  const E* trow = static_cast<const E*>(a.target) + (static_cast<size_t>(b) * W + pos) * V;
  const E* drow = residual ? static_cast<const E*>(a.draft) + (static_cast<size_t>(b) * a.gmax + pos) * V : nullptr;
  const bool aligned = geo.aligned != 0;
  const size_t pi_idx = static_cast<size_t>(b) * W + pi;
  float* psum = a.psum + pi_idx * NP;

  // This warp's pieces (geo.ppw of them, one after the other): their weight
  // sums, then one arrival for all of them.  With the pieces ready (the
  // Saguaro residual pass summed every position's draw row the same way),
  // warp 0 of the request's one CTA draws from row n's sums directly.
  const int ppw = geo.ppw;
  const int p0 = (c * kW2 + warp) * ppw;
  if (a.pieces_ready) {
    if (warp != 0) return;
    psum = a.psum + (static_cast<size_t>(b) * W + pos) * NP;
  } else if (p0 >= NP) {
    return;
  }
  const int pn = min(ppw, NP - p0);
  bool last = a.pieces_ready != 0;
  if (!a.pieces_ready) {
    for (int j = 0; j < pn; ++j) {
      const int lo = (p0 + j) * pelems;
      PieceRows<E> pr;
      pr.load(trow + lo, drow ? drow + lo : nullptr, min(pelems, V - lo), aligned);
      const float ps = warp_sum(residual ? piece_lane_sum(pr, rw) : piece_lane_sum(pr, tw));
      if (lane == 0) psum[p0 + j] = ps;
    }
    int is_last = 0;
    if (lane == 0) is_last = ticket_add(a.ticket + pi_idx) == (NP + ppw - 1) / ppw - 1;
    last = __shfl_sync(0xFFFFFFFFu, is_last, 0) != 0;
  }
  if (!last) return;
  __syncwarp();  // the arrival's acquire (lane 0) orders every lane's loads below

  // The last warp: the piece sums in order, the piece holding u * S, then
  // that piece reloaded and scanned.
  if (lane == 0 && !a.pieces_ready) a.ticket[pi_idx] = 0;  // the last arrival of this call: reset for the next
  RowPieces rp;
  rp.load(psum, NP, s_pieces);
  if (a.stats && residual && lane == 0)
    a.stats[pi_idx * SSD_NSTAT_VERIFY + 6] = static_cast<float>(rp.total / static_cast<double>(s.ts));
  if (pos != n) return;
  if (residual && rp.total > 0.0) {
    warp_draw_row<E>(a, b, n, pi_idx, rp, ures, trow, drow, aligned, rw, tok_x);
  } else {
    // The bonus draw, or a zero residual mass (a rounding corner case): draw
    // from q_pos.  For the latter this warp first sums the target pieces.
    if (residual) {
      for (int q = 0; q < NP; ++q) {
        const int lo = q * pelems;
        PieceRows<E> pr;
        pr.load(trow + lo, nullptr, min(pelems, V - lo), aligned);
        const float ps = warp_sum(piece_lane_sum(pr, tw));
        if (lane == 0) psum[q] = ps;
      }
      __syncwarp();
      rp.load(psum, NP, s_pieces);
    }
    warp_draw_row<E>(a, b, n, pi_idx, rp, ures, trow, nullptr, aligned, tw, tok_x);
  }
}

// ---------------------------------------------------------------------------
// Small vocabularies (V <= kSmallV): one warp verifies one request in
// registers -- no records, no workspace, one launch.  Lane L holds elements
// [L*E, L*E + E) of a row, E = ceil(V / 32) <= 8, so lane sums in lane order
// are the row's running sums in index order.
// ---------------------------------------------------------------------------
namespace {

constexpr int kSmallE = kSmallV / 32;

template <typename E>
__device__ __forceinline__ void small_load(const E* row, int V, int lo, int ne, float (&x)[kSmallE]) {
#pragma unroll
  for (int k = 0; k < kSmallE; ++k) x[k] = (k < ne && lo + k < V) ? Elem<E>::to_float(row[lo + k]) : -INFINITY;
}

// Warp max and sum of exp2(x*c - fl(m*c)) of a row held as above.
__device__ __forceinline__ MaxSum small_stats(const float (&x)[kSmallE], float c) {
  float m = x[0];
#pragma unroll
  for (int k = 1; k < kSmallE; ++k) m = fmaxf(m, x[k]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  float s = 0.f;
  if (m != -INFINITY) {
    const float nm = -scaled_max(m, c);
#pragma unroll
    for (int k = 0; k < kSmallE; ++k) s += fast_exp2(fmaf(x[k], c, nm));
  }
  return MaxSum{m, warp_sum(s)};
}

// The element of a lane-blocked row (weights w) whose running weight first
// exceeds u * sum (float-float across lanes, fp32 within a lane), falling back
// to the last element with positive weight; -1 if every weight is zero.
__device__ __forceinline__ int small_draw(const float (&w)[kSmallE], int lo, float u) {
  const int lane = threadIdx.x & 31;
  float ls = 0.f;
#pragma unroll
  for (int k = 0; k < kSmallE; ++k) ls += w[k];
  const FF tot = ff_warp_sum(ls);
  if (!(tot.hi > 0.f)) return -1;
  const FF target = ff_mul(tot, u);
  FF before;
  const int L = lane_locate(ls, target, &before);
  int el = -1;
  if (lane == L) {
    const float t = ff_float(ff_sub(target, before));
    float acc = 0.f;
    bool done = false;
#pragma unroll
    for (int k = 0; k < kSmallE; ++k) {
      if (!done && w[k] > 0.f) {
        el = lo + k;
        done = t < acc + w[k];
      }
      acc += w[k];
    }
  }
  return __shfl_sync(0xFFFFFFFFu, el, L >= 0 ? L : 0);
}

// Element k (a runtime index) of a lane's block.
__device__ __forceinline__ float small_pick(const float (&x)[kSmallE], int k) {
  float v = -INFINITY;
#pragma unroll
  for (int j = 0; j < kSmallE; ++j)
    if (j == k) v = x[j];
  return v;
}

}  // namespace

template <typename E>
__global__ void __launch_bounds__(256) small_verify_kernel(const VerifyArgs a) {
  __shared__ int tok_s[8][SSD_MAX_GAMMA];
  griddep_wait();  // the previous kernel on the stream is complete (inputs and outputs)
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * 8 + warp;
  if (b >= a.B) return;
  const int V = a.geo.V, W = a.gmax + 1;
  const int g = a.gamma ? a.gamma[b] : a.gmax;
  const float T = a.temps ? a.temps[b] : a.temp_scalar;
  const bool bad_gamma = g > a.gmax, bad_temp = !temperature_ok(T);
  if (g < 0 || bad_gamma || bad_temp) {  // padded or invalid request
    if (lane == 0) {
      write_error(a, b);
      if (bad_gamma) atomicOr(a.status, 1 << SSD_ERR_GAMMA);
      if (bad_temp && g >= 0) atomicOr(a.status, 1 << SSD_ERR_TEMPERATURE);
    }
    return;
  }
  int* tok_x = tok_s[warp];
  bool bad = false;
  if (lane < g) {
    const int x = a.draft_tokens[static_cast<size_t>(b) * a.gmax + lane];
    bad = x < 0 || x >= V;
    tok_x[lane] = x;
  }
  if (__any_sync(0xFFFFFFFFu, bad)) {
    if (lane == 0) {
      write_error(a, b);
      atomicOr(a.status, 1 << SSD_ERR_TOKEN_RANGE);
    }
    return;
  }
  __syncwarp();
  const int ne = (V + 31) / 32;
  const int lo = lane * ne;
  const E* trows = static_cast<const E*>(a.target) + static_cast<size_t>(b) * W * V;
  const E* drows = static_cast<const E*>(a.draft) + static_cast<size_t>(b) * a.gmax * V;
  const uint32_t rid = static_cast<uint32_t>(a.req_base + b);
  int n = g, last = -1;
  float xt[kSmallE], xd[kSmallE], w[kSmallE];
  if (T == 0.f) {
    // greedy: accept while the draft token is the target argmax
    for (int i = 0; i <= g; ++i) {
      small_load(trows + static_cast<size_t>(i) * V, V, lo, ne, xt);
      ArgMax am{-INFINITY, -1};
#pragma unroll
      for (int k = 0; k < kSmallE; ++k)
        if (k < ne && lo + k < V && (am.i < 0 || xt[k] > am.v)) am = ArgMax{xt[k], lo + k};
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const ArgMax oa{__shfl_xor_sync(0xFFFFFFFFu, am.v, o), __shfl_xor_sync(0xFFFFFFFFu, am.i, o)};
        am = better_arg(am, oa);
      }
      if (i == g || tok_x[i] != am.i) {
        n = i;
        last = am.i;
        break;
      }
    }
  } else {
    const float c = kLog2e / T;
    for (int i = 0; i < g; ++i) {
      small_load(trows + static_cast<size_t>(i) * V, V, lo, ne, xt);
      small_load(drows + static_cast<size_t>(i) * V, V, lo, ne, xd);
      const MaxSum st = small_stats(xt, c), sd = small_stats(xd, c);
      const int x = tok_x[i];
      const float lx_t = __shfl_sync(0xFFFFFFFFu, small_pick(xt, x % ne), x / ne);
      const float lx_d = __shfl_sync(0xFFFFFFFFu, small_pick(xd, x % ne), x / ne);
      const float mct = scaled_max(st.m, c), mcd = scaled_max(sd.m, c);
      float ratio = 1.f;  // a -inf draft logit: p(x) = 0, accepted
      if (lx_d != -INFINITY)
        ratio = fminf(1.f, fast_exp2(fmaf(lx_t, c, -mct) - fmaf(lx_d, c, -mcd)) * (sd.s / st.s));
      const Draws dr = unit_draws(a.seed, rid, i);
      if (dr.accept < ratio) continue;
      // rejected at i: the correction from (q_i - p_i)+ (q_i if that is empty)
      const float kr = st.s / sd.s;
#pragma unroll
      for (int k = 0; k < kSmallE; ++k)
        w[k] = fmaxf(fmaf(-kr, fast_exp2(fmaf(xd[k], c, -mcd)), fast_exp2(fmaf(xt[k], c, -mct))), 0.f);
      const float ures = dr.resample;
      last = small_draw(w, lo, ures);
      if (last < 0) {
#pragma unroll
        for (int k = 0; k < kSmallE; ++k) w[k] = fast_exp2(fmaf(xt[k], c, -mct));
        last = small_draw(w, lo, ures);
      }
      n = i;
      break;
    }
    if (n == g) {  // every draft token accepted: the bonus from q_g
      small_load(trows + static_cast<size_t>(g) * V, V, lo, ne, xt);
      const MaxSum st = small_stats(xt, c);
      const float mct = scaled_max(st.m, c);
#pragma unroll
      for (int k = 0; k < kSmallE; ++k) w[k] = fast_exp2(fmaf(xt[k], c, -mct));
      last = small_draw(w, lo, unit_draws(a.seed, rid, g).resample);
    }
  }
  if (lane == 0) {
    if (last < 0) {
      write_error(a, b);
      atomicOr(a.status, 1 << SSD_ERR_DRAW);
    } else {
      write_outputs(a, b, n, last, tok_x);
    }
  }
}

template __global__ void small_verify_kernel<uint16_t>(const VerifyArgs);
template __global__ void small_verify_kernel<float>(const VerifyArgs);

template __global__ void stream_kernel<uint16_t>(const VerifyArgs);
template __global__ void stream_kernel<float>(const VerifyArgs);
template __global__ void stream_reg_kernel<uint16_t, 4>(const VerifyArgs);
template __global__ void stream_reg_kernel<float, 4>(const VerifyArgs);
template __global__ void stream_reg_kernel<uint16_t, 6>(const VerifyArgs);
template __global__ void stream_reg_kernel<float, 6>(const VerifyArgs);
template __global__ void stream_reg_kernel<uint16_t, 8>(const VerifyArgs);
template __global__ void stream_reg_kernel<float, 8>(const VerifyArgs);
template __global__ void sample_kernel<uint16_t, kModePlain>(const VerifyArgs);
template __global__ void sample_kernel<float, kModePlain>(const VerifyArgs);
template __global__ void sample_kernel<uint16_t, kModeSag>(const VerifyArgs);
template __global__ void sample_kernel<float, kModeSag>(const VerifyArgs);
template __global__ void sample_kernel<uint16_t, kModeTopP>(const VerifyArgs);
template __global__ void sample_kernel<float, kModeTopP>(const VerifyArgs);

__global__ void uniforms_kernel(uint64_t seed, int B, int W, float* out) {
  const long long n = static_cast<long long>(B) * W;
  for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < n;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    const Draws d = unit_draws(seed, static_cast<int>(t / W), static_cast<int>(t % W));
    out[3 * t + 0] = d.accept;
    out[3 * t + 1] = d.resample;
    out[3 * t + 2] = d.saguaro;
  }
}

cudaError_t launch_uniforms(uint64_t seed, int B, int W, float* out, cudaStream_t stream) {
  const long long n = static_cast<long long>(B) * W;
  const int blocks = static_cast<int>(n / 256 + 1 < 4096 ? n / 256 + 1 : 4096);
  uniforms_kernel<<<blocks, 256, 0, stream>>>(seed, B, W, out);
  return cudaGetLastError();
}

namespace {

// The register form takes aligned rows whose chunks hold at most kRegVecs
// vectors per thread.
bool use_register_stream(const ChunkGeometry& geo, int vec) {
  return geo.aligned && geo.chunk <= kRegVecs * kThreads * vec;
}

// cudaFuncSetAttribute once per (kernel, size) on the current device.
cudaError_t ensure_smem(const void* fn, int smem_bytes, int* cached) {
  if (*cached == smem_bytes) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e == cudaSuccess) *cached = smem_bytes;
  return e;
}

template <typename E>
cudaError_t launch_stream_t(const VerifyArgs& a, int smem_bytes, cudaStream_t stream) {
  static thread_local int dev_cached = -1, smem1 = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev != dev_cached) {
    smem1 = -1;
    dev_cached = dev;
  }
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t c1 = {};
  c1.gridDim = a.req_major ? dim3(a.geo.nchunk, a.gmax + 1, a.B) : dim3(a.geo.nchunk, a.B, a.gmax + 1);
  c1.blockDim = dim3(kThreads, 1, 1);
  c1.stream = stream;
  c1.attrs = pdl;
  c1.numAttrs = 1;
  if (use_register_stream(a.geo, Elem<E>::kVec)) {
    c1.dynamicSmemBytes = 0;
    const int per = (a.geo.chunk / Elem<E>::kVec + kThreads - 1) / kThreads;  // vectors per thread
    if (per <= 4) return cudaLaunchKernelEx(&c1, stream_reg_kernel<E, 4>, a);
    if (per <= 6) return cudaLaunchKernelEx(&c1, stream_reg_kernel<E, 6>, a);
    return cudaLaunchKernelEx(&c1, stream_reg_kernel<E, 8>, a);
  }
  e = ensure_smem(reinterpret_cast<const void*>(&stream_kernel<E>), smem_bytes, &smem1);
  if (e != cudaSuccess) return e;
  c1.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  return cudaLaunchKernelEx(&c1, stream_kernel<E>, a);
}

template <typename E>
cudaError_t launch_sample_t(const VerifyArgs& a, cudaStream_t stream) {
  const int P = a.debug ? a.gmax + 1 : 1;  // position slots of the sampling grid
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = a.pieces_ready ? dim3(1, 1, a.B)
                               : dim3((a.geo.npiece + kW2 * a.geo.ppw - 1) / (kW2 * a.geo.ppw), P, a.B);
  cfg.blockDim = dim3(kT2, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(a.geo.npiece) * sizeof(float);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return a.sag_S  ? cudaLaunchKernelEx(&cfg, sample_kernel<E, kModeSag>, a)
         : a.tp_th ? cudaLaunchKernelEx(&cfg, sample_kernel<E, kModeTopP>, a)
                   : cudaLaunchKernelEx(&cfg, sample_kernel<E, kModePlain>, a);
}

template <typename E>
cudaError_t launch_verify_t(const VerifyArgs& a, int smem_bytes, cudaStream_t stream) {
  cudaError_t e = launch_stream_t<E>(a, smem_bytes, stream);
  if (e != cudaSuccess) return e;
  return launch_sample_t<E>(a, stream);
}

}  // namespace

cudaError_t launch_verify(const VerifyArgs& a, int esize, int smem_bytes, cudaStream_t stream) {
  return esize == 2 ? launch_verify_t<uint16_t>(a, smem_bytes, stream) : launch_verify_t<float>(a, smem_bytes, stream);
}

cudaError_t launch_small_verify(const VerifyArgs& a, int esize, cudaStream_t stream) {
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.B + 7) / 8, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  return esize == 2 ? cudaLaunchKernelEx(&cfg, small_verify_kernel<uint16_t>, a)
                    : cudaLaunchKernelEx(&cfg, small_verify_kernel<float>, a);
}

cudaError_t launch_sample(const VerifyArgs& a, int esize, cudaStream_t stream) {
  return esize == 2 ? launch_sample_t<uint16_t>(a, stream) : launch_sample_t<float>(a, stream);
}

cudaError_t launch_stream(const VerifyArgs& a, int esize, int smem_bytes, cudaStream_t stream) {
  return esize == 2 ? launch_stream_t<uint16_t>(a, smem_bytes, stream) : launch_stream_t<float>(a, smem_bytes, stream);
}

}  // namespace ssdv
