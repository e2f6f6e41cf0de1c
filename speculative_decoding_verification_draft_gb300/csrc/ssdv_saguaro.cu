// ssdv_saguaro.cu -- Saguaro pre-speculation.
//
// Method (notes "Speculative Speculative Decoding (Saguaro)", section 3.1 bonus
// prediction by top-k, section 3.2 Saguaro sampling): while the target verifies,
// predict the bonus token for every possible acceptance length j = 0..gamma.
// For j < gamma the bonus would be drawn from the residual
// r_j = (q_j - p_j)+ / sum (q_j - p_j)+ (q_j when that mass is zero); for
// j = gamma from q_gamma.  Outputs per (request, j): the k largest entries of
// r_j, and one sample from p_saguaro proportional to
// sqrt(p_D(v) * max(r_j(v), 1e-8)), p_D = p_j (q_gamma at j = gamma).
//
// Three kernels per segment of requests, chained by programmatic dependent
// launch (each waits for its predecessor before reading its results):
//  1. the verification streaming kernel: per-chunk (max, sum) records of every
//     target row and draft row -- one HBM read of every logit;
//  2. residual_kernel: warps over 128-vector pieces of every unit's rows: the
//     residual weights (target weights at j = gamma), the pieces' sums and a
//     top-4 (k <= 4) or top-8 per lane, merged per warp; the last warp of a
//     unit fixes S_j and merges the top-k;
//  3. mix_kernel: warps over the same pieces: the Saguaro weights, their
//     piece sums; the last warp of a unit draws the token (and, when S_j = 0,
//     merges the top-k of q_j instead).
// A round that also verifies (the fused call) runs the verification's
// sampling kernel between 2 and 3: the residual kernel's piece sums of unit
// (b, j) are, in the same order and arithmetic, the sums of the weights the
// verification draws from when n = j, so the draw needs no pass over the rows.
#include "ssdv_device.cuh"

namespace ssdv {

namespace {

template <typename E>
struct PassAW {  // residual (scaled by Z_t) or target weights
  float c, mct, mcd, kr;
  int target_only;
  __device__ __forceinline__ void operator()(const float (&xt)[Elem<E>::kVec], const float (&xd)[Elem<E>::kVec],
                                             float (&w)[Elem<E>::kVec]) const {
#pragma unroll
    for (int e = 0; e < Elem<E>::kVec; ++e) {
      const float et = fast_exp2(fmaf(xt[e], c, -mct));
      if (target_only) {
        w[e] = et;
      } else {
        const float ed = fast_exp2(fmaf(xd[e], c, -mcd));
        w[e] = fmaxf(fmaf(-kr, ed, et), 0.f);
      }
    }
  }
};

// sqrt.approx: one MUFU operation (relative error within about 2^-22),
// against several instructions for the IEEE-rounded square root.
__device__ __forceinline__ float sqrt_fast(float x) {
  float y;
  asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Saguaro mix weights sqrt(p_D * max(r, 1e-8)) in probability units.
template <typename E>
struct MixW {
  float c, mct, mcd, kr;
  int target_only;  // r from q instead of the residual
  int pd_target;    // p_D = q (bonus position) instead of p
  float inv_s;      // 1 / (sum of the pass-A weights)
  float inv_zp;     // 1 / Z of p_D's row
  __device__ __forceinline__ void operator()(const float (&xt)[Elem<E>::kVec], const float (&xd)[Elem<E>::kVec],
                                             float (&w)[Elem<E>::kVec]) const {
#pragma unroll
    for (int e = 0; e < Elem<E>::kVec; ++e) {
      const float et = fast_exp2(fmaf(xt[e], c, -mct));
      float ed = 0.f;
      if (!pd_target) ed = fast_exp2(fmaf(xd[e], c, -mcd));
      const float wa = target_only ? et : fmaxf(fmaf(-kr, ed, et), 0.f);
      const float r = wa * inv_s;
      const float pd = (pd_target ? et : ed) * inv_zp;
      w[e] = sqrt_fast(pd * fmaxf(r, 1e-8f));
    }
  }
};


constexpr int kS = 128;  // threads of a residual / mix CTA
constexpr int kSW = kS / 32;
// Resident CTAs per SM the residual and mix kernels are built for.  Both
// passes wait on HBM with few warps per SM, so fp32 rows trade registers for
// warps: 6 and 8 CTAs per SM (80 and 64 registers, against 90 and 80 left
// free), measured 0.999 against 1.070 ms per Saguaro round at B=256, gamma 6,
// V=152064.  bf16 rows measured slower that way and keep the allocation they
// get unconstrained (the residual kernel without top-k: 72 registers, 7 CTAs
// per SM; with top-k: up to 128, 4; the mix kernel: 80, 6).
// kK: the per-lane top-k list (4 when k <= 4, else 8): the shorter list frees
// registers for a seventh fp32 CTA per SM.
template <typename E, int kKey, int kK = 8>
constexpr int resid_min_blocks() { return sizeof(E) == 4 ? (kK <= 4 ? 7 : 6) : (kKey == 0 ? 7 : 4); }
template <typename E>
constexpr int mix_min_blocks() { return sizeof(E) == 4 ? 8 : 6; }
constexpr int kTopK = SSD_MAX_TOPK;  // every warp tracks the top 8; the first k are written

// Row statistics of unit u from its chunk records (one warp; lanes < NC hold
// a record each), valid in every lane: target and draft (max, sum).
__device__ __forceinline__ void unit_stats(const SagArgs& a, size_t u, float c, MaxSum* t, MaxSum* d) {
  const int lane = threadIdx.x & 31, NC = a.geo.nchunk;
  MaxSum tt{-INFINITY, 0.f}, dd{-INFINITY, 0.f};
  ArgMax am{-INFINITY, -1};
  if (lane < NC) {
    const float4 r0 = __ldcg(a.part + (u * NC + lane) * 2);
    tt = MaxSum{r0.x, r0.y};
    dd = MaxSum{r0.z, r0.w};
  }
  butterfly_stats(tt, dd, am, c);
  *t = tt;
  *d = dd;
}

// One warp: the k best of n candidates (value, index), descending, the lower
// index first among equal values; every lane gets the list.  Candidates are
// distinct, so each round takes the best one ranking after the previous pick;
// empty slots (index 0x7FFFFFFF) rank after everything.
__device__ __forceinline__ void merge_candidates(const float* cv, const int* ci, int n, int k, float* ov, int* oi) {
  const int lane = threadIdx.x & 31;
  float lv = INFINITY;
  int li = -1;
  for (int s = 0; s < k; ++s) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
    for (int q = lane; q < n; q += 32) {
      const float v = cv[q];
      const int i = ci[q];
      if (i == 0x7FFFFFFF || !ranks_before(lv, li, v, i)) continue;  // taken already, or empty
      if (ranks_before(v, i, bv, bi)) {
        bv = v;
        bi = i;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
      const int i2 = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
      if (ranks_before(v2, i2, bv, bi)) {
        bv = v2;
        bi = i2;
      }
    }
    ov[s] = bv;
    oi[s] = bi;
    lv = bv;
    li = bi;
  }
}

// Top-k keys of the residual kernel: the weights, or (draft source) the
// draft logits -- the target logits at the bonus position.
enum { kKeyNone = 0, kKeyWeight = 1, kKeyLogit = 2 };

// This warp's pieces: weight sums into psum, top-8 (by kKey) into the unit's
// candidate slots.  Returns true in the last warp of the unit to arrive
// (every lane), after which the other warps' sums are visible.
template <typename E, typename WFun, int kKey, int kK = kTopK>
__device__ __forceinline__ bool unit_pieces(const SagArgs& a, size_t u, int wi, const E* trow, const E* drow,
                                            const WFun& wfun, float* psum, int32_t* ticket) {
  constexpr bool kTop = kKey != kKeyNone;
  constexpr int kVec = Elem<E>::kVec;
  const int lane = threadIdx.x & 31;
  const int V = a.geo.V, NP = a.geo.npiece, ppw = a.geo.ppw;
  const int pelems = kPieceVecs * kVec;
  const int p0 = wi * ppw;
  const int pn = min(ppw, NP - p0);
  TopK<kK, kKey == kKeyLogit> tk;
  tk.init();
  // tau: the k-th largest of the lanes' best keys so far.  The warp holds k
  // elements at or above it, so a smaller key is not among the row's k
  // largest and is not pushed.
  const bool key_target = drow == nullptr;
  float tau = -INFINITY;
  for (int j = 0; j < pn; ++j) {
    const int lo = (p0 + j) * pelems;
    PieceRows<E> pr;
    pr.load(trow + lo, drow ? drow + lo : nullptr, min(pelems, V - lo), a.geo.aligned != 0);
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float w[kVec];
      pr.weights(k, wfun, w);
      s += pair_sum(w);
      if constexpr (kTop) {
        float key[kVec];
        if constexpr (kKey == kKeyLogit) {
          float xt[kVec], xd[kVec];
          pr.raw(k, xt, xd);
#pragma unroll
          for (int e = 0; e < kVec; ++e) key[e] = key_target ? xt[e] : xd[e];
        } else {
#pragma unroll
          for (int e = 0; e < kVec; ++e) key[e] = w[e];
        }
        const int base = lo + (4 * lane + k) * kVec;
        float km = key[0];  // elements past V are padding: weight 0, logit -inf
#pragma unroll
        for (int e = 1; e < kVec; ++e) km = fmaxf(km, key[e]);
        if (__any_sync(0xFFFFFFFFu, km >= tau)) {
#pragma unroll
          for (int e = 0; e < kVec; ++e)
            if (key[e] >= tau && base + e < V) tk.push(key[e], base + e);
        }
      }
    }
    s = warp_sum(s);
    if (lane == 0) psum[u * NP + p0 + j] = s;
    // tau after the first piece, then after every fourth: an older tau is
    // still a lower bound on the warp's k-th key, so it only lets a few more
    // elements be pushed
    if (kTop && (j == 0 || (j & 3) == 3)) {
      float x = tk.v[0];
      for (int r = 0; r < a.k; ++r) {
        float m = x;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        tau = m;
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, x == m);
        if (lane == __ffs(hit) - 1) x = -INFINITY;
      }
    }
  }
  if constexpr (kTop) {
    float mv[kK];
    int mi[kK];
    warp_merge_topk(tk, mv, mi);
    if (lane < kTopK) {  // the warp's kTopK candidate slots; past kK they stay empty
      float v = -INFINITY;
      int i = 0x7FFFFFFF;
#pragma unroll
      for (int r = 0; r < kK; ++r)
        if (lane == r) {
          v = mv[r];
          i = mi[r];
        }
      a.cand_v[(u * a.npw + wi) * kTopK + lane] = v;
      a.cand_i[(u * a.npw + wi) * kTopK + lane] = i;
      __threadfence();  // before lane 0's arrival below publishes them
    }
    __syncwarp();
  }
  int is_last = 0;
  if (lane == 0) is_last = ticket_add(ticket + u) == a.npw - 1;
  const bool last = __shfl_sync(0xFFFFFFFFu, is_last, 0) != 0;
  if (last) __syncwarp();  // the arrival's acquire (lane 0) orders every lane's loads after it
  return last;
}

// The last warp of a unit: its top-k from the warps' candidates (copied to
// shared memory first) into bonus_topk, and the statistics of slots 0 and k-1
// as probabilities: weights over `total`, or (logit keys) exp2(x*c - mc) / z.
__device__ __forceinline__ void write_topk(const SagArgs& a, size_t u, double total, float* s_cv, int* s_ci,
                                          float* st, bool logit_keys = false, float c = 0.f, float mc = 0.f,
                                          float z = 1.f) {
  const int lane = threadIdx.x & 31;
  const int n = a.npw * kTopK;
  for (int q = lane; q < n; q += 32) {
    s_cv[q] = __ldcg(a.cand_v + u * n + q);
    s_ci[q] = __ldcg(a.cand_i + u * n + q);
  }
  __syncwarp();
  float ov[kTopK];
  int oi[kTopK];
  merge_candidates(s_cv, s_ci, n, a.k, ov, oi);
  if (lane == 0) {
    int32_t* out = a.bonus_topk + u * a.k;
    for (int s = 0; s < a.k; ++s) out[s] = (oi[s] >= 0 && oi[s] < a.geo.V) ? oi[s] : -1;
    if (st && logit_keys) {
      st[5] = fast_exp2(fmaf(ov[0], c, -mc)) / z;
      st[6] = fast_exp2(fmaf(ov[a.k - 1], c, -mc)) / z;
    } else if (st) {
      st[5] = static_cast<float>(static_cast<double>(ov[0]) / total);
      st[6] = static_cast<float>(static_cast<double>(ov[a.k - 1]) / total);
    }
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// The residual pass of one unit, warp by warp: residual weights (target
// weights at j = gamma), their piece sums and the warps' top-8 candidates;
// the last warp of the unit fixes S_j, writes the row statistics and merges
// the top-k.  s4 = the unit's row statistics (target max, sum, draft max,
// sum).  Returns true in (every lane of) that last warp.
// ---------------------------------------------------------------------------
template <typename E, int kKey, int kK = kTopK>
__device__ __forceinline__ bool residual_unit(const SagArgs& a, int b, int j, int wi, uint8_t* dyn_smem,
                                              float4 s4) {
  const int W = a.g + 1;
  const int lane = threadIdx.x & 31;
  const size_t u = static_cast<size_t>(b) * W + j;
  const bool bonus = (j == a.g);
  const float c = kLog2e / a.temperature;
  const int V = a.geo.V;
  const E* trow = static_cast<const E*>(a.target) + u * V;
  const E* drow = bonus ? nullptr : static_cast<const E*>(a.draft) + (static_cast<size_t>(b) * a.g + j) * V;
  const PassAW<E> wf{c, scaled_max(s4.x, c), bonus ? 0.f : scaled_max(s4.z, c), bonus ? 0.f : s4.y / s4.w,
                     bonus ? 1 : 0};
  if (!unit_pieces<E, PassAW<E>, kKey, kK>(a, u, wi, trow, drow, wf, a.psum2, a.ticket2)) return false;

  // The last warp: S_j, and the top-k unless the residual is empty (then the
  // mix pass takes the top-k of q_j).
  RowPieces rp;
  // one copy per CTA: a CTA's warps all cover unit u, whose last warp is unique
  float* s_pieces = reinterpret_cast<float*>(dyn_smem);
  rp.load(a.psum2 + u * a.geo.npiece, a.geo.npiece, s_pieces);
  const double S = rp.total;
  float* st = a.stats ? a.stats + u * SSD_NSTAT_SAGUARO : nullptr;
  if (lane == 0) {
    a.rowstat[u] = s4;
    a.rowsum[u] = S;
    a.ticket3[u] = 0;  // the mix kernel's counter starts at zero (read after this grid completes)
    a.ticket2[u] = 0;  // the last arrival: zero again for a later kernel of the call
    if (st) {
      st[0] = logf(s4.y) - fmaf(s4.x, c, -scaled_max(s4.x, c)) * 0.6931471805599453f;
      st[1] = bonus ? NAN : logf(s4.w) - fmaf(s4.z, c, -scaled_max(s4.z, c)) * 0.6931471805599453f;
      st[2] = bonus ? 1.f : static_cast<float>(S / static_cast<double>(s4.y));
    }
  }
  const bool logit_keys = kKey == kKeyLogit;
  if (kKey != kKeyNone && (logit_keys || bonus || S > 0.0)) {
    __syncwarp();
    float* s_cv = reinterpret_cast<float*>(dyn_smem) + a.geo.npiece;
    int* s_ci = reinterpret_cast<int*>(s_cv + a.npw * kTopK);
    // logit keys report p_j (q_gamma at the bonus position) of the slots
    const float mc = bonus ? scaled_max(s4.x, c) : scaled_max(s4.z, c);
    write_topk(a, u, S, s_cv, s_ci, st, logit_keys, c, mc, bonus ? s4.y : s4.w);
  }
  return true;
}

// ---------------------------------------------------------------------------
// The mix pass of one unit, warp by warp: the Saguaro weights
// sqrt(p_D max(r, 1e-8)) and their piece sums; the last warp of the unit
// keeps Zs, draws the token (and, when S_j = 0, merges the top-k of q_j).
// Reads the residual pass's row statistics and S_j of the unit.  Returns true
// in (every lane of) that last warp.
// ---------------------------------------------------------------------------
template <typename E>
__device__ __forceinline__ bool mix_unit(const SagArgs& a, int b, int j, int wi, uint8_t* dyn_smem) {
  const int W = a.g + 1;
  const int lane = threadIdx.x & 31;
  const size_t u = static_cast<size_t>(b) * W + j;
  const bool bonus = (j == a.g);
  const float c = kLog2e / a.temperature;
  const float4 s4 = __ldcg(a.rowstat + u);
  const double S = __ldcg(a.rowsum + u);
  const bool target_only = bonus || !(S > 0.0);  // r = q_j: the bonus position or an empty residual
  const double sum_a = (bonus || S > 0.0) ? S : static_cast<double>(s4.y);
  const int V = a.geo.V;
  const E* trow = static_cast<const E*>(a.target) + u * V;
  const E* drow = bonus ? nullptr : static_cast<const E*>(a.draft) + (static_cast<size_t>(b) * a.g + j) * V;
  const float mct = scaled_max(s4.x, c), mcd = bonus ? 0.f : scaled_max(s4.z, c);
  const MixW<E> mw{c, mct, mcd, bonus ? 0.f : s4.y / s4.w, target_only ? 1 : 0, bonus ? 1 : 0,
                   static_cast<float>(1.0 / sum_a), bonus ? 1.f / s4.y : 1.f / s4.w};
  // empty residual with the residual as the top-k source: the top-k of q_j
  // is taken here
  const bool fallback = a.k > 0 && a.topk_src == 0 && !bonus && !(S > 0.0);
  if (!unit_pieces<E, MixW<E>, kKeyNone>(a, u, wi, trow, drow, mw, a.psum3, a.ticket3)) return false;

  // The last warp: Zs, the draw, and (empty residual) the top-k of q_j.
  RowPieces rp;
  float* s_pieces = reinterpret_cast<float*>(dyn_smem);  // one copy per CTA, as in the residual pass
  rp.load(a.psum3 + u * a.geo.npiece, a.geo.npiece, s_pieces);
  if (a.zsum && lane == 0) a.zsum[u] = static_cast<float>(rp.total);
  if (!a.saguaro_tokens) return true;  // the normaliser is all a later kernel needs
  const float u_sag = unit_draws(a.seed, a.req_base + b, j).saguaro;
  const RowDraw d = warp_locate_row<E>(rp, u_sag, trow, drow, V, a.geo.aligned != 0, mw);
  float* st = a.stats ? a.stats + u * SSD_NSTAT_SAGUARO : nullptr;
  if (lane == 0) {
    const bool ok = d.elem >= 0 && rp.total > 0.0;
    a.saguaro_tokens[u] = ok ? d.elem : -1;
    if (!ok) atomicOr(a.status, 1 << SSD_ERR_DRAW);
    if (st && ok) {
      st[3] = static_cast<float>(rp.total);
      st[4] = static_cast<float>(static_cast<double>(d.w) / rp.total);
      const double edge = ff_double(d.edge);
      st[8] = static_cast<float>(static_cast<double>(u_sag) - edge / rp.total);
      st[9] = static_cast<float>((edge + static_cast<double>(d.w)) / rp.total - static_cast<double>(u_sag));
    }
  }
  if (fallback) {
    // Empty residual: r_j = q_j, whose top-k is the top-k of the target
    // logits.  This warp scans the row once (a rare corner case).
    TopK<kTopK> tk;
    tk.init();
    const int pelems = kPieceVecs * Elem<E>::kVec;
    const PassAW<E> tw{c, mct, 0.f, 0.f, 1};
    for (int q = 0; q < a.geo.npiece; ++q) {
      const int lo = q * pelems;
      PieceRows<E> pr;
      pr.load(trow + lo, nullptr, min(pelems, V - lo), a.geo.aligned != 0);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float w[Elem<E>::kVec];
        pr.weights(k, tw, w);
        const int base = lo + (4 * lane + k) * Elem<E>::kVec;
#pragma unroll
        for (int e = 0; e < Elem<E>::kVec; ++e)
          if (base + e < V) tk.push(w[e], base + e);
      }
    }
    float mv[kTopK];
    int mi[kTopK];
    warp_merge_topk<kTopK>(tk, mv, mi);
    if (lane == 0) {
      int32_t* out = a.bonus_topk + u * a.k;
      for (int s = 0; s < a.k; ++s) out[s] = (mi[s] >= 0 && mi[s] < V) ? mi[s] : -1;
      if (st) {
        st[5] = static_cast<float>(static_cast<double>(mv[0]) / static_cast<double>(s4.y));
        st[6] = static_cast<float>(static_cast<double>(mv[a.k - 1]) / static_cast<double>(s4.y));
      }
    }
  }
  return true;
}

// The row statistics of unit u into sh (warp 0), visible to the CTA after the
// barrier.
__device__ __forceinline__ void cta_unit_stats(const SagArgs& a, size_t u, float4* sh) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    MaxSum t, d;
    unit_stats(a, u, kLog2e / a.temperature, &t, &d);
    if (lane == 0) *sh = make_float4(t.m, t.s, d.m, d.s);
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Kernel 2: residual sums and top-k.  Grid (warp groups, j, request).
// ---------------------------------------------------------------------------
template <typename E, int kKey, int kK>
__global__ void __launch_bounds__(kS, resid_min_blocks<E, kKey, kK>()) residual_kernel(const SagArgs a) {
  extern __shared__ __align__(16) uint8_t dyn_smem[];
  __shared__ float4 sh_stats;
  griddep_launch_dependents();  // the mix kernel may become resident (it waits for this grid)
  const int W = a.g + 1, j = blockIdx.y, b = blockIdx.z;
  const int wi = blockIdx.x * kSW + (threadIdx.x >> 5);
  griddep_wait();  // the streaming kernel's records are complete and visible
  cta_unit_stats(a, static_cast<size_t>(b) * W + j, &sh_stats);
  if (wi >= a.npw) return;
  residual_unit<E, kKey, kK>(a, b, j, wi, dyn_smem, sh_stats);
}

// ---------------------------------------------------------------------------
// Kernel 3: the Saguaro mix and its draw.  Grid as kernel 2.
// ---------------------------------------------------------------------------
template <typename E>
__global__ void __launch_bounds__(kS, mix_min_blocks<E>()) mix_kernel(const SagArgs a) {
  extern __shared__ __align__(16) uint8_t dyn_smem[];
  griddep_launch_dependents();  // the next kernel may become resident (it waits for this grid)
  const int j = blockIdx.y, b = blockIdx.z;
  const int wi = blockIdx.x * kSW + (threadIdx.x >> 5);
  if (wi >= a.npw) return;
  griddep_wait();  // the residual kernel's sums are complete and visible
  mix_unit<E>(a, b, j, wi, dyn_smem);
}

template __global__ void residual_kernel<uint16_t, kKeyWeight, 8>(const SagArgs);
template __global__ void residual_kernel<float, kKeyWeight, 8>(const SagArgs);
template __global__ void residual_kernel<uint16_t, kKeyLogit, 8>(const SagArgs);
template __global__ void residual_kernel<float, kKeyLogit, 8>(const SagArgs);
template __global__ void residual_kernel<uint16_t, kKeyWeight, 4>(const SagArgs);
template __global__ void residual_kernel<float, kKeyWeight, 4>(const SagArgs);
template __global__ void residual_kernel<uint16_t, kKeyLogit, 4>(const SagArgs);
template __global__ void residual_kernel<float, kKeyLogit, 4>(const SagArgs);
template __global__ void residual_kernel<uint16_t, kKeyNone, 8>(const SagArgs);
template __global__ void residual_kernel<float, kKeyNone, 8>(const SagArgs);
template __global__ void mix_kernel<uint16_t>(const SagArgs);
template __global__ void mix_kernel<float>(const SagArgs);

namespace {

template <typename E>
cudaError_t launch_saguaro_t(const SagArgs& a, cudaStream_t stream, int passes) {
  const int smem = static_cast<int>(sizeof(float) * a.geo.npiece + 8 * a.npw * kTopK);
  const int key = a.k == 0 ? kKeyNone : (a.topk_src == 1 ? kKeyLogit : kKeyWeight);
  const bool short_list = a.k <= 4;  // per-lane top-4 lists: 72 registers, 7 fp32 CTAs per SM
  const void* resid =
      key == kKeyLogit    ? (short_list ? reinterpret_cast<const void*>(&residual_kernel<E, kKeyLogit, 4>)
                                        : reinterpret_cast<const void*>(&residual_kernel<E, kKeyLogit, 8>))
      : key == kKeyWeight ? (short_list ? reinterpret_cast<const void*>(&residual_kernel<E, kKeyWeight, 4>)
                                        : reinterpret_cast<const void*>(&residual_kernel<E, kKeyWeight, 8>))
                          : reinterpret_cast<const void*>(&residual_kernel<E, kKeyNone, 8>);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(resid, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&mix_kernel<E>),
                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.npw + kSW - 1) / kSW, a.nj, a.B);
  cfg.blockDim = dim3(kS, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  if (passes & kSagResidual) {
    cudaError_t e;
    if (key == kKeyLogit)
      e = short_list ? cudaLaunchKernelEx(&cfg, residual_kernel<E, kKeyLogit, 4>, a)
                     : cudaLaunchKernelEx(&cfg, residual_kernel<E, kKeyLogit, 8>, a);
    else if (key == kKeyWeight)
      e = short_list ? cudaLaunchKernelEx(&cfg, residual_kernel<E, kKeyWeight, 4>, a)
                     : cudaLaunchKernelEx(&cfg, residual_kernel<E, kKeyWeight, 8>, a);
    else
      e = cudaLaunchKernelEx(&cfg, residual_kernel<E, kKeyNone, 8>, a);
    if (e != cudaSuccess) return e;
  }
  return (passes & kSagMix) ? cudaLaunchKernelEx(&cfg, mix_kernel<E>, a) : cudaSuccess;
}

}  // namespace

// ---------------------------------------------------------------------------
// The cache check (SSD notes, sections 3.3 and 4.1): a round's outcome hits
// the pre-speculated cache when its correction / bonus token is among the
// predicted bonus tokens for its acceptance length.  One CTA over the batch.
// ---------------------------------------------------------------------------
constexpr int kCheckThreads = 1024;

__global__ void __launch_bounds__(kCheckThreads) cache_check_kernel(const int32_t* bonus_topk,
                                                                   const int32_t* out_tokens,
                                                                   const int32_t* n_accepted, int B, int W, int k,
                                                                   int32_t* hit, int32_t* n_hits) {
  __shared__ int wsum[kCheckThreads / 32];
  griddep_wait();  // the verification and Saguaro outputs are complete and visible
  int count = 0;
  for (int b = threadIdx.x; b < B; b += kCheckThreads) {
    const int n = n_accepted[b];
    int h = -1;
    if (n >= 0 && n < W) {
      const int tok = out_tokens[static_cast<size_t>(b) * W + n];
      const int32_t* row = bonus_topk + (static_cast<size_t>(b) * W + n) * k;
      for (int s = k - 1; s >= 0; --s)
        if (tok >= 0 && row[s] == tok) h = s;
    }
    if (hit) hit[b] = h;
    count += h >= 0 ? 1 : 0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) count += __shfl_xor_sync(0xFFFFFFFFu, count, o);
  if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = count;
  __syncthreads();
  if (threadIdx.x == 0 && n_hits) {
    int t = 0;
    for (int w = 0; w < kCheckThreads / 32; ++w) t += wsum[w];
    n_hits[0] = t;
  }
}

cudaError_t launch_cache_check(const int32_t* bonus_topk, const int32_t* out_tokens, const int32_t* n_accepted, int B,
                               int W, int k, int32_t* hit, int32_t* n_hits, cudaStream_t stream) {
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, 1);
  cfg.blockDim = dim3(kCheckThreads, 1, 1);
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, cache_check_kernel, bonus_topk, out_tokens, n_accepted, B, W, k, hit, n_hits);
}

cudaError_t launch_saguaro(const SagArgs& a, int esize, cudaStream_t stream, int passes) {
  return esize == 2 ? launch_saguaro_t<uint16_t>(a, stream, passes) : launch_saguaro_t<float>(a, stream, passes);
}

}  // namespace ssdv
