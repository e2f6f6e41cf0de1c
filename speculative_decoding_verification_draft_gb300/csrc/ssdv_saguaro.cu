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
// One cluster per (request, j) unit, slices resident in shared memory: the
// statistics pass reads HBM once; the residual pass (sum and top-k), the mix
// pass (normaliser) and the inverse-CDF search run on-chip.
#include "ssdv_device.cuh"

namespace ssdv {

namespace {

constexpr int kTopK = SSD_MAX_TOPK;  // every unit tracks the top 8; the first k are written

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
      w[e] = sqrtf(pd * fmaxf(r, 1e-8f));
    }
  }
};

}  // namespace

template <typename E>
__global__ void __launch_bounds__(kThreads) saguaro_kernel(const SaguaroArgs a) {
  constexpr int kVec = Elem<E>::kVec;
  extern __shared__ __align__(128) uint8_t dyn_smem[];
  __shared__ __align__(8) uint64_t bars[kMaxStages];
  __shared__ __align__(8) uint64_t xbar[kNumX];
  __shared__ __align__(16) Inbox inbox;
  __shared__ __align__(16) float cta_top_v[kTopK];
  __shared__ __align__(16) int cta_top_i[kTopK];
  __shared__ float red_f[5 * kWarps];
  __shared__ int red_i[2 * kWarps];
  __shared__ float wsum[kWarps];
  __shared__ float wtop_v[kWarps][kTopK];
  __shared__ int wtop_i[kWarps][kTopK];
  __shared__ int sh_warp, sh_result, sh_owner, sh_err;
  __shared__ double sh_base, sh_local, sh_total, sh_prefix, sh_edge;
  __shared__ float sh_edge_w;
  __shared__ float sh_mt, sh_zt, sh_md, sh_zd;

  const Geometry& geo = a.geo;
  const int V = geo.V;
  const int C = geo.csize;
  const int rank = static_cast<int>(cluster_rank());
  const int unit = blockIdx.x / C;
  const int W = a.g + 1;
  const int b = unit / W;
  const int j = unit % W;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  const bool bonus = (j == a.g);
  const size_t trow = (static_cast<size_t>(b) * W + j) * V;
  const size_t drow = (static_cast<size_t>(b) * a.g + j) * V;
  const int lo = rank * geo.slice;
  const int n = max(0, min(geo.slice, V - lo));

  Slice<E> sl;
  sl.gt = static_cast<const E*>(a.target) + trow + lo;
  sl.gd = bonus ? nullptr : static_cast<const E*>(a.draft) + drow + lo;
  sl.st = reinterpret_cast<E*>(dyn_smem);
  sl.sd = reinterpret_cast<E*>(dyn_smem + geo.row_smem);
  sl.n = n;
  sl.nvec = (n + kVec - 1) / kVec;
  sl.nstage = (n + geo.stage_elems - 1) / geo.stage_elems;
  sl.bulk = geo.bulk != 0;

  if (tid == 0) inbox_init(xbar, C, rank == 0);
  const float c = kLog2e / a.temperature;
  stage_issue(sl, bars, geo.stage_elems);
  cluster_arrive_release();
  const ThreadStats<E> ts = stats_pass(sl, bars, geo.stage_elems / kVec, c, true, false, lo);
  const BlockStats bs = block_reduce_stats(ts, c, red_f, red_i);
  cluster_wait_acquire();
  const float u_sag = unit_draws(a.seed, b, j).saguaro;
  const size_t out_idx = static_cast<size_t>(b) * W + j;
  float* st = (a.stats && rank == 0) ? a.stats + out_idx * SSD_NSTAT_SAGUARO : nullptr;
  if (warp == 0) {
    push_stats(&inbox, xbar, C, rank, bs);
    const BlockStats all = gather_stats(&inbox, xbar, C, c);
    if (tid == 0) {
      sh_mt = all.t.m;
      sh_zt = all.t.s;
      sh_md = all.d.m;
      sh_zd = all.d.s;
      sh_err = all.timeout;
      if (st) {
        st[0] = logf(all.t.s) - fmaf(all.t.m, c, -scaled_max(all.t.m, c)) * 0.6931471805599453f;
        st[1] = bonus ? NAN : logf(all.d.s) - fmaf(all.d.m, c, -scaled_max(all.d.m, c)) * 0.6931471805599453f;
        st[7] = NAN;
      }
    }
  }
  __syncthreads();

  const float mct = scaled_max(sh_mt, c);
  const float mcd = bonus ? 0.f : scaled_max(sh_md, c);
  const float kr = bonus ? 0.f : sh_zt / sh_zd;

  // Pass A: residual weights (or q at the bonus position / on zero residual
  // mass), their cluster sum, and this CTA's top-8.
  int target_only = bonus ? 1 : 0;
  int p = 0;
  double sum_a = 0.0, resid_mass = 1.0;
  for (;;) {
    TopK<kTopK> tk;
    tk.init();
    const PassAW<E> wf{c, mct, mcd, kr, target_only};
    const double cta = weighted_pass<E, kTopK>(sl, lo, wf, wsum, tk);
    float mv[kTopK];
    int mi[kTopK];
    warp_merge_topk<kTopK>(tk, mv, mi);
    if (lane == 0) {
#pragma unroll
      for (int r = 0; r < kTopK; ++r) {
        wtop_v[warp][r] = mv[r];
        wtop_i[warp][r] = mi[r];
      }
    }
    __syncthreads();
    if (warp == 0) {
      if (tid == 0) {
        int head[kWarps] = {0};
        for (int r = 0; r < kTopK; ++r) {
          int best = -1;
          for (int w = 0; w < kWarps; ++w) {
            if (head[w] >= kTopK) continue;
            if (best < 0 || ranks_before(wtop_v[w][head[w]], wtop_i[w][head[w]], wtop_v[best][head[best]],
                                         wtop_i[best][head[best]]))
              best = w;
          }
          cta_top_v[r] = wtop_v[best][head[best]];
          cta_top_i[r] = wtop_i[best][head[best]];
          ++head[best];
        }
      }
      push_sum(&inbox, xbar, C, rank, p, cta);
      int owner, to = 0;
      double local, prefix;
      const double total = gather_sums(&inbox, xbar, C, p, 0.5, &owner, &local, &prefix, &to);
      if (tid == 0) {
        sh_total = total;
        sh_err |= to;
      }
    }
    __syncthreads();
    if (p == 0 && !bonus) resid_mass = sh_total / static_cast<double>(sh_zt);
    if (!(sh_total > 0.0) && !target_only) {
      target_only = 1;
      ++p;
      continue;
    }
    sum_a = sh_total;
    break;
  }

  // Bonus prediction: every CTA sends its top-8 to rank 0, which merges them.
  if (tid == 0) {
    const uint32_t bar = dsmem_addr(&xbar[kXTop], 0);
    const float4* v4 = reinterpret_cast<const float4*>(cta_top_v);
    const float4* i4 = reinterpret_cast<const float4*>(cta_top_i);
    st_async_v4(dsmem_addr(&inbox.top[rank][0], 0), v4[0], bar);
    st_async_v4(dsmem_addr(&inbox.top[rank][1], 0), v4[1], bar);
    st_async_v4(dsmem_addr(&inbox.top[rank][2], 0), i4[0], bar);
    st_async_v4(dsmem_addr(&inbox.top[rank][3], 0), i4[1], bar);
  }
  if (rank == 0 && tid == 0) {
    if (!xbar_wait_bounded(&xbar[kXTop])) sh_err = 1;
    int head[kMaxCluster];
    for (int r = 0; r < C; ++r) head[r] = 0;
    int32_t* out = a.bonus_topk + out_idx * a.k;
    for (int s = 0; s < a.k; ++s) {
      int best = -1;
      float bv = 0.f;
      int bi = 0;
      for (int r = 0; r < C; ++r) {
        if (head[r] >= a.k) continue;
        const float* tv = reinterpret_cast<const float*>(&inbox.top[r][0]);
        const int* ti = reinterpret_cast<const int*>(&inbox.top[r][2]);
        if (best < 0 || ranks_before(tv[head[r]], ti[head[r]], bv, bi)) {
          best = r;
          bv = tv[head[r]];
          bi = ti[head[r]];
        }
      }
      ++head[best];
      out[s] = (bi >= 0 && bi < V && !sh_err) ? bi : -1;
      if (st && s == 0) st[5] = static_cast<float>(bv / sum_a);
      if (st && s == a.k - 1) st[6] = static_cast<float>(bv / sum_a);
    }
    if (st) st[2] = static_cast<float>(resid_mass);
  }

  // Saguaro mix pass and its inverse-CDF draw.
  const MixW<E> mw{c, mct, mcd, kr, target_only, bonus ? 1 : 0, static_cast<float>(1.0 / sum_a),
                   bonus ? 1.f / sh_zt : 1.f / sh_zd};
  {
    TopK<0> none;
    const double cta = weighted_pass<E, 0>(sl, lo, mw, wsum, none);
    if (warp == 0) {
      push_sum(&inbox, xbar, C, rank, 2, cta);
      int owner, to = 0;
      double local, prefix;
      const double total = gather_sums(&inbox, xbar, C, 2, static_cast<double>(u_sag), &owner, &local, &prefix, &to);
      if (tid == 0) {
        sh_total = total;
        sh_owner = owner;
        sh_local = local;
        sh_prefix = prefix;
        sh_err |= to;
      }
    }
    __syncthreads();
  }
  if (sh_owner == rank) {
    cdf_search(sl, lo, mw, wsum, sh_local, &sh_warp, &sh_base, &sh_result, &sh_edge, &sh_edge_w);
    if (tid == 0) a.saguaro_tokens[out_idx] = sh_err ? -1 : sh_result;
    if (a.stats && tid == 0 && sh_result >= lo) {
      // p_saguaro of the drawn token (debug statistics only)
      const int v = (sh_result - lo) / kVec, e = (sh_result - lo) % kVec;
      float xt[kVec], xd[kVec], w[kVec];
      load_vec(sl.st, v, xt);
      if (sl.gd) load_vec(sl.sd, v, xd);
      mw(xt, xd, w);
      float* st0 = a.stats + out_idx * SSD_NSTAT_SAGUARO;
      st0[3] = static_cast<float>(sh_total);
      st0[4] = static_cast<float>(w[e] / sh_total);
      st0[8] = static_cast<float>(static_cast<double>(u_sag) - (sh_prefix + sh_edge) / sh_total);
      st0[9] = static_cast<float>((sh_prefix + sh_edge + static_cast<double>(sh_edge_w)) / sh_total -
                                  static_cast<double>(u_sag));
    }
  } else if (sh_owner < 0 && rank == 0 && tid == 0) {
    a.saguaro_tokens[out_idx] = -1;
  }
  if (sh_err) stage_drain(sl, bars);
}

template __global__ void saguaro_kernel<uint16_t>(const SaguaroArgs);
template __global__ void saguaro_kernel<float>(const SaguaroArgs);

cudaError_t launch_saguaro(const SaguaroArgs& a, int esize, int smem_bytes, cudaStream_t stream) {
  const void* fn = esize == 2 ? reinterpret_cast<const void*>(&saguaro_kernel<uint16_t>)
                              : reinterpret_cast<const void*>(&saguaro_kernel<float>);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  if (a.geo.csize > 8) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  const long long units = static_cast<long long>(a.B) * (a.g + 1);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units * a.geo.csize), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.geo.csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (esize == 2) return cudaLaunchKernelEx(&cfg, saguaro_kernel<uint16_t>, a);
  return cudaLaunchKernelEx(&cfg, saguaro_kernel<float>, a);
}

}  // namespace ssdv
