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
// One cluster handles one (request b, position i) unit: it stages target row i
// (and draft row i for a sampled draft position) into shared memory, reduces
// the softmax statistics of both rows in the same pass, takes the accept
// decision, and -- only if position i rejects, or i is the bonus position --
// runs the on-chip residual pass and inverse-CDF search.  Every position is
// decided independently; the last unit of a request to finish (arrival
// ticket in the workspace, no spinning) scans the decisions to the first
// rejection and writes the request's outputs.
#include "ssdv_device.cuh"

namespace ssdv {

namespace {

// Residual weights scaled by Z_t: w = max(e_t - (Z_t/Z_d) e_d, 0) with
// e = exp2(x*c - fl(m*c)).  Its sum is Z_t * sum (q - p)+.
template <typename E>
struct ResidualW {
  float c, mct, mcd, kr;
  __device__ __forceinline__ void operator()(const float (&xt)[Elem<E>::kVec], const float (&xd)[Elem<E>::kVec],
                                             float (&w)[Elem<E>::kVec]) const {
#pragma unroll
    for (int e = 0; e < Elem<E>::kVec; ++e) {
      const float et = exp2f(fmaf(xt[e], c, -mct));
      const float ed = exp2f(fmaf(xd[e], c, -mcd));
      w[e] = fmaxf(fmaf(-kr, ed, et), 0.f);
    }
  }
};

// Target weights: w = e_t (proportional to q).
template <typename E>
struct TargetW {
  float c, mct;
  __device__ __forceinline__ void operator()(const float (&xt)[Elem<E>::kVec], const float (&)[Elem<E>::kVec],
                                             float (&w)[Elem<E>::kVec]) const {
#pragma unroll
    for (int e = 0; e < Elem<E>::kVec; ++e) w[e] = exp2f(fmaf(xt[e], c, -mct));
  }
};

__device__ __forceinline__ bool temperature_ok(float T) {
  return T == 0.f || (T >= 1e-6f && T <= 3.0e38f);
}

// Last unit of request b: scan the per-position decisions and write outputs.
__device__ void finish_request(const VerifyArgs& a, int b, int g) {
  const int W = a.gmax + 1;
  int32_t* wflag = a.unit_flag + static_cast<size_t>(b) * W;
  int32_t* wtok = a.unit_tok + static_cast<size_t>(b) * W;
  int32_t* out = a.out_tokens + static_cast<size_t>(b) * W;
  int32_t flags[SSD_MAX_GAMMA + 1];
#pragma unroll 4
  for (int k = 0; k <= g; ++k) flags[k] = ld_volatile(wflag + k);
  bool err = false;
  int n = g;
  for (int k = g; k >= 0; --k) {
    err |= flags[k] < 0;
    if (k < g && flags[k] == 0) n = k;
  }
  if (err) {
    for (int k = 0; k < W; ++k) out[k] = -1;
    a.n_accepted[b] = -1;
  } else {
    const int32_t last = ld_volatile(wtok + n);
    for (int k = 0; k < n; ++k) out[k] = a.draft_tokens[static_cast<size_t>(b) * a.gmax + k];
    out[n] = last;
    for (int k = n + 1; k < W; ++k) out[k] = -1;
    a.n_accepted[b] = n;
  }
  // Leave the whole workspace zeroed (its layout depends on B and gamma, so a
  // later call with another shape may read these words as arrival counters).
  for (int k = 0; k < W; ++k) {
    wflag[k] = 0;
    wtok[k] = 0;
  }
  a.ticket[b] = 0;
}

// Record unit (b, i)'s decision and count it; the last unit of the request
// writes the outputs.  Called by one thread per unit.
__device__ __forceinline__ void arrive_unit(const VerifyArgs& a, int b, int i, int g, int flag, int tok,
                                            bool write_tok) {
  const int out_idx = b * (a.gmax + 1) + i;
  if (write_tok) a.unit_tok[out_idx] = tok;
  a.unit_flag[out_idx] = flag;
  __threadfence();
  if (atomicAdd(a.ticket + b, 1) == g) {
    __threadfence();
    finish_request(a, b, g);
  }
}

}  // namespace

template <typename E>
__global__ void __launch_bounds__(kThreads) verify_kernel(const VerifyArgs a) {
  constexpr int kVec = Elem<E>::kVec;
  extern __shared__ __align__(128) uint8_t dyn_smem[];
  __shared__ __align__(8) uint64_t bars[kMaxStages];
  __shared__ __align__(8) uint64_t xbar[kNumX];
  __shared__ __align__(16) Inbox inbox;
  __shared__ float red_f[5 * kWarps];
  __shared__ int red_i[2 * kWarps];
  __shared__ float wsum[kWarps];
  __shared__ int sh_warp, sh_result, sh_owner, sh_accept, sh_pass, sh_err;
  __shared__ double sh_base, sh_local, sh_prefix, sh_total, sh_edge;
  __shared__ float sh_edge_w;
  __shared__ float sh_mt, sh_zt, sh_md, sh_zd;

  const Geometry& geo = a.geo;
  const int V = geo.V;
  const int C = geo.csize;
  const int rank = static_cast<int>(cluster_rank());
  const int unit = blockIdx.x / C;
  const int W = a.gmax + 1;
  const int b = unit / W;
  const int i = unit % W;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;

  const int g = a.gamma ? a.gamma[b] : a.gmax;
  const float T = a.temps ? a.temps[b] : a.temp_scalar;
  const bool bad_gamma = g > a.gmax;
  const bool bad_temp = !temperature_ok(T);
  if (g < 0 || bad_gamma || bad_temp) {  // padded or invalid request: position 0 writes -1s
    if (i == 0 && rank == 0 && tid == 0) {
      int32_t* out = a.out_tokens + static_cast<size_t>(b) * W;
      for (int k = 0; k < W; ++k) out[k] = -1;
      a.n_accepted[b] = -1;
      if (bad_gamma) atomicOr(a.status, 1 << SSD_ERR_GAMMA);
      if (bad_temp && g >= 0) atomicOr(a.status, 1 << SSD_ERR_TEMPERATURE);
    }
    return;
  }
  if (i > g) return;

  const bool greedy = (T == 0.f);
  const bool bonus = (i == g);
  const bool has_draft = !greedy && !bonus;
  int x = -1;
  bool tok_err = false;
  if (!bonus) {
    x = a.draft_tokens[static_cast<size_t>(b) * a.gmax + i];
    tok_err = (x < 0 || x >= V);
  }
  const int out_idx = b * W + i;
  if (tok_err) {  // the whole cluster agrees: no staging, no exchange
    if (rank == 0 && tid == 0) {
      atomicOr(a.status, 1 << SSD_ERR_TOKEN_RANGE);
      arrive_unit(a, b, i, g, -1, 0, false);
    }
    return;
  }

  const size_t trow = (static_cast<size_t>(b) * W + i) * V;
  const size_t drow = (static_cast<size_t>(b) * a.gmax + i) * V;
  const E* tbase = static_cast<const E*>(a.target);
  const E* dbase = has_draft ? static_cast<const E*>(a.draft) : nullptr;
  const int lo = rank * geo.slice;
  const int n = max(0, min(geo.slice, V - lo));

  Slice<E> sl;
  sl.gt = tbase + trow + lo;
  sl.gd = has_draft ? dbase + drow + lo : nullptr;
  sl.st = reinterpret_cast<E*>(dyn_smem);
  sl.sd = reinterpret_cast<E*>(dyn_smem + geo.row_smem);
  sl.n = n;
  sl.nvec = (n + kVec - 1) / kVec;
  sl.nstage = (n + geo.stage_elems - 1) / geo.stage_elems;
  sl.bulk = geo.bulk != 0;

  // The two token logits of the accept test (sampled draft positions).
  float xt_tok = 0.f, xd_tok = 0.f;
  if (has_draft && tid == 0) {
    xt_tok = Elem<E>::to_float(tbase[trow + x]);
    xd_tok = Elem<E>::to_float(dbase[drow + x]);
  }

  if (tid == 0) inbox_init(xbar, C, false);
  const float c = greedy ? 1.f : kLog2e / T;
  stage_issue(sl, bars, geo.stage_elems);  // (its __syncthreads also publishes the inbox barriers)
  cluster_arrive_release();                // this CTA's inbox is ready
  const ThreadStats<E> ts =
      stats_pass(sl, bars, geo.stage_elems / kVec, c, /*want_exp=*/!greedy, /*want_arg=*/greedy, lo);
  const BlockStats bs = block_reduce_stats(ts, c, red_f, red_i);
  cluster_wait_acquire();  // every inbox of the cluster is ready
  const Draws u = unit_draws(a.seed, b, i);
  if (warp == 0) {
    push_stats(&inbox, xbar, C, rank, bs);
    const BlockStats all = gather_stats(&inbox, xbar, C, c);
    if (tid == 0) {
      int accept = 0, need_pass = 0, err = all.timeout;
      if (greedy) {
        accept = (!bonus && x == all.a.i) ? 1 : 0;
        sh_result = all.a.i;
      } else if (bonus) {
        need_pass = 1;
      } else {
        // a = min(1, q(x)/p(x)) with q(x) = e_t(x)/Z_t, p(x) = e_d(x)/Z_d, the
        // ratio taken as one exp2 of the exponent difference.
        const float mct = scaled_max(all.t.m, c), mcd = scaled_max(all.d.m, c);
        float ratio_acc;
        if (xd_tok == -INFINITY) {
          ratio_acc = 1.f;
        } else {
          const float lt = fmaf(xt_tok, c, -mct), ld = fmaf(xd_tok, c, -mcd);
          const float ratio = exp2f(lt - ld) * (all.d.s / all.t.s);
          ratio_acc = fminf(1.f, ratio);
        }
        accept = u.accept < ratio_acc ? 1 : 0;
        need_pass = (!accept || a.force_residual) ? 1 : 0;
        if (a.stats && rank == 0) {
          float* st = a.stats + static_cast<size_t>(out_idx) * SSD_NSTAT_VERIFY;
          st[2] = all.d.m;
          st[3] = logf(all.d.s) - fmaf(all.d.m, c, -mcd) * 0.6931471805599453f;
          st[4] = exp2f(fmaf(xt_tok, c, -mct)) / all.t.s;
          st[5] = exp2f(fmaf(xd_tok, c, -mcd)) / all.d.s;
          st[7] = ratio_acc;
        }
      }
      if (err) need_pass = 0;
      if (a.stats && rank == 0) {
        float* st = a.stats + static_cast<size_t>(out_idx) * SSD_NSTAT_VERIFY;
        st[0] = greedy ? all.a.v : all.t.m;
        // ln sum exp((x - m)/T): the sums carry the factor exp2(m*c - fl(m*c)).
        if (!greedy) st[1] = logf(all.t.s) - fmaf(all.t.m, c, -scaled_max(all.t.m, c)) * 0.6931471805599453f;
      }
      sh_accept = accept;
      sh_pass = need_pass;
      sh_err = err;
      sh_mt = all.t.m;
      sh_zt = all.t.s;
      sh_md = all.d.m;
      sh_zd = all.d.s;
    }
  }
  __syncthreads();

  if (!sh_pass) {
    // Decided without a draw (accepted, greedy, or an error): rank 0 reports.
    if (rank == 0 && tid == 0)
      arrive_unit(a, b, i, g, sh_err ? -1 : sh_accept, sh_result, greedy && !sh_err);
    if (sh_err) stage_drain(sl, bars);
    return;
  }

  // Residual (or bonus) pass over the resident slice, the cluster-wide sums,
  // and the inverse-CDF draw in the CTA that owns the target.
  const float mct = scaled_max(sh_mt, c);
  TopK<0> none;
  int p = 0;
  int use_target = bonus ? 1 : 0;
  double resid_mass = 0.0;
  for (;;) {
    double cta;
    if (use_target) {
      const TargetW<E> wf{c, mct};
      cta = weighted_pass<E, 0>(sl, lo, wf, wsum, none);
    } else {
      const ResidualW<E> wf{c, mct, scaled_max(sh_md, c), sh_zt / sh_zd};
      cta = weighted_pass<E, 0>(sl, lo, wf, wsum, none);
    }
    if (warp == 0) {
      push_sum(&inbox, xbar, C, rank, p, cta);
      int owner, to = 0;
      double local, prefix;
      const double total =
          gather_sums(&inbox, xbar, C, p, static_cast<double>(u.resample), &owner, &local, &prefix, &to);
      if (tid == 0) {
        sh_owner = owner;
        sh_local = local;
        sh_prefix = prefix;
        sh_total = total;
        sh_err |= to;
        if (!use_target && p == 0) resid_mass = total;
      }
    }
    __syncthreads();
    // Rejected with no residual mass: sample from q instead (the same decision
    // in every CTA: all of them received the same sums).
    if (sh_owner < 0 && !use_target) {
      use_target = 1;
      ++p;
      continue;
    }
    break;
  }
  if (a.stats && rank == 0 && tid == 0 && !bonus)
    a.stats[static_cast<size_t>(out_idx) * SSD_NSTAT_VERIFY + 6] = static_cast<float>(resid_mass / sh_zt);

  const bool draws = !sh_accept || bonus;  // debug runs may pass accepted positions here
  if (!draws) {
    if (rank == 0 && tid == 0) arrive_unit(a, b, i, g, sh_err ? -1 : 1, 0, false);
    if (sh_err) stage_drain(sl, bars);
    return;
  }
  if (sh_owner < 0) {  // no positive weight at all: only possible for invalid input
    if (rank == 0 && tid == 0) arrive_unit(a, b, i, g, -1, 0, false);
    return;
  }
  if (sh_owner != rank) {
    if (sh_err) stage_drain(sl, bars);
    return;
  }
  if (use_target) {
    const TargetW<E> wf{c, mct};
    cdf_search(sl, lo, wf, wsum, sh_local, &sh_warp, &sh_base, &sh_result, &sh_edge, &sh_edge_w);
  } else {
    const ResidualW<E> wf{c, mct, scaled_max(sh_md, c), sh_zt / sh_zd};
    cdf_search(sl, lo, wf, wsum, sh_local, &sh_warp, &sh_base, &sh_result, &sh_edge, &sh_edge_w);
  }
  if (tid == 0) {
    if (a.stats) {  // distances of u to the drawn token's CDF edges (debug statistics)
      float* st = a.stats + static_cast<size_t>(out_idx) * SSD_NSTAT_VERIFY;
      const double ur = static_cast<double>(u.resample);
      st[8] = static_cast<float>(ur - (sh_prefix + sh_edge) / sh_total);
      st[9] = static_cast<float>((sh_prefix + sh_edge + static_cast<double>(sh_edge_w)) / sh_total - ur);
    }
    if (sh_err) atomicOr(a.status, 1 << SSD_ERR_TIMEOUT);
    arrive_unit(a, b, i, g, sh_err ? -1 : (bonus ? 1 : 0), sh_result, true);
  }
  if (sh_err) stage_drain(sl, bars);
}

template __global__ void verify_kernel<uint16_t>(const VerifyArgs);
template __global__ void verify_kernel<float>(const VerifyArgs);

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

cudaError_t launch_verify(const VerifyArgs& a, int esize, int smem_bytes, cudaStream_t stream) {
  const void* fn = esize == 2 ? reinterpret_cast<const void*>(&verify_kernel<uint16_t>)
                              : reinterpret_cast<const void*>(&verify_kernel<float>);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  if (a.geo.csize > 8) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  const long long units = static_cast<long long>(a.B) * (a.gmax + 1);
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
  if (esize == 2) return cudaLaunchKernelEx(&cfg, verify_kernel<uint16_t>, a);
  return cudaLaunchKernelEx(&cfg, verify_kernel<float>, a);
}

}  // namespace ssdv
