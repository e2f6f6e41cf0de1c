// ssdv_api.cu -- the C ABI of libssdv (declared in include/ssdv.h): argument
// validation, launch geometry, workspace layout, status reporting.
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <list>
#include <mutex>
#include <string>
#include <unordered_map>
#include <vector>

#include "ssdv_device.cuh"
#include "ssdv_internal.h"

namespace ssdv {

namespace {

thread_local std::string g_last_error;

ssd_status fail(ssd_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
ssd_status fail(ssd_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

ssd_status cuda_fail(cudaError_t e, const char* what) {
  return fail(SSD_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int esize_of(ssd_dtype dt) { return dt == SSD_BF16 ? 2 : (dt == SSD_F32 ? 4 : 0); }

constexpr int kMaxChunkElems = SSD_MAX_V / kMaxChunks;  // 16384

bool temperature_valid(float T) { return T == 0.f || (T >= 1e-6f && isfinite(T)); }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int env_int(const char* name, int fallback) {
  const char* v = getenv(name);
  if (!v || !*v) return fallback;
  return atoi(v);
}

}  // namespace

WorkspaceLayout workspace_layout(int B, int gmax) {
  WorkspaceLayout L;
  const size_t units = static_cast<size_t>(B) * static_cast<size_t>(gmax + 1);
  L.status = 0;
  L.half0 = 256;
  L.ticket = 0;  // offsets within a half
  L.part = round_up(L.ticket + 4 * units, 256);
  L.blocks = L.part + units * kMaxChunks * 2 * sizeof(float4);
  L.half_bytes = round_up(L.blocks + units * kMaxPieces * sizeof(float), 256);
  L.total = L.half0 + 2 * L.half_bytes;
  return L;
}

SagLayout saguaro_layout(int B, int g, int V) {
  SagLayout L;
  const size_t units = static_cast<size_t>(B) * static_cast<size_t>(g + 1);
  // sized for fp32 rows (the most pieces per row) and the fewest pieces per warp
  const size_t np = (static_cast<size_t>(V) + 511) / 512;
  const size_t npw = (np + kSagMinPpw - 1) / kSagMinPpw;
  L.ticket2 = 256;  // after the status word
  L.ticket3 = round_up(L.ticket2 + 4 * units, 256);
  L.rowstat = round_up(L.ticket3 + 4 * units, 256);
  L.rowsum = L.rowstat + units * sizeof(float4);
  L.zsum = L.rowsum + units * sizeof(double);
  L.part = round_up(L.zsum + units * sizeof(float), 256);
  L.psum2 = L.part + units * kMaxChunks * 2 * sizeof(float4);
  L.psum3 = round_up(L.psum2 + units * np * sizeof(float), 256);
  L.cand_v = round_up(L.psum3 + units * np * sizeof(float), 256);
  L.cand_i = round_up(L.cand_v + units * npw * SSD_MAX_TOPK * sizeof(float), 256);
  L.total = round_up(L.cand_i + units * npw * SSD_MAX_TOPK * sizeof(int32_t), 256);
  return L;
}

// Top-p extension of the verification workspace: per row slot (B, gmax+1, 2)
// the select state, the thresholds and kept masses, then every level's
// histograms (fp32's 256 + 2048 + 2048 + 1024 bins, the most).
struct TopPLayout {
  size_t prefix, bstar, above, goal, th, z, todo, todo_count, hist, total;
};
constexpr int kTopPBins = 256 + 2048 + 2048 + 1024;
static TopPLayout topp_layout(int B, int gmax) {
  TopPLayout T;
  const size_t slots = static_cast<size_t>(B) * static_cast<size_t>(gmax + 1) * 2;
  T.prefix = round_up(workspace_layout(B, gmax).total, 256);
  T.bstar = T.prefix + 4 * slots;
  T.above = round_up(T.bstar + 4 * slots, 256);
  T.goal = T.above + 8 * slots;
  T.th = T.goal + 8 * slots;
  T.z = T.th + 4 * slots;
  T.todo = round_up(T.z + 4 * slots, 256);
  T.todo_count = round_up(T.todo + 4 * slots, 256);  // zeroed with the histograms
  T.hist = T.todo_count + 256;
  T.total = T.hist + slots * kTopPBins * 8;
  return T;
}

namespace {

// Consecutive calls on one workspace use alternate halves, so a pipelined
// call's streaming kernel may run while the previous call's sampling kernel
// reads the other half.  The parity is kept on the host per workspace
// address, for the kHalfSlots most recently used addresses (least recently
// used first out): a workspace evicted from the table was last used at least
// kHalfSlots calls on other workspaces ago, and starts again from half 0.
constexpr size_t kHalfSlots = 4096;
std::mutex g_half_mutex;
std::list<std::pair<const void*, unsigned long long>> g_half_lru;  // most recent first
std::unordered_map<const void*, std::list<std::pair<const void*, unsigned long long>>::iterator> g_half;

int next_half(const void* workspace) {
  std::lock_guard<std::mutex> lock(g_half_mutex);
  auto it = g_half.find(workspace);
  if (it == g_half.end()) {
    if (g_half_lru.size() >= kHalfSlots) {
      g_half.erase(g_half_lru.back().first);
      g_half_lru.pop_back();
    }
    g_half_lru.emplace_front(workspace, 0ull);
    it = g_half.emplace(workspace, g_half_lru.begin()).first;
  } else if (it->second != g_half_lru.begin()) {
    g_half_lru.splice(g_half_lru.begin(), g_half_lru, it->second);
  }
  return static_cast<int>(it->second->second++ & 1ull);
}

}  // namespace

int max_dynamic_smem() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
  return v - 8 * 1024;  // leave room for the kernels' static shared memory
}

// Split a row of V elements into chunks for verification: about 24 KB of each
// row per CTA (SSDV_CHUNK_BYTES overrides), at most kMaxChunks chunks, each a
// multiple of 8 elements.
ssd_status choose_chunks(int V, int esize, bool aligned, ChunkGeometry* geo, int* smem_bytes) {
  const int max_smem = max_dynamic_smem();
  if (max_smem <= 0) return fail(SSD_ERR_CUDA, "cannot query the device's shared-memory limit");
  const long long row_bytes = static_cast<long long>(V) * esize;
  const int want = env_int("SSDV_CHUNK_BYTES", 24 * 1024);
  long long nc = (row_bytes + want - 1) / want;
  if (nc < 1) nc = 1;
  if (nc > kMaxChunks) nc = kMaxChunks;
  // at most kMaxChunkElems elements a chunk (top-p's level 0 counts a chunk's
  // masses in 32-bit words sized for that); V <= 2^19 keeps nc <= kMaxChunks
  if (nc < (V + kMaxChunkElems - 1) / kMaxChunkElems) nc = (V + kMaxChunkElems - 1) / kMaxChunkElems;
  const int chunk = static_cast<int>(round_up((static_cast<size_t>(V) + nc - 1) / nc, 8));
  const int row_smem = static_cast<int>(round_up(static_cast<size_t>(chunk) * esize, 128));
  if (2 * row_smem > max_smem)
    return fail(SSD_ERR_UNSUPPORTED, "V=%d: a chunk of %d elements does not fit in shared memory", V, chunk);
  geo->V = V;
  geo->chunk = chunk;
  geo->nchunk = (V + chunk - 1) / chunk;
  geo->row_smem = row_smem;
  geo->aligned = aligned ? 1 : 0;
  // pieces of the sampling kernel: 128 vectors of a row each
  geo->npiece = static_cast<int>((static_cast<long long>(V) + 128 * (16 / esize) - 1) / (128 * (16 / esize)));
  if (geo->npiece > kMaxPieces) return fail(SSD_ERR_UNSUPPORTED, "V=%d: more than %d pieces per row", V, kMaxPieces);
  *smem_bytes = 2 * row_smem;
  return SSD_OK;
}

namespace {

ssd_status verify_common(const void* target, const void* draft, ssd_dtype dtype, const int32_t* draft_tokens, int B,
                         int gmax, int V, const int32_t* gamma, const float* temps, float temp_scalar,
                         bool all_greedy, uint64_t seed, int32_t* out_tokens, int32_t* n_accepted, void* workspace,
                         size_t ws_bytes, float* stats, void* stream, bool pipelined = false, float top_p = 1.f) {
  const bool use_topp = top_p < 1.f && !all_greedy;
  const int es = esize_of(dtype);
  if (es == 0) return fail(SSD_ERR_DTYPE, "unknown dtype %d", static_cast<int>(dtype));
  if (!target || !out_tokens || !n_accepted || !workspace) return fail(SSD_ERR_NULL, "a required pointer is NULL");
  if (!draft && !all_greedy && gmax > 0)
    return fail(SSD_ERR_NULL, "draft_logits is NULL but some request samples");
  if (gmax > 0 && !draft_tokens) return fail(SSD_ERR_NULL, "draft_tokens is NULL");
  if (B < 1 || gmax < 0 || gmax > SSD_MAX_GAMMA || V < 1 || V > SSD_MAX_V)
    return fail(SSD_ERR_SHAPE, "bad shape B=%d gamma=%d V=%d", B, gmax, V);
  if (!aligned_to(target, es) || (draft && !aligned_to(draft, es)) || !aligned_to(out_tokens, 4) ||
      !aligned_to(n_accepted, 4) || (draft_tokens && !aligned_to(draft_tokens, 4)) || !aligned_to(workspace, 16) ||
      (stats && !aligned_to(stats, 4)) || (gamma && !aligned_to(gamma, 4)) || (temps && !aligned_to(temps, 4)))
    return fail(SSD_ERR_ALIGN, "a pointer is not aligned to its element size (workspace: 16 bytes)");
  const WorkspaceLayout L = workspace_layout(B, gmax);
  const size_t need = use_topp ? topp_layout(B, gmax).total : L.total;
  if (ws_bytes < need) return fail(SSD_ERR_WORKSPACE, "workspace of %zu bytes < %zu required", ws_bytes, need);
  if (use_topp && (B > 65535 || stats))
    return fail(SSD_ERR_UNSUPPORTED, "top-p verification takes at most 65535 requests and no statistics");
  const bool aligned = aligned_to(target, 16) && (!draft || aligned_to(draft, 16)) &&
                       ((static_cast<size_t>(V) * es) % 16 == 0);
  ChunkGeometry geo;
  int smem = 0;
  ssd_status st = choose_chunks(V, es, aligned, &geo, &smem);
  if (st != SSD_OK) return st;
  const long long ctas = static_cast<long long>(B) * (gmax + 1) * geo.nchunk;
  if (ctas >= (1LL << 31)) return fail(SSD_ERR_SHAPE, "grid too large");
  // Pieces per warp of the sampling kernel (SSDV_PPW overrides).  A plain
  // call takes one piece per warp (one round of loads) when the sampling grid
  // then still fits in one wave of 8 small CTAs per SM, else two.  A pipelined
  // call takes four, so that the sampling grid becomes resident while the
  // streaming kernel still runs and the next call's streaming kernel can
  // launch early.
  int ppw_default = pipelined ? 4 : 2;
  if (!pipelined) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
        static_cast<long long>(B) * ((geo.npiece + 3) / 4) <= 8LL * sms)
      ppw_default = 1;
  }
  geo.ppw = env_int("SSDV_PPW", ppw_default);
  if (geo.ppw < 1) geo.ppw = 1;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  VerifyArgs a;
  a.target = target;
  a.draft = draft;
  a.draft_tokens = draft_tokens;
  a.B = B;
  a.gmax = gmax;
  a.req_base = 0;
  a.gamma = gamma;
  a.temps = temps;
  a.temp_scalar = temp_scalar;
  a.seed = seed;
  a.out_tokens = out_tokens;
  a.n_accepted = n_accepted;
  a.status = reinterpret_cast<int32_t*>(ws + L.status);
  uint8_t* half = ws + L.half0 + static_cast<size_t>(next_half(workspace)) * L.half_bytes;
  a.ticket = reinterpret_cast<int32_t*>(half + L.ticket);
  a.part = reinterpret_cast<float4*>(half + L.part);
  a.psum = reinterpret_cast<float*>(half + L.blocks);
  a.stats = stats;
  a.debug = stats ? 1 : 0;
  a.sag_S = nullptr;
  a.sag_Zs = nullptr;
  a.tp_th = nullptr;
  a.tp_z = nullptr;
  a.pieces_ready = 0;
  // streaming order: request-major for pipelined calls of one gamma, where it
  // measured faster; position-major for plain and ragged calls
  a.req_major = (pipelined && !gamma) ? 1 : 0;
  a.geo = geo;
  if (use_topp) {
    // The streaming kernel, the radix-select levels of every row's nucleus
    // threshold, then the sampling kernel on the truncated distributions.
    const TopPLayout TL = topp_layout(B, gmax);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // level 0: 256 mass bins; then the key digits inside the chosen bin
    const int levels = es == 2 ? 3 : 4;
    const int shifts[4] = {0, es == 2 ? 24 : 21, es == 2 ? 16 : 10, 0};
    const int bits[4] = {8, es == 2 ? 8 : 11, es == 2 ? 8 : 11, 10};
    const size_t slots = static_cast<size_t>(B) * (gmax + 1) * 2;
    size_t hist_bytes = 0;
    for (int l = 0; l < levels; ++l) hist_bytes += slots * (static_cast<size_t>(8) << bits[l]);
    cudaError_t e = cudaMemsetAsync(ws + TL.todo_count, 0, (TL.hist - TL.todo_count) + hist_bytes, st);
    if (e != cudaSuccess) return cuda_fail(e, "top-p histogram memset");
    a.first = 1;
    a.tp_th = reinterpret_cast<float*>(ws + TL.th);
    a.tp_z = reinterpret_cast<float*>(ws + TL.z);
    e = launch_stream(a, es, smem, st);
    if (e != cudaSuccess) return cuda_fail(e, "verify launch");
    TopPArgs t = {};
    t.target = target;
    t.draft = draft;
    t.B = B;
    t.gmax = gmax;
    t.gamma = gamma;
    t.temps = temps;
    t.temp_scalar = temp_scalar;
    t.top_p = top_p;
    t.part = a.part;
    t.geo = geo;
    t.nlevels = levels;
    t.prefix = reinterpret_cast<uint32_t*>(ws + TL.prefix);
    t.bstar = reinterpret_cast<uint32_t*>(ws + TL.bstar);
    t.above = reinterpret_cast<unsigned long long*>(ws + TL.above);
    t.goal = reinterpret_cast<unsigned long long*>(ws + TL.goal);
    t.th = reinterpret_cast<float*>(ws + TL.th);
    t.z = reinterpret_cast<float*>(ws + TL.z);
    t.todo = reinterpret_cast<uint32_t*>(ws + TL.todo);
    t.todo_count = reinterpret_cast<uint32_t*>(ws + TL.todo_count);
    size_t off = TL.hist;
    for (int l = 0; l < levels; ++l) {
      t.level = l;
      t.shift = shifts[l];
      t.bits = bits[l];
      t.hist = reinterpret_cast<unsigned long long*>(ws + off);
      off += slots * (static_cast<size_t>(8) << bits[l]);
      e = launch_topp_level(t, es, st);
      if (e != cudaSuccess) return cuda_fail(e, "top-p launch");
    }
    e = launch_sample(a, es, st);
    if (e != cudaSuccess) return cuda_fail(e, "verify launch");
    return SSD_OK;
  }
  // Launch in segments of at most 65535 requests (the grid's third
  // dimension; SSDV_SEGMENT sets a smaller size).  Each segment keeps its
  // requests' global indices for the Philox counters and its own rows of the
  // workspace; a segment's sampling kernel may run while the next segment
  // streams.
  int seg = env_int("SSDV_SEGMENT", 65535);
  seg = std::max(1, std::min(seg, 65535));
  const int NP = geo.npiece;
  const int W = gmax + 1;
  for (int b0 = 0; b0 < B; b0 += seg) {
    VerifyArgs s = a;
    s.B = B - b0 < seg ? B - b0 : seg;
    s.req_base = b0;
    s.first = (b0 == 0 && !pipelined) ? 1 : 0;
    s.target = static_cast<const uint8_t*>(target) + static_cast<size_t>(b0) * W * V * es;
    if (draft) s.draft = static_cast<const uint8_t*>(draft) + static_cast<size_t>(b0) * gmax * V * es;
    if (draft_tokens) s.draft_tokens = draft_tokens + static_cast<size_t>(b0) * gmax;
    if (gamma) s.gamma = gamma + b0;
    if (temps) s.temps = temps + b0;
    s.out_tokens = out_tokens + static_cast<size_t>(b0) * W;
    s.n_accepted = n_accepted + b0;
    if (stats) s.stats = stats + static_cast<size_t>(b0) * W * SSD_NSTAT_VERIFY;
    const size_t u0 = static_cast<size_t>(b0) * W;  // the segment's first (request, position) unit
    s.ticket = a.ticket + u0;
    s.part = a.part + u0 * geo.nchunk * 2;
    s.psum = a.psum + u0 * NP;
    // small vocabularies (no statistics wanted): one warp per request
    const cudaError_t e = (V <= kSmallV && !stats && env_int("SSDV_SMALL_V", 1) != 0)
                              ? launch_small_verify(s, es, static_cast<cudaStream_t>(stream))
                              : launch_verify(s, es, smem, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "verify launch");
  }
  return SSD_OK;
}

}  // namespace

}  // namespace ssdv

// Scratch of ssd_verify_noalloc: one fixed array per device, so that entry
// point never allocates.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SSD_NOALLOC_SCRATCH_BYTES];

namespace ssdv {
namespace {

// Device addresses of the array already zeroed.  Keyed by the address, not
// the device ordinal: after a device reset the module is loaded again and the
// array may sit elsewhere, and that new copy is zeroed before first use.
std::mutex g_noalloc_mutex;
std::vector<void*> g_noalloc_zeroed;

// The current device's scratch address, looked up on every call (a host-side
// query that allocates nothing); an address seen for the first time is zeroed
// on `stream`.
ssd_status noalloc_scratch(cudaStream_t stream, void** out) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the no-alloc scratch");
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (std::find(g_noalloc_zeroed.begin(), g_noalloc_zeroed.end(), p) == g_noalloc_zeroed.end()) {
    e = cudaMemsetAsync(p, 0, SSD_NOALLOC_SCRATCH_BYTES, stream);
    if (e != cudaSuccess) return cuda_fail(e, "no-alloc scratch memset");
    g_noalloc_zeroed.push_back(p);
  }
  *out = p;
  return SSD_OK;
}

}  // namespace
}  // namespace ssdv

using namespace ssdv;

extern "C" {

size_t ssd_workspace_bytes(int B, int gamma_max) {
  if (B < 1 || gamma_max < 0) return 0;
  return workspace_layout(B, gamma_max).total;
}

size_t ssd_saguaro_workspace_bytes(int B, int gamma, int V) {
  if (B < 1 || gamma < 0 || V < 1) return 0;
  return saguaro_layout(B, gamma, V).total;
}

ssd_status ssd_workspace_init(void* workspace, size_t ws_bytes, void* stream) {
  if (!workspace) return fail(SSD_ERR_NULL, "workspace is NULL");
  const cudaError_t e = cudaMemsetAsync(workspace, 0, ws_bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "workspace memset");
  return SSD_OK;
}

ssd_status ssd_verify(const void* target_logits, const void* draft_logits, ssd_dtype dtype,
                      const int32_t* draft_tokens, int B, int gamma, int V, float temperature, uint64_t seed,
                      int32_t* out_tokens, int32_t* n_accepted, void* workspace, size_t ws_bytes, void* stream) {
  g_last_error.clear();
  if (!temperature_valid(temperature))
    return fail(SSD_ERR_TEMPERATURE, "temperature %g is not 0 or in [1e-6, inf)", static_cast<double>(temperature));
  return verify_common(target_logits, draft_logits, dtype, draft_tokens, B, gamma, V, nullptr, nullptr, temperature,
                       temperature == 0.f, seed, out_tokens, n_accepted, workspace, ws_bytes, nullptr, stream);
}

size_t ssd_verify_top_p_workspace_bytes(int B, int gamma_max) {
  if (B < 1 || gamma_max < 0) return 0;
  return topp_layout(B, gamma_max).total;
}

ssd_status ssd_verify_top_p(const void* target_logits, const void* draft_logits, ssd_dtype dtype,
                            const int32_t* draft_tokens, int B, int gamma, int V, float temperature, float top_p,
                            uint64_t seed, int32_t* out_tokens, int32_t* n_accepted, void* workspace, size_t ws_bytes,
                            void* stream) {
  g_last_error.clear();
  if (!temperature_valid(temperature))
    return fail(SSD_ERR_TEMPERATURE, "temperature %g is not 0 or in [1e-6, inf)", static_cast<double>(temperature));
  if (!(top_p > 0.f) || !(top_p <= 1.f))
    return fail(SSD_ERR_SHAPE, "top_p %g is not in (0, 1]", static_cast<double>(top_p));
  return verify_common(target_logits, draft_logits, dtype, draft_tokens, B, gamma, V, nullptr, nullptr, temperature,
                       temperature == 0.f, seed, out_tokens, n_accepted, workspace, ws_bytes, nullptr, stream, false,
                       top_p);
}

ssd_status ssd_verify_pipelined(const void* target_logits, const void* draft_logits, ssd_dtype dtype,
                                const int32_t* draft_tokens, int B, int gamma, int V, float temperature,
                                uint64_t seed, int32_t* out_tokens, int32_t* n_accepted, void* workspace,
                                size_t ws_bytes, void* stream) {
  g_last_error.clear();
  if (!temperature_valid(temperature))
    return fail(SSD_ERR_TEMPERATURE, "temperature %g is not 0 or in [1e-6, inf)", static_cast<double>(temperature));
  return verify_common(target_logits, draft_logits, dtype, draft_tokens, B, gamma, V, nullptr, nullptr, temperature,
                       temperature == 0.f, seed, out_tokens, n_accepted, workspace, ws_bytes, nullptr, stream, true);
}

ssd_status ssd_verify_noalloc(const void* target_logits, const void* draft_logits, ssd_dtype dtype,
                              const int32_t* draft_tokens, int B, int gamma, int V, float temperature, uint64_t seed,
                              int32_t* out_tokens, int32_t* n_accepted, void* stream) {
  g_last_error.clear();
  if (!temperature_valid(temperature))
    return fail(SSD_ERR_TEMPERATURE, "temperature %g is not 0 or in [1e-6, inf)", static_cast<double>(temperature));
  if (B < 1 || gamma < 0 || gamma > SSD_MAX_GAMMA)
    return fail(SSD_ERR_SHAPE, "bad shape B=%d gamma=%d V=%d", B, gamma, V);
  const size_t need = workspace_layout(B, gamma).total;
  if (need > SSD_NOALLOC_SCRATCH_BYTES)
    return fail(SSD_ERR_WORKSPACE,
                "B=%d gamma=%d needs %zu bytes of scratch, above the fixed %u-byte array of ssd_verify_noalloc "
                "(B*(gamma+1) <= 1600 always fits); call ssd_verify with a workspace instead",
                B, gamma, need, SSD_NOALLOC_SCRATCH_BYTES);
  void* scratch = nullptr;
  const ssd_status st = noalloc_scratch(static_cast<cudaStream_t>(stream), &scratch);
  if (st != SSD_OK) return st;
  return verify_common(target_logits, draft_logits, dtype, draft_tokens, B, gamma, V, nullptr, nullptr, temperature,
                       temperature == 0.f, seed, out_tokens, n_accepted, scratch, SSD_NOALLOC_SCRATCH_BYTES, nullptr,
                       stream);
}

ssd_status ssd_verify_ragged(const void* target_logits, const void* draft_logits, ssd_dtype dtype,
                             const int32_t* draft_tokens, int B, int gamma_max, int V, const int32_t* gamma,
                             const float* temperature, uint64_t seed, int32_t* out_tokens, int32_t* n_accepted,
                             void* workspace, size_t ws_bytes, void* stream) {
  g_last_error.clear();
  if (!gamma || !temperature) return fail(SSD_ERR_NULL, "gamma / temperature arrays are NULL");
  return verify_common(target_logits, draft_logits, dtype, draft_tokens, B, gamma_max, V, gamma, temperature, 0.f,
                       false, seed, out_tokens, n_accepted, workspace, ws_bytes, nullptr, stream);
}

ssd_status ssd_verify_ragged_pipelined(const void* target_logits, const void* draft_logits, ssd_dtype dtype,
                                       const int32_t* draft_tokens, int B, int gamma_max, int V,
                                       const int32_t* gamma, const float* temperature, uint64_t seed,
                                       int32_t* out_tokens, int32_t* n_accepted, void* workspace, size_t ws_bytes,
                                       void* stream) {
  g_last_error.clear();
  if (!gamma || !temperature) return fail(SSD_ERR_NULL, "gamma / temperature arrays are NULL");
  return verify_common(target_logits, draft_logits, dtype, draft_tokens, B, gamma_max, V, gamma, temperature, 0.f,
                       false, seed, out_tokens, n_accepted, workspace, ws_bytes, nullptr, stream, true);
}

ssd_status ssd_debug_rowstats(const void* target_logits, const void* draft_logits, ssd_dtype dtype,
                              const int32_t* draft_tokens, int B, int gamma, int V, float temperature,
                              uint64_t seed, int32_t* out_tokens, int32_t* n_accepted, float* stats, void* workspace,
                              size_t ws_bytes, void* stream) {
  g_last_error.clear();
  if (!stats) return fail(SSD_ERR_NULL, "stats is NULL");
  if (!temperature_valid(temperature))
    return fail(SSD_ERR_TEMPERATURE, "temperature %g is not 0 or in [1e-6, inf)", static_cast<double>(temperature));
  if (B < 1 || gamma < 0 || gamma > SSD_MAX_GAMMA) return fail(SSD_ERR_SHAPE, "bad shape");
  const size_t n_stats = static_cast<size_t>(B) * (gamma + 1) * SSD_NSTAT_VERIFY;
  cudaError_t e = cudaMemsetAsync(stats, 0xFF, n_stats * sizeof(float), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stats memset");
  return verify_common(target_logits, draft_logits, dtype, draft_tokens, B, gamma, V, nullptr, nullptr, temperature,
                       temperature == 0.f, seed, out_tokens, n_accepted, workspace, ws_bytes, stats, stream);
}

// Verification outputs of a fused call (ssd_verify_saguaro); null members
// mean a Saguaro-only call.
struct FusedVerify {
  const int32_t* draft_tokens = nullptr;
  int32_t* out_tokens = nullptr;
  int32_t* n_accepted = nullptr;
  int32_t* hit = nullptr;
  int32_t* n_hits = nullptr;
};

static ssd_status saguaro_common(const void* target, const void* draft, ssd_dtype dtype, int B, int g, int V, int k,
                                 ssd_topk_source src, float temperature, uint64_t seed, int32_t* bonus_topk,
                                 int32_t* tokens, float* stats,
                                 void* workspace, size_t ws_bytes, void* stream, const FusedVerify& fv = FusedVerify()) {
  const int es = esize_of(dtype);
  const bool fused = fv.out_tokens != nullptr;
  if (es == 0) return fail(SSD_ERR_DTYPE, "unknown dtype %d", static_cast<int>(dtype));
  if (!target || !bonus_topk || !tokens || !workspace || (g > 0 && !draft))
    return fail(SSD_ERR_NULL, "a required pointer is NULL");
  if (fused && (!fv.n_accepted || (g > 0 && !fv.draft_tokens)))
    return fail(SSD_ERR_NULL, "n_accepted / draft_tokens is NULL");
  if (fused && (!aligned_to(fv.out_tokens, 4) || !aligned_to(fv.n_accepted, 4) ||
                (fv.draft_tokens && !aligned_to(fv.draft_tokens, 4)) || (fv.hit && !aligned_to(fv.hit, 4)) ||
                (fv.n_hits && !aligned_to(fv.n_hits, 4))))
    return fail(SSD_ERR_ALIGN, "a token / output pointer is not 4-byte aligned");
  if (B < 1 || g < 0 || g > SSD_MAX_GAMMA || V < 1 || V > SSD_MAX_V || k < 1 || k > SSD_MAX_TOPK || k > V)
    return fail(SSD_ERR_SHAPE, "bad shape B=%d gamma=%d V=%d k=%d", B, g, V, k);
  if (src != SSD_TOPK_RESIDUAL && src != SSD_TOPK_DRAFT)
    return fail(SSD_ERR_SHAPE, "unknown top-k source %d", static_cast<int>(src));
  if (!(temperature >= 1e-6f) || !isfinite(temperature))
    return fail(SSD_ERR_TEMPERATURE, "Saguaro needs a temperature in [1e-6, inf), got %g",
                static_cast<double>(temperature));
  if (!aligned_to(target, es) || (draft && !aligned_to(draft, es)) || !aligned_to(bonus_topk, 4) ||
      !aligned_to(tokens, 4) || (stats && !aligned_to(stats, 4)) || !aligned_to(workspace, 16))
    return fail(SSD_ERR_ALIGN, "a pointer is not aligned to its element size (workspace: 16 bytes)");
  const SagLayout L = saguaro_layout(B, g, V);
  if (ws_bytes < L.total)
    return fail(SSD_ERR_WORKSPACE, "workspace of %zu bytes < %zu required", ws_bytes, L.total);
  const bool aligned =
      aligned_to(target, 16) && (!draft || aligned_to(draft, 16)) && ((static_cast<size_t>(V) * es) % 16 == 0);
  ChunkGeometry geo;
  int smem = 0;
  ssd_status st = choose_chunks(V, es, aligned, &geo, &smem);
  if (st != SSD_OK) return st;
  // Pieces per warp of the residual and mix kernels (SSDV_SAG_PPW overrides).
  geo.ppw = std::max(kSagMinPpw, env_int("SSDV_SAG_PPW", 16));
  const int npw = (geo.npiece + geo.ppw - 1) / geo.ppw;
  const int W = g + 1;
  if (static_cast<long long>(B) * W * geo.nchunk >= (1LL << 31)) return fail(SSD_ERR_SHAPE, "grid too large");
  if (stats) {
    const size_t n_stats = static_cast<size_t>(B) * W * SSD_NSTAT_SAGUARO;
    cudaError_t e = cudaMemsetAsync(stats, 0xFF, n_stats * sizeof(float), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "stats memset");
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* status = reinterpret_cast<int32_t*>(ws);
  // Segments of requests (SSDV_SAG_SEGMENT; at most 65535, the grid's third
  // dimension): each runs the streaming, residual and mix kernels on its own
  // workspace rows; a later segment streams while the previous one finishes.
  int seg = env_int("SSDV_SAG_SEGMENT", 65535);
  seg = std::max(1, std::min(seg, 65535));
  for (int b0 = 0; b0 < B; b0 += seg) {
    const int nb = B - b0 < seg ? B - b0 : seg;
    const size_t u0 = static_cast<size_t>(b0) * W;
    const void* t = static_cast<const uint8_t*>(target) + u0 * V * es;
    const void* d = draft ? static_cast<const uint8_t*>(draft) + static_cast<size_t>(b0) * g * V * es : nullptr;
    VerifyArgs v = {};
    v.target = t;
    v.draft = d;
    v.draft_tokens = nullptr;
    v.B = nb;
    v.gmax = g;
    v.req_base = b0;
    v.gamma = nullptr;
    v.temps = nullptr;
    v.temp_scalar = temperature;
    v.seed = seed;
    v.part = reinterpret_cast<float4*>(ws + L.part) + u0 * geo.nchunk * 2;
    v.ticket = reinterpret_cast<int32_t*>(ws + L.ticket2) + u0;  // cleared by the streaming kernel
    v.status = status;
    v.stats = nullptr;
    v.debug = 0;
    v.first = b0 == 0 ? 1 : 0;
    v.req_major = 1;  // request-major streaming: measured faster for the Saguaro passes
    v.geo = geo;
    // The streaming kernel: one read of every row, whose records serve
    // verification and Saguaro alike.
    cudaError_t e = launch_stream(v, es, smem, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "saguaro streaming launch");
    if (fused) {
      // Verification draws after the residual pass, from its piece sums: for
      // every acceptance length j they are the sums, in the same order and
      // arithmetic, of the very weights the verification's draw at n = j
      // uses ((q_j - p_j)+ scaled by Z_t, or q_gamma at the bonus), so the
      // draw rows are not read again.
      v.draft_tokens = fv.draft_tokens ? fv.draft_tokens + static_cast<size_t>(b0) * g : nullptr;
      v.out_tokens = fv.out_tokens + u0;
      v.n_accepted = fv.n_accepted + b0;
      v.psum = reinterpret_cast<float*>(ws + L.psum2) + u0 * geo.npiece;
      v.pieces_ready = 1;
    }
    SagArgs a;
    a.target = t;
    a.draft = d;
    a.B = nb;
    a.g = g;
    a.k = k;
    a.nj = W;
    a.topk_src = src == SSD_TOPK_DRAFT ? 1 : 0;
    a.req_base = b0;
    a.temperature = temperature;
    a.seed = seed;
    a.npw = npw;
    a.bonus_topk = bonus_topk + u0 * k;
    a.saguaro_tokens = tokens + u0;
    a.stats = stats ? stats + u0 * SSD_NSTAT_SAGUARO : nullptr;
    a.part = v.part;
    a.psum2 = reinterpret_cast<float*>(ws + L.psum2) + u0 * geo.npiece;
    a.psum3 = reinterpret_cast<float*>(ws + L.psum3) + u0 * geo.npiece;
    a.cand_v = reinterpret_cast<float*>(ws + L.cand_v) + u0 * npw * SSD_MAX_TOPK;
    a.cand_i = reinterpret_cast<int32_t*>(ws + L.cand_i) + u0 * npw * SSD_MAX_TOPK;
    a.rowstat = reinterpret_cast<float4*>(ws + L.rowstat) + u0;
    a.rowsum = reinterpret_cast<double*>(ws + L.rowsum) + u0;
    a.zsum = nullptr;
    a.ticket2 = v.ticket;
    a.ticket3 = reinterpret_cast<int32_t*>(ws + L.ticket3) + u0;
    a.status = status;
    a.geo = geo;
    if (fused) {
      e = launch_saguaro(a, es, static_cast<cudaStream_t>(stream), kSagResidual);
      if (e == cudaSuccess) e = launch_sample(v, es, static_cast<cudaStream_t>(stream));
      if (e == cudaSuccess) e = launch_saguaro(a, es, static_cast<cudaStream_t>(stream), kSagMix);
    } else {
      e = launch_saguaro(a, es, static_cast<cudaStream_t>(stream));
    }
    if (e != cudaSuccess) return cuda_fail(e, "saguaro launch");
  }
  if (fused && (fv.hit || fv.n_hits)) {
    const cudaError_t e = launch_cache_check(bonus_topk, fv.out_tokens, fv.n_accepted, B, W, k, fv.hit, fv.n_hits,
                                             static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cache check launch");
  }
  return SSD_OK;
}

ssd_status ssd_saguaro_prespec(const void* target_logits, const void* draft_logits, ssd_dtype dtype, int B, int gamma,
                               int V, int k, ssd_topk_source topk_source, float temperature, uint64_t seed,
                               int32_t* bonus_topk,
                               int32_t* saguaro_tokens, void* workspace, size_t ws_bytes, void* stream) {
  g_last_error.clear();
  return saguaro_common(target_logits, draft_logits, dtype, B, gamma, V, k, topk_source, temperature, seed,
                        bonus_topk, saguaro_tokens, nullptr, workspace, ws_bytes, stream);
}

ssd_status ssd_debug_saguaro_stats(const void* target_logits, const void* draft_logits, ssd_dtype dtype, int B,
                                   int gamma, int V, int k, ssd_topk_source topk_source, float temperature,
                                   uint64_t seed, int32_t* bonus_topk,
                                   int32_t* saguaro_tokens, float* stats, void* workspace, size_t ws_bytes,
                                   void* stream) {
  g_last_error.clear();
  if (!stats) return fail(SSD_ERR_NULL, "stats is NULL");
  return saguaro_common(target_logits, draft_logits, dtype, B, gamma, V, k, topk_source, temperature, seed,
                        bonus_topk, saguaro_tokens, stats, workspace, ws_bytes, stream);
}

ssd_status ssd_verify_saguaro(const void* target_logits, const void* draft_logits, ssd_dtype dtype,
                              const int32_t* draft_tokens, int B, int gamma, int V, int k,
                              ssd_topk_source topk_source, float temperature, uint64_t seed, int32_t* out_tokens,
                              int32_t* n_accepted, int32_t* bonus_topk,
                              int32_t* saguaro_tokens, int32_t* hit, int32_t* n_hits, void* workspace,
                              size_t ws_bytes, void* stream) {
  g_last_error.clear();
  if (!out_tokens) return fail(SSD_ERR_NULL, "out_tokens is NULL");
  FusedVerify fv;
  fv.draft_tokens = draft_tokens;
  fv.out_tokens = out_tokens;
  fv.n_accepted = n_accepted;
  fv.hit = hit;
  fv.n_hits = n_hits;
  return saguaro_common(target_logits, draft_logits, dtype, B, gamma, V, k, topk_source, temperature, seed,
                        bonus_topk, saguaro_tokens, nullptr, workspace, ws_bytes, stream, fv);
}

ssd_status ssd_verify_saguaro_draft(const void* target_logits, const void* draft_logits, ssd_dtype dtype,
                                    const int32_t* draft_tokens, int B, int gamma, int V, float temperature,
                                    uint64_t seed, int32_t* out_tokens, int32_t* n_accepted, void* workspace,
                                    size_t ws_bytes, void* stream) {
  g_last_error.clear();
  const int es = esize_of(dtype);
  const int g = gamma;
  if (es == 0) return fail(SSD_ERR_DTYPE, "unknown dtype %d", static_cast<int>(dtype));
  if (!target_logits || !out_tokens || !n_accepted || !workspace || (g > 0 && (!draft_logits || !draft_tokens)))
    return fail(SSD_ERR_NULL, "a required pointer is NULL");
  if (B < 1 || g < 0 || g > SSD_MAX_GAMMA || V < 1 || V > SSD_MAX_V)
    return fail(SSD_ERR_SHAPE, "bad shape B=%d gamma=%d V=%d", B, g, V);
  if (!(temperature >= 1e-6f) || !isfinite(temperature))
    return fail(SSD_ERR_TEMPERATURE, "Saguaro sampling needs a temperature in [1e-6, inf), got %g",
                static_cast<double>(temperature));
  if (!aligned_to(target_logits, es) || (draft_logits && !aligned_to(draft_logits, es)) ||
      !aligned_to(out_tokens, 4) || !aligned_to(n_accepted, 4) || (draft_tokens && !aligned_to(draft_tokens, 4)) ||
      !aligned_to(workspace, 16))
    return fail(SSD_ERR_ALIGN, "a pointer is not aligned to its element size (workspace: 16 bytes)");
  const SagLayout L = saguaro_layout(B, g, V);
  if (ws_bytes < L.total)
    return fail(SSD_ERR_WORKSPACE, "workspace of %zu bytes < %zu required", ws_bytes, L.total);
  const bool aligned = aligned_to(target_logits, 16) && (!draft_logits || aligned_to(draft_logits, 16)) &&
                       ((static_cast<size_t>(V) * es) % 16 == 0);
  ChunkGeometry geo;
  int smem = 0;
  ssd_status st = choose_chunks(V, es, aligned, &geo, &smem);
  if (st != SSD_OK) return st;
  const int W = g + 1;
  if (static_cast<long long>(B) * W * geo.nchunk >= (1LL << 31)) return fail(SSD_ERR_SHAPE, "grid too large");
  ChunkGeometry sgeo = geo;
  sgeo.ppw = std::max(kSagMinPpw, env_int("SSDV_SAG_PPW", 16));
  const int npw = (geo.npiece + sgeo.ppw - 1) / sgeo.ppw;
  geo.ppw = std::max(1, env_int("SSDV_PPW", 2));
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* status = reinterpret_cast<int32_t*>(ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Per segment of requests: the streaming kernel (records and the draft
  // tokens' logits), the Saguaro residual and mix passes over positions
  // 0..gamma-1 (residual masses S_i and normalisers Zs, no top-k, no draw),
  // then the sampling kernel with p' in place of p.
  int seg = env_int("SSDV_SAG_SEGMENT", 65535);
  seg = std::max(1, std::min(seg, 65535));
  for (int b0 = 0; b0 < B; b0 += seg) {
    const int nb = B - b0 < seg ? B - b0 : seg;
    const size_t u0 = static_cast<size_t>(b0) * W;
    VerifyArgs v = {};
    v.target = static_cast<const uint8_t*>(target_logits) + u0 * V * es;
    v.draft = draft_logits ? static_cast<const uint8_t*>(draft_logits) + static_cast<size_t>(b0) * g * V * es
                           : nullptr;
    v.draft_tokens = draft_tokens ? draft_tokens + static_cast<size_t>(b0) * g : nullptr;
    v.B = nb;
    v.gmax = g;
    v.req_base = b0;
    v.temp_scalar = temperature;
    v.seed = seed;
    v.out_tokens = out_tokens + u0;
    v.n_accepted = n_accepted + b0;
    v.part = reinterpret_cast<float4*>(ws + L.part) + u0 * geo.nchunk * 2;
    v.psum = reinterpret_cast<float*>(ws + L.psum2) + u0 * geo.npiece;
    v.ticket = reinterpret_cast<int32_t*>(ws + L.ticket2) + u0;
    v.status = status;
    v.sag_S = reinterpret_cast<double*>(ws + L.rowsum) + u0;
    v.sag_Zs = reinterpret_cast<float*>(ws + L.zsum) + u0;
    v.first = b0 == 0 ? 1 : 0;
    v.req_major = 1;  // request-major streaming: measured faster for the Saguaro passes
    v.geo = geo;
    cudaError_t e = launch_stream(v, es, smem, s);
    if (e != cudaSuccess) return cuda_fail(e, "streaming launch");
    if (g > 0) {
      SagArgs a = {};
      a.target = v.target;
      a.draft = v.draft;
      a.B = nb;
      a.g = g;
      a.k = 0;
      a.nj = g;
      a.req_base = b0;
      a.temperature = temperature;
      a.seed = seed;
      a.npw = npw;
      a.part = v.part;
      a.psum2 = reinterpret_cast<float*>(ws + L.psum2) + u0 * geo.npiece;
      a.psum3 = reinterpret_cast<float*>(ws + L.psum3) + u0 * geo.npiece;
      a.rowstat = reinterpret_cast<float4*>(ws + L.rowstat) + u0;
      a.rowsum = const_cast<double*>(v.sag_S);
      a.zsum = const_cast<float*>(v.sag_Zs);
      a.ticket2 = v.ticket;
      a.ticket3 = reinterpret_cast<int32_t*>(ws + L.ticket3) + u0;
      a.status = status;
      a.geo = sgeo;
      e = launch_saguaro(a, es, s);
      if (e != cudaSuccess) return cuda_fail(e, "saguaro launch");
    }
    e = launch_sample(v, es, s);
    if (e != cudaSuccess) return cuda_fail(e, "sampling launch");
  }
  return SSD_OK;
}

ssd_status ssd_cache_check(const int32_t* bonus_topk, const int32_t* out_tokens, const int32_t* n_accepted, int B,
                           int gamma, int k, int32_t* hit, int32_t* n_hits, void* stream) {
  g_last_error.clear();
  if (!bonus_topk || !out_tokens || !n_accepted || (!hit && !n_hits))
    return fail(SSD_ERR_NULL, "a required pointer is NULL");
  if (B < 1 || gamma < 0 || gamma > SSD_MAX_GAMMA || k < 1 || k > SSD_MAX_TOPK)
    return fail(SSD_ERR_SHAPE, "bad shape B=%d gamma=%d k=%d", B, gamma, k);
  if (!aligned_to(bonus_topk, 4) || !aligned_to(out_tokens, 4) || !aligned_to(n_accepted, 4) ||
      (hit && !aligned_to(hit, 4)) || (n_hits && !aligned_to(n_hits, 4)))
    return fail(SSD_ERR_ALIGN, "a pointer is not 4-byte aligned");
  const cudaError_t e = launch_cache_check(bonus_topk, out_tokens, n_accepted, B, gamma + 1, k, hit, n_hits,
                                           static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cache check launch");
  return SSD_OK;
}

ssd_status ssd_debug_uniforms(uint64_t seed, int B, int W, float* out, void* stream) {
  g_last_error.clear();
  if (!out) return fail(SSD_ERR_NULL, "out is NULL");
  if (B < 1 || W < 1 || static_cast<long long>(B) * W >= (1LL << 31)) return fail(SSD_ERR_SHAPE, "bad shape");
  const cudaError_t e = launch_uniforms(seed, B, W, out, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "uniforms launch");
  return SSD_OK;
}

ssd_status ssd_read_status(void* workspace, size_t ws_bytes, int* status, void* stream) {
  g_last_error.clear();
  if (!workspace || !status) return fail(SSD_ERR_NULL, "a required pointer is NULL");
  if (ws_bytes < 16) return fail(SSD_ERR_WORKSPACE, "workspace too small");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t bits = 0;
  cudaError_t e = cudaMemcpyAsync(&bits, workspace, sizeof bits, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof bits, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  *status = SSD_OK;
  for (int c = 1; c < 32; ++c)
    if (bits & (1 << c)) {
      *status = c;
      break;
    }
  return SSD_OK;
}

const char* ssd_status_str(ssd_status status) {
  switch (status) {
    case SSD_OK: return "SSD_OK";
    case SSD_ERR_NULL: return "SSD_ERR_NULL: a required pointer is NULL";
    case SSD_ERR_SHAPE: return "SSD_ERR_SHAPE: B, gamma, V or k out of range";
    case SSD_ERR_DTYPE: return "SSD_ERR_DTYPE: unknown dtype";
    case SSD_ERR_ALIGN: return "SSD_ERR_ALIGN: misaligned pointer";
    case SSD_ERR_TOKEN_RANGE: return "SSD_ERR_TOKEN_RANGE: a draft token outside [0, V)";
    case SSD_ERR_TEMPERATURE: return "SSD_ERR_TEMPERATURE: invalid temperature";
    case SSD_ERR_CUDA: return "SSD_ERR_CUDA: a CUDA runtime call failed";
    case SSD_ERR_UNSUPPORTED: return "SSD_ERR_UNSUPPORTED: no launch configuration fits";
    case SSD_ERR_WORKSPACE: return "SSD_ERR_WORKSPACE: workspace missing or too small";
    case SSD_ERR_GAMMA: return "SSD_ERR_GAMMA: a per-request gamma above gamma_max";
    case SSD_ERR_DRAW: return "SSD_ERR_DRAW: a draw found no token of positive weight";
  }
  return "unknown ssd_status";
}

const char* ssd_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
