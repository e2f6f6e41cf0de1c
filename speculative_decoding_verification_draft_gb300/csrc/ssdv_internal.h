// ssdv_internal.h -- launch arguments shared by the host launchers and the
// kernels of libssdv (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "ssdv.h"

namespace ssdv {

// How verification splits each row: the streaming kernel runs one CTA per
// (request, position, chunk); the sampling kernel one warp per piece (128
// vectors) of each request's draw row (of every row in the debug mode).
struct ChunkGeometry {
  int V;         // vocabulary size
  int chunk;     // elements per chunk, a multiple of 8
  int nchunk;    // chunks per row, 1..kMaxChunks
  int row_smem;  // shared-memory bytes per row chunk of the shared-memory form (a multiple of 128)
  int aligned;   // 1: rows 16-byte aligned (read with 16-byte vector loads)
  int npiece;    // pieces (128 vectors) per row, at most kMaxPieces
  int ppw;       // pieces per warp of the sampling kernel
};
constexpr int kMaxChunks = 32;
constexpr int kMaxPieces = 1024;  // 2^19 fp32 elements / 512

struct VerifyArgs {
  const void* target;          // [B, gmax+1, V]
  const void* draft;           // [B, gmax, V] (may be null if every request is greedy)
  const int32_t* draft_tokens; // [B, gmax]
  int B, gmax;
  int req_base;                // request index of row 0 in the Philox counters
  const int32_t* gamma;        // [B] or null (every request uses gmax)
  const float* temps;          // [B] or null (temp_scalar)
  float temp_scalar;
  uint64_t seed;
  int32_t* out_tokens;         // [B, gmax+1]
  int32_t* n_accepted;         // [B]
  float4* part;                // workspace [B, gmax+1, nchunk, 2]: per-chunk row statistics
  float* psum;                 // workspace [B, gmax+1, npiece]: per-piece weight sums of the draw rows
  int32_t* ticket;             // workspace [B, gmax+1]: pieces arrived
  int32_t* status;             // workspace [1]: device error bits
  float* stats;                // [B, gmax+1, SSD_NSTAT_VERIFY] or null (debug)
  int debug;                   // 1: decide and report every position (statistics)
  const double* sag_S;         // [B, gmax+1] or null: residual masses S_i (weight units) of the Saguaro
                               // passes; given, the draft tokens were sampled from the Saguaro
                               // distribution p' of their position, which replaces p in the accept test
                               // and the residual
  const float* sag_Zs;         // [B, gmax+1]: the Saguaro normalisers sum_v sqrt(p max(r, 1e-8))
  const float* tp_th;          // [B, gmax+1, 2] or null: top-p nucleus thresholds (logits) of each
                               // target (slot 0) and draft (slot 1) row; given, both distributions are
                               // truncated to their nuclei
  const float* tp_z;           // [B, gmax+1, 2]: the nuclei's masses, in units of exp2(x c - fl(m c))
  int pieces_ready;            // 1: psum already holds the piece sums of every position's draw row,
                               // [B, gmax+1, npiece] (the Saguaro residual pass's): one CTA per request
                               // takes the decision and draws, with no pass over the rows
  int first;                   // 1: every streaming CTA waits for the previous kernel (the first
                               // segment of a call); 0: only the first CTA waits (a later segment, or
                               // a pipelined call)
  int req_major;               // streaming grid order: 1 request by request (chunk, position, request);
                               // 0 position-major (chunk, request, position)
  ChunkGeometry geo;
};

// Saguaro pre-speculation (the residual and mix kernels; the streaming kernel
// of verification supplies the per-chunk records).  Pointers are offset to
// the segment of requests this launch covers; unit u = b * (g + 1) + j.
struct SagArgs {
  const void* target;       // [B, g+1, V]
  const void* draft;        // [B, g, V]
  int B, g, k;               // k = 0: no top-k
  int nj;                   // positions j = 0 .. nj-1 of every request are processed (g + 1, or g)
  int topk_src;             // 0: top-k of the residual; 1: of the draft logits (target logits at j = g)
  int req_base;             // request index of row 0 in the Philox counters
  float temperature;
  uint64_t seed;
  int npw;                  // warps per unit (ceil(npiece / ppw))
  int32_t* bonus_topk;      // [B, g+1, k]
  int32_t* saguaro_tokens;  // [B, g+1], or null: no draw (the normalisers Zs are still kept)
  float* zsum;              // workspace [units] or null: Zs of every unit
  float* stats;             // [B, g+1, SSD_NSTAT_SAGUARO] or null
  const float4* part;       // workspace [units, nchunk, 2]: the streaming kernel's records
  float* psum2;             // workspace [units, npiece]: residual (or target) piece sums
  float* psum3;             // workspace [units, npiece]: Saguaro-weight piece sums
  float* cand_v;            // workspace [units, npw, 8]: every warp's top-8 weights
  int32_t* cand_i;          // workspace [units, npw, 8]: and their indices
  float4* rowstat;          // workspace [units]: target max, target sum, draft max, draft sum
  double* rowsum;           // workspace [units]: S_j in weight units (NaN: the unit failed)
  int32_t* ticket2;         // workspace [units]: residual-kernel warps arrived
  int32_t* ticket3;         // workspace [units]: mix-kernel warps arrived
  int32_t* status;          // workspace [1]: device error bits
  ChunkGeometry geo;
};

// One level of the top-p select.  Level 0: digit = 255 - (mass bin of the
// element); later levels: digit = (key >> shift) & ((1 << bits) - 1) of the
// elements in the chosen bin.
struct TopPArgs {
  const void* target;   // [B, gmax+1, V]
  const void* draft;    // [B, gmax, V]
  int B, gmax;
  const int32_t* gamma; // [B] or null
  const float* temps;   // [B] or null (temp_scalar)
  float temp_scalar;
  float top_p;
  const float4* part;   // the streaming kernel's records
  ChunkGeometry geo;
  int level, nlevels, shift, bits;
  unsigned long long* hist;    // [B, gmax+1, 2, 1 << bits]: this level's histograms (zeroed by the caller)
  uint32_t* bstar;             // [B, gmax+1, 2]: the mass bin holding the threshold (level 0's result)
  uint32_t* prefix;            // [B, gmax+1, 2]: the key digits fixed so far
  unsigned long long* above;   // [B, gmax+1, 2]: mass of keys above the prefix's range
  unsigned long long* goal;    // [B, gmax+1, 2]: ceil(top_p * total mass)
  float* th;                   // [B, gmax+1, 2]: the nucleus threshold (logit), after the last level
  float* z;                    // [B, gmax+1, 2]: the nucleus mass, after the last level
  uint32_t* todo;              // [B, gmax+1, 2]: row slots that level 1 left open (bf16 rows)
  uint32_t* todo_count;        // [1]: their number (zeroed by the caller)
};
cudaError_t launch_topp_level(const TopPArgs& a, int esize, cudaStream_t stream);

// Workspace layout (byte offsets), shared by the launchers and the API: the
// status word, then two halves used by alternate calls, each holding the
// arrival counters (cleared by every call), chunk records and piece sums of
// the call's shape (ticket .. blocks are offsets within a half).
struct WorkspaceLayout {
  size_t status, half0, half_bytes, ticket, part, blocks, total;
};
WorkspaceLayout workspace_layout(int B, int gmax);

ssd_status choose_chunks(int V, int esize, bool aligned, ChunkGeometry* geo, int* smem_bytes);

// Streaming statistics kernel followed by the decision / sampling kernel (both
// with programmatic dependent launch; each waits for its predecessor).
cudaError_t launch_verify(const VerifyArgs& a, int esize, int smem_bytes, cudaStream_t stream);
// Small vocabularies: one warp per request, the whole verification in one
// kernel (no workspace but the status word; no statistics).
constexpr int kSmallV = 256;
cudaError_t launch_small_verify(const VerifyArgs& a, int esize, cudaStream_t stream);
// The sampling kernel alone (after the Saguaro passes it reads).
cudaError_t launch_sample(const VerifyArgs& a, int esize, cudaStream_t stream);
// The streaming kernel alone (Saguaro's first kernel).
cudaError_t launch_stream(const VerifyArgs& a, int esize, int smem_bytes, cudaStream_t stream);
// Saguaro's residual and mix kernels (each waits for its predecessor).
// passes: 1 the residual kernel, 2 the mix kernel, 3 both.
constexpr int kSagResidual = 1, kSagMix = 2;
cudaError_t launch_saguaro(const SagArgs& a, int esize, cudaStream_t stream, int passes = kSagResidual | kSagMix);

// The cache check: hit[b] = the slot of bonus_topk[b, n_b, :] holding
// out_tokens[b, n_b] (-1 if none), n_hits[0] = the number of hits (either
// output may be null).  One kernel, launched after its predecessor.
cudaError_t launch_cache_check(const int32_t* bonus_topk, const int32_t* out_tokens, const int32_t* n_accepted, int B,
                               int W, int k, int32_t* hit, int32_t* n_hits, cudaStream_t stream);

// Saguaro workspace layout (byte offsets from the workspace start; status at 0).
struct SagLayout {
  size_t ticket2, ticket3, rowstat, rowsum, zsum, part, psum2, psum3, cand_v, cand_i, total;
};
constexpr int kSagMinPpw = 2;  // pieces per warp of the Saguaro kernels, at least
SagLayout saguaro_layout(int B, int g, int V);

cudaError_t launch_uniforms(uint64_t seed, int B, int W, float* out, cudaStream_t stream);

// Largest dynamic shared memory one CTA may use (bytes).
int max_dynamic_smem();

}  // namespace ssdv
