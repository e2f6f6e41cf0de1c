// ssdv_internal.h -- launch arguments shared by the host launchers and the
// kernels of libssdv (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "ssdv.h"

namespace ssdv {

// How a unit's rows are split across the CTAs of its cluster.
struct Geometry {
  int V;            // vocabulary size
  int slice;        // elements per CTA slice, a multiple of 8 (16 bytes for bf16 and fp32)
  int csize;        // CTAs per cluster (1..16)
  int row_smem;     // shared-memory bytes reserved per staged row slice
  int stage_elems;  // elements per staged copy (one stage)
  int bulk;         // 1: rows 16-byte aligned, staged with bulk async copies
};

// How verification splits each row: the streaming kernel runs one CTA per
// (request, position, chunk); the sampling kernel one warp per piece (128
// vectors) of each request's draw row (of every row in the debug mode).
struct ChunkGeometry {
  int V;         // vocabulary size
  int chunk;     // elements per chunk, a multiple of 8
  int nchunk;    // chunks per row, 1..kMaxChunks
  int row_smem;  // shared-memory bytes per staged row chunk (a multiple of 128)
  int bulk;      // 1: rows 16-byte aligned, staged with bulk async copies
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
  int first;                   // 1: every streaming CTA waits for the previous kernel (the first
                               // segment of a call); 0: only the first CTA waits (a later segment, or
                               // a pipelined call)
  ChunkGeometry geo;
};

struct SaguaroArgs {
  const void* target;  // [B, g+1, V]
  const void* draft;   // [B, g, V]
  int B, g, k;
  float temperature;
  uint64_t seed;
  int32_t* bonus_topk;      // [B, g+1, k]
  int32_t* saguaro_tokens;  // [B, g+1]
  float* stats;             // [B, g+1, SSD_NSTAT_SAGUARO] or null
  Geometry geo;
};

// Workspace layout (byte offsets), shared by the launchers and the API: the
// status word, then two halves used by alternate calls, each holding the
// arrival counters (cleared by every call), chunk records and piece sums of
// the call's shape (ticket .. blocks are offsets within a half).
struct WorkspaceLayout {
  size_t status, half0, half_bytes, ticket, part, csum, blocks, total;
};
WorkspaceLayout workspace_layout(int B, int gmax);

ssd_status choose_chunks(int V, int esize, bool aligned, ChunkGeometry* geo, int* smem_bytes);

// Launch configuration for one call; returns SSD_OK or an error.
ssd_status choose_geometry(int V, int esize, bool aligned, bool two_rows, Geometry* geo, int* smem_bytes);

// Streaming statistics kernel followed by the decision / sampling kernel (both
// with programmatic dependent launch; each waits for its predecessor).
cudaError_t launch_verify(const VerifyArgs& a, int esize, int smem_bytes, cudaStream_t stream);
cudaError_t launch_saguaro(const SaguaroArgs& a, int esize, int smem_bytes, cudaStream_t stream);

cudaError_t launch_uniforms(uint64_t seed, int B, int W, float* out, cudaStream_t stream);

// Largest dynamic shared memory one CTA may use (bytes).
int max_dynamic_smem();

}  // namespace ssdv
