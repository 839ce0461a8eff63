// Internal launch parameters and launchers of the Vegas kernels (host + device).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "vg.h"

namespace vg {

// Keys per verify tile: the unit of TMA transfer and of the work split.
constexpr int kVerifyTileKeys = 64;
// Longest draft-token tail a sparse draft step attends besides the selection (the
// draft tokens of one iteration number at most gamma + 1 <= 16).
constexpr int kDraftMaxTail = 16;
constexpr int kDraftChunk = 16;   // entries of one pipeline stage of the draft kernel
// Most CTAs in one thread-block cluster of the draft step.
constexpr int kDraftMaxCluster = 16;
// Largest sequence the top-k kernel holds (in shared memory, across a cluster of up to 16).
constexpr int kTopkMaxLen = 262144;
constexpr int kMaxBatch = 1024;

struct VerifyParams {
  const __nv_bfloat16* q;      // [B][R][Hq][D]
  const __nv_bfloat16* k_new;  // [B][R][Hkv][D] or null (read from the cache)
  const __nv_bfloat16* v_new;
  __nv_bfloat16* K;            // cache [capacity][Hkv][D]
  __nv_bfloat16* V;
  const int64_t* seq_offset;   // [B] (slot pool) or null (paged)
  const int32_t* ptab;         // [B][pstride] page table, or null (slot pool)
  int psize, pstride;          // tokens per page, pages per sequence
  int box_rows;                // rows of one K/V TMA box: 64 for the slot pool, else min(page size, 64)
  const int32_t* prefix_len;   // [B]
  int64_t capacity;
  int B, Hq, Hkv, G, R, D, M, Mpad;  // M = G * R rows per KV head, Mpad = 16 * ceil(M / 16)
  int sc_row0;       // first score row of the MMA's A operand (after the query rows, see verify_sc_row0)
  int max_len;
  float scale;       // natural-log units (scores)
  float scale_log2;  // scale * log2(e) (softmax)
  uint32_t mask0, mask1;
  int nctas;         // verify grid size
  // workspace
  int32_t* meta;     // [B + 1] tiles-per-head prefix sums, then [B] checked lengths
  float* part_o;     // [nctas + B*Hkv][Mpad][D]  unnormalised partial outputs
  float* part_ml;    // [nctas + B*Hkv][Mpad][2]  (running max in log2 units, sum)
  float* part_s;     // [2][B][Hkv][2][s_stride]  per-(KV head, high / low part) partial scores
  int s_stride;      // max_len rounded up to a multiple of 64
  // outputs
  float* scores0;    // [B][score_stride] or null
  float* scores1;
  int64_t score_stride;
  __nv_bfloat16* out;  // [B][R][Hq][D]
  int32_t* status;
};

struct TopkParams {
  const float* scores;
  int64_t score_stride;
  const int32_t* len;
  int B, max_len, k;
  int per_cta;  // positions held by one CTA of the cluster
  int32_t* idx;
  int32_t* count;
  int32_t* status;
};

struct DraftParams {
  const __nv_bfloat16* q;      // [B][Hq][D]
  const __nv_bfloat16* k_new;  // [B][Hkv][D] or null
  const __nv_bfloat16* v_new;
  __nv_bfloat16* K;
  __nv_bfloat16* V;
  const int64_t* seq_offset;   // [B] (slot pool) or null (paged)
  const int32_t* ptab;         // [B][pstride] page table, or null (slot pool)
  int psize, pstride;
  int64_t capacity;
  const int32_t* idx;          // [B][k_stride]
  const int32_t* count;        // [B]
  int k_stride;
  const int32_t* tail_start;   // [B]
  const int32_t* tail_len;     // [B] or null -> tail_len_const
  int tail_len_const;
  int slots;                   // entry slots per sequence in the work split: k_stride + the tail bound
  int settled;                 // the selection predates the previous kernel: gather before the wait
  int B, Hq, Hkv, G, D;
  float scale, scale_log2;
  int nctas;
  int nstage;                  // ring stages of the draft kernel (2 or 3)
  float* part_o;               // [nctas + B][Hq][D]  unnormalised partial outputs
  float* part_ml;              // [nctas + B][Hq][2]
  __nv_bfloat16* out;          // [B][Hq][D]
  int32_t* status;
};

// Most 4096-entry tiles of the vocabulary the acceptance step draws from (V <= 2^20).
constexpr int kMaxAcceptTiles = 256;

struct AcceptParams {
  const float* p_logits;   // [B][gamma+1][V]
  const float* q_logits;   // [B][gamma][V] (sampling only)
  const int32_t* draft;    // [B][gamma]
  const float* u;          // [B][gamma] (sampling only)
  const float* u_res;      // [B] (sampling only)
  int B, gamma, V, nchunk, sample;
  float* stats;            // [rows][nchunk] (max, sum, argmax value, argmax) per chunk
  float* dec;              // [B] decision records (sampling): a, row a's statistics
  float* tiles;            // [B][2][ntiles] tile sums of row a's weights: excess, then p
  int ntiles;
  int32_t* n_accept;       // [B]
  int32_t* next_token;     // [B]
  int32_t* advance_len;    // [B] or null
  int32_t* status;
};

// Launchers (return a cudaError_t from the launch).
cudaError_t launch_verify(const VerifyParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                          cudaStream_t stream);
// First score row of the verify MMA's A operand for M query rows and nsc score rows: the
// start of the next lane quadrant (16 rows at M = 64, 32 at M = 128) when the rows still
// fit the same MMA shape, so that the score rows' stores fall to row warps that hold no
// query row; else right after the query rows.
int verify_sc_row0(int M, int nsc);
size_t verify_smem_bytes(int D, int B);
cudaError_t launch_topk(const TopkParams& p, int cluster, cudaStream_t stream, bool pdl);
size_t topk_smem_bytes(int per_cta);
cudaError_t launch_window(const int32_t* len, int B, int max_len, int k, int32_t* idx, int32_t* count,
                          int32_t* status, cudaStream_t stream);
cudaError_t launch_draft(const DraftParams& p, cudaStream_t stream, bool pdl);
size_t draft_smem_bytes(int D, int Hkv, int nstage);  // dynamic shared memory of a draft CTA
int draft_stages(int D, int Hkv, int B, int slots, int nctas, size_t smem_optin);  // 2 or 3
int draft_grid(int B, int slots, int sms);  // CTAs of a draft step
cudaError_t launch_accept(const AcceptParams& p, cudaStream_t stream);
int accept_chunks(int V);  // vocabulary chunks of the statistics kernel
int accept_tiles(int V);   // tiles of the sampling draw over a row of V entries
// Warps of the draft step's combine kernel (4, 8 or 16 from the most partials a
// sequence has), or 0 when every sequence's entries sit in one CTA (no combine runs).
int draft_combine_warps(int B, int slots, int nctas);

}  // namespace vg
