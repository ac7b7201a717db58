// Internal launch interface between the C ABI (capi.cu) and the kernels.
// Every launcher only enqueues work on `stream` and returns the launch error.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace csa2 {

// Sets the thread-local text returned by csa2_last_error(); returns `code`.
int record_error(int code, const char* msg);

// Host checks of a Reindex call (batch, ratio m, pointers, alignment, page
// table); CSA2_OK or the failing status with its error text set.
int check_reindex(const uint8_t* q_codes, const uint8_t* q_scales, const float* w, const int64_t* seq_len, int B,
                  int n_q, const int32_t* block_table, int max_pages, int64_t n_pages, const uint8_t* idx_pages,
                  const int32_t* pool, const int32_t* topk, int m);

// Each kernel translation unit keeps its own device status word; these read
// (and optionally clear) it. Synchronous with respect to `stream`.
cudaError_t status_append(cudaStream_t stream, int* code, int* where, bool clear);
cudaError_t status_indexer(cudaStream_t stream, int* code, int* where, bool clear);
cudaError_t status_topk(cudaStream_t stream, int* code, int* where, bool clear);
cudaError_t status_attn(cudaStream_t stream, int* code, int* where, bool clear);
// Sets the forced-timeout site of each translation unit's bounded waits (0 = off).
cudaError_t force_timeout_append(int site, cudaStream_t stream);
cudaError_t force_timeout_indexer(int site, cudaStream_t stream);
cudaError_t force_timeout_topk(int site, cudaStream_t stream);
cudaError_t force_timeout_attn(int site, cudaStream_t stream);

cudaError_t launch_append_kv(const void* latent, const void* idx_key, const int32_t* seq_idx,
                             const int64_t* pos, int T, const int32_t* block_table, int B,
                             int max_pages, int64_t n_pages, uint8_t* main_pages,
                             uint8_t* idx_pages, cudaStream_t stream);
// One decode step's appends and indexer-query quantisations in one launch:
// the main append (as launch_append_kv), then per layer its window entries
// (as launch_append_swa, with the call's pos and T; swa == NULL: none) and
// its query (as launch_quant_mxfp4; q_idx == NULL: none). kv_blocks is set
// by the launcher.
constexpr int kMaxAppendLayers = 16;
struct DecodeAppendsLayer {
  const void* swa;
  const int32_t* ring_idx;
  int64_t n_rings;
  uint8_t* rings;
  const void* q_idx;
  int64_t q_n;
  uint8_t* q_codes;
  uint8_t* q_scales;
};
struct DecodeAppends {
  const void* latent;
  const void* idx_key;
  const int32_t* seq_idx;
  const int64_t* pos;
  int T;
  const int32_t* block_table;
  int B, max_pages;
  int64_t n_pages;
  uint8_t* main_pages;
  uint8_t* idx_pages;
  int n_layers, kv_blocks;
  DecodeAppendsLayer layer[kMaxAppendLayers];
};
cudaError_t launch_decode_appends(const DecodeAppends& P, cudaStream_t stream);
// Encoder-side append at ratio m (1 or 2): entries from groups of m tokens
// (softmax of their logits per channel), MXFP4 into entry pages; pending
// tokens into tail [B][m-1][1280] bf16.
cudaError_t launch_compress_append(const void* kv, const void* kv_gate, const void* idx_key, const void* idx_gate,
                                   const int32_t* seq_idx, const int64_t* pos, int T, int m, void* tail,
                                   const int32_t* block_table, int B, int max_pages, int64_t n_pages,
                                   uint8_t* main_pages, uint8_t* idx_pages, cudaStream_t stream);
// ring_idx == NULL: E4M3 of T entries into rings viewed as [T, 512] (pos unused).
cudaError_t launch_append_swa(const void* x, const int32_t* ring_idx, const int64_t* pos, int T,
                              int64_t n_rings, uint8_t* rings, cudaStream_t stream);
// The last min(n, 128) of n E4M3 entries per sequence into their ring slots.
cudaError_t launch_ring_refill(const uint8_t* entries, const int64_t* seq_len, int B, int n,
                               const int32_t* ring_idx, int64_t n_rings, uint8_t* rings, cudaStream_t stream);
cudaError_t launch_quant_mxfp4(const void* x, int64_t n, uint8_t* codes, uint8_t* scales,
                               cudaStream_t stream);
cudaError_t launch_dequant_mxfp4(const uint8_t* codes, const uint8_t* scales, int64_t n,
                                 float* out, cudaStream_t stream);
cudaError_t launch_quant_fp8(const float* x, int64_t n, uint8_t* out, cudaStream_t stream);

// Full-mode scan -> block maxima.
cudaError_t launch_indexer_scan(const uint8_t* q_codes, const uint8_t* q_scales, const float* w,
                                const int64_t* seq_len, int B, int n_q, int64_t max_ctx,
                                const int32_t* block_table, int max_pages, int64_t n_pages,
                                const uint8_t* idx_pages, float* block_max, int64_t max_blocks,
                                cudaStream_t stream, int m = 1);
// Pool rescore -> per-slot scores [B*n_q, 2048*8] (-inf for empty / future slots).
cudaError_t launch_pool_scores(const uint8_t* q_codes, const uint8_t* q_scales, const float* w,
                               const int64_t* seq_len, int B, int n_q,
                               const int32_t* block_table, int max_pages, int64_t n_pages,
                               const uint8_t* idx_pages, const int32_t* pool, float* scores,
                               cudaStream_t stream, int m = 1);

// Top-k selections (one CTA per query token).
cudaError_t launch_block_topk(const float* block_max, const int64_t* seq_len, int B, int n_q,
                              int64_t max_blocks, int32_t* pool, cudaStream_t stream, int m = 1);
cudaError_t launch_pool_topk(const float* scores, const int64_t* seq_len, int B, int n_q,
                             const int32_t* pool, int32_t* topk, cudaStream_t stream);

// Sparse attention: split partials + combine.
size_t attn_workspace_bytes(int64_t queries);
cudaError_t launch_sparse_attn(const void* q, const int32_t* topk, const int64_t* seq_len, int B,
                               int n_q, const int32_t* block_table, int max_pages,
                               int64_t n_pages, const uint8_t* main_pages, const uint8_t* rings,
                               const int32_t* ring_idx, int64_t n_rings, const uint8_t* swa_chunk,
                               float softmax_scale, int out_dtype, void* out, float* lse, void* ws,
                               cudaStream_t stream, int m = 1);

}  // namespace csa2
