// Reindex-mode indexer for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: plug-ins whose host framework
// owns every device allocation, and decode loops that forbid allocation on
// the decode path (an allocation there can synchronise the device or fail
// under memory pressure in the middle of a step). csa2_indexer_reindex needs
// a caller workspace for its per-slot scores; csa2_indexer_reindex_noalloc
// keeps those scores in a fixed array of device memory inside this library
// instead.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it until the process exits. In host code its name is only a
// host-side stand-in, so the device address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and passed to the kernels.
#include <nvtx3/nvToolsExt.h>
#include <cstdio>
#include <mutex>

#include "csa2.h"
#include "kernels.h"

namespace {

constexpr int kMaxQueries = 64;                 // B * n_q per call
constexpr size_t kSlotsPerQuery = 2048 * 8;     // pool blocks x positions
constexpr int kMaxDevices = 64;

// 64 x 16384 fp32 = 4 MiB. Every call overwrites every slot it reads (the
// rescore kernel writes all 16384 slots of each query before the top-k kernel
// reads them), so nothing has to start at zero.
static __device__ __align__(256) float g_noalloc_scores[kMaxQueries * kSlotsPerQuery];

std::mutex g_mu;
float* g_scores_ptr[kMaxDevices] = {};

}  // namespace

extern "C" {

// Documented in include/csa2.h next to csa2_indexer_reindex.
int csa2_indexer_reindex_noalloc(const uint8_t* q_codes, const uint8_t* q_scales, const float* w,
                                 const int64_t* seq_len, int B, int n_q,
                                 const int32_t* block_table, int max_pages, int64_t n_pages,
                                 const uint8_t* idx_pages, const int32_t* pool, int32_t* topk, int m,
                                 void* stream) {
  nvtxRangePushA(__func__);
  struct Pop {
    ~Pop() { nvtxRangePop(); }
  } pop;
  // The same checks (and status codes) as csa2_indexer_reindex, then the
  // limit of the fixed scratch array.
  if (int st = csa2::check_reindex(q_codes, q_scales, w, seq_len, B, n_q, block_table, max_pages, n_pages,
                                   idx_pages, pool, topk, m))
    return st;
  if (B == 0) return CSA2_OK;
  char msg[256];
  if (static_cast<int64_t>(B) * n_q > kMaxQueries) {
    snprintf(msg, sizeof(msg),
             "reindex_noalloc: B * n_q = %lld exceeds the fixed scratch of %d query tokens (4 MiB); "
             "split the batch or use csa2_indexer_reindex with a workspace",
             static_cast<long long>(B) * n_q, kMaxQueries);
    return csa2::record_error(CSA2_ERR_UNSUPPORTED, msg);
  }

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return csa2::record_error(CSA2_ERR_CUDA, "reindex_noalloc: no usable current device");
  float* scores = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scores_ptr[dev]) {
      // First call on this device: look up the array's device address.
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scores);
      if (e != cudaSuccess || !p) {
        snprintf(msg, sizeof(msg), "reindex_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
        return csa2::record_error(CSA2_ERR_CUDA, msg);
      }
      g_scores_ptr[dev] = static_cast<float*>(p);
    }
    scores = g_scores_ptr[dev];
  }
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = csa2::launch_pool_scores(q_codes, q_scales, w, seq_len, B, n_q, block_table, max_pages,
                                           n_pages, idx_pages, pool, scores, s, m);
  if (e == cudaSuccess) e = csa2::launch_pool_topk(scores, seq_len, B, n_q, pool, topk, s);
  if (e != cudaSuccess) {
    snprintf(msg, sizeof(msg), "reindex_noalloc launch: %s", cudaGetErrorString(e));
    return csa2::record_error(CSA2_ERR_CUDA, msg);
  }
  return CSA2_OK;
}

}  // extern "C"
