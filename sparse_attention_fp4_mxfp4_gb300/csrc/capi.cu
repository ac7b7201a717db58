// C ABI of libcsa2.so: host-side validation, workspace carving and the
// Full / Reindex / Reuse mode dispatcher ("DeepSeek V4.1: model architecture
// and system design, a close reading" section 2.2; "DeepSeek-V4.1-Flash:
// Pushing the Limits of KV Cache Compression" section 3.3). No allocation, no
// synchronisation except in csa2_check_device_status.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "csa2.h"
#include "kernels.h"
#include <nvtx3/nvToolsExt.h>

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(CSA2_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaStream_t S(void* s) { return static_cast<cudaStream_t>(s); }

constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t reindex_ws(int64_t Q) { return align256(static_cast<size_t>(Q) * 16384 * sizeof(float)); }
size_t blockmax_ws(int64_t Q, int64_t max_ctx) {
  return align256(static_cast<size_t>(Q) * static_cast<size_t>((max_ctx + 7) / 8) * sizeof(float));
}

#define CHECK_PTR(p, name)                                                      \
  do {                                                                          \
    if (!(p)) return fail(CSA2_ERR_INVALID_ARG, "%s is NULL", name);            \
  } while (0)
#define CHECK_A16(p, name)                                                      \
  do {                                                                          \
    if (!(p)) return fail(CSA2_ERR_INVALID_ARG, "%s is NULL", name);            \
    if (!aligned16(p)) return fail(CSA2_ERR_INVALID_ARG, "%s is not 16-byte aligned", name); \
  } while (0)

// max_nq: CSA2_MAX_NQ for the decode attention, CSA2_MAX_PREFILL_NQ elsewhere.
int check_batch(int B, int n_q, int max_nq = CSA2_MAX_PREFILL_NQ) {
  if (B < 0) return fail(CSA2_ERR_INVALID_ARG, "B = %d < 0", B);
  if (B > CSA2_MAX_TOKENS) return fail(CSA2_ERR_UNSUPPORTED, "B = %d > %d", B, CSA2_MAX_TOKENS);
  if (n_q < 1) return fail(CSA2_ERR_INVALID_ARG, "n_q = %d < 1", n_q);
  if (n_q > max_nq) return fail(CSA2_ERR_UNSUPPORTED, "n_q = %d > %d", n_q, max_nq);
  if (static_cast<int64_t>(B) * n_q > CSA2_MAX_TOKENS)
    return fail(CSA2_ERR_UNSUPPORTED, "B * n_q = %lld > %d", static_cast<long long>(B) * n_q, CSA2_MAX_TOKENS);
  return CSA2_OK;
}

int check_ratio(int m) {
  if (m != 1 && m != 2) return fail(CSA2_ERR_UNSUPPORTED, "tokens per entry m = %d (1 or 2 supported)", m);
  return CSA2_OK;
}

int check_pages(const int32_t* block_table, int max_pages, int64_t n_pages) {
  CHECK_PTR(block_table, "block_table");
  if (max_pages < 1) return fail(CSA2_ERR_INVALID_ARG, "max_pages = %d < 1", max_pages);
  if (n_pages < 1 || n_pages > (int64_t(1) << 31) - 1)
    return fail(CSA2_ERR_INVALID_ARG, "n_pages = %lld out of range", static_cast<long long>(n_pages));
  return CSA2_OK;
}

}  // namespace

namespace csa2 {
int record_error(int code, const char* msg) { return fail(code, "%s", msg); }
}  // namespace csa2

extern "C" {

// Every compute call of the C ABI opens an NVTX range named after it, so that
// a profiler tracing NVTX shows the library's calls around their kernels
// (without such a tool attached a push and a pop cost a few nanoseconds).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
#define CSA2_NVTX_RANGE() NvtxRange csa2_nvtx_range_(__func__)

const char* csa2_status_string(int status) {
  switch (status) {
    case CSA2_OK: return "ok";
    case CSA2_ERR_INVALID_ARG: return "invalid argument";
    case CSA2_ERR_UNSUPPORTED: return "unsupported shape";
    case CSA2_ERR_WORKSPACE: return "workspace missing or too small";
    case CSA2_ERR_CUDA: return "CUDA error";
    case CSA2_ERR_DEVICE_TIMEOUT: return "a bounded device wait timed out";
    case CSA2_ERR_DEVICE_BOUNDS: return "a device-side index check failed";
    case CSA2_ERR_DEVICE_RANGE: return "an input value outside the supported range";
    default: return "unknown status";
  }
}

const char* csa2_last_error(void) { return g_err; }

int csa2_version(void) { return 1; }

int csa2_page_bytes(int plane, size_t* bytes) {
  CHECK_PTR(bytes, "bytes");
  if (plane == CSA2_PLANE_MAIN) *bytes = CSA2_PAGE_TOKENS * CSA2_MAIN_ENTRY_BYTES;
  else if (plane == CSA2_PLANE_INDEX) *bytes = CSA2_PAGE_TOKENS * CSA2_IDX_ENTRY_BYTES;
  else return fail(CSA2_ERR_INVALID_ARG, "unknown plane %d", plane);
  return CSA2_OK;
}

int csa2_ring_bytes(size_t* bytes) {
  CHECK_PTR(bytes, "bytes");
  *bytes = static_cast<size_t>(CSA2_WINDOW) * CSA2_LATENT_DIM;
  return CSA2_OK;
}

int csa2_workspace_bytes(int op, int B, int n_q, int64_t max_ctx, size_t* bytes) {
  CHECK_PTR(bytes, "bytes");
  if (int st = check_batch(B, n_q)) return st;
  if (max_ctx < 0) return fail(CSA2_ERR_INVALID_ARG, "max_ctx < 0");
  const int64_t Q = static_cast<int64_t>(B) * n_q;
  switch (op) {
    case CSA2_OP_INDEXER_REINDEX: *bytes = reindex_ws(Q); break;
    case CSA2_OP_INDEXER_FULL: *bytes = blockmax_ws(Q, max_ctx) + reindex_ws(Q); break;
    case CSA2_OP_SPARSE_ATTN: *bytes = csa2::attn_workspace_bytes(Q); break;
    case CSA2_OP_DECODE_LAYER: {
      const size_t idx = blockmax_ws(Q, max_ctx) + reindex_ws(Q);
      const size_t att = csa2::attn_workspace_bytes(Q);
      *bytes = idx > att ? idx : att;
      break;
    }
    default: return fail(CSA2_ERR_INVALID_ARG, "unknown op %d", op);
  }
  return CSA2_OK;
}

int csa2_append_kv(const void* latent, const void* idx_key, const int32_t* seq_idx,
                   const int64_t* pos, int T, const int32_t* block_table, int B, int max_pages,
                   int64_t n_pages, uint8_t* main_pages, uint8_t* idx_pages, void* stream) {
  CSA2_NVTX_RANGE();
  if (T < 0) return fail(CSA2_ERR_INVALID_ARG, "T = %d < 0", T);
  if (T == 0) return CSA2_OK;
  CHECK_A16(latent, "latent");
  CHECK_A16(idx_key, "idx_key");
  CHECK_PTR(seq_idx, "seq_idx");
  CHECK_PTR(pos, "pos");
  CHECK_A16(main_pages, "main_pages");
  CHECK_A16(idx_pages, "idx_pages");
  if (B < 1) return fail(CSA2_ERR_INVALID_ARG, "B = %d < 1", B);
  if (int st = check_pages(block_table, max_pages, n_pages)) return st;
  cudaError_t e = csa2::launch_append_kv(latent, idx_key, seq_idx, pos, T, block_table, B, max_pages,
                                         n_pages, main_pages, idx_pages, S(stream));
  return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "append_kv launch");
}

int csa2_decode_appends(const void* latent, const void* idx_key, const int32_t* seq_idx, const int64_t* pos, int T,
                        const int32_t* block_table, int B, int max_pages, int64_t n_pages, uint8_t* main_pages,
                        uint8_t* idx_pages, const csa2_append_layer* layers, int n_layers, void* stream) {
  CSA2_NVTX_RANGE();
  if (T < 0) return fail(CSA2_ERR_INVALID_ARG, "T = %d < 0", T);
  if (n_layers < 0) return fail(CSA2_ERR_INVALID_ARG, "n_layers = %d < 0", n_layers);
  if (n_layers > csa2::kMaxAppendLayers)
    return fail(CSA2_ERR_UNSUPPORTED, "n_layers = %d > %d", n_layers, csa2::kMaxAppendLayers);
  if (n_layers > 0) CHECK_PTR(layers, "layers");
  csa2::DecodeAppends P{};
  P.T = T;
  if (T > 0) {
    CHECK_A16(latent, "latent");
    CHECK_A16(idx_key, "idx_key");
    CHECK_PTR(seq_idx, "seq_idx");
    CHECK_PTR(pos, "pos");
    CHECK_A16(main_pages, "main_pages");
    CHECK_A16(idx_pages, "idx_pages");
    if (B < 1) return fail(CSA2_ERR_INVALID_ARG, "B = %d < 1", B);
    if (int st = check_pages(block_table, max_pages, n_pages)) return st;
  }
  P.latent = latent;
  P.idx_key = idx_key;
  P.seq_idx = seq_idx;
  P.pos = pos;
  P.block_table = block_table;
  P.B = B;
  P.max_pages = max_pages;
  P.n_pages = n_pages;
  P.main_pages = main_pages;
  P.idx_pages = idx_pages;
  P.n_layers = n_layers;
  for (int i = 0; i < n_layers; ++i) {
    const csa2_append_layer& a = layers[i];
    csa2::DecodeAppendsLayer& d = P.layer[i];
    if (a.swa && T > 0) {
      if (!aligned16(a.swa)) return fail(CSA2_ERR_INVALID_ARG, "layer %d: swa is not 16-byte aligned", i);
      if (!a.ring_idx) return fail(CSA2_ERR_INVALID_ARG, "layer %d: ring_idx is NULL", i);
      if (!a.rings || !aligned16(a.rings))
        return fail(CSA2_ERR_INVALID_ARG, "layer %d: rings is NULL or not 16-byte aligned", i);
      if (a.n_rings < 1) return fail(CSA2_ERR_INVALID_ARG, "layer %d: n_rings < 1", i);
      d.swa = a.swa;
      d.ring_idx = a.ring_idx;
      d.n_rings = a.n_rings;
      d.rings = a.rings;
    }
    if (a.q_idx) {
      if (a.q_n < 0 || a.q_n % 16)
        return fail(CSA2_ERR_INVALID_ARG, "layer %d: q_n = %lld is not a multiple of 16", i,
                    static_cast<long long>(a.q_n));
      if (!aligned16(a.q_idx)) return fail(CSA2_ERR_INVALID_ARG, "layer %d: q_idx is not 16-byte aligned", i);
      if (!a.q_codes || (reinterpret_cast<uintptr_t>(a.q_codes) & 7u))
        return fail(CSA2_ERR_INVALID_ARG, "layer %d: q_codes is NULL or not 8-byte aligned", i);
      if (!a.q_scales) return fail(CSA2_ERR_INVALID_ARG, "layer %d: q_scales is NULL", i);
      if (a.q_n > 0) {
        d.q_idx = a.q_idx;
        d.q_n = a.q_n;
        d.q_codes = a.q_codes;
        d.q_scales = a.q_scales;
      }
    }
  }
  cudaError_t e = csa2::launch_decode_appends(P, S(stream));
  return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "decode_appends launch");
}
int csa2_append_swa(const void* x, const int32_t* ring_idx, const int64_t* pos, int T,
                    int64_t n_rings, uint8_t* rings, void* stream) {
  CSA2_NVTX_RANGE();
  if (T < 0) return fail(CSA2_ERR_INVALID_ARG, "T = %d < 0", T);
  if (T == 0) return CSA2_OK;
  CHECK_A16(x, "x");
  CHECK_PTR(ring_idx, "ring_idx");
  CHECK_PTR(pos, "pos");
  CHECK_A16(rings, "rings");
  if (n_rings < 1) return fail(CSA2_ERR_INVALID_ARG, "n_rings < 1");
  cudaError_t e = csa2::launch_append_swa(x, ring_idx, pos, T, n_rings, rings, S(stream));
  return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "append_swa launch");
}

int csa2_compress_append(const void* kv, const void* kv_gate, const void* idx_key, const void* idx_gate,
                         const int32_t* seq_idx, const int64_t* pos, int T, int m, void* tail,
                         const int32_t* block_table, int B, int max_pages, int64_t n_pages,
                         uint8_t* main_pages, uint8_t* idx_pages, void* stream) {
  CSA2_NVTX_RANGE();
  if (T < 0) return fail(CSA2_ERR_INVALID_ARG, "T = %d < 0", T);
  if (int st = check_ratio(m)) return st;
  if (T == 0) return CSA2_OK;
  CHECK_A16(kv, "kv");
  CHECK_A16(kv_gate, "kv_gate");
  CHECK_A16(idx_key, "idx_key");
  CHECK_A16(idx_gate, "idx_gate");
  CHECK_PTR(seq_idx, "seq_idx");
  CHECK_PTR(pos, "pos");
  if (m > 1) CHECK_A16(tail, "tail");
  CHECK_A16(main_pages, "main_pages");
  CHECK_A16(idx_pages, "idx_pages");
  if (B < 1) return fail(CSA2_ERR_INVALID_ARG, "B = %d < 1", B);
  if (int st = check_pages(block_table, max_pages, n_pages)) return st;
  cudaError_t e = csa2::launch_compress_append(kv, kv_gate, idx_key, idx_gate, seq_idx, pos, T, m, tail, block_table,
                                               B, max_pages, n_pages, main_pages, idx_pages, S(stream));
  return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "compress_append launch");
}

int csa2_quant_fp8_entries(const void* x, int T, uint8_t* out, void* stream) {
  CSA2_NVTX_RANGE();
  if (T < 0) return fail(CSA2_ERR_INVALID_ARG, "T = %d < 0", T);
  if (T == 0) return CSA2_OK;
  CHECK_A16(x, "x");
  CHECK_A16(out, "out");
  cudaError_t e = csa2::launch_append_swa(x, nullptr, nullptr, T, 0, out, S(stream));
  return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "quant_fp8_entries launch");
}

int csa2_ring_refill(const uint8_t* entries, const int64_t* seq_len, int B, int n,
                     const int32_t* ring_idx, int64_t n_rings, uint8_t* rings, void* stream) {
  CSA2_NVTX_RANGE();
  if (B < 0 || B > CSA2_MAX_TOKENS) return fail(CSA2_ERR_INVALID_ARG, "B = %d out of range", B);
  if (n < 0) return fail(CSA2_ERR_INVALID_ARG, "n = %d < 0", n);
  if (B == 0 || n == 0) return CSA2_OK;
  CHECK_A16(entries, "entries");
  CHECK_PTR(seq_len, "seq_len");
  CHECK_PTR(ring_idx, "ring_idx");
  CHECK_A16(rings, "rings");
  if (n_rings < 1) return fail(CSA2_ERR_INVALID_ARG, "n_rings < 1");
  cudaError_t e = csa2::launch_ring_refill(entries, seq_len, B, n, ring_idx, n_rings, rings, S(stream));
  return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "ring_refill launch");
}

int csa2_quant_mxfp4(const void* x, int64_t n, uint8_t* codes, uint8_t* scales, void* stream) {
  CSA2_NVTX_RANGE();
  if (n < 0 || n % 16) return fail(CSA2_ERR_INVALID_ARG, "n = %lld is not a multiple of 16", static_cast<long long>(n));
  if (n == 0) return CSA2_OK;
  CHECK_A16(x, "x");
  CHECK_PTR(codes, "codes");
  CHECK_PTR(scales, "scales");
  if (reinterpret_cast<uintptr_t>(codes) & 7u) return fail(CSA2_ERR_INVALID_ARG, "codes is not 8-byte aligned");
  cudaError_t e = csa2::launch_quant_mxfp4(x, n, codes, scales, S(stream));
  return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "quant_mxfp4 launch");
}

int csa2_dequant_mxfp4(const uint8_t* codes, const uint8_t* scales, int64_t n, float* out,
                       void* stream) {
  CSA2_NVTX_RANGE();
  if (n < 0 || n % 16) return fail(CSA2_ERR_INVALID_ARG, "n = %lld is not a multiple of 16", static_cast<long long>(n));
  if (n == 0) return CSA2_OK;
  CHECK_PTR(codes, "codes");
  CHECK_PTR(scales, "scales");
  CHECK_PTR(out, "out");
  if (reinterpret_cast<uintptr_t>(codes) & 7u) return fail(CSA2_ERR_INVALID_ARG, "codes is not 8-byte aligned");
  cudaError_t e = csa2::launch_dequant_mxfp4(codes, scales, n, out, S(stream));
  return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "dequant_mxfp4 launch");
}

int csa2_quant_fp8(const float* x, int64_t n, uint8_t* out, void* stream) {
  CSA2_NVTX_RANGE();
  if (n < 0) return fail(CSA2_ERR_INVALID_ARG, "n < 0");
  if (n == 0) return CSA2_OK;
  CHECK_PTR(x, "x");
  CHECK_PTR(out, "out");
  cudaError_t e = csa2::launch_quant_fp8(x, n, out, S(stream));
  return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "quant_fp8 launch");
}

static int check_indexer_inputs(const uint8_t* q_codes, const uint8_t* q_scales, const float* w,
                                const int64_t* seq_len, const uint8_t* idx_pages) {
  CHECK_A16(q_codes, "q_codes");
  CHECK_PTR(q_scales, "q_scales");
  if (reinterpret_cast<uintptr_t>(q_scales) & 1u) return fail(CSA2_ERR_INVALID_ARG, "q_scales is not 2-byte aligned");
  CHECK_PTR(w, "w");
  CHECK_PTR(seq_len, "seq_len");
  CHECK_A16(idx_pages, "idx_pages");
  return CSA2_OK;
}

int csa2_indexer_scan(const uint8_t* q_codes, const uint8_t* q_scales, const float* w,
                      const int64_t* seq_len, int B, int n_q, int64_t max_ctx,
                      const int32_t* block_table, int max_pages, int64_t n_pages,
                      const uint8_t* idx_pages, float* block_max, int64_t max_blocks, int m,
                      void* stream) {
  CSA2_NVTX_RANGE();
  if (int st = check_batch(B, n_q)) return st;
  if (int st = check_ratio(m)) return st;
  if (B == 0) return CSA2_OK;
  if (int st = check_indexer_inputs(q_codes, q_scales, w, seq_len, idx_pages)) return st;
  if (int st = check_pages(block_table, max_pages, n_pages)) return st;
  CHECK_PTR(block_max, "block_max");
  if (max_ctx < 1) return fail(CSA2_ERR_INVALID_ARG, "max_ctx < 1");
  if (max_blocks < (max_ctx / m + 7) / 8) return fail(CSA2_ERR_INVALID_ARG, "max_blocks < ceil(max_ctx / m / 8)");
  cudaError_t e = csa2::launch_indexer_scan(q_codes, q_scales, w, seq_len, B, n_q, max_ctx, block_table,
                                            max_pages, n_pages, idx_pages, block_max, max_blocks, S(stream), m);
  return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "indexer_scan launch");
}

int csa2_block_topk(const float* block_max, const int64_t* seq_len, int B, int n_q,
                    int64_t max_blocks, int32_t* pool, int m, void* stream) {
  CSA2_NVTX_RANGE();
  if (int st = check_batch(B, n_q)) return st;
  if (int st = check_ratio(m)) return st;
  if (B == 0) return CSA2_OK;
  CHECK_PTR(block_max, "block_max");
  CHECK_PTR(seq_len, "seq_len");
  CHECK_PTR(pool, "pool");
  if (max_blocks < 1) return fail(CSA2_ERR_INVALID_ARG, "max_blocks < 1");
  cudaError_t e = csa2::launch_block_topk(block_max, seq_len, B, n_q, max_blocks, pool, S(stream), m);
  return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "block_topk launch");
}

}  // extern "C"

namespace csa2 {
// Host checks of a Reindex call (shared by csa2_indexer_reindex and
// csa2_indexer_reindex_noalloc, so both accept and reject the same shapes
// with the same status codes). Pointers are checked only when B > 0.
int check_reindex(const uint8_t* q_codes, const uint8_t* q_scales, const float* w, const int64_t* seq_len, int B,
                  int n_q, const int32_t* block_table, int max_pages, int64_t n_pages, const uint8_t* idx_pages,
                  const int32_t* pool, const int32_t* topk, int m) {
  if (int st = check_batch(B, n_q)) return st;
  if (int st = check_ratio(m)) return st;
  if (B == 0) return CSA2_OK;
  if (int st = check_indexer_inputs(q_codes, q_scales, w, seq_len, idx_pages)) return st;
  if (int st = check_pages(block_table, max_pages, n_pages)) return st;
  CHECK_PTR(pool, "pool");
  CHECK_PTR(topk, "topk");
  return CSA2_OK;
}
}  // namespace csa2

extern "C" {

int csa2_indexer_reindex(const uint8_t* q_codes, const uint8_t* q_scales, const float* w,
                         const int64_t* seq_len, int B, int n_q, const int32_t* block_table,
                         int max_pages, int64_t n_pages, const uint8_t* idx_pages,
                         const int32_t* pool, int32_t* topk, void* ws, size_t ws_bytes, int m,
                         void* stream) {
  CSA2_NVTX_RANGE();
  if (int st = csa2::check_reindex(q_codes, q_scales, w, seq_len, B, n_q, block_table, max_pages, n_pages,
                                   idx_pages, pool, topk, m))
    return st;
  if (B == 0) return CSA2_OK;
  const int64_t Q = static_cast<int64_t>(B) * n_q;
  if (!ws || ws_bytes < reindex_ws(Q)) return fail(CSA2_ERR_WORKSPACE, "reindex needs %zu workspace bytes", reindex_ws(Q));
  if (!aligned16(ws)) return fail(CSA2_ERR_INVALID_ARG, "ws is not 16-byte aligned");
  float* scores = static_cast<float*>(ws);
  cudaError_t e = csa2::launch_pool_scores(q_codes, q_scales, w, seq_len, B, n_q, block_table, max_pages,
                                           n_pages, idx_pages, pool, scores, S(stream), m);
  if (e != cudaSuccess) return cuda_fail(e, "pool rescore launch");
  e = csa2::launch_pool_topk(scores, seq_len, B, n_q, pool, topk, S(stream));
  return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "pool top-k launch");
}

int csa2_indexer_full(const uint8_t* q_codes, const uint8_t* q_scales, const float* w,
                      const int64_t* seq_len, int B, int n_q, int64_t max_ctx,
                      const int32_t* block_table, int max_pages, int64_t n_pages,
                      const uint8_t* idx_pages, int32_t* pool, int32_t* topk, void* ws,
                      size_t ws_bytes, int m, void* stream) {
  CSA2_NVTX_RANGE();
  if (int st = check_batch(B, n_q)) return st;
  if (int st = check_ratio(m)) return st;
  if (B == 0) return CSA2_OK;
  if (max_ctx < 1) return fail(CSA2_ERR_INVALID_ARG, "max_ctx < 1");
  const int64_t Q = static_cast<int64_t>(B) * n_q;
  const size_t need = blockmax_ws(Q, max_ctx) + reindex_ws(Q);
  if (!ws || ws_bytes < need) return fail(CSA2_ERR_WORKSPACE, "indexer_full needs %zu workspace bytes", need);
  if (!aligned16(ws)) return fail(CSA2_ERR_INVALID_ARG, "ws is not 16-byte aligned");
  CHECK_PTR(pool, "pool");
  float* bm = static_cast<float*>(ws);
  const int64_t max_blocks = (max_ctx / m + 7) / 8;
  if (int st = csa2_indexer_scan(q_codes, q_scales, w, seq_len, B, n_q, max_ctx, block_table, max_pages,
                                 n_pages, idx_pages, bm, max_blocks, m, stream))
    return st;
  if (int st = csa2_block_topk(bm, seq_len, B, n_q, max_blocks, pool, m, stream)) return st;
  return csa2_indexer_reindex(q_codes, q_scales, w, seq_len, B, n_q, block_table, max_pages, n_pages,
                              idx_pages, pool, topk, static_cast<uint8_t*>(ws) + blockmax_ws(Q, max_ctx),
                              ws_bytes - blockmax_ws(Q, max_ctx), m, stream);
}

static int sparse_attn(const void* q, const int32_t* topk, const int64_t* seq_len, int B, int n_q,
                       const int32_t* block_table, int max_pages, int64_t n_pages,
                       const uint8_t* main_pages, const uint8_t* rings, const int32_t* ring_idx,
                       int64_t n_rings, const uint8_t* swa_chunk, float softmax_scale, int out_dtype,
                       void* out, float* lse, void* ws, size_t ws_bytes, int m, void* stream) {
  if (int st = check_batch(B, n_q, swa_chunk ? CSA2_MAX_PREFILL_NQ : CSA2_MAX_NQ)) return st;
  if (int st = check_ratio(m)) return st;
  if (B == 0) return CSA2_OK;
  if (swa_chunk && !aligned16(swa_chunk)) return fail(CSA2_ERR_INVALID_ARG, "swa_chunk is not 16-byte aligned");
  CHECK_A16(q, "q");
  CHECK_PTR(topk, "topk");
  CHECK_PTR(seq_len, "seq_len");
  if (int st = check_pages(block_table, max_pages, n_pages)) return st;
  CHECK_A16(main_pages, "main_pages");
  CHECK_A16(rings, "rings");
  CHECK_PTR(ring_idx, "ring_idx");
  if (n_rings < 1) return fail(CSA2_ERR_INVALID_ARG, "n_rings < 1");
  CHECK_PTR(out, "out");
  const int base_dtype = out_dtype & ~CSA2_OUT_DEROTATE;
  if (base_dtype != CSA2_OUT_F32 && base_dtype != CSA2_OUT_BF16)
    return fail(CSA2_ERR_INVALID_ARG, "unknown out_dtype %d", out_dtype);
  if (!(softmax_scale > 0.f) || softmax_scale > 1e30f) return fail(CSA2_ERR_INVALID_ARG, "softmax_scale must be positive and finite");
  const int64_t Q = static_cast<int64_t>(B) * n_q;
  const size_t need = csa2::attn_workspace_bytes(Q);
  if (need > 0) {
    if (!ws || ws_bytes < need) return fail(CSA2_ERR_WORKSPACE, "sparse_attn needs %zu workspace bytes", need);
    if (!aligned16(ws)) return fail(CSA2_ERR_INVALID_ARG, "ws is not 16-byte aligned");
  }
  cudaError_t e = csa2::launch_sparse_attn(q, topk, seq_len, B, n_q, block_table, max_pages, n_pages,
                                           main_pages, rings, ring_idx, n_rings, swa_chunk, softmax_scale,
                                           out_dtype, out, lse, ws, S(stream), m);
  return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "sparse_attn launch");
}

int csa2_sparse_attn(const void* q, const int32_t* topk, const int64_t* seq_len, int B, int n_q,
                     const int32_t* block_table, int max_pages, int64_t n_pages,
                     const uint8_t* main_pages, const uint8_t* rings, const int32_t* ring_idx,
                     int64_t n_rings, float softmax_scale, int out_dtype, void* out, float* lse,
                     void* ws, size_t ws_bytes, int m, void* stream) {
  CSA2_NVTX_RANGE();
  return sparse_attn(q, topk, seq_len, B, n_q, block_table, max_pages, n_pages, main_pages, rings, ring_idx,
                     n_rings, nullptr, softmax_scale, out_dtype, out, lse, ws, ws_bytes, m, stream);
}

int csa2_sparse_attn_prefill(const void* q, const int32_t* topk, const int64_t* seq_len, int B,
                             int n_q, const int32_t* block_table, int max_pages, int64_t n_pages,
                             const uint8_t* main_pages, const uint8_t* rings,
                             const int32_t* ring_idx, int64_t n_rings, const uint8_t* swa_chunk,
                             float softmax_scale, int out_dtype, void* out, float* lse, void* ws,
                             size_t ws_bytes, int m, void* stream) {
  CSA2_NVTX_RANGE();
  CHECK_A16(swa_chunk, "swa_chunk");
  return sparse_attn(q, topk, seq_len, B, n_q, block_table, max_pages, n_pages, main_pages, rings, ring_idx,
                     n_rings, swa_chunk, softmax_scale, out_dtype, out, lse, ws, ws_bytes, m, stream);
}

static int run_layer(const csa2_layer_args* a, int32_t* pool, int32_t* topk, void* stream) {
  const int m = a->tokens_per_entry == 0 ? 1 : a->tokens_per_entry;
  switch (a->mode) {
    case CSA2_MODE_FULL:
      CHECK_PTR(pool, "pool (FULL)");
      CHECK_PTR(topk, "topk (FULL)");
      if (int st = csa2_indexer_full(a->q_idx_codes, a->q_idx_scales, a->w, a->seq_len, a->B, a->n_q,
                                     a->max_ctx, a->block_table, a->max_pages, a->n_pages, a->idx_pages,
                                     pool, topk, a->ws, a->ws_bytes, m, stream))
        return st;
      break;
    case CSA2_MODE_REINDEX:
      if (!pool) return fail(CSA2_ERR_INVALID_ARG, "REINDEX layer without a pool (none given, no earlier FULL layer)");
      CHECK_PTR(topk, "topk (REINDEX)");
      if (int st = csa2_indexer_reindex(a->q_idx_codes, a->q_idx_scales, a->w, a->seq_len, a->B, a->n_q,
                                        a->block_table, a->max_pages, a->n_pages, a->idx_pages, pool, topk,
                                        a->ws, a->ws_bytes, m, stream))
        return st;
      break;
    case CSA2_MODE_REUSE:
      if (!topk) return fail(CSA2_ERR_INVALID_ARG, "REUSE layer without a top-k (none given, no earlier indexer layer)");
      break;
    default:
      return fail(CSA2_ERR_INVALID_ARG, "unknown mode %d", a->mode);
  }
  return sparse_attn(a->q, topk, a->seq_len, a->B, a->n_q, a->block_table, a->max_pages, a->n_pages,
                     a->main_pages, a->rings, a->ring_idx, a->n_rings, a->swa_chunk, a->softmax_scale,
                     a->out_dtype, a->out, a->lse, a->ws, a->ws_bytes, m, stream);
}

int csa2_decode_layer(const csa2_layer_args* layer, void* stream) {
  CSA2_NVTX_RANGE();
  CHECK_PTR(layer, "layer");
  return run_layer(layer, layer->pool, layer->topk, stream);
}

int csa2_decode_group(const csa2_layer_args* layers, int n_layers, void* stream) {
  CSA2_NVTX_RANGE();
  CHECK_PTR(layers, "layers");
  if (n_layers < 1) return fail(CSA2_ERR_INVALID_ARG, "n_layers < 1");
  int32_t* latest_pool = nullptr;
  int32_t* latest_topk = nullptr;
  for (int i = 0; i < n_layers; ++i) {
    const csa2_layer_args* a = &layers[i];
    int32_t* pool = a->pool;
    int32_t* topk = a->topk;
    if (a->mode == CSA2_MODE_REINDEX && !pool) pool = latest_pool;
    if (a->mode == CSA2_MODE_REUSE && !topk) topk = latest_topk;
    if (int st = run_layer(a, pool, topk, stream)) {
      char tmp[512];
      snprintf(tmp, sizeof(tmp), "layer %d: %s", i, g_err);
      return fail(st, "%s", tmp);
    }
    if (a->mode == CSA2_MODE_FULL) latest_pool = pool;
    if (a->mode != CSA2_MODE_REUSE) latest_topk = topk;
  }
  return CSA2_OK;
}

int csa2_debug_force_wait_timeout(int site, void* stream) {
  if (site < 0) return fail(CSA2_ERR_INVALID_ARG, "site = %d < 0", site);
  cudaError_t (*setters[4])(int, cudaStream_t) = {csa2::force_timeout_append, csa2::force_timeout_indexer,
                                                   csa2::force_timeout_topk, csa2::force_timeout_attn};
  for (auto set : setters) {
    const cudaError_t e = set(site, S(stream));
    if (e != cudaSuccess) return cuda_fail(e, "setting the forced-timeout site");
  }
  return CSA2_OK;
}

int csa2_check_device_status(void* stream, int* status) {
  CHECK_PTR(status, "status");
  int worst = CSA2_OK;
  const char* which = "";
  int where_worst = 0;
  cudaError_t (*readers[4])(cudaStream_t, int*, int*, bool) = {csa2::status_append, csa2::status_indexer,
                                                               csa2::status_topk, csa2::status_attn};
  const char* names[4] = {"append", "indexer", "topk", "attention"};
  for (int i = 0; i < 4; ++i) {
    int code = 0, where = 0;
    cudaError_t e = readers[i](S(stream), &code, &where, true);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device status");
    if (code != CSA2_OK && worst == CSA2_OK) {
      worst = code;
      which = names[i];
      where_worst = where;
    }
  }
  *status = worst;
  if (worst != CSA2_OK) fail(worst, "device status from %s kernels (site %d): %s", which, where_worst, csa2_status_string(worst));
  return CSA2_OK;
}

}  // extern "C"
