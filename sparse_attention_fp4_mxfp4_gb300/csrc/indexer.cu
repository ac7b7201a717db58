// Hierarchical sparse indexer on the tensor cores ("DeepSeek V4.1: model
// architecture and system design, a close reading" section 2.2;
// "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" section
// 3.4): s(p) = sum_h w_h * max(0, qhat_h . khat_p) over 32 heads x 128 dims.
//
// One kernel serves both uses:
//   * Full scan: a tile is one 128-entry page of the indexer plane; the
//     epilogue reduces scores to the maximum over 8-position blocks. All n_q
//     query tokens of a sequence share the tile: N = 32 * n_q MMA columns.
//   * Pool rescore (Reindex, and the end of Full): a tile is 16 pool blocks of
//     8 positions, gathered block by block; the epilogue writes every score.
//
// Per CTA: warp 4 streams tiles into a ring of shared-memory stages with bulk
// copies; warps 0-3 dequantise a stage to an f16 128 x 128 operand (exact:
// E2M1 x E4M3 fits f16) in the 128-byte-swizzled K-major layout and run the
// epilogue of the previous tile; warp 5 issues tcgen05.mma (M = 128
// positions, N = 32 * n_q, K = 128) into a double-buffered TMEM accumulator.
#include <algorithm>

#include "formats.cuh"
#include "kernels.h"
#include "sm103.cuh"

namespace csa2 {
namespace {

constexpr int kStages = 4;
constexpr int kTileBytes = 16 * 576;     // one indexer page / 16 pool blocks
constexpr int kABytes = 128 * 128 * 2;   // f16 operand tile
constexpr int kThreads = 192;
constexpr int kIdxPageBytes = 16 * 576;

struct ScanParams {
  const uint8_t* q_codes;
  const uint8_t* q_scales;
  const float* w;
  const int64_t* seq_len;
  int B, n_q;
  const int32_t* block_table;
  int max_pages;
  int64_t n_pages;
  const uint8_t* idx_pages;
  // Full scan
  float* block_max;
  int64_t max_blocks;
  // Pool rescore
  const int32_t* pool;
  float* scores;
  int tiles_per_cta;
};

__host__ __device__ constexpr uint32_t tmem_cols_for(int n_cols) {
  uint32_t c = 32;
  while (c < static_cast<uint32_t>(2 * n_cols)) c <<= 1;
  return c;
}

__host__ __device__ constexpr int smem_bytes_for(int n_q) {
  return 1024 /*align*/ + 2 * kABytes + 32 * n_q * 256 /*q operand*/ + kStages * kTileBytes +
         2048 /*barriers, flags, head weights*/;
}

// Dequantises one staged tile (16 groups of 8 entries in the indexer-page
// layout) into the swizzled f16 operand; thread t handles row t.
__device__ __forceinline__ void dequant_tile(const uint8_t* stage, uint8_t* a, int t) {
  const uint8_t* grp = stage + (t >> 3) * 576;
  const int row = t & 7;
  const uint2 sc = *reinterpret_cast<const uint2*>(grp + 512 + row * 8);
  const uint64_t sc8 = (static_cast<uint64_t>(sc.y) << 32) | sc.x;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 codes = *reinterpret_cast<const uint4*>(grp + c * 128 + row * 16);
    uint4 out[4];
    dequant32_f16(codes, static_cast<uint16_t>((sc8 >> (16 * c)) & 0xFFFFu), out);
    uint8_t* kb = a + (c >> 1) * 16384;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<uint4*>(kb + sw128_offset(t, (c & 1) * 4 + j)) = out[j];
  }
}

template <bool kPool>
__global__ void __launch_bounds__(kThreads, 1) indexer_kernel(const ScanParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int n_q = kPool ? 1 : P.n_q;
  const int n_cols = 32 * n_q;
  uint8_t* abuf = smem;                                  // 2 x 32 KB
  uint8_t* qbuf = smem + 2 * kABytes;                    // n_cols x 256 B
  uint8_t* stages = qbuf + n_cols * 256;                 // kStages x 9216 B
  uint8_t* misc = stages + kStages * kTileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc);    // 16 barriers
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 128);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 132);
  uint32_t* stage_mask = reinterpret_cast<uint32_t*>(misc + 136);  // kStages words
  float* wsm = reinterpret_cast<float*>(misc + 256);                 // n_cols floats

  const uint32_t full0 = smem_u32(&bars[0]), empty0 = smem_u32(&bars[4]);
  const uint32_t afull0 = smem_u32(&bars[8]), aempty0 = smem_u32(&bars[10]);
  const uint32_t dfull0 = smem_u32(&bars[12]), dempty0 = smem_u32(&bars[14]);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Work of this CTA.
  int b, jq = 0;  // sequence, query token (pool mode)
  int64_t first_tile, n_tiles, tile_stride;
  if (kPool) {
    const int q = blockIdx.y;
    b = q / P.n_q;
    jq = q % P.n_q;
    first_tile = static_cast<int64_t>(blockIdx.x) * P.tiles_per_cta;
    n_tiles = 128 - first_tile < P.tiles_per_cta ? 128 - first_tile : P.tiles_per_cta;
    if (n_tiles < 0) n_tiles = 0;
    tile_stride = 1;
  } else {
    b = blockIdx.y;
    const int64_t pages = (P.seq_len[b] + 127) >> 7;
    first_tile = blockIdx.x;
    tile_stride = gridDim.x;
    n_tiles = pages > first_tile ? (pages - first_tile + tile_stride - 1) / tile_stride : 0;
  }
  const int64_t seq_n = P.seq_len[b];
  if (!kPool && (seq_n + 7) / 8 > P.max_blocks) {
    if (threadIdx.x == 0) report(CSA2_ERR_DEVICE_BOUNDS, 204);
    n_tiles = 0;
  }

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, 128);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(afull0 + 8 * i, 128);
      mbar_init(aempty0 + 8 * i, 1);
      mbar_init(dfull0 + 8 * i, 1);
      mbar_init(dempty0 + 8 * i, 128);
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  const uint32_t ncols = tmem_cols_for(n_cols);
  if (warp == 5) tmem_alloc(smem_u32(tmem_slot), ncols);

  // Query operand: qhat of the CTA's query tokens, f16 [n_cols rows x 128].
  if (tid < 128) {
    for (int task = tid; task < n_cols * 4; task += 128) {
      const int n = task >> 2, c = task & 3;
      const int jj = kPool ? jq : n >> 5, h = n & 31;
      const int64_t qrow = (static_cast<int64_t>(b) * P.n_q + jj) * 32 + h;
      const uint4 codes = *reinterpret_cast<const uint4*>(P.q_codes + qrow * 64 + c * 16);
      const uint16_t s2 = *reinterpret_cast<const uint16_t*>(P.q_scales + qrow * 8 + 2 * c);
      uint4 out[4];
      dequant32_f16(codes, s2, out);
      uint8_t* kb = qbuf + (c >> 1) * (n_cols * 128);
#pragma unroll
      for (int j = 0; j < 4; ++j) *reinterpret_cast<uint4*>(kb + sw128_offset(n, (c & 1) * 4 + j)) = out[j];
    }
    for (int i = tid; i < n_cols; i += 128) {
      const int jj = kPool ? jq : i >> 5;
      wsm[i] = P.w[(static_cast<int64_t>(b) * P.n_q + jj) * 32 + (i & 31)];
    }
    fence_proxy_async();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ---- producer ----
    if (lane == 0) {
      for (int64_t i = 0; i < n_tiles; ++i) {
        const int s = static_cast<int>(i % kStages);
        const int64_t u = i / kStages;
        if (u > 0 && !mbar_wait(empty0 + 8 * s, (u - 1) & 1, 201, abort_flag)) { *abort_flag = 1; break; }
        if (*abort_flag) break;
        const int64_t tile = first_tile + i * tile_stride;
        const uint32_t dst = smem_u32(stages + s * kTileBytes);
        if (!kPool) {
          const int32_t page = (tile < P.max_pages)
                                   ? P.block_table[static_cast<int64_t>(b) * P.max_pages + tile]
                                   : -1;
          if (page < 0 || page >= P.n_pages) {
            report(CSA2_ERR_DEVICE_BOUNDS, 202);
            stage_mask[s] = 0;
            mbar_arrive(full0 + 8 * s);
            continue;
          }
          stage_mask[s] = 0xFFFFu;
          mbar_arrive_expect_tx(full0 + 8 * s, kTileBytes);
          bulk_g2s(dst, P.idx_pages + static_cast<int64_t>(page) * kIdxPageBytes, kTileBytes, full0 + 8 * s);
        } else {
          const int64_t t_q = seq_n - P.n_q + jq;
          const int32_t* prow = P.pool + (static_cast<int64_t>(b) * P.n_q + jq) * 2048 + tile * 16;
          uint32_t mask = 0, nvalid = 0;
          int32_t pages[16];
          for (int g = 0; g < 16; ++g) {
            const int32_t blk = prow[g];
            pages[g] = -1;
            if (blk < 0 || static_cast<int64_t>(blk) * 8 > t_q) continue;
            const int64_t lp = static_cast<int64_t>(blk) >> 4;
            const int32_t page = lp < P.max_pages ? P.block_table[static_cast<int64_t>(b) * P.max_pages + lp] : -1;
            if (page < 0 || page >= P.n_pages) {
              report(CSA2_ERR_DEVICE_BOUNDS, 203);
              continue;
            }
            pages[g] = page;
            mask |= 1u << g;
            ++nvalid;
          }
          stage_mask[s] = mask;
          if (nvalid == 0) {
            mbar_arrive(full0 + 8 * s);
            continue;
          }
          mbar_arrive_expect_tx(full0 + 8 * s, nvalid * 576);
          for (int g = 0; g < 16; ++g) {
            if (pages[g] < 0) continue;
            const int32_t blk = prow[g];
            bulk_g2s(dst + g * 576,
                     P.idx_pages + static_cast<int64_t>(pages[g]) * kIdxPageBytes + (blk & 15) * 576,
                     576, full0 + 8 * s);
          }
        }
      }
    }
  } else if (warp == 5) {
    // ---- MMA issuer ----
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(128, n_cols, false, false);
      int64_t issued = 0;
      for (int64_t i = 0; i < n_tiles; ++i) {
        const int a = static_cast<int>(i & 1);
        const int64_t ua = i >> 1;
        if (!mbar_wait(afull0 + 8 * a, ua & 1, 211, abort_flag)) { *abort_flag = 1; break; }
        if (ua > 0 && !mbar_wait(dempty0 + 8 * a, (ua - 1) & 1, 212, abort_flag)) { *abort_flag = 1; break; }
        if (*abort_flag) break;
        tc_fence_after();
        const uint32_t a_base = smem_u32(abuf + a * kABytes);
        const uint32_t b_base = smem_u32(qbuf);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t ad = sdesc(a_base + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024, kSwizzle128B);
          const uint64_t bd = sdesc(b_base + (k >> 2) * (n_cols * 128) + (k & 3) * 32, 16, 1024, kSwizzle128B);
          umma_f16(tmem + a * n_cols, ad, bd, idesc, k > 0 ? 1u : 0u);
        }
        umma_commit(aempty0 + 8 * a);
        umma_commit(dfull0 + 8 * a);
        issued = i + 1;
      }
      // Before TMEM is released, the last MMAs must have finished (they have on
      // the normal path: the epilogue waited for them).
      if (issued > 0) mbar_wait(dfull0 + 8 * ((issued - 1) & 1), ((issued - 1) >> 1) & 1, 213);
    }
  } else {
    // ---- dequant + epilogue (warps 0-3, thread t <-> row t) ----
    uint32_t valid_rows[2] = {0, 0};  // bit set per 8-row group of the tile in flight
    auto epilogue = [&](int64_t i) -> bool {
      const int a = static_cast<int>(i & 1);
      const int64_t ua = i >> 1;
      if (!mbar_wait(dfull0 + 8 * a, ua & 1, 221, abort_flag)) return false;
      tc_fence_after();
      const int64_t tile = first_tile + i * tile_stride;
      const bool row_ok = (valid_rows[a] >> (tid >> 3)) & 1u;
      for (int jj = 0; jj < n_q; ++jj) {
        uint32_t r[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + a * n_cols + jj * 32, r);
        tmem_wait_ld();
        if (jj == n_q - 1) {
          tc_fence_before();
          mbar_arrive(dempty0 + 8 * a);
        }
        float s = 0.f;
#pragma unroll
        for (int h = 0; h < 32; ++h) s = fmaf(wsm[jj * 32 + h], fmaxf(__uint_as_float(r[h]), 0.f), s);
        if (!kPool) {
          const int64_t t_q = seq_n - P.n_q + jj;
          const int64_t p = tile * 128 + tid;
          float m = (row_ok && p <= t_q) ? s : -INFINITY;
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
          if ((tid & 7) == 0 && row_ok && p <= t_q)
            P.block_max[(static_cast<int64_t>(b) * P.n_q + jj) * P.max_blocks + (p >> 3)] = m;
        } else {
          const int64_t t_q = seq_n - P.n_q + jq;
          const int32_t blk = P.pool[(static_cast<int64_t>(b) * P.n_q + jq) * 2048 + tile * 16 + (tid >> 3)];
          const int64_t p = static_cast<int64_t>(blk) * 8 + (tid & 7);
          const float v = (row_ok && p <= t_q) ? s : -INFINITY;
          P.scores[(static_cast<int64_t>(b) * P.n_q + jq) * 16384 + tile * 128 + tid] = v;
        }
      }
      return true;
    };
    bool ok = true;
    for (int64_t i = 0; i < n_tiles && ok; ++i) {
      const int s = static_cast<int>(i % kStages);
      const int64_t u = i / kStages;
      const int a = static_cast<int>(i & 1);
      const int64_t ua = i >> 1;
      if (!mbar_wait(full0 + 8 * s, u & 1, 231, abort_flag)) { ok = false; break; }
      if (ua > 0 && !mbar_wait(aempty0 + 8 * a, (ua - 1) & 1, 232, abort_flag)) { ok = false; break; }
      const uint32_t mask = stage_mask[s];
      valid_rows[a] = mask;
      if ((mask >> (tid >> 3)) & 1u) dequant_tile(stages + s * kTileBytes, abuf + a * kABytes, tid);
      fence_proxy_async();
      mbar_arrive(empty0 + 8 * s);
      mbar_arrive(afull0 + 8 * a);
      if (i > 0) ok = epilogue(i - 1);
    }
    if (ok && n_tiles > 0) ok = epilogue(n_tiles - 1);
    if (!ok) *abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

template <bool kPool>
cudaError_t launch(const ScanParams& p, dim3 grid, int n_q, cudaStream_t stream) {
  const int smem = smem_bytes_for(kPool ? 1 : n_q);
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(indexer_kernel<kPool>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem_bytes_for(8));
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev] = true;
  }
  indexer_kernel<kPool><<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

int num_sms() {
  static int sms[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64) return 148;
  if (!sms[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    sms[dev] = v > 0 ? v : 148;
  }
  return sms[dev];
}

}  // namespace

cudaError_t status_indexer(cudaStream_t stream, int* code, int* where, bool clear) {
  int h[2] = {0, 0};
  cudaError_t e = cudaMemcpyFromSymbolAsync(h, g_status, sizeof(h), 0, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess && clear) {
    const int z[2] = {0, 0};
    e = cudaMemcpyToSymbolAsync(g_status, z, sizeof(z), 0, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  }
  *code = h[0];
  *where = h[1];
  return e;
}

cudaError_t launch_indexer_scan(const uint8_t* q_codes, const uint8_t* q_scales, const float* w,
                                const int64_t* seq_len, int B, int n_q, int64_t max_ctx,
                                const int32_t* block_table, int max_pages, int64_t n_pages,
                                const uint8_t* idx_pages, float* block_max, int64_t max_blocks,
                                cudaStream_t stream) {
  if (B == 0 || max_ctx <= 0) return cudaSuccess;
  ScanParams p{};
  p.q_codes = q_codes;
  p.q_scales = q_scales;
  p.w = w;
  p.seq_len = seq_len;
  p.B = B;
  p.n_q = n_q;
  p.block_table = block_table;
  p.max_pages = max_pages;
  p.n_pages = n_pages;
  p.idx_pages = idx_pages;
  p.block_max = block_max;
  p.max_blocks = max_blocks;
  const int64_t pages = (max_ctx + 127) / 128;
  const int64_t target = 2LL * num_sms();
  const int64_t per_seq = std::max<int64_t>(1, std::min<int64_t>(pages, (target + B - 1) / B));
  return launch<false>(p, dim3(static_cast<unsigned>(per_seq), B), n_q, stream);
}

cudaError_t launch_pool_scores(const uint8_t* q_codes, const uint8_t* q_scales, const float* w,
                               const int64_t* seq_len, int B, int n_q,
                               const int32_t* block_table, int max_pages, int64_t n_pages,
                               const uint8_t* idx_pages, const int32_t* pool, float* scores,
                               cudaStream_t stream) {
  const int64_t Q = static_cast<int64_t>(B) * n_q;
  if (Q == 0) return cudaSuccess;
  ScanParams p{};
  p.q_codes = q_codes;
  p.q_scales = q_scales;
  p.w = w;
  p.seq_len = seq_len;
  p.B = B;
  p.n_q = n_q;
  p.block_table = block_table;
  p.max_pages = max_pages;
  p.n_pages = n_pages;
  p.idx_pages = idx_pages;
  p.pool = pool;
  p.scores = scores;
  const int64_t target = 2LL * num_sms();
  int splits = static_cast<int>(std::min<int64_t>(128, std::max<int64_t>(1, (target + Q - 1) / Q)));
  const int per = (128 + splits - 1) / splits;
  splits = (128 + per - 1) / per;
  p.tiles_per_cta = per;
  return launch<true>(p, dim3(splits, static_cast<unsigned>(Q)), 1, stream);
}

}  // namespace csa2
