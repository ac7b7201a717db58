// Top-k selections of the hierarchical sparse indexer ("DeepSeek V4.1: model
// architecture and system design, a close reading" section 2.2;
// "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" section
// 3.4): the 2048 best 8-position blocks by block maximum form the candidate
// pool; the 512 best pool positions form the top-k.
//
// Exact radix select on the
// order-preserving integer image of the fp32 scores (digits of 11, 11 and 10
// bits), then an ordered compaction: everything above the threshold, plus the
// lowest-index elements equal to it until k are taken. The output is in
// ascending index order and padded with -1. Invalid elements (masked slots,
// -inf, NaN) are never selected. The cluster kernel below keeps the row in
// shared memory; the single-CTA global-memory kernel serves rows too long for
// a 16-CTA cluster.
#include "kernels.h"
#include "sm103.cuh"

namespace csa2 {
namespace {

constexpr int kThreads = 1024;

__device__ __forceinline__ uint32_t ordered_key(float f) {
  if (!(f > -INFINITY)) return 0u;  // -inf and NaN: invalid
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive prefix sum over 1024 threads; returns the total in *total.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* warp_sums, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t s = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;  // inclusive
  }
  __syncthreads();
  const uint32_t base = warp > 0 ? warp_sums[warp - 1] : 0u;
  const uint32_t tot = warp_sums[31];
  __syncthreads();
  *total = tot;
  return base + x - v;
}

// Adds 1 to hist[bin] for every lane with take == true; lanes of a warp that
// hit the same bin are combined first (scores cluster in a few bins of the
// first digit, so per-element shared atomics would serialise).
__device__ __forceinline__ void warp_hist_add(uint32_t* hist, bool take, uint32_t bin) {
  const uint32_t key = take ? bin : 0xFFFFFFFFu;
  const uint32_t peers = __match_any_sync(0xffffffffu, key);
  if (take && (threadIdx.x & 31) == static_cast<uint32_t>(__ffs(peers) - 1)) atomicAdd(&hist[bin], __popc(peers));
}

// Row of n keys, pick k. `map` turns an element index into the output value.
// mode 0: block top-k (value = block id); mode 1: pool top-k (value = position
// pool[i / 8] * 8 + i % 8).
template <int kMode>
__global__ void __launch_bounds__(kThreads) radix_topk_kernel(const float* __restrict__ keys,
                                                              int64_t row_stride,
                                                              const int64_t* __restrict__ seq_len,
                                                              int n_q, int k,
                                                              const int32_t* __restrict__ pool,
                                                              int32_t* __restrict__ out) {
  __shared__ uint32_t hist[2048];
  __shared__ uint32_t warp_sums[32];
  __shared__ uint32_t s_sel[2];

  const int q = blockIdx.x;
  const int b = q / n_q, j = q % n_q;
  const int tid = threadIdx.x;
  const float* row = keys + static_cast<int64_t>(q) * row_stride;
  int32_t* orow = out + static_cast<int64_t>(q) * k;
  int64_t n;
  if (kMode == 0) {
    const int64_t t = seq_len[b] - n_q + j;
    n = t >= 0 ? (t + 8) / 8 : 0;
    if (n > row_stride) {
      if (tid == 0) report(CSA2_ERR_DEVICE_BOUNDS, 301);
      n = row_stride;
    }
  } else {
    n = row_stride;
  }
  const int32_t* prow = pool + static_cast<int64_t>(q) * 2048;

  // Radix passes. prefix/mask describe the bits fixed so far; `remaining`
  // counts how many elements still have to be taken among those matching.
  uint32_t prefix = 0, mask = 0, remaining = static_cast<uint32_t>(k);
  uint32_t valid = 0;
  const int shifts[3] = {21, 10, 0};
  const int widths[3] = {11, 11, 10};
  bool all_valid = false;
  for (int pass = 0; pass < 3; ++pass) {
    const int sh = shifts[pass];
    const uint32_t nb = 1u << widths[pass];
    for (uint32_t i = tid; i < 2048; i += kThreads) hist[i] = 0;
    __syncthreads();
    const int64_t n_round = (n + kThreads - 1) / kThreads * kThreads;  // whole warps iterate together
    for (int64_t i = tid; i < n_round; i += kThreads) {
      const uint32_t u = i < n ? ordered_key(row[i]) : 0u;
      warp_hist_add(hist, u != 0u && (u & mask) == prefix, (u >> sh) & (nb - 1));
    }
    __syncthreads();
    // Counts from the top: thread t owns bins [2t, 2t+1] in descending order.
    const uint32_t hi_bin = nb - 1 - 2 * tid, lo_bin = hi_bin - 1;
    uint32_t c_hi = 0, c_lo = 0;
    if (2 * static_cast<uint32_t>(tid) < nb) {
      c_hi = hist[hi_bin];
      c_lo = hist[lo_bin];
    }
    uint32_t total;
    const uint32_t before = block_excl_scan(c_hi + c_lo, warp_sums, &total);
    if (pass == 0) {
      valid = total;
      if (valid <= static_cast<uint32_t>(k)) {
        all_valid = true;
        break;
      }
    }
    if (2 * static_cast<uint32_t>(tid) < nb) {
      if (before < remaining && before + c_hi >= remaining) {
        s_sel[0] = hi_bin;
        s_sel[1] = before;
      } else if (before + c_hi < remaining && before + c_hi + c_lo >= remaining) {
        s_sel[0] = lo_bin;
        s_sel[1] = before + c_hi;
      }
    }
    __syncthreads();
    const uint32_t bin = s_sel[0];
    remaining -= s_sel[1];
    prefix |= bin << sh;
    mask |= (nb - 1) << sh;
    __syncthreads();
  }

  // Threshold T: take u > T, and the first `need_eq` elements with u == T.
  const uint32_t T = all_valid ? 0u : prefix;
  const uint32_t need_eq = all_valid ? 0u : remaining;
  const int64_t seg = (n + kThreads - 1) / kThreads;
  const int64_t lo = static_cast<int64_t>(tid) * seg, hi = lo + seg < n ? lo + seg : n;
  uint32_t gt = 0, eq = 0;
  for (int64_t i = lo; i < hi; ++i) {
    const uint32_t u = ordered_key(row[i]);
    if (u > T) ++gt;
    else if (u == T && u != 0u) ++eq;
  }
  uint32_t tot_eq;
  const uint32_t eq_base = block_excl_scan(eq, warp_sums, &tot_eq);
  const uint32_t take_eq = need_eq > eq_base ? min(eq, need_eq - eq_base) : 0u;
  uint32_t tot_sel;
  uint32_t o = block_excl_scan(gt + take_eq, warp_sums, &tot_sel);
  uint32_t taken_eq = 0;
  for (int64_t i = lo; i < hi; ++i) {
    const uint32_t u = ordered_key(row[i]);
    bool sel = u > T;
    if (!sel && u == T && u != 0u && taken_eq < take_eq) {
      sel = true;
      ++taken_eq;
    }
    if (sel) {
      int32_t v;
      if (kMode == 0) {
        v = static_cast<int32_t>(i);
      } else {
        v = prow[i >> 3] * 8 + static_cast<int32_t>(i & 7);
      }
      if (o < static_cast<uint32_t>(k)) orow[o] = v;  // never past the row, whatever the counts say
      ++o;
    }
  }
  for (int i = static_cast<int>(tot_sel) + tid; i < k; i += kThreads) orow[i] = -1;
}

// ---- cluster version: the row lives in shared memory ------------------------
//
// A cluster of C CTAs (C <= 16) selects from one row; CTA r keeps elements
// [r * chunk, (r + 1) * chunk) of the row in its shared memory as ordered keys,
// so the row is read from global memory once. Each radix pass builds a local
// histogram; every CTA then sums all C histograms through distributed shared
// memory and derives the same threshold digit. The ordered compaction uses
// the per-CTA counts exchanged the same way. Control flow is uniform across
// the cluster: every CTA executes every cluster barrier.
constexpr int kChunk = 16384;  // elements per CTA

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t dsmem_ld(const uint32_t* local, uint32_t rank) {
  uint32_t ra, v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(ra) : "memory");
  return v;
}

template <int kMode>
__global__ void __launch_bounds__(kThreads) cluster_topk_kernel(const float* __restrict__ keys,
                                                                int64_t row_stride,
                                                                const int64_t* __restrict__ seq_len,
                                                                int n_q, int k, int C,
                                                                const int32_t* __restrict__ pool,
                                                                int32_t* __restrict__ out) {
  extern __shared__ uint32_t sm[];
  uint32_t* key = sm;                    // [kChunk] ordered keys of this CTA's slice
  uint32_t* hist = sm + kChunk;          // [2048] local histogram
  uint32_t* tot = hist + 2048;           // [2048] cluster-wide histogram
  uint32_t* warp_sums = tot + 2048;      // [32]
  uint32_t* xchg = warp_sums + 32;       // [4]: gt, eq of this CTA
  uint32_t* s_sel = xchg + 4;            // [2]

  const uint32_t r = cluster_rank();
  const int q = blockIdx.y;
  const int b = q / n_q, j = q % n_q;
  const int tid = threadIdx.x;
  int64_t n;
  if (kMode == 0) {
    const int64_t t = seq_len[b] - n_q + j;
    n = t >= 0 ? (t + 8) / 8 : 0;
    if (n > row_stride || n > static_cast<int64_t>(C) * kChunk) {
      if (tid == 0 && r == 0) report(CSA2_ERR_DEVICE_BOUNDS, 311);
      n = min(row_stride, static_cast<int64_t>(C) * kChunk);
    }
  } else {
    n = row_stride;
  }
  const int64_t chunk = (n + C - 1) / C;
  const int64_t lo = static_cast<int64_t>(r) * chunk;
  const int64_t hi = min(n, lo + chunk);
  const int m = hi > lo ? static_cast<int>(hi - lo) : 0;
  const float* row = keys + static_cast<int64_t>(q) * row_stride + lo;
#pragma unroll 4
  for (int i = tid; i < m; i += kThreads) key[i] = ordered_key(row[i]);
  __syncthreads();

  uint32_t prefix = 0, mask = 0, remaining = static_cast<uint32_t>(k);
  bool all_valid = false;
  const int shifts[3] = {21, 10, 0};
  const int widths[3] = {11, 11, 10};
  for (int pass = 0; pass < 3; ++pass) {
    const int sh = shifts[pass];
    const uint32_t nb = 1u << widths[pass];
    for (int i = tid; i < 2048; i += kThreads) hist[i] = 0;
    __syncthreads();
    const int m_round = (m + kThreads - 1) / kThreads * kThreads;  // whole warps iterate together
    for (int i = tid; i < m_round; i += kThreads) {
      const uint32_t u = i < m ? key[i] : 0u;
      warp_hist_add(hist, u != 0u && (u & mask) == prefix, (u >> sh) & (nb - 1));
    }
    cluster_sync_all();  // every local histogram is complete
    for (int i = tid; i < 2048; i += kThreads) {
      uint32_t s = 0;
      for (int c = 0; c < C; ++c) s += dsmem_ld(&hist[i], c);
      tot[i] = s;
    }
    cluster_sync_all();  // nobody reads a remote histogram any more
    const uint32_t hi_bin = nb - 1 - 2 * tid, lo_bin = hi_bin - 1;
    uint32_t c_hi = 0, c_lo = 0;
    if (2 * static_cast<uint32_t>(tid) < nb) {
      c_hi = tot[hi_bin];
      c_lo = tot[lo_bin];
    }
    uint32_t total;
    const uint32_t before = block_excl_scan(c_hi + c_lo, warp_sums, &total);
    if (pass == 0 && total <= static_cast<uint32_t>(k)) {
      all_valid = true;
      break;
    }
    if (2 * static_cast<uint32_t>(tid) < nb) {
      if (before < remaining && before + c_hi >= remaining) {
        s_sel[0] = hi_bin;
        s_sel[1] = before;
      } else if (before + c_hi < remaining && before + c_hi + c_lo >= remaining) {
        s_sel[0] = lo_bin;
        s_sel[1] = before + c_hi;
      }
    }
    __syncthreads();
    remaining -= s_sel[1];
    prefix |= s_sel[0] << sh;
    mask |= (nb - 1) << sh;
    __syncthreads();
  }
  const uint32_t T = all_valid ? 0u : prefix;
  const uint32_t need_eq = all_valid ? 0u : remaining;

  // Per-thread contiguous segments of this CTA's slice keep index order.
  const int seg = (m + kThreads - 1) / kThreads;
  const int s0 = tid * seg, s1 = min(m, s0 + seg);
  uint32_t gt = 0, eq = 0;
  for (int i = s0; i < s1; ++i) {
    const uint32_t u = key[i];
    if (u > T) ++gt;
    else if (u == T && u != 0u) ++eq;
  }
  uint32_t cta_eq, cta_gt;
  const uint32_t eq_base_local = block_excl_scan(eq, warp_sums, &cta_eq);
  block_excl_scan(gt, warp_sums, &cta_gt);
  if (tid == 0) {
    xchg[0] = cta_gt;
    xchg[1] = cta_eq;
  }
  cluster_sync_all();
  // Ties go to the lowest indices: CTA slices are in index order.
  uint32_t eq_before = 0, sel_before = 0, total_sel = 0, eq_cta_before = 0;
  for (uint32_t c = 0; c < static_cast<uint32_t>(C); ++c) {
    const uint32_t g = dsmem_ld(&xchg[0], c), e = dsmem_ld(&xchg[1], c);
    const uint32_t take = need_eq > eq_before ? min(e, need_eq - eq_before) : 0u;
    if (c < r) {
      sel_before += g + take;
      eq_cta_before += e;
    }
    total_sel += g + take;
    eq_before += e;
  }
  const uint32_t eq_base = eq_cta_before + eq_base_local;
  const uint32_t take_eq = need_eq > eq_base ? min(eq, need_eq - eq_base) : 0u;
  uint32_t cta_sel;
  uint32_t o = sel_before + block_excl_scan(gt + take_eq, warp_sums, &cta_sel);
  int32_t* orow = out + static_cast<int64_t>(q) * k;
  const int32_t* prow = pool + static_cast<int64_t>(q) * 2048;
  uint32_t taken_eq = 0;
  for (int i = s0; i < s1; ++i) {
    const uint32_t u = key[i];
    bool sel = u > T;
    if (!sel && u == T && u != 0u && taken_eq < take_eq) {
      sel = true;
      ++taken_eq;
    }
    if (sel) {
      const int64_t gi = lo + i;
      const int32_t v = kMode == 0 ? static_cast<int32_t>(gi) : prow[gi >> 3] * 8 + static_cast<int32_t>(gi & 7);
      if (o < static_cast<uint32_t>(k)) orow[o] = v;  // never past the row, whatever the counts say
      ++o;
    }
  }
  if (r == 0)
    for (int i = static_cast<int>(min(total_sel, static_cast<uint32_t>(k))) + tid; i < k; i += kThreads) orow[i] = -1;
  cluster_sync_all();  // keep this CTA's shared memory alive until every remote read is done
}

constexpr size_t kClusterSmem = (kChunk + 2048 + 2048 + 32 + 4 + 4) * sizeof(uint32_t);

template <int kMode>
cudaError_t launch_cluster_topk(const float* keys, int64_t row_stride, const int64_t* seq_len, int Q,
                                int n_q, int k, int C, const int32_t* pool, int32_t* out,
                                cudaStream_t stream) {
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(cluster_topk_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kClusterSmem));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(cluster_topk_kernel<kMode>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, Q, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kClusterSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, cluster_topk_kernel<kMode>, keys, row_stride, seq_len, n_q, k, C, pool, out);
}

}  // namespace

cudaError_t status_topk(cudaStream_t stream, int* code, int* where, bool clear) {
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

cudaError_t launch_block_topk(const float* block_max, const int64_t* seq_len, int B, int n_q,
                              int64_t max_blocks, int32_t* pool, cudaStream_t stream) {
  const int Q = B * n_q;
  if (Q == 0) return cudaSuccess;
  const int64_t C = (max_blocks + kChunk - 1) / kChunk;
  if (C <= 16) {
    const cudaError_t e = launch_cluster_topk<0>(block_max, max_blocks, seq_len, Q, n_q, 2048,
                                                 static_cast<int>(C < 1 ? 1 : C), nullptr, pool, stream);
    if (e == cudaSuccess || C <= 8) return e;
    cudaGetLastError();  // a 16-CTA cluster may not fit this GPU: use the global-memory select
  }
  radix_topk_kernel<0><<<Q, kThreads, 0, stream>>>(block_max, max_blocks, seq_len, n_q, 2048,
                                                   nullptr, pool);
  return cudaGetLastError();
}

cudaError_t launch_pool_topk(const float* scores, const int64_t* seq_len, int B, int n_q,
                             const int32_t* pool, int32_t* topk, cudaStream_t stream) {
  const int Q = B * n_q;
  if (Q == 0) return cudaSuccess;
  // 16384 scores per token, 2048 per CTA of an 8-CTA cluster.
  return launch_cluster_topk<1>(scores, 16384, seq_len, Q, n_q, 512, 8, pool, topk, stream);
}

}  // namespace csa2
