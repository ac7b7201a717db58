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

// Block-wide exclusive prefix sum over kWarps warps (the whole block); returns
// the total in *total.
template <int kWarps = 32>
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
    uint32_t s = lane < kWarps ? warp_sums[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < kWarps) warp_sums[lane] = s;  // inclusive
  }
  __syncthreads();
  const uint32_t base = warp > 0 ? warp_sums[warp - 1] : 0u;
  const uint32_t tot = warp_sums[kWarps - 1];
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

// Block top-k of one row of block maxima (n = the causal blocks of the token),
// pick k; the output values are block ids. Reads the row from global memory
// on every pass: it serves rows too long for a cluster.
__global__ void __launch_bounds__(kThreads) radix_topk_kernel(const float* __restrict__ keys,
                                                              int64_t row_stride,
                                                              const int64_t* __restrict__ seq_len,
                                                              int n_q, int k, int m_shift,
                                                              int32_t* __restrict__ out) {
  griddep_wait();
  griddep_launch();
  __shared__ uint32_t hist[2048];
  __shared__ uint32_t warp_sums[32];
  __shared__ uint32_t s_sel[2];

  const int q = blockIdx.x;
  const int b = q / n_q, j = q % n_q;
  const int tid = threadIdx.x;
  const float* row = keys + static_cast<int64_t>(q) * row_stride;
  int32_t* orow = out + static_cast<int64_t>(q) * k;
  const int64_t t = ((seq_len[b] - n_q + j + 1) >> m_shift) - 1;  // the token's last visible entry
  int64_t n = t >= 0 ? (t + 8) / 8 : 0;
  if (n > row_stride) {
    if (tid == 0) report(CSA2_ERR_DEVICE_BOUNDS, 301);
    n = row_stride;
  }

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
      if (o < static_cast<uint32_t>(k)) orow[o] = static_cast<int32_t>(i);  // never past the row, whatever the counts say
      ++o;
    }
  }
  for (int i = static_cast<int>(tot_sel) + tid; i < k; i += kThreads) orow[i] = -1;
}

// ---- exact selection over a key set held by the block ------------------------
constexpr int kDigit = 12;
constexpr int kBins = 1 << kDigit;

struct SelectShared {
  uint32_t hist[kBins];
  uint32_t wtot[32];  // per-warp bin totals
  uint32_t bc[5];     // crossing warp and keys above it; selected bin, keys above it and keys in it
};

// The bin that holds the remaining-th largest counted key, scanning bins from
// the top, the number of keys in the bins above it and in it; every thread
// gets all three.
// Warp w owns 128 consecutive bins from the top, lane l four of them; warp 0
// finds the warp whose range holds the crossing, that warp finds the bin.
// Three barriers; the block has 32 warps.
__device__ __forceinline__ void find_bin(SelectShared& S, uint32_t remaining, uint32_t& bin, uint32_t& above,
                                         uint32_t& in_bin) {
  constexpr int kR = kBins / 32, kL = kR / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t c[kL], own = 0;
#pragma unroll
  for (int i = 0; i < kL; ++i) {
    c[i] = S.hist[kBins - 1 - (warp * kR + lane * kL + i)];
    own += c[i];
  }
  const uint32_t wsum = __reduce_add_sync(0xffffffffu, own);
  if (lane == 0) S.wtot[warp] = wsum;
  __syncthreads();
  if (warp == 0) {
    const uint32_t wt = S.wtot[lane];
    uint32_t incl = wt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (incl - wt < remaining && incl >= remaining) {
      S.bc[0] = static_cast<uint32_t>(lane);
      S.bc[1] = incl - wt;
    }
  }
  __syncthreads();
  if (warp == static_cast<int>(S.bc[0])) {
    uint32_t incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    uint32_t before = S.bc[1] + incl - own;
#pragma unroll
    for (int i = 0; i < kL; ++i) {
      if (before < remaining && before + c[i] >= remaining) {
        S.bc[2] = static_cast<uint32_t>(kBins - 1 - (warp * kR + lane * kL + i));
        S.bc[3] = before;
        S.bc[4] = c[i];
      }
      before += c[i];
    }
  }
  __syncthreads();
  bin = S.bc[2];
  above = S.bc[3];
  in_bin = S.bc[4];
}

// Radix select over the valid keys >= lo (all of them <= hi) that visit()
// hands to its callback: T and need_eq such that the keys > T plus the first
// need_eq keys equal to T are the top k (at least k exist). Digits of 12 bits
// from the top of the span hi - lo; at most three passes. It stops early when
// the bin holding the k-th largest key holds exactly the keys still needed:
// every key from that bin's lower bound up is then taken, exactly k keys with
// no tie across the boundary, so T = that bound - 1 and need_eq = 0 select the
// same set as the exact k-th largest would.
template <class Visit>
__device__ __forceinline__ void radix_threshold(const Visit& visit, uint32_t k, uint32_t lo, uint32_t hi,
                                                SelectShared& S, uint32_t& T, uint32_t& need_eq) {
  const uint32_t span = hi - lo;
  const int bits = span ? 32 - __clz(span) : 0;
  int shift = bits > kDigit ? bits - kDigit : 0;
  uint32_t pref = 0u, hmask = 0u, remaining = k;
  for (int pass = 0; pass < 3; ++pass) {
    for (int i = threadIdx.x; i < kBins; i += blockDim.x) S.hist[i] = 0;
    __syncthreads();
    visit([&](uint32_t u) {
      const uint32_t d = u - lo;
      if (u != 0u && u >= lo && (d & hmask) == pref) atomicAdd(&S.hist[(d >> shift) & (kBins - 1)], 1u);
    });
    __syncthreads();
    uint32_t bin, above, in_bin;
    find_bin(S, remaining, bin, above, in_bin);
    remaining -= above;
    pref |= bin << shift;
    hmask = ~((1u << shift) - 1u);
    if (in_bin == remaining) {  // the whole bin is taken
      T = lo + pref - 1u;
      need_eq = 0u;
      return;
    }
    if (shift == 0) break;
    shift = shift > kDigit ? shift - kDigit : 0;
  }
  T = lo + pref;
  need_eq = remaining;
}

// ---- cluster version: the row lives in registers -----------------------------
//
// A cluster of C CTAs (C <= 16) selects from one row; CTA r keeps elements
// [r * chunk, (r + 1) * chunk) of the row buffer in registers as ordered keys
// (thread t holds the 16 consecutive elements from 16 t), so the row is read
// from global memory once. chunk follows from the buffer's row stride, not
// from the token's length, so the loads are issued before the length is known.
//
// The threshold search first narrows the row to a candidate set with samples:
// each warp sorts one sample per lane and takes the j-th largest, j chosen so
// that about 2k/n of the row lies above it; a CTA takes the median over its
// warps, the cluster the median over CTAs (T0). When between k and 8192 keys
// are >= T0, every CTA writes its candidates into CTA 0's shared memory and
// CTA 0 runs the span-based 12-bit radix select on them alone. Otherwise (short
// rows, heavy ties) every pass runs over the whole row: each CTA builds a local
// histogram, every CTA sums all C histograms through distributed shared memory
// and derives the same threshold digit. Either way the result is the same.
// The ordered compaction is one block prefix sum of each thread's packed
// counts of keys above and equal to the threshold; with the counts of lower
// CTAs it gives every selected key its output position in index order.
// Control flow is uniform across the cluster: every CTA executes every cluster
// barrier (a block barrier when the cluster is one CTA).
constexpr int kChunk = 16384;  // elements per CTA at most
constexpr int kMaxC = 16;
constexpr int kSlots = kChunk / kThreads;  // register slots per thread
constexpr int kBlkCandMax = 8192;  // candidate set of the sample filter (in CTA 0)

struct ClusterShared {
  SelectShared S;               // histogram and bin search
  uint32_t tot[kBins];          // cluster-wide histogram slice (whole-row passes)
  uint32_t cand[kBlkCandMax];   // CTA 0: the candidates of the whole row
  uint32_t wred[4][32];         // per warp: min, max, valid count, sample statistic
  uint32_t woff[32];            // per warp: offset of its candidates within the CTA
  uint32_t wsel[2][32];         // per warp: packed (above, equal) counts, then their exclusive prefix
  uint32_t warp_sums[32];
  uint32_t xchg[16];            // read by other CTAs: 0-3 min/max/valid/sample median,
                                // 4 candidate count, 5 slice total, 6-7 gt/eq counts,
                                // 8-9 threshold and equal-key takes (CTA 0)
  uint32_t bc[16];              // block-wide broadcasts
};

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t dsmem_addr(const void* local, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local)), "r"(rank));
  return ra;
}

__device__ __forceinline__ uint32_t dsmem_ld(const uint32_t* local, uint32_t rank) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(dsmem_addr(local, rank)) : "memory");
  return v;
}

__device__ __forceinline__ void dsmem_st(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Ascending bitonic sort of one value per lane (lane 0 ends with the smallest).
__device__ __forceinline__ uint32_t warp_sort_asc(uint32_t v, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint32_t o = __shfl_xor_sync(0xffffffffu, v, stride);
      const bool asc = (lane & size) == 0;
      const bool low = (lane & stride) == 0;
      v = (low == asc) ? min(v, o) : max(v, o);
    }
  }
  return v;
}

__global__ void __launch_bounds__(kThreads, 1) cluster_topk_kernel(const float* __restrict__ keys,
                                                                int64_t row_stride,
                                                                const int64_t* __restrict__ seq_len,
                                                                int n_q, int k, int C, int m_shift,
                                                                int32_t* __restrict__ out) {
  extern __shared__ __align__(16) uint8_t cs_raw[];
  ClusterShared& cs = *reinterpret_cast<ClusterShared*>(cs_raw);
  uint32_t* hist = cs.S.hist;
  uint32_t* tot = cs.tot;
  uint32_t* warp_sums = cs.warp_sums;
  uint32_t* xchg = cs.xchg;
  uint32_t* bc = cs.bc;

  griddep_wait();
  griddep_launch();
  const uint32_t r = cluster_rank();
  const int q = blockIdx.y;
  const int b = q / n_q, j = q % n_q;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // CTA r's slice of the row buffer (the launcher makes C * kChunk >= row_stride).
  const int chunk = static_cast<int>(((row_stride + C - 1) / C + 15) & ~int64_t(15));
  const int lo = static_cast<int>(r) * chunk;
  const int avail = static_cast<int>(max(int64_t(0), min(static_cast<int64_t>(chunk), row_stride - lo)));
  const float* row = keys + static_cast<int64_t>(q) * row_stride + lo;
  const int base = tid * kSlots;  // this thread's first element of the slice
  float f[kSlots];
  if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0 && base + kSlots <= avail) {
#pragma unroll
    for (int i = 0; i < kSlots / 4; ++i) {
      const float4 v = reinterpret_cast<const float4*>(row + base)[i];
      f[4 * i] = v.x;
      f[4 * i + 1] = v.y;
      f[4 * i + 2] = v.z;
      f[4 * i + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < kSlots; ++i) f[i] = base + i < avail ? row[base + i] : -INFINITY;
  }
  const int64_t t = ((seq_len[b] - n_q + j + 1) >> m_shift) - 1;  // the token's last visible entry
  int64_t n64 = t >= 0 ? (t + 8) / 8 : 0;
  if (n64 > row_stride) {
    if (tid == 0 && r == 0) report(CSA2_ERR_DEVICE_BOUNDS, 311);
    n64 = row_stride;
  }
  const int n = static_cast<int>(n64);  // at most 16 * 16384
  const int m = max(0, min(n - lo, chunk));  // valid elements of the slice
  // One cluster-wide barrier; a block barrier when the cluster is one CTA.
  auto csync = [&]() {
    if (C > 1) cluster_sync_all();
    else __syncthreads();
  };

  // Sample statistic: the j-th largest of a warp's 32 samples sits near the
  // (j - 1/3) / (32 + 1/3) quantile; aim at 2k/n, j = floor((2k/n) 97/3 + 5/6),
  // in integers. Rows where 2k/n >= 1/2 skip the sample filter.
  const bool try_filter = n > 4 * k;
  int jrank = n > 0 ? (194 * k + 5 * (n / 2)) / (3 * n) : 32;
  jrank = jrank < 1 ? 1 : (jrank > 32 ? 32 : jrank);

  uint32_t u[kSlots];
#pragma unroll
  for (int it = 0; it < kSlots; ++it) u[it] = base + it < m ? ordered_key(f[it]) : 0u;
  const uint32_t smp = (lane & 1) ? u[kSlots / 2] : u[0];
  uint32_t vmin = 0xFFFFFFFFu, vmax = 0u, nvalid = 0u;
#pragma unroll
  for (int it = 0; it < kSlots; ++it) {
    vmin = min(vmin, u[it] - 1u);  // invalid keys (0) wrap above every valid one
    vmax = max(vmax, u[it]);
    nvalid += u[it] != 0u ? 1u : 0u;
  }
  vmin = nvalid ? vmin + 1u : 0xFFFFFFFFu;
  vmin = __reduce_min_sync(0xffffffffu, vmin);
  vmax = __reduce_max_sync(0xffffffffu, vmax);
  nvalid = __reduce_add_sync(0xffffffffu, nvalid);
  const uint32_t stat = __shfl_sync(0xffffffffu, warp_sort_asc(smp, lane), 32 - jrank);
  if (lane == 0) {
    cs.wred[0][warp] = vmin;
    cs.wred[1][warp] = vmax;
    cs.wred[2][warp] = nvalid;
    cs.wred[3][warp] = stat;
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t mn = __reduce_min_sync(0xffffffffu, cs.wred[0][lane]);
    const uint32_t mx = __reduce_max_sync(0xffffffffu, cs.wred[1][lane]);
    const uint32_t nv = __reduce_add_sync(0xffffffffu, cs.wred[2][lane]);
    const uint32_t med = __shfl_sync(0xffffffffu, warp_sort_asc(cs.wred[3][lane], lane), 16);
    if (lane == 0) {
      xchg[0] = mn;
      xchg[1] = mx;
      xchg[2] = nv;
      xchg[3] = med;
    }
  }
  csync();
  if (warp == 0) {
    const bool in = lane < C;
    const uint32_t mn = __reduce_min_sync(0xffffffffu, in ? dsmem_ld(&xchg[0], lane) : 0xFFFFFFFFu);
    const uint32_t mx = __reduce_max_sync(0xffffffffu, in ? dsmem_ld(&xchg[1], lane) : 0u);
    const uint32_t nv = __reduce_add_sync(0xffffffffu, in ? dsmem_ld(&xchg[2], lane) : 0u);
    const uint32_t tr = in ? dsmem_ld(&xchg[3], lane) : 0u;
    uint32_t rank = 0;  // among the C CTA medians, ties by rank
#pragma unroll
    for (int l = 0; l < kMaxC; ++l) {
      const uint32_t x = __shfl_sync(0xffffffffu, tr, l);
      rank += (l < C && (x > tr || (x == tr && l < lane))) ? 1u : 0u;
    }
    const int pick = __ffs(__ballot_sync(0xffffffffu, in && rank == static_cast<uint32_t>(C / 2))) - 1;
    const uint32_t T0 = __shfl_sync(0xffffffffu, tr, pick);
    if (lane == 0) {
      bc[0] = mn;
      bc[1] = mx;
      bc[2] = nv;
      bc[3] = T0;
    }
  }
  __syncthreads();
  const uint32_t umin = bc[0], umax = bc[1], total_valid = bc[2], T0 = bc[3];

  // Threshold: take keys > T and the first need_eq keys equal to T.
  uint32_t T = 0u, need_eq = 0u;
  if (total_valid > static_cast<uint32_t>(k)) {
    bool filtered = false;
    if (try_filter && T0 != 0u) {
      uint32_t c = 0;  // T0 >= 1, so invalid keys never count
#pragma unroll
      for (int it = 0; it < kSlots; ++it) c += u[it] >= T0 ? 1u : 0u;
      const uint32_t cw = __reduce_add_sync(0xffffffffu, c);
      if (lane == 0) cs.wred[0][warp] = cw;  // wred[0] was last read before the cluster barrier
      __syncthreads();
      if (warp == 0) {
        const uint32_t wv = cs.wred[0][lane];
        uint32_t incl = wv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        cs.woff[lane] = incl - wv;
        if (lane == 31) xchg[4] = incl;
      }
      csync();
      if (warp == 0) {
        const uint32_t cr = lane < C ? dsmem_ld(&xchg[4], lane) : 0u;
        uint32_t incl = cr;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const uint32_t base = __shfl_sync(0xffffffffu, incl - cr, static_cast<int>(r));
        const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
        if (lane == 0) {
          bc[4] = base;
          bc[5] = total;
        }
      }
      __syncthreads();
      const uint32_t n_cand = bc[5];
      if (n_cand >= static_cast<uint32_t>(k) && n_cand <= static_cast<uint32_t>(kBlkCandMax)) {
        filtered = true;
        // Candidates into CTA 0's shared memory (any order).
        uint32_t incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const uint32_t dst0 = dsmem_addr(cs.cand, 0);
        uint32_t pos = bc[4] + cs.woff[warp] + incl - c;
#pragma unroll
        for (int it = 0; it < kSlots; ++it) {
          if (u[it] >= T0) {
            dsmem_st(dst0 + 4u * pos, u[it]);
            ++pos;
          }
        }
        csync();  // every candidate is in CTA 0
        if (r == 0) {
          radix_threshold([&](auto&& fn) {
            for (int i = tid; i < static_cast<int>(n_cand); i += kThreads) fn(cs.cand[i]);
          }, static_cast<uint32_t>(k), T0, umax, cs.S, T, need_eq);
          if (tid == 0) {
            xchg[8] = T;
            xchg[9] = need_eq;
          }
        }
        csync();  // CTA 0's threshold is published
        if (tid == 0) {
          bc[6] = dsmem_ld(&xchg[8], 0);
          bc[7] = dsmem_ld(&xchg[9], 0);
        }
        __syncthreads();
        T = bc[6];
        need_eq = bc[7];
      }
    }
    if (!filtered) {
      const uint32_t span = umax - umin;
      const int bits = span ? 32 - __clz(span) : 0;
      int shift = bits > kDigit ? bits - kDigit : 0;
      uint32_t pref = 0u, hmask = 0u, remaining = static_cast<uint32_t>(k);
      bool whole_bin = false;  // stopped early: every key from the selected bin up is taken
      for (int pass = 0; pass < 3; ++pass) {
        for (int i = tid; i < kBins; i += kThreads) hist[i] = 0;
        __syncthreads();
#pragma unroll
        for (int it = 0; it < kSlots; ++it) {
          const uint32_t uu = u[it];
          const uint32_t d = uu - umin;
          if (uu != 0u && (d & hmask) == pref) atomicAdd(&hist[(d >> shift) & (kBins - 1)], 1u);
        }
        csync();  // every local histogram is complete
        // CTA r sums the bins of its slice [r * Sn, (r + 1) * Sn) over the cluster
        // (the last slice may be short); a single CTA uses its own histogram as is.
        const int Sn = (kBins + C - 1) / C;
        const uint32_t* totals = hist;
        if (C > 1) {
          uint32_t part = 0;
          for (int bi = tid; bi < Sn; bi += kThreads) {
            const int bin = static_cast<int>(r) * Sn + bi;
            if (bin >= kBins) break;
            uint32_t sum = 0;
            for (int cc = 0; cc < C; ++cc) sum += dsmem_ld(&hist[bin], cc);
            tot[bin] = sum;
            part += sum;
          }
          uint32_t slice_total;
          block_excl_scan(part, warp_sums, &slice_total);
          if (tid == 0) xchg[5] = slice_total;
          totals = tot;
        }
        csync();  // slice sums complete; nobody reads a remote histogram any more
        // The slice that holds the remaining-th largest key (slices of higher ranks
        // hold higher digits), and the keys above it.
        if (warp == 0) {
          const uint32_t st = lane < C ? (C > 1 ? dsmem_ld(&xchg[5], lane) : 0u) : 0u;
          uint32_t incl = st;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_down_sync(0xffffffffu, incl, o);
            if (lane + o < 32) incl += y;
          }
          const uint32_t above = incl - st;
          if (lane == 0) {
            bc[8] = 0;
            bc[9] = 0;
          }
          __syncwarp();
          if (C > 1 && lane < C && above < remaining && above + st >= remaining) {
            bc[8] = lane;
            bc[9] = above;
          }
        }
        __syncthreads();
        const uint32_t target = min(bc[8], static_cast<uint32_t>(C - 1));  // always a rank of this cluster
        const uint32_t above_t = bc[9];
        __syncthreads();
        // Thread t owns kPer consecutive bins of the target slice counted from the top.
        constexpr int kPer = kBins / kThreads;
        uint32_t c4[kPer], own = 0;
#pragma unroll
        for (int it = 0; it < kPer; ++it) {
          const int rank = tid * kPer + it;
          c4[it] = 0;
          const int bin = static_cast<int>(target) * Sn + (Sn - 1 - rank);
          if (rank < Sn && bin < kBins) c4[it] = C > 1 ? dsmem_ld(&totals[bin], target) : totals[bin];
          own += c4[it];
        }
        uint32_t total;
        uint32_t before = above_t + block_excl_scan(own, warp_sums, &total);
#pragma unroll
        for (int it = 0; it < kPer; ++it) {
          const int rank = tid * kPer + it;
          if (rank < Sn && before < remaining && before + c4[it] >= remaining) {
            bc[10] = static_cast<uint32_t>(static_cast<int>(target) * Sn + (Sn - 1 - rank));
            bc[11] = before;
            bc[15] = c4[it];
          }
          before += c4[it];
        }
        __syncthreads();
        remaining -= bc[11];
        pref |= bc[10] << shift;
        hmask = ~((1u << shift) - 1u);
        // The same cluster-wide counts in every CTA: all stop at the same pass.
        whole_bin = bc[15] == remaining;
        __syncthreads();
        if (whole_bin || shift == 0) break;
        shift = shift > kDigit ? shift - kDigit : 0;
      }
      // Stopped early (see radix_threshold): T = the bin's lower bound - 1, no equal keys.
      T = whole_bin ? umin + pref - 1u : umin + pref;
      need_eq = whole_bin ? 0u : remaining;
    }
  }

  // Ordered compaction. Keys equal to T are all valid when T > 0; when T = 0
  // every valid key is taken and need_eq = 0 takes no "equal" (invalid) key.
  // Index order is (CTA, thread, slot): one block prefix sum of the packed
  // (above, equal) counts (16 bits each; a slice has at most 16384 of either).
  uint32_t gm = 0, em = 0;  // per-slot masks: above T, equal to T
#pragma unroll
  for (int it = 0; it < kSlots; ++it) {
    gm |= (u[it] > T ? 1u : 0u) << it;
    em |= (u[it] == T && u[it] != 0u ? 1u : 0u) << it;
  }
  const uint32_t v = (static_cast<uint32_t>(__popc(gm)) << 16) | static_cast<uint32_t>(__popc(em));
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) cs.wsel[0][warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const uint32_t wt = cs.wsel[0][lane];
    uint32_t wi = wt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    cs.wsel[1][lane] = wi - wt;
    if (lane == 31) {
      xchg[6] = wi >> 16;      // keys above T in this CTA
      xchg[7] = wi & 0xFFFFu;  // keys equal to T in this CTA
    }
  }
  csync();
  if (warp == 0) {  // ties go to the lowest indices: CTA slices are in index order
    const uint32_t g = lane < C ? dsmem_ld(&xchg[6], lane) : 0u;
    const uint32_t e = lane < C ? dsmem_ld(&xchg[7], lane) : 0u;
    uint32_t g_incl = g, e_incl = e;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t yg = __shfl_up_sync(0xffffffffu, g_incl, o), ye = __shfl_up_sync(0xffffffffu, e_incl, o);
      if (lane >= o) {
        g_incl += yg;
        e_incl += ye;
      }
    }
    const uint32_t gt_all = __shfl_sync(0xffffffffu, g_incl, 31);
    const uint32_t eq_all = __shfl_sync(0xffffffffu, e_incl, 31);
    if (lane == static_cast<int>(r)) {
      bc[12] = g_incl - g;  // keys above T in lower CTAs
      bc[13] = e_incl - e;  // keys equal to T in lower CTAs
    }
    if (lane == 0) bc[14] = gt_all + min(eq_all, need_eq);  // keys selected in the whole row
  }
  __syncthreads();
  const uint32_t total_sel = bc[14];
  const uint32_t before = cs.wsel[1][warp] + incl - v;  // packed counts of lower threads of this CTA
  const uint32_t gb = bc[12] + (before >> 16), eb = bc[13] + (before & 0xFFFFu);
  // This thread's equal keys that are taken: the lowest min(popc, need_eq - eb) of them.
  uint32_t take = need_eq > eb ? need_eq - eb : 0u;
  uint32_t sel = gm, rest = em;
  while (take > 0u && rest != 0u) {
    const uint32_t lowest = rest & (0u - rest);
    sel |= lowest;
    rest ^= lowest;
    --take;
  }
  int32_t* orow = out + static_cast<int64_t>(q) * k;
  uint32_t pos = gb + min(eb, need_eq);
  while (sel != 0u) {
    const int i = __ffs(sel) - 1;
    sel &= sel - 1u;
    if (pos < static_cast<uint32_t>(k)) orow[pos] = lo + base + i;  // never past the row
    ++pos;
  }
  if (r == 0)
    for (int i = static_cast<int>(min(total_sel, static_cast<uint32_t>(k))) + tid; i < k; i += kThreads) orow[i] = -1;
  csync();  // keep this CTA's shared memory alive until every remote read is done
}

constexpr size_t kClusterSmem = sizeof(ClusterShared);

cudaError_t launch_cluster_topk(const float* keys, int64_t row_stride, const int64_t* seq_len, int Q,
                                int n_q, int k, int C, int m_shift, int32_t* out, cudaStream_t stream) {
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(cluster_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kClusterSmem));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(cluster_topk_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev] = true;
  }
  return launch_pdl(cluster_topk_kernel, dim3(C, Q, 1), dim3(kThreads), kClusterSmem, stream,
                    static_cast<unsigned>(C), keys, row_stride, seq_len, n_q, k, C, m_shift, out);
}

// ---- pool top-k: one CTA per token, the row in registers --------------------
//
// A token's pool row holds 16384 scores (2048 blocks x 8 positions). Each of
// 1024 threads keeps 16 consecutive ordered keys in registers (4 float4 loads
// in flight at once), so the row is read once and no pass touches global
// memory. Warp shuffles are the scarce resource here (one warp instruction per
// clock per SM), so reductions use redux.sync and work that needs a shuffle
// scan is done by one warp, not redundantly by all 32.
//
// The threshold search first narrows the row to a candidate set: T0 = the
// median over warps of each warp's second-largest sample (one sample per
// lane) sits near the 6% quantile, so usually between k and 2048 keys are
// >= T0. Those candidates go to shared memory and the span-based 12-bit radix
// select runs on them alone (two keys per thread at most, hence few
// shared-memory atomics). When the count falls outside [k, 2048] (heavy ties,
// adversarial orders) the radix select runs on all keys instead; the result is
// the same either way, only the cost differs. The compaction is one block
// prefix sum of each thread's count of keys above and equal to the threshold,
// packed into one word (16 bits each; a row has at most 16384 of either).
constexpr int kPoolRow = 16384;
constexpr int kPoolThreads = 1024;
constexpr int kPoolKeys = kPoolRow / kPoolThreads;  // 16 consecutive keys per thread
constexpr int kCandMax = 2048;

__global__ void __launch_bounds__(kPoolThreads, 1) pool_topk_kernel(const float* __restrict__ scores,
                                                                    const int32_t* __restrict__ pool, int k,
                                                                    int32_t* __restrict__ out) {
  __shared__ SelectShared S;
  __shared__ uint32_t cand[kCandMax];
  __shared__ int32_t pool_sm[2048];
  __shared__ uint32_t red[7 * 32];  // per-warp values; every use has its own 32 slots
  __shared__ uint32_t misc[4];      // candidate count, T0, packed selection total

  griddep_wait();
  griddep_launch();
  const int q = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float4* row = reinterpret_cast<const float4*>(scores + static_cast<int64_t>(q) * kPoolRow);
  float4 f[kPoolKeys / 4];
#pragma unroll
  for (int j = 0; j < kPoolKeys / 4; ++j) f[j] = row[tid * (kPoolKeys / 4) + j];
  const int32_t* prow = pool + static_cast<int64_t>(q) * 2048;
#pragma unroll
  for (int i = 0; i < 2048 / kPoolThreads; ++i) pool_sm[tid + i * kPoolThreads] = prow[tid + i * kPoolThreads];
  if (tid == 0) misc[0] = 0;

  uint32_t u[kPoolKeys];
#pragma unroll
  for (int j = 0; j < kPoolKeys / 4; ++j) {
    u[4 * j + 0] = ordered_key(f[j].x);
    u[4 * j + 1] = ordered_key(f[j].y);
    u[4 * j + 2] = ordered_key(f[j].z);
    u[4 * j + 3] = ordered_key(f[j].w);
  }
  // One sample per thread: the first or the eighth key of its run.
  const uint32_t smp = (lane & 1) ? u[7] : u[0];
  // Invalid keys are 0: u - 1 wraps them above every valid key for the minimum.
  uint32_t vmin = 0xFFFFFFFFu, vmax = 0u, nvalid = 0u;
#pragma unroll
  for (int i = 0; i < kPoolKeys; ++i) {
    vmin = min(vmin, u[i] - 1u);
    vmax = max(vmax, u[i]);
    nvalid += u[i] != 0u ? 1u : 0u;
  }
  vmin += 1u;  // 0 when every key of the thread is invalid: then vmax is 0 too
  if (nvalid == 0u) vmin = 0xFFFFFFFFu;
  // The warp's second-largest sample (the largest taken once).
  const uint32_t m1 = __reduce_max_sync(0xffffffffu, smp);
  const int first = __ffs(__ballot_sync(0xffffffffu, smp == m1)) - 1;
  const uint32_t m2 = __reduce_max_sync(0xffffffffu, lane == first ? 0u : smp);
  vmin = __reduce_min_sync(0xffffffffu, vmin);
  vmax = __reduce_max_sync(0xffffffffu, vmax);
  nvalid = __reduce_add_sync(0xffffffffu, nvalid);
  if (lane == 0) {
    red[warp] = vmin;
    red[32 + warp] = vmax;
    red[64 + warp] = nvalid;
    red[96 + warp] = m2;
  }
  __syncthreads();
  const uint32_t umin = __reduce_min_sync(0xffffffffu, red[lane]);
  const uint32_t umax = __reduce_max_sync(0xffffffffu, red[32 + lane]);
  const uint32_t total_valid = __reduce_add_sync(0xffffffffu, red[64 + lane]);

  // Threshold: take keys > T and the first need_eq keys equal to T.
  uint32_t T = 0u, need_eq = 0u;
  if (total_valid > static_cast<uint32_t>(k)) {
    if (warp == 0) {  // T0 = the 16th largest of the warps' second-largest samples
      const uint32_t v = red[96 + lane];
      uint32_t rank = 0;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const uint32_t x = __shfl_sync(0xffffffffu, v, j);
        rank += (x > v || (x == v && j < lane)) ? 1u : 0u;
      }
      if (rank == 15u) misc[1] = v;
    }
    __syncthreads();
    const uint32_t T0 = misc[1];
    uint32_t c = 0;  // T0 >= 1 whenever it is used, so invalid keys never count
#pragma unroll
    for (int i = 0; i < kPoolKeys; ++i) c += u[i] >= T0 ? 1u : 0u;
    const uint32_t cw = __reduce_add_sync(0xffffffffu, c);
    if (lane == 0) red[128 + warp] = cw;
    __syncthreads();
    const uint32_t n_cand = __reduce_add_sync(0xffffffffu, red[128 + lane]);
    if (T0 != 0u && n_cand >= static_cast<uint32_t>(k) && n_cand <= static_cast<uint32_t>(kCandMax)) {
      // Candidates to shared memory (any order).
      uint32_t incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      uint32_t base = 0;
      if (lane == 31) base = atomicAdd(&misc[0], incl);
      uint32_t o = __shfl_sync(0xffffffffu, base, 31) + incl - c;
#pragma unroll
      for (int i = 0; i < kPoolKeys; ++i)
        if (u[i] >= T0) cand[o++] = u[i];
      __syncthreads();
      radix_threshold([&](auto&& fn) {
        for (int i = tid; i < static_cast<int>(n_cand); i += kPoolThreads) fn(cand[i]);
      }, static_cast<uint32_t>(k), T0, umax, S, T, need_eq);
    } else {
      radix_threshold([&](auto&& fn) {
#pragma unroll
        for (int i = 0; i < kPoolKeys; ++i) fn(u[i]);
      }, static_cast<uint32_t>(k), umin, umax, S, T, need_eq);
    }
  }

  // Ordered compaction: one block prefix sum of the packed (above, equal)
  // counts, then each thread writes its selected slots in order. When T = 0
  // (every valid key is taken) the "equal" keys are the invalid ones and
  // need_eq = 0 takes none of them.
  uint32_t gm = 0, em = 0;  // per-key masks: above T, equal to T
#pragma unroll
  for (int i = 0; i < kPoolKeys; ++i) {
    gm |= (u[i] > T ? 1u : 0u) << i;
    em |= (u[i] == T ? 1u : 0u) << i;
  }
  const uint32_t v = (static_cast<uint32_t>(__popc(gm)) << 16) | static_cast<uint32_t>(__popc(em));
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) red[160 + warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const uint32_t wt = red[160 + lane];
    uint32_t wi = wt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    red[192 + lane] = wi - wt;
    if (lane == 31) misc[2] = wi;
  }
  __syncthreads();
  const uint32_t tot = misc[2];
  const uint32_t n_sel = min((tot >> 16) + min(tot & 0xFFFFu, need_eq), static_cast<uint32_t>(k));
  int32_t* orow = out + static_cast<int64_t>(q) * k;
  const uint32_t base = red[192 + warp] + incl - v;
  const uint32_t gb = base >> 16, eb = base & 0xFFFFu;  // keys above / equal to T in lower threads
  // This thread's equal keys that are taken: the lowest min(popc, need_eq - eb) of them.
  uint32_t take = need_eq > eb ? need_eq - eb : 0u;
  uint32_t sel = gm, rest = em;
  while (take > 0u && rest != 0u) {
    const uint32_t lowest = rest & (0u - rest);
    sel |= lowest;
    rest ^= lowest;
    --take;
  }
  uint32_t pos = gb + min(eb, need_eq);
  while (sel != 0u) {
    const int i = __ffs(sel) - 1;
    sel &= sel - 1u;
    const int slot = tid * kPoolKeys + i;
    if (pos < static_cast<uint32_t>(k)) orow[pos] = pool_sm[slot >> 3] * 8 + (slot & 7);
    ++pos;
  }
  for (int i = static_cast<int>(n_sel) + tid; i < k; i += kPoolThreads) orow[i] = -1;
}

}  // namespace

cudaError_t force_timeout_topk(int site, cudaStream_t stream) { return set_force_timeout_site(site, stream); }

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
                              int64_t max_blocks, int32_t* pool, cudaStream_t stream, int m) {
  const int Q = B * n_q;
  if (Q == 0) return cudaSuccess;
  // Half-full CTAs (8192 elements) while few rows make few 16-CTA clusters
  // (a cluster of 16 needs 16 free SMs of one GPC), else full ones.
  int64_t C = (max_blocks + 8191) / 8192;
  if (C > 16 || static_cast<int64_t>(Q) * C > 64) C = (max_blocks + kChunk - 1) / kChunk;
  if (C <= 16) {
    const cudaError_t e = launch_cluster_topk(block_max, max_blocks, seq_len, Q, n_q, 2048,
                                              static_cast<int>(C < 1 ? 1 : C), m == 2 ? 1 : 0, pool, stream);
    if (e == cudaSuccess || C <= 8) return e;
    cudaGetLastError();  // a 16-CTA cluster may not fit this GPU: use the global-memory select
  }
  return launch_pdl(radix_topk_kernel, dim3(Q), dim3(kThreads), 0, stream, 0, block_max, max_blocks, seq_len, n_q,
                    2048, m == 2 ? 1 : 0, pool);
}

cudaError_t launch_pool_topk(const float* scores, const int64_t* seq_len, int B, int n_q,
                             const int32_t* pool, int32_t* topk, cudaStream_t stream) {
  (void)seq_len;  // causality is already in the scores: masked slots are -inf
  const int Q = B * n_q;
  if (Q == 0) return cudaSuccess;
  return launch_pdl(pool_topk_kernel, dim3(Q), dim3(kPoolThreads), 0, stream, 0, scores, pool, 512, topk);
}

}  // namespace csa2
