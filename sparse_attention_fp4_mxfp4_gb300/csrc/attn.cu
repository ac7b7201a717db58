// Reuse-mode sparse attention ("DeepSeek V4.1: model architecture and system
// design, a close reading" sections 1 and 2.2; "DeepSeek-V4.1-Flash: Pushing
// the Limits of KV Cache Compression" sections 3.3 and 3.6; "DeepSeek-V4 model
// structure (7): structure decides the system", closing summary): 64 query
// heads attend, with K = V = the 512-channel latent, to the query's top-k
// main entries (MXFP4, dequantised before attention) and to its FP8
// sliding-window entries.
//
// Split-KV: a query's 640 key slots are cut into five splits of 128 (four of
// top-k entries, one of window entries), one CTA each. A CTA gathers its keys,
// dequantises them to f16 (exact) into one 128-byte-swizzled tile, and runs
//   S^T[128 keys x 64 heads] = K Q^T    (tcgen05, M = 128, N = 64, K = 512)
//   exact softmax over its keys (fp32), P^T in f16
//   O^T[512 dims x 64 heads] = V^T P^T  (tcgen05, 4 x M = 128, N = 64, K = 128)
// where V^T is the same shared-memory tile read as an MN-major operand. The
// partial (max, sum, O) of every split is merged by a second kernel.
#include <algorithm>

#include "formats.cuh"
#include "kernels.h"
#include "sm103.cuh"

namespace csa2 {
namespace {

constexpr int kSplits = 5;
constexpr int kThreads = 256;
constexpr int kKtOff = 0;                 // 128 keys x 512 f16: 8 K-blocks of 16 KB
constexpr int kQsOff = 131072;            // 64 heads x 512 f16: 8 K-blocks of 8 KB
constexpr int kSOff = kQsOff;             // after S = K Q^T: fp32 [128][65]
constexpr int kPtOff = kQsOff + 40960;    // P^T f16 [64 heads x 128 keys]: 2 K-blocks of 8 KB
constexpr int kMiscOff = kQsOff + 65536;  // barriers, flags, reductions
constexpr int kSmemBytes = 1024 + kMiscOff + 4096;
constexpr int kSStride = 65;
constexpr float kLog2e = 1.4426950408889634f;

struct AttnParams {
  const uint16_t* q;
  const int32_t* topk;
  const int64_t* seq_len;
  int B, n_q;
  const int32_t* block_table;
  int max_pages;
  int64_t n_pages;
  const uint8_t* main_pages;
  const uint8_t* rings;
  const int32_t* ring_idx;
  int64_t n_rings;
  float scale_log2;   // softmax_scale * log2(e)
  float* part;        // [Q][5][64][512]
  float2* stats;      // [Q][5][64] (max in log2 units, sum)
};

__global__ void __launch_bounds__(kThreads, 1) attn_split_kernel(const AttnParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Kt = smem + kKtOff;
  uint8_t* Qs = smem + kQsOff;
  float* Ss = reinterpret_cast<float*>(smem + kSOff);
  uint8_t* Pt = smem + kPtOff;
  uint8_t* misc = smem + kMiscOff;
  uint64_t* bar = reinterpret_cast<uint64_t*>(misc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 8);
  int64_t* key_off = reinterpret_cast<int64_t*>(misc + 64);       // [128] byte offsets, -1 = none
  float* red = reinterpret_cast<float*>(misc + 64 + 1024);         // [4][64]
  float* mh = red + 256;                                           // [64]
  float* lh = mh + 64;                                             // [64]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x;
  const int q = blockIdx.y;
  const int b = q / P.n_q, j = q % P.n_q;
  const int64_t N = P.seq_len[b];
  const int64_t t = N - P.n_q + j;
  const uint32_t mbar = smem_u32(bar);

  if (tid == 0) {
    mbar_init(mbar, 1);
    mbar_init_fence();
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), 512);

  // Issue this thread's 16 Q loads first: they do not depend on anything and
  // overlap with the key-slot lookups below.
  const uint4* qg = reinterpret_cast<const uint4*>(P.q + static_cast<int64_t>(q) * 64 * 512);
  uint4 qv[16];
#pragma unroll
  for (int it = 0; it < 16; ++it) qv[it] = qg[tid + it * kThreads];

  // ---- key slots of this split ----
  if (tid < 128) {
    int64_t off = -1;
    if (split < 4) {
      const int32_t p = P.topk[static_cast<int64_t>(q) * 512 + split * 128 + tid];
      if (p >= 0) {
        if (p > t || (p >> 7) >= P.max_pages) {
          report(CSA2_ERR_DEVICE_BOUNDS, 401);
        } else {
          const int32_t page = P.block_table[static_cast<int64_t>(b) * P.max_pages + (p >> 7)];
          if (page < 0 || page >= P.n_pages) report(CSA2_ERR_DEVICE_BOUNDS, 402);
          else off = static_cast<int64_t>(page) * (128 * 288) + (p & 127) * 288;
        }
      }
    } else {
      const int32_t r = P.ring_idx[b];
      const int64_t base = N - 128;  // the ring holds positions N-128 .. N-1
      int64_t d = (static_cast<int64_t>(tid) - base) % 128;
      if (d < 0) d += 128;
      const int64_t p = base + d;   // the position stored in slot tid
      int64_t lo = t - 127;
      if (lo < base) lo = base;
      if (lo < 0) lo = 0;
      if (r < 0 || r >= P.n_rings) {
        if (tid == 0) report(CSA2_ERR_DEVICE_BOUNDS, 403);
      } else if (p >= lo && p <= t) {
        off = (static_cast<int64_t>(r) * 128 + tid) * 512;
      }
    }
    key_off[tid] = off;
  }

  __syncthreads();  // key slots are known

  // ---- gather + dequantise keys into the swizzled A operand ----
  // All of a thread's key loads are issued before any is used. A missing key
  // becomes zero codes with a zero scale, which dequantises to zeros.
  if (split < 4) {
    uint4 cv[8];
    uint32_t sv[8];
#pragma unroll
    for (int it = 0; it < 8; ++it) {
      const int i = tid + it * kThreads;
      const int r = i >> 4, c = i & 15;  // key row, 32-channel chunk
      const int64_t off = key_off[r];
      cv[it] = make_uint4(0, 0, 0, 0);
      sv[it] = 0;
      if (off >= 0) {
        const uint8_t* e = P.main_pages + off;
        cv[it] = *reinterpret_cast<const uint4*>(e + c * 16);
        sv[it] = *reinterpret_cast<const uint16_t*>(e + 256 + 2 * c);
      }
    }
#pragma unroll
    for (int it = 0; it < 8; ++it) {
      const int i = tid + it * kThreads;
      const int r = i >> 4, c = i & 15;
      uint4 out[4];
      dequant32_f16(cv[it], static_cast<uint16_t>(sv[it]), out);
      uint8_t* kb = Kt + (c >> 1) * 16384;
#pragma unroll
      for (int k = 0; k < 4; ++k) *reinterpret_cast<uint4*>(kb + sw128_offset(r, (c & 1) * 4 + k)) = out[k];
    }
  } else {
    uint4 rv[16];
#pragma unroll
    for (int it = 0; it < 16; ++it) {
      const int i = tid + it * kThreads;
      const int r = i >> 5, c = i & 31;  // key row, 16-channel chunk
      const int64_t off = key_off[r];
      rv[it] = off >= 0 ? *reinterpret_cast<const uint4*>(P.rings + off + c * 16) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int it = 0; it < 16; ++it) {
      const int i = tid + it * kThreads;
      const int r = i >> 5, c = i & 31;
      const uint32_t w[4] = {rv[it].x, rv[it].y, rv[it].z, rv[it].w};
      uint32_t h[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        h[2 * k] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[k] & 0xFFFFu));
        h[2 * k + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[k] >> 16));
      }
      uint8_t* kb = Kt + (c >> 2) * 16384;
      *reinterpret_cast<uint4*>(kb + sw128_offset(r, (c & 3) * 2)) = make_uint4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<uint4*>(kb + sw128_offset(r, (c & 3) * 2 + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
    }
  }
  // ---- Q (bf16 -> f16) into the swizzled B operand ----
#pragma unroll
  for (int it = 0; it < 16; ++it) {
    const int i = tid + it * kThreads;
    const int h = i >> 6, c = i & 63;
    float f[8];
    bf16x8_to_f32(qv[it], f);
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      __half2 hv = __floats2half2_rn(f[2 * k], f[2 * k + 1]);
      o[k] = *reinterpret_cast<uint32_t*>(&hv);
    }
    *reinterpret_cast<uint4*>(Qs + (c >> 3) * 8192 + sw128_offset(h, c & 7)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // ---- S^T = K Q^T on the tensor cores ----
  if (tid == 0) {
    const uint32_t idesc = idesc_f16(128, 64, false, false);
    const uint32_t kt = smem_u32(Kt), qs = smem_u32(Qs);
#pragma unroll 4
    for (int k = 0; k < 32; ++k) {
      const uint64_t ad = sdesc(kt + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024, kSwizzle128B);
      const uint64_t bd = sdesc(qs + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024, kSwizzle128B);
      umma_f16(tmem, ad, bd, idesc, k > 0 ? 1u : 0u);
    }
    umma_commit(mbar);
  }
  const bool ok1 = mbar_wait(mbar, 0, 411);
  tc_fence_after();

  // ---- softmax over this split's keys ----
  const int quarter = warp & 3, half = warp >> 2;
  const int r = quarter * 32 + lane;  // key row of this thread
  const bool kvalid = key_off[r] >= 0;
  float l[32];
  {
    uint32_t raw[32];
    tmem_ld32(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + half * 32, raw);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) l[i] = (kvalid && ok1) ? __uint_as_float(raw[i]) * P.scale_log2 : -INFINITY;
  }
  // Q is no longer needed: its region now holds the logits (padded rows).
#pragma unroll
  for (int i = 0; i < 32; ++i) Ss[r * kSStride + half * 32 + i] = l[i];
  __syncthreads();
  {
    const int h = tid & 63, kq = tid >> 6;
    float m = -INFINITY;
    for (int i = 0; i < 32; ++i) m = fmaxf(m, Ss[(kq * 32 + i) * kSStride + h]);
    red[kq * 64 + h] = m;
  }
  __syncthreads();
  if (tid < 64) mh[tid] = fmaxf(fmaxf(red[tid], red[64 + tid]), fmaxf(red[128 + tid], red[192 + tid]));
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int h = half * 32 + i;
    const float m = fmaxf(fmaxf(red[h], red[64 + h]), fmaxf(red[128 + h], red[192 + h]));
    const float p = (m == -INFINITY) ? 0.f : exp2f(l[i] - m);
    const __half ph = __float2half_rn(p);
    // P^T is the K-major B operand [64 heads x 128 keys].
    *reinterpret_cast<__half*>(Pt + (r >> 6) * 8192 + sw128_offset(h, (r & 63) >> 3) + (r & 7) * 2) = ph;
    Ss[r * kSStride + h] = __half2float(ph);
  }
  __syncthreads();  // every read of the maxima in red[] is done
  {
    const int h = tid & 63, kq = tid >> 6;
    float s = 0.f;
    for (int i = 0; i < 32; ++i) s += Ss[(kq * 32 + i) * kSStride + h];
    red[kq * 64 + h] = s;
  }
  __syncthreads();
  if (tid < 64) lh[tid] = (red[tid] + red[64 + tid]) + (red[128 + tid] + red[192 + tid]);
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---- O^T = V^T P^T on the tensor cores (V^T: the key tile read MN-major) ----
  if (tid == 0) {
    const uint32_t idesc = idesc_f16(128, 64, true, false);
    const uint32_t kt = smem_u32(Kt), pt = smem_u32(Pt);
    for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint64_t ad = sdesc(kt + mt * 32768 + ks * 2048, 16384, 1024, kSwizzle128B);
        const uint64_t bd = sdesc(pt + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024, kSwizzle128B);
        umma_f16(tmem + 64 + 64 * mt, ad, bd, idesc, ks > 0 ? 1u : 0u);
      }
    }
    umma_commit(mbar);
  }
  const bool ok2 = mbar_wait(mbar, 1, 412);
  tc_fence_after();

  // ---- partial output ----
  const int64_t pidx = static_cast<int64_t>(q) * kSplits + split;
  float* part = P.part + pidx * (64 * 512);
  for (int mt = 0; mt < 4; ++mt) {
    uint32_t raw[32];
    tmem_ld32(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + 64 + 64 * mt + half * 32, raw);
    tmem_wait_ld();
    const int d = mt * 128 + quarter * 32 + lane;
#pragma unroll
    for (int i = 0; i < 32; ++i) part[(half * 32 + i) * 512 + d] = ok2 ? __uint_as_float(raw[i]) : 0.f;
  }
  if (tid < 64) P.stats[pidx * 64 + tid] = make_float2((ok1 && ok2) ? mh[tid] : -INFINITY, (ok1 && ok2) ? lh[tid] : 0.f);

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Merges the five splits of one query: O = sum_s 2^(m_s - M) O_s / L.
__global__ void __launch_bounds__(256) attn_combine_kernel(const float* __restrict__ part,
                                                           const float2* __restrict__ stats,
                                                           int out_dtype, void* __restrict__ out,
                                                           float* __restrict__ lse) {
  const int q = blockIdx.x;
  const int h = blockIdx.y;
  const int tid = threadIdx.x;
  float m[kSplits], l[kSplits];
  float M = -INFINITY;
#pragma unroll
  for (int s = 0; s < kSplits; ++s) {
    const float2 st = stats[(static_cast<int64_t>(q) * kSplits + s) * 64 + h];
    m[s] = st.x;
    l[s] = st.y;
    M = fmaxf(M, st.x);
  }
  float wsum = 0.f, f[kSplits];
#pragma unroll
  for (int s = 0; s < kSplits; ++s) {
    f[s] = (m[s] == -INFINITY) ? 0.f : exp2f(m[s] - M);
    wsum += f[s] * l[s];
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  for (int d = tid; d < 512; d += 256) {
    float acc = 0.f;
#pragma unroll
    for (int s = 0; s < kSplits; ++s)
      acc += f[s] * part[((static_cast<int64_t>(q) * kSplits + s) * 64 + h) * 512 + d];
    const float o = acc * inv;
    const int64_t oi = (static_cast<int64_t>(q) * 64 + h) * 512 + d;
    if (out_dtype == CSA2_OUT_F32) static_cast<float*>(out)[oi] = o;
    else static_cast<__nv_bfloat16*>(out)[oi] = __float2bfloat16_rn(o);
  }
  if (tid == 0 && lse)
    lse[static_cast<int64_t>(q) * 64 + h] = wsum > 0.f ? (M + log2f(wsum)) * 0.6931471805599453f : -INFINITY;
}

}  // namespace

cudaError_t status_attn(cudaStream_t stream, int* code, int* where, bool clear) {
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

size_t attn_workspace_bytes(int64_t queries) {
  const size_t part = static_cast<size_t>(queries) * kSplits * 64 * 512 * sizeof(float);
  const size_t stats = static_cast<size_t>(queries) * kSplits * 64 * sizeof(float2);
  return ((part + 255) & ~size_t(255)) + ((stats + 255) & ~size_t(255));
}

cudaError_t launch_sparse_attn(const void* q, const int32_t* topk, const int64_t* seq_len, int B,
                               int n_q, const int32_t* block_table, int max_pages,
                               int64_t n_pages, const uint8_t* main_pages, const uint8_t* rings,
                               const int32_t* ring_idx, int64_t n_rings, float softmax_scale,
                               int out_dtype, void* out, float* lse, void* ws,
                               cudaStream_t stream) {
  const int64_t Q = static_cast<int64_t>(B) * n_q;
  if (Q == 0) return cudaSuccess;
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev] = true;
  }
  AttnParams p{};
  p.q = static_cast<const uint16_t*>(q);
  p.topk = topk;
  p.seq_len = seq_len;
  p.B = B;
  p.n_q = n_q;
  p.block_table = block_table;
  p.max_pages = max_pages;
  p.n_pages = n_pages;
  p.main_pages = main_pages;
  p.rings = rings;
  p.ring_idx = ring_idx;
  p.n_rings = n_rings;
  p.scale_log2 = softmax_scale * kLog2e;
  const size_t part_bytes = static_cast<size_t>(Q) * kSplits * 64 * 512 * sizeof(float);
  p.part = static_cast<float*>(ws);
  p.stats = reinterpret_cast<float2*>(static_cast<uint8_t*>(ws) + ((part_bytes + 255) & ~size_t(255)));
  attn_split_kernel<<<dim3(kSplits, static_cast<unsigned>(Q)), kThreads, kSmemBytes, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_combine_kernel<<<dim3(static_cast<unsigned>(Q), 64), 256, 0, stream>>>(p.part, p.stats, out_dtype, out, lse);
  return cudaGetLastError();
}

}  // namespace csa2
