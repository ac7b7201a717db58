// MXFP4 append of new main-KV latents and indexer keys into their pages, FP8
// append of new sliding-window entries into their rings, and the standalone
// codec kernels. "DeepSeek V4.1: model architecture and system design, a close
// reading" section 2.3 and "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache
// Compression" section 3.6 (E2M1 + one E4M3 scale per 16 channels, quantised
// after RoPE; sliding-window KV kept in FP8). Latency-bound at decode: one warp
// per new entry, one 16-channel block per lane.
#include "formats.cuh"
#include "kernels.h"
#include "sm103.cuh"

namespace csa2 {
namespace {

constexpr int kMainPageBytes = 128 * 288;
constexpr int kIdxPageBytes = 16 * 576;

__global__ void __launch_bounds__(256) append_kv_kernel(
    const uint16_t* __restrict__ latent, const uint16_t* __restrict__ idx_key,
    const int32_t* __restrict__ seq_idx, const int64_t* __restrict__ pos, int T,
    const int32_t* __restrict__ block_table, int B, int max_pages, int64_t n_pages,
    uint8_t* __restrict__ main_pages, uint8_t* __restrict__ idx_pages) {
  griddep_wait();
  griddep_launch();
  const int tok = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (tok >= T) return;
  // The entry's values do not depend on where it goes: load them first, so
  // their latency overlaps the position and page lookups.
  const uint4* lsrc = reinterpret_cast<const uint4*>(latent + static_cast<int64_t>(tok) * 512) + 2 * lane;
  const uint4 l0 = lsrc[0], l1 = lsrc[1];
  uint4 k0 = make_uint4(0, 0, 0, 0), k1 = k0;
  if (lane < 8) {
    const uint4* ksrc = reinterpret_cast<const uint4*>(idx_key + static_cast<int64_t>(tok) * 128) + 2 * lane;
    k0 = ksrc[0];
    k1 = ksrc[1];
  }
  const int b = seq_idx[tok];
  const int64_t p = pos[tok];
  if (b < 0 || b >= B || p < 0 || (p >> 7) >= max_pages) {
    if (lane == 0) report(CSA2_ERR_DEVICE_BOUNDS, 101);
    return;
  }
  const int32_t page = block_table[static_cast<int64_t>(b) * max_pages + (p >> 7)];
  if (page < 0 || page >= n_pages) {
    if (lane == 0) report(CSA2_ERR_DEVICE_BOUNDS, 102);
    return;
  }
  const int slot = static_cast<int>(p & 127);

  // Main latent: lane -> channels 16*lane .. 16*lane+15.
  {
    float v[16];
    bf16x8_to_f32(l0, v);
    bf16x8_to_f32(l1, v + 8);
    uint8_t sc;
    uint32_t lo, hi;
    mxfp4_block(v, sc, lo, hi);
    uint8_t* e = main_pages + static_cast<int64_t>(page) * kMainPageBytes + slot * 288;
    *reinterpret_cast<uint2*>(e + 8 * lane) = make_uint2(lo, hi);
    e[256 + lane] = sc;
  }
  // Indexer key: lanes 0..7 -> channel blocks 0..7.
  if (lane < 8) {
    float v[16];
    bf16x8_to_f32(k0, v);
    bf16x8_to_f32(k1, v + 8);
    uint8_t sc;
    uint32_t lo, hi;
    mxfp4_block(v, sc, lo, hi);
    const int row = slot & 7;
    uint8_t* g = idx_pages + static_cast<int64_t>(page) * kIdxPageBytes + (slot >> 3) * 576;
    *reinterpret_cast<uint2*>(g + (lane >> 1) * 128 + row * 16 + (lane & 1) * 8) = make_uint2(lo, hi);
    g[512 + row * 8 + lane] = sc;
  }
}

__global__ void __launch_bounds__(256) append_swa_kernel(const uint16_t* __restrict__ x,
                                                         const int32_t* __restrict__ ring_idx,
                                                         const int64_t* __restrict__ pos, int T,
                                                         int64_t n_rings,
                                                         uint8_t* __restrict__ rings) {
  griddep_wait();
  griddep_launch();
  const int tok = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (tok >= T) return;
  // ring_idx == NULL: entry tok goes to row tok of a plain [T, 512] array
  // (a prefill chunk's own window entries).
  int64_t row = tok;
  if (ring_idx) {
    const int r = ring_idx[tok];
    const int64_t p = pos[tok];
    if (r < 0 || r >= n_rings || p < 0) {
      if (lane == 0) report(CSA2_ERR_DEVICE_BOUNDS, 111);
      return;
    }
    row = static_cast<int64_t>(r) * 128 + (p & 127);
  }
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(tok) * 512) + 2 * lane;
  float v[16];
  bf16x8_to_f32(src[0], v);
  bf16x8_to_f32(src[1], v + 8);
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w[i] = static_cast<uint32_t>(e4m3x2_from_f32(v[4 * i], v[4 * i + 1])) |
           (static_cast<uint32_t>(e4m3x2_from_f32(v[4 * i + 2], v[4 * i + 3])) << 16);
  uint8_t* dst = rings + row * 512 + 16 * lane;
  *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
}

// Ring refill: entries [B][n][512] (E4M3) hold positions seq_len[b] - n ..
// seq_len[b] - 1; the last min(n, 128) of them go to slot position % 128 of
// their sequence's ring. One warp per entry, 16 bytes per lane.
__global__ void __launch_bounds__(256) ring_refill_kernel(const uint8_t* __restrict__ entries,
                                                          const int64_t* __restrict__ seq_len, int n,
                                                          const int32_t* __restrict__ ring_idx,
                                                          int64_t n_rings, uint8_t* __restrict__ rings) {
  griddep_wait();
  griddep_launch();
  const int b = blockIdx.y;
  const int m = n < 128 ? n : 128;
  const int k = blockIdx.x * 8 + (threadIdx.x >> 5);  // k-th of the last m entries
  const int lane = threadIdx.x & 31;
  if (k >= m) return;
  const int i = n - m + k;
  const int64_t p = seq_len[b] - n + i;
  const int r = ring_idx[b];
  if (r < 0 || r >= n_rings || p < 0) {
    if (lane == 0) report(CSA2_ERR_DEVICE_BOUNDS, 112);
    return;
  }
  const uint4 v = reinterpret_cast<const uint4*>(entries + (static_cast<int64_t>(b) * n + i) * 512)[lane];
  reinterpret_cast<uint4*>(rings + (static_cast<int64_t>(r) * 128 + (p & 127)) * 512)[lane] = v;
}

__global__ void quant_mxfp4_kernel(const uint16_t* __restrict__ x, int64_t nblocks,
                                   uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  griddep_wait();
  griddep_launch();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= nblocks) return;
  const uint4* src = reinterpret_cast<const uint4*>(x + 16 * i);
  float v[16];
  bf16x8_to_f32(src[0], v);
  bf16x8_to_f32(src[1], v + 8);
  uint8_t sc;
  uint32_t lo, hi;
  mxfp4_block(v, sc, lo, hi);
  *reinterpret_cast<uint2*>(codes + 8 * i) = make_uint2(lo, hi);
  scales[i] = sc;
}

__global__ void dequant_mxfp4_kernel(const uint8_t* __restrict__ codes,
                                     const uint8_t* __restrict__ scales, int64_t nblocks,
                                     float* __restrict__ out) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= nblocks) return;
  const uint2 c = *reinterpret_cast<const uint2*>(codes + 8 * i);
  const float sf = e4m3_to_f32(scales[i]);
  const uint32_t w[2] = {c.x, c.y};
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t h2 = e2m1x2_to_f16x2((w[k >> 2] >> (8 * (k & 3))) & 0xFFu);
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
    out[16 * i + 2 * k] = f.x * sf;
    out[16 * i + 2 * k + 1] = f.y * sf;
  }
}

__global__ void quant_fp8_kernel(const float* __restrict__ x, int64_t n, uint8_t* __restrict__ out) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) out[i] = e4m3_from_f32(x[i]);
}

}  // namespace

cudaError_t status_append(cudaStream_t stream, int* code, int* where, bool clear) {
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

cudaError_t launch_append_kv(const void* latent, const void* idx_key, const int32_t* seq_idx,
                             const int64_t* pos, int T, const int32_t* block_table, int B,
                             int max_pages, int64_t n_pages, uint8_t* main_pages,
                             uint8_t* idx_pages, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  return launch_pdl(append_kv_kernel, dim3((T + 7) / 8), dim3(256), 0, stream, 0,
                    static_cast<const uint16_t*>(latent), static_cast<const uint16_t*>(idx_key), seq_idx, pos, T,
                    block_table, B, max_pages, n_pages, main_pages, idx_pages);
}

cudaError_t launch_append_swa(const void* x, const int32_t* ring_idx, const int64_t* pos, int T,
                              int64_t n_rings, uint8_t* rings, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  return launch_pdl(append_swa_kernel, dim3((T + 7) / 8), dim3(256), 0, stream, 0,
                    static_cast<const uint16_t*>(x), ring_idx, pos, T, n_rings, rings);
}

cudaError_t launch_ring_refill(const uint8_t* entries, const int64_t* seq_len, int B, int n,
                               const int32_t* ring_idx, int64_t n_rings, uint8_t* rings, cudaStream_t stream) {
  if (B == 0 || n == 0) return cudaSuccess;
  const int m = n < 128 ? n : 128;
  return launch_pdl(ring_refill_kernel, dim3((m + 7) / 8, B), dim3(256), 0, stream, 0, entries, seq_len, n,
                    ring_idx, n_rings, rings);
}

cudaError_t launch_quant_mxfp4(const void* x, int64_t n, uint8_t* codes, uint8_t* scales,
                               cudaStream_t stream) {
  const int64_t nb = n / 16;
  if (nb == 0) return cudaSuccess;
  return launch_pdl(quant_mxfp4_kernel, dim3(static_cast<unsigned>((nb + 255) / 256)), dim3(256), 0, stream, 0,
                    static_cast<const uint16_t*>(x), nb, codes, scales);
}

cudaError_t launch_dequant_mxfp4(const uint8_t* codes, const uint8_t* scales, int64_t n,
                                 float* out, cudaStream_t stream) {
  const int64_t nb = n / 16;
  if (nb == 0) return cudaSuccess;
  dequant_mxfp4_kernel<<<static_cast<unsigned>((nb + 255) / 256), 256, 0, stream>>>(codes, scales,
                                                                                     nb, out);
  return cudaGetLastError();
}

cudaError_t launch_quant_fp8(const float* x, int64_t n, uint8_t* out, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  quant_fp8_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(x, n, out);
  return cudaGetLastError();
}

}  // namespace csa2
