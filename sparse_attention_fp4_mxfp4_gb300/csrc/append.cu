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
constexpr int kTailRow = 512 + 512 + 128 + 128;  // bf16 per pending token: kv, kv logits, key, key logits

// One 16-channel block of an entry into its page: the main latent block of
// lane `lane` and, for lanes 0-7, the indexer-key block.
__device__ __forceinline__ void store_entry(uint8_t* __restrict__ main_pages, uint8_t* __restrict__ idx_pages,
                                            int32_t page, int slot, int lane, const float (&lat)[16],
                                            const float (&key)[16]) {
  uint8_t sc;
  uint32_t lo, hi;
  mxfp4_block(lat, sc, lo, hi);
  uint8_t* e = main_pages + static_cast<int64_t>(page) * kMainPageBytes + slot * 288;
  *reinterpret_cast<uint2*>(e + 8 * lane) = make_uint2(lo, hi);
  e[256 + lane] = sc;
  if (lane < 8) {
    mxfp4_block(key, sc, lo, hi);
    const int row = slot & 7;
    uint8_t* g = idx_pages + static_cast<int64_t>(page) * kIdxPageBytes + (slot >> 3) * 576;
    *reinterpret_cast<uint2*>(g + (lane >> 1) * 128 + row * 16 + (lane & 1) * 8) = make_uint2(lo, hi);
    g[512 + row * 8 + lane] = sc;
  }
}

// fp64 -> bf16, nearest with ties to even, from the double's bits in one step.
__device__ __forceinline__ uint16_t bf16_from_f64(double d) {
  const uint64_t u = static_cast<uint64_t>(__double_as_longlong(d));
  const uint32_t sign = static_cast<uint32_t>(u >> 63) << 15;
  const int ex = static_cast<int>((u >> 52) & 0x7FF);
  if (ex == 0) return static_cast<uint16_t>(sign);  // zero or far below bf16's range
  const uint64_t m = (u & ((uint64_t(1) << 52) - 1)) | (uint64_t(1) << 52);  // 53 significant bits
  int e8 = ex - 1023 + 127;
  // Normal bf16 keeps 8 significant bits; below 2^-126 the quantum is 2^-133.
  const int drop = e8 >= 1 ? 45 : 45 + (1 - e8);
  if (drop > 54) return static_cast<uint16_t>(sign);
  uint64_t q = m >> drop;
  const uint64_t rem = m & ((uint64_t(1) << drop) - 1), half = uint64_t(1) << (drop - 1);
  if (rem > half || (rem == half && (q & 1))) ++q;
  if (e8 < 1) return static_cast<uint16_t>(sign | static_cast<uint32_t>(q));  // q = 128 is the smallest normal
  if (q == (uint64_t(1) << 8)) {
    q >>= 1;
    ++e8;
  }
  if (e8 >= 255) return static_cast<uint16_t>(sign | 0x7F80u);
  return static_cast<uint16_t>(sign | (static_cast<uint32_t>(e8) << 7) | static_cast<uint32_t>(q & 0x7F));
}

// Entry of ratio m: per channel, the softmax of the m tokens' logits weights
// their candidates (fp64), rounded once to bf16, returned as fp32.
template <int kM>
__device__ __forceinline__ void compress16(const float (&x)[kM][16], const float (&z)[kM][16], float (&out)[16]) {
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    double zmax = z[0][c];
#pragma unroll
    for (int i = 1; i < kM; ++i) zmax = fmax(zmax, static_cast<double>(z[i][c]));
    double num = 0.0, den = 0.0;
#pragma unroll
    for (int i = 0; i < kM; ++i) {
      const double w = exp(static_cast<double>(z[i][c]) - zmax);
      num += w * static_cast<double>(x[i][c]);
      den += w;
    }
    out[c] = __uint_as_float(static_cast<uint32_t>(bf16_from_f64(num / den)) << 16);
  }
}

// Encoder-side append at ratio kM: the warp of a token at position p with
// p % kM == kM - 1 builds entry p / kM from its kM tokens (earlier ones from
// this call when they are the rows just before it, else from the sequence's
// tail state) and stores it; other tokens do nothing here.
template <int kM>
__global__ void __launch_bounds__(256) compress_append_kernel(
    const uint16_t* __restrict__ kv, const uint16_t* __restrict__ kv_gate, const uint16_t* __restrict__ idx_key,
    const uint16_t* __restrict__ idx_gate, const int32_t* __restrict__ seq_idx, const int64_t* __restrict__ pos,
    int T, const uint16_t* __restrict__ tail, const int32_t* __restrict__ block_table, int B, int max_pages,
    int64_t n_pages, uint8_t* __restrict__ main_pages, uint8_t* __restrict__ idx_pages) {
  griddep_wait();
  griddep_launch();
  const int tok = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (tok >= T) return;
  const int b = seq_idx[tok];
  const int64_t p = pos[tok];
  if (b < 0 || b >= B || p < 0) {
    if (lane == 0) report(CSA2_ERR_DEVICE_BOUNDS, 121);
    return;
  }
  if (p % kM != kM - 1) return;
  const int64_t e = p / kM;
  if ((e >> 7) >= max_pages) {
    if (lane == 0) report(CSA2_ERR_DEVICE_BOUNDS, 122);
    return;
  }
  const int32_t page = block_table[static_cast<int64_t>(b) * max_pages + (e >> 7)];
  if (page < 0 || page >= n_pages) {
    if (lane == 0) report(CSA2_ERR_DEVICE_BOUNDS, 123);
    return;
  }
  float x[kM][16], z[kM][16], kx[kM][16], kz[kM][16];
#pragma unroll
  for (int i = 0; i < kM; ++i) {
    // Token m*e + i: row tok - (kM - 1 - i) of this call, or tail slot i.
    const int r = tok - (kM - 1 - i);
    const bool in_call = i == kM - 1 || (r >= 0 && seq_idx[r] == b && pos[r] == p - (kM - 1 - i));
    const uint16_t *xs, *zs, *ks, *kzs;
    if (in_call) {
      xs = kv + static_cast<int64_t>(r) * 512;
      zs = kv_gate + static_cast<int64_t>(r) * 512;
      ks = idx_key + static_cast<int64_t>(r) * 128;
      kzs = idx_gate + static_cast<int64_t>(r) * 128;
    } else {
      const uint16_t* row = tail + (static_cast<int64_t>(b) * (kM - 1) + i) * kTailRow;
      xs = row;
      zs = row + 512;
      ks = row + 1024;
      kzs = row + 1152;
    }
    const uint4* xv = reinterpret_cast<const uint4*>(xs) + 2 * lane;
    const uint4* zv = reinterpret_cast<const uint4*>(zs) + 2 * lane;
    bf16x8_to_f32(xv[0], x[i]);
    bf16x8_to_f32(xv[1], x[i] + 8);
    bf16x8_to_f32(zv[0], z[i]);
    bf16x8_to_f32(zv[1], z[i] + 8);
    if (lane < 8) {
      const uint4* kv4 = reinterpret_cast<const uint4*>(ks) + 2 * lane;
      const uint4* kz4 = reinterpret_cast<const uint4*>(kzs) + 2 * lane;
      bf16x8_to_f32(kv4[0], kx[i]);
      bf16x8_to_f32(kv4[1], kx[i] + 8);
      bf16x8_to_f32(kz4[0], kz[i]);
      bf16x8_to_f32(kz4[1], kz[i] + 8);
    } else {
#pragma unroll
      for (int c = 0; c < 16; ++c) kx[i][c] = kz[i][c] = 0.f;
    }
  }
  float lat[16], key[16];
  compress16<kM>(x, z, lat);
  compress16<kM>(kx, kz, key);
  store_entry(main_pages, idx_pages, page, static_cast<int>(e & 127), lane, lat, key);
}

// After compress_append_kernel: a token whose entry is not completed within
// this call (its completing token is not among the rows after it) goes to
// tail slot p % kM of its sequence.
template <int kM>
__global__ void __launch_bounds__(256) compress_tail_kernel(
    const uint16_t* __restrict__ kv, const uint16_t* __restrict__ kv_gate, const uint16_t* __restrict__ idx_key,
    const uint16_t* __restrict__ idx_gate, const int32_t* __restrict__ seq_idx, const int64_t* __restrict__ pos,
    int T, int B, uint16_t* __restrict__ tail) {
  griddep_wait();
  griddep_launch();
  const int tok = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (tok >= T) return;
  const int b = seq_idx[tok];
  const int64_t p = pos[tok];
  if (b < 0 || b >= B || p < 0 || p % kM == kM - 1) return;
  const int d = static_cast<int>(kM - 1 - p % kM);
  const int r = tok + d;
  if (r < T && seq_idx[r] == b && pos[r] == p + d) return;  // completed in this call
  uint16_t* row = tail + (static_cast<int64_t>(b) * (kM - 1) + p % kM) * kTailRow;
  // 1280 bf16 = 160 x 16 B: lane copies chunks lane, lane + 32, ...
  for (int c = lane; c < kTailRow / 8; c += 32) {
    const uint16_t* src;
    int off;
    if (c < 64) { src = kv; off = c; }
    else if (c < 128) { src = kv_gate; off = c - 64; }
    else if (c < 144) { src = idx_key; off = c - 128; }
    else { src = idx_gate; off = c - 144; }
    const int width = c < 128 ? 512 : 128;
    reinterpret_cast<uint4*>(row)[c] =
        reinterpret_cast<const uint4*>(src + static_cast<int64_t>(tok) * width)[off];
  }
}


// Entry tok of an MXFP4 append, by the 32 lanes of one warp.
__device__ __forceinline__ void append_kv_entry(
    int tok, int lane, const uint16_t* __restrict__ latent, const uint16_t* __restrict__ idx_key,
    const int32_t* __restrict__ seq_idx, const int64_t* __restrict__ pos,
    const int32_t* __restrict__ block_table, int B, int max_pages, int64_t n_pages,
    uint8_t* __restrict__ main_pages, uint8_t* __restrict__ idx_pages) {
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

__global__ void __launch_bounds__(256) append_kv_kernel(
    const uint16_t* __restrict__ latent, const uint16_t* __restrict__ idx_key,
    const int32_t* __restrict__ seq_idx, const int64_t* __restrict__ pos, int T,
    const int32_t* __restrict__ block_table, int B, int max_pages, int64_t n_pages,
    uint8_t* __restrict__ main_pages, uint8_t* __restrict__ idx_pages) {
  griddep_wait();
  griddep_launch();
  const int tok = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (tok >= T) return;
  append_kv_entry(tok, threadIdx.x & 31, latent, idx_key, seq_idx, pos, block_table, B, max_pages, n_pages,
                  main_pages, idx_pages);
}

// Window entry tok (E4M3), by the 32 lanes of one warp.
__device__ __forceinline__ void append_swa_entry(int tok, int lane, const uint16_t* __restrict__ x,
                                                 const int32_t* __restrict__ ring_idx,
                                                 const int64_t* __restrict__ pos, int64_t n_rings,
                                                 uint8_t* __restrict__ rings) {
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

__global__ void __launch_bounds__(256) append_swa_kernel(const uint16_t* __restrict__ x,
                                                         const int32_t* __restrict__ ring_idx,
                                                         const int64_t* __restrict__ pos, int T,
                                                         int64_t n_rings,
                                                         uint8_t* __restrict__ rings) {
  griddep_wait();
  griddep_launch();
  const int tok = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (tok >= T) return;
  append_swa_entry(tok, threadIdx.x & 31, x, ring_idx, pos, n_rings, rings);
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

// 16-value block i of an MXFP4 quantisation.
__device__ __forceinline__ void quant_mxfp4_block(int64_t i, const uint16_t* __restrict__ x,
                                                  uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
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

__global__ void quant_mxfp4_kernel(const uint16_t* __restrict__ x, int64_t nblocks,
                                   uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  griddep_wait();
  griddep_launch();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= nblocks) return;
  quant_mxfp4_block(i, x, codes, scales);
}

// A decode step's appends and indexer-query quantisations in one launch
// (the same work as append_kv_kernel, then append_swa_kernel per layer, then
// quant_mxfp4_kernel per indexed layer; they touch disjoint memory). Block
// ranges: [0, kv_blocks) append entries, 8 per block; then per layer its
// window entries (8 per block) and its query's 16-value blocks (256 per block).
__global__ void __launch_bounds__(256) decode_appends_kernel(const DecodeAppends P) {
  griddep_wait();
  griddep_launch();
  const int tid = threadIdx.x, lane = tid & 31;
  int blk = blockIdx.x;
  if (blk < P.kv_blocks) {
    const int tok = blk * 8 + (tid >> 5);
    if (tok < P.T)
      append_kv_entry(tok, lane, static_cast<const uint16_t*>(P.latent), static_cast<const uint16_t*>(P.idx_key),
                      P.seq_idx, P.pos, P.block_table, P.B, P.max_pages, P.n_pages, P.main_pages, P.idx_pages);
    return;
  }
  blk -= P.kv_blocks;
  for (int l = 0; l < P.n_layers; ++l) {
    const DecodeAppendsLayer& L = P.layer[l];
    const int swa_blocks = L.swa ? (P.T + 7) / 8 : 0;
    if (blk < swa_blocks) {
      const int tok = blk * 8 + (tid >> 5);
      if (tok < P.T)
        append_swa_entry(tok, lane, static_cast<const uint16_t*>(L.swa), L.ring_idx, P.pos, L.n_rings, L.rings);
      return;
    }
    blk -= swa_blocks;
    const int64_t qb = L.q_idx ? L.q_n / 16 : 0;
    const int q_blocks = static_cast<int>((qb + 255) / 256);
    if (blk < q_blocks) {
      const int64_t i = static_cast<int64_t>(blk) * 256 + tid;
      if (i < qb) quant_mxfp4_block(i, static_cast<const uint16_t*>(L.q_idx), L.q_codes, L.q_scales);
      return;
    }
    blk -= q_blocks;
  }
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

cudaError_t force_timeout_append(int site, cudaStream_t stream) { return set_force_timeout_site(site, stream); }

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

cudaError_t launch_decode_appends(const DecodeAppends& P, cudaStream_t stream) {
  DecodeAppends p = P;
  p.kv_blocks = (p.T + 7) / 8;
  int64_t blocks = p.kv_blocks;
  for (int l = 0; l < p.n_layers; ++l) {
    if (p.layer[l].swa) blocks += (p.T + 7) / 8;
    if (p.layer[l].q_idx) blocks += (p.layer[l].q_n / 16 + 255) / 256;
  }
  if (blocks == 0) return cudaSuccess;
  return launch_pdl(decode_appends_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, 0, p);
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

template <int kM>
cudaError_t launch_compress_m(const void* kv, const void* kv_gate, const void* idx_key, const void* idx_gate,
                              const int32_t* seq_idx, const int64_t* pos, int T, void* tail,
                              const int32_t* block_table, int B, int max_pages, int64_t n_pages,
                              uint8_t* main_pages, uint8_t* idx_pages, cudaStream_t stream) {
  const dim3 grid((T + 7) / 8);
  cudaError_t e = launch_pdl(compress_append_kernel<kM>, grid, dim3(256), 0, stream, 0,
                             static_cast<const uint16_t*>(kv), static_cast<const uint16_t*>(kv_gate),
                             static_cast<const uint16_t*>(idx_key), static_cast<const uint16_t*>(idx_gate), seq_idx,
                             pos, T, static_cast<const uint16_t*>(tail), block_table, B, max_pages, n_pages,
                             main_pages, idx_pages);
  if (e != cudaSuccess || kM == 1) return e;
  return launch_pdl(compress_tail_kernel<kM>, grid, dim3(256), 0, stream, 0, static_cast<const uint16_t*>(kv),
                    static_cast<const uint16_t*>(kv_gate), static_cast<const uint16_t*>(idx_key),
                    static_cast<const uint16_t*>(idx_gate), seq_idx, pos, T, B, static_cast<uint16_t*>(tail));
}

cudaError_t launch_compress_append(const void* kv, const void* kv_gate, const void* idx_key, const void* idx_gate,
                                   const int32_t* seq_idx, const int64_t* pos, int T, int m, void* tail,
                                   const int32_t* block_table, int B, int max_pages, int64_t n_pages,
                                   uint8_t* main_pages, uint8_t* idx_pages, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  switch (m) {
    case 1: return launch_compress_m<1>(kv, kv_gate, idx_key, idx_gate, seq_idx, pos, T, tail, block_table, B,
                                        max_pages, n_pages, main_pages, idx_pages, stream);
    case 2: return launch_compress_m<2>(kv, kv_gate, idx_key, idx_gate, seq_idx, pos, T, tail, block_table, B,
                                        max_pages, n_pages, main_pages, idx_pages, stream);
    default: return cudaErrorInvalidValue;
  }
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
