// Reuse-mode sparse attention ("DeepSeek V4.1: model architecture and system
// design, a close reading" sections 1 and 2.2; "DeepSeek-V4.1-Flash: Pushing
// the Limits of KV Cache Compression" sections 3.3 and 3.6; "DeepSeek-V4 model
// structure (7): structure decides the system", closing summary): 64 query
// heads attend, with K = V = the 512-channel latent, to the query's top-k
// main entries (MXFP4, dequantised before attention) and to its FP8
// sliding-window entries.
//
// A query's 640 key slots form five chunks of 128 (four of top-k entries, one
// of window entries). A CTA takes a run of consecutive chunks of one query
// (all five when there are enough queries to fill the GPU, otherwise the
// chunks are split over up to five CTAs whose partial results a second kernel
// merges) and walks them with an online softmax:
//   S^T[128 keys x 64 heads] = K Q^T    (tcgen05, M = 128, N = 64, K = 512)
//   softmax of the chunk against a running per-head stabiliser, P^T in f16
//   O^T[512 dims x 64 heads] += V^T P^T (tcgen05, 4 x M = 128, N = 64, K = 128)
// V^T is the key tile itself read as an MN-major operand; O^T stays in TMEM
// across chunks. Roles: warps 8-15 gather the next chunk's stored keys into
// registers while the current chunk is on the tensor cores, then dequantise
// them (exactly) to f16 into the 128-byte-swizzled key tile, one half of the
// dimensions at a time, so that the next chunk's first half is written while
// the tensor cores still read the second half for the current one; warps 0-7
// own the softmax (S^T row = key, 32 heads per warp) and the output, and their
// thread 0 issues the MMAs.
//
// The stabiliser is only raised when a chunk's logit exceeds it by more than
// 8 (log2 units), as in lazy-rescaling flash attention: p = 2^(l - m) <= 256
// stays exact enough in f16, and O^T and the running sums are rescaled only on
// those (rare) raises. The result is the same softmax either way.
#include <algorithm>

#include "formats.cuh"
#include "kernels.h"
#include "sm103.cuh"

namespace csa2 {
namespace {

constexpr int kChunks = 5;  // four top-k chunks of 128 entries, one window chunk
constexpr int kSxWarps = 8;
constexpr int kGdWarps = 8;
constexpr int kGdThreads = kGdWarps * 32;
constexpr int kSxThreads = kSxWarps * 32;
constexpr int kThreads = kSxThreads + kGdThreads;
constexpr int kKtOff = 0;                // 128 keys x 512 f16: 8 K-blocks of 16 KB
constexpr int kQsOff = 131072;           // 64 heads x 512 f16: 8 K-blocks of 8 KB
constexpr int kPtOff = 196608;           // P^T, MN-major: 128 keys x 64 heads f16
constexpr int kMiscOff = kPtOff + 16384;  // barriers, key offsets, per-head state
constexpr int kSmemBytes = 1024 + kMiscOff + 4096;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazy = 8.f;  // headroom (log2 units) before the stabiliser is raised
constexpr int kBarGd = 1, kBarSxOr = 2, kBarSx = 3;  // named barriers
constexpr int64_t kChunkSrc = int64_t(1) << 62;     // key offset tag: the call's own window entries
// Tokens from which a query's chunks are never split over several CTAs (so no
// partial-output workspace is needed), whatever the SM count.
constexpr int64_t kNoSplitQueries = 256;

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
  // Prefill: FP8 window entries of the call's own positions N-n_q .. N-1,
  // [B][n_q][512]; the rings then hold the positions before them. NULL:
  // decode, every window entry comes from the ring.
  const uint8_t* swa_chunk;
  int m_shift;        // log2 of the tokens per entry: top-k entries of token t are < (t + 1) >> m_shift
  float scale_log2;   // softmax_scale * log2(e)
  int nsplit;         // CTAs per query (1..5)
  int out_dtype;
  void* out;          // final output (nsplit == 1)
  float* lse;
  float* part;        // [Q][5][64][512] unnormalised partial outputs (nsplit > 1)
  float2* stats;      // [Q][5][64] (stabiliser in log2 units, sum)
};

// 32 values per lane -> lane L holds op over the warp of entry L. Each step
// halves the range a lane keeps (the upper half when the lane's bit for that
// step is set) and combines it with the partner's copy of that half.
template <class Op>
__device__ __forceinline__ void warp_reduce_scatter32(float (&v)[32], int lane, Op op) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool up = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = up ? v[i] : v[i + w];
      const float keep = up ? v[i + w] : v[i];
      v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, w));
    }
  }
}

// cos and sin of -t * theta_i, theta_i = 10000^(-2i/64) (output de-rotation).
// The angle is formed and reduced to [-pi, pi] in double precision (t * theta
// reaches 1e9 rad), then evaluated in single precision.
__device__ __forceinline__ void derotate_cs(int64_t t, int i, float& c, float& s) {
  const double theta = exp2(-static_cast<double>(i) * (13.287712379549449 / 32.0));  // log2(10000) = 13.2877...
  double a = -static_cast<double>(t) * theta;
  a -= 6.283185307179586 * rint(a * 0.15915494309189535);
  sincosf(static_cast<float>(a), &s, &c);
}

// Rotates this lane's value x of output channel d (pairs (448 + 2i, 449 + 2i))
// by -t * theta_i, given its partner lane's value y (lane ^ 1 holds channel d ^ 1).
__device__ __forceinline__ float derotate_value(float x, float y, int d, float c, float s) {
  return (d & 1) ? (y * s + x * c) : (x * c - y * s);
}

__global__ void __launch_bounds__(kThreads, 1) attn_kernel(const AttnParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Kt = smem + kKtOff;
  uint8_t* Qs = smem + kQsOff;
  uint8_t* Pt = smem + kPtOff;
  uint8_t* misc = smem + kMiscOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 64);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 68);
  int64_t* key_off = reinterpret_cast<int64_t*>(misc + 128);  // [2][128] byte offsets, -1 = none
  float* mst = reinterpret_cast<float*>(misc + 2176);         // [64] running stabiliser (log2)
  float* fac = reinterpret_cast<float*>(misc + 2432);         // [64] rescale factors
  float* lsum = reinterpret_cast<float*>(misc + 2688);        // [64] sums, then their inverses
  float* red = reinterpret_cast<float*>(misc + 2944);         // [4][64] per-lane-quarter partials
  // Key tile halves: "lo" = dimensions 0-255 (K-blocks 0-3), "hi" = 256-511.
  const uint32_t kfull_lo = smem_u32(&bars[0]), kfull_hi = smem_u32(&bars[1]);
  const uint32_t kfree_lo = smem_u32(&bars[2]), kfree_hi = smem_u32(&bars[3]);
  const uint32_t sfull = smem_u32(&bars[4]), drain = smem_u32(&bars[5]);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(kfull_lo, kGdThreads);
    mbar_init(kfull_hi, kGdThreads);
    mbar_init(kfree_lo, 1);
    mbar_init(kfree_hi, 1);
    mbar_init(sfull, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (tid < 64) {
    mst[tid] = -INFINITY;
    lsum[tid] = 0.f;
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), 512);
  griddep_wait();  // everything below may read what earlier kernels wrote
  griddep_launch();
  const int split = blockIdx.x;
  const int q = blockIdx.y;
  const int b = q / P.n_q, jq = q % P.n_q;
  const int64_t N = P.seq_len[b];
  const int64_t t = N - P.n_q + jq;
  const int per = kChunks / P.nsplit, rem = kChunks % P.nsplit;
  const int c0 = split * per + (split < rem ? split : rem);
  const int nc = per + (split < rem ? 1 : 0);

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= kSxWarps) {
    // ============ gather + dequantise (256 threads, two per key) ============
    // Thread (key r, sub) owns dimensions sub*128 .. +127 of each tile half:
    // lo = sub*128 + [0,128), hi = 256 + sub*128 + [0,128).
    const int gt = tid - kSxThreads;
    const int r = gt >> 1, sub = gt & 1;
    auto resolve = [&](int c, int64_t* dst) {  // threads gt < 128: byte offset of key slot gt
      if (gt >= 128) return;
      int64_t off = -1;
      if (c < 4) {
        const int32_t p = P.topk[static_cast<int64_t>(q) * 512 + c * 128 + gt];
        if (p >= 0) {
          if (p > ((t + 1) >> P.m_shift) - 1 || (p >> 7) >= P.max_pages) {
            report(CSA2_ERR_DEVICE_BOUNDS, 401);
          } else {
            const int32_t page = P.block_table[static_cast<int64_t>(b) * P.max_pages + (p >> 7)];
            if (page < 0 || page >= P.n_pages) report(CSA2_ERR_DEVICE_BOUNDS, 402);
            else off = static_cast<int64_t>(page) * (128 * 288) + (p & 127) * 288;
          }
        }
      } else if (!P.swa_chunk) {
        const int32_t ri = P.ring_idx[b];
        const int64_t base = N - 128;  // the ring holds positions N-128 .. N-1
        int64_t d = (static_cast<int64_t>(gt) - base) % 128;
        if (d < 0) d += 128;
        const int64_t p = base + d;  // the position stored in slot gt
        int64_t lo = t - 127;
        if (lo < base) lo = base;
        if (lo < 0) lo = 0;
        if (ri < 0 || ri >= P.n_rings) {
          if (gt == 0) report(CSA2_ERR_DEVICE_BOUNDS, 403);
        } else if (p >= lo && p <= t) {
          off = (static_cast<int64_t>(ri) * 128 + gt) * 512;
        }
      } else {
        // Prefill: key slot gt holds position t - 127 + gt, from the call's
        // own entries when it is one of the new positions, else from the ring
        // (which still holds the 128 positions before them).
        const int64_t p = t - 127 + gt, first_new = N - P.n_q;
        if (p >= 0) {
          if (p >= first_new) {
            off = kChunkSrc | ((static_cast<int64_t>(b) * P.n_q + (p - first_new)) * 512);
          } else {
            const int32_t ri = P.ring_idx[b];
            if (ri < 0 || ri >= P.n_rings) report(CSA2_ERR_DEVICE_BOUNDS, 404);
            else off = (static_cast<int64_t>(ri) * 128 + (p & 127)) * 512;
          }
        }
      }
      dst[gt] = off;
    };
    // Stored bytes of this thread's share of key r. FP4: code bytes
    // [sub*64, +64) and [128 + sub*64, +64), scale bytes [256 + sub*8, +8) and
    // [272 + sub*8, +8). FP8: bytes [sub*128, +128) and [256 + sub*128, +128).
    uint4 raw[16];
    uint2 scl[2];
    auto load = [&](int c, const int64_t* offs) {
      const int64_t off = offs[r];
#pragma unroll
      for (int i = 0; i < 16; ++i) raw[i] = make_uint4(0, 0, 0, 0);
      scl[0] = scl[1] = make_uint2(0, 0);
      if (off < 0) return;
      if (c < 4) {
        const uint8_t* e = P.main_pages + off;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
          for (int i = 0; i < 4; ++i) raw[4 * hf + i] = reinterpret_cast<const uint4*>(e + hf * 128 + sub * 64)[i];
          scl[hf] = *reinterpret_cast<const uint2*>(e + 256 + hf * 16 + sub * 8);
        }
      } else {
        const uint8_t* e = (off & kChunkSrc) ? P.swa_chunk + (off & ~kChunkSrc) : P.rings + off;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
          for (int i = 0; i < 8; ++i) raw[8 * hf + i] = reinterpret_cast<const uint4*>(e + hf * 256 + sub * 128)[i];
        }
      }
    };
    auto dequant = [&](int c, int hf) {  // one tile half of this thread's share
      const int d0 = hf * 256 + sub * 128;
      if (c < 4) {
        const uint32_t sw[2] = {scl[hf].x, scl[hf].y};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint4 o[4];
          dequant32_f16(raw[4 * hf + i], static_cast<uint16_t>(sw[i >> 1] >> (16 * (i & 1))), o);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int d = d0 + 32 * i + 8 * k;
            *reinterpret_cast<uint4*>(Kt + (d >> 6) * 16384 + sw128_offset(r, (d & 63) >> 3)) = o[k];
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 v = raw[8 * hf + i];
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
          uint32_t h[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            h[2 * k] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[k] & 0xFFFFu));
            h[2 * k + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[k] >> 16));
          }
          const int d = d0 + 16 * i;
          uint8_t* kb = Kt + (d >> 6) * 16384;
          *reinterpret_cast<uint4*>(kb + sw128_offset(r, (d & 63) >> 3)) = make_uint4(h[0], h[1], h[2], h[3]);
          *reinterpret_cast<uint4*>(kb + sw128_offset(r, ((d & 63) >> 3) + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
        }
      }
    };

    // Q loads first: they depend on nothing and overlap the slot lookups.
    const uint4* qg = reinterpret_cast<const uint4*>(P.q + static_cast<int64_t>(q) * 64 * 512);
    uint4 qv[16];
#pragma unroll
    for (int it = 0; it < 16; ++it) qv[it] = qg[gt + it * kGdThreads];
    resolve(c0, key_off);
#pragma unroll
    for (int it = 0; it < 16; ++it) {  // Q (bf16 -> f16) into the swizzled B operand
      const int i = gt + it * kGdThreads;
      const int h = i >> 6, c = i & 63;
      float f[8];
      bf16x8_to_f32(qv[it], f);
      uint32_t o[4];
      bool bad = false;  // f16 holds |q| < 65520 (65504 after rounding); larger or non-finite q is out of range
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        bad |= !(fabsf(f[2 * k]) < 65520.f) || !(fabsf(f[2 * k + 1]) < 65520.f);
        __half2 hv = __floats2half2_rn(f[2 * k], f[2 * k + 1]);
        o[k] = *reinterpret_cast<uint32_t*>(&hv);
      }
      if (bad) report(CSA2_ERR_DEVICE_RANGE, 405);
      *reinterpret_cast<uint4*>(Qs + (c >> 3) * 8192 + sw128_offset(h, c & 7)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    named_bar_sync(kBarGd, kGdThreads);  // slots of the first chunk are known
    load(c0, key_off);
    for (int jj = 0; jj < nc; ++jj) {
      // A tile half is free once the previous chunk's O^T MMAs that read it are done.
      const bool ok = jj == 0 || mbar_wait(kfree_lo, (jj - 1) & 1, 421, abort_flag);
      if (named_bar_or(kBarGd, kGdThreads, !ok || *abort_flag)) {
        *abort_flag = 1;
        break;
      }
      dequant(c0 + jj, 0);
      fence_proxy_async();
      mbar_arrive(kfull_lo);
      if (jj == 0 || mbar_wait(kfree_hi, (jj - 1) & 1, 422, abort_flag)) {
        dequant(c0 + jj, 1);
        fence_proxy_async();
        mbar_arrive(kfull_hi);
      } else {
        *abort_flag = 1;  // the next check (or the waiting roles) stops everyone
      }
      if (jj + 1 < nc) {
        int64_t* nxt = key_off + ((jj + 1) & 1) * 128;
        resolve(c0 + jj + 1, nxt);
        named_bar_sync(kBarGd, kGdThreads);
        load(c0 + jj + 1, nxt);
      }
    }
  } else {
    // ============ softmax + output (256 threads) ============
    // Warp w: TMEM lane quarter qt = w % 4, heads 32*hh .. +31 with hh = w / 4.
    // In S^T a thread owns key row qt*32 + lane; in O^T dimension row
    // qt*32 + lane of every M tile.
    const int qt = warp & 3, hh = warp >> 2;
    const int row = qt * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(qt * 32) << 16;
    float l[32], acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = 0.f;
    auto load_logits = [&](bool kvalid) {
      uint32_t v[32];
      tmem_ld32(tmem + lane_base + 32 * hh, v);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) l[i] = kvalid ? __uint_as_float(v[i]) * P.scale_log2 : -INFINITY;
    };
    const uint32_t id_s = idesc_f16(128, 64, false, false);
    const uint32_t id_o = idesc_f16(128, 64, true, true);
    const uint32_t kt = smem_u32(Kt), qs = smem_u32(Qs), pt = smem_u32(Pt);
    bool ok = true;
    for (int jj = 0; jj < nc; ++jj) {
      bool got = mbar_wait(kfull_lo, jj & 1, 441, abort_flag);
      if (tid == 0 && got) {  // S^T = K Q^T, a tile half at a time
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          if (hf == 1 && !(got = mbar_wait(kfull_hi, jj & 1, 444, abort_flag))) break;
          tc_fence_after();
#pragma unroll 4
          for (int k = 16 * hf; k < 16 * hf + 16; ++k) {
            const uint64_t ad = sdesc(kt + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024, kSwizzle128B);
            const uint64_t bd = sdesc(qs + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024, kSwizzle128B);
            umma_f16(tmem, ad, bd, id_s, k > 0 ? 1u : 0u);
          }
        }
        if (got) umma_commit(sfull);
      }
      if (!got) *abort_flag = 1;
      got = got && mbar_wait(sfull, jj & 1, 442, abort_flag);
      if (named_bar_or(kBarSxOr, kSxThreads, !got)) {
        ok = false;
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const bool kvalid = key_off[(jj & 1) * 128 + row] >= 0;
      load_logits(kvalid);
      bool over = false;
#pragma unroll
      for (int i = 0; i < 32; ++i) over |= l[i] > mst[32 * hh + i] + kLazy;
      if (named_bar_or(kBarSxOr, kSxThreads, over)) {
        // Raise the stabiliser to this chunk's per-head maximum where it is larger.
        warp_reduce_scatter32(l, lane, [](float a, float c) { return fmaxf(a, c); });
        red[qt * 64 + 32 * hh + lane] = l[0];
        named_bar_sync(kBarSx, kSxThreads);
        if (tid < 64) {
          const float cm = fmaxf(fmaxf(red[tid], red[64 + tid]), fmaxf(red[128 + tid], red[192 + tid]));
          const float m_old = mst[tid];
          const float m_new = fmaxf(m_old, cm);
          fac[tid] = m_old == -INFINITY ? 0.f : (m_new == m_old ? 1.f : exp2f(m_old - m_new));
          mst[tid] = m_new;
        }
        named_bar_sync(kBarSx, kSxThreads);
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[i] *= fac[32 * hh + i];
        if (jj > 0) {  // O^T columns of this warp's heads, every M tile
          uint32_t v[32];
#pragma unroll 1
          for (int mt = 0; mt < 4; ++mt) {
            const uint32_t a = tmem + lane_base + 64 + 64 * mt + 32 * hh;
            tmem_ld32(a, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * fac[32 * hh + i]);
            tmem_st32(a, v);
          }
          tmem_wait_st();
        }
        load_logits(kvalid);  // the reduction consumed l
      }
      // P^T row of this key: heads 32*hh .. +31 as f16, MN-major (heads contiguous).
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i = 8 * c + 2 * k;
          const float m0 = mst[32 * hh + i], m1 = mst[32 * hh + i + 1];
          const float p0 = m0 == -INFINITY ? 0.f : exp2f(l[i] - m0);
          const float p1 = m1 == -INFINITY ? 0.f : exp2f(l[i + 1] - m1);
          __half2 hv = __floats2half2_rn(p0, p1);
          w[k] = *reinterpret_cast<uint32_t*>(&hv);
          const float2 back = __half22float2(hv);  // the sums use exactly what the MMA sees
          acc[i] += back.x;
          acc[i + 1] += back.y;
        }
        *reinterpret_cast<uint4*>(Pt + sw128_offset(row, 4 * hh + c)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async();
      tc_fence_before();
      named_bar_sync(kBarSx, kSxThreads);  // P^T complete (and O^T rescaled)
      if (tid == 0) {  // O^T += V^T P^T, one commit per tile half
        tc_fence_after();
#pragma unroll 1
        for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint64_t ad = sdesc(kt + mt * 32768 + ks * 2048, 16384, 1024, kSwizzle128B);
            const uint64_t bd = sdesc(pt + ks * 2048, 16384, 1024, kSwizzle128B);
            umma_f16(tmem + 64 + 64 * mt, ad, bd, id_o, (jj > 0 || ks > 0) ? 1u : 0u);
          }
          if (mt == 1) umma_commit(kfree_lo);
        }
        umma_commit(kfree_hi);
      }
    }
    if (ok && nc > 0) {
      ok = mbar_wait(kfree_hi, (nc - 1) & 1, 443, abort_flag);
      ok = !named_bar_or(kBarSxOr, kSxThreads, !ok);
    }
    if (ok) {
      tc_fence_after();
      // Per-head sums over the keys of all chunks.
      warp_reduce_scatter32(acc, lane, [](float a, float c) { return a + c; });
      red[qt * 64 + 32 * hh + lane] = acc[0];
      named_bar_sync(kBarSx, kSxThreads);
      const bool final_out = P.nsplit == 1;
      if (tid < 64) {
        const float s = (red[tid] + red[64 + tid]) + (red[128 + tid] + red[192 + tid]);
        if (final_out) {
          lsum[tid] = s > 0.f ? 1.f / s : 0.f;
          if (P.lse)
            P.lse[static_cast<int64_t>(q) * 64 + tid] = s > 0.f ? (mst[tid] + log2f(s)) * 0.6931471805599453f : -INFINITY;
        } else {
          P.stats[(static_cast<int64_t>(q) * kChunks + split) * 64 + tid] = make_float2(mst[tid], s);
        }
      }
      named_bar_sync(kBarSx, kSxThreads);
      float* part = P.part + (static_cast<int64_t>(q) * kChunks + split) * (64 * 512);
#pragma unroll 1
      for (int mt = 0; mt < 4; ++mt) {
        const int d = mt * 128 + row;
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + 64 + 64 * mt + 32 * hh, v);
        tmem_wait_ld();
        if (final_out) {
          float y[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) y[i] = __uint_as_float(v[i]) * lsum[32 * hh + i];
          if ((P.out_dtype & CSA2_OUT_DEROTATE) && d >= 448) {  // whole warps: rows 64..127 of the last M tile
            float c, sn;
            derotate_cs(t, (d - 448) >> 1, c, sn);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float other = __shfl_xor_sync(0xffffffffu, y[i], 1);
              y[i] = derotate_value(y[i], other, d, c, sn);
            }
          }
          if ((P.out_dtype & ~CSA2_OUT_DEROTATE) == CSA2_OUT_F32) {
            float* o = static_cast<float*>(P.out) + (static_cast<int64_t>(q) * 64 + 32 * hh) * 512 + d;
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i * 512] = y[i];
          } else {
            __nv_bfloat16* o = static_cast<__nv_bfloat16*>(P.out) + (static_cast<int64_t>(q) * 64 + 32 * hh) * 512 + d;
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i * 512] = __float2bfloat16_rn(y[i]);
          }
        } else {
          float* o = part + (32 * hh) * 512 + d;
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i * 512] = __uint_as_float(v[i]);
        }
      }
    }
  }

  if (tid == 0) {  // every MMA issued has completed before TMEM is released
    umma_commit(drain);
    mbar_wait(drain, 0, 433);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Merges the splits of one query: O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) L_s.
__global__ void __launch_bounds__(256) attn_combine_kernel(const float* __restrict__ part,
                                                           const float2* __restrict__ stats, int nsplit,
                                                           int out_dtype, void* __restrict__ out,
                                                           float* __restrict__ lse,
                                                           const int64_t* __restrict__ seq_len, int n_q) {
  griddep_wait();
  griddep_launch();
  const int q = blockIdx.x;
  const int h = blockIdx.y;
  const int tid = threadIdx.x;
  float m[kChunks], l[kChunks];
  float M = -INFINITY;
#pragma unroll
  for (int s = 0; s < kChunks; ++s) {
    m[s] = -INFINITY;
    l[s] = 0.f;
    if (s < nsplit) {
      const float2 st = stats[(static_cast<int64_t>(q) * kChunks + s) * 64 + h];
      m[s] = st.x;
      l[s] = st.y;
      M = fmaxf(M, st.x);
    }
  }
  float wsum = 0.f, f[kChunks];
#pragma unroll
  for (int s = 0; s < kChunks; ++s) {
    f[s] = (m[s] == -INFINITY) ? 0.f : exp2f(m[s] - M);
    wsum += f[s] * l[s];
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  for (int d = tid; d < 512; d += 256) {
    float acc = 0.f;
#pragma unroll
    for (int s = 0; s < kChunks; ++s)
      if (s < nsplit) acc += f[s] * part[((static_cast<int64_t>(q) * kChunks + s) * 64 + h) * 512 + d];
    float o = acc * inv;
    if ((out_dtype & CSA2_OUT_DEROTATE) && d >= 448) {  // whole warps: threads 192..255, second pass
      const int64_t t = seq_len[q / n_q] - n_q + q % n_q;
      float c, sn;
      derotate_cs(t, (d - 448) >> 1, c, sn);
      const float other = __shfl_xor_sync(0xffffffffu, o, 1);
      o = derotate_value(o, other, d, c, sn);
    }
    const int64_t oi = (static_cast<int64_t>(q) * 64 + h) * 512 + d;
    if ((out_dtype & ~CSA2_OUT_DEROTATE) == CSA2_OUT_F32) static_cast<float*>(out)[oi] = o;
    else static_cast<__nv_bfloat16*>(out)[oi] = __float2bfloat16_rn(o);
  }
  if (tid == 0 && lse)
    lse[static_cast<int64_t>(q) * 64 + h] = wsum > 0.f ? (M + log2f(wsum)) * 0.6931471805599453f : -INFINITY;
}

int attn_num_sms() {
  static int sms[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (!sms[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    sms[dev] = v > 0 ? v : 148;
  }
  return sms[dev];
}

}  // namespace

cudaError_t force_timeout_attn(int site, cudaStream_t stream) { return set_force_timeout_site(site, stream); }

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
  if (queries >= kNoSplitQueries) return 0;
  const size_t part = static_cast<size_t>(queries) * kChunks * 64 * 512 * sizeof(float);
  const size_t stats = static_cast<size_t>(queries) * kChunks * 64 * sizeof(float2);
  return ((part + 255) & ~size_t(255)) + ((stats + 255) & ~size_t(255));
}

cudaError_t launch_sparse_attn(const void* q, const int32_t* topk, const int64_t* seq_len, int B,
                               int n_q, const int32_t* block_table, int max_pages,
                               int64_t n_pages, const uint8_t* main_pages, const uint8_t* rings,
                               const int32_t* ring_idx, int64_t n_rings, const uint8_t* swa_chunk,
                               float softmax_scale, int out_dtype, void* out, float* lse, void* ws,
                               cudaStream_t stream, int m) {
  const int64_t Q = static_cast<int64_t>(B) * n_q;
  if (Q == 0) return cudaSuccess;
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
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
  p.swa_chunk = swa_chunk;
  p.m_shift = m == 2 ? 1 : 0;
  p.scale_log2 = softmax_scale * kLog2e;
  // Split a query's chunks over several CTAs only while that is what fills the GPU.
  p.nsplit = Q >= kNoSplitQueries
                 ? 1 : static_cast<int>(std::min<int64_t>(kChunks, std::max<int64_t>(1, attn_num_sms() / Q)));
  p.out_dtype = out_dtype;
  p.out = out;
  p.lse = lse;
  const size_t part_bytes = static_cast<size_t>(Q) * kChunks * 64 * 512 * sizeof(float);
  p.part = static_cast<float*>(ws);
  p.stats = reinterpret_cast<float2*>(static_cast<uint8_t*>(ws) + ((part_bytes + 255) & ~size_t(255)));
  cudaError_t e = launch_pdl(attn_kernel, dim3(static_cast<unsigned>(p.nsplit), static_cast<unsigned>(Q)),
                             dim3(kThreads), kSmemBytes, stream, 0, p);
  if (e != cudaSuccess || p.nsplit == 1) return e;
  return launch_pdl(attn_combine_kernel, dim3(static_cast<unsigned>(Q), 64), dim3(256), 0, stream, 0,
                    static_cast<const float*>(p.part), static_cast<const float2*>(p.stats), p.nsplit, out_dtype,
                    out, lse, seq_len, n_q);
}

}  // namespace csa2
