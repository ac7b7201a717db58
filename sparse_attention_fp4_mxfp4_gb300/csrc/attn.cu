// Reuse-mode sparse attention ("DeepSeek V4.1: model architecture and system
// design, a close reading" sections 1 and 2.2; "DeepSeek-V4.1-Flash: Pushing
// the Limits of KV Cache Compression" sections 3.3 and 3.6; "DeepSeek-V4 model
// structure (7): structure decides the system", closing summary): 64 query
// heads attend, with K = V = the 512-channel latent, to the query's top-k
// main entries (MXFP4, dequantised before attention) and to its FP8
// sliding-window entries.
//
// A query's 640 key slots form five chunks of 128 (four of top-k entries, one
// of window entries). A work item is a run of consecutive chunks of one query
// (all five when there are enough queries to fill the GPU; otherwise the
// chunks are split over up to five items whose partial results a second
// kernel merges), and it runs on a cluster of two CTAs that split the 512
// latent dimensions: CTA r holds dimensions 256 r .. 256 r + 255 of the query
// and of every key. Per chunk, with an online softmax:
//   S_r^T[128 keys x 64 heads] = K_r Q_r^T   (tcgen05, M = 128, N = 64, K = 256)
//   S^T = S_0^T + S_1^T                       (each CTA sends its partial to the
//                                              other through distributed shared
//                                              memory; both add them in the same
//                                              order, so both hold the same S^T)
//   softmax against a running per-head stabiliser (computed identically in
//   both CTAs), P^T in f16
//   O_r^T[256 dims x 64 heads] += V_r^T P^T  (tcgen05, 2 x M = 128, N = 64, K = 128)
// V_r^T is the CTA's key half-tile itself read as an MN-major operand; O_r^T
// stays in TMEM across chunks.
//
// An M = 128, K = 16 MMA takes the same time for any N <= 128, so the N = 64
// (heads) MMAs run well below the tensor pipe's peak whatever the layout;
// what this design buys is overlap. Half the dimensions per CTA halve the key
// tile (64 KB of f16 per 128 keys), so each CTA double-buffers it, and the
// tensor pipe runs S^T of chunk j + 1 and O^T of chunk j - 1 while the
// softmax warps work on chunk j: pipe order S(0) S(1) O(0) S(2) O(1) ...
// Roles per CTA: warps 8-11 gather the stored bytes of the CTA's half of each
// key (one thread per key) into registers ahead of time and dequantise them
// (exactly) to f16 into the 128-byte-swizzled key tile, a quarter of the
// dimensions (two K-blocks) at a time, so that a tile's first half is filled
// while the tensor pipe still reads its second half for the chunk before;
// their thread 0 issues each S^T quarter right after the warps wrote it.
// Warps 0-7 exchange partial scores, run the softmax (thread = key row x 32
// heads), write P^T, and their thread 0 issues the chunk's O^T MMAs; they
// also write the output.
//
// The CTA pairs are persistent: pair p walks work items p, p + pairs, ...
// with one running chunk counter, so barrier phases and buffers continue
// across items. While an item's last chunk is in flight the gather warps look
// up the next item's key slots and load its first keys, and they reload Q as
// soon as the last S^T MMA that reads it has completed; the first item's Q is
// loaded by the softmax warps, idle until its first S^T.
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
constexpr int kXWarps = 8;  // scores exchange, softmax, output
constexpr int kGWarps = 4;  // gather + dequantise; their thread 0 issues the MMAs
constexpr int kXThreads = kXWarps * 32;
constexpr int kGThreads = kGWarps * 32;
constexpr int kTmemWarp = kXWarps;  // the first gather warp allocates and frees TMEM
constexpr int kThreads = kXThreads + kGThreads;
constexpr int kTmemCols = 256;           // S^T x 2 buffers (64 columns each), O^T (2 M tiles x 64)
constexpr int kQsOff = 0;                // Q half: 64 heads x 256 dims f16, 4 K-blocks of 8 KB
constexpr int kKtOff = 32768;            // 2 key half-tiles: 128 keys x 256 dims f16, 4 K-blocks of 16 KB each
constexpr int kKtBytes = 65536;
constexpr int kPtOff = kKtOff + 2 * kKtBytes;  // P^T, MN-major: 128 keys x 64 heads f16
constexpr int kSxOff = kPtOff + 16384;         // the other CTA's partial S^T: 128 keys x 64 heads fp32
constexpr int kSxBytes = 32768;
constexpr int kMiscOff = kSxOff + kSxBytes;    // barriers, key offsets, per-head state
constexpr int kMiscBytes = 3072;
constexpr int kSmemBytes = 1024 + kMiscOff + kMiscBytes;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazy = 8.f;  // headroom (log2 units) before the stabiliser is raised
// Initial stabiliser: below every finite logit, so the first valid key raises
// it, and finite, so 2^(l - m) needs no special case (-inf logits give 0).
constexpr float kNoMax = -1e30f;
constexpr int kBarG = 1, kBarXOr = 2, kBarX = 3;  // named barriers
constexpr int64_t kChunkSrc = int64_t(1) << 62;   // key offset tag: the call's own window entries
// Tokens from which a query's chunks are never split over several work items
// (so no partial-output workspace is needed), whatever the SM count.
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
  int nsplit;         // work items per query (1..5)
  int n_items;        // Q * nsplit; each CTA pair walks items pair, pair + pairs, ...
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

// Byte offset, in the partial-score exchange buffer (128 keys x 64 heads
// fp32), of the 16 bytes that softmax thread (lane quarter qt, head half hh,
// lane) sends as its c-th group of 4 heads (c = 0..7): the 32 lanes of a warp
// cover 512 contiguous bytes for each c, so a warp's asynchronous remote
// stores, and the receiving warp's loads, are contiguous.
__device__ __forceinline__ uint32_t sx_offset(int qt, int hh, int lane, int c) {
  return static_cast<uint32_t>((((c * 2 + hh) * 4 + qt) * 32 + lane) * 16);
}

// 2^x on the special-function unit (x <= 8 here; -inf gives +0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One work item: a run of consecutive chunks of one query token.
struct Item {
  int q, split, b;
  int64_t N, t;
  int c0, nc;
};

__device__ __forceinline__ Item item_of(const AttnParams& P, int w) {
  Item it;
  it.q = w / P.nsplit;
  it.split = w % P.nsplit;
  it.b = it.q / P.n_q;
  it.N = P.seq_len[it.b];
  it.t = it.N - P.n_q + it.q % P.n_q;
  const int per = kChunks / P.nsplit, rem = kChunks % P.nsplit;
  it.c0 = it.split * per + (it.split < rem ? it.split : rem);
  it.nc = per + (it.split < rem ? 1 : 0);
  return it;
}

__global__ void __launch_bounds__(kThreads, 1) attn_kernel(const AttnParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Qs = smem + kQsOff;
  uint8_t* Kt = smem + kKtOff;
  uint8_t* Pt = smem + kPtOff;
  uint8_t* Sx = smem + kSxOff;
  uint8_t* misc = smem + kMiscOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc);          // barriers 2..16
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 260);
  uint32_t* vbits = reinterpret_cast<uint32_t*>(misc + 512);   // [8 chunk slots][4 words]: key row holds a key
  float* mst = reinterpret_cast<float*>(misc + 1024);          // [64] running stabiliser (log2)
  float* fac = reinterpret_cast<float*>(misc + 1280);          // [64] rescale factors
  float* lsum = reinterpret_cast<float*>(misc + 1536);         // [64] inverse sums
  float* red = reinterpret_cast<float*>(misc + 1792);          // [4][64] per-lane-quarter partials
  // Key tile quarters: "lo" = dimensions 0-127 of the CTA's half (K-blocks 0-1), "hi" = 128-255.
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t qready = bar(0), kfull_hi0 = bar(2), kfree_lo0 = bar(4), kfree_hi0 = bar(6);
  const uint32_t sfull0 = bar(8), sfree0 = bar(10);
  const uint32_t odone = bar(12), drain_o = bar(13), sxfull = bar(14), sxfree = bar(15), drain = bar(16);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(kfull_hi0 + 8 * i, kGThreads);
      mbar_init(kfree_lo0 + 8 * i, 1);
      mbar_init(kfree_hi0 + 8 * i, 1);
      mbar_init(sfull0 + 8 * i, 1);
      mbar_init(sfree0 + 8 * i, kXThreads);
    }
    mbar_init(odone, 1);
    mbar_init(drain_o, 1);
    mbar_init(qready, kXThreads);  // the first item's Q, written by the softmax warps
    mbar_init(sxfull, 1);  // armed here with the bytes expected from the other CTA (st.async)
    mbar_init(sxfree, 1);  // one remote arrival per chunk: the other CTA has read its partials
    mbar_init(drain, 1);
    *abort_flag = 0;
    mbar_init_fence();
    mbar_arrive_expect_tx(sxfull, kSxBytes);  // the first chunk's partials
  }
  if (warp == kTmemWarp) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  cl_sync();       // both CTAs' barriers exist before either arrives remotely
  griddep_wait();  // everything below may read what earlier kernels wrote
  griddep_launch();
  const int rk = static_cast<int>(cl_rank());  // this CTA's dimension half
  // Work items w = pair, pair + pairs, ...; both CTAs of the pair walk the same ones.
  const int pair = blockIdx.x >> 1, pairs = gridDim.x >> 1;

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= kXWarps) {
    // ============ gather + dequantise (128 threads, one per key row), MMAs ============
    const int gt = tid - kXThreads;
    const int r = gt;
    int64_t offs[kChunks];  // byte offsets of key slot gt of the current item's chunks (-1 = no key)
    // Resolves this thread's slot of every chunk of item `it`: the top-k
    // reads of all chunks are issued together, then their block-table reads,
    // so an item's lookups cost two dependent round trips.
    auto resolve_item = [&](const Item& it) {
      int32_t pos[kChunks], page[kChunks];
#pragma unroll
      for (int k = 0; k < kChunks; ++k) {
        const int c = it.c0 + k;
        pos[k] = (k < it.nc && c < 4) ? P.topk[static_cast<int64_t>(it.q) * 512 + c * 128 + gt] : -1;
      }
#pragma unroll
      for (int k = 0; k < kChunks; ++k) {
        page[k] = -1;
        const int32_t p = pos[k];
        if (p >= 0) {
          if (p > ((it.t + 1) >> P.m_shift) - 1 || (p >> 7) >= P.max_pages) {
            report(CSA2_ERR_DEVICE_BOUNDS, 401);
            pos[k] = -1;
          } else {
            page[k] = P.block_table[static_cast<int64_t>(it.b) * P.max_pages + (p >> 7)];
          }
        }
      }
#pragma unroll
      for (int k = 0; k < kChunks; ++k) {
        const int c = it.c0 + k;
        int64_t off = -1;
        if (k >= it.nc) {
        } else if (c < 4) {
          if (pos[k] >= 0) {
            if (page[k] < 0 || page[k] >= P.n_pages) report(CSA2_ERR_DEVICE_BOUNDS, 402);
            else off = static_cast<int64_t>(page[k]) * (128 * 288) + (pos[k] & 127) * 288;
          }
        } else if (!P.swa_chunk) {
          const int32_t ri = P.ring_idx[it.b];
          const int64_t base = it.N - 128;  // the ring holds positions N-128 .. N-1
          int64_t d = (static_cast<int64_t>(gt) - base) % 128;
          if (d < 0) d += 128;
          const int64_t p = base + d;  // the position stored in slot gt
          int64_t lo = it.t - 127;
          if (lo < base) lo = base;
          if (lo < 0) lo = 0;
          if (ri < 0 || ri >= P.n_rings) {
            if (gt == 0) report(CSA2_ERR_DEVICE_BOUNDS, 403);
          } else if (p >= lo && p <= it.t) {
            off = (static_cast<int64_t>(ri) * 128 + gt) * 512;
          }
        } else {
          // Prefill: key slot gt holds position t - 127 + gt, from the call's
          // own entries when it is one of the new positions, else from the
          // ring (which still holds the 128 positions before them).
          const int64_t p = it.t - 127 + gt, first_new = it.N - P.n_q;
          if (p >= 0) {
            if (p >= first_new) {
              off = kChunkSrc | ((static_cast<int64_t>(it.b) * P.n_q + (p - first_new)) * 512);
            } else {
              const int32_t ri = P.ring_idx[it.b];
              if (ri < 0 || ri >= P.n_rings) report(CSA2_ERR_DEVICE_BOUNDS, 404);
              else off = (static_cast<int64_t>(ri) * 128 + (p & 127)) * 512;
            }
          }
        }
        offs[k] = off;
      }
    };
    // Stored bytes of this CTA's half of key r. FP4: code bytes
    // [128 rk, +128) and scale bytes [256 + 16 rk, +16). FP8: bytes
    // [256 rk, +256).
    uint4 raw[16];
    uint4 scl;
    bool raw_valid = false;
    auto load = [&](int c, int64_t off) {
#pragma unroll
      for (int i = 0; i < 16; ++i) raw[i] = make_uint4(0, 0, 0, 0);
      scl = make_uint4(0, 0, 0, 0);
      raw_valid = off >= 0;
      if (off < 0) return;
      if (c < 4) {
        const uint8_t* e = P.main_pages + off;
#pragma unroll
        for (int i = 0; i < 8; ++i) raw[i] = reinterpret_cast<const uint4*>(e + 128 * rk)[i];
        scl = *reinterpret_cast<const uint4*>(e + 256 + 16 * rk);
      } else {
        const uint8_t* e = (off & kChunkSrc) ? P.swa_chunk + (off & ~kChunkSrc) : P.rings + off;
#pragma unroll
        for (int i = 0; i < 16; ++i) raw[i] = reinterpret_cast<const uint4*>(e + 256 * rk)[i];
      }
    };
    auto dequant = [&](int c, uint8_t* kt, int hf) {  // dimensions 128 hf .. +127 of the half
      if (c < 4) {
        const uint32_t sw[4] = {scl.x, scl.y, scl.z, scl.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint4 o[4];
          const int ib = 4 * hf + i;  // 32-dim group: 16 code bytes, 2 scale bytes
          dequant32_f16(raw[ib], static_cast<uint16_t>(sw[ib >> 1] >> (16 * (ib & 1))), o);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int d = 32 * ib + 8 * k;
            *reinterpret_cast<uint4*>(kt + (d >> 6) * 16384 + sw128_offset(r, (d & 63) >> 3)) = o[k];
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
          const int d = 128 * hf + 16 * i;
          uint8_t* kb = kt + (d >> 6) * 16384;
          *reinterpret_cast<uint4*>(kb + sw128_offset(r, (d & 63) >> 3)) = make_uint4(h[0], h[1], h[2], h[3]);
          *reinterpret_cast<uint4*>(kb + sw128_offset(r, ((d & 63) >> 3) + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
        }
      }
    };
    // The CTA's half of an item's Q: 64 heads x 256 dims, 16 x 16 bytes per
    // thread, in two batches of loads, bf16 -> f16 into the swizzled B operand.
    bool bad = false;  // f16 holds |q| < 65520 (65504 after rounding); larger or non-finite q is out of range
    auto load_q = [&](const Item& it) {
      const uint4* qg = reinterpret_cast<const uint4*>(P.q + static_cast<int64_t>(it.q) * 64 * 512);
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint4 qv[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int i = gt + (8 * half + k) * kGThreads;  // (head, 8-dim group) = (i >> 5, i & 31)
          qv[k] = qg[(i >> 5) * 64 + 32 * rk + (i & 31)];
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int i = gt + (8 * half + k) * kGThreads;
          const int h = i >> 5, g = i & 31;
          float f[8];
          bf16x8_to_f32(qv[k], f);
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            bad |= !(fabsf(f[2 * e]) < 65520.f) || !(fabsf(f[2 * e + 1]) < 65520.f);
            __half2 hv = __floats2half2_rn(f[2 * e], f[2 * e + 1]);
            o[e] = *reinterpret_cast<uint32_t*>(&hv);
          }
          *reinterpret_cast<uint4*>(Qs + (g >> 3) * 8192 + sw128_offset(h, g & 7)) =
              make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      fence_proxy_async();
    };

    // S^T MMAs, issued by thread gt == 0 right after a named barrier of the
    // gather warps (their shared-memory writes, each followed by a proxy
    // fence, are then visible to the tensor cores).
    const uint32_t id_s = idesc_f16(128, 64, false, false);
    const uint32_t qs = smem_u32(Qs);
    bool mma_ok = true;  // gt == 0: every MMA wait so far succeeded
    // S_r^T = K_r Q_r^T, one key tile quarter (8 K-steps) of chunk g.
    auto issue_s = [&](int g, int hf) {
      const int bf = g & 1;
      const uint32_t kt = smem_u32(Kt + bf * kKtBytes);
      tc_fence_after();
#pragma unroll
      for (int k = 8 * hf; k < 8 * hf + 8; ++k) {
        const uint64_t ad = sdesc(kt + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024, kSwizzle128B);
        const uint64_t bd = sdesc(qs + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024, kSwizzle128B);
        umma_f16(tmem + 64 * bf, ad, bd, id_s, k > 0 ? 1u : 0u);
      }
      if (hf == 1) umma_commit(sfull0 + 8 * bf);
    };

    int g = 0;          // global chunk counter of this CTA
    bool live = true;   // no abort seen
    if (pair < P.n_items) {
      const Item it0 = item_of(P, pair);
      resolve_item(it0);
      load(it0.c0, offs[0]);
    }
    for (int w = pair; w < P.n_items && live; w += pairs) {
      const Item it = item_of(P, w);
      // Q of this item: the previous item's last S^T MMAs must have read Qs.
      // The first item's Q is loaded by the softmax warps (idle until its
      // first S^T), while these warps look up its keys.
      bool ok = g == 0 || mbar_wait(sfull0 + 8 * ((g - 1) & 1), ((g - 1) >> 1) & 1, 456, abort_flag);
      if (ok && g > 0) load_q(it);
      if (named_bar_or(kBarG, kGThreads, !ok || *abort_flag)) {
        *abort_flag = 1;
        live = false;
        break;
      }
      for (int jj = 0; jj < it.nc; ++jj, ++g) {
        const int c = it.c0 + jj, bf = g & 1;
        uint8_t* kt = Kt + bf * kKtBytes;
        // A tile quarter is free once the O^T MMAs of the chunk two back that read it are done.
        const uint32_t ph = ((g >> 1) - 1) & 1;
        ok = g < 2 || mbar_wait(kfree_lo0 + 8 * bf, ph, 421, abort_flag);
        if (named_bar_or(kBarG, kGThreads, !ok || *abort_flag)) {
          *abort_flag = 1;
          live = false;
          break;
        }
        dequant(c, kt, 0);
        fence_proxy_async();
        named_bar_sync(kBarG, kGThreads);
        if (gt == 0 && mma_ok) {
          // The S^T buffer is free once the softmax has read chunk g - 2 from
          // it; the first S^T needs the first item's Q.
          if ((g == 0 && !mbar_wait(qready, 0, 457, abort_flag)) ||
              (g >= 2 && !mbar_wait(sfree0 + 8 * bf, ph, 451, abort_flag))) {
            mma_ok = false;
            *abort_flag = 1;
          } else {
            issue_s(g, 0);
          }
        }
        ok = g < 2 || mbar_wait(kfree_hi0 + 8 * bf, ph, 422, abort_flag);
        if (named_bar_or(kBarG, kGThreads, !ok || *abort_flag)) {
          *abort_flag = 1;
          live = false;
          break;
        }
        dequant(c, kt, 1);
        fence_proxy_async();
        // Which key rows hold a key (read by the softmax after this chunk's tile is complete).
        const uint32_t vb = __ballot_sync(0xffffffffu, raw_valid);
        if (lane == 0) vbits[(g & 7) * 4 + (warp - kXWarps)] = vb;
        mbar_arrive(kfull_hi0 + 8 * bf);
        named_bar_sync(kBarG, kGThreads);
        if (gt == 0 && mma_ok) issue_s(g, 1);
        // The next chunk's bytes (of this item, or the next item's first) are
        // on their way while the MMAs run; each thread loads its own key row.
        if (jj + 1 < it.nc) {
          load(c + 1, offs[jj + 1]);
        } else if (w + pairs < P.n_items) {
          const Item nx = item_of(P, w + pairs);
          resolve_item(nx);
          load(nx.c0, offs[0]);
        }
      }
    }
    if (bad) report(CSA2_ERR_DEVICE_RANGE, 405);
    if (gt == 0) {  // every S^T MMA issued has completed before TMEM is released
      umma_commit(drain);
      mbar_wait(drain, 0, 433);
    }
  } else {
    // ============ score exchange, softmax, output (256 threads) ============
    // Warp w: TMEM lane quarter qt = w % 4, heads 32 hh .. +31 with hh = w / 4.
    // In S^T a thread owns key row qt*32 + lane; in O^T dimension row
    // qt*32 + lane of both M tiles.
    const int qt = warp & 3, hh = warp >> 2;
    const int row = qt * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(qt * 32) << 16;
    const uint32_t peer = static_cast<uint32_t>(rk ^ 1);
    const uint32_t sx_peer = cl_map(smem_u32(Sx), peer);
    const uint32_t sxfull_peer = cl_map(sxfull, peer), sxfree_peer = cl_map(sxfree, peer);
    const uint32_t id_o = idesc_f16(128, 64, true, true);
    float l[32], acc[32];
    bool ok = true;
    int g = 0;
    if (pair < P.n_items) {
      // The first item's half of Q (64 heads x 256 dims): 8 x 16 bytes per
      // thread in one batch, bf16 -> f16 into the swizzled B operand.
      const Item it0 = item_of(P, pair);
      const uint4* qg = reinterpret_cast<const uint4*>(P.q + static_cast<int64_t>(it0.q) * 64 * 512);
      uint4 qv[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int i = tid + k * kXThreads;  // (head, 8-dim group) = (i >> 5, i & 31)
        qv[k] = qg[(i >> 5) * 64 + 32 * rk + (i & 31)];
      }
      bool qbad = false;  // f16 holds |q| < 65520; larger or non-finite q is out of range
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int i = tid + k * kXThreads;
        const int h = i >> 5, g8 = i & 31;
        float f[8];
        bf16x8_to_f32(qv[k], f);
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          qbad |= !(fabsf(f[2 * e]) < 65520.f) || !(fabsf(f[2 * e + 1]) < 65520.f);
          __half2 hv = __floats2half2_rn(f[2 * e], f[2 * e + 1]);
          o[e] = *reinterpret_cast<uint32_t*>(&hv);
        }
        *reinterpret_cast<uint4*>(Qs + (g8 >> 3) * 8192 + sw128_offset(h, g8 & 7)) =
            make_uint4(o[0], o[1], o[2], o[3]);
      }
      if (qbad) report(CSA2_ERR_DEVICE_RANGE, 405);
      fence_proxy_async();
      mbar_arrive(qready);
    }
    for (int w = pair; w < P.n_items && ok; w += pairs) {
      const Item it = item_of(P, w);
      const bool more_after = w + pairs < P.n_items;  // another item follows this one
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[i] = 0.f;
      if (tid < 64) mst[tid] = kNoMax;
      named_bar_sync(kBarX, kXThreads);  // the previous item's epilogue is done with the per-head state
      for (int jj = 0; jj < it.nc; ++jj, ++g) {
        const int bf = g & 1;
        bool got = mbar_wait(sfull0 + 8 * bf, (g >> 1) & 1, 441, abort_flag);
        tc_fence_after();
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + 64 * bf + 32 * hh, v);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(sfree0 + 8 * bf);
        // Partial scores to the other CTA (asynchronous stores counted on its
        // barrier), once it has read the previous ones.
        got = got && (g == 0 || mbar_wait_cluster(sxfree, (g - 1) & 1, 445, abort_flag));
        if (got) {
#pragma unroll
          for (int c = 0; c < 8; ++c)
            cl_st_async_v4(sx_peer + sx_offset(qt, hh, lane, c),
                           make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]), sxfull_peer);
        }
        got = got && mbar_wait_cluster(sxfull, g & 1, 446, abort_flag);
        // The key rows' validity (written by the gather warps before this chunk's tile).
        got = got && mbar_wait(kfull_hi0 + 8 * bf, (g >> 1) & 1, 447, abort_flag);
        if (named_bar_or(kBarXOr, kXThreads, !got)) {
          ok = false;
          *abort_flag = 1;
          break;
        }
        const bool kvalid = (vbits[(g & 7) * 4 + qt] >> lane) & 1u;
        bool over = false;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 wv = *reinterpret_cast<const uint4*>(Sx + sx_offset(qt, hh, lane, c));
          const float4 m4 = *reinterpret_cast<const float4*>(mst + 32 * hh + 4 * c);
          // Own partial + the other CTA's (IEEE addition is commutative: both
          // CTAs get the same logit).
          l[4 * c] = kvalid ? (__uint_as_float(v[4 * c]) + __uint_as_float(wv.x)) * P.scale_log2 : -INFINITY;
          l[4 * c + 1] = kvalid ? (__uint_as_float(v[4 * c + 1]) + __uint_as_float(wv.y)) * P.scale_log2 : -INFINITY;
          l[4 * c + 2] = kvalid ? (__uint_as_float(v[4 * c + 2]) + __uint_as_float(wv.z)) * P.scale_log2 : -INFINITY;
          l[4 * c + 3] = kvalid ? (__uint_as_float(v[4 * c + 3]) + __uint_as_float(wv.w)) * P.scale_log2 : -INFINITY;
          over |= (l[4 * c] > m4.x + kLazy) || (l[4 * c + 1] > m4.y + kLazy) || (l[4 * c + 2] > m4.z + kLazy) ||
                  (l[4 * c + 3] > m4.w + kLazy);
        }
        // Every X thread has read its partials once past this barrier.
        const bool raise = named_bar_or(kBarXOr, kXThreads, over);
        if (tid == 0 && (jj + 1 < it.nc || more_after)) {
          mbar_arrive_expect_tx(sxfull, kSxBytes);  // the next chunk's partials
          // This CTA's exchange buffer may take them: every read of it has
          // completed (its values were used before the barrier above). After
          // the last chunk nobody waits for this.
          cl_arrive_remote_relaxed(sxfree_peer);
        }
        if (raise) {
          // Raise the stabiliser to this chunk's per-head maximum where it is larger.
          float mx[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) mx[i] = l[i];
          warp_reduce_scatter32(mx, lane, [](float a, float c) { return fmaxf(a, c); });
          red[qt * 64 + 32 * hh + lane] = mx[0];
          named_bar_sync(kBarX, kXThreads);
          if (tid < 64) {
            const float cm = fmaxf(fmaxf(red[tid], red[64 + tid]), fmaxf(red[128 + tid], red[192 + tid]));
            const float m_old = mst[tid];
            const float m_new = fmaxf(m_old, cm);
            fac[tid] = m_new == m_old ? 1.f : ex2(m_old - m_new);  // 0 on the first raise
            mst[tid] = m_new;
          }
          named_bar_sync(kBarX, kXThreads);
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[i] *= fac[32 * hh + i];
        }
        // P^T row of this key: heads 32*hh .. +31 as f16 (into registers first).
        uint32_t pw[16];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float4 m4 = *reinterpret_cast<const float4*>(mst + 32 * hh + 4 * c);
          __half2 h01 = __floats2half2_rn(ex2(l[4 * c] - m4.x), ex2(l[4 * c + 1] - m4.y));
          __half2 h23 = __floats2half2_rn(ex2(l[4 * c + 2] - m4.z), ex2(l[4 * c + 3] - m4.w));
          pw[2 * c] = *reinterpret_cast<uint32_t*>(&h01);
          pw[2 * c + 1] = *reinterpret_cast<uint32_t*>(&h23);
          const float2 b01 = __half22float2(h01), b23 = __half22float2(h23);  // the sums use exactly what the MMA sees
          acc[4 * c] += b01.x;
          acc[4 * c + 1] += b01.y;
          acc[4 * c + 2] += b23.x;
          acc[4 * c + 3] += b23.y;
        }
        // O^T and P^T are free once the previous chunk's O^T MMAs are done
        // (for an item's first chunk, the previous item's last, which its
        // epilogue already waited for).
        got = jj == 0 || mbar_wait(odone, (g - 1) & 1, 443, abort_flag);
        if (named_bar_or(kBarXOr, kXThreads, !got)) {
          ok = false;
          *abort_flag = 1;
          break;
        }
        if (raise && jj > 0) {  // O^T columns of this warp's heads, both M tiles
          tc_fence_after();
          uint32_t o[32];
#pragma unroll 1
          for (int mt = 0; mt < 2; ++mt) {
            const uint32_t a = tmem + lane_base + 128 + 64 * mt + 32 * hh;
            tmem_ld32(a, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * fac[32 * hh + i]);
            tmem_st32(a, o);
          }
          tmem_wait_st();
        }
        // MN-major (heads contiguous).
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *reinterpret_cast<uint4*>(Pt + sw128_offset(row, 4 * hh + c)) =
              make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
        fence_proxy_async();
        tc_fence_before();
        named_bar_sync(kBarX, kXThreads);  // P^T complete (and O^T rescaled)
        if (tid == 0) {
          // O_r^T (+)= V_r^T P^T; an item's first chunk overwrites O^T. Frees
          // the key tile quarter by quarter.
          tc_fence_after();
          const uint32_t kt = smem_u32(Kt + bf * kKtBytes), pt = smem_u32(Pt);
#pragma unroll 1
          for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint64_t ad = sdesc(kt + mt * 32768 + ks * 2048, 16384, 1024, kSwizzle128B);
              const uint64_t bd = sdesc(pt + ks * 2048, 16384, 1024, kSwizzle128B);
              umma_f16(tmem + 128 + 64 * mt, ad, bd, id_o, (jj > 0 || ks > 0) ? 1u : 0u);
            }
            umma_commit((mt == 0 ? kfree_lo0 : kfree_hi0) + 8 * bf);
          }
          umma_commit(odone);
        }
      }
      if (!ok) break;
      // ---- this item's output ----
      ok = mbar_wait(odone, (g - 1) & 1, 448, abort_flag);
      if (named_bar_or(kBarXOr, kXThreads, !ok)) {
        ok = false;
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      // Per-head sums over the keys of all chunks (the same in both CTAs).
      warp_reduce_scatter32(acc, lane, [](float a, float c) { return a + c; });
      red[qt * 64 + 32 * hh + lane] = acc[0];
      named_bar_sync(kBarX, kXThreads);
      const bool final_out = P.nsplit == 1;
      if (tid < 64) {
        const float s = (red[tid] + red[64 + tid]) + (red[128 + tid] + red[192 + tid]);
        lsum[tid] = final_out ? (s > 0.f ? 1.f / s : 0.f) : 1.f;
        if (rk == 0) {
          if (final_out) {
            if (P.lse)
              P.lse[static_cast<int64_t>(it.q) * 64 + tid] =
                  s > 0.f ? (mst[tid] + log2f(s)) * 0.6931471805599453f : -INFINITY;
          } else {
            P.stats[(static_cast<int64_t>(it.q) * kChunks + it.split) * 64 + tid] = make_float2(mst[tid], s);
          }
        }
      }
      named_bar_sync(kBarX, kXThreads);
      float* part = P.part + (static_cast<int64_t>(it.q) * kChunks + it.split) * (64 * 512);
#pragma unroll 1
      for (int mt = 0; mt < 2; ++mt) {
        const int d = 256 * rk + 128 * mt + row;
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + 128 + 64 * mt + 32 * hh, v);
        tmem_wait_ld();
        if (final_out) {
          float y[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) y[i] = __uint_as_float(v[i]) * lsum[32 * hh + i];
          if ((P.out_dtype & CSA2_OUT_DEROTATE) && d >= 448) {  // whole warps: rows 64..127 of the last M tile
            float cs, sn;
            derotate_cs(it.t, (d - 448) >> 1, cs, sn);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float other = __shfl_xor_sync(0xffffffffu, y[i], 1);
              y[i] = derotate_value(y[i], other, d, cs, sn);
            }
          }
          if ((P.out_dtype & ~CSA2_OUT_DEROTATE) == CSA2_OUT_F32) {
            float* o = static_cast<float*>(P.out) + (static_cast<int64_t>(it.q) * 64 + 32 * hh) * 512 + d;
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i * 512] = y[i];
          } else {
            __nv_bfloat16* o =
                static_cast<__nv_bfloat16*>(P.out) + (static_cast<int64_t>(it.q) * 64 + 32 * hh) * 512 + d;
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i * 512] = __float2bfloat16_rn(y[i]);
          }
        } else {
          float* o = part + (32 * hh) * 512 + d;
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i * 512] = __uint_as_float(v[i]);
        }
      }
      tc_fence_before();  // the O^T reads precede the next item's first O^T MMAs
    }
    if (tid == 0) {  // every O^T MMA issued has completed before TMEM is released
      umma_commit(drain_o);
      mbar_wait(drain_o, 0, 434);
    }
  }

  tc_fence_before();
  __syncthreads();
  cl_sync();  // the other CTA no longer touches this CTA's shared memory
  if (warp == kTmemWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
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
  // Split a query's chunks over several work items (two CTAs each) only while
  // that is what fills the GPU.
  p.nsplit = Q >= kNoSplitQueries
                 ? 1 : static_cast<int>(std::min<int64_t>(kChunks, std::max<int64_t>(1, attn_num_sms() / (2 * Q))));
  p.out_dtype = out_dtype;
  p.out = out;
  p.lse = lse;
  const size_t part_bytes = static_cast<size_t>(Q) * kChunks * 64 * 512 * sizeof(float);
  p.part = static_cast<float*>(ws);
  p.stats = reinterpret_cast<float2*>(static_cast<uint8_t*>(ws) + ((part_bytes + 255) & ~size_t(255)));
  // One CTA pair per SM pair, each walking its share of the work items (or
  // one pair per item when there are fewer items than SM pairs).
  p.n_items = static_cast<int>(Q * p.nsplit);
  const int pairs = static_cast<int>(std::min<int64_t>(p.n_items, std::max(1, attn_num_sms() / 2)));
  cudaError_t e = launch_pdl(attn_kernel, dim3(static_cast<unsigned>(2 * pairs)), dim3(kThreads), kSmemBytes, stream,
                             2, p);
  if (e != cudaSuccess || p.nsplit == 1) return e;
  return launch_pdl(attn_combine_kernel, dim3(static_cast<unsigned>(Q), 64), dim3(256), 0, stream, 0,
                    static_cast<const float*>(p.part), static_cast<const float2*>(p.stats), p.nsplit, out_dtype,
                    out, lse, seq_len, n_q);
}

}  // namespace csa2
