// Hierarchical sparse indexer on the tensor cores ("DeepSeek V4.1: model
// architecture and system design, a close reading" section 2.2;
// "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" section
// 3.4): s(p) = sum_h w_h * max(0, qhat_h . khat_p) over 32 heads x 128 dims.
//
// The keys stay in their stored MXFP4 form: the tensor cores multiply packed
// E2M1 codes with one E4M3 scale per 16 channels (tcgen05.mma
// kind::mxf4nvf4, scale_vec::4X), which is exactly the storage format, so
// nothing is dequantised. The indexer page layout (16 groups of 8 entries:
// [chunk][row][16 B] codes, then 8 scale bytes per row) is itself a K-major
// operand of 8-row x 16-byte core matrices: K-adjacent core matrices are 128 B
// apart, 8-row groups 576 B apart.
//
// One kernel serves both uses:
//   * Full scan: a tile is one 128-entry page; the epilogue reduces scores to
//     the maximum over 8-position blocks. The query tokens of a sequence are
//     cut into groups (one group of one or two tokens; groups of 7 from three
//     tokens on, draft tokens or a prefill chunk); a group's tokens share the
//     tile: N = 32 * tokens MMA columns. A group walks the pages up to its last token's position, and
//     CTAs of different groups that read the same pages run side by side, so
//     the repeated reads of a prefill chunk come from L2.
//   * Pool rescore (Reindex, and the end of Full): a tile is 16 pool blocks of
//     8 positions, gathered block by block; the epilogue writes every score.
//
// Per CTA: warp E streams tiles into a ring of shared-memory stages with bulk
// copies; warps 0-3 move each row's 8 scale bytes into TMEM; warps 0..E-1 run
// the epilogue (warp w reads TMEM lane quarter w % 4, i.e. rows 32 (w % 4) ..
// +31, for the tokens j = w / 4 (mod E / 4)); warp E + 1 issues the two
// K = 64 MMAs of a tile (M = 128 positions) straight from the stage. E = 4 for
// one or two tokens and in the pool rescore; E = 16 for groups of 7 tokens,
// whose epilogue fp32 work is the bound.
#include <algorithm>

#include "kernels.h"
#include "sm103.cuh"

namespace csa2 {
namespace {

constexpr int kStages = 5;
constexpr int kTileBytes = 16 * 576;     // one indexer page / 16 pool blocks
constexpr int kIdxPageBytes = 16 * 576;
constexpr int kGroup = 8;      // one or two tokens: all in one CTA (the shared memory is sized for 8)
constexpr int kWideGroup = 7;  // prefill: tokens per scan CTA (two N = 224 accumulators fit TMEM)
constexpr int kWideSub = 4;    // prefill: epilogue warps per TMEM lane quarter

// Epilogue warps 4 * kSub, then the producer and the MMA warp.
__host__ __device__ constexpr int threads_for(int kSub) { return 32 * (4 * kSub + 2); }

struct ScanParams {
  const uint8_t* q_codes;
  const uint8_t* q_scales;
  const float* w;
  const int64_t* seq_len;
  int B, n_q;
  int m_shift;   // log2 of the tokens per entry (0 decoder, 1 encoder): token t sees entries < (t + 1) >> m_shift
  int n_grp;     // scan: query groups per sequence
  int grp_size;  // scan: tokens per group (the last group may hold fewer)
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

// TMEM columns: accumulators (two buffers when N <= 128), then, 32-aligned,
// two buffers of 8 scale columns for A (4 per K step) and 16 scale columns for
// B (8 per K step, n_q of them used).
struct TmemPlan {
  uint32_t nacc, sfa, sfb, ncols;
};

__host__ __device__ constexpr TmemPlan tmem_plan(int n_q) {
  const uint32_t n = 32u * n_q;
  const uint32_t nacc = 2u * n + 32u <= 512u ? 2u : 1u;
  const uint32_t sf = (nacc * n + 31u) & ~31u;
  uint32_t cols = 32;
  while (cols < sf + 32u) cols <<= 1;
  return TmemPlan{nacc, sf, sf + 16u, cols};
}

// Pool rescore: per pool slot of the CTA's tiles, the source (page * 16 + block
// in page, or kNoSlot) and the number of causal positions in the block.
constexpr uint32_t kNoSlot = 0xFFFFFFFFu;

__host__ __device__ constexpr int pool_table_bytes(int pool_tiles) { return (pool_tiles * 16 * 5 + 15) & ~15; }

// pool_tiles: tiles per CTA in pool mode (sizes the slot table), 0 for the scan.
__host__ __device__ constexpr int smem_bytes_for(int n_q, int pool_tiles) {
  return 1024 /*align*/ + kStages * kTileBytes + 32 * n_q * 64 /*q operand*/ + 2048 /*barriers, w*/ +
         pool_table_bytes(pool_tiles);
}

// fp32 fused multiply-add of two lanes at once (each lane an IEEE fma.rn).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

template <bool kPool, int kSub>
__global__ void __launch_bounds__(threads_for(kSub), kSub == 1 ? 4 : 1) indexer_kernel(const ScanParams P) {
  static_assert(!kPool || kSub == 1, "the pool rescore has one token per CTA");
  constexpr int kEpi = 4 * kSub;  // epilogue warps; producer = warp kEpi, MMA issuer = warp kEpi + 1
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // Scan: this CTA's query group, tokens j0 .. j0 + n_q - 1 of its sequence.
  const int grp = kPool ? 0 : static_cast<int>(blockIdx.y % P.n_grp);
  const int j0 = grp * P.grp_size;
  const int n_q = kPool ? 1 : (P.n_q - j0 < P.grp_size ? P.n_q - j0 : P.grp_size);
  const int n_cols = 32 * n_q;
  const TmemPlan plan = tmem_plan(n_q);
  uint8_t* stages = smem;                                   // kStages x 9216 B
  uint8_t* qbuf = stages + kStages * kTileBytes;            // n_cols x 64 B, core-matrix order
  uint8_t* misc = qbuf + n_cols * 64;
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc);       // 20 barriers
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 192);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 196);
  uint32_t* stage_mask = reinterpret_cast<uint32_t*>(misc + 200);  // kStages words
  float* wsm = reinterpret_cast<float*>(misc + 256);                 // n_cols floats
  uint32_t* slot_src = reinterpret_cast<uint32_t*>(misc + 2048);      // pool mode: [tiles_per_cta * 16]
  uint8_t* slot_n = misc + 2048 + (kPool ? P.tiles_per_cta * 16 * 4 : 0);  // pool mode: [tiles_per_cta * 16]

  const uint32_t full0 = smem_u32(&bars[0]), empty0 = smem_u32(&bars[kStages]);
  const uint32_t sfull0 = smem_u32(&bars[2 * kStages]);
  const uint32_t dfull0 = smem_u32(&bars[2 * kStages + 2]), dempty0 = smem_u32(&bars[2 * kStages + 4]);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(sfull0 + 8 * i, 128);
      mbar_init(dfull0 + 8 * i, 1);
      mbar_init(dempty0 + 8 * i, 32 * kEpi);
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == kEpi + 1) tmem_alloc(smem_u32(tmem_slot), plan.ncols);
  griddep_wait();  // everything below may read what earlier kernels wrote
  griddep_launch();
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
    b = blockIdx.y / P.n_grp;
    // The group's last token and the last entry it sees.
    const int64_t e_last = ((P.seq_len[b] - P.n_q + j0 + n_q) >> P.m_shift) - 1;
    const int64_t pages = e_last >= 0 ? (e_last + 128) >> 7 : 0;
    first_tile = blockIdx.x;
    tile_stride = gridDim.x;
    n_tiles = pages > first_tile ? (pages - first_tile + tile_stride - 1) / tile_stride : 0;
  }
  const int64_t seq_n = P.seq_len[b];
  if (!kPool && ((seq_n >> P.m_shift) + 7) / 8 > P.max_blocks) {
    if (threadIdx.x == 0) report(CSA2_ERR_DEVICE_BOUNDS, 204);
    n_tiles = 0;
  }


  // Pool rescore: the source (page * 16 + block in page, or kNoSlot) and the
  // causal positions of pool slot e of this CTA's tiles.
  const int64_t t_slot = ((seq_n - P.n_q + jq + 1) >> P.m_shift) - 1;  // pool mode: the token's last visible entry
  const int32_t* pool_row = kPool ? P.pool + (static_cast<int64_t>(b) * P.n_q + jq) * 2048 + first_tile * 16 : nullptr;
  // The page of pool block blk (-1: not causal or not mapped).
  auto slot_page = [&](int32_t blk) -> int32_t {
    if (blk < 0 || static_cast<int64_t>(blk) * 8 > t_slot) return -1;
    const int64_t lp = static_cast<int64_t>(blk) >> 4;
    return lp < P.max_pages ? P.block_table[static_cast<int64_t>(b) * P.max_pages + lp] : -2;
  };
  auto store_slot = [&](int e, int32_t blk, int32_t page) {
    uint32_t src = kNoSlot;
    int nv = 0;
    if (page != -1) {
      if (page < 0 || page >= P.n_pages) {
        report(CSA2_ERR_DEVICE_BOUNDS, 203);
      } else {
        src = static_cast<uint32_t>(page) * 16u + static_cast<uint32_t>(blk & 15);
        const int64_t left = t_slot - static_cast<int64_t>(blk) * 8 + 1;
        nv = left < 8 ? static_cast<int>(left) : 8;
      }
    }
    slot_src[e] = src;
    slot_n[e] = static_cast<uint8_t>(nv);
  };
  auto resolve_slot = [&](int e) {
    const int32_t blk = pool_row[e];
    store_slot(e, blk, slot_page(blk));
  };
  // The pool producer resolves the first two tiles' slots itself and starts;
  // warps 0-3 resolve the rest and meet it at named barrier 2 before tile 2.
  const bool pool_split = kPool && n_tiles > 2;

  // The producer needs neither the query nor TMEM: once the mbarriers are
  // visible it starts, while the other warps set the query up among
  // themselves (named barrier 1).
  const bool early_producer = warp == kEpi;
  __syncthreads();
  auto setup_sync = [&]() { named_bar_sync(1, 32 * (kEpi + 1)); };

  // Query operand: packed E2M1 codes of the CTA's query tokens, rows
  // n = token * 32 + head, in core-matrix order [n / 8][chunk][n % 8][16 B].
  if (tid < 128) {
    for (int task = tid; task < n_cols * 4; task += 128) {
      const int n = task >> 2, c = task & 3;
      const int jj = kPool ? jq : j0 + (n >> 5), h = n & 31;
      const int64_t qrow = (static_cast<int64_t>(b) * P.n_q + jj) * 32 + h;
      const uint4 codes = *reinterpret_cast<const uint4*>(P.q_codes + qrow * 64 + c * 16);
      *reinterpret_cast<uint4*>(qbuf + ((n >> 3) * 4 + c) * 128 + (n & 7) * 16) = codes;
    }
    for (int i = tid; i < n_cols; i += 128) {
      const int jj = kPool ? jq : j0 + (i >> 5);
      wsm[i] = P.w[(static_cast<int64_t>(b) * P.n_q + jj) * 32 + (i & 31)];
    }
    if (kPool) {
      // Slots 32.. in batches of 8 per thread: the batch's pool reads, then
      // its page-table reads, so each batch costs two dependent round trips.
      const int n_slots = static_cast<int>(n_tiles) * 16;
      for (int e0 = 32 + tid; e0 < n_slots; e0 += 8 * 128) {
        int32_t blk[8], page[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const int e = e0 + r * 128;
          blk[r] = e < n_slots ? pool_row[e] : -1;
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) page[r] = slot_page(blk[r]);
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const int e = e0 + r * 128;
          if (e < n_slots) store_slot(e, blk[r], page[r]);
        }
      }
      if (pool_split) named_bar_sync(2, 160);
    }
    fence_proxy_async();
  }
  uint32_t tmem = 0;
  if (!early_producer) {
    tc_fence_before();
    setup_sync();
    tc_fence_after();
    tmem = *tmem_slot;
  }

  // Query scales: column n of B has its scales in lane n % 32 of column
  // sfb + 8 * step + n / 32, replicated in all four 32-lane quarters (each
  // quarter of the M = 128 datapath reads B's scales from its own lanes), so
  // warps 0-3 each write their quarter. Every scale-factor address handed to
  // the MMA is 4-column aligned.
  if (warp < 4) {
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    for (int jj = 0; jj < n_q; ++jj) {
      const int jt = kPool ? jq : j0 + jj;
      const int64_t qrow = (static_cast<int64_t>(b) * P.n_q + jt) * 32 + lane;
      const uint8_t* sp = P.q_scales + qrow * 8;  // only 2-byte alignment is promised
      const uint32_t lo = sp[0] | (sp[1] << 8) | (sp[2] << 16) | (static_cast<uint32_t>(sp[3]) << 24);
      const uint32_t hi = sp[4] | (sp[5] << 8) | (sp[6] << 16) | (static_cast<uint32_t>(sp[7]) << 24);
      tmem_st1(tmem + lane_base + plan.sfb + jj, lo);
      tmem_st1(tmem + lane_base + plan.sfb + 8 + jj, hi);
    }
    tmem_wait_st();
  }
  if (!early_producer) {
    tc_fence_before();
    setup_sync();
    tc_fence_after();
  }

  if (warp == kEpi) {
    // ---- producer (whole warp: lookups in parallel, one bulk copy per lane) ----
    if (kPool) {
      // The first two tiles' slots (one per lane); the consumers read the
      // table after the stage barriers, which this warp arrives on afterwards.
      if (lane < n_tiles * 16) resolve_slot(lane);
      __syncwarp();
    }
    int32_t next_pages = -1;  // scan: page id of tile (i & ~31) + lane
    bool met = false;         // pool: named barrier 2 passed
    const int nt = static_cast<int>(n_tiles);
    int issued = 0;    // tiles whose copies (or empty arrival) this warp has issued
    int s = 0, u = 0;  // stage of tile i and the round of the ring it is in (i = u * kStages + s)
    for (int i = 0; i < nt; ++i, s = (s + 1 == kStages) ? 0 : s + 1, u += (s == 0) ? 1 : 0) {
      int go = 1;
      if (lane == 0) {
        if (u > 0 && !mbar_wait(empty0 + 8 * s, (u - 1) & 1, 201, abort_flag)) *abort_flag = 1;
        go = *abort_flag ? 0 : 1;
      }
      if (!__shfl_sync(0xffffffffu, go, 0)) break;
      const uint32_t dst = smem_u32(stages + s * kTileBytes);
      if (pool_split && i == 2) {  // the other slots are resolved
        named_bar_sync(2, 160);
        met = true;
      }
      if (!kPool) {
        if ((i & 31) == 0) {  // page ids of the next 32 tiles, one per lane
          const int64_t tl = first_tile + (i + lane) * tile_stride;
          next_pages = (i + lane < n_tiles && tl < P.max_pages)
                           ? P.block_table[static_cast<int64_t>(b) * P.max_pages + tl] : -1;
        }
        const int32_t page = __shfl_sync(0xffffffffu, next_pages, static_cast<int>(i & 31));
        if (lane == 0) {
          if (page < 0 || page >= P.n_pages) {
            report(CSA2_ERR_DEVICE_BOUNDS, 202);
            stage_mask[s] = 0;
            mbar_arrive(full0 + 8 * s);
          } else {
            stage_mask[s] = 0xFFFFu;
            mbar_arrive_expect_tx(full0 + 8 * s, kTileBytes);
            bulk_g2s(dst, P.idx_pages + static_cast<int64_t>(page) * kIdxPageBytes, kTileBytes, full0 + 8 * s);
          }
        }
      } else {
        // Lane g < 16 copies pool slot g of this tile (resolved at start).
        const uint32_t src = lane < 16 ? slot_src[i * 16 + lane] : kNoSlot;
        const bool valid = src != kNoSlot;
        const uint32_t mask = __ballot_sync(0xffffffffu, valid) & 0xFFFFu;
        if (lane == 0) {
          stage_mask[s] = mask;
          if (mask == 0) mbar_arrive(full0 + 8 * s);
          else mbar_arrive_expect_tx(full0 + 8 * s, __popc(mask) * 576u);
        }
        __syncwarp();
        if (valid)
          bulk_g2s(dst + lane * 576, P.idx_pages + static_cast<int64_t>(src >> 4) * kIdxPageBytes + (src & 15) * 576,
                   576, full0 + 8 * s);
      }
      issued = i + 1;
    }
    if (pool_split && !met) named_bar_sync(2, 160);  // stopped early: still meet warps 0-3
    // Every copy issued must have landed before the CTA's shared memory is
    // released. On the normal path the consumers already waited for all of
    // them; after an abort, wait here for the last round issued on each stage
    // (earlier rounds of a stage completed before its next round was issued).
    if (lane == 0) {
      for (int st = 0; st < kStages && st < issued; ++st) {
        const int last = st + kStages * ((issued - 1 - st) / kStages);
        mbar_wait(full0 + 8 * st, (last / kStages) & 1, 205);
      }
    }
  } else if (warp == kEpi + 1) {
    // ---- MMA issuer ----
    if (lane == 0) {
      const uint32_t idesc = idesc_mxf4nvf4(128, n_cols);
      const uint32_t qb = smem_u32(qbuf);
      const bool two = plan.nacc == 2;
      const int nt = static_cast<int>(n_tiles);
      int issued = 0;
      int s = 0, u = 0;
      for (int i = 0; i < nt; ++i, s = (s + 1 == kStages) ? 0 : s + 1, u += (s == 0) ? 1 : 0) {
        const int a = static_cast<int>(i & 1);
        const int acc = two ? (i & 1) : 0;
        const int ub = two ? (i >> 1) : i;
        if (!mbar_wait(full0 + 8 * s, u & 1, 210, abort_flag)) { *abort_flag = 1; break; }
        if (!mbar_wait(sfull0 + 8 * a, (i >> 1) & 1, 211, abort_flag)) { *abort_flag = 1; break; }
        if (ub > 0 && !mbar_wait(dempty0 + 8 * acc, (ub - 1) & 1, 212, abort_flag)) { *abort_flag = 1; break; }
        if (*abort_flag) break;
        tc_fence_after();
        const uint32_t st = smem_u32(stages + s * kTileBytes);
        const uint32_t sfa = tmem + plan.sfa + 8 * a;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const uint64_t ad = sdesc(st + k * 256, 128, 576, 0);
          const uint64_t bd = sdesc(qb + k * 256, 128, 512, 0);
          umma_mxf4nvf4(tmem + acc * n_cols, ad, bd, idesc, sfa + 4 * k, tmem + plan.sfb + k * 8,
                        k > 0 ? 1u : 0u);
        }
        umma_commit(empty0 + 8 * s);
        umma_commit(dfull0 + 8 * acc);
        issued = i + 1;
      }
      // Before TMEM is released, the last MMAs must have finished (they have on
      // the normal path: the epilogue waited for them).
      if (issued > 0)
        mbar_wait(dfull0 + 8 * (two ? ((issued - 1) & 1) : 0), (two ? ((issued - 1) >> 1) : (issued - 1)) & 1, 213);
    }
  } else {
    // ---- scales to TMEM (warps 0-3, thread t <-> row t) + epilogue ----
    const int quarter = warp & 3, sub = warp >> 2;
    const int row = quarter * 32 + lane;  // the tile row (TMEM lane) this thread owns
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t valid_rows[2] = {0, 0};  // kSub == 1: per 8-row group, tiles i and i-1 (from the stage)
    int32_t next_pages = -1;          // kSub > 1: page ids of tiles (i & ~31) + lane
    const bool two = plan.nacc == 2;
    // This warp's tokens of the group: j = sub, sub + kSub, ...
    const int mine = sub < n_q ? (n_q - sub + kSub - 1) / kSub : 0;
    auto epilogue = [&](int i) -> bool {
      const int acc = two ? (i & 1) : 0;
      bool row_ok;
      if (kSub == 1) {
        row_ok = (valid_rows[i & 1] >> (row >> 3)) & 1u;
      } else {
        // A wide CTA's epilogue warps run up to two tiles behind the
        // producer's stage bookkeeping, so they look the page up themselves.
        if ((i & 31) == 0) {
          const int64_t tl = first_tile + (i + lane) * tile_stride;
          next_pages = (i + lane < n_tiles && tl < P.max_pages)
                           ? P.block_table[static_cast<int64_t>(b) * P.max_pages + tl] : -1;
        }
        const int32_t page = __shfl_sync(0xffffffffu, next_pages, i & 31);
        row_ok = page >= 0 && page < P.n_pages;
      }
      if (!mbar_wait(dfull0 + 8 * acc, (two ? (i >> 1) : i) & 1, 221, abort_flag)) return false;
      tc_fence_after();
      const int64_t tile = first_tile + i * tile_stride;
      // The score of this thread's row for token jj from its 32 head dot products.
      auto finish = [&](const uint32_t (&r)[32], int jj) {
        // Heads h = 0, 1, 2, 3 (mod 4) in four fp32 sums, two per packed fma.
        float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
        const float4* wj = reinterpret_cast<const float4*>(wsm + jj * 32);  // 16-byte aligned
#pragma unroll
        for (int h = 0; h < 32; h += 4) {
          const float4 wv = wj[h >> 2];
          a01 = ffma2(make_float2(fmaxf(__uint_as_float(r[h]), 0.f), fmaxf(__uint_as_float(r[h + 1]), 0.f)),
                      make_float2(wv.x, wv.y), a01);
          a23 = ffma2(make_float2(fmaxf(__uint_as_float(r[h + 2]), 0.f), fmaxf(__uint_as_float(r[h + 3]), 0.f)),
                      make_float2(wv.z, wv.w), a23);
        }
        const float s = (a01.x + a01.y) + (a23.x + a23.y);
        if (!kPool) {
          const int64_t t_q = ((seq_n - P.n_q + j0 + jj + 1) >> P.m_shift) - 1;  // the token's last visible entry
          const int64_t p = tile * 128 + row;
          float m = (row_ok && p <= t_q) ? s : -INFINITY;
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
          if ((row & 7) == 0 && row_ok && p <= t_q)
            P.block_max[(static_cast<int64_t>(b) * P.n_q + j0 + jj) * P.max_blocks + (p >> 3)] = m;
        } else {
          const bool causal = (row & 7) < slot_n[i * 16 + (row >> 3)];
          const float v = (row_ok && causal) ? s : -INFINITY;
          P.scores[(static_cast<int64_t>(b) * P.n_q + jq) * 16384 + tile * 128 + row] = v;
        }
      };
      if (mine == 0) {
        tc_fence_before();
        mbar_arrive(dempty0 + 8 * acc);
      }
      for (int k = 0; k < mine; ++k) {
        const int jj = sub + k * kSub;
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + acc * n_cols + jj * 32, r);
        tmem_wait_ld();
        if (k == mine - 1) {
          tc_fence_before();
          mbar_arrive(dempty0 + 8 * acc);
        }
        finish(r, jj);
      }
      return true;
    };
    bool ok = true;
    const int nt = static_cast<int>(n_tiles);
    if (warp < 4) {
      int s = 0, u = 0;
      for (int i = 0; i < nt && ok; ++i, s = (s + 1 == kStages) ? 0 : s + 1, u += (s == 0) ? 1 : 0) {
        const int a = static_cast<int>(i & 1);
        if (!mbar_wait(full0 + 8 * s, u & 1, 231, abort_flag)) { ok = false; break; }
        if (kSub == 1) valid_rows[a] = stage_mask[s];
        // Row t's 8 scale bytes: blocks 0-3 feed the first K = 64 step, 4-7 the second.
        const uint8_t* grp_bytes = stages + s * kTileBytes + (row >> 3) * 576;
        const uint2 sc = *reinterpret_cast<const uint2*>(grp_bytes + 512 + (row & 7) * 8);
        const uint32_t sfa = tmem + lane_base + plan.sfa + 8 * a;
        tmem_st1(sfa + quarter, sc.x);
        tmem_st1(sfa + 4 + quarter, sc.y);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(sfull0 + 8 * a);
        if (i > 0) ok = epilogue(i - 1);
      }
      if (ok && nt > 0) ok = epilogue(nt - 1);
    } else {
      for (int i = 0; i < nt && ok; ++i) ok = epilogue(i);
    }
    if (!ok) *abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kEpi + 1) {
    tc_fence_after();
    tmem_dealloc(tmem, plan.ncols);
  }
}

template <bool kPool, int kSub>
cudaError_t launch(const ScanParams& p, dim3 grid, int n_q, cudaStream_t stream) {
  const int smem = smem_bytes_for(kPool ? 1 : n_q, kPool ? p.tiles_per_cta : 0);
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(indexer_kernel<kPool, kSub>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem_bytes_for(kPool ? 1 : kGroup, kPool ? 128 : 0));
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev] = true;
  }
  return launch_pdl(indexer_kernel<kPool, kSub>, grid, dim3(threads_for(kSub)), smem, stream, 0, p);
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

// Resident CTAs per SM, bounded by shared memory, TMEM columns and threads.
int ctas_per_sm(int n_q, int pool_tiles, int sub = 1) {
  const int by_smem = (228 * 1024) / (smem_bytes_for(n_q, pool_tiles) + 1024);
  const int by_tmem = 512 / static_cast<int>(tmem_plan(n_q).ncols);
  const int by_threads = 2048 / threads_for(sub);
  return std::max(1, std::min(std::min(by_smem, by_tmem), by_threads));
}

}  // namespace

cudaError_t force_timeout_indexer(int site, cudaStream_t stream) { return set_force_timeout_site(site, stream); }

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
                                cudaStream_t stream, int m) {
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
  p.m_shift = m == 2 ? 1 : 0;
  // One or two tokens per sequence: one group, 4 epilogue warps. Three or
  // more (draft tokens at decode, a prefill chunk): groups of 7 tokens, each
  // CTA with 16 epilogue warps (at 4 and 6 tokens per sequence and 256K
  // context this halves the scan's time against one group with 4 warps).
  const bool wide = n_q >= 3;
  p.grp_size = wide ? kWideGroup : kGroup;
  p.n_grp = (n_q + p.grp_size - 1) / p.grp_size;
  const int tile_q = std::min(n_q, p.grp_size);
  const int64_t rows = static_cast<int64_t>(B) * p.n_grp;
  const int64_t pages = (max_ctx / m + 127) / 128;
  const int64_t target = static_cast<int64_t>(ctas_per_sm(tile_q, 0, wide ? kWideSub : 1)) * num_sms();
  const int64_t per_seq = std::max<int64_t>(1, std::min<int64_t>(pages, (target + rows - 1) / rows));
  const dim3 grid(static_cast<unsigned>(per_seq), static_cast<unsigned>(rows));
  return wide ? launch<false, kWideSub>(p, grid, tile_q, stream) : launch<false, 1>(p, grid, tile_q, stream);
}

cudaError_t launch_pool_scores(const uint8_t* q_codes, const uint8_t* q_scales, const float* w,
                               const int64_t* seq_len, int B, int n_q,
                               const int32_t* block_table, int max_pages, int64_t n_pages,
                               const uint8_t* idx_pages, const int32_t* pool, float* scores,
                               cudaStream_t stream, int m) {
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
  p.n_grp = 1;
  p.grp_size = 1;
  p.m_shift = m == 2 ? 1 : 0;
  // The 128 tiles of a token are cut into equal runs so that all CTAs are
  // resident at once (one wave) where the batch allows it; a run's slot table
  // is sized to the run, so short runs leave room for more CTAs per SM.
  int splits = 1, per = 128;
  for (int cps = 4; cps >= 1; --cps) {
    const int64_t target = static_cast<int64_t>(cps) * num_sms();
    splits = static_cast<int>(std::min<int64_t>(128, std::max<int64_t>(1, target / Q)));
    per = (128 + splits - 1) / splits;
    splits = (128 + per - 1) / per;
    if (ctas_per_sm(1, per) >= cps) break;
  }
  p.tiles_per_cta = per;
  return launch<true, 1>(p, dim3(splits, static_cast<unsigned>(Q)), 1, stream);
}

}  // namespace csa2
