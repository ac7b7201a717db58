/*
 * csa2.h -- C ABI of libcsa2.so, the sm_103a (GB300) decode hot path of
 * DeepSeek-V4.1-Flash's CSA2 sparse attention.
 *
 * Sources (public pages the method is taken from):
 *   [RN] "DeepSeek V4.1: model architecture and system design, a close reading"
 *        (blog.keqichen.top): section 1 (configuration: indexer 32 heads x 128,
 *        top-k 512, query 64 heads x 512, 2048 blocks x 8 positions = 16384
 *        candidates, window 128), section 2.2 (CSA2 modes Full / Reindex /
 *        Reuse and the hierarchical sparse indexer), section 2.3 (FP4 main KV:
 *        E2M1 with one E4M3 scale per 16 channels, no global scale, quantised
 *        after RoPE; sliding-window KV kept in FP8).
 *   [AB] "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression"
 *        (abstract notes): section 3.3 (what each mode reuses), section 3.4
 *        (block selection by the maximum score of a block's positions, pool
 *        shared by later Reindex layers), section 3.6 (FP4 main KV, dequantised
 *        before attention).
 *   [SY] "DeepSeek-V4 model structure (7): structure decides the system": the
 *        paged KV cache in 128-token blocks and the per-sequence sliding-window
 *        state; attention over the top-k entries plus 128 window entries with
 *        K = V single-head MQA on a 512-dim latent.
 *
 * Conventions
 *   - Every function returns a csa2 status (int); CSA2_OK is 0. Functions
 *     validate their host-side arguments first and never abort or exit.
 *     csa2_last_error() gives a thread-local text for the last failure.
 *   - All tensor pointers are DEVICE pointers unless a comment says host.
 *     The caller allocates and frees every buffer; the library allocates no
 *     memory and keeps no per-call state. Device pointers that the kernels
 *     read or write with vector accesses must be 16-byte aligned
 *     (CSA2_ERR_INVALID_ARG otherwise).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Every call is asynchronous on that stream. Index checks done on
 *     the device (page ids, positions, ring slots) do not fail the call: the
 *     offending access is skipped and a device status word is set, which
 *     csa2_check_device_status() reads after the stream's work is done. Every
 *     wait inside a kernel is bounded (about 2 s) and records
 *     CSA2_ERR_DEVICE_TIMEOUT instead of hanging.
 *   - bf16 tensors are passed as void* and hold IEEE bfloat16 bit patterns.
 *
 * Data layout in HBM (decoder CSA2 at m = 1: one entry per token)
 *   - Main KV page (CSA2_PLANE_MAIN): 128 entries x 288 bytes. Entry e of a
 *     page starts at e * 288: 256 bytes of E2M1 codes (channel 2i in the low
 *     nibble of byte i, channel 2i+1 in the high nibble), then 32 E4M3 scale
 *     bytes (scale j covers channels 16j..16j+15).
 *   - Indexer-key page (CSA2_PLANE_INDEX): 16 groups of 8 entries, 576 bytes
 *     per group (9216 bytes per page). Group g covers entries 8g..8g+7:
 *     bytes [0, 512) hold codes ordered [chunk c = 0..3][row r = 0..7][16
 *     bytes = channels 32c..32c+31 of entry 8g+r]; bytes [512, 576) hold the
 *     8 scale bytes of each row, row-major.
 *   - Block table: int32 [B, max_pages]; entry (b, i) is the physical page of
 *     positions 128i..128i+127 of sequence b (-1 = unmapped). Main and
 *     indexer planes share the table: physical page P is main_pages + P*36864
 *     and idx_pages + P*9216. n_pages = number of physical pages of each pool.
 *   - Sliding-window ring: [n_rings, 128, 512] E4M3 bytes, no scale; position
 *     p of a sequence lives in slot p % 128 of its ring.
 *   - Query token j of n_q of sequence b sits at position
 *     t = seq_len[b] - n_q + j (seq_len counts the entries already appended,
 *     including this step's tokens). At decode (csa2_sparse_attn) its sliding
 *     window is the positions max(0, t - 127, seq_len[b] - 128) .. t still
 *     resident in the ring; in a prefill call (csa2_sparse_attn_prefill) it is
 *     exactly max(0, t - 127) .. t.
 *   - Tokens per entry m (argument m of the indexer and attention calls): 1
 *     for the decoder's CSA2 layers, where entry p is token p; 2 for the
 *     encoder's ([RN] 1, [AB] 3.1), where entry e summarises tokens 2e and
 *     2e + 1 (csa2_compress_append). Pages, block tables, top-k positions and
 *     block ids then count entries; seq_len and t still count tokens: token t
 *     sees the complete entries 0 .. floor((t + 1) / m) - 1, and its sliding
 *     window stays in tokens.
 *   - Query tokens per sequence: the indexer calls and the prefill attention
 *     take n_q <= CSA2_MAX_PREFILL_NQ (the Full scan serves them in groups of
 *     8 tokens), the decode attention n_q <= CSA2_MAX_NQ; every call takes
 *     B * n_q <= CSA2_MAX_TOKENS. Larger shapes return CSA2_ERR_UNSUPPORTED.
 */
#ifndef CSA2_H_
#define CSA2_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status ---------------------------------------------------------------- */
#define CSA2_OK 0
#define CSA2_ERR_INVALID_ARG 1     /* null/misaligned pointer, bad size or count */
#define CSA2_ERR_UNSUPPORTED 2     /* a shape the library does not implement */
#define CSA2_ERR_WORKSPACE 3       /* workspace missing or too small */
#define CSA2_ERR_CUDA 4            /* a CUDA runtime call or launch failed */
#define CSA2_ERR_DEVICE_TIMEOUT 5  /* a bounded wait inside a kernel gave up */
#define CSA2_ERR_DEVICE_BOUNDS 6   /* a device-side index check failed */
#define CSA2_ERR_DEVICE_RANGE 7    /* an input value outside the supported range (read on the device) */

/* ---- fixed geometry of the decoder CSA2 layer ([RN] 1, [AB] 3.1) ----------- */
#define CSA2_LATENT_DIM 512    /* main KV latent channels (K = V) */
#define CSA2_Q_HEADS 64        /* attention query heads */
#define CSA2_IDX_HEADS 32      /* indexer heads */
#define CSA2_IDX_DIM 128       /* indexer head dim */
#define CSA2_TOPK 512          /* selected positions per query */
#define CSA2_POOL_BLOCKS 2048  /* candidate blocks per query */
#define CSA2_BLOCK 8           /* positions per candidate block */
#define CSA2_WINDOW 128        /* sliding-window entries */
#define CSA2_PAGE_TOKENS 128   /* entries per page */
#define CSA2_MAIN_ENTRY_BYTES 288
#define CSA2_IDX_ENTRY_BYTES 72
#define CSA2_MAX_NQ 8          /* query tokens per sequence in one decode call */
#define CSA2_MAX_PREFILL_NQ 4096  /* query tokens per sequence in one prefill call */
#define CSA2_MAX_TOKENS 65535  /* B * n_q in one call */

#define CSA2_PLANE_MAIN 0
#define CSA2_PLANE_INDEX 1

#define CSA2_OUT_F32 0
#define CSA2_OUT_BF16 1
/* OR'ed into out_dtype: rotate the output back by the query position
 * ("DeepSeek-V4 model structure (7): structure decides the system", closing
 * summary: the output is rotated back to restore relative position). The last
 * 64 channels of every output row, as pairs (448 + 2i, 449 + 2i), are rotated
 * by -t * theta_i with theta_i = 10000^(-2i/64) and t the token's position
 * N - n_q + j, the inverse of the rotary layout of the stored latents. */
#define CSA2_OUT_DEROTATE 0x100

#define CSA2_MODE_FULL 0
#define CSA2_MODE_REINDEX 1
#define CSA2_MODE_REUSE 2

#define CSA2_OP_INDEXER_FULL 1
#define CSA2_OP_INDEXER_REINDEX 2
#define CSA2_OP_SPARSE_ATTN 3
#define CSA2_OP_DECODE_LAYER 4

const char* csa2_status_string(int status);
/* Thread-local detail text of the last failing call on this thread. */
const char* csa2_last_error(void);
int csa2_version(void);

/* ---- size queries (host only, no GPU needed) ------------------------------- */
/* Bytes of one page of a plane: 36864 (main) or 9216 (indexer). */
int csa2_page_bytes(int plane, size_t* bytes);
/* Bytes of one sliding-window ring: 128 * 512 = 65536. */
int csa2_ring_bytes(size_t* bytes);
/* Workspace bytes that an op needs for B sequences, n_q tokens each and a
 * context of at most max_ctx entries. */
int csa2_workspace_bytes(int op, int B, int n_q, int64_t max_ctx, size_t* bytes);

/* ---- append: MXFP4 main KV + indexer keys, FP8 window ([RN] 2.3, [AB] 3.6) -- */
/* Quantises T new entries and stores each into slot pos % 128 of page
 * block_table[seq_idx[i], pos / 128] of both planes.
 *   latent:  bf16 [T, 512], post-RoPE main-KV entries
 *   idx_key: bf16 [T, 128], indexer keys
 *   seq_idx: int32 [T] in [0, B); pos: int64 [T]; block_table: int32 [B, max_pages]
 * Per 16-channel block: scale = E4M3(amax / 6) (fp32 IEEE division, round to
 * nearest even, saturating at 448); code = nearest E2M1 value of |v| / scale,
 * ties to the even code. Entries with an unmapped or out-of-range page are
 * skipped and set CSA2_ERR_DEVICE_BOUNDS. */
int csa2_append_kv(const void* latent, const void* idx_key, const int32_t* seq_idx,
                   const int64_t* pos, int T, const int32_t* block_table, int B, int max_pages,
                   int64_t n_pages, uint8_t* main_pages, uint8_t* idx_pages, void* stream);

/* E4M3 (round to nearest even, saturating, no scale) of T new window entries
 * x: bf16 [T, 512] into slot pos % 128 of ring ring_idx[i] of rings
 * [n_rings, 128, 512]. Entries of one call must go to distinct slots (at most
 * 128 consecutive positions per ring); a prefill chunk longer than that uses
 * csa2_quant_fp8_entries + csa2_ring_refill. */
int csa2_append_swa(const void* x, const int32_t* ring_idx, const int64_t* pos, int T,
                    int64_t n_rings, uint8_t* rings, void* stream);

/* One layer's share of csa2_decode_appends: its window entries and its
 * indexer query. swa == NULL: no window append for this layer; q_idx == NULL:
 * no quantisation. */
typedef struct {
  const void* swa;          /* bf16 [T, 512] window entries, 16-byte aligned, or NULL */
  const int32_t* ring_idx;  /* int32 [T]: ring of each entry */
  int64_t n_rings;
  uint8_t* rings;           /* [n_rings, 128, 512], 16-byte aligned */
  const void* q_idx;        /* bf16 [q_n] indexer query, 16-byte aligned, or NULL */
  int64_t q_n;              /* a multiple of 16 */
  uint8_t* q_codes;         /* [q_n / 2], 8-byte aligned */
  uint8_t* q_scales;        /* [q_n / 16] */
} csa2_append_layer;

/* A decode step's stores and query quantisations in ONE kernel launch: the
 * same bytes as csa2_append_kv(latent, idx_key, seq_idx, pos, T, ...) (main
 * KV at one token per entry), then, for each of the n_layers layers,
 * csa2_append_swa(swa, ring_idx, pos, T, n_rings, rings) and
 * csa2_quant_mxfp4(q_idx, q_n, q_codes, q_scales). The parts run
 * concurrently, so no part may write memory another part reads or writes
 * (distinct rings per layer and distinct code buffers, as a decode step has).
 * T = 0: only the quantisations run (latent .. idx_pages and every swa may
 * then be NULL). n_layers <= 16 (else CSA2_ERR_UNSUPPORTED). Errors and
 * device-side bounds reports are those of the three calls ([RN] 2.3 and
 * [AB] 3.6 for the stores, [AB] 3.4 for the indexer query). */
int csa2_decode_appends(const void* latent, const void* idx_key, const int32_t* seq_idx, const int64_t* pos, int T,
                        const int32_t* block_table, int B, int max_pages, int64_t n_pages, uint8_t* main_pages,
                        uint8_t* idx_pages, const csa2_append_layer* layers, int n_layers, void* stream);

/* Encoder-side append at m tokens per entry (m = 1 or 2; [RN] 1 / [AB] 3.1
 * give m = 2 for the encoder's CSA2 layers; "DeepSeek-V4 model structure
 * (7)", KV cache of hybrid attention: an unfinished entry's tail tokens and
 * their compression weights are per-sequence state). T new tokens: kv, kv_gate
 * bf16 [T, 512] (candidate latent and its compression logits), idx_key,
 * idx_gate bf16 [T, 128] (the same for the indexer key), seq_idx int32 [T],
 * pos int64 [T] token positions. The rows of one sequence must be consecutive
 * positions in order. The token at position p with p % m == m - 1 completes
 * entry e = p / m: per channel, out_c = sum_i exp(z_ic - max z) x_ic /
 * sum_i exp(z_ic - max z) over tokens m*e .. p (fp64), rounded once to bf16,
 * then stored like csa2_append_kv at entry e (page block_table[b, e / 128],
 * slot e % 128). The tokens of the entry that precede this call come from
 * tail: bf16 [B, m - 1, 1280] (per token: kv 512, kv_gate 512, idx_key 128,
 * idx_gate 128; slot = position % m), owned by the caller, one per (layer,
 * sequence group); tokens whose entry stays unfinished after the call are
 * written there. m = 1 stores every token as is (tail unused, may be NULL).
 * Two kernels run in order on the stream (entries, then tails). */
int csa2_compress_append(const void* kv, const void* kv_gate, const void* idx_key, const void* idx_gate,
                         const int32_t* seq_idx, const int64_t* pos, int T, int m, void* tail,
                         const int32_t* block_table, int B, int max_pages, int64_t n_pages,
                         uint8_t* main_pages, uint8_t* idx_pages, void* stream);

/* The same E4M3 encoding of T window entries x: bf16 [T, 512] into out: u8
 * [T, 512] (16-byte aligned), row for row. A prefill chunk's own window
 * entries are encoded this way for csa2_sparse_attn_prefill before the ring
 * receives the last 128 of them (csa2_ring_refill). */
int csa2_quant_fp8_entries(const void* x, int T, uint8_t* out, void* stream);

/* Ring refill ([RN] 2.4, SWA Bounded Replay: the window state is rebuilt from
 * the last n_win tokens alone). entries: E4M3 [B, n, 512], the window entries
 * of positions seq_len[b] - n .. seq_len[b] - 1 of sequence b; the last
 * min(n, 128) of them go to slot position % 128 of ring ring_idx[b] of rings
 * [n_rings, 128, 512]; the other slots keep their bytes. With n >= 128 the
 * ring afterwards holds exactly positions seq_len[b] - 128 .. seq_len[b] - 1.
 * Entries at a negative position or of a ring index out of range are skipped
 * and set CSA2_ERR_DEVICE_BOUNDS. */
int csa2_ring_refill(const uint8_t* entries, const int64_t* seq_len, int B, int n,
                     const int32_t* ring_idx, int64_t n_rings, uint8_t* rings, void* stream);

/* ---- codec utilities -------------------------------------------------------- */
/* MXFP4 quantisation of n bf16 values (n % 16 == 0): codes [n/2], scales
 * [n/16]. Used for the indexer query (32 heads x 128 per token) and tests. */
int csa2_quant_mxfp4(const void* x, int64_t n, uint8_t* codes, uint8_t* scales, void* stream);
/* Dequantisation to fp32 (exact). */
int csa2_dequant_mxfp4(const uint8_t* codes, const uint8_t* scales, int64_t n, float* out,
                       void* stream);
/* fp32 -> E4M3 (round to nearest even, saturating to +-448). */
int csa2_quant_fp8(const float* x, int64_t n, uint8_t* out, void* stream);

/* ---- hierarchical sparse indexer ([RN] 2.2, [AB] 3.4) ----------------------- */
/* Full-mode scan: for every causal position p <= t of every query token,
 * s(p) = sum_h w_h * max(0, qhat_h . khat_p) (fp32 accumulation of exact FP4
 * products on the tensor cores), then the maximum over each block of 8 causal
 * positions.
 *   q_codes: [B, n_q, 32, 64] bytes, q_scales: [B, n_q, 32, 8] (MXFP4 of the
 *   indexer query, as written by csa2_quant_mxfp4 on a [B, n_q, 32, 128]
 *   tensor); w: fp32 [B, n_q, 32]; seq_len: int64 [B].
 *   block_max: fp32 [B, n_q, max_blocks], max_blocks >= ceil(max_ctx / m / 8);
 *   entries at or past ceil(floor((t + 1) / m) / 8) are left untouched.
 * max_ctx is a host-side upper bound of seq_len (sizes the grid); m: tokens
 * per entry (1 or 2; positions p are entries then). */
int csa2_indexer_scan(const uint8_t* q_codes, const uint8_t* q_scales, const float* w,
                      const int64_t* seq_len, int B, int n_q, int64_t max_ctx,
                      const int32_t* block_table, int max_pages, int64_t n_pages,
                      const uint8_t* idx_pages, float* block_max, int64_t max_blocks, int m,
                      void* stream);

/* Top 2048 blocks of each query token by block maximum (higher first, then
 * lower block id); all causal blocks when there are at most 2048.
 *   pool: int32 [B, n_q, 2048], block ids ascending, -1 padded. */
int csa2_block_topk(const float* block_max, const int64_t* seq_len, int B, int n_q,
                    int64_t max_blocks, int32_t* pool, int m, void* stream);

/* Reindex: scores only the positions 8b..8b+7 (<= t) of each pool block b
 * with this layer's indexer query and takes the top 512 (higher score first,
 * then lower position).
 *   pool: int32 [B, n_q, 2048] (-1 entries ignored); topk: int32 [B, n_q,
 *   512], positions ascending, -1 padded.
 *   ws: workspace of csa2_workspace_bytes(CSA2_OP_INDEXER_REINDEX, ...). */
int csa2_indexer_reindex(const uint8_t* q_codes, const uint8_t* q_scales, const float* w,
                         const int64_t* seq_len, int B, int n_q, const int32_t* block_table,
                         int max_pages, int64_t n_pages, const uint8_t* idx_pages,
                         const int32_t* pool, int32_t* topk, void* ws, size_t ws_bytes, int m,
                         void* stream);

/* Same computation and outputs as csa2_indexer_reindex (same arguments,
 * including the ratio m, and the same host checks and status codes), for
 * callers that cannot allocate device memory: plug-ins whose host framework
 * owns every device allocation, and decode loops that must not allocate
 * because an allocation there can synchronise the device or fail under
 * memory pressure in the middle of a step. The per-slot scores live in a
 * fixed 4 MiB device array inside the library instead of a caller workspace.
 * The pages have no counterpart of this entry point; it only changes where
 * scratch lives.
 *   - At most 64 query tokens per call (B * n_q <= 64); larger calls return
 *     CSA2_ERR_UNSUPPORTED and launch nothing.
 *   - Every GPU that loads the library holds the array until the process
 *     exits. The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) and keeps it for the process; make that first
 *     call before any stream capture. A device reset (cudaDeviceReset)
 *     invalidates the kept address: do not call this entry point on a device
 *     after resetting it.
 *   - All calls share the one array: calls that overlap on the GPU (other
 *     streams, other threads) race and must be serialised by the caller. No
 *     content has to start at zero: each call writes every slot it reads.
 *   - No cudaMalloc / cudaFree or allocating library routine is called. */
int csa2_indexer_reindex_noalloc(const uint8_t* q_codes, const uint8_t* q_scales, const float* w,
                                 const int64_t* seq_len, int B, int n_q,
                                 const int32_t* block_table, int max_pages, int64_t n_pages,
                                 const uint8_t* idx_pages, const int32_t* pool, int32_t* topk, int m,
                                 void* stream);

/* Full-mode indexer = scan + block top-2048 + rescore of the pool + top-512.
 * The final top-512 over the pool equals the top-512 over all causal
 * positions up to ties. ws: csa2_workspace_bytes(CSA2_OP_INDEXER_FULL, ...). */
int csa2_indexer_full(const uint8_t* q_codes, const uint8_t* q_scales, const float* w,
                      const int64_t* seq_len, int B, int n_q, int64_t max_ctx,
                      const int32_t* block_table, int max_pages, int64_t n_pages,
                      const uint8_t* idx_pages, int32_t* pool, int32_t* topk, void* ws,
                      size_t ws_bytes, int m, void* stream);

/* ---- sparse attention (Reuse mode; [RN] 2.2, [AB] 3.3 / 3.6, [SY]) ---------- */
/* o_h = softmax(scale * q_h K^T) V with K = V = the dequantised keys: the main
 * entries at the query's top-k positions (-1 skipped) followed by its FP8
 * window entries, duplicates kept. 64 heads x 512 dims, fp32 softmax.
 *   q: bf16 [B, n_q, 64, 512], every element finite with |q| < 65520: the
 *   tensor cores take q in f16 (exact for such values, whose f16 rounding
 *   stays finite); a larger or non-finite element records
 *   CSA2_ERR_DEVICE_RANGE and makes that token's output undefined (the other
 *   tokens are unaffected).
 *   topk: int32 [B, n_q, 512]; ring_idx: int32 [B]
 *   out: [B, n_q, 64, 512] fp32 (out_dtype CSA2_OUT_F32) or bf16
 *   (CSA2_OUT_BF16), optionally | CSA2_OUT_DEROTATE (see its definition;
 *   lse is unchanged by it); lse: fp32 [B, n_q, 64] natural-log sum of exp of the
 *   scaled logits (may be NULL).
 *   ws: csa2_workspace_bytes(CSA2_OP_SPARSE_ATTN, ...). */
int csa2_sparse_attn(const void* q, const int32_t* topk, const int64_t* seq_len, int B, int n_q,
                     const int32_t* block_table, int max_pages, int64_t n_pages,
                     const uint8_t* main_pages, const uint8_t* rings, const int32_t* ring_idx,
                     int64_t n_rings, float softmax_scale, int out_dtype, void* out, float* lse,
                     void* ws, size_t ws_bytes, int m, void* stream);

/* Prefill (chunked prefill) of n_q <= CSA2_MAX_PREFILL_NQ new tokens per
 * sequence ([RN] 2.2, [AB] 3.3: the same attention over a causal run of query
 * tokens). As csa2_sparse_attn, except for the window: token t sees exactly
 * the entries of positions max(0, t - 127) .. t. Those of the call's own
 * positions N - n_q .. N - 1 come from swa_chunk: E4M3 [B, n_q, 512]
 * (csa2_quant_fp8_entries), 16-byte aligned; older ones from the rings, which
 * must still hold the 128 positions before the chunk (refill them with
 * csa2_ring_refill after the call). ws: csa2_workspace_bytes(CSA2_OP_SPARSE_ATTN,
 * ...), zero bytes (ws may be NULL) from 256 tokens on. */
int csa2_sparse_attn_prefill(const void* q, const int32_t* topk, const int64_t* seq_len, int B,
                             int n_q, const int32_t* block_table, int max_pages, int64_t n_pages,
                             const uint8_t* main_pages, const uint8_t* rings,
                             const int32_t* ring_idx, int64_t n_rings, const uint8_t* swa_chunk,
                             float softmax_scale, int out_dtype, void* out, float* lse, void* ws,
                             size_t ws_bytes, int m, void* stream);

/* ---- mode dispatcher ([RN] 2.2, [AB] 3.3) ----------------------------------- */
typedef struct csa2_layer_args {
  int mode;                 /* CSA2_MODE_FULL / _REINDEX / _REUSE */
  int B, n_q;
  int64_t max_ctx;          /* host-side upper bound of seq_len */
  const int64_t* seq_len;   /* [B] */
  const int32_t* block_table;
  int max_pages;
  int64_t n_pages;
  const uint8_t* main_pages;
  const uint8_t* idx_pages;
  const uint8_t* rings;     /* this layer's rings [n_rings, 128, 512] */
  const int32_t* ring_idx;  /* [B] */
  int64_t n_rings;
  const uint8_t* q_idx_codes;  /* FULL / REINDEX: this layer's indexer query */
  const uint8_t* q_idx_scales;
  const float* w;
  const void* q;            /* bf16 [B, n_q, 64, 512], this layer's query */
  int32_t* pool;            /* FULL: written. REINDEX: read; NULL = the group's latest pool */
  int32_t* topk;            /* FULL / REINDEX: written. REUSE: read; NULL = latest top-k */
  float softmax_scale;
  int out_dtype;
  void* out;
  float* lse;               /* may be NULL */
  void* ws;
  size_t ws_bytes;          /* csa2_workspace_bytes(CSA2_OP_DECODE_LAYER, ...) */
  const uint8_t* swa_chunk; /* NULL: decode (n_q <= CSA2_MAX_NQ, window from the ring).
                               Else prefill: the chunk's E4M3 window entries
                               [B, n_q, 512], attention as csa2_sparse_attn_prefill */
  int tokens_per_entry;     /* m: 0 or 1 = decoder layer, 2 = encoder layer */
} csa2_layer_args;

/* One layer: FULL = indexer_full then sparse_attn; REINDEX = indexer_reindex
 * (on the given or latest pool) then sparse_attn; REUSE = sparse_attn on the
 * given or latest top-k. With swa_chunk set, the attention is
 * csa2_sparse_attn_prefill (the ring is not written: refill it after the
 * chunk's last layer). */
int csa2_decode_layer(const csa2_layer_args* layer, void* stream);

/* Layers in order on one stream. A REINDEX layer with pool == NULL uses the
 * latest FULL layer's pool of the group; a REUSE layer with topk == NULL uses
 * the latest top-k written by an earlier layer of the group. Layers may share
 * one workspace: they run one after another on the stream. */
int csa2_decode_group(const csa2_layer_args* layers, int n_layers, void* stream);

/* ---- device status ---------------------------------------------------------- */
/* Waits for the stream, then reads (and clears) the device status words:
 * *status = CSA2_OK, CSA2_ERR_DEVICE_TIMEOUT, CSA2_ERR_DEVICE_BOUNDS or
 * CSA2_ERR_DEVICE_RANGE (the first one recorded since the last read). */
int csa2_check_device_status(void* stream, int* status);

/* Test utility (fault injection without a fault): from this call on, every
 * bounded wait inside this library's kernels whose internal site number equals
 * `site` gives up at once, exactly as if its time limit had run out: it
 * records CSA2_ERR_DEVICE_TIMEOUT (read by csa2_check_device_status), and the
 * kernel stops its work, waits for its own copies and tensor-core operations
 * in flight, releases its tensor memory and returns. site = 0 turns it off.
 * Site 210 is the indexer's tensor-core issuer waiting for a tile's copy (the
 * Full scan and the pool rescore). Synchronises `stream`. */
int csa2_debug_force_wait_timeout(int site, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CSA2_H_ */
