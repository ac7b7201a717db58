// CPU oracle of the CSA2 decode path (DeepSeek-V4.1-Flash).
//
// TEST INFRASTRUCTURE ONLY. Only tests/, the smoke check and the benchmark's
// CPU-baseline arm may load this file's library. It shares no code, header,
// table or constant generator with the CUDA library, and neither includes the
// other. It is deliberately plain and slow: every step is the definition of
// what the method computes, written out in fp64 (the formats are integer /
// exact by definition).
//
// Sources (the three public pages this implementation is written from):
//   [RN] "DeepSeek V4.1: model architecture and system design, a close reading"
//        (blog.keqichen.top, 2026-09): section 1 (model configuration),
//        section 2.2 (CSA2, three modes, hierarchical sparse indexer),
//        section 2.3 (FP4 main KV cache).
//   [AB] "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression"
//        (abstract notes, git.hyonglin.top): section 3.1 (configuration),
//        section 3.3 (CSA2 reuse modes), section 3.4 (hierarchical sparse
//        indexer), section 3.6 (FP4 main KV cache).
//   [SY] "DeepSeek-V4 model structure (7): structure decides the system"
//        (blog.javazero.top): "KV cache of hybrid attention" (128-token
//        blocks, sliding window kept as per-sequence state) and the closing
//        summary (K = V single-head MQA over top-k entries plus 128 window
//        entries).
//
// Readings where the pages are silent (each stated once, here):
//   * The scale of a 16-channel block is RNE_E4M3(amax / 6) with the division
//     in IEEE fp32 and saturation to 448; no second-level scale ([RN] 2.3,
//     [AB] 3.6 fix E2M1 + one E4M3 scale per 16 channels and no global scale).
//   * An element's E2M1 code is the grid value nearest to |v| / scale, ties to
//     the even code, saturating at 6; -0 and values that round to 0 get code 0.
//   * Indexer score s(p) = sum_h w_h * max(0, qhat_h . khat_p) (the pages give
//     none; 32 heads x 128 dims from [RN] 1 / [AB] 3.1). The indexer query is
//     MXFP4-quantised like the keys.
//   * Block score = max over the causal positions of an 8-position block; pool
//     = top 2048 blocks (all when there are fewer); final top-512 over all
//     causal positions of the Full layer, which equals the top-512 of its pool
//     up to ties; Reindex scores only pool positions p <= t.
//   * Ties: higher score first, then lower index. Selections are returned in
//     ascending index order.
//   * Attention: K = V = the 512-channel latent, 64 query heads, logits
//     tau * q . k, softmax in fp64; the key multiset is the dequantised top-k
//     entries followed by the FP8 window entries, duplicates kept.
//   * Window of query t when the ring holds the last W positions of a
//     sequence of N entries: positions max(0, t - W + 1, N - W) .. t.
//   * Compressed entries at ratio m (encoder-side CSA2, m = 2): entry e covers
//     tokens m*e .. m*e + m - 1; per channel it is the softmax over those m
//     tokens of their compression logits, weighting their candidate values
//     (fp64, then rounded to bf16); a token at position t sees the complete
//     entries 0 .. floor((t + 1) / m) - 1, and its window stays in tokens.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <thread>
#include <vector>

namespace {

template <class F>
void parallel_for(int64_t n, int threads, F&& f) {
  if (threads < 1) threads = 1;
  if (threads == 1 || n < 64) {
    f(0, n);
    return;
  }
  std::vector<std::thread> pool;
  const int64_t chunk = (n + threads - 1) / threads;
  for (int i = 0; i < threads; ++i) {
    const int64_t lo = i * chunk, hi = std::min<int64_t>(n, lo + chunk);
    if (lo >= hi) break;
    pool.emplace_back([&f, lo, hi] { f(lo, hi); });
  }
  for (auto& t : pool) t.join();
}

float bf16_value(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// Round a non-negative, exactly represented double to the nearest integer,
// ties to even.
double round_half_even(double q) {
  const double fl = std::floor(q);
  const double d = q - fl;
  if (d > 0.5) return fl + 1.0;
  if (d < 0.5) return fl;
  return std::fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0;
}

// E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit, no inf/NaN.
double e2m1_value(int code) {
  const int e = (code >> 1) & 3, m = code & 1;
  const double mag = (e == 0) ? 0.5 * m : (1.0 + 0.5 * m) * std::ldexp(1.0, e - 1);
  return (code & 8) ? -mag : mag;
}

// E4M3 ("fn" variant): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits, no
// infinities, S.1111.111 is NaN, largest finite 448, subnormals m * 2^-9.
double e4m3_value(int byte) {
  const int s = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
  if (e == 15 && m == 7) return std::nan("");
  const double mag = (e == 0) ? m * std::ldexp(1.0, -9) : (1.0 + m / 8.0) * std::ldexp(1.0, e - 7);
  return s ? -mag : mag;
}

// fp32 -> E4M3, round to nearest even, saturating to +-448 (infinities too).
// NaN -> 0x7F.
uint8_t e4m3_encode(float xf) {
  if (std::isnan(xf)) return 0x7F;
  const uint8_t sign = std::signbit(xf) ? 0x80 : 0x00;
  const double a = std::fabs(static_cast<double>(xf));
  if (a >= 448.0) return sign | 0x7E;
  if (a == 0.0) return sign;
  int e2;
  std::frexp(a, &e2);  // a = f * 2^e2, f in [0.5, 1)
  int E = e2 - 1;      // a = (1.xxx) * 2^E
  if (E < -6) {        // below the smallest normal 2^-6: multiples of 2^-9
    const double m = round_half_even(std::ldexp(a, 9));
    return sign | static_cast<uint8_t>(m);  // m == 8 is exactly the encoding of 2^-6
  }
  double m = round_half_even(std::ldexp(a, 3 - E));  // in [8, 16]
  if (m >= 16.0) {
    m = 8.0;
    E += 1;
  }
  const int biased = E + 7;
  if (biased > 15 || (biased == 15 && m - 8.0 > 6.0)) return sign | 0x7E;
  return sign | static_cast<uint8_t>((biased << 3) | static_cast<int>(m - 8.0));
}

// E2M1 magnitude code of a >= 0 against scale sf > 0: the grid value g*sf
// nearest to a, ties to the even code, saturating at g = 6. Midpoints between
// neighbouring grid values times sf are exact doubles.
int e2m1_magnitude_code(double a, double sf) {
  static const double grid[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  int k = 0;
  for (int i = 0; i < 7; ++i) {
    const double mid = 0.5 * (grid[i] + grid[i + 1]) * sf;
    const bool up = a > mid || (a == mid && ((i + 1) % 2 == 0));
    if (!up) break;
    k = i + 1;
  }
  return k;
}

// One 16-channel MXFP4 block.
void quant_block(const float* v, uint8_t* codes /*8 bytes*/, uint8_t* scale) {
  float amax = 0.0f;
  for (int i = 0; i < 16; ++i) amax = std::max(amax, std::fabs(v[i]));
  const float s32 = amax / 6.0f;
  const uint8_t sb = e4m3_encode(s32);
  const double sf = e4m3_value(sb);
  *scale = sb;
  for (int i = 0; i < 8; ++i) {
    int c[2];
    for (int h = 0; h < 2; ++h) {
      const float x = v[2 * i + h];
      int k = (sf > 0.0) ? e2m1_magnitude_code(std::fabs(static_cast<double>(x)), sf) : 0;
      if (k != 0 && x < 0.0f) k |= 8;
      c[h] = k;
    }
    codes[i] = static_cast<uint8_t>(c[0] | (c[1] << 4));  // even channel in the low nibble
  }
}

void dequant_row(const uint8_t* codes, const uint8_t* scales, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) {
    const int nib = (codes[i / 2] >> (4 * (i & 1))) & 15;
    out[i] = e2m1_value(nib) * e4m3_value(scales[i / 16]);
  }
}

// khat of one 128-dim bf16 row: quantise then dequantise.
void fp4_roundtrip_row(const uint16_t* row, int dim, double* out) {
  float v[512];
  uint8_t codes[256], scales[32];
  for (int c = 0; c < dim; ++c) v[c] = bf16_value(row[c]);
  for (int b = 0; b < dim / 16; ++b) quant_block(v + 16 * b, codes + 8 * b, scales + b);
  dequant_row(codes, scales, dim, out);
}

double index_score(const double* qhat, const double* w, int heads, int dim, const double* k) {
  double s = 0.0;
  for (int h = 0; h < heads; ++h) {
    double d = 0.0;
    for (int c = 0; c < dim; ++c) d += qhat[h * dim + c] * k[c];
    s += w[h] * std::max(0.0, d);
  }
  return s;
}

// Indices of the k largest scores (higher score first, then lower index),
// written ascending.
int64_t topk_indices(const double* s, int64_t n, int64_t k, int64_t* out) {
  std::vector<int64_t> idx(static_cast<size_t>(n));
  std::iota(idx.begin(), idx.end(), 0);
  const int64_t m = std::min(n, k);
  std::partial_sort(idx.begin(), idx.begin() + m, idx.end(), [s](int64_t a, int64_t b) {
    return s[a] > s[b] || (s[a] == s[b] && a < b);
  });
  std::sort(idx.begin(), idx.begin() + m);
  for (int64_t i = 0; i < m; ++i) out[i] = idx[i];
  return m;
}

// fp64 -> bf16, round to nearest, ties to even, in one step (no intermediate
// float). Finite inputs within the bf16 range (the compressor's convex
// combinations of bf16 values always are).
uint16_t bf16_round(double d) {
  if (d == 0.0) return std::signbit(d) ? 0x8000u : 0u;
  const bool neg = d < 0;
  double a = neg ? -d : d;
  int e = 0;
  std::frexp(a, &e);  // a = f * 2^e, f in [0.5, 1)
  // bf16 keeps 8 significant bits down to 2^-126, then a fixed quantum 2^-133.
  int q_exp = e - 8;
  if (q_exp < -133) q_exp = -133;
  double r = std::nearbyint(std::ldexp(a, -q_exp));  // default mode: nearest, ties to even
  const float v = static_cast<float>(std::ldexp(r, q_exp));  // exact: at most 8 significant bits
  uint32_t u;
  std::memcpy(&u, &v, 4);
  return static_cast<uint16_t>((u >> 16) | (neg ? 0x8000u : 0u));
}

}  // namespace

extern "C" {

double orc_e2m1_value(int code) { return e2m1_value(code); }
double orc_e4m3_value(int byte) { return e4m3_value(byte); }
int orc_e4m3_encode(float x) { return e4m3_encode(x); }

void orc_e4m3_encode_array(const float* x, int64_t n, uint8_t* out, int threads) {
  parallel_for(n, threads, [=](int64_t lo, int64_t hi) {
    for (int64_t i = lo; i < hi; ++i) out[i] = e4m3_encode(x[i]);
  });
}

// MXFP4 quantisation of n values (n % 16 == 0): codes[n/2], scales[n/16].
void orc_mxfp4_quant(const float* x, int64_t n, uint8_t* codes, uint8_t* scales, int threads) {
  parallel_for(n / 16, threads, [=](int64_t lo, int64_t hi) {
    for (int64_t b = lo; b < hi; ++b) quant_block(x + 16 * b, codes + 8 * b, scales + b);
  });
}

void orc_mxfp4_dequant(const uint8_t* codes, const uint8_t* scales, int64_t n, double* out) {
  dequant_row(codes, scales, n, out);
}

void orc_fp8_quant(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_encode(x[i]);
}

void orc_fp8_dequant(const uint8_t* in, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_value(in[i]);
}

// Indexer scores of n dequantised keys [n, dim] against qhat [heads, dim].
void orc_index_scores(const double* qhat, const double* w, int heads, int dim, const double* keys,
                      int64_t n, double* out, int threads) {
  parallel_for(n, threads, [=](int64_t lo, int64_t hi) {
    for (int64_t p = lo; p < hi; ++p) out[p] = index_score(qhat, w, heads, dim, keys + p * dim);
  });
}

// Block maxima of s[0..n): out[b] = max over positions 8b..min(8b+7, n-1).
void orc_block_max(const double* s, int64_t n, int block, double* out) {
  for (int64_t b = 0; b * block < n; ++b) {
    double m = -INFINITY;
    for (int64_t p = b * block; p < std::min<int64_t>(n, (b + 1) * block); ++p) m = std::max(m, s[p]);
    out[b] = m;
  }
}

int64_t orc_topk(const double* s, int64_t n, int64_t k, int64_t* out) {
  return topk_indices(s, n, k, out);
}

// Full-mode hierarchical indexer for one query token at position t.
//   qidx: bf16 [heads, dim] indexer query (MXFP4-quantised here);
//   w: fp32 [heads]; keys: bf16 [t+1, dim] indexer keys of positions 0..t
//   (MXFP4-quantised here).
// Outputs: scores[t+1] (fp64, may be null), blockmax[ceil((t+1)/block)] (may
// be null), pool[n_pool] block ids ascending with -1 padding, topk[k]
// positions ascending with -1 padding. Returns the number of top-k positions.
int64_t orc_full_indexer(const uint16_t* qidx, const float* w, int heads, int dim,
                         const uint16_t* keys, int64_t t, int block, int64_t n_pool, int64_t k,
                         double* scores, double* blockmax, int32_t* pool, int32_t* topk,
                         int threads) {
  const int64_t n = t + 1;
  std::vector<double> qhat(static_cast<size_t>(heads) * dim), wd(heads);
  for (int h = 0; h < heads; ++h) {
    fp4_roundtrip_row(qidx + static_cast<int64_t>(h) * dim, dim, qhat.data() + h * dim);
    wd[h] = w[h];
  }
  std::vector<double> own;
  if (!scores) {
    own.resize(static_cast<size_t>(n));
    scores = own.data();
  }
  const double* qp = qhat.data();
  const double* wp = wd.data();
  parallel_for(n, threads, [=](int64_t lo, int64_t hi) {
    double kh[512];
    for (int64_t p = lo; p < hi; ++p) {
      fp4_roundtrip_row(keys + p * dim, dim, kh);
      scores[p] = index_score(qp, wp, heads, dim, kh);
    }
  });
  const int64_t nb = (n + block - 1) / block;
  std::vector<double> bm(static_cast<size_t>(nb));
  orc_block_max(scores, n, block, bm.data());
  if (blockmax) std::copy(bm.begin(), bm.end(), blockmax);
  std::vector<int64_t> sel(static_cast<size_t>(std::max(n_pool, k)));
  const int64_t npool = topk_indices(bm.data(), nb, n_pool, sel.data());
  for (int64_t i = 0; i < n_pool; ++i) pool[i] = i < npool ? static_cast<int32_t>(sel[i]) : -1;
  const int64_t nk = topk_indices(scores, n, k, sel.data());
  for (int64_t i = 0; i < k; ++i) topk[i] = i < nk ? static_cast<int32_t>(sel[i]) : -1;
  return nk;
}

// Reindex-mode indexer for one query token at position t: scores only the
// positions 8b..8b+7 (<= t) of the pool's blocks b (-1 entries ignored).
//   keys: bf16 indexer keys of positions 0..t (row p at keys + p*dim).
// Outputs: pos_scores[n_pool*block] (score of pool slot i, -inf when the slot
// is not a causal position; may be null), topk[k] ascending, -1 padded.
int64_t orc_reindex(const uint16_t* qidx, const float* w, int heads, int dim, const uint16_t* keys,
                    int64_t t, int block, const int32_t* pool, int64_t n_pool, int64_t k,
                    double* pos_scores, int32_t* topk, int threads) {
  std::vector<double> qhat(static_cast<size_t>(heads) * dim), wd(heads);
  for (int h = 0; h < heads; ++h) {
    fp4_roundtrip_row(qidx + static_cast<int64_t>(h) * dim, dim, qhat.data() + h * dim);
    wd[h] = w[h];
  }
  std::vector<int64_t> cand;
  for (int64_t i = 0; i < n_pool; ++i) {
    if (pool[i] < 0) continue;
    for (int j = 0; j < block; ++j) {
      const int64_t p = static_cast<int64_t>(pool[i]) * block + j;
      if (p <= t) cand.push_back(p);
    }
  }
  std::vector<double> cs(cand.size());
  const double* qp = qhat.data();
  const double* wp = wd.data();
  const int64_t* cp = cand.data();
  double* csp = cs.data();
  parallel_for(static_cast<int64_t>(cand.size()), threads, [=](int64_t lo, int64_t hi) {
    double kh[512];
    for (int64_t i = lo; i < hi; ++i) {
      fp4_roundtrip_row(keys + cp[i] * dim, dim, kh);
      csp[i] = index_score(qp, wp, heads, dim, kh);
    }
  });
  if (pos_scores) {
    for (int64_t i = 0; i < n_pool * block; ++i) pos_scores[i] = -INFINITY;
    size_t c = 0;
    for (int64_t i = 0; i < n_pool; ++i) {
      if (pool[i] < 0) continue;
      for (int j = 0; j < block; ++j) {
        const int64_t p = static_cast<int64_t>(pool[i]) * block + j;
        if (p <= t) pos_scores[i * block + j] = cs[c++];
      }
    }
  }
  // Order of cand is ascending position when the pool is ascending, and ties
  // go to the lower position either way because selection compares positions.
  std::vector<int64_t> order(cand.size());
  std::iota(order.begin(), order.end(), 0);
  const int64_t m = std::min<int64_t>(k, static_cast<int64_t>(cand.size()));
  std::partial_sort(order.begin(), order.begin() + m, order.end(), [&](int64_t a, int64_t b) {
    return cs[a] > cs[b] || (cs[a] == cs[b] && cand[a] < cand[b]);
  });
  std::vector<int64_t> sel(static_cast<size_t>(m));
  for (int64_t i = 0; i < m; ++i) sel[i] = cand[order[i]];
  std::sort(sel.begin(), sel.end());
  for (int64_t i = 0; i < k; ++i) topk[i] = i < m ? static_cast<int32_t>(sel[i]) : -1;
  return m;
}

// Positions of the sliding window of query t (see the header's reading);
// returns the count written to out (<= window).
int64_t orc_window_positions(int64_t t, int64_t n_ctx, int64_t window, int64_t* out) {
  const int64_t lo = std::max<int64_t>({0, t - window + 1, n_ctx - window});
  int64_t m = 0;
  for (int64_t p = lo; p <= t; ++p) out[m++] = p;
  return m;
}

// Sparse attention of one query token.
//   q: bf16 [heads, dim]; main_rows: raw bf16 latents [n_main, dim] of the
//   selected positions (MXFP4-quantised here); win_rows: raw bf16 window
//   entries [n_win, dim] (FP8-quantised here).
//   out[heads, dim] = softmax(tau * q K^T) V with V = K; lse[heads] in the
//   natural-log units of the scaled logits (-inf when there are no keys).
void orc_sparse_attention(const uint16_t* q, int heads, int dim, const uint16_t* main_rows,
                          int64_t n_main, const uint16_t* win_rows, int64_t n_win, double tau,
                          double* out, double* lse) {
  const int64_t m = n_main + n_win;
  std::vector<double> K(static_cast<size_t>(m) * dim);
  for (int64_t i = 0; i < n_main; ++i) fp4_roundtrip_row(main_rows + i * dim, dim, K.data() + i * dim);
  for (int64_t i = 0; i < n_win; ++i)
    for (int c = 0; c < dim; ++c)
      K[(n_main + i) * dim + c] = e4m3_value(e4m3_encode(bf16_value(win_rows[i * dim + c])));
  std::vector<double> logit(static_cast<size_t>(m));
  for (int h = 0; h < heads; ++h) {
    double* o = out + static_cast<int64_t>(h) * dim;
    std::fill(o, o + dim, 0.0);
    if (m == 0) {
      lse[h] = -INFINITY;
      continue;
    }
    double mx = -INFINITY;
    for (int64_t i = 0; i < m; ++i) {
      double d = 0.0;
      for (int c = 0; c < dim; ++c) d += static_cast<double>(bf16_value(q[h * dim + c])) * K[i * dim + c];
      logit[i] = tau * d;
      mx = std::max(mx, logit[i]);
    }
    double den = 0.0;
    for (int64_t i = 0; i < m; ++i) {
      const double p = std::exp(logit[i] - mx);
      den += p;
      for (int c = 0; c < dim; ++c) o[c] += p * K[i * dim + c];
    }
    for (int c = 0; c < dim; ++c) o[c] /= den;
    lse[h] = mx + std::log(den);
  }
}

// Compressed entries ([RN] section 1 / [AB] section 3.1: the encoder's CSA2
// layers compress m = 2 tokens per entry; "DeepSeek-V4 model structure (7)",
// KV cache of hybrid attention: the compressor keeps an unfinished entry's
// tail tokens and their compression weights as state). The pages give no
// formula; per channel c of entry e:
//   out_c = sum_i exp(z_ic - zmax_c) x_ic / sum_i exp(z_ic - zmax_c),
// i over the entry's m tokens, in fp64, rounded once to bf16.
//   x, z: bf16 [n, m, dim] candidates and logits; out: bf16 [n, dim].
void orc_compress(const uint16_t* x, const uint16_t* z, int m, int dim, int64_t n, uint16_t* out) {
  for (int64_t e = 0; e < n; ++e) {
    for (int c = 0; c < dim; ++c) {
      double zmax = -INFINITY;
      for (int i = 0; i < m; ++i) zmax = std::max(zmax, static_cast<double>(bf16_value(z[(e * m + i) * dim + c])));
      double num = 0.0, den = 0.0;
      for (int i = 0; i < m; ++i) {
        const double w = std::exp(static_cast<double>(bf16_value(z[(e * m + i) * dim + c])) - zmax);
        num += w * static_cast<double>(bf16_value(x[(e * m + i) * dim + c]));
        den += w;
      }
      out[e * dim + c] = bf16_round(num / den);
    }
  }
}

// Output de-rotation ("DeepSeek-V4 model structure (7): structure decides the
// system", closing summary: the output is rotated back to restore relative
// position). K = V carries the rotary position of its own entry on the last 64
// channels, as interleaved pairs (448 + 2i, 449 + 2i) rotated by p * theta_i,
// theta_i = 10000^(-2i/64). Rotating an output row's pairs by -t * theta_i,
// t the query position, leaves every value term rotated by (p - t) * theta_i:
// relative position. rows: [n, dim] fp64, in place.
void orc_output_derotate(double* rows, int64_t n, int dim, int64_t t) {
  for (int i = 0; i < 32; ++i) {
    const double theta = std::pow(10000.0, -2.0 * i / 64.0);
    const double a = -static_cast<double>(t) * theta;
    const double c = std::cos(a), s = std::sin(a);
    for (int64_t r = 0; r < n; ++r) {
      double* x = rows + r * dim + (dim - 64) + 2 * i;
      const double x0 = x[0], x1 = x[1];
      x[0] = x0 * c - x1 * s;
      x[1] = x0 * s + x1 * c;
    }
  }
}

}  // extern "C"
