// Seeded synthetic inputs for the CSA2 decode path.
//
// This module only draws numbers. It holds none of the method's arithmetic
// (no quantiser, no score, no selection, no attention): both the CPU oracle
// and the CUDA library consume what it writes, so it must not depend on
// either of them.
//
// Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable
// pseudorandom number generators", OOPSLA 2014), used counter-style. Every
// value is a pure function of (seed, tensor id, sequence, position, draw
// index), so the result does not depend on the thread count or on the order
// in which rows are produced.
//
//   key(seed, tensor, seq, pos) = mix(mix(mix(seed ^ (tensor << 48)) ^ seq) ^ pos)
//   draw(key, c)                = mix(key + (c + 1) * GAMMA)   (the (c+1)-th
//                                                               SplitMix64 output
//                                                               of a stream at key)
//   uniform u in [0,1)          = (draw >> 11) * 2^-53
//   normal pair (Box-Muller)    = sqrt(-2 ln u1) * (cos 2 pi u2, sin 2 pi u2),
//                                 u1 = ((draw(2i) >> 11) + 1) * 2^-53,
//                                 u2 = (draw(2i+1) >> 11) * 2^-53
//
// Latent recipe (the 512-channel post-RoPE entry of the decoder KV):
//   z_c ~ N(0,1); with probability 1e-3 (uniform of draw 1024 + c) z_c is
//   replaced by +-11.1 (sign = lowest bit of that draw); RMSNorm without gain,
//   x = z / sqrt(mean(z^2) + 1e-6), so that ||x||_2 <= sqrt(512); then RoPE on
//   the last 64 channels as interleaved pairs (448+2i, 449+2i), angle
//   pos * 10000^(-2i/64). All of it in fp64, then rounded to bf16 (RNE).
//
// Compile with -ffp-contract=off so that x86 and Arm hosts give the same bits.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

constexpr uint64_t GAMMA = 0x9E3779B97F4A7C15ull;

inline uint64_t mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

inline uint64_t row_key(uint64_t seed, uint32_t tensor, int64_t seq, int64_t pos) {
  uint64_t k = mix(seed ^ (static_cast<uint64_t>(tensor) << 48));
  k = mix(k ^ static_cast<uint64_t>(seq));
  return mix(k ^ static_cast<uint64_t>(pos));
}

inline uint64_t draw(uint64_t key, uint64_t c) { return mix(key + (c + 1) * GAMMA); }

inline double unit(uint64_t d) { return static_cast<double>(d >> 11) * 0x1.0p-53; }

inline void normal_pair(uint64_t key, uint64_t i, double* z0, double* z1) {
  const double u1 = (static_cast<double>(draw(key, 2 * i) >> 11) + 1.0) * 0x1.0p-53;
  const double u2 = unit(draw(key, 2 * i + 1));
  const double r = std::sqrt(-2.0 * std::log(u1));
  const double a = 2.0 * M_PI * u2;
  *z0 = r * std::cos(a);
  *z1 = r * std::sin(a);
}

// fp32 -> bf16, round to nearest even (finite inputs only; the recipe makes no
// non-finite values).
inline uint16_t to_bf16(double v) {
  float f = static_cast<float>(v);
  uint32_t u;
  std::memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

template <class F>
void parallel_rows(int64_t n, int threads, F&& f) {
  if (threads < 1) threads = 1;
  if (n < 256 || threads == 1) {
    f(0, n);
    return;
  }
  std::vector<std::thread> pool;
  const int64_t chunk = (n + threads - 1) / threads;
  for (int t = 0; t < threads; ++t) {
    const int64_t lo = t * chunk, hi = std::min<int64_t>(n, lo + chunk);
    if (lo >= hi) break;
    pool.emplace_back([&f, lo, hi] { f(lo, hi); });
  }
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

// Rows (seq, pos0 + r) for r < n, `dim` i.i.d. N(0,1) values each, as bf16.
void synth_normal_bf16(uint64_t seed, uint32_t tensor, int64_t seq, int64_t pos0, int64_t n,
                       int dim, uint16_t* out, int threads) {
  parallel_rows(n, threads, [=](int64_t lo, int64_t hi) {
    for (int64_t r = lo; r < hi; ++r) {
      const uint64_t key = row_key(seed, tensor, seq, pos0 + r);
      for (int i = 0; i < dim / 2; ++i) {
        double z0, z1;
        normal_pair(key, i, &z0, &z1);
        out[r * dim + 2 * i] = to_bf16(z0);
        out[r * dim + 2 * i + 1] = to_bf16(z1);
      }
    }
  });
}

// Same values as synth_normal_bf16 for an explicit list of (seq, pos) rows.
void synth_normal_bf16_rows(uint64_t seed, uint32_t tensor, const int64_t* seq,
                            const int64_t* pos, int64_t n, int dim, uint16_t* out, int threads) {
  parallel_rows(n, threads, [=](int64_t lo, int64_t hi) {
    for (int64_t r = lo; r < hi; ++r) {
      const uint64_t key = row_key(seed, tensor, seq[r], pos[r]);
      for (int i = 0; i < dim / 2; ++i) {
        double z0, z1;
        normal_pair(key, i, &z0, &z1);
        out[r * dim + 2 * i] = to_bf16(z0);
        out[r * dim + 2 * i + 1] = to_bf16(z1);
      }
    }
  });
}

static void latent_row(uint64_t seed, uint32_t tensor, int64_t seq, int64_t pos, uint16_t* o) {
  const uint64_t key = row_key(seed, tensor, seq, pos);
  double z[512];
  for (int i = 0; i < 256; ++i) normal_pair(key, i, &z[2 * i], &z[2 * i + 1]);
  for (int c = 0; c < 512; ++c) {
    const uint64_t d = draw(key, 1024 + c);
    if (unit(d) < 1e-3) z[c] = (d & 1u) ? -11.1 : 11.1;
  }
  double ms = 0.0;
  for (int c = 0; c < 512; ++c) ms += z[c] * z[c];
  const double inv = 1.0 / std::sqrt(ms / 512.0 + 1e-6);
  for (int c = 0; c < 512; ++c) z[c] *= inv;
  for (int i = 0; i < 32; ++i) {
    const double theta = std::pow(10000.0, -2.0 * i / 64.0);
    const double a = static_cast<double>(pos) * theta;
    const double cs = std::cos(a), sn = std::sin(a);
    const double x0 = z[448 + 2 * i], x1 = z[449 + 2 * i];
    z[448 + 2 * i] = x0 * cs - x1 * sn;
    z[449 + 2 * i] = x0 * sn + x1 * cs;
  }
  for (int c = 0; c < 512; ++c) o[c] = to_bf16(z[c]);
}

// Rows (seq, pos0 + r): 512-channel latents per the recipe above, bf16.
void synth_latent_bf16(uint64_t seed, uint32_t tensor, int64_t seq, int64_t pos0, int64_t n,
                       uint16_t* out, int threads) {
  parallel_rows(n, threads, [=](int64_t lo, int64_t hi) {
    for (int64_t r = lo; r < hi; ++r) latent_row(seed, tensor, seq, pos0 + r, out + r * 512);
  });
}

// Latents for an explicit list of (seq, pos) rows.
void synth_latent_bf16_rows(uint64_t seed, uint32_t tensor, const int64_t* seq,
                            const int64_t* pos, int64_t n, uint16_t* out, int threads) {
  parallel_rows(n, threads, [=](int64_t lo, int64_t hi) {
    for (int64_t r = lo; r < hi; ++r) latent_row(seed, tensor, seq[r], pos[r], out + r * 512);
  });
}

// Rows (seq, pos0 + r), `dim` values uniform in [lo, hi), fp32.
void synth_uniform_f32(uint64_t seed, uint32_t tensor, int64_t seq, int64_t pos0, int64_t n,
                       int dim, double lo, double hi, float* out) {
  for (int64_t r = 0; r < n; ++r) {
    const uint64_t key = row_key(seed, tensor, seq, pos0 + r);
    for (int c = 0; c < dim; ++c)
      out[r * dim + c] = static_cast<float>(lo + (hi - lo) * unit(draw(key, c)));
  }
}

// k distinct integers drawn uniformly without replacement from [0, range),
// written ascending (Floyd's algorithm, driven by the (seq, pos) stream).
// If k >= range every integer of the range is written. Returns the count.
int64_t synth_sample_sorted(uint64_t seed, uint32_t tensor, int64_t seq, int64_t pos,
                            int64_t range, int64_t k, int32_t* out) {
  if (range <= 0) return 0;
  if (k >= range) {
    for (int64_t i = 0; i < range; ++i) out[i] = static_cast<int32_t>(i);
    return range;
  }
  const uint64_t key = row_key(seed, tensor, seq, pos);
  std::vector<uint8_t> taken(static_cast<size_t>(range), 0);
  int64_t c = 0;
  for (int64_t j = range - k; j < range; ++j, ++c) {
    const int64_t t = static_cast<int64_t>(draw(key, c) % static_cast<uint64_t>(j + 1));
    if (!taken[t]) taken[t] = 1; else taken[j] = 1;
  }
  int64_t m = 0;
  for (int64_t i = 0; i < range; ++i)
    if (taken[i]) out[m++] = static_cast<int32_t>(i);
  return m;
}

}  // extern "C"
