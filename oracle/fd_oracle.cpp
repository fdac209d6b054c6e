// FP64 CPU oracle for single-token decode attention over a position-addressed
// bf16 KV cache.
//
// TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or load
// this file; only the test suite, the smoke check and the benchmark's CPU
// baseline leg do. It shares no code, header, table or constant with the CUDA
// library.
//
// What it computes follows "Hand-Writing Gemma 4 Flash-Decoding + an FP4
// Matvec Bonus (Part 2)", section "One KV head breaks the textbook":
//   * one query token per sequence; Q head h belongs to the KV group
//     kvh = h / (NH / NKV) (the [B,1,NH*HS] and [B*NKV,GS,HS] layouts are the
//     same bytes, so the groups are contiguous runs of Q heads);
//   * the cache is addressed by absolute position: position pos lives in slot
//     pos % capacity;
//   * only the live band [max(0, len - window), len) takes part.
// and the same page's section "The test that catches what parity misses":
// an FP64 host reference over the bf16 values exactly as stored.
//
// Readings taken where the page is silent:
//   * window <= 0 means "no window";
//   * a cache holds at most `capacity` positions, so the band is clamped to
//     [max(0, len - min(W, capacity)), len);
//   * len == 0 gives an all-zero output (empty softmax);
//   * the scale is applied to the q.k dot product before the softmax.
//
// The oracle is the plain definition written out: gather the band's K and V
// rows into contiguous arrays, score every row, take the maximum, then the
// two-pass softmax-weighted sum of V. No tiling, no online rescale.
//
// A second function restates the split form (partition the band into S
// contiguous pieces, keep an unnormalised (O, m, l) per piece, merge) in FP64.
// It exists so the tests can show that the merge algebra is exact; the plain
// function above is the oracle proper.
//
// A third computes the same attention over an FP8 (E4M3) cache: the same
// page's section "What we'd tell the next person" says FP8 KV storage needs
// no special hardware and is dequantised inline: the type a cache is stored
// in need not be the type the arithmetic runs in. Reading taken: K and V are stored as E4M3 codes with one
// fp32 scale per (sequence, KV head) for K and one for V; the value of a code
// is its E4M3 number times that scale. E4M3 (1 sign, 4 exponent bits with
// bias 7, 3 mantissa bits; exponent field 0 = subnormal; code x111_1111 =
// NaN; no infinity) is decoded from that definition.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

double bf16_bits_to_double(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

struct Problem {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  const int32_t* lens;
  int B, NH, NKV, HS, capacity, window;
  double scale;
  const uint8_t* want;  // optional: which (b, h) outputs to compute
  // FP8 cache (k8/v8 non-null): E4M3 codes and per-(b, kvh) fp32 scales
  const uint8_t* k8 = nullptr;
  const uint8_t* v8 = nullptr;
  const float* k_scale = nullptr;
  const float* v_scale = nullptr;
};

// Value of an E4M3 code: (-1)^s * 2^(e-7) * (1 + m/8) for e > 0,
// (-1)^s * 2^-6 * (m/8) for e = 0, NaN for e = 15 and m = 7.
double e4m3_to_double(uint8_t code) {
  const int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return std::numeric_limits<double>::quiet_NaN();
  const double mag = e == 0 ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

// Live band of one sequence: positions [lo, hi).
void live_band(const Problem& p, int len, int64_t* lo, int64_t* hi) {
  int64_t w = p.window > 0 ? p.window : std::numeric_limits<int32_t>::max();
  int64_t keep = std::min<int64_t>(w, p.capacity);
  *hi = len;
  *lo = std::max<int64_t>(0, static_cast<int64_t>(len) - keep);
}

// Copies the K and V rows of the band's positions into contiguous arrays,
// position by position, in increasing position order.
void gather_band(const Problem& p, int b, int kvh, int64_t lo, int64_t hi,
                 std::vector<double>& kb, std::vector<double>& vb) {
  const int64_t n = hi - lo;
  kb.assign(static_cast<size_t>(n * p.HS), 0.0);
  vb.assign(static_cast<size_t>(n * p.HS), 0.0);
  for (int64_t i = 0; i < n; ++i) {
    const int64_t pos = lo + i;
    const int64_t slot = pos % p.capacity;
    const int64_t row = (static_cast<int64_t>(b) * p.NKV + kvh) * p.capacity + slot;
    if (p.k8) {
      const double ks = p.k_scale[static_cast<int64_t>(b) * p.NKV + kvh];
      const double vs = p.v_scale[static_cast<int64_t>(b) * p.NKV + kvh];
      for (int d = 0; d < p.HS; ++d) {
        kb[i * p.HS + d] = e4m3_to_double(p.k8[row * p.HS + d]) * ks;
        vb[i * p.HS + d] = e4m3_to_double(p.v8[row * p.HS + d]) * vs;
      }
      continue;
    }
    for (int d = 0; d < p.HS; ++d) {
      kb[i * p.HS + d] = bf16_bits_to_double(p.k[row * p.HS + d]);
      vb[i * p.HS + d] = bf16_bits_to_double(p.v[row * p.HS + d]);
    }
  }
}

// Plain softmax attention of one query row over the gathered band.
void attend_one(const Problem& p, int b, int h, double* out) {
  const int group = p.NH / p.NKV;
  const int kvh = h / group;
  const int len = p.lens[b];
  int64_t lo, hi;
  live_band(p, len, &lo, &hi);
  const int64_t n = hi - lo;
  double* o = out + (static_cast<int64_t>(b) * p.NH + h) * p.HS;
  for (int d = 0; d < p.HS; ++d) o[d] = 0.0;
  if (n <= 0) return;

  std::vector<double> kb, vb;
  gather_band(p, b, kvh, lo, hi, kb, vb);

  std::vector<double> q(p.HS);
  const uint16_t* qrow = p.q + (static_cast<int64_t>(b) * p.NH + h) * p.HS;
  for (int d = 0; d < p.HS; ++d) q[d] = bf16_bits_to_double(qrow[d]);

  std::vector<double> s(static_cast<size_t>(n));
  for (int64_t i = 0; i < n; ++i) {
    double dot = 0.0;
    for (int d = 0; d < p.HS; ++d) dot += q[d] * kb[i * p.HS + d];
    s[i] = p.scale * dot;
  }
  double m = s[0];
  for (int64_t i = 1; i < n; ++i) m = std::max(m, s[i]);
  // std::max drops a NaN that is not the first argument; keep NaN visible.
  for (int64_t i = 0; i < n; ++i)
    if (std::isnan(s[i])) m = s[i];

  double denom = 0.0;
  std::vector<double> w(static_cast<size_t>(n));
  for (int64_t i = 0; i < n; ++i) {
    w[i] = std::exp(s[i] - m);
    denom += w[i];
  }
  for (int64_t i = 0; i < n; ++i)
    for (int d = 0; d < p.HS; ++d) o[d] += w[i] * vb[i * p.HS + d];
  for (int d = 0; d < p.HS; ++d) o[d] /= denom;
}

// Split form: the band cut into `splits` contiguous pieces of near-equal size,
// an unnormalised partial per piece, then the online-softmax merge.
void attend_one_split(const Problem& p, int b, int h, int splits, double* out) {
  const int group = p.NH / p.NKV;
  const int kvh = h / group;
  const int len = p.lens[b];
  int64_t lo, hi;
  live_band(p, len, &lo, &hi);
  const int64_t n = hi - lo;
  double* o = out + (static_cast<int64_t>(b) * p.NH + h) * p.HS;
  for (int d = 0; d < p.HS; ++d) o[d] = 0.0;
  if (n <= 0) return;

  std::vector<double> kb, vb;
  gather_band(p, b, kvh, lo, hi, kb, vb);
  std::vector<double> q(p.HS);
  const uint16_t* qrow = p.q + (static_cast<int64_t>(b) * p.NH + h) * p.HS;
  for (int d = 0; d < p.HS; ++d) q[d] = bf16_bits_to_double(qrow[d]);

  const double neg_inf = -std::numeric_limits<double>::infinity();
  std::vector<double> part_o(static_cast<size_t>(splits) * p.HS, 0.0);
  std::vector<double> part_m(splits, neg_inf), part_l(splits, 0.0);
  for (int s = 0; s < splits; ++s) {
    const int64_t a = n * s / splits, e = n * (s + 1) / splits;
    if (a >= e) continue;  // an empty piece keeps m = -inf, l = 0, O = 0
    std::vector<double> sc(static_cast<size_t>(e - a));
    for (int64_t i = a; i < e; ++i) {
      double dot = 0.0;
      for (int d = 0; d < p.HS; ++d) dot += q[d] * kb[i * p.HS + d];
      sc[i - a] = p.scale * dot;
    }
    double m = *std::max_element(sc.begin(), sc.end());
    double l = 0.0;
    for (int64_t i = a; i < e; ++i) {
      const double wi = std::exp(sc[i - a] - m);
      l += wi;
      for (int d = 0; d < p.HS; ++d) part_o[s * p.HS + d] += wi * vb[i * p.HS + d];
    }
    part_m[s] = m;
    part_l[s] = l;
  }
  double big_m = neg_inf;
  for (int s = 0; s < splits; ++s) big_m = std::max(big_m, part_m[s]);
  double big_l = 0.0;
  for (int s = 0; s < splits; ++s) {
    if (part_l[s] == 0.0) continue;
    const double c = std::exp(part_m[s] - big_m);
    big_l += c * part_l[s];
    for (int d = 0; d < p.HS; ++d) o[d] += c * part_o[s * p.HS + d];
  }
  for (int d = 0; d < p.HS; ++d) o[d] /= big_l;
}

int check_args(const Problem& p, double* out) {
  if (!p.q || !p.lens || !out) return 1;
  if (p.k8 ? (!p.v8 || !p.k_scale || !p.v_scale) : (!p.k || !p.v)) return 1;
  if (p.B < 0 || p.NH <= 0 || p.NKV <= 0 || p.HS <= 0 || p.capacity <= 0) return 1;
  if (p.NH % p.NKV != 0) return 1;
  for (int b = 0; b < p.B; ++b)
    if (p.lens[b] < 0) return 1;
  return 0;
}

template <class Fn>
void for_each_row(const Problem& p, int nthreads, Fn fn) {
  const int64_t total = static_cast<int64_t>(p.B) * p.NH;
  if (nthreads <= 0) nthreads = static_cast<int>(std::max(1u, std::thread::hardware_concurrency()));
  nthreads = static_cast<int>(std::min<int64_t>(nthreads, std::max<int64_t>(1, total)));
  std::vector<std::thread> pool;
  for (int t = 0; t < nthreads; ++t) {
    pool.emplace_back([&, t] {
      for (int64_t r = t; r < total; r += nthreads) {
        if (p.want && !p.want[r]) continue;
        fn(static_cast<int>(r / p.NH), static_cast<int>(r % p.NH));
      }
    });
  }
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

// out: float64 [B][NH][HS]. want: nullable uint8 [B*NH]; rows with want == 0
// are left untouched. nthreads <= 0 uses every hardware thread.
// Returns 0 on success, 1 on invalid arguments.
int fd_oracle_decode(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                     const int32_t* lens, int B, int NH, int NKV, int HS,
                     int capacity, int window, double scale,
                     const uint8_t* want, int nthreads, double* out) {
  Problem p{q, k, v, lens, B, NH, NKV, HS, capacity, window, scale, want};
  if (check_args(p, out)) return 1;
  for_each_row(p, nthreads, [&](int b, int h) { attend_one(p, b, h, out); });
  return 0;
}

// The same over an FP8 (E4M3) cache: k8/v8 codes [B][NKV][capacity][HS],
// k_scale/v_scale fp32 [B][NKV].
int fd_oracle_decode_fp8(const uint16_t* q, const uint8_t* k8, const uint8_t* v8, const float* k_scale,
                         const float* v_scale, const int32_t* lens, int B, int NH, int NKV, int HS,
                         int capacity, int window, double scale, const uint8_t* want, int nthreads,
                         double* out) {
  Problem p{q, nullptr, nullptr, lens, B, NH, NKV, HS, capacity, window, scale, want, k8, v8, k_scale, v_scale};
  if (check_args(p, out)) return 1;
  for_each_row(p, nthreads, [&](int b, int h) { attend_one(p, b, h, out); });
  return 0;
}

// Value of every E4M3 code 0..255 (for the tests' decoding pin).
void fd_oracle_e4m3_table(double* out256) {
  for (int c = 0; c < 256; ++c) out256[c] = e4m3_to_double(static_cast<uint8_t>(c));
}

// FP64 restatement of the split form with `splits` near-equal pieces.
int fd_oracle_decode_split(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                           const int32_t* lens, int B, int NH, int NKV, int HS,
                           int capacity, int window, double scale, int splits,
                           int nthreads, double* out) {
  Problem p{q, k, v, lens, B, NH, NKV, HS, capacity, window, scale, nullptr};
  if (check_args(p, out) || splits <= 0) return 1;
  for_each_row(p, nthreads, [&](int b, int h) { attend_one_split(p, b, h, splits, out); });
  return 0;
}

}  // extern "C"
