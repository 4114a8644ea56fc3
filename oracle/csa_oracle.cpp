// CPU oracle for the compressed-sparse-attention KV Compressor.
//
// TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
// benchmark's CPU-baseline leg, never by the product path.  Plain loops, no
// blocking or fusion; threads only split independent tokens, groups or
// sequences.  Page citations are given per function (see csa_oracle.h for
// the page keys [V41], [RUST], [CSA4]).
#include "csa_oracle.h"

#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------------------
// Number formats, written from the format definitions.
//
// Every rounding below uses one recipe: pick the quantum (spacing of
// representable values) of the binade holding |v|, divide (exact: a power of
// two), round to the nearest integer with ties to even (std::nearbyint in the
// default rounding mode), multiply back.

double quantum_round(double a, double quantum) { return std::nearbyint(a / quantum) * quantum; }

// binade exponent E with 2^E <= a < 2^(E+1), for a > 0
int binade(double a) {
  int e;
  std::frexp(a, &e);  // a = m * 2^e, m in [0.5, 1)
  return e - 1;
}

uint32_t f32_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return u;
}

float f32_from_bits(uint32_t u) {
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// bf16: 1 sign, 8 exponent (bias 127), 7 mantissa bits; the upper half of a float32.
uint16_t bf16_round(double v) {
  if (std::isnan(v)) return 0x7FC0;
  const uint16_t sign = std::signbit(v) ? 0x8000 : 0;
  double a = std::fabs(v);
  if (a == 0.0) return sign;
  // largest finite bf16 is (2 - 2^-7) * 2^127; the midpoint to 2^128 rounds up to inf
  if (a >= std::ldexp(2.0 - std::ldexp(1.0, -8), 127)) return sign | 0x7F80;
  int e = binade(a);
  double q = e < -126 ? std::ldexp(1.0, -133) : std::ldexp(1.0, e - 7);
  double r = quantum_round(a, q);  // exactly a bf16 value, so exact in float32
  return sign | (uint16_t)(f32_bits((float)r) >> 16);
}

double bf16_value(uint16_t h) { return (double)f32_from_bits((uint32_t)h << 16); }

// e4m3 ("fn" flavour): 1 sign, 4 exponent (bias 7), 3 mantissa; largest finite 448,
// no infinities; smallest subnormal 2^-9.  Saturating: magnitudes rounding above 448 give 448.
uint8_t e4m3_round(double v) {
  if (std::isnan(v)) return 0x7F;
  const uint8_t sign = std::signbit(v) ? 0x80 : 0;
  double a = std::fabs(v);
  if (a == 0.0) return sign;
  int e = binade(a);
  if (e < -6) e = -6;  // subnormal range shares the quantum of the lowest normal binade
  double r = quantum_round(a, std::ldexp(1.0, e - 3));
  if (r > 448.0) r = 448.0;
  if (r == 0.0) return sign;
  int er = binade(r);
  if (er < -6) return sign | (uint8_t)(r / std::ldexp(1.0, -9));  // subnormal: mantissa * 2^-9
  int mant = (int)((r / std::ldexp(1.0, er) - 1.0) * 8.0);
  return sign | (uint8_t)((er + 7) << 3) | (uint8_t)mant;
}

double e4m3_value(uint8_t b) {
  int s = b >> 7, ex = (b >> 3) & 15, m = b & 7;
  if (ex == 15 && m == 7) return std::numeric_limits<double>::quiet_NaN();
  double mag = ex == 0 ? m * std::ldexp(1.0, -9) : (1.0 + m / 8.0) * std::ldexp(1.0, ex - 7);
  return s ? -mag : mag;
}

// e2m1: 1 sign, 2 exponent (bias 1), 1 mantissa.  Magnitudes by code 0..7:
// 0, 0.5, 1, 1.5, 2, 3, 4, 6.  [RUST] to_e2m1_rne: round onto this grid,
// ties to the even code, keeping the sign; the fp4 round trip saturates at 6.
const double kE2M1[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

uint8_t e2m1_round(float v) {
  const uint8_t sign = std::signbit(v) ? 0x8 : 0;
  double a = std::fabs((double)v);
  if (std::isnan(a)) return sign | 7;
  double q = a < 2.0 ? 0.5 : (a < 4.0 ? 1.0 : 2.0);  // quantum of the binade (0 and [1,2) share 0.5)
  double r = quantum_round(a, q);
  if (r > 6.0) r = 6.0;
  uint8_t code = 0;
  for (uint8_t k = 0; k < 8; ++k)
    if (kE2M1[k] == r) code = k;
  return sign | code;
}

double e2m1_value(uint8_t c) { return (c & 8 ? -1.0 : 1.0) * kE2M1[c & 7]; }

// [RUST] fp4_quant_e4m3_inplace with block LATENT_BLOCK = 16:
// amax floored at 6*2^-9; scale = amax/6 (float32 division) rounded through e4m3;
// each value divided by the scale (float32 division) to e2m1; dequantised
// (exact: <= 6 significant bits) and rounded to bf16.
void fp4_block(const uint16_t* in, uint8_t* codes, uint8_t* scale, uint16_t* out) {
  float amax = 0.0f;
  for (int i = 0; i < 16; ++i) amax = std::fmax(amax, (float)std::fabs(bf16_value(in[i])));
  const float floor_amax = std::ldexp(6.0f, -9);
  float sq = std::fmax(amax, floor_amax) / 6.0f;
  uint8_t sb = e4m3_round((double)sq);
  float s = (float)e4m3_value(sb);
  *scale = sb;
  for (int i = 0; i < 16; ++i) {
    float q = (float)bf16_value(in[i]) / s;
    uint8_t c = e2m1_round(q);
    if (codes) {
      if (i % 2 == 0)
        codes[i / 2] = c;
      else
        codes[i / 2] |= (uint8_t)(c << 4);
    }
    out[i] = bf16_round(e2m1_value(c) * (double)s);
  }
}

// [RUST] fp4_quant_e8m0_inplace with block FP4_BLOCK = 32 (the indexer's fp4 round trip):
// amax floored at 6*2^-126; scale = the power-of-two ceiling of amax/6 (float32 division),
// kept as an e8m0 byte (an 8-bit biased exponent, bias 127, value 2^(byte-127)); each value
// divided by the scale (exact: a power of two) to e2m1; dequantised and rounded to bf16.
void fp4_block_e8m0(const uint16_t* in, uint8_t* codes, uint8_t* scale, uint16_t* out) {
  float amax = 0.0f;
  for (int i = 0; i < 32; ++i) amax = std::fmax(amax, (float)std::fabs(bf16_value(in[i])));
  const float q = std::fmax(amax, std::ldexp(6.0f, -126)) / 6.0f;
  int e = binade((double)q);                 // 2^e <= q < 2^(e+1)
  if (std::ldexp(1.0, e) < (double)q) ++e;   // the smallest power of two >= q
  const double s = std::ldexp(1.0, e);
  *scale = (uint8_t)(e + 127);
  for (int i = 0; i < 32; ++i) {
    uint8_t c = e2m1_round((float)(bf16_value(in[i]) / s));
    if (codes) {
      if (i % 2 == 0)
        codes[i / 2] = c;
      else
        codes[i / 2] |= (uint8_t)(c << 4);
    }
    out[i] = bf16_round(e2m1_value(c) * s);
  }
}

// ---------------------------------------------------------------------------
// YaRN RoPE ([RUST] yarn_freqs_cis; [CSA4] "RoPE sub-dimension 64", applied
// after normalisation).  NTK-by-parts frequency correction of Peng et al.
// (2023): dims rotating fewer than beta_slow times over the original context
// are interpolated (divided by factor), dims rotating more than beta_fast times
// keep their frequency, a linear ramp in between.

double correction_dim(double rotations, int d, double base, int orig_len) {
  return d * std::log(orig_len / (rotations * 2.0 * M_PI)) / (2.0 * std::log(base));
}

void yarn_bounds(int d, double base, int orig_len, double beta_fast, double beta_slow, double* lo, double* hi) {
  double l = std::floor(correction_dim(beta_fast, d, base, orig_len));
  double h = std::ceil(correction_dim(beta_slow, d, base, orig_len));
  *lo = std::fmax(l, 0.0);
  *hi = std::fmin(h, (double)(d - 1));
}

void yarn_freqs(int d, double base, double factor, int orig_len, double beta_fast, double beta_slow,
                double* f) {
  double lo, hi;
  yarn_bounds(d, base, orig_len, beta_fast, beta_slow, &lo, &hi);
  if (hi == lo) hi += 0.001;
  for (int i = 0; i < d / 2; ++i) {
    double base_f = 1.0 / std::pow(base, (2.0 * i) / d);
    double ramp = std::fmin(std::fmax((i - lo) / (hi - lo), 0.0), 1.0);
    // ramp 0: keep the frequency; ramp 1: interpolate (divide by factor)
    f[i] = base_f * (1.0 - ramp) + (base_f / factor) * ramp;
  }
}

template <class F>
void parallel_for(int64_t n, int nthreads, F fn) {
  if (nthreads <= 1 || n < 2) {
    for (int64_t i = 0; i < n; ++i) fn(i);
    return;
  }
  if (nthreads > n) nthreads = (int)n;
  std::vector<std::thread> th;
  for (int t = 0; t < nthreads; ++t)
    th.emplace_back([=, &fn] {
      for (int64_t i = t; i < n; i += nthreads) fn(i);
    });
  for (auto& x : th) x.join();
}

}  // namespace

// ---------------------------------------------------------------------------

struct oracle_compressor {
  int dim, H, ratio, overlap;
  oracle_options opt;
  std::vector<float> wkv, wgate, gain;  // [C][dim], [C][dim], [H]
  std::vector<float> ape;               // gate positional bias [ratio][C], empty = none
  std::vector<double> freqs;            // [rope_dim/2]
  std::vector<float> kv_state, score_state;
  int width() const { return (1 + overlap) * H; }
  int slots() const { return overlap ? 8 : ratio; }  // overlap: 2 parities x 4
  int slot_width() const { return overlap ? 2 * H : H; }
  int scale_block() const { return opt.fp4 == 2 ? 32 : 16; }  // values per fp4 scale
};

namespace {

// [CSA4] "wgate(x) + positional bias": the gate logits of n projected tokens at positions
// p0, p0 + 1, ... get the bias row of their position within the group, ape[p % ratio][c],
// one float32 addition each.  No bias set: unchanged.
void add_gate_bias(const oracle_compressor* c, float* sp, int64_t n, int64_t p0) {
  if (c->ape.empty()) return;
  const int W = c->width();
  for (int64_t t = 0; t < n; ++t)
    for (int k = 0; k < W; ++k) sp[t * W + k] = sp[t * W + k] + c->ape[((p0 + t) % c->ratio) * W + k];
}

}  // namespace

extern "C" {

uint16_t oracle_bf16_from_f32(float v) { return bf16_round((double)v); }
uint16_t oracle_bf16_from_f64(double v) { return bf16_round(v); }
float oracle_bf16_to_f32(uint16_t h) { return (float)bf16_value(h); }
uint8_t oracle_e4m3_from_f32(float v) { return e4m3_round((double)v); }
double oracle_e4m3_to_f64(uint8_t b) { return e4m3_value(b); }
uint8_t oracle_e2m1_from_f32(float v) { return e2m1_round(v); }
double oracle_e2m1_to_f64(uint8_t c) { return e2m1_value(c); }

void oracle_fp4_e4m3(const uint16_t* in, int64_t n_blocks, uint8_t* codes, uint8_t* scales, uint16_t* out) {
  for (int64_t b = 0; b < n_blocks; ++b)
    fp4_block(in + 16 * b, codes ? codes + 8 * b : nullptr, scales + b, out + 16 * b);
}

void oracle_fp4_e8m0(const uint16_t* in, int64_t n_blocks, uint8_t* codes, uint8_t* scales, uint16_t* out) {
  for (int64_t b = 0; b < n_blocks; ++b)
    fp4_block_e8m0(in + 32 * b, codes ? codes + 16 * b : nullptr, scales + b, out + 32 * b);
}

void oracle_yarn_freqs(int d, double base, double factor, int orig_len, double bf, double bs, double* f) {
  yarn_freqs(d, base, factor, orig_len, bf, bs, f);
}

void oracle_yarn_bounds(int d, double base, int orig_len, double bf, double bs, double* lo, double* hi) {
  yarn_bounds(d, base, orig_len, bf, bs, lo, hi);
}

// [RUST] linear_f32: x . w^T, w laid out [out_dim][in_dim]; [V41] x.float() then wkv(x).
// Each output is the exact dot product (products of a bf16 and a float32 are
// exact in double) accumulated in double and rounded once to float32.
void oracle_linear(const uint16_t* x, int64_t M, int dim, const float* w, int C, float* out, int nthreads) {
  parallel_for(M, nthreads, [&](int64_t t) {
    std::vector<double> xr(dim);
    for (int k = 0; k < dim; ++k) xr[k] = bf16_value(x[t * dim + k]);
    for (int c = 0; c < C; ++c) {
      const float* wr = w + (int64_t)c * dim;
      double acc = 0.0;
      for (int k = 0; k < dim; ++k) acc += xr[k] * (double)wr[k];
      out[t * C + c] = (float)acc;
    }
  });
}

// [V41] pooling formula k^p_j = sum_i softmax_i(g_i) (.) k_i, per feature, and
// (kv * score.softmax(dim=2)).sum(dim=2).  Candidate i of feature h is kv[i*H+h].
void oracle_pool(const float* kv, const float* score, int n, int H, float* out, double* weights) {
  for (int h = 0; h < H; ++h) {
    double m = -std::numeric_limits<double>::infinity();
    for (int i = 0; i < n; ++i) m = std::fmax(m, (double)score[i * H + h]);
    double den = 0.0, num = 0.0;
    for (int i = 0; i < n; ++i) {
      double e = std::exp((double)score[i * H + h] - m);  // exp(-inf) = 0 for padded slots
      den += e;
      num += e * (double)kv[i * H + h];
    }
    out[h] = (float)(num / den);  // the pooled result is float32 ([V41] "Computed in float32")
    if (weights)
      for (int i = 0; i < n; ++i) weights[i * H + h] = std::exp((double)score[i * H + h] - m) / den;
  }
}

// [V41] norm(kv.to(bf16)); [CSA4] "normalized, rotary position is applied";
// [RUST] the pooled result is rounded to bf16 for the RMSNorm.
void oracle_epilogue(const oracle_compressor* c, const float* pooled, int64_t pos, uint16_t* prequant) {
  const int H = c->H;
  std::vector<double> u(H);
  double ss = 0.0;
  for (int h = 0; h < H; ++h) {
    u[h] = bf16_value(bf16_round((double)pooled[h]));
    ss += u[h] * u[h];
  }
  double inv = 1.0 / std::sqrt(ss / H + c->opt.eps);
  for (int h = 0; h < H; ++h) prequant[h] = bf16_round(u[h] * inv * (double)c->gain[h]);
  const int rd = c->opt.rope_dim;
  for (int i = 0; rd > 0 && i < rd / 2; ++i) {
    int ia = H - rd + 2 * i, ib = ia + 1;  // adjacent pairs of the trailing rotary slice
    double a = bf16_value(prequant[ia]), b = bf16_value(prequant[ib]);
    double th = (double)pos * c->freqs[i];
    double cs = std::cos(th), sn = std::sin(th);
    prequant[ia] = bf16_round(a * cs - b * sn);
    prequant[ib] = bf16_round(a * sn + b * cs);
  }
}

oracle_compressor* oracle_create(int dim, int H, int ratio, int overlap, const oracle_options* opt) {
  if (dim <= 0 || H <= 0 || H % 16 != 0 || ratio < 1 || (overlap && ratio != 4) || !opt) return nullptr;
  if (opt->rope_dim < 0 || opt->rope_dim % 2 || opt->rope_dim > H || opt->max_batch < 1) return nullptr;
  if (opt->fp4 < 0 || opt->fp4 > 2 || (opt->fp4 == 2 && H % 32)) return nullptr;
  auto* c = new oracle_compressor();
  c->dim = dim;
  c->H = H;
  c->ratio = ratio;
  c->overlap = overlap ? 1 : 0;
  c->opt = *opt;
  if (opt->rope_dim > 0) {
    c->freqs.resize(opt->rope_dim / 2);
    yarn_freqs(opt->rope_dim, opt->rope_base, opt->rope_factor, opt->rope_orig_len, opt->beta_fast,
               opt->beta_slow, c->freqs.data());
  }
  int64_t n = oracle_state_elems(c);
  c->kv_state.assign(n, 0.0f);
  c->score_state.assign(n, -std::numeric_limits<float>::infinity());
  return c;
}

void oracle_destroy(oracle_compressor* c) { delete c; }

void oracle_set_weights(oracle_compressor* c, const float* wkv, const float* wgate, const float* gain) {
  int64_t n = (int64_t)c->width() * c->dim;
  c->wkv.assign(wkv, wkv + n);
  if (wgate)
    c->wgate.assign(wgate, wgate + n);
  else
    c->wgate.assign(n, 0.0f);  // ratio 1: the gate does not matter (softmax over one candidate)
  c->gain.assign(gain, gain + c->H);
}

void oracle_set_gate_bias(oracle_compressor* c, const float* ape) {
  if (ape)
    c->ape.assign(ape, ape + (int64_t)c->ratio * c->width());
  else
    c->ape.clear();
}

int64_t oracle_state_elems(const oracle_compressor* c) {
  return (int64_t)c->opt.max_batch * c->slots() * c->slot_width();
}

void oracle_state_reset(oracle_compressor* c) {
  std::fill(c->kv_state.begin(), c->kv_state.end(), 0.0f);
  std::fill(c->score_state.begin(), c->score_state.end(), -std::numeric_limits<float>::infinity());
}

void oracle_state_export(const oracle_compressor* c, float* kv, float* score) {
  std::memcpy(kv, c->kv_state.data(), c->kv_state.size() * 4);
  std::memcpy(score, c->score_state.data(), c->score_state.size() * 4);
}

}  // extern "C"

namespace {

// Candidates of group j from projected rows.  Row 0 of kvp/sp is token t_base of the
// sequence; row stride W = width().  [V41] non-overlapped: tokens r*j .. r*j+r-1.  [CSA4] ratio 4
// overlapped: branch B (columns H..2H-1) of the previous group's 4 tokens, then branch A
// (columns 0..H-1) of the current group's 4 tokens; for j = 0 the previous branch is padded
// (score -inf, kv 0).
void gather_group(const oracle_compressor* c, const float* kvp, const float* sp, int64_t t_base, int64_t j,
                  float* kv, float* sc) {
  const int H = c->H, W = c->width(), r = c->ratio;
  auto row = [&](int64_t tok) { return (tok - t_base) * W; };
  if (!c->overlap) {
    for (int i = 0; i < r; ++i)
      for (int h = 0; h < H; ++h) {
        kv[i * H + h] = kvp[row(r * j + i) + h];
        sc[i * H + h] = sp[row(r * j + i) + h];
      }
    return;
  }
  for (int i = 0; i < 4; ++i)
    for (int h = 0; h < H; ++h) {
      if (j == 0) {
        kv[i * H + h] = 0.0f;
        sc[i * H + h] = -std::numeric_limits<float>::infinity();
      } else {
        kv[i * H + h] = kvp[row(4 * j - 4 + i) + H + h];
        sc[i * H + h] = sp[row(4 * j - 4 + i) + H + h];
      }
      kv[(4 + i) * H + h] = kvp[row(4 * j + i) + h];
      sc[(4 + i) * H + h] = sp[row(4 * j + i) + h];
    }
}

void finish_entry(const oracle_compressor* c, const float* pooled, int64_t pos, uint16_t* latent, uint8_t* codes,
                  uint8_t* scales, uint16_t* prequant) {
  const int H = c->H;
  std::vector<uint16_t> pq(H), lat(H);
  std::vector<uint8_t> cd(H / 2), sc(H / 16);
  oracle_epilogue(c, pooled, pos, pq.data());
  if (c->opt.fp4 == 1)  // the latent: e4m3 scales, block 16
    oracle_fp4_e4m3(pq.data(), H / 16, cd.data(), sc.data(), lat.data());
  else if (c->opt.fp4 == 2)  // the indexer's keys: power-of-two scales, block 32
    oracle_fp4_e8m0(pq.data(), H / 32, cd.data(), sc.data(), lat.data());
  else
    lat = pq;
  if (latent) std::memcpy(latent, lat.data(), H * 2);
  if (prequant) std::memcpy(prequant, pq.data(), H * 2);
  if (codes && c->opt.fp4) std::memcpy(codes, cd.data(), H / 2);
  if (scales && c->opt.fp4) std::memcpy(scales, sc.data(), H / c->scale_block());
}

float* state_row(std::vector<float>& st, const oracle_compressor* c, int b, int slot) {
  return st.data() + ((int64_t)b * c->slots() + slot) * c->slot_width();
}

}  // namespace

extern "C" {

int oracle_prefill(oracle_compressor* c, const uint16_t* x, int B, int N, int slot_offset, uint16_t* latent,
                   uint8_t* codes, uint8_t* scales, uint16_t* prequant, int nthreads) {
  if (!c || B < 1 || N < 1 || slot_offset < 0 || slot_offset + B > c->opt.max_batch || c->wkv.empty()) return -1;
  const int H = c->H, W = c->width(), r = c->ratio, D = c->dim;
  const int64_t G = N / r, rem = N % r;  // [V41] cutoff = seqlen - remainder; emit iff seqlen >= ratio
  const int ncand = c->overlap ? 8 : r;
  std::vector<float> kvp((int64_t)N * W), sp((int64_t)N * W);
  for (int b = 0; b < B; ++b) {
    const uint16_t* xs = x + (int64_t)b * N * D;
    oracle_linear(xs, N, D, c->wkv.data(), W, kvp.data(), nthreads);
    oracle_linear(xs, N, D, c->wgate.data(), W, sp.data(), nthreads);
    add_gate_bias(c, sp.data(), N, 0);
    parallel_for(G, nthreads, [&](int64_t j) {
      std::vector<float> kv((int64_t)ncand * H), sc((int64_t)ncand * H), pooled(H);
      gather_group(c, kvp.data(), sp.data(), 0, j, kv.data(), sc.data());
      oracle_pool(kv.data(), sc.data(), ncand, H, pooled.data(), nullptr);
      int64_t e = (int64_t)b * G + j;
      finish_entry(c, pooled.data(), r * j, latent ? latent + e * H : nullptr, codes ? codes + e * H / 2 : nullptr,
                   scales ? scales + e * H / c->scale_block() : nullptr, prequant ? prequant + e * H : nullptr);
    });
    // [V41] the trailing partial group waits in the state (slots 0..rem-1).
    const int sb = slot_offset + b, sw = c->slot_width();
    if (!c->overlap) {
      for (int i = 0; i < rem; ++i) {
        std::memcpy(state_row(c->kv_state, c, sb, i), &kvp[(G * r + i) * W], sw * 4);
        std::memcpy(state_row(c->score_state, c, sb, i), &sp[(G * r + i) * W], sw * 4);
      }
    } else {
      // Overlapped state: two parities of 4 slots, each slot the token's full 2H columns.
      // The group being filled (index G) lives in parity G%2; the last complete group
      // (G-1), whose branch B the next entry needs, in the other parity.
      const int q = (int)(G % 2);
      for (int i = 0; i < rem; ++i) {
        std::memcpy(state_row(c->kv_state, c, sb, 4 * q + i), &kvp[(G * 4 + i) * W], sw * 4);
        std::memcpy(state_row(c->score_state, c, sb, 4 * q + i), &sp[(G * 4 + i) * W], sw * 4);
      }
      for (int i = 0; i < 4; ++i) {
        float* k = state_row(c->kv_state, c, sb, 4 * (1 - q) + i);
        float* s = state_row(c->score_state, c, sb, 4 * (1 - q) + i);
        if (G >= 1) {
          std::memcpy(k, &kvp[((G - 1) * 4 + i) * W], sw * 4);
          std::memcpy(s, &sp[((G - 1) * 4 + i) * W], sw * 4);
        } else {  // no complete group yet: the previous branch is the padded one
          for (int h = 0; h < sw; ++h) {
            k[h] = 0.0f;
            s[h] = -std::numeric_limits<float>::infinity();
          }
        }
      }
    }
  }
  return (int)G;
}

int oracle_prefill_groups(const oracle_compressor* c, const uint16_t* x, int N, const int* groups, int ng,
                          uint16_t* latent, uint8_t* codes, uint8_t* scales, uint16_t* prequant, int nthreads) {
  if (!c || N < 1 || ng < 0 || c->wkv.empty()) return -1;
  const int H = c->H, W = c->width(), r = c->ratio, D = c->dim;
  const int ncand = c->overlap ? 8 : r;
  for (int g = 0; g < ng; ++g)
    if (groups[g] < 0 || (int64_t)(groups[g] + 1) * r > N) return -1;
  parallel_for(ng, nthreads, [&](int64_t g) {
    const int64_t j = groups[g];
    // project only the tokens the group reads: [r*j - r*overlap, r*j + r)
    const int64_t t0 = c->overlap && j > 0 ? 4 * j - 4 : r * j;
    const int64_t nt = r * j + r - t0;
    std::vector<float> kvp(nt * W), sp(nt * W);
    oracle_linear(x + t0 * D, nt, D, c->wkv.data(), W, kvp.data(), 1);
    oracle_linear(x + t0 * D, nt, D, c->wgate.data(), W, sp.data(), 1);
    add_gate_bias(c, sp.data(), nt, t0);
    std::vector<float> kv((int64_t)ncand * H), sc((int64_t)ncand * H), pooled(H);
    gather_group(c, kvp.data(), sp.data(), t0, j, kv.data(), sc.data());
    oracle_pool(kv.data(), sc.data(), ncand, H, pooled.data(), nullptr);
    finish_entry(c, pooled.data(), r * j, latent ? latent + g * H : nullptr, codes ? codes + g * H / 2 : nullptr,
                 scales ? scales + g * H / c->scale_block() : nullptr, prequant ? prequant + g * H : nullptr);
  });
  return ng;
}

// A prefill chunk that starts at start_pos > 0 (every sequence at the same position): the N
// tokens continue sequences whose earlier tokens went through prefill, chunks or decode.
// The pages define prefill only at start_pos 0 and decode one token at a time; [CSA4]
// "Prefill and decode use the same rule" fixes what a chunk must compute: the entries of the
// groups that complete inside [start_pos, start_pos + N), each pooled over its candidates
// whatever call projected them, and a state that later calls can continue from.  Candidates
// of earlier calls are read from the state slots the decode rule puts them in (non-overlapped:
// slot p % r; ratio 4 overlapped: parity (p / 4) % 2, slot p % 4).  The state then receives,
// as [V41]'s prefill branch does for its remainder, the new tokens of the unfinished group and
// (overlapped) of the last complete group; no other slot changes.  start_pos 0 is the prefill.
// Entries go to latent [B][G][H] etc., G = (start_pos + N) / r - start_pos / r.
int oracle_prefill_chunk(oracle_compressor* c, const uint16_t* x, int B, int N, int start_pos, int slot_offset,
                         uint16_t* latent, uint8_t* codes, uint8_t* scales, uint16_t* prequant, int nthreads) {
  if (start_pos == 0) return oracle_prefill(c, x, B, N, slot_offset, latent, codes, scales, prequant, nthreads);
  if (!c || B < 1 || N < 1 || start_pos < 0 || slot_offset < 0 || slot_offset + B > c->opt.max_batch ||
      c->wkv.empty())
    return -1;
  const int H = c->H, W = c->width(), r = c->ratio, D = c->dim, sw = c->slot_width();
  const int64_t p0 = start_pos, p1 = p0 + N;
  const int64_t g_first = p0 / r, g_end = p1 / r, G = g_end - g_first;
  const int ncand = c->overlap ? 8 : r;
  auto slot_of = [&](int64_t p) { return c->overlap ? (int)(4 * ((p / 4) % 2) + p % 4) : (int)(p % r); };
  std::vector<float> kvp((int64_t)N * W), sp((int64_t)N * W);
  for (int b = 0; b < B; ++b) {
    const int sb = slot_offset + b;
    const uint16_t* xs = x + (int64_t)b * N * D;
    oracle_linear(xs, N, D, c->wkv.data(), W, kvp.data(), nthreads);
    oracle_linear(xs, N, D, c->wgate.data(), W, sp.data(), nthreads);
    add_gate_bias(c, sp.data(), N, p0);
    // the kv / score row (W columns) of token p: this call's projection, or its state slot
    auto kv_row = [&](int64_t p) -> const float* {
      return p >= p0 ? &kvp[(p - p0) * W] : state_row(c->kv_state, c, sb, slot_of(p));
    };
    auto sc_row = [&](int64_t p) -> const float* {
      return p >= p0 ? &sp[(p - p0) * W] : state_row(c->score_state, c, sb, slot_of(p));
    };
    parallel_for(G, nthreads, [&](int64_t jj) {
      const int64_t g = g_first + jj;
      std::vector<float> kv((int64_t)ncand * H), sc((int64_t)ncand * H), pooled(H);
      for (int i = 0; i < (c->overlap ? 4 : r); ++i)
        for (int h = 0; h < H; ++h) {
          if (!c->overlap) {
            kv[i * H + h] = kv_row(r * g + i)[h];
            sc[i * H + h] = sc_row(r * g + i)[h];
            continue;
          }
          if (g == 0) {  // [CSA4] padded previous branch
            kv[i * H + h] = 0.0f;
            sc[i * H + h] = -std::numeric_limits<float>::infinity();
          } else {  // branch B (columns H..2H-1) of the previous group's tokens
            kv[i * H + h] = kv_row(4 * g - 4 + i)[H + h];
            sc[i * H + h] = sc_row(4 * g - 4 + i)[H + h];
          }
          kv[(4 + i) * H + h] = kv_row(4 * g + i)[h];  // branch A of the group's own tokens
          sc[(4 + i) * H + h] = sc_row(4 * g + i)[h];
        }
      oracle_pool(kv.data(), sc.data(), ncand, H, pooled.data(), nullptr);
      const int64_t e = (int64_t)b * G + jj;
      finish_entry(c, pooled.data(), r * g, latent ? latent + e * H : nullptr, codes ? codes + e * H / 2 : nullptr,
                   scales ? scales + e * H / c->scale_block() : nullptr, prequant ? prequant + e * H : nullptr);
    });
    // state: the new tokens of the unfinished group g_end and, overlapped, of group g_end - 1
    const int64_t keep_from = std::max(p0, (g_end - c->overlap) * r);
    for (int64_t p = keep_from; p < p1; ++p) {
      std::memcpy(state_row(c->kv_state, c, sb, slot_of(p)), &kvp[(p - p0) * W], sw * 4);
      std::memcpy(state_row(c->score_state, c, sb, slot_of(p)), &sp[(p - p0) * W], sw * 4);
    }
    if (c->overlap && g_end == 0)  // no complete group yet: the previous branch stays padded
      for (int i = 0; i < 4; ++i)
        for (int h = 0; h < sw; ++h) {
          state_row(c->kv_state, c, sb, 4 + i)[h] = 0.0f;
          state_row(c->score_state, c, sb, 4 + i)[h] = -std::numeric_limits<float>::infinity();
        }
  }
  return (int)G;
}

// [V41] decode branch (start_pos > 0, one token): slot = start_pos % ratio; pool over the
// state when (start_pos+1) % ratio == 0.  start_pos == 0 takes the prefill branch with one
// token.  [CSA4] "Prefill and decode use the same rule": at ratio 4 overlapped, the entry
// completing at p = 4j+3 pools branch B of group j-1 (other parity) and branch A of group j.
int oracle_decode(oracle_compressor* c, const uint16_t* x_tok, int B, const int32_t* start_pos, uint16_t* latent,
                  uint8_t* codes, uint8_t* scales, uint16_t* prequant, uint8_t* emitted, int nthreads) {
  if (!c || B < 1 || B > c->opt.max_batch || c->wkv.empty()) return -1;
  for (int b = 0; b < B; ++b)
    if (start_pos[b] < 0) return -1;
  const int H = c->H, W = c->width(), r = c->ratio, D = c->dim;
  std::vector<int> emit(B, 0);
  parallel_for(B, nthreads, [&](int64_t b) {
    const int64_t p = start_pos[b];
    const uint16_t* xt = x_tok + b * D;
    if (p == 0) {
      std::vector<uint16_t> lat(H), pq(H);
      std::vector<uint8_t> cd(H / 2), sc(H / 16);
      // a one-token prefill into slot b
      int g = oracle_prefill(c, xt, 1, 1, (int)b, lat.data(), cd.data(), sc.data(), pq.data(), 1);
      if (g > 0) {
        emit[b] = 1;
        if (latent) std::memcpy(latent + b * H, lat.data(), H * 2);
        if (prequant) std::memcpy(prequant + b * H, pq.data(), H * 2);
        if (codes && c->opt.fp4) std::memcpy(codes + b * H / 2, cd.data(), H / 2);
        if (scales && c->opt.fp4) std::memcpy(scales + b * H / c->scale_block(), sc.data(), H / c->scale_block());
      }
      return;
    }
    std::vector<float> kv(W), sc(W);
    oracle_linear(xt, 1, D, c->wkv.data(), W, kv.data(), 1);
    oracle_linear(xt, 1, D, c->wgate.data(), W, sc.data(), 1);
    add_gate_bias(c, sc.data(), 1, p);
    const int sw = c->slot_width();
    if (!c->overlap) {
      const int slot = (int)(p % r);
      std::memcpy(state_row(c->kv_state, c, (int)b, slot), kv.data(), sw * 4);
      std::memcpy(state_row(c->score_state, c, (int)b, slot), sc.data(), sw * 4);
      if ((p + 1) % r != 0) return;
      std::vector<float> pooled(H);
      oracle_pool(state_row(c->kv_state, c, (int)b, 0), state_row(c->score_state, c, (int)b, 0), r, H,
                  pooled.data(), nullptr);
      emit[b] = 1;
      finish_entry(c, pooled.data(), p + 1 - r, latent ? latent + b * H : nullptr,
                   codes ? codes + b * H / 2 : nullptr, scales ? scales + b * H / c->scale_block() : nullptr,
                   prequant ? prequant + b * H : nullptr);
      return;
    }
    const int q = (int)((p / 4) % 2), slot = (int)(p % 4);
    std::memcpy(state_row(c->kv_state, c, (int)b, 4 * q + slot), kv.data(), sw * 4);
    std::memcpy(state_row(c->score_state, c, (int)b, 4 * q + slot), sc.data(), sw * 4);
    if ((p + 1) % 4 != 0) return;
    std::vector<float> ck(8 * H), cs(8 * H), pooled(H);
    for (int i = 0; i < 4; ++i)
      for (int h = 0; h < H; ++h) {
        ck[i * H + h] = state_row(c->kv_state, c, (int)b, 4 * (1 - q) + i)[H + h];
        cs[i * H + h] = state_row(c->score_state, c, (int)b, 4 * (1 - q) + i)[H + h];
        ck[(4 + i) * H + h] = state_row(c->kv_state, c, (int)b, 4 * q + i)[h];
        cs[(4 + i) * H + h] = state_row(c->score_state, c, (int)b, 4 * q + i)[h];
      }
    oracle_pool(ck.data(), cs.data(), 8, H, pooled.data(), nullptr);
    emit[b] = 1;
    finish_entry(c, pooled.data(), p - 3, latent ? latent + b * H : nullptr, codes ? codes + b * H / 2 : nullptr,
                 scales ? scales + b * H / c->scale_block() : nullptr, prequant ? prequant + b * H : nullptr);
  });
  int n = 0;
  for (int b = 0; b < B; ++b) {
    if (emitted) emitted[b] = (uint8_t)emit[b];
    n += emit[b];
  }
  return n;
}

}  // extern "C"
