// ORACLE -- test infrastructure, not part of the product.
//
// A plain, slow CPU restatement of the rotated 4-bit KV-cache decode path of
// "Serving Kolibri-1 with a 4-bit KV cache" (sevren.ai), written to check the
// CUDA library against. Only tests/, __graft_entry__.smoke() and bench.py's CPU
// baseline leg may load it. It shares no code, header or table with the CUDA
// library, and the library never calls it.
//
// Precision: fp64 everywhere, except the two steps whose exact fp32 formula is
// part of the specification (the key/query prologue and the int4 quantiser),
// which are emulated bit for bit in fp32 because the 4-bit codes must match the
// GPU exactly. Attention is evaluated in fp64 on the dequantised cache.
//
// Readings taken where the page is silent (each also listed in the design notes):
//  * H is the Sylvester-ordered 128x128 Hadamard matrix; "a random sign per
//    column" is diag(s) on the right: R = H diag(s) / sqrt(128).
//  * s_j = +1 when the top bit of the j-th splitmix64 output of the seed is 0.
//  * the RMS norm is n(x) = x / sqrt(mean(x^2) + eps); no positional map sits
//    between the norm and the dot product (the full layers are read as NoPE).
//  * the fp16 offset rounds toward -inf and the fp16 scale toward +inf, so every
//    input lies on the code grid's span; codes round half to even.
//  * the softmax scale 1/sqrt(128) is applied to the scores, not folded.
//
// Parity pins: every function here is checked in tests/test_oracle_pins.py
// against closed forms, invariants or brute force; the page's attention-error
// percentages are real-model numbers and stay unpinned (see the claims test).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

// Planted-mistake switch for tests/test_oracle_mutations.py: a variant build with
// -DORACLE_MUTATION=n introduces one deliberate error so the test can show that
// some pin fails. The normal build has ORACLE_MUTATION == 0 and every MUT(n) is false.
#ifndef ORACLE_MUTATION
#define ORACLE_MUTATION 0
#endif
#define MUT(n) (ORACLE_MUTATION == (n))

namespace {

// ---------------------------------------------------------------- threading

template <class F>
void for_range(int64_t n, int threads, F f) {
  if (threads <= 1 || n < 2) {
    f((int64_t)0, n);
    return;
  }
  threads = (int)std::min<int64_t>(threads, n);
  std::vector<std::thread> pool;
  int64_t per = (n + threads - 1) / threads;
  for (int t = 0; t < threads; ++t) {
    int64_t a = t * per, b = std::min(n, a + per);
    if (a >= b) break;
    pool.emplace_back([=] { f(a, b); });
  }
  for (auto& th : pool) th.join();
}

// ---------------------------------------------------------------- splitmix64
// Published definition (Steele, Lea, Flood 2014): state += golden gamma, then
// the variant-13 finaliser.
uint64_t splitmix64_next(uint64_t& state) {
  state += 0x9E3779B97F4A7C15ull;
  uint64_t z = state;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// ---------------------------------------------------------------- fp16 / e4m3
// Rounding of an exactly known real value (held in a double) to a binary
// floating-point format with `sig` significant bits, smallest normal exponent
// `emin` (value 2^emin) and subnormal quantum 2^(emin - sig + 1).
// dir: 0 = nearest, ties to even; -1 = toward -inf; +1 = toward +inf.
double round_to_format(double x, int sig, int emin, int dir) {
  if (std::isnan(x) || std::isinf(x) || x == 0.0) return x;
  bool neg = x < 0;
  double m = neg ? -x : x;
  // rounding direction on the magnitude
  int mdir = dir == 0 ? 0 : ((neg && !MUT(10)) ? -dir : dir);
  int e;
  std::frexp(m, &e);              // m = f * 2^e, f in [0.5, 1): leading bit has weight 2^(e-1)
  int q = std::max(e - sig, emin - sig + 1);  // weight of the last kept bit
  double scaled = std::ldexp(m, -q);  // exact: power-of-two scaling of a double
  double fl = std::floor(scaled);
  double frac = scaled - fl;
  double r;
  if (mdir == 0) {
    if (frac > 0.5)
      r = fl + 1;
    else if (frac < 0.5)
      r = fl;
    else
      r = (std::fmod(fl, 2.0) == 0.0) ? fl : fl + 1;
  } else if (mdir < 0) {
    r = fl;
  } else {
    r = frac > 0 ? fl + 1 : fl;
  }
  double v = std::ldexp(r, q);
  return neg ? -v : v;
}

constexpr double kHalfMax = 65504.0;

// fp16 rounding of an fp32 value. Overflow follows IEEE: nearest and the
// outward direction go to infinity, the inward direction stops at 65504.
double fp16_round(float xf, int dir) {
  double x = (double)xf;
  if (std::isnan(x)) return x;
  double v = round_to_format(x, 11, -14, dir);
  if (std::fabs(v) > kHalfMax) {
    bool neg = v < 0;
    bool inward = (dir == -1 && !neg) || (dir == 1 && neg);
    double mag = (std::isinf(x) || !inward) ? std::numeric_limits<double>::infinity() : kHalfMax;
    v = neg ? -mag : mag;
  }
  return v;
}

uint16_t fp16_bits(double v) {
  uint16_t sign = std::signbit(v) ? 0x8000 : 0;
  double m = std::fabs(v);
  if (std::isnan(v)) return 0x7E00;
  if (std::isinf(m)) return sign | 0x7C00;
  if (m == 0.0) return sign;
  int e;
  double f = std::frexp(m, &e);  // m = f 2^e, f in [0.5,1) -> unbiased exponent e-1
  int ue = e - 1;
  (void)f;
  if (ue < -14) return sign | (uint16_t)std::ldexp(m, 24);  // subnormal: units of 2^-24
  uint16_t mant = (uint16_t)(std::ldexp(m, 10 - ue) - 1024.0);
  return sign | (uint16_t)((ue + 15) << 10) | mant;
}

double fp16_value(uint16_t h) {
  int s = h >> 15, ex = (h >> 10) & 31, mant = h & 1023;
  double v;
  if (ex == 31)
    v = mant ? std::numeric_limits<double>::quiet_NaN() : std::numeric_limits<double>::infinity();
  else if (ex == 0)
    v = std::ldexp((double)mant, -24);
  else
    v = std::ldexp(1024.0 + mant, ex - 25);
  return s ? -v : v;
}

// OCP FP8 E4M3 ("e4m3fn"): 4 significant bits, bias 7, no infinities,
// 0x7F/0xFF are NaN, largest finite 448. Conversion: nearest-even with
// saturation to +-448 (infinities saturate too); NaN stays NaN.
uint8_t e4m3_encode(float xf) {
  double x = (double)xf;
  uint8_t sign = std::signbit(x) ? 0x80 : 0;
  if (std::isnan(x)) return sign | 0x7F;
  double m = std::fabs(x);
  double v = std::isinf(m) ? 448.0 : round_to_format(m, 4, -6, 0);
  if (v > 448.0 && !MUT(9)) v = 448.0;
  if (v == 0.0) return sign;
  int e;
  std::frexp(v, &e);
  int ue = e - 1;
  if (ue < -6) return sign | (uint8_t)std::ldexp(v, 9);  // subnormal: units of 2^-9
  uint8_t mant = (uint8_t)(std::ldexp(v, 3 - ue) - 8.0);
  return sign | (uint8_t)((ue + 7) << 3) | mant;
}

double e4m3_value(uint8_t c) {
  int s = c >> 7, ex = (c >> 3) & 15, mant = c & 7;
  double v;
  if (ex == 15 && mant == 7)
    v = std::numeric_limits<double>::quiet_NaN();
  else if (ex == 0)
    v = std::ldexp((double)mant, -9);
  else
    v = std::ldexp(8.0 + mant, ex - 10);
  return s ? -v : v;
}

// ---------------------------------------------------------------- prologue
// fp32 specification of the per-vector prologue (section "What we do": the RMS
// norm and a fixed 128x128 matrix applied by one kernel). The arithmetic order
// below IS the specification; the CUDA kernel performs the same operations.
//   lanes l = 0..31 hold x[4l..4l+3]
//   t_l = fma(x3,x3, fma(x2,x2, fma(x1,x1, x0*x0)))
//   butterfly: for o in 16,8,4,2,1: t_l <- t_l + t_(l xor o); ss = t_0
//   inv = 1 / sqrt(ss/128 + eps)       (IEEE division and square root)
//   n_i = x_i * inv
//   y_j = fma chain over i = 0..127 of M[j][i] * n_i, starting from 0
// The normalisation n(x) of the specification above (shared by both prologue forms).
void normalize_one(const float* x, float eps, float* n) {
  float t[32];
  for (int l = 0; l < 32; ++l) {
    const float* p = x + 4 * l;
    float a = p[0] * p[0];
    a = std::fmaf(p[1], p[1], a);
    a = std::fmaf(p[2], p[2], a);
    a = std::fmaf(p[3], p[3], a);
    t[l] = a;
  }
  for (int o = 16; o >= 1; o >>= 1) {
    float u[32];
    for (int l = 0; l < 32; ++l) u[l] = t[l] + t[l ^ o];
    std::memcpy(t, u, sizeof(t));
  }
  float ss = t[0];
  float inv = MUT(6) ? 1.0f : 1.0f / std::sqrt(ss / 128.0f + eps);
  for (int i = 0; i < 128; ++i) n[i] = x[i] * inv;
}

void prologue_one(const float* M, const float* x, float eps, float* y) {
  float n[128];
  normalize_one(x, eps, n);
  for (int j = 0; j < 128; ++j) {
    float acc = 0.0f;
    for (int i = 0; i < 128; ++i) acc = std::fmaf(M[j * 128 + i], n[i], acc);
    y[j] = acc;
  }
}

// Second codec specification: the same rotation through a fast Walsh-Hadamard transform.
// Since R = H diag(s) / sqrt(128) (H Sylvester-ordered), R x = H (s * x) / sqrt(128) and
// R diag(g) x = H (s * g * x) / sqrt(128), computed in fp32 as
//   n = n(x) (as above);  u_i = w_i * n_i   (w = s for keys, w = fp32(s * g_q * g_k) for queries)
//   for h = 1, 2, 4, ..., 64, for every i with (i & h) == 0:
//       (u_i, u_{i+h}) <- (u_i + u_{i+h}, u_i - u_{i+h})
//   y_j = c * u_j with c = fp32(1 / sqrt(128)).
void prologue_fwht_one(const float* w, const float* x, float eps, float* y) {
  float u[128];
  normalize_one(x, eps, u);
  for (int i = 0; i < 128; ++i) u[i] = w[i] * u[i];
  for (int h = 1; h < 128; h <<= 1)
    for (int i = 0; i < 128; ++i) {
      if (i & h) continue;
      const float a = u[i], b = u[i + h];
      u[i] = a + b;
      u[i + h] = MUT(13) ? b - a : a - b;
    }
  const float c = (float)(1.0 / std::sqrt(128.0));
  for (int j = 0; j < 128; ++j) y[j] = MUT(14) ? u[j] : c * u[j];
}

bool all_finite(const float* x, int n) {
  for (int i = 0; i < n; ++i)
    if (!std::isfinite(x[i])) return false;
  return true;
}

// ---------------------------------------------------------------- int4 quantiser
// Section "What we do": 4-bit codes with one fp16 scale and one fp16 offset per
// token and head. fp32 specification:
//   mn = min y, mx = max y
//   o = fp16_down(mn)  (-0 stored as +0)
//   s = fp16_up((mx - o) / 15)  (-0 stored as +0)
//   c_i = 0 if s == 0, else clamp(round_half_even((y_i - o) / s), 0, 15)
// Flags: 1 = non-finite input (record not produced), 2 = fp16 range saturated.
int quantize_one(const float* y, uint8_t* codes, uint16_t* sbits, uint16_t* obits) {
  if (!all_finite(y, 128)) return 1;
  int flags = 0;
  float mn = y[0], mx = y[0];
  for (int i = 1; i < 128; ++i) {
    mn = std::min(mn, y[i]);
    mx = std::max(mx, y[i]);
  }
  double od = fp16_round(mn, MUT(11) ? 0 : -1);
  if (std::isinf(od)) {
    od = -kHalfMax;
    flags |= 2;
  }
  if (od == 0.0) od = 0.0;  // canonical +0
  float o = (float)od;
  float span = (mx - o) / 15.0f;
  double sd = fp16_round(span, MUT(4) ? 0 : +1);
  if (std::isinf(sd)) {
    sd = kHalfMax;
    flags |= 2;
  }
  if (sd == 0.0) sd = 0.0;  // canonical +0 (a row of zeros whose largest element is -0)
  float s = (float)sd;
  for (int i = 0; i < 128; ++i) {
    if (s == 0.0f) {
      codes[i] = 0;
      continue;
    }
    float q = (y[i] - o) / s;
    float r = MUT(5) ? std::round(q) : std::nearbyint(q);  // default mode: nearest, ties to even
    if (r < 0.0f) r = 0.0f;
    if (r > 15.0f) r = 15.0f;
    codes[i] = (uint8_t)r;
  }
  *sbits = fp16_bits(sd);
  *obits = fp16_bits(od);
  return flags;
}

// ---------------------------------------------------------------- attention
// Plain definition: for a query row, scores z_j = sm_scale * (q . k_j) over the
// visible keys, p = softmax(z) (max subtracted), output sum_j p_j v_j.
void softmax_attention_row(const double* q, int64_t L, int64_t lo, int64_t hi,
                           const double* K /* [L][128] */, const double* V, double sm_scale, double* out) {
  std::vector<double> z(std::max<int64_t>(hi - lo, 0));
  double zmax = -std::numeric_limits<double>::infinity();
  for (int64_t j = lo; j < hi; ++j) {
    double d = 0.0;
    for (int i = 0; i < 128; ++i) d += q[i] * K[j * 128 + i];
    z[j - lo] = (MUT(2) ? 1.0 : sm_scale) * d;
    zmax = std::max(zmax, z[j - lo]);
  }
  if (MUT(16)) zmax = 0.0;
  double den = 0.0;
  for (int i = 0; i < 128; ++i) out[i] = 0.0;
  for (int64_t j = lo; j < hi; ++j) {
    double p = std::exp(z[j - lo] - zmax);
    den += p;
    for (int i = 0; i < 128; ++i) out[i] += p * V[j * 128 + i];
  }
  for (int i = 0; i < 128; ++i) out[i] /= den;
  (void)L;
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------- rotation

// Sylvester construction: H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]].
void orc_hadamard(int n, int8_t* H) {
  std::vector<int8_t> cur(1, 1);
  int m = 1;
  while (m < n) {
    std::vector<int8_t> nxt((size_t)4 * m * m);
    for (int i = 0; i < m; ++i)
      for (int j = 0; j < m; ++j) {
        int8_t h = cur[(size_t)i * m + j];
        nxt[(size_t)i * 2 * m + j] = h;
        nxt[(size_t)i * 2 * m + j + m] = h;
        nxt[(size_t)(i + m) * 2 * m + j] = h;
        nxt[(size_t)(i + m) * 2 * m + j + m] = (int8_t)-h;
      }
    cur.swap(nxt);
    m *= 2;
  }
  std::memcpy(H, cur.data(), (size_t)n * n);
}

// Section "What we do": "a random sign per column", drawn from the seed.
void orc_signs(uint64_t seed, int n, int8_t* s) {
  uint64_t st = seed;
  for (int j = 0; j < n; ++j) s[j] = (splitmix64_next(st) >> 63) ? -1 : 1;
}

// R = H diag(s) / sqrt(n) in fp64, and its fp32 copy (round to nearest).
void orc_rotation(uint64_t seed, int n, double* R64, float* R32) {
  std::vector<int8_t> H((size_t)n * n), s(n);
  orc_hadamard(n, H.data());
  orc_signs(seed, n, s.data());
  double root = std::sqrt((double)n);
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < n; ++j) {
      double v = (double)(H[(size_t)i * n + j] * (MUT(3) ? s[i] : s[j])) / root;
      R64[(size_t)i * n + j] = v;
      R32[(size_t)i * n + j] = (float)v;
    }
}

// Section "What we do", QK-norm gain folding: scores depend on q.k only, so g_k
// moves to the query side and both gains join R in the query matrix:
//   M_q = R diag(g_q * g_k),  M_k = R.
// Each M_q entry: fp64 product R32[j][i] * (g_q[i] * g_k[i]) rounded once to fp32.
void orc_fold(const float* R32, const float* gq, const float* gk, int n, float* Mq, float* Mk) {
  for (int j = 0; j < n; ++j)
    for (int i = 0; i < n; ++i) {
      int gi = MUT(12) ? j : i;  // MUT(12): diag(g) R instead of R diag(g)
      double g = (double)gq[gi] * (MUT(7) ? 1.0 : (double)gk[gi]);
      Mq[(size_t)j * n + i] = (float)((double)R32[(size_t)j * n + i] * g);
      Mk[(size_t)j * n + i] = R32[(size_t)j * n + i];
    }
}

// Multipliers of the FWHT prologue: w_k = s (keys), w_q = fp32(s * g_q * g_k) (the
// product in fp64, rounded once), i.e. the diagonal that R = H diag(s)/sqrt(128) and the
// gain fold put in front of H.
void orc_fold_fwht(const int8_t* s, const float* gq, const float* gk, int n, float* wq, float* wk) {
  for (int i = 0; i < n; ++i) {
    const double sg = MUT(15) ? 1.0 : (double)s[i];
    wq[i] = (float)(sg * (double)gq[i] * (double)gk[i]);
    wk[i] = (float)s[i];
  }
}

// ---------------------------------------------------------------- codec

// y[v] = w-weighted FWHT prologue of x[v] (second specification); non-finite rows give NaN.
void orc_prologue_fwht(const float* w, const float* x, int64_t nvec, float eps, float* y, int threads) {
  for_range(nvec, threads, [&](int64_t a, int64_t b) {
    for (int64_t v = a; v < b; ++v) {
      if (!all_finite(x + v * 128, 128)) {
        for (int i = 0; i < 128; ++i) y[v * 128 + i] = std::numeric_limits<float>::quiet_NaN();
        continue;
      }
      prologue_fwht_one(w, x + v * 128, eps, y + v * 128);
    }
  });
}

// y[v] = M n(x[v]) with the fp32 specification above; x rows that are not all
// finite give a row of NaN.
void orc_prologue(const float* M, const float* x, int64_t nvec, float eps, float* y, int threads) {
  for_range(nvec, threads, [&](int64_t a, int64_t b) {
    for (int64_t v = a; v < b; ++v) {
      if (!all_finite(x + v * 128, 128)) {
        for (int i = 0; i < 128; ++i) y[v * 128 + i] = std::numeric_limits<float>::quiet_NaN();
        continue;
      }
      prologue_one(M, x + v * 128, eps, y + v * 128);
    }
  });
}

// Per 128-vector: codes (one byte per code, logical order), fp16 scale/offset
// bits and flags (1 non-finite, 2 range saturated).
void orc_quantize_int4(const float* y, int64_t nvec, uint8_t* codes, uint16_t* sbits, uint16_t* obits,
                       int32_t* flags, int threads) {
  for_range(nvec, threads, [&](int64_t a, int64_t b) {
    for (int64_t v = a; v < b; ++v) {
      uint16_t s = 0, o = 0;
      std::memset(codes + v * 128, 0, 128);
      int f = quantize_one(y + v * 128, codes + v * 128, &s, &o);
      sbits[v] = s;
      obits[v] = o;
      flags[v] = f;
    }
  });
}

// Dequantised value c*s + o, exact in fp64.
void orc_dequant_int4(const uint8_t* codes, const uint16_t* sbits, const uint16_t* obits, int64_t nvec,
                      double* out) {
  for (int64_t v = 0; v < nvec; ++v) {
    double s = fp16_value(sbits[v]), o = fp16_value(obits[v]);
    for (int i = 0; i < 128; ++i) out[v * 128 + i] = (double)codes[v * 128 + i] * s + (MUT(1) ? 0.0 : o);
  }
}

uint16_t orc_fp16_round_bits(float x, int dir) { return fp16_bits(fp16_round(x, dir)); }

// The converters above over n consecutive fp32 bit patterns first, first+1, ... (wrapping
// at 2^32), for the exhaustive pins: fp16 bits rounded to nearest-even (rn), toward -inf
// (rd), toward +inf (ru), and the saturating e4m3 code (e4). Any output may be NULL.
void orc_convert_range(uint32_t first, int64_t n, uint16_t* rn, uint16_t* rd, uint16_t* ru, uint8_t* e4,
                       int threads) {
  for_range(n, threads, [&](int64_t a, int64_t b) {
    for (int64_t i = a; i < b; ++i) {
      const uint32_t bits = first + (uint32_t)i;
      float x;
      std::memcpy(&x, &bits, sizeof(x));
      if (rn) rn[i] = fp16_bits(fp16_round(x, 0));
      if (rd) rd[i] = fp16_bits(fp16_round(x, -1));
      if (ru) ru[i] = fp16_bits(fp16_round(x, +1));
      if (e4) e4[i] = e4m3_encode(x);
    }
  });
}
double orc_fp16_value(uint16_t h) { return fp16_value(h); }
uint8_t orc_e4m3_encode(float x) { return e4m3_encode(x); }
double orc_e4m3_value(uint8_t c) { return e4m3_value(c); }

// Stock FP8 cache write: code = e4m3(x / scale) with an IEEE fp32 division.
void orc_quantize_fp8(const float* x, int64_t n, float scale, uint8_t* codes, int threads) {
  for_range(n, threads, [&](int64_t a, int64_t b) {
    for (int64_t e = a; e < b; ++e) codes[e] = e4m3_encode(x[e] / scale);
  });
}

// ---------------------------------------------------------------- attention (fp64)

// Rotated-int4 decode attention (section "What we do": decode reads the 4-bit
// codes and nothing is rotated back). Query row r attends to cache positions
// 0..vis_len[r]-1 of the dequantised cache k_j = c_j s_j + o_j (same for v).
//   q      [nrows][128] fp32 (already rotated and folded)
//   kc,vc  [L][128] logical codes; ks/ko/vs/vo fp16 bits per position
//   out    [nrows][128] fp64
void orc_attention_int4(const float* q, int64_t nrows, const int64_t* vis_len, const uint8_t* kc,
                        const uint16_t* ks, const uint16_t* ko, const uint8_t* vc, const uint16_t* vs,
                        const uint16_t* vo, int64_t L, double sm_scale, double* out, int threads) {
  std::vector<double> K((size_t)L * 128), V((size_t)L * 128);
  for_range(L, threads, [&](int64_t a, int64_t b) {
    orc_dequant_int4(kc + a * 128, ks + a, ko + a, b - a, K.data() + a * 128);
    orc_dequant_int4(vc + a * 128, vs + a, vo + a, b - a, V.data() + a * 128);
  });
  for_range(nrows, threads, [&](int64_t a, int64_t b) {
    for (int64_t r = a; r < b; ++r) {
      double qd[128];
      for (int i = 0; i < 128; ++i) qd[i] = (double)q[r * 128 + i];
      softmax_attention_row(qd, L, 0, vis_len[r] - (MUT(8) ? 1 : 0), K.data(), V.data(), sm_scale, out + r * 128);
    }
  });
}

// Stock FP8 sliding-window attention: row r attends to positions lo[r]..hi[r]
// (inclusive) of a cache held here by position, k_j = e4m3(kc_j) * k_scale.
void orc_attention_fp8(const float* q, int64_t nrows, const int64_t* lo, const int64_t* hi, const uint8_t* kc,
                       const uint8_t* vc, int64_t L, double k_scale, double v_scale, double sm_scale,
                       double* out, int threads) {
  std::vector<double> K((size_t)L * 128), V((size_t)L * 128);
  for (int64_t e = 0; e < L * 128; ++e) {
    K[e] = e4m3_value(kc[e]) * k_scale;
    V[e] = e4m3_value(vc[e]) * v_scale;
  }
  for_range(nrows, threads, [&](int64_t a, int64_t b) {
    for (int64_t r = a; r < b; ++r) {
      double qd[128];
      for (int i = 0; i < 128; ++i) qd[i] = (double)q[r * 128 + i];
      softmax_attention_row(qd, L, lo[r], hi[r] + 1, K.data(), V.data(), sm_scale, out + r * 128);
    }
  });
}

// The same softmax attention on explicit fp64 keys and values (all L visible).
void orc_attention_f64(const double* q, int64_t nrows, const double* K, const double* V, int64_t L,
                       double sm_scale, double* out, int threads) {
  for_range(nrows, threads, [&](int64_t a, int64_t b) {
    for (int64_t r = a; r < b; ++r) softmax_attention_row(q + r * 128, L, 0, L, K, V, sm_scale, out + r * 128);
  });
}

// ---------------------------------------------------------------- claim statistics

// Section "What we do": largest channel vs the average channel of the cached
// keys, measured as max_c mean_t |k_tc| / mean_c mean_t |k_tc|.
double orc_channel_ratio(const double* keys, int64_t n, int d) {
  std::vector<double> m(d, 0.0);
  for (int64_t t = 0; t < n; ++t)
    for (int c = 0; c < d; ++c) {
      const double k = keys[t * d + c];
      m[c] += MUT(17) ? k * k : std::fabs(k);  // MUT(17): root-mean-square per channel
    }
  if (MUT(17))
    for (int c = 0; c < d; ++c) m[c] = std::sqrt(m[c]);
  double mx = 0.0, mean = 0.0;
  for (int c = 0; c < d; ++c) {
    mx = std::max(mx, m[c]);
    mean += m[c];
  }
  mean /= d;
  return mx / mean;
}

// Section "What we do", attention-output error of 4-bit keys: how far quantised
// keys move the attention output, relative L2, averaged over query rows. Values
// stay exact; only the keys are quantised. Three caches are compared with the
// exact model scores (g_q n(q)).(g_k n(k)):
//   err[0] int4 without rotation: keys n(k), queries diag(g_q g_k) n(q)
//   err[1] int4 with rotation:    keys R n(k), queries R diag(g_q g_k) n(q)
//   err[2] FP8 e4m3 keys g_k n(k) with per-tensor scale max|k|/448, queries g_q n(q)
// ratio[0], ratio[1]: channel ratio of n(k) and of R n(k).
// Inputs: q [nq][128], k, v [L][128] fp32 pre-norm; R32 the fp32 rotation.
void orc_claim_errors(const float* q, int64_t nq, const float* k, const float* v, int64_t L, const float* gq,
                      const float* gk, const float* R32, float eps, double* err, double* ratio, int threads) {
  const int D = 128;
  std::vector<float> I((size_t)D * D, 0.0f), Mq_unrot((size_t)D * D, 0.0f), Mq_rot((size_t)D * D);
  std::vector<float> Gk((size_t)D * D, 0.0f), Gq((size_t)D * D, 0.0f);
  for (int i = 0; i < D; ++i) {
    I[(size_t)i * D + i] = 1.0f;
    Mq_unrot[(size_t)i * D + i] = (float)((double)gq[i] * (double)gk[i]);
    Gk[(size_t)i * D + i] = gk[i];
    Gq[(size_t)i * D + i] = gq[i];
  }
  std::vector<float> Mk_dummy((size_t)D * D);
  orc_fold(R32, gq, gk, D, Mq_rot.data(), Mk_dummy.data());

  // normalised keys and queries in fp32 per the prologue specification
  std::vector<float> nk((size_t)L * D), rk((size_t)L * D), gkk((size_t)L * D);
  orc_prologue(I.data(), k, L, eps, nk.data(), threads);
  orc_prologue(R32, k, L, eps, rk.data(), threads);
  orc_prologue(Gk.data(), k, L, eps, gkk.data(), threads);
  std::vector<float> qu((size_t)nq * D), qr((size_t)nq * D), qg((size_t)nq * D);
  orc_prologue(Mq_unrot.data(), q, nq, eps, qu.data(), threads);
  orc_prologue(Mq_rot.data(), q, nq, eps, qr.data(), threads);
  orc_prologue(Gq.data(), q, nq, eps, qg.data(), threads);

  std::vector<double> Vd((size_t)L * D);
  for (int64_t e = 0; e < L * D; ++e) Vd[e] = v[e];
  double sm = 1.0 / std::sqrt((double)D);

  // exact reference: (g_q n(q)) . (g_k n(k))
  std::vector<double> Kx((size_t)L * D), Qx((size_t)nq * D), ref((size_t)nq * D);
  for (int64_t e = 0; e < L * D; ++e) Kx[e] = gkk[e];
  for (int64_t e = 0; e < nq * D; ++e) Qx[e] = qg[e];
  orc_attention_f64(Qx.data(), nq, Kx.data(), Vd.data(), L, sm, ref.data(), threads);

  auto rel_err = [&](const std::vector<double>& o) {
    double acc = 0.0;
    for (int64_t r = 0; r < nq; ++r) {
      double num = 0.0, den = 0.0;
      for (int i = 0; i < D; ++i) {
        double d = o[r * D + i] - ref[r * D + i];
        num += d * d;
        den += ref[r * D + i] * ref[r * D + i];
      }
      acc += std::sqrt(num / den);
    }
    return acc / (double)nq;
  };

  auto int4_case = [&](const std::vector<float>& keys, const std::vector<float>& qs) {
    std::vector<uint8_t> c((size_t)L * D);
    std::vector<uint16_t> sb(L), ob(L);
    std::vector<int32_t> fl(L);
    orc_quantize_int4(keys.data(), L, c.data(), sb.data(), ob.data(), fl.data(), threads);
    std::vector<double> Kq((size_t)L * D), Qd((size_t)nq * D), o((size_t)nq * D);
    orc_dequant_int4(c.data(), sb.data(), ob.data(), L, Kq.data());
    for (int64_t e = 0; e < nq * D; ++e) Qd[e] = qs[e];
    orc_attention_f64(Qd.data(), nq, Kq.data(), Vd.data(), L, sm, o.data(), threads);
    return rel_err(o);
  };
  err[0] = int4_case(nk, qu);
  err[1] = int4_case(rk, qr);

  float amax = 0.0f;
  for (int64_t e = 0; e < L * D; ++e) amax = std::max(amax, std::fabs(gkk[e]));
  float scale = amax / 448.0f;
  std::vector<uint8_t> c8((size_t)L * D);
  orc_quantize_fp8(gkk.data(), L * D, scale, c8.data(), threads);
  std::vector<double> K8((size_t)L * D), o8((size_t)nq * D);
  for (int64_t e = 0; e < L * D; ++e) K8[e] = e4m3_value(c8[e]) * (double)scale;
  orc_attention_f64(Qx.data(), nq, K8.data(), Vd.data(), L, sm, o8.data(), threads);
  err[2] = rel_err(o8);

  std::vector<double> a((size_t)L * D), b((size_t)L * D);
  for (int64_t e = 0; e < L * D; ++e) {
    a[e] = nk[e];
    b[e] = rk[e];
  }
  ratio[0] = orc_channel_ratio(a.data(), L, D);
  ratio[1] = orc_channel_ratio(b.data(), L, D);
}

}  // extern "C"
