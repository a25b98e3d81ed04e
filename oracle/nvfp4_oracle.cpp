// NVFP4 MoE oracle — TEST INFRASTRUCTURE ONLY.
//
// A plain, slow CPU statement of what the NVFP4 Mixture-of-Experts expert
// forward computes. Only the tests, the smoke check and the CPU-baseline leg
// of the benchmark may load this library. It shares no code, header, table or
// helper with the CUDA path under nvfp4_block_scaled_05_gb300/csrc.
//
// Sources (the pages describe a CuTeDSL kernel library, "NVFP4 MegaMoE Kernel"):
//   * README "What We Have" / "ScaledGroupedGemmKernel": NVFP4 = E2M1 codes in
//     16-element blocks, FP8 (E4M3) block scale on both operands, FP32 global
//     scale per expert; 2D x 3D grouped GEMM A(M,K) x B(E,K,N) -> C(M,N).
//   * README "Bridge Layer": quantize_to_nvfp4 (with global scale),
//     quantize_activation_nvfp4 (pre-computed global scale),
//     interleave_l1_weights (gate/up at granularity 8).
//   * README "MoE Runner": the six-step forward (quantize, L1 GEMM, SiLU(gate)*up,
//     requantize, L2 GEMM, scatter with routing weights).
//   * README "Correctness Bugs Fixed": bug 3 (all-zero block -> exact-0 scale),
//     bug 4 (underflow block -> zero codes), bug 2 (dequantize->requantize is
//     byte-identical), bug 5 (expert counting by bincount).
//   * README "Fused SwiGLU - How It Works": column interleave at granularity 8,
//     silu(gate)*up pairing; "Key Lessons" 10 (SiLU on all columns is not SwiGLU).
//   * CURRENT_BUG.md "What Works": activation global scale recomputed per call.
//
// Readings where the pages are silent (each is listed in the design notes):
//   R1 E2M1 encode = round-to-nearest-even onto {0,.5,1,1.5,2,3,4,6}, saturating
//      at 6; the sign bit of the input is kept (a negative value that rounds to
//      magnitude 0 gives code 0x8). Two codes per byte, even element in the low
//      nibble.
//   R2 E4M3 encode = round-to-nearest-even, saturating at 448 (never NaN).
//   R3 global scale gs = 2688 / amax (2688 = 6 * 448) in f32; gs = 1 if amax == 0.
//   R4 block rule: p = amax_block * gs (f32). If amax_block == 0 (bug 3) or
//      p < 6 * 2^-9 (bug 4, compared where the block scale lives, i.e. after
//      the global scale), the block gets scale byte 0 and all codes 0.
//      Otherwise sf = E4M3(p / 6), s = value(sf), code_i = E2M1((x_i * gs) / s),
//      every step one f32 operation rounded to nearest.
//   R5 top-k: the k largest logits, ties to the lower expert index, ordered by
//      descending logit; weights = softmax over the k selected logits.
//   R16 a NaN router logit ranks as -inf: below every finite logit, never
//      chosen before one, and never leaves a token without k experts.
//   R6 permutation: rows of one expert are ordered by ascending flat slot
//      f = t*k + j (stable counting sort).
//   R7 dequantized value = code * s / gs; GEMMs accumulate in fp64.
//   R13 RMS norm (README "THE PLAN", item 3: "Q norm -> RoPE -> NVFP4 quant" in
//      one pass): y_i = x_i / sqrt(mean_i(x_i^2) + eps) * gamma_i over the D
//      elements of a row, in fp64.
//   R14 RoPE on the last R elements of the row: adjacent pairs (2j, 2j+1)
//      counted from the first rope element are rotated by the angle whose
//      cosine and sine are the caller's tables at [position][j]; the first
//      D - R elements are left as normed.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>
#include <algorithm>
#include <numeric>

extern "C" {

// ---------------------------------------------------------------- formats

// E2M1 magnitudes indexed by the low three bits of a code (README "What We
// Have": 4-bit E2M1 values; the value set is {0, 0.5, 1, 1.5, 2, 3, 4, 6}).
static const double kE2M1[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_decode(uint8_t code) {
  double m = kE2M1[code & 7];
  return (code & 8) ? -m : m;
}

// R1: nearest representable magnitude, ties to the even code (mantissa bit 0),
// saturating at 6. Works on the exact value of the f32 input.
uint8_t orc_e2m1_encode(float v) {
  uint8_t sign = std::signbit(v) ? 8 : 0;
  double a = std::fabs((double)v);
  if (std::isnan(a)) return sign | 7;
  if (a >= 6.0) return sign | 7;
  int best = 0;
  double best_err = a;  // distance to magnitude 0
  for (int i = 1; i < 8; ++i) {
    double err = std::fabs(a - kE2M1[i]);
    if (err < best_err || (err == best_err && (i % 2) == 0)) {
      best = i;
      best_err = err;
    }
  }
  return sign | (uint8_t)best;
}

// E4M3 (OCP FP8, "fn" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits;
// exponent field 0 is subnormal (m * 2^-9); 0x7F / 0xFF are NaN; max 448.
double orc_e4m3_decode(uint8_t code) {
  int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = std::ldexp((double)m, -9);
  else v = std::ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

// R2: round to nearest even, saturate to 448.
uint8_t orc_e4m3_encode(float vf) {
  double v = (double)vf;
  uint8_t sign = std::signbit(v) ? 0x80 : 0;
  double a = std::fabs(v);
  if (std::isnan(a)) return sign | 0x7F;
  if (a >= 448.0) return sign | 0x7E;
  if (a < std::ldexp(1.0, -6)) {
    // subnormal grid: multiples of 2^-9; m == 8 is the first normal (code 8)
    double m = std::nearbyint(std::ldexp(a, 9));  // default mode: nearest-even
    return sign | (uint8_t)m;
  }
  int e;
  double fr = std::frexp(a, &e);  // a = fr * 2^e, fr in [0.5, 1)
  int ue = e - 1;                 // a = (2 fr) * 2^ue, 2 fr in [1, 2)
  double m = std::nearbyint((2.0 * fr - 1.0) * 8.0);
  if (m == 8.0) { m = 0.0; ue += 1; }
  int field = ue + 7;
  if (field > 15 || (field == 15 && m == 7.0)) return sign | 0x7E;
  return sign | (uint8_t)((field << 3) | (int)m);
}

// R3
float orc_global_scale(float amax) {
  if (amax == 0.0f) return 1.0f;
  volatile float num = 2688.0f;
  return num / amax;
}

static int g_threads = 0;

void orc_set_threads(int n) { g_threads = n; }

int orc_get_threads() {
  if (g_threads > 0) return g_threads;
  unsigned h = std::thread::hardware_concurrency();
  return h ? (int)h : 1;
}

}  // extern "C"

template <class F>
static void parallel_rows(int64_t rows, F fn) {
  int nt = (int)std::min<int64_t>(orc_get_threads(), std::max<int64_t>(rows, 1));
  if (nt <= 1) {
    for (int64_t r = 0; r < rows; ++r) fn(r);
    return;
  }
  std::vector<std::thread> th;
  for (int i = 0; i < nt; ++i)
    th.emplace_back([&, i] {
      for (int64_t r = i; r < rows; r += nt) fn(r);
    });
  for (auto& t : th) t.join();
}

extern "C" {

static inline float bf16_to_f32(uint16_t b);
static inline double bf16_to_double(uint16_t b) { return (double)bf16_to_f32(b); }
static inline float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

float orc_amax_bf16(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx) {
  float m = 0.0f;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) {
      float a = std::fabs(bf16_to_f32(x[r * ldx + c]));
      if (a > m) m = a;
    }
  return m;
}

float orc_amax_f32(const float* x, int64_t n) {
  float m = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float a = std::fabs(x[i]);
    if (a > m) m = a;
  }
  return m;
}

// R4 applied to one 16-element block of f32 values.
// Writes 8 code bytes (element 2j in the low nibble of byte j) and returns the
// scale byte.
static uint8_t quantize_block(const float* v, float gs, uint8_t* out8) {
  float amax = 0.0f;
  for (int i = 0; i < 16; ++i) amax = std::max(amax, std::fabs(v[i]));
  volatile float p = amax * gs;
  const float underflow = 6.0f * 0.001953125f;  // 6 * 2^-9
  if (amax == 0.0f || p < underflow) {           // bug 3 and bug 4
    std::memset(out8, 0, 8);
    return 0;
  }
  volatile float ps = p / 6.0f;
  uint8_t sf = orc_e4m3_encode(ps);
  float s = (float)orc_e4m3_decode(sf);
  for (int j = 0; j < 8; ++j) {
    uint8_t c[2];
    for (int h = 0; h < 2; ++h) {
      volatile float scaled = v[2 * j + h] * gs;
      volatile float norm = scaled / s;
      c[h] = orc_e2m1_encode(norm);
    }
    out8[j] = (uint8_t)(c[0] | (c[1] << 4));
  }
  return sf;
}

// Block-quantize rows x cols (cols % 16 == 0) BF16 values with global scale gs.
// codes: rows x cols/2 bytes, row-major. sf: rows x cols/16 bytes, row-major.
void orc_quantize_bf16(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx, float gs,
                       uint8_t* codes, uint8_t* sf) {
  parallel_rows(rows, [&](int64_t r) {
    float blk[16];
    for (int64_t b = 0; b < cols / 16; ++b) {
      for (int i = 0; i < 16; ++i) blk[i] = bf16_to_f32(x[r * ldx + b * 16 + i]);
      sf[r * (cols / 16) + b] = quantize_block(blk, gs, codes + r * (cols / 2) + b * 8);
    }
  });
}

// Same for f32 input (the requantization of h, and the round-trip identity).
void orc_quantize_f32(const float* x, int64_t rows, int64_t cols, float gs, uint8_t* codes,
                      uint8_t* sf) {
  parallel_rows(rows, [&](int64_t r) {
    for (int64_t b = 0; b < cols / 16; ++b)
      sf[r * (cols / 16) + b] =
          quantize_block(x + r * cols + b * 16, gs, codes + r * (cols / 2) + b * 8);
  });
}

// R7 in f32 (used for the byte round-trip of README bug 2): v = (code*s)/gs.
void orc_dequantize_f32(const uint8_t* codes, const uint8_t* sf, int64_t rows, int64_t cols,
                        float gs, float* out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) {
      uint8_t byte = codes[r * (cols / 2) + c / 2];
      uint8_t code = (c & 1) ? (byte >> 4) : (byte & 15);
      float s = (float)orc_e4m3_decode(sf[r * (cols / 16) + c / 16]);
      volatile float cs = (float)orc_e2m1_decode(code) * s;
      out[r * cols + c] = cs / gs;
    }
}

// R7 in fp64.
void orc_dequantize_f64(const uint8_t* codes, const uint8_t* sf, int64_t rows, int64_t cols,
                        float gs, double* out) {
  parallel_rows(rows, [&](int64_t r) {
    for (int64_t c = 0; c < cols; ++c) {
      uint8_t byte = codes[r * (cols / 2) + c / 2];
      uint8_t code = (c & 1) ? (byte >> 4) : (byte & 15);
      double s = orc_e4m3_decode(sf[r * (cols / 16) + c / 16]);
      out[r * cols + c] = orc_e2m1_decode(code) * s / (double)gs;
    }
  });
}

// ---------------------------------------------------------------- layout

// README "Fused SwiGLU - How It Works": W1's 2I output rows hold gate rows
// [0, I) then up rows [I, 2I); the interleaved order alternates blocks of g
// rows: [gate 0..g-1, up 0..g-1, gate g..2g-1, up g..2g-1, ...].
// Interleaved row 2g*(n/g) + n%g is gate row n; row 2g*(n/g) + g + n%g is up row n.
void orc_interleave_rows(const uint8_t* src, uint8_t* dst, int64_t two_i, int64_t row_bytes,
                         int64_t g) {
  int64_t inter = two_i / 2;
  for (int64_t n = 0; n < inter; ++n) {
    int64_t base = 2 * g * (n / g) + n % g;
    std::memcpy(dst + base * row_bytes, src + n * row_bytes, row_bytes);
    std::memcpy(dst + (base + g) * row_bytes, src + (inter + n) * row_bytes, row_bytes);
  }
}

void orc_deinterleave_rows(const uint8_t* src, uint8_t* dst, int64_t two_i, int64_t row_bytes,
                           int64_t g) {
  int64_t inter = two_i / 2;
  for (int64_t n = 0; n < inter; ++n) {
    int64_t base = 2 * g * (n / g) + n % g;
    std::memcpy(dst + n * row_bytes, src + base * row_bytes, row_bytes);
    std::memcpy(dst + (inter + n) * row_bytes, src + (base + g) * row_bytes, row_bytes);
  }
}

// ---------------------------------------------------------------- routing

// R5 for T tokens over E experts. R16: a NaN logit ranks as -inf (below every
// finite logit, tied with -inf, ties to the lower index), so the sort key is a
// strict weak order and a token with NaN logits still gets k valid experts.
void orc_route_topk(const float* logits, int64_t T, int E, int k, int32_t* ids, double* w) {
  std::vector<int> idx(E);
  std::vector<double> key(E);
  for (int64_t t = 0; t < T; ++t) {
    const float* l = logits + t * E;
    for (int e = 0; e < E; ++e) key[e] = std::isnan(l[e]) ? -INFINITY : (double)l[e];
    std::iota(idx.begin(), idx.end(), 0);
    std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) { return key[a] > key[b]; });
    double lmax = key[idx[0]];
    double den = 0.0;
    for (int j = 0; j < k; ++j) den += std::exp(key[idx[j]] - lmax);
    for (int j = 0; j < k; ++j) {
      ids[t * k + j] = idx[j];
      w[t * k + j] = std::exp(key[idx[j]] - lmax) / den;
    }
  }
}

// R6 with README bug 5 (per-expert counts by bincount, then exclusive sum).
void orc_permute(const int32_t* ids, int64_t T, int k, int E, int32_t* offsets,
                 int32_t* perm_to_flat, int32_t* flat_to_perm) {
  std::vector<int64_t> count(E, 0);
  for (int64_t f = 0; f < T * k; ++f) count[ids[f]]++;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + (int32_t)count[e];
  std::vector<int64_t> next(offsets, offsets + E);
  for (int64_t f = 0; f < T * k; ++f) {
    int64_t pos = next[ids[f]]++;
    perm_to_flat[pos] = (int32_t)f;
    flat_to_perm[f] = (int32_t)pos;
  }
}

// ---------------------------------------------------------------- GEMM



// C[r][n] = sum_k A[r][k] * B[n][k], fp64, plain loops (threads over rows).
void orc_matmul_nt(const double* A, const double* B, int64_t M, int64_t N, int64_t K, double* C) {
  parallel_rows(M, [&](int64_t r) {
    const double* a = A + r * K;
    for (int64_t n = 0; n < N; ++n) {
      const double* b = B + n * K;
      double acc = 0.0;
      for (int64_t kk = 0; kk < K; ++kk) acc += a[kk] * b[kk];
      C[r * N + n] = acc;
    }
  });
}

// README "ScaledGroupedGemmKernel": rows [offsets[e], offsets[e+1]) of A use
// expert e of B. A is (M, K) NVFP4 with row-major scales and global scale gs_a;
// B is (E, N, K) NVFP4 (K contiguous) with per-expert global scales gs_b[e].
// C (M, N) fp64.
void orc_grouped_gemm(const uint8_t* a_codes, const uint8_t* a_sf, float gs_a,
                      const uint8_t* b_codes, const uint8_t* b_sf, const float* gs_b,
                      const int32_t* offsets, int64_t N, int64_t K, int E, double* C) {
  for (int e = 0; e < E; ++e) {
    int64_t r0 = offsets[e], r1 = offsets[e + 1];
    if (r1 <= r0) continue;
    std::vector<double> A((r1 - r0) * K), B(N * K);
    orc_dequantize_f64(a_codes + r0 * (K / 2), a_sf + r0 * (K / 16), r1 - r0, K, gs_a, A.data());
    orc_dequantize_f64(b_codes + (int64_t)e * N * (K / 2), b_sf + (int64_t)e * N * (K / 16), N, K,
                       gs_b[e], B.data());
    orc_matmul_nt(A.data(), B.data(), r1 - r0, N, K, C + r0 * N);
  }
}

// README "MoE Runner" step 3 and "Key Lessons" 10: h = silu(gate) * up with
// gate = columns [0, I) and up = columns [I, 2I) of the L1 output v (M, 2I).
// silu(g) = g / (1 + exp(-g)). Result rounded once to f32.
void orc_swiglu(const double* v, int64_t M, int64_t I, float* h) {
  for (int64_t r = 0; r < M; ++r)
    for (int64_t i = 0; i < I; ++i) {
      double g = v[r * 2 * I + i], u = v[r * 2 * I + I + i];
      double silu = g / (1.0 + std::exp(-g));
      h[r * I + i] = (float)(silu * u);
    }
}

// README "MoE Runner" step 6: y[t] = sum_j w[t][j] * out[flat_to_perm[t*k+j]],
// summed in fp64 in j order.
void orc_combine(const double* out, int64_t K, const double* w, const int32_t* flat_to_perm,
                 int64_t T, int k, double* y) {
  for (int64_t t = 0; t < T; ++t)
    for (int64_t c = 0; c < K; ++c) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j) acc += w[t * k + j] * out[(int64_t)flat_to_perm[t * k + j] * K + c];
      y[t * K + c] = acc;
    }
}

// R13 + R14: RMS norm, then rotary embedding of the last R elements.
// x: rows x D BF16 bits (leading dimension ldx); gamma[D]; pos[rows];
// cos_t / sin_t: (max_pos x R/2), row-major; y: rows x D fp64.
void orc_rmsnorm_rope(const uint16_t* x, int64_t rows, int64_t D, int64_t ldx, const double* gamma,
                      double eps, int64_t R, const int32_t* pos, const double* cos_t,
                      const double* sin_t, double* y) {
  for (int64_t r = 0; r < rows; ++r) {
    double ss = 0.0;
    for (int64_t i = 0; i < D; ++i) {
      const double v = bf16_to_double(x[r * ldx + i]);
      ss += v * v;
    }
    const double inv = 1.0 / std::sqrt(ss / (double)D + eps);
    double* yr = y + r * D;
    for (int64_t i = 0; i < D; ++i) yr[i] = bf16_to_double(x[r * ldx + i]) * inv * gamma[i];
    const int64_t s0 = D - R;
    for (int64_t j = 0; j < R / 2; ++j) {
      const double c = cos_t[(int64_t)pos[r] * (R / 2) + j], s = sin_t[(int64_t)pos[r] * (R / 2) + j];
      const double a = yr[s0 + 2 * j], b = yr[s0 + 2 * j + 1];
      yr[s0 + 2 * j] = a * c - b * s;
      yr[s0 + 2 * j + 1] = a * s + b * c;
    }
  }
}

}  // extern "C"
