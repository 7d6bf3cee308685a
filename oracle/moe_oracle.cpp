// CPU oracle of one routed MoE layer forward pass, in FP64 (test
// infrastructure only: the tests, the smoke check and the bench's CPU
// baseline call it; the CUDA library never links or calls it, and the two
// share no code).
//
// The FreeToken pages ("FreeToken：把 284B MoE 塞进游戏 PC", zhichai.net, §二;
// the ananclaw.com explainer, §核心方法 1 and 4; the juejin.cn overview, §二
// and §五) describe an edge MoE serving engine whose layers route each token to
// a few experts held in a GPU LRU expert cache, with MXFP4 / NVFP4 weights.
// They print no formula for the layer, so each function below writes out the
// standard definition the pages' names refer to, as plain loops:
//
//   formats   E2M1 / E8M0 / E4M3 values (OCP Microscaling v1.0; NVIDIA's
//             NVFP4), block dequantisation (two codes per byte, low nibble =
//             even K; scales row-major [rows, K / block]);
//   quant     the FP4 activation quantisers of the prefill regime (fp32
//             decisions, as the reading in the package notes fixes them);
//   router    logits in FP64, top-k on the logits (ties to the lower expert
//             id), gates = softmax over the selected logits (or the full
//             softmax probabilities), ids ascending;
//   permute   counts, exclusive prefix sum over ascending expert id, rows of
//             one expert in ascending token order;
//   expert    out = W_d (SiLU(W_g x) * (W_u x)), SiLU(z) = z / (1 + e^-z);
//   combine   y[t] = sum_j g[t, j] out_j + shared (weight 1);
//   lru       the per-step slot table: hits first (ascending id), then misses
//             (ascending id); a miss takes the lowest free slot, else evicts
//             the least recently used expert (smallest recency stamp).
//
// Every reduction runs in a fixed order (ascending index), so a result does
// not depend on the thread count; OpenMP only spreads independent rows or
// tokens over the cores.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

constexpr int kMXFP4 = 0;
constexpr int kNVFP4 = 1;
constexpr int kMXFP8 = 2;   // E4M3 elements, E8M0 per 32
constexpr int kBF16 = 3;    // bf16 elements, no scales

double e2m1_value(int c) {
  const int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
  const double mag = e == 0 ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

double e8m0_value(int x) { return x == 255 ? std::nan("") : std::ldexp(1.0, x - 127); }

double e4m3_value(int b) {
  const int s = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
  if (e == 15 && m == 7) return std::nan("");
  const double mag = e == 0 ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

// Nearest E2M1 code of q: ties to the even code, saturating at 6, sign kept
// (a negative value that rounds to zero is -0, code 8).
int e2m1_encode(double q) {
  static const double mags[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  const double a = std::fabs(q);
  int pick = 7;
  if (a < 6.0) {
    double best = INFINITY;
    for (int c = 0; c < 8; ++c) {
      const double dist = std::fabs(a - mags[c]);
      if (dist < best || (dist == best && (c % 2 == 0) && (pick % 2 != 0))) {
        best = dist;
        pick = c;
      }
    }
  }
  return pick | (std::signbit(q) ? 8 : 0);
}

// Nearest non-negative finite E4M3 byte of v >= 0: ties to the even byte,
// values of 448 and above give 448.
int e4m3_encode_satfinite(double v) {
  if (v >= 448.0) return 0x7E;
  int pick = 0;
  double best = INFINITY;
  for (int b = 0; b < 0x7F; ++b) {
    const double dist = std::fabs(v - e4m3_value(b));
    if (dist < best || (dist == best && (b % 2 == 0) && (pick % 2 != 0))) {
      best = dist;
      pick = b;
    }
  }
  return pick;
}

// bf16 bits -> value: the fp32 whose upper half they are.
double bf16_value(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

// fp32 -> bf16 bits, nearest even (NaN stays NaN).
uint16_t bf16_round_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x7FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
  return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

double silu(double z) { return z / (1.0 + std::exp(-z)); }

int nthreads(int want) {
#ifdef _OPENMP
  return want > 0 ? want : omp_get_max_threads();
#else
  (void)want;
  return 1;
#endif
}

int g_threads = 0;   // 0: all the cores OpenMP sees

}  // namespace

extern "C" {

// ---------------------------------------------------------------- threads
void orc_set_threads(int n) { g_threads = n < 0 ? 0 : n; }
int orc_threads() { return nthreads(g_threads); }

// ---------------------------------------------------------------- formats
double orc_e2m1(int code) { return e2m1_value(code & 15); }
double orc_e8m0(int x) { return e8m0_value(x & 255); }
double orc_e4m3(int b) { return e4m3_value(b & 255); }

// One weight matrix [rows, K] to FP64:
// MXFP4 w = E2M1(c) E8M0(s) (block 32), NVFP4 w = E2M1(c) E4M3(s) t (block 16),
// MXFP8 w = E4M3(c) E8M0(s) (block 32, one byte per element), BF16 w = the
// bf16 value of each little-endian byte pair.
void orc_dequant(const uint8_t* codes, const uint8_t* scales, int rows, int K, int fmt, float tscale,
                 double* out) {
  if (fmt == kMXFP8 || fmt == kBF16) {
#pragma omp parallel for num_threads(nthreads(g_threads)) schedule(static)
    for (int r = 0; r < rows; ++r)
      for (int i = 0; i < K; ++i) {
        if (fmt == kBF16) {
          const uint8_t* b = codes + (size_t)r * K * 2 + (size_t)i * 2;
          out[(size_t)r * K + i] = bf16_value((uint16_t)(b[0] | (b[1] << 8)));
        } else {
          out[(size_t)r * K + i] =
              e4m3_value(codes[(size_t)r * K + i]) * e8m0_value(scales[(size_t)r * (K / 32) + i / 32]);
        }
      }
    return;
  }
  const int blk = fmt == kMXFP4 ? 32 : 16;
  const double t = fmt == kMXFP4 ? 1.0 : (double)tscale;
#pragma omp parallel for num_threads(nthreads(g_threads)) schedule(static)
  for (int r = 0; r < rows; ++r) {
    for (int i = 0; i < K; ++i) {
      const uint8_t byte = codes[(size_t)r * (K / 2) + i / 2];
      const int c = (i & 1) ? byte >> 4 : byte & 15;
      const int sb = scales[(size_t)r * (K / blk) + i / blk];
      const double sc = fmt == kMXFP4 ? e8m0_value(sb) : e4m3_value(sb);
      out[(size_t)r * K + i] = e2m1_value(c) * sc * t;
    }
  }
}

// Element-wise encoders and SiLU over arrays (for the pins).
void orc_e2m1_encode_n(const double* q, long long n, uint8_t* out) {
  for (long long i = 0; i < n; ++i) out[i] = (uint8_t)e2m1_encode(q[i]);
}
void orc_e4m3_encode_n(const double* v, long long n, uint8_t* out) {
  for (long long i = 0; i < n; ++i) out[i] = (uint8_t)e4m3_encode_satfinite(v[i]);
}
void orc_silu_n(const double* z, long long n, double* out) {
  for (long long i = 0; i < n; ++i) out[i] = silu(z[i]);
}

// ---------------------------------------------------------------- quant
// MXFP4 activation quantiser (OCP MX v1.0 conversion) of fp32 rows v [rows, K]:
// per 32-block X = floor(log2(amax)) - 2 clamped to [-127, 127] (-127 for an
// all-zero block), codes = E2M1(v / 2^X) formed in fp32.
void orc_quant_mxfp4(const float* v, int rows, int K, uint8_t* codes, uint8_t* scales) {
#pragma omp parallel for num_threads(nthreads(g_threads)) schedule(static)
  for (int r = 0; r < rows; ++r) {
    for (int b = 0; b < K / 32; ++b) {
      const float* blk = v + (size_t)r * K + (size_t)b * 32;
      float amax = 0.f;
      for (int i = 0; i < 32; ++i) amax = std::fmax(amax, std::fabs(blk[i]));
      int X = -127;
      if (amax > 0.f) {
        int ex;
        std::frexp((double)amax, &ex);   // amax = m 2^ex, m in [0.5, 1)
        X = (ex - 1) - 2;
        X = X < -127 ? -127 : X > 127 ? 127 : X;
      }
      scales[(size_t)r * (K / 32) + b] = (uint8_t)(X + 127);
      for (int i = 0; i < 32; i += 2) {
        const float q0 = (float)((double)blk[i] * std::ldexp(1.0, -X));
        const float q1 = (float)((double)blk[i + 1] * std::ldexp(1.0, -X));
        codes[(size_t)r * (K / 2) + (size_t)b * 16 + i / 2] =
            (uint8_t)(e2m1_encode(q0) | (e2m1_encode(q1) << 4));
      }
    }
  }
}

// NVFP4 activation quantiser with static fp32 activation scale g: per
// 16-block scale = E4M3(amax / 6 / g) (fp32 IEEE quotients, nearest-even,
// saturating), codes = E2M1(v / (scale g)) in fp32; scale 0 gives zero codes.
void orc_quant_nvfp4(const float* v, int rows, int K, float g, uint8_t* codes, uint8_t* scales) {
#pragma omp parallel for num_threads(nthreads(g_threads)) schedule(static)
  for (int r = 0; r < rows; ++r) {
    for (int b = 0; b < K / 16; ++b) {
      const float* blk = v + (size_t)r * K + (size_t)b * 16;
      float amax = 0.f;
      for (int i = 0; i < 16; ++i) amax = std::fmax(amax, std::fabs(blk[i]));
      const float s_raw = (amax / 6.0f) / g;
      const int sb = e4m3_encode_satfinite((double)s_raw);
      scales[(size_t)r * (K / 16) + b] = (uint8_t)sb;
      const float denom = (float)e4m3_value(sb) * g;
      for (int i = 0; i < 16; i += 2) {
        const float q0 = denom > 0.f ? blk[i] / denom : 0.0f;
        const float q1 = denom > 0.f ? blk[i + 1] / denom : 0.0f;
        codes[(size_t)r * (K / 2) + (size_t)b * 8 + i / 2] = (uint8_t)(e2m1_encode(q0) | (e2m1_encode(q1) << 4));
      }
    }
  }
}

// MXFP8 activation quantiser (OCP MX v1.0 conversion) of fp32 rows v [rows, K]:
// per 32-block X = floor(log2(amax)) - 8 clamped to [-127, 127] (-127 for an
// all-zero block), codes = E4M3(v / 2^X) (nearest even, saturating at 448,
// sign kept) formed in fp32; one code byte per element.
void orc_quant_mxfp8(const float* v, int rows, int K, uint8_t* codes, uint8_t* scales) {
#pragma omp parallel for num_threads(nthreads(g_threads)) schedule(static)
  for (int r = 0; r < rows; ++r) {
    for (int b = 0; b < K / 32; ++b) {
      const float* blk = v + (size_t)r * K + (size_t)b * 32;
      float amax = 0.f;
      for (int i = 0; i < 32; ++i) amax = std::fmax(amax, std::fabs(blk[i]));
      int X = -127;
      if (amax > 0.f) {
        int ex;
        std::frexp((double)amax, &ex);
        X = (ex - 1) - 8;
        X = X < -127 ? -127 : X > 127 ? 127 : X;
      }
      scales[(size_t)r * (K / 32) + b] = (uint8_t)(X + 127);
      for (int i = 0; i < 32; ++i) {
        const float q = (float)((double)blk[i] * std::ldexp(1.0, -X));
        codes[(size_t)r * K + (size_t)b * 32 + i] =
            (uint8_t)(e4m3_encode_satfinite(std::fabs((double)q)) | (std::signbit(q) ? 0x80 : 0));
      }
    }
  }
}

// v (FP64) rounded to fp32, then to bf16, nearest even, as FP64.
void orc_round_bf16_n(const double* v, long long n, double* out) {
  for (long long i = 0; i < n; ++i) out[i] = bf16_value(bf16_round_bits((float)v[i]));
}

// The values the prefill activation quantiser hands to the MMA, in FP64: v
// (rows x K, FP64) rounded to fp32, quantised to the weight's block format
// (FP4 weights), MXFP8 (MXFP8 weights) or rounded to bf16 (BF16 weights),
// dequantised (x g for NVFP4).
void orc_act_roundtrip(const double* v, int rows, int K, int fmt, float g, double* out) {
  if (fmt == kBF16) {
    orc_round_bf16_n(v, (long long)rows * K, out);
    return;
  }
  std::vector<float> v32((size_t)rows * K);
  for (size_t i = 0; i < v32.size(); ++i) v32[i] = (float)v[i];
  if (fmt == kMXFP8) {
    std::vector<uint8_t> c((size_t)rows * K), s((size_t)rows * K / 32);
    orc_quant_mxfp8(v32.data(), rows, K, c.data(), s.data());
    orc_dequant(c.data(), s.data(), rows, K, fmt, 1.0f, out);
    return;
  }
  const int blk = fmt == kMXFP4 ? 32 : 16;
  std::vector<uint8_t> c((size_t)rows * K / 2), s((size_t)rows * K / blk);
  if (fmt == kMXFP4) orc_quant_mxfp4(v32.data(), rows, K, c.data(), s.data());
  else orc_quant_nvfp4(v32.data(), rows, K, g, c.data(), s.data());
  orc_dequant(c.data(), s.data(), rows, K, fmt, 1.0f, out);
  if (fmt == kNVFP4)
    for (size_t i = 0; i < (size_t)rows * K; ++i) out[i] *= (double)g;
}

// ---------------------------------------------------------------- router
// logits[t, e] = sum_i x[t, i] W_r[e, i] (+ b[e]) in FP64 (i ascending); the
// k largest logits, ties to the lower id, emitted ascending; gates = softmax
// over the selected logits (norm_topk) or the full softmax probabilities.
void orc_router(const double* x, const float* Wr, const float* bias, int N, int d, int E, int k, int norm_topk,
                int* idx, double* gates, double* logits) {
#pragma omp parallel for num_threads(nthreads(g_threads)) schedule(static)
  for (int t = 0; t < N; ++t) {
    std::vector<double> L(E);
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int i = 0; i < d; ++i) acc += x[(size_t)t * d + i] * (double)Wr[(size_t)e * d + i];
      L[e] = acc + (bias ? (double)bias[e] : 0.0);
      if (logits) logits[(size_t)t * E + e] = L[e];
    }
    // selection: k rounds of "largest remaining, lowest id on ties"
    std::vector<char> taken(E, 0);
    std::vector<int> sel;
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || L[e] > L[best])) best = e;
      taken[best] = 1;
      sel.push_back(best);
    }
    double m = L[0];
    for (int e = 1; e < E; ++e) m = std::fmax(m, L[e]);
    // ascending expert order
    std::vector<int> asc;
    for (int e = 0; e < E; ++e)
      if (taken[e]) asc.push_back(e);
    double den = 0.0;
    if (norm_topk) {
      for (int e : asc) den += std::exp(L[e] - m);
    } else {
      for (int e = 0; e < E; ++e) den += std::exp(L[e] - m);
    }
    for (int j = 0; j < k; ++j) {
      idx[(size_t)t * k + j] = asc[j];
      gates[(size_t)t * k + j] = std::exp(L[asc[j]] - m) / den;
    }
  }
}

// ---------------------------------------------------------------- permute
// counts[e]; offsets = exclusive prefix sum (ascending e), offsets[E] = N k;
// row_of[t, j] = offsets[e] + #{t' < t routed to e}; tok_of[row] = t.
void orc_permute(const int* idx, int N, int k, int E, long long* counts, long long* offsets, long long* row_of,
                 long long* tok_of) {
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (long long p = 0; p < (long long)N * k; ++p) counts[idx[p]] += 1;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  std::vector<long long> fill(offsets, offsets + E);
  for (int t = 0; t < N; ++t)
    for (int j = 0; j < k; ++j) {
      const int e = idx[(size_t)t * k + j];
      row_of[(size_t)t * k + j] = fill[e];
      tok_of[fill[e]] = t;
      fill[e] += 1;
    }
}

// ---------------------------------------------------------------- expert
// out[r] = W_d (SiLU(W_g X[r]) * (W_u X[r])) for n rows X [n, d] (FP64
// dequantised weights Wg, Wu [f, d], Wd [d, f]).  regime 1 (prefill): X and
// h pass through the block quantiser of the activation format `fmt` first
// (the weights' own format, or MXFP8 on MXFP4 weights; NVFP4 scales gx, gh).
void orc_expert_ffn(const double* X, int n, int d, int f, const double* Wg, const double* Wu, const double* Wd,
                    int regime, int fmt, float gx, float gh, double* out) {
  std::vector<double> Xq;
  const double* xin = X;
  if (regime == 1) {
    Xq.resize((size_t)n * d);
    orc_act_roundtrip(X, n, d, fmt, gx, Xq.data());
    xin = Xq.data();
  }
  std::vector<double> h((size_t)n * f);
#pragma omp parallel for num_threads(nthreads(g_threads)) schedule(static)
  for (int r = 0; r < n; ++r) {
    const double* xr = xin + (size_t)r * d;
    for (int o = 0; o < f; ++o) {
      double a = 0.0, u = 0.0;
      for (int i = 0; i < d; ++i) {
        a += Wg[(size_t)o * d + i] * xr[i];
        u += Wu[(size_t)o * d + i] * xr[i];
      }
      h[(size_t)r * f + o] = silu(a) * u;
    }
  }
  if (regime == 1) {
    std::vector<double> hq((size_t)n * f);
    orc_act_roundtrip(h.data(), n, f, fmt, gh, hq.data());
    h.swap(hq);
  }
#pragma omp parallel for num_threads(nthreads(g_threads)) schedule(static)
  for (int r = 0; r < n; ++r) {
    for (int o = 0; o < d; ++o) {
      double acc = 0.0;
      for (int i = 0; i < f; ++i) acc += Wd[(size_t)o * f + i] * h[(size_t)r * f + i];
      out[(size_t)r * d + o] = acc;
    }
  }
}

// ---------------------------------------------------------------- combine
// y[t] = sum_j gates[t, j] O[row_of[t, j]] (j ascending) + shared[t] (if any).
void orc_combine(const double* O, const double* gates, const long long* row_of, int N, int k, int d,
                 const double* shared, double* y) {
#pragma omp parallel for num_threads(nthreads(g_threads)) schedule(static)
  for (int t = 0; t < N; ++t)
    for (int c = 0; c < d; ++c) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j) acc += gates[(size_t)t * k + j] * O[(size_t)row_of[(size_t)t * k + j] * d + c];
      if (shared) acc += shared[(size_t)t * d + c];
      y[(size_t)t * d + c] = acc;
    }
}

// ---------------------------------------------------------------- LRU
// The textbook slot table: expert per slot (-1 free), a recency stamp per
// slot from a counter that ticks once per access, the victim is the occupied
// slot with the smallest stamp.
struct OrcLru {
  int E, S;
  std::vector<int> slot_of, expert_of;
  std::vector<unsigned long long> stamp;
  unsigned long long clock;
};

void* orc_lru_new(int E, int S) {
  OrcLru* L = new OrcLru();
  L->E = E;
  L->S = S;
  L->slot_of.assign(E, -1);
  L->expert_of.assign(S, -1);
  L->stamp.assign(S, 0);
  L->clock = 0;
  return L;
}

void orc_lru_free(void* h) { delete static_cast<OrcLru*>(h); }

// Put expert e into slot s as most recently used.
void orc_lru_install(void* h, int e, int s) {
  OrcLru* L = static_cast<OrcLru*>(h);
  if (L->slot_of[e] >= 0) L->expert_of[L->slot_of[e]] = -1;
  const int old = L->expert_of[s];
  if (old >= 0) L->slot_of[old] = -1;
  L->expert_of[s] = e;
  L->slot_of[e] = s;
  L->clock += 1;
  L->stamp[s] = L->clock;
}

// One step: the distinct experts of routed[0..n), hits first (ascending id),
// then misses (ascending id).  Per access (in order): expert, slot, hit,
// evicted expert (-1 none).  Returns the number of accesses.
int orc_lru_step(void* h, const int* routed, int n, int* acc_e, int* acc_s, int* acc_hit, int* acc_ev) {
  OrcLru* L = static_cast<OrcLru*>(h);
  std::vector<char> in(L->E, 0);
  for (int i = 0; i < n; ++i) in[routed[i]] = 1;
  std::vector<int> hits, misses;
  for (int e = 0; e < L->E; ++e)
    if (in[e]) (L->slot_of[e] >= 0 ? hits : misses).push_back(e);
  int a = 0;
  for (int e : hits) {
    const int s = L->slot_of[e];
    L->clock += 1;
    L->stamp[s] = L->clock;
    acc_e[a] = e;
    acc_s[a] = s;
    acc_hit[a] = 1;
    acc_ev[a] = -1;
    ++a;
  }
  for (int e : misses) {
    int s = -1;
    for (int q = 0; q < L->S && s < 0; ++q)
      if (L->expert_of[q] < 0) s = q;   // lowest free slot
    if (s < 0) {
      s = 0;
      for (int q = 1; q < L->S; ++q)
        if (L->stamp[q] < L->stamp[s]) s = q;   // least recently used
    }
    const int ev = L->expert_of[s];
    if (ev >= 0) L->slot_of[ev] = -1;
    L->expert_of[s] = e;
    L->slot_of[e] = s;
    L->clock += 1;
    L->stamp[s] = L->clock;
    acc_e[a] = e;
    acc_s[a] = s;
    acc_hit[a] = 0;
    acc_ev[a] = ev;
    ++a;
  }
  return a;
}

// Resize between steps (the pages' elastic expert cache: resized at safe
// points, nothing reloaded): the min(S_new, occupied) most recently used
// experts stay with their stamps, moved to slots 0, 1, ... in the order of
// their old slots; the other slots are free; the clock is unchanged.
void orc_lru_resize(void* h, int S_new) {
  OrcLru* L = static_cast<OrcLru*>(h);
  std::vector<int> occ;
  for (int s = 0; s < L->S; ++s)
    if (L->expert_of[s] >= 0) occ.push_back(s);
  // the S_new largest stamps (stamps of occupied slots are distinct)
  std::vector<char> keep(L->S, 0);
  for (int n = 0; n < S_new && n < (int)occ.size(); ++n) {
    int best = -1;
    for (int s : occ)
      if (!keep[s] && (best < 0 || L->stamp[s] > L->stamp[best])) best = s;
    keep[best] = 1;
  }
  std::vector<int> eo(S_new, -1);
  std::vector<unsigned long long> st(S_new, 0);
  int i = 0;
  for (int s = 0; s < L->S; ++s)
    if (keep[s]) {
      eo[i] = L->expert_of[s];
      st[i] = L->stamp[s];
      ++i;
    }
  L->S = S_new;
  L->expert_of = eo;
  L->stamp = st;
  L->slot_of.assign(L->E, -1);
  for (int s = 0; s < S_new; ++s)
    if (eo[s] >= 0) L->slot_of[eo[s]] = s;
}

void orc_lru_state(void* h, int* expert_of, unsigned long long* stamp, unsigned long long* clock, int* slot_of) {
  OrcLru* L = static_cast<OrcLru*>(h);
  if (expert_of) std::memcpy(expert_of, L->expert_of.data(), sizeof(int) * L->S);
  if (stamp) std::memcpy(stamp, L->stamp.data(), sizeof(unsigned long long) * L->S);
  if (clock) *clock = L->clock;
  if (slot_of) std::memcpy(slot_of, L->slot_of.data(), sizeof(int) * L->E);
}

// Replace the table (e.g. to drop experts whose fill failed): expert_of [S]
// (-1 free) and stamps [S]; slot_of follows.
void orc_lru_set(void* h, const int* expert_of, const unsigned long long* stamp, unsigned long long clock) {
  OrcLru* L = static_cast<OrcLru*>(h);
  L->slot_of.assign(L->E, -1);
  for (int s = 0; s < L->S; ++s) {
    L->expert_of[s] = expert_of[s];
    L->stamp[s] = stamp[s];
    if (expert_of[s] >= 0) L->slot_of[expert_of[s]] = s;
  }
  L->clock = clock;
}

}  // extern "C"
