// ovc_oracle.cpp -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow CPU restatement of ExpCast FP8 attention (Open-VC attention)
// and of its V residual repair.  Only the test suite, the smoke check and the
// CPU-baseline leg of the benchmark use it; the product path never links it.
// It shares no source, header, table or constant generator with the CUDA
// library: every definition below is written again from the pages.
//
// Sources, by page title and section:
//   [OVC-news]   "Open-VC attention" news item (aikraft.ru): sections
//                "Problem: the MUFU bottleneck", "Solution: ExpCast",
//                "Architectural optimisations", "Results".
//   [OVC-mlllm]  "MachGen opened the sources of Open-VC Attention" (mlllm.io):
//                sections "What happened", "Context", "For users".
//   [OVC-lib]    "Open VC Attention" catalogue entry (ailibri.com).
//   [VC-summary] Bengali summary of "VC-Attention" (redirect domain):
//                sections "V-Smooth" and "ExpCast-FP8".
//
// Precision: the quantisation steps (per-block Q/K scales, per-head V scale,
// the E4M3 codes, the repair residuals and their energies) are defined in
// FP32 arithmetic so that codes and repair indices can be compared bit for
// bit; every FP32 step goes through a volatile so that neither FMA
// contraction nor extended precision changes it (the file is also compiled
// with -ffp-contract=off).  Everything downstream of the codes (scores,
// running max, row sum, output) is computed in double.
//
// Readings of the pages fixed here:
//   * stored probability v = 2^8 p, i.e. c0 = 120 in code = 8 log2(p) + c0 + beta;
//   * beta = -0.35, round half to even, clamp to [0, 126];
//   * lazy rescale threshold tau = 0.75 log2 units;
//   * the running reference m8 (units of 1/8 log2) is raised, when the block
//     max passes m8 + 8 tau, to the smallest value >= the block max on the
//     grid {k + frac(c0 + beta)}, so that c0 + beta - m8 is an integer;
//   * key blocks of 128 are visited cyclically from block floor(nb/2);
//   * the row sum l adds the decoded codes that enter P.V;
//   * repair: n = ceil(budget S) tokens per head, ranked by FP32 residual
//     energy (ties to the lower index), one residual scale per head.
// The tests pin every function against facts the pages or mathematics fix.

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

constexpr double kLog2e = 1.4426950408889634074;

// ---------------------------------------------------------------------------
// Rounding helpers.
// ---------------------------------------------------------------------------
double round_half_even(double x) {        // any sign, exact for |x| < 2^52
  const double f = std::floor(x);
  const double d = x - f;
  if (d > 0.5) return f + 1.0;
  if (d < 0.5) return f;
  return (std::fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

// ---------------------------------------------------------------------------
// E4M3 "fn" format, from its definition: 1 sign bit, 4 exponent bits (bias 7),
// 3 mantissa bits; no infinities; 0x7F and 0xFF are NaN; largest finite 448;
// exponent field 0 holds subnormals m * 2^-9.
// ---------------------------------------------------------------------------
double e4m3_value(uint8_t code) {
  const int sign = code >> 7;
  const int e = (code >> 3) & 15;
  const int m = code & 7;
  if (e == 15 && m == 7) return std::nan("");
  const double mag = (e == 0) ? std::ldexp(static_cast<double>(m), -9)
                              : std::ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -mag : mag;
}

// FP32 -> E4M3, round to nearest even, saturating to +-448.
uint8_t e4m3_from_float(float x) {
  if (std::isnan(x)) return 0x7F;
  const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  const double a = std::fabs(static_cast<double>(x));
  if (a >= 448.0) return sign | 0x7E;
  double quantum;   // spacing of representable values around |x|
  int first_code;   // code of the first value with that spacing
  if (a < std::ldexp(1.0, -6)) {
    quantum = std::ldexp(1.0, -9);
    first_code = 0;
  } else {
    int e2;
    std::frexp(a, &e2);           // a in [2^(e2-1), 2^e2)
    const int E = e2 - 1;
    quantum = std::ldexp(1.0, E - 3);
    first_code = (E + 7) * 8 - 8;  // 2^E has code (E+7)*8 = first_code + 8
  }
  const double steps = round_half_even(a / quantum);
  return sign | static_cast<uint8_t>(first_code + static_cast<int>(steps));
}

float bf16_bits_to_float(uint16_t b) {
  const uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// IEEE binary16 bits -> value, from the format definition: 1 sign bit, 5
// exponent bits (bias 15), 10 fraction bits; exponent 0 is subnormal
// (f * 2^-24), exponent 31 is Inf/NaN.  Every binary16 value is exact in FP32.
float half_bits_to_float(uint16_t h) {
  const int sign = h >> 15, e = (h >> 10) & 31, f = h & 1023;
  double v;
  if (e == 0) v = std::ldexp(static_cast<double>(f), -24);
  else if (e == 31) v = f ? NAN : INFINITY;
  else v = std::ldexp(1.0 + f / 1024.0, e - 15);
  return static_cast<float>(sign ? -v : v);
}

// Input element (BF16 or FP16 bits, the two input types of the API
// ["Open VC Attention" catalogue entry: FP16 or BF16 inputs]) -> FP32.
float input_bits_to_float(uint16_t b, int fp16) { return fp16 ? half_bits_to_float(b) : bf16_bits_to_float(b); }

// double -> BF16 with a single round to nearest even.
uint16_t bf16_from_double(double x) {
  if (std::isnan(x)) return 0x7FC0;
  const uint16_t sign = std::signbit(x) ? 0x8000 : 0;
  const double a = std::fabs(x);
  if (a == 0.0) return sign;
  int e2;
  std::frexp(a, &e2);
  int E = e2 - 1;
  if (E < -126) E = -126;                      // subnormal spacing 2^-133
  const double quantum = std::ldexp(1.0, E - 7);
  const double r = round_half_even(a / quantum) * quantum;
  if (r >= std::ldexp(1.0, 128)) return sign | 0x7F80;
  const float f = static_cast<float>(r);       // exact: <= 8 significant bits
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return sign | static_cast<uint16_t>(u >> 16);
}

// ---------------------------------------------------------------------------
// FP32-defined quantisation.  [OVC-lib: Q/K scales per block, V per head]
// s = fl(amax / 448), r = fl(448 / amax); amax = 0 -> s = r = 1;
// code = E4M3(fl(x * r)).
// ---------------------------------------------------------------------------
struct Scale {
  float s;
  float r;
};

Scale scale_from_amax(float amax) {
  if (amax == 0.0f) return {1.0f, 1.0f};
  volatile float a = amax;
  volatile float s = a / 448.0f;
  volatile float r = 448.0f / a;
  return {s, r};
}

uint8_t quantize_value(float x, float r) {
  volatile float y = x * r;
  return e4m3_from_float(y);
}

// V residual of one element: R = fl(v - fl(s_v * dec(code))).
float v_residual(float v, uint8_t code, float sv) {
  volatile float deq = sv * static_cast<float>(e4m3_value(code));
  volatile float r = v - deq;
  return r;
}

// Residual energy of one token in FP32, in a fixed order: sixteen partial
// sums over channels 8g..8g+7 taken left to right, then the pairwise tree
// p_g <- p_g + p_(g+w) for w = 8, 4, 2, 1.  Squares are rounded before they
// are added (no FMA).
float residual_energy(const float* R) {
  float p[16];
  for (int g = 0; g < 16; ++g) {
    volatile float acc = R[8 * g] * R[8 * g];
    for (int i = 1; i < 8; ++i) {
      volatile float sq = R[8 * g + i] * R[8 * g + i];
      acc = acc + sq;
    }
    p[g] = acc;
  }
  for (int w = 8; w >= 1; w /= 2) {
    for (int g = 0; g < w; ++g) {
      volatile float t = p[g] + p[g + w];
      p[g] = t;
    }
  }
  return p[0];
}

// ---------------------------------------------------------------------------
// Attention.
// ---------------------------------------------------------------------------
struct Params {
  double c0;        // code offset of p = 1 before beta (120 <=> v = 2^8 p)
  double beta;      // centring constant of the byte relation (-0.35)
  double tau;       // lazy-rescale threshold, log2 units (0.75)
  double sm;        // softmax scale
  int exact;        // 1: p = 2^((Z - m8)/8) exactly, no codes (skeleton pin)
  int mid_window;   // 1: cyclic from block floor(nb/2); 0: natural order
  int snap;         // 1: reference on the {k + frac(c0+beta)} grid; 0: = max
  int cast;         // 1: exp-then-cast bytes (the baseline) instead of ExpCast
};

// Key-block visiting order over the blocks [b0, b1) (the whole sequence, or
// one key range of a split).  [OVC-news "Architectural optimisations";
// OVC-lib: keys traversed from the middle of the window]
std::vector<int64_t> key_block_order(int64_t b0, int64_t b1, int mid_window) {
  const int64_t n = b1 - b0;
  std::vector<int64_t> order(n);
  const int64_t start = mid_window ? n / 2 : 0;
  for (int64_t i = 0; i < n; ++i) order[i] = b0 + (start + i) % n;
  return order;
}

// Key range of split s of n: blocks [floor(s nb / n), floor((s+1) nb / n)).
void split_range(int64_t nb, int64_t n, int64_t s, int64_t* b0, int64_t* b1) {
  *b0 = s * nb / n;
  *b1 = (s + 1) * nb / n;
}

// One head, decoded to double.  Keys and values are token-major [S][128].
struct HeadView {
  int64_t S = 0;
  int64_t nb = 0;
  const double* K = nullptr;       // key values (decoded codes or raw)
  const double* kscale = nullptr;  // [nb]
  const double* V = nullptr;       // value values, unscaled
  double vscale = 1.0;
  const double* kbias = nullptr;   // Q smoothing: beta_t = mu_q . k_t per key (NULL: none)
  int64_t n_rep = 0;               // repair set
  const int32_t* rep_idx = nullptr;
  const double* dV = nullptr;      // [n_rep][128] decoded residual codes
  double rscale = 1.0;
};

struct RowResult {
  double O[128];
  double m8;
  double l;
  int32_t nrescale;
  int32_t nrescale_repair;
};

// ExpCast probability of a score.  Z is the log2-domain score in code units
// (Z = 8 z); code = clamp(rint(Z - m8 + c0 + beta), 0, 126), p = dec(code).
// [VC-summary "ExpCast-FP8": an E4M3 byte read as an integer is about
// 8 log2(v) + 56; one FMA writes it; beta = -0.35]  [OVC-news "Solution"]
double expcast_p(double Z, double m8, const Params& P, uint8_t* code_out) {
  if (P.exact) {
    if (code_out) *code_out = 0;
    return std::exp2((Z - m8) / 8.0);
  }
  double t = round_half_even(Z - m8 + P.c0 + P.beta);
  t = std::min(126.0, std::max(0.0, t));
  const uint8_t c = static_cast<uint8_t>(t);
  if (code_out) *code_out = c;
  return e4m3_value(c);
}

// Exp-then-cast probability, the path ExpCast replaces: the stored value
// v = 2^((Z - m8 + c0 - 56) / 8) (= 2^8 p for c0 = 120) is computed, held in
// FP32 and converted to E4M3 with round to nearest even and saturation;
// p = dec(code).  [OVC-news "Problem": one exponent per score and a
// conversion to FP8; VC-summary "ExpCast-FP8": the exp-then-cast path whose
// bytes ExpCast matches on 79.6% of entries]
double exp_cast_p(double Z, double m8, const Params& P, uint8_t* code_out) {
  const double v = std::exp2((Z - m8 + P.c0 - 56.0) / 8.0);
  const uint8_t c = e4m3_from_float(static_cast<float>(v));
  if (code_out) *code_out = c;
  return e4m3_value(c);
}

// Probability of one score under the configured byte path.
double prob(double Z, double m8, const Params& P, uint8_t* code_out) {
  return (P.cast && !P.exact) ? exp_cast_p(Z, m8, P, code_out) : expcast_p(Z, m8, P, code_out);
}

// Lazy rescale of the running state.  [OVC-mlllm "Context": fewer rescales]
void maybe_rescale(double bm, const Params& P, double* m8, double* l, double* O, double* O2,
                   int32_t* count) {
  if (!(bm > *m8 + 8.0 * P.tau)) return;
  const double frac = (P.c0 + P.beta) - std::floor(P.c0 + P.beta);
  const double m_new = P.snap ? std::ceil(bm - frac) + frac : bm;
  const double f = std::exp2((*m8 - m_new) / 8.0);   // 0 for the first block
  for (int d = 0; d < 128; ++d) O[d] *= f;
  if (O2)
    for (int d = 0; d < 128; ++d) O2[d] *= f;
  *l *= f;
  *m8 = m_new;
  ++*count;
}

double dot128(const double* a, const double* b) {
  double s = 0.0;
  for (int d = 0; d < 128; ++d) s += a[d] * b[d];
  return s;
}

// One query row against every key of its head.  [OVC-lib: non-causal
// forward MHA, head dim 128; OVC-news "Solution"; VC-summary "V-Smooth":
// the row sum kept by online softmax]
void attend_row(const double* q, double qscale, const HeadView& hv, const Params& P,
                RowResult* res, int64_t dump_block, uint8_t* dump_codes, double* dump_m8,
                int64_t b0 = 0, int64_t b1 = -1) {
  if (b1 < 0) b1 = hv.nb;
  double m8 = -INFINITY;
  double l = 0.0;
  double O[128], Orep[128];
  for (int d = 0; d < 128; ++d) O[d] = Orep[d] = 0.0;
  int32_t nres = 0, nres_rep = 0;
  double Z[128];

  const std::vector<int64_t> order = key_block_order(b0, b1, P.mid_window);
  for (int64_t i = 0; i < b1 - b0; ++i) {
    const int64_t j = order[i];
    const int64_t k0 = j * 128;
    const int64_t nk = std::min<int64_t>(128, hv.S - k0);   // tail block
    const double a = 8.0 * kLog2e * P.sm * qscale * hv.kscale[j];
    const double ab = 8.0 * kLog2e * P.sm * hv.kscale[j];   // Q smoothing's bias term
    double bm = -INFINITY;
    for (int64_t c = 0; c < nk; ++c) {
      Z[c] = a * dot128(q, hv.K + (k0 + c) * 128);
      if (hv.kbias) Z[c] += ab * hv.kbias[k0 + c];
      bm = std::max(bm, Z[c]);
    }
    maybe_rescale(bm, P, &m8, &l, O, nullptr, &nres);
    const bool dump = dump_codes && j == dump_block;
    if (dump && dump_m8) *dump_m8 = m8;
    for (int64_t c = 0; c < nk; ++c) {
      uint8_t code = 0;
      const double p = prob(Z[c], m8, P, &code);
      if (dump) dump_codes[c] = code;
      l += p;
      const double* vr = hv.V + (k0 + c) * 128;
      for (int d = 0; d < 128; ++d) O[d] += p * vr[d];
    }
    if (dump)
      for (int64_t c = nk; c < 128; ++c) dump_codes[c] = 0;
  }

  // V residual repair: the selected keys once more, with their quantised
  // residuals as values; they add to the output, not to the row sum.
  // [OVC-lib: prepare_v_repair(budget) and attention_v_repair;
  //  OVC-mlllm "What happened": residuals re-added for the worst tokens]
  for (int64_t r0 = 0; r0 < hv.n_rep; r0 += 128) {
    const int64_t nk = std::min<int64_t>(128, hv.n_rep - r0);
    double bm = -INFINITY;
    for (int64_t c = 0; c < nk; ++c) {
      const int64_t t = hv.rep_idx[r0 + c];
      const double a = 8.0 * kLog2e * P.sm * qscale * hv.kscale[t / 128];
      Z[c] = a * dot128(q, hv.K + t * 128);
      if (hv.kbias) Z[c] += 8.0 * kLog2e * P.sm * hv.kscale[t / 128] * hv.kbias[t];
      bm = std::max(bm, Z[c]);
    }
    maybe_rescale(bm, P, &m8, &l, O, Orep, &nres_rep);   // never fires: keys already seen
    for (int64_t c = 0; c < nk; ++c) {
      const double p = prob(Z[c], m8, P, nullptr);
      const double* dv = hv.dV + (r0 + c) * 128;
      for (int d = 0; d < 128; ++d) Orep[d] += p * dv[d];
    }
  }

  for (int d = 0; d < 128; ++d) res->O[d] = (hv.vscale * O[d] + hv.rscale * Orep[d]) / l;
  res->m8 = m8;
  res->l = l;
  res->nrescale = nres;
  res->nrescale_repair = nres_rep;
}

// Split key ranges (short sequences): each of the n ranges runs its own
// online softmax (own reference m8_s, row sum l_s, output O_s = s_v O_acc/l_s),
// then the ranges are merged exactly: with M = max m8_s and
// w_s = l_s 2^((m8_s - M)/8), O = sum w_s O_s / sum w_s.  This is the
// standard merge of partial softmax results; it changes only where each
// range's ExpCast reference sits.  No repair set (the caller checks).
void attend_row_split(const double* q, double qscale, const HeadView& hv, const Params& P, int64_t nsplit,
                      RowResult* res, int64_t dump_block, uint8_t* dump_codes, double* dump_m8) {
  if (nsplit <= 1) {
    attend_row(q, qscale, hv, P, res, dump_block, dump_codes, dump_m8);
    return;
  }
  std::vector<RowResult> part(nsplit);
  double M = -INFINITY;
  int32_t nres = 0;
  for (int64_t s = 0; s < nsplit; ++s) {
    int64_t b0, b1;
    split_range(hv.nb, nsplit, s, &b0, &b1);
    const bool mine = dump_block >= b0 && dump_block < b1;
    attend_row(q, qscale, hv, P, &part[s], mine ? dump_block : -1, mine ? dump_codes : nullptr,
               mine ? dump_m8 : nullptr, b0, b1);
    M = std::max(M, part[s].m8);
    nres += part[s].nrescale;
  }
  double W = 0.0, O[128];
  for (int d = 0; d < 128; ++d) O[d] = 0.0;
  for (int64_t s = 0; s < nsplit; ++s) {
    const double w = part[s].l * std::exp2((part[s].m8 - M) / 8.0);
    W += w;
    for (int d = 0; d < 128; ++d) O[d] += w * part[s].O[d];
  }
  for (int d = 0; d < 128; ++d) res->O[d] = O[d] / W;
  res->m8 = M;
  res->l = W;
  res->nrescale = nres;
  res->nrescale_repair = 0;
}

template <class F>
void parallel_for(int64_t n, int nthreads, F&& fn) {
  if (nthreads <= 1 || n <= 1) {
    for (int64_t i = 0; i < n; ++i) fn(i);
    return;
  }
  std::atomic<int64_t> next{0};
  std::vector<std::thread> pool;
  const int nt = static_cast<int>(std::min<int64_t>(nthreads, n));
  for (int t = 0; t < nt; ++t)
    pool.emplace_back([&]() {
      for (int64_t i = next.fetch_add(1); i < n; i = next.fetch_add(1)) fn(i);
    });
  for (auto& th : pool) th.join();
}

struct Dims {
  int64_t B, S, H, nb, S_pad;
};

Dims make_dims(int64_t B, int64_t S, int64_t H) {
  const int64_t nb = (S + 127) / 128;
  return {B, S, H, nb, nb * 128};
}

}  // namespace

extern "C" {

double ovc_oracle_e4m3_value(uint8_t code) { return e4m3_value(code); }
uint8_t ovc_oracle_e4m3_from_float(float x) { return e4m3_from_float(x); }
uint16_t ovc_oracle_bf16_from_double(double x) { return bf16_from_double(x); }
float ovc_oracle_residual_energy(const float* R) { return residual_energy(R); }
float ovc_oracle_half_bits_to_float(uint16_t h) { return half_bits_to_float(h); }

// ExpCast code of one score: clamp(rint(Z - m8 + c0 + beta), 0, 126).
uint8_t ovc_oracle_expcast_code(double Z, double m8, double c0, double beta) {
  const Params P{c0, beta, 0.75, 1.0, 0, 1, 1, 0};
  uint8_t code = 0;
  expcast_p(Z, m8, P, &code);
  return code;
}

// Exp-then-cast code of one score: E4M3(fl32(2^((Z - m8 + c0 - 56) / 8))).
uint8_t ovc_oracle_exp_cast_code(double Z, double m8, double c0) {
  const Params P{c0, -0.35, 0.75, 1.0, 0, 1, 1, 1};
  uint8_t code = 0;
  exp_cast_p(Z, m8, P, &code);
  return code;
}

// K smoothing (optional; prior art the VC-Attention summary names in "Why
// attention is the video bottleneck": earlier low-bit kernels smooth Q and K).
// For non-causal attention, subtracting a per-channel constant mu from every
// key changes each score row by the constant q.mu, so the softmax is
// unchanged; what changes is the quantisation, whose per-block amax no
// longer carries the channel offset.  mu is defined in FP32 with a fixed
// order: per 128-token block a sequential sum over its tokens, then a
// sequential sum of the block sums, then one division by S.
//   mean: [B,H,128]
void ovc_oracle_k_mean(const uint16_t* x, int fp16, int64_t B, int64_t S, int64_t H, int64_t sb,
                       int64_t ss, int64_t sh, float* mean) {
  const Dims dm = make_dims(B, S, H);
  for (int64_t b = 0; b < B; ++b)
    for (int64_t h = 0; h < H; ++h)
      for (int d = 0; d < 128; ++d) {
        volatile float total = 0.0f;
        for (int64_t j = 0; j < dm.nb; ++j) {
          volatile float part = 0.0f;
          for (int64_t t = j * 128; t < std::min(S, j * 128 + 128); ++t)
            part = part + input_bits_to_float(x[b * sb + t * ss + h * sh + d], fp16);
          total = total + part;
        }
        volatile float m = total / static_cast<float>(S);
        mean[(b * H + h) * 128 + d] = m;
      }
}

// Q or K quantisation.  x: BF16 (fp16 = 0) or FP16 bits of a [B,S,H,128] tensor with element
// strides (sb, ss, sh) and unit channel stride; mean: NULL, or [B,H,128]
// channel means subtracted (in FP32) before quantising (K smoothing).
// codes: [B,H,S_pad,128], rows >= S are zero.  scales: [B,H,nb].
void ovc_oracle_quantize_blocks(const uint16_t* x, int fp16, int64_t B, int64_t S, int64_t H, int64_t sb,
                                int64_t ss, int64_t sh, const float* mean, uint8_t* codes, float* scales) {
  const Dims dm = make_dims(B, S, H);
  for (int64_t b = 0; b < B; ++b)
    for (int64_t h = 0; h < H; ++h)
      for (int64_t j = 0; j < dm.nb; ++j) {
        const int64_t t0 = j * 128, t1 = std::min(S, t0 + 128);
        const float* mu = mean ? mean + (b * H + h) * 128 : nullptr;
        auto value = [&](int64_t t, int d) {
          const float v = input_bits_to_float(x[b * sb + t * ss + h * sh + d], fp16);
          if (!mu) return v;
          volatile float r = v - mu[d];
          return static_cast<float>(r);
        };
        float amax = 0.0f;
        for (int64_t t = t0; t < t1; ++t)
          for (int d = 0; d < 128; ++d) amax = std::max(amax, std::fabs(value(t, d)));
        const Scale sc = scale_from_amax(amax);
        scales[(b * H + h) * dm.nb + j] = sc.s;
        uint8_t* out = codes + ((b * H + h) * dm.S_pad + t0) * 128;
        for (int64_t t = t0; t < t0 + 128; ++t)
          for (int d = 0; d < 128; ++d) out[(t - t0) * 128 + d] = (t < S) ? quantize_value(value(t, d), sc.r) : 0;
      }
}

// V quantisation with one scale per head.  codes: token-major [B,H,S_pad,128]
// (rows >= S zero); sv: [B,H]; energy: [B,H,S] residual energy per token.
void ovc_oracle_quantize_v(const uint16_t* v, int fp16, int64_t B, int64_t S, int64_t H, int64_t sb,
                           int64_t ss, int64_t sh, uint8_t* codes, float* sv, float* energy) {
  const Dims dm = make_dims(B, S, H);
  for (int64_t b = 0; b < B; ++b)
    for (int64_t h = 0; h < H; ++h) {
      float amax = 0.0f;
      for (int64_t t = 0; t < S; ++t)
        for (int d = 0; d < 128; ++d)
          amax = std::max(amax, std::fabs(input_bits_to_float(v[b * sb + t * ss + h * sh + d], fp16)));
      const Scale sc = scale_from_amax(amax);
      sv[b * H + h] = sc.s;
      uint8_t* out = codes + (b * H + h) * dm.S_pad * 128;
      for (int64_t t = 0; t < dm.S_pad; ++t) {
        float R[128];
        for (int d = 0; d < 128; ++d) {
          if (t < S) {
            const float x = input_bits_to_float(v[b * sb + t * ss + h * sh + d], fp16);
            const uint8_t c = quantize_value(x, sc.r);
            out[t * 128 + d] = c;
            R[d] = v_residual(x, c, sc.s);
          } else {
            out[t * 128 + d] = 0;
          }
        }
        if (t < S && energy) energy[(b * H + h) * S + t] = residual_energy(R);
      }
    }
}

// V-Smooth, the VC-Attention paper's treatment of V ([VC-summary "V-Smooth"]:
// each 128-token hardware block subtracts its mean, only the residual is
// quantised, and the mean is added back through the row sums that online
// softmax keeps).  Per head and block b (the tail block: its valid tokens):
//   mu_b  = bf16( fl( (sum of v_t over the block, FP32 in token order) / n_b ) )
//   R_t   = fl(v_t - mu_b)
//   one scale per head from amax |R| (as for V),  code_t = E4M3(fl(R_t r))
// The value restored for token t is s dec(code_t) + mu_b, with mu_b as
// stored: 16 bits per 128 elements of a channel (0.125 bit per element, as
// the summary states).  The restore itself is exact here (attention_rows
// adds mu_b / s in double before the final multiplication by s).
//   codes [B,H,S_pad,128] token-major; sv [B,H]; mu [B,H,nb,128].
void ovc_oracle_vsmooth_v(const uint16_t* v, int fp16, int64_t B, int64_t S, int64_t H, int64_t sb, int64_t ss,
                          int64_t sh, uint8_t* codes, float* sv, float* mu) {
  const Dims dm = make_dims(B, S, H);
  std::vector<float> R(static_cast<size_t>(S) * 128);
  for (int64_t b = 0; b < B; ++b)
    for (int64_t h = 0; h < H; ++h) {
      const int64_t bh = b * H + h;
      float amax = 0.0f;
      for (int64_t j = 0; j < dm.nb; ++j) {
        const int64_t t0 = j * 128, t1 = std::min(S, t0 + 128);
        for (int d = 0; d < 128; ++d) {
          volatile float sum = 0.0f;
          for (int64_t t = t0; t < t1; ++t) sum = sum + input_bits_to_float(v[b * sb + t * ss + h * sh + d], fp16);
          volatile float mean = sum / static_cast<float>(t1 - t0);
          const float m = bf16_bits_to_float(bf16_from_double(static_cast<double>(mean)));
          mu[(bh * dm.nb + j) * 128 + d] = m;
          for (int64_t t = t0; t < t1; ++t) {
            volatile float r = input_bits_to_float(v[b * sb + t * ss + h * sh + d], fp16) - m;
            R[t * 128 + d] = r;
            amax = std::max(amax, std::fabs(static_cast<float>(r)));
          }
        }
      }
      const Scale sc = scale_from_amax(amax);
      sv[bh] = sc.s;
      uint8_t* out = codes + bh * dm.S_pad * 128;
      for (int64_t t = 0; t < dm.S_pad; ++t)
        for (int d = 0; d < 128; ++d) out[t * 128 + d] = t < S ? quantize_value(R[t * 128 + d], sc.r) : 0;
    }
}

// V-Smooth's grouping step ([VC-summary "V-Smooth": online k-means clusters
// each head's value tokens; keys and values are permuted together, which
// leaves non-causal attention unchanged): Lloyd's k-means with C clusters and
// `iters` assignment steps, then the tokens ordered by (cluster, index).  The
// summary gives neither C, the iteration count nor the start; the reading
// here is the plainest one, computed in double:
//   start:   mu_c = x_(floor(c S / C)), c = 0..C-1
//   assign:  the cluster with the smallest squared distance sum_d (x_d - mu_cd)^2,
//            ties to the lower c
//   update:  mu_c = mean of its tokens; a cluster with no token keeps its
//            centroid
// One iteration is assign then update; the labels returned are those of the
// last assignment, and centroids [B,H,C,128] the centroids it used.
int ovc_oracle_kmeans_group(const uint16_t* v, int fp16, int64_t B, int64_t S, int64_t H, int64_t sb, int64_t ss,
                            int64_t sh, int64_t C, int64_t iters, int32_t* labels, double* centroids, int32_t* perm) {
  if (C < 1 || C > S || iters < 1) return 1;
  std::vector<double> x(static_cast<size_t>(S) * 128), mu(static_cast<size_t>(C) * 128);
  std::vector<double> sum(static_cast<size_t>(C) * 128);
  std::vector<int64_t> cnt(C);
  for (int64_t b = 0; b < B; ++b)
    for (int64_t h = 0; h < H; ++h) {
      const int64_t bh = b * H + h;
      for (int64_t t = 0; t < S; ++t)
        for (int d = 0; d < 128; ++d) x[t * 128 + d] = input_bits_to_float(v[b * sb + t * ss + h * sh + d], fp16);
      for (int64_t c = 0; c < C; ++c)
        std::memcpy(&mu[c * 128], &x[(c * S / C) * 128], 128 * sizeof(double));
      int32_t* lab = labels + bh * S;
      for (int64_t it = 0; it < iters; ++it) {
        if (it + 1 == iters) std::memcpy(centroids + bh * C * 128, mu.data(), C * 128 * sizeof(double));
        for (int64_t t = 0; t < S; ++t) {
          double best = INFINITY;
          int32_t arg = 0;
          for (int64_t c = 0; c < C; ++c) {
            double dist = 0.0;
            for (int d = 0; d < 128; ++d) {
              const double e = x[t * 128 + d] - mu[c * 128 + d];
              dist += e * e;
            }
            if (dist < best) best = dist, arg = static_cast<int32_t>(c);
          }
          lab[t] = arg;
        }
        if (it + 1 == iters) break;
        std::fill(sum.begin(), sum.end(), 0.0);
        std::fill(cnt.begin(), cnt.end(), 0);
        for (int64_t t = 0; t < S; ++t) {
          ++cnt[lab[t]];
          for (int d = 0; d < 128; ++d) sum[lab[t] * 128 + d] += x[t * 128 + d];
        }
        for (int64_t c = 0; c < C; ++c)
          if (cnt[c] > 0)
            for (int d = 0; d < 128; ++d) mu[c * 128 + d] = sum[c * 128 + d] / static_cast<double>(cnt[c]);
      }
      // tokens ordered by (cluster, index)
      std::vector<int32_t> order(S);
      for (int64_t t = 0; t < S; ++t) order[t] = static_cast<int32_t>(t);
      std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t c) { return lab[a] < lab[c]; });
      std::memcpy(perm + bh * S, order.data(), S * sizeof(int32_t));
    }
  return 0;
}

// Number of repaired tokens per head: n = ceil(budget * S), at least 1.
int64_t ovc_oracle_repair_count(int64_t S, float budget) {
  const double n = std::ceil(static_cast<double>(budget) * static_cast<double>(S));
  return std::max<int64_t>(1, std::min<int64_t>(S, static_cast<int64_t>(n)));
}

// Repair selection: per head the n tokens with the largest energy, ties to
// the lower index, returned in ascending index order.  energy: [BH,S];
// idx: [BH,n].
void ovc_oracle_repair_select(const float* energy, int64_t BH, int64_t S, int64_t n, int32_t* idx) {
  std::vector<int32_t> order(S);
  for (int64_t bh = 0; bh < BH; ++bh) {
    const float* e = energy + bh * S;
    for (int64_t t = 0; t < S; ++t) order[t] = static_cast<int32_t>(t);
    std::stable_sort(order.begin(), order.end(),
                     [&](int32_t a, int32_t b) { return e[a] > e[b]; });
    std::vector<int32_t> top(order.begin(), order.begin() + n);
    std::sort(top.begin(), top.end());
    std::memcpy(idx + bh * n, top.data(), n * sizeof(int32_t));
  }
}

// Repair quantisation: residuals of the selected tokens, one scale per head
// s_r = amax|R_sel| / 448, codes E4M3(fl(R * r_r)).  vcodes: token-major
// [B,H,S_pad,128]; idx: [B,H,n]; dcodes: [B,H,n,128]; sr: [B,H].
void ovc_oracle_repair_quantize(const uint16_t* v, int fp16, int64_t B, int64_t S, int64_t H, int64_t sb,
                                int64_t ss, int64_t sh, const uint8_t* vcodes, const float* sv,
                                const int32_t* idx, int64_t n, uint8_t* dcodes, float* sr) {
  const Dims dm = make_dims(B, S, H);
  std::vector<float> R(n * 128);
  for (int64_t b = 0; b < B; ++b)
    for (int64_t h = 0; h < H; ++h) {
      const int64_t bh = b * H + h;
      float amax = 0.0f;
      for (int64_t i = 0; i < n; ++i) {
        const int64_t t = idx[bh * n + i];
        for (int d = 0; d < 128; ++d) {
          const float x = input_bits_to_float(v[b * sb + t * ss + h * sh + d], fp16);
          R[i * 128 + d] = v_residual(x, vcodes[(bh * dm.S_pad + t) * 128 + d], sv[bh]);
          amax = std::max(amax, std::fabs(R[i * 128 + d]));
        }
      }
      const Scale sc = scale_from_amax(amax);
      sr[bh] = sc.s;
      for (int64_t i = 0; i < n * 128; ++i) dcodes[bh * n * 128 + i] = quantize_value(R[i], sc.r);
    }
}

// Codes of one key block for one query row against a given reference m8
// (used to compare the device's P bytes under the device's own reference);
// cast = 1 gives the exp-then-cast bytes.
void ovc_oracle_block_codes(const uint8_t* qrow, float sq, const uint8_t* kcodes_head,
                            const float* sk_head, const double* kbias_head, int64_t S, int64_t j, double m8,
                            double c0, double beta, double sm, int cast, uint8_t* codes) {
  double q[128];
  for (int d = 0; d < 128; ++d) q[d] = e4m3_value(qrow[d]);
  Params P{c0, beta, 0.75, sm, 0, 1, 1, cast};
  const double a = 8.0 * kLog2e * sm * static_cast<double>(sq) * static_cast<double>(sk_head[j]);
  for (int c = 0; c < 128; ++c) {
    const int64_t t = j * 128 + c;
    if (t >= S) {
      codes[c] = 0;
      continue;
    }
    double k[128];
    for (int d = 0; d < 128; ++d) k[d] = e4m3_value(kcodes_head[t * 128 + d]);
    double Z = a * dot128(q, k);
    if (kbias_head) Z += 8.0 * kLog2e * sm * static_cast<double>(sk_head[j]) * kbias_head[t];
    uint8_t code;
    prob(Z, m8, P, &code);
    codes[c] = code;
  }
}

// ExpCast attention (cast = 1: the exp-then-cast baseline; mid_window = 0:
// natural key order) for a list of query rows (b*H+h, s).  Inputs are the
// oracle's own quantised tensors: qc/kc [B,H,S_pad,128], sq/sk [B,H,nb],
// vc token-major [B,H,S_pad,128], sv [B,H].  Optional repair set: rep_idx
// [B,H,n_rep], rep_dcodes [B,H,n_rep,128], sr [B,H].  vmu (V-Smooth, not
// with repair): [B,H,nb,128] block means mu_b in V's own units; token t of
// block b is restored as s_v dec(code_t) + mu_b (the row-sum restore:
// sum_t p_t mu_b(t) = sum_b l_b mu_b), in double.  kbias (Q smoothing, else
// NULL): [B,H,S] beta_t = mu_q . dec(code_t), the per-key bias; each score of
// key t gains 8 log2(e) sm s_k beta_t, so the score is the exact product of
// the query mu_q + s_q dec(Q^') with the key s_k dec(K^_t).
// Outputs per row: out
// [nrows,128] (double), m8, l, nres [nrows,2] (main, repair).  If dump_codes
// is given, the codes of key block dump_block are written per row
// ([nrows,128]) with the reference used for them in dump_m8 ([nrows]).
int ovc_oracle_attention_rows(const uint8_t* qc, const float* sq, const uint8_t* kc, const float* sk,
                              const uint8_t* vc, const float* sv, int64_t B, int64_t S, int64_t H,
                              const int32_t* rep_idx, const uint8_t* rep_dcodes, const float* sr,
                              int64_t n_rep, const float* vmu, const double* kbias, const int64_t* row_bh,
                              const int64_t* row_s,
                              int64_t nrows, double c0, double beta, double tau, double sm,
                              int mid_window, int snap, int cast, int64_t nsplit, double* out, double* m8_out, double* l_out,
                              int32_t* nres_out, int64_t dump_block, uint8_t* dump_codes,
                              double* dump_m8, int nthreads) {
  const Dims dm = make_dims(B, S, H);
  const Params P{c0, beta, tau, sm, 0, mid_window, snap, cast};
  if (nsplit < 1 || nsplit > dm.nb || (nsplit > 1 && n_rep > 0) || (vmu && n_rep > 0)) return 3;
  // Process the rows head by head so that one head's keys are decoded once.
  std::vector<int64_t> perm(nrows);
  for (int64_t i = 0; i < nrows; ++i) perm[i] = i;
  std::stable_sort(perm.begin(), perm.end(), [&](int64_t a, int64_t b) { return row_bh[a] < row_bh[b]; });
  int64_t i0 = 0;
  std::vector<double> K, V, dV, ks;
  while (i0 < nrows) {
    const int64_t bh = row_bh[perm[i0]];
    int64_t i1 = i0;
    while (i1 < nrows && row_bh[perm[i1]] == bh) ++i1;
    if (bh < 0 || bh >= B * H) return 1;
    K.assign(S * 128, 0.0);
    V.assign(S * 128, 0.0);
    for (int64_t t = 0; t < S; ++t)
      for (int d = 0; d < 128; ++d) {
        K[t * 128 + d] = e4m3_value(kc[(bh * dm.S_pad + t) * 128 + d]);
        V[t * 128 + d] = e4m3_value(vc[(bh * dm.S_pad + t) * 128 + d]) +
                         (vmu ? static_cast<double>(vmu[(bh * dm.nb + t / 128) * 128 + d]) /
                                    static_cast<double>(sv[bh])
                              : 0.0);
      }
    ks.assign(sk + bh * dm.nb, sk + (bh + 1) * dm.nb);
    HeadView hv;
    hv.S = S;
    hv.nb = dm.nb;
    hv.K = K.data();
    hv.kscale = ks.data();
    hv.V = V.data();
    hv.vscale = sv[bh];
    hv.kbias = kbias ? kbias + bh * S : nullptr;
    if (n_rep > 0 && rep_idx) {
      dV.assign(n_rep * 128, 0.0);
      for (int64_t i = 0; i < n_rep * 128; ++i) dV[i] = e4m3_value(rep_dcodes[bh * n_rep * 128 + i]);
      hv.n_rep = n_rep;
      hv.rep_idx = rep_idx + bh * n_rep;
      hv.dV = dV.data();
      hv.rscale = sr[bh];
    }
    bool bad = false;
    parallel_for(i1 - i0, nthreads, [&](int64_t ii) {
      const int64_t r = perm[i0 + ii];
      const int64_t s = row_s[r];
      if (s < 0 || s >= S) {
        bad = true;
        return;
      }
      double q[128];
      for (int d = 0; d < 128; ++d) q[d] = e4m3_value(qc[(bh * dm.S_pad + s) * 128 + d]);
      RowResult rr;
      attend_row_split(q, sq[bh * dm.nb + s / 128], hv, P, nsplit, &rr, dump_block,
                       dump_codes ? dump_codes + r * 128 : nullptr, dump_m8 ? dump_m8 + r : nullptr);
      std::memcpy(out + r * 128, rr.O, sizeof(rr.O));
      if (m8_out) m8_out[r] = rr.m8;
      if (l_out) l_out[r] = rr.l;
      if (nres_out) {
        nres_out[2 * r] = rr.nrescale;
        nres_out[2 * r + 1] = rr.nrescale_repair;
      }
    });
    if (bad) return 2;
    i0 = i1;
  }
  return 0;
}

// The same online-softmax skeleton (traversal, lazy rescale, tail mask) on
// raw double inputs with p = 2^((Z - m8)/8) exactly: must equal plain
// softmax attention.  q/k/v: [BH,S,128]; rows as above; kbias (or NULL):
// [BH,S] a per-key term added to every score (Q smoothing's bias).
int ovc_oracle_attention_exact_rows(const double* q, const double* k, const double* v, const double* kbias,
                                    int64_t BH, int64_t S, const int64_t* row_bh, const int64_t* row_s,
                                    int64_t nrows, double tau, double sm, int mid_window, int snap,
                                    int64_t nsplit, double* out, int32_t* nres_out, int nthreads) {
  const Dims dm = make_dims(1, S, 1);
  const Params P{120.0, -0.35, tau, sm, 1, mid_window, snap, 0};
  if (nsplit < 1 || nsplit > dm.nb) return 3;
  std::vector<double> ones(dm.nb, 1.0);
  bool bad = false;
  parallel_for(nrows, nthreads, [&](int64_t r) {
    const int64_t bh = row_bh[r], s = row_s[r];
    if (bh < 0 || bh >= BH || s < 0 || s >= S) {
      bad = true;
      return;
    }
    HeadView hv;
    hv.S = S;
    hv.nb = dm.nb;
    hv.K = k + bh * S * 128;
    hv.kscale = ones.data();
    hv.V = v + bh * S * 128;
    hv.kbias = kbias ? kbias + bh * S : nullptr;
    RowResult rr;
    attend_row_split(q + (bh * S + s) * 128, 1.0, hv, P, nsplit, &rr, -1, nullptr, nullptr);
    std::memcpy(out + r * 128, rr.O, sizeof(rr.O));
    if (nres_out) nres_out[r] = rr.nrescale;
  });
  return bad ? 2 : 0;
}

}  // extern "C"
