// dflash2_oracle.cpp -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.
//
// A plain, slow, obviously-correct CPU restatement of the DFlash 2 draft-block
// head, written from "DFlash 2: Keep Drafting Parallel" (Inco AI).  Only the
// test suite, the smoke check and the benchmark's CPU-baseline leg may load
// this library.  It shares no code, header, table or helper with the CUDA
// library; the two meet only through the seeded input generator, which holds
// none of the method's arithmetic.
//
// Conventions
//   * bf16 tensors arrive as raw uint16 bit patterns; they are widened exactly
//     (bits << 16) to float and then to double.
//   * Everything is accumulated in double unless a function says otherwise.
//   * Loops follow the definitions directly: no blocking, fusion or reordering.
//   * `nthreads` <= 1 runs single-threaded; larger values split the outermost
//     loop over independent rows / sequences with OpenMP (results do not
//     depend on the thread count: every row is computed by one thread).
//
// Readings where the pages are silent (each is listed in the design notes):
//   R1  top-16 order: value descending, ties by lowest vocabulary id; -0 == +0;
//       NaN ranks below -inf.
//   R2  context gate H(h_t) = sigmoid(W_H h_t + b_H), one 256-vector per position.
//   R3  position t = 0 has a single predecessor, the last verified token; the 16
//       rows of its 16x16 score block are identical.
//   R4  greedy walk = myopic best successor at every step, lowest slot on ties;
//       a NaN score never beats a number (R1's order: NaN below -inf), so a
//       row's choice is the lowest slot of its largest non-NaN score (slot 0
//       if every score is NaN).
//   R5  sampled walk = softmax(S/T) over the 16 successors of the chosen
//       predecessor, inverse CDF in slot order with a Philox4x32-10 uniform.
//       The draw is an integer decided by floating point, so it is taken in
//       the kernel's precision (fp32) with 2^x evaluated by a named method
//       (Cody-Waite reduction + degree-7 Taylor polynomial, exp2_neg below):
//       every step is a correctly rounded IEEE fp32 operation, so any
//       implementation of the same steps draws the same slot.  A row with no
//       positive weight (every score NaN or -inf) takes the greedy choice,
//       with q one-hot there.
//   R6  conv correction [c0; c1] = W_c h_t (+ b_c), linear, no activation;
//       rows [0, d/16) give c0, rows [d/16, 2d/16) give c1; channel ch belongs
//       to group ch/16; h defaults to the conv input x; no residual.
//   R7  verification at T > 0 is standard speculative rejection sampling with
//       proposal q = the walk's per-step 16-slot distribution (zero elsewhere).
//   R21 the target distribution of R7 in exact fixed point.  Every accept test
//       and draw is an integer decided by floating point, so both sides take
//       the weights in one precision and sum them exactly:
//         c = fp32(log2 e) / T (fp32), M = the row's largest non-NaN logit,
//         w_v = exp2_neg((l_v - M) * c) (fp32, R5's function),
//         W_v = floor(w_v * 2^40) (an integer; weights below 2^-40 of the
//         row's largest count as 0), Z = sum_v W_v (exact in 64 bits for
//         V < 2^23), p(v) = W_v / Z.
//       Integer sums do not depend on their order, so any parallel split of a
//       row gives the same Z and the same prefix sums.  Accept t iff
//       (u1 * q) * Z < W_x in fp64 (u1 * q is exact; one rounding).  The
//       residual of a rejection is R_v = max(0, W_v - sum_{j: c_j = v} Q_j) with
//       Q_j = floor(q_j * Z) (fp64 product, truncated); the draw target is
//       floor(U * R / 2^24) for the 24-bit Philox integer U and R = sum_v R_v,
//       and the token is the lowest id whose inclusive prefix of R exceeds it.
//       If R = 0 the draw uses W; if Z = 0 (no finite logit) the token is the
//       row's arg-max in R1's order.  The bonus row draws from W the same way.
//   R8  Philox counter = (b, t | stream << 24, offset_lo, offset_hi),
//       key = (seed_lo, seed_hi); a uniform is (x0 >> 8) * 2^-24.
//   R17 exact best-path walk (the pages call pairwise scoring "the simplest
//       selector" and leave more to explore): the slot path j_0..j_{L-1}
//       maximising S[0][0][j_0] + sum_{t>=1} S[t][j_{t-1}][j_t], the sum taken
//       left to right in fp32 (the precision the scores are stored in, so the
//       integer path is decided in one precision); ties keep the lowest
//       predecessor, then the lowest final slot.
//   R19 projection-form selector: A(a) = W_A E(a) and B(b) = W_B E(b), with E
//       the shared [V, d] token embedding and W_A, W_B [256, d] (the form whose
//       parameter count, 3 x 256 x d for W_A, W_B and W_H, matches the 2.0M
//       the pages state at d = 2560).  The projections are exact sums, not
//       rounded to bf16 (the tables of R10 are this form folded offline).
//   R20 conv fused into the producing GEMM: x = A W^T (the sublayer's output
//       projection) is exact, with no rounding to bf16 between the GEMM and the
//       taps, and the correction reads a given hidden state h (a GEMM epilogue
//       sees one tile of x, never the whole row that W_c x would need).
//   R18 selector evaluation (Table 1): recall at position t counts sequences
//       whose earlier positions were all correct under the same rule (top-1
//       equal to the true token, or the true token among the 16); the
//       acceptance length of a rule is 1 + its number of leading correct
//       positions (the verifier's next token included).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

double widen_bf16(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

float widen_bf16_f(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}

int threads_for(int nthreads) { return nthreads < 1 ? 1 : nthreads; }

// ---------------------------------------------------------------------------
// Philox4x32-10, from Salmon, Moraes, Dror and Shaw, "Parallel Random Numbers:
// As Easy as 1, 2, 3" (SC'11): ten rounds of the 4x32 S-box/P-box round with
// multipliers 0xD2511F53 and 0xCD9E8D57 and the Weyl key schedule
// (0x9E3779B9, 0xBB67AE85).  The pages name no generator (reading R8).
// ---------------------------------------------------------------------------
void philox_round(uint32_t c[4], const uint32_t k[2]) {
  const uint64_t p0 = static_cast<uint64_t>(0xD2511F53u) * c[0];
  const uint64_t p1 = static_cast<uint64_t>(0xCD9E8D57u) * c[2];
  const uint32_t hi0 = static_cast<uint32_t>(p0 >> 32), lo0 = static_cast<uint32_t>(p0);
  const uint32_t hi1 = static_cast<uint32_t>(p1 >> 32), lo1 = static_cast<uint32_t>(p1);
  const uint32_t n0 = hi1 ^ c[1] ^ k[0];
  const uint32_t n2 = hi0 ^ c[3] ^ k[1];
  c[0] = n0;
  c[1] = lo1;
  c[2] = n2;
  c[3] = lo0;
}

void philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
  uint32_t k[2] = {key[0], key[1]};
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k[0] += 0x9E3779B9u;
      k[1] += 0xBB67AE85u;
    }
    philox_round(c, k);
  }
  for (int i = 0; i < 4; ++i) out[i] = c[i];
}

// Uniform in [0, 1) with 24 random bits (reading R8).
double uniform24(uint64_t seed, uint64_t b, uint64_t t, uint32_t stream, uint64_t offset) {
  const uint32_t ctr[4] = {static_cast<uint32_t>(b),
                           static_cast<uint32_t>(t) | (stream << 24),
                           static_cast<uint32_t>(offset),
                           static_cast<uint32_t>(offset >> 32)};
  const uint32_t key[2] = {static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32)};
  uint32_t out[4];
  philox4x32_10(ctr, key, out);
  return static_cast<double>(out[0] >> 8) * (1.0 / 16777216.0);
}

// 2^x for x <= 0 in fp32 (reading R5).  Cody and Waite's range reduction
// (Software Manual for the Elementary Functions, 1980): x = n + f with
// n = rint(x) and f in [-1/2, 1/2]; 2^f = e^(f ln 2) by the degree-7 Taylor
// polynomial, coefficients (ln 2)^k / k! rounded to fp32, in Horner form with
// fused multiply-adds; then an exact scaling by 2^n.  0 below -126 (and for NaN).
// Truncation error (f ln 2)^8 / 8! < 4e-10, below half an fp32 ulp.
float exp2_neg(float x) {
  if (!(x >= -126.0f)) return 0.0f;
  const float n = std::nearbyint(x);
  const float f = x - n;
  float p = 1.525273365e-05f;            // (ln 2)^7 / 7!
  p = std::fma(p, f, 1.540352969e-04f);  // (ln 2)^6 / 6!
  p = std::fma(p, f, 1.333355787e-03f);  // (ln 2)^5 / 5!
  p = std::fma(p, f, 9.618128650e-03f);  // (ln 2)^4 / 4!
  p = std::fma(p, f, 5.550410971e-02f);  // (ln 2)^3 / 3!
  p = std::fma(p, f, 2.402265072e-01f);  // (ln 2)^2 / 2!
  p = std::fma(p, f, 6.931471825e-01f);  // ln 2
  p = std::fma(p, f, 1.0f);
  return std::ldexp(p, static_cast<int>(n));
}

// Reading R1: does (va, ia) come strictly before (vb, ib) in top-k order?
bool ranks_before(double va, int64_t ia, double vb, int64_t ib) {
  const bool na = std::isnan(va), nb = std::isnan(vb);
  if (na != nb) return nb;  // the non-NaN one comes first
  if (!na && va != vb) return va > vb;
  return ia < ib;
}

int64_t clamp_id(int64_t id, int64_t V, int* flag) {
  if (id < 0 || id >= V) {
    if (flag) *flag = 1;
    return id < 0 ? 0 : V - 1;
  }
  return id;
}

// The 24-bit Philox integer behind uniform24 (reading R8): u = U * 2^-24.
uint64_t uniform24_bits(uint64_t seed, uint64_t b, uint64_t t, uint32_t stream, uint64_t offset) {
  return static_cast<uint64_t>(uniform24(seed, b, t, stream, offset) * 16777216.0);
}

// Reading R21: floor(w * 2^40) for an fp32 weight w (0 for w <= 0 and NaN).
// w * 2^40 is exact in double (a 24-bit mantissa scaled by a power of two) and
// the conversion truncates toward zero.
uint64_t fixed_weight(float w) {
  if (!(w > 0.0f)) return 0;
  return static_cast<uint64_t>(std::ldexp(static_cast<double>(w), 40));
}

// Reading R21: the fixed-point weights W_v of one target row at inverse
// temperature c, returning Z = sum_v W_v (exact).  M is the largest non-NaN
// logit (NaN if there is none, which makes every weight 0).
uint64_t fixed_row_weights(const uint16_t* row, int64_t V, float c, uint64_t* W) {
  float M = std::numeric_limits<float>::quiet_NaN();
  for (int64_t v = 0; v < V; ++v) {
    const float l = widen_bf16_f(row[v]);
    if (!std::isnan(l) && (std::isnan(M) || l > M)) M = l;
  }
  uint64_t Z = 0;
  for (int64_t v = 0; v < V; ++v) {
    const float x = (widen_bf16_f(row[v]) - M) * c;
    W[v] = fixed_weight(exp2_neg(x));
    Z += W[v];
  }
  return Z;
}

// floor(U * total / 2^24) exactly, for U < 2^24 (the draw target of reading R21).
uint64_t scaled_target(uint64_t U, uint64_t total) {
  const unsigned __int128 p = static_cast<unsigned __int128>(U) * total;
  return static_cast<uint64_t>(p >> 24);
}

}  // namespace

extern "C" {

// Philox4x32-10 block function, exported so tests can check it against the
// published known-answer vectors.
void oracle_philox4x32_10(const uint32_t* ctr, const uint32_t* key, uint32_t* out) {
  philox4x32_10(ctr, key, out);
}

double oracle_uniform24(uint64_t seed, uint64_t b, uint64_t t, uint32_t stream, uint64_t offset) {
  return uniform24(seed, b, t, stream, offset);
}

float oracle_exp2_neg(float x) { return exp2_neg(x); }

// Reading R21's fixed-point weights of one target row (bf16 bits, V ids) at
// temperature T: W[v] = floor(exp2_neg((l_v - M) * c) * 2^40), c = fp32(log2 e) / T;
// returns Z = sum_v W[v].
uint64_t oracle_verify_weights(const uint16_t* row, int64_t V, double temperature, uint64_t* W) {
  const float c = 1.44269504f / static_cast<float>(temperature);
  return fixed_row_weights(row, V, c, W);
}

// ---------------------------------------------------------------------------
// Stage 1: per-position top-k candidates.
// "A Lightweight Path Selector": DFlash 2 keeps the top 16 candidates of the
// drafter's own logits U_t at every block position instead of the top-1.
// Definition: order all V entries of a row by reading R1 and keep the first k
// (std::partial_sort with that comparator).
// logits: [rows, ld] bf16 bits; vals/idx: [rows, k].
// ---------------------------------------------------------------------------
void oracle_topk(const uint16_t* logits, int64_t rows, int64_t V, int64_t ld, int k,
                 float* vals, int32_t* idx, int nthreads) {
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads_for(nthreads))
  for (int64_t r = 0; r < rows; ++r) {
    const uint16_t* row = logits + r * ld;
    std::vector<int64_t> order(static_cast<size_t>(V));
    for (int64_t v = 0; v < V; ++v) order[v] = v;
    std::partial_sort(order.begin(), order.begin() + k, order.end(),
                      [row](int64_t a, int64_t b) {
                        return ranks_before(widen_bf16(row[a]), a, widen_bf16(row[b]), b);
                      });
    for (int j = 0; j < k; ++j) {
      vals[r * k + j] = widen_bf16_f(row[order[j]]);
      idx[r * k + j] = static_cast<int32_t>(order[j]);
    }
  }
}

// ---------------------------------------------------------------------------
// Stage 2a: context gate (reading R2), "A Lightweight Path Selector":
// H(h_t) decides which parts of the embedding match count.
// H[m, q] = 1 / (1 + exp(-(sum_k W_H[q, k] h[m, k] + b_H[q]))), in double.
// h: [M, d] bf16; W_H: [r, d] bf16; b_H: [r] fp32 or null; H: [M, r] double.
// ---------------------------------------------------------------------------
void oracle_gate(const uint16_t* h, const uint16_t* W_H, const float* b_H, int64_t M,
                 int64_t d, int64_t r, double* H, int nthreads) {
#pragma omp parallel for schedule(static) num_threads(threads_for(nthreads))
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t q = 0; q < r; ++q) {
      double acc = b_H ? static_cast<double>(b_H[q]) : 0.0;
      for (int64_t kk = 0; kk < d; ++kk)
        acc += widen_bf16(W_H[q * d + kk]) * widen_bf16(h[m * d + kk]);
      H[m * r + q] = 1.0 / (1.0 + std::exp(-acc));
    }
  }
}

// ---------------------------------------------------------------------------
// Stage 2b: pairwise path-selector scores, "A Lightweight Path Selector",
// score equation S_t(a, b) = U_t(b) + <A(a) (.) H(h_t), B(b)>:
//   S[b, t, i, j] = U_t(c_t[j]) + sum_q A[p_i, q] * H[b, t, q] * B[c_t[j], q]
// with p_i = c_{t-1}[i] for t >= 1 and p = last_verified[b] for t = 0
// (reading R3).  U_t(c_t[j]) is cand_val[b, t, j].
// cand_idx/cand_val: [B, L, K]; H: [B, L, r] double; A, Bt: [V, r] bf16;
// S: [B, L, K, K] double.  Out-of-range ids are clamped and reported.
// Returns 1 if any id was out of range, else 0.
// ---------------------------------------------------------------------------
int oracle_pair_scores(const int32_t* cand_idx, const float* cand_val,
                       const int32_t* last_verified, const double* H, const uint16_t* A,
                       const uint16_t* Bt, int64_t B, int64_t L, int64_t K, int64_t r,
                       int64_t V, double* S, int nthreads) {
  int any_bad = 0;
#pragma omp parallel for schedule(static) num_threads(threads_for(nthreads)) reduction(| : any_bad)
  for (int64_t b = 0; b < B; ++b) {
    for (int64_t t = 0; t < L; ++t) {
      const double* Ht = H + (b * L + t) * r;
      for (int64_t i = 0; i < K; ++i) {
        int bad = 0;
        int64_t pred = (t == 0) ? last_verified[b] : cand_idx[(b * L + t - 1) * K + i];
        pred = clamp_id(pred, V, &bad);
        for (int64_t j = 0; j < K; ++j) {
          int64_t cur = clamp_id(cand_idx[(b * L + t) * K + j], V, &bad);
          double acc = 0.0;
          for (int64_t q = 0; q < r; ++q)
            acc += widen_bf16(A[pred * r + q]) * Ht[q] * widen_bf16(Bt[cur * r + q]);
          S[((b * L + t) * K + i) * K + j] = static_cast<double>(cand_val[(b * L + t) * K + j]) + acc;
        }
        any_bad |= bad;
      }
    }
  }
  return any_bad;
}

// ---------------------------------------------------------------------------
// Stage 2b, projection form (reading R19): the same score with the embeddings
// projected on the fly from the shared token embedding,
//   A(a)_q = sum_k W_A[q, k] E[a, k],   B(b)_q = sum_k W_B[q, k] E[b, k],
//   S[b, t, i, j] = U_t(c_t[j]) + sum_q A(p_i)_q * H[b, t, q] * B(c_t[j])_q,
// predecessors as in the table form.  E: [V, d] bf16; W_A, W_B: [r, d] bf16;
// H: [B, L, r] double; S: [B, L, K, K] double.  Ids are clamped and reported
// as in the table form.  Returns 1 if any id was out of range, else 0.
// ---------------------------------------------------------------------------
static void project_row(const uint16_t* E, const uint16_t* W, int64_t id, int64_t r, int64_t d, double* out) {
  for (int64_t q = 0; q < r; ++q) {
    double acc = 0.0;
    for (int64_t k = 0; k < d; ++k) acc += widen_bf16(W[q * d + k]) * widen_bf16(E[id * d + k]);
    out[q] = acc;
  }
}

int oracle_pair_scores_proj(const int32_t* cand_idx, const float* cand_val, const int32_t* last_verified,
                            const double* H, const uint16_t* E, const uint16_t* W_A, const uint16_t* W_B,
                            int64_t B, int64_t L, int64_t K, int64_t r, int64_t V, int64_t d, double* S,
                            int nthreads) {
  int any_bad = 0;
#pragma omp parallel for collapse(2) schedule(static) num_threads(threads_for(nthreads)) reduction(| : any_bad)
  for (int64_t b = 0; b < B; ++b) {
    for (int64_t t = 0; t < L; ++t) {
      int bad = 0;
      std::vector<double> Ap(static_cast<size_t>(K * r)), Bc(static_cast<size_t>(K * r));
      for (int64_t i = 0; i < K; ++i) {
        int64_t pred = (t == 0) ? last_verified[b] : cand_idx[(b * L + t - 1) * K + i];
        pred = clamp_id(pred, V, &bad);
        project_row(E, W_A, pred, r, d, &Ap[i * r]);
        const int64_t cur = clamp_id(cand_idx[(b * L + t) * K + i], V, &bad);
        project_row(E, W_B, cur, r, d, &Bc[i * r]);
      }
      const double* Ht = H + (b * L + t) * r;
      for (int64_t i = 0; i < K; ++i)
        for (int64_t j = 0; j < K; ++j) {
          double acc = 0.0;
          for (int64_t q = 0; q < r; ++q) acc += Ap[i * r + q] * Ht[q] * Bc[j * r + q];
          S[((b * L + t) * K + i) * K + j] = static_cast<double>(cand_val[(b * L + t) * K + j]) + acc;
        }
      any_bad |= bad;
    }
  }
  return any_bad;
}

// ---------------------------------------------------------------------------
// Stage 3: the walk over precomputed scores, "A Lightweight Path Selector":
// starting from the last verified token, greedy follows the best successor at
// each step; sampling draws from the same scores.
//   row(t) = 0 for t = 0 (all rows are equal there), else slot(t - 1).
//   temperature <= 0: slot(t) = lowest j maximising S[b, t, row, j] over the
//                     non-NaN scores (R4; 0 if all are NaN);
//                     q[b, t, :] = one-hot at slot(t).
//   temperature  > 0 (R5, all in fp32): c = log2(e) / T, m = the greedy slot's
//                     score, w_j = exp2_neg((S_j - m) * c), Z = w_0 + ... + w_15
//                     summed in slot order, u = uniform24(seed, b, t, 0, offset)
//                     (exact in fp32), slot(t) = smallest j with u * Z < w_0 + ... + w_j;
//                     q[b, t, j] = w_j / Z.  If Z = 0 (every score NaN or -inf),
//                     slot(t) = the greedy slot and q is one-hot there.
// S: [B, L, K, K] fp32 (the walk reads scores at the precision they are stored);
// outputs draft_tok, draft_slot: [B, L]; q: [B, L, K] or null;
// margin: [B, L] or null -- the decision margin of every step (greedy: best -
// runner-up; sampled: distance of u*Z to the nearest CDF boundary of the chosen
// slot, relative to Z).
// ---------------------------------------------------------------------------
void oracle_walk(const float* S, const int32_t* cand_idx, int64_t B, int64_t L, int64_t K,
                 double temperature, uint64_t seed, uint64_t offset, int32_t* draft_tok,
                 int32_t* draft_slot, float* q, double* margin, int nthreads) {
#pragma omp parallel for schedule(static) num_threads(threads_for(nthreads))
  for (int64_t b = 0; b < B; ++b) {
    int64_t prev = 0;
    for (int64_t t = 0; t < L; ++t) {
      double step_margin = 0.0;
      const int64_t row = (t == 0) ? 0 : prev;
      const float* s = S + ((b * L + t) * K + row) * K;
      // lowest slot of the largest non-NaN score (R4); slot 0 if all are NaN
      int64_t best = 0;
      for (int64_t j = 1; j < K; ++j)
        if (!std::isnan(s[j]) && (std::isnan(s[best]) || s[j] > s[best])) best = j;
      int64_t chosen;
      if (temperature <= 0.0) {
        chosen = best;
        double runner = -std::numeric_limits<double>::infinity();
        for (int64_t j = 0; j < K; ++j)
          if (j != best) runner = std::max(runner, static_cast<double>(s[j]));
        step_margin = static_cast<double>(s[best]) - runner;
        if (q)
          for (int64_t j = 0; j < K; ++j) q[(b * L + t) * K + j] = (j == chosen) ? 1.0f : 0.0f;
      } else {
        const float m = s[best];
        const float c = 1.44269504f / static_cast<float>(temperature);
        float w[64], cdf[64];
        float Z = 0.0f;
        for (int64_t j = 0; j < K; ++j) {
          w[j] = exp2_neg((s[j] - m) * c);
          Z += w[j];
          cdf[j] = Z;
        }
        if (!(Z > 0.0f)) {
          // no positive weight (every score NaN or -inf): the greedy choice (R5)
          chosen = best;
          step_margin = std::numeric_limits<double>::infinity();
          if (q)
            for (int64_t j = 0; j < K; ++j) q[(b * L + t) * K + j] = (j == chosen) ? 1.0f : 0.0f;
        } else {
          const float u = static_cast<float>(uniform24(seed, static_cast<uint64_t>(b), static_cast<uint64_t>(t), 0, offset));
          const float target = u * Z;
          chosen = -1;
          for (int64_t j = 0; j < K; ++j)
            if (target < cdf[j]) {
              chosen = j;
              break;
            }
          if (chosen < 0)
            for (int64_t j = K - 1; j >= 0; --j)
              if (w[j] > 0.0f) {
                chosen = j;
                break;
              }
          double gap = static_cast<double>(cdf[chosen]) - target;
          if (chosen > 0) gap = std::min(gap, static_cast<double>(target) - cdf[chosen - 1]);
          step_margin = gap / Z;
          if (q)
            for (int64_t j = 0; j < K; ++j) q[(b * L + t) * K + j] = w[j] / Z;
        }
      }
      draft_slot[b * L + t] = static_cast<int32_t>(chosen);
      draft_tok[b * L + t] = cand_idx[(b * L + t) * K + chosen];
      if (margin) margin[b * L + t] = step_margin;
      prev = chosen;
    }
  }
}

// ---------------------------------------------------------------------------
// Stage 4: two-tap dynamic depthwise convolution, "A Lightweight Local
// Convolution": Conv_k(x)_t = k_{t,0} (.) x_t + k_{t,1} (.) x_{t-1}, each
// coefficient = learned base + a correction from the current hidden state,
// shared by every 16 channels; position 0 reads the last verified token's
// representation (reading R6):
//   c[m, n]  = sum_k W_c[n, k] h[m, k] (+ b_c[n]),   n in [0, 2G), G = d / 16
//   y[m, ch] = (k0[ch] + c[m, g]) x[m, ch] + (k1[ch] + c[m, G + g]) xp[ch]
// with g = ch / 16, m = b * L + t, and xp = x[m - 1] for t > 0, x_prev[b] at t = 0.
// x: [B, L, d]; x_prev: [B, d]; h: [B, L, d] or null (then h = x); k0, k1: [d];
// W_c: [2G, d] bf16; b_c: [2G] fp32 or null; y: [B, L, d] double.
// ---------------------------------------------------------------------------
void oracle_conv2tap(const uint16_t* x, const uint16_t* x_prev, const uint16_t* h,
                     const uint16_t* k0, const uint16_t* k1, const uint16_t* W_c,
                     const float* b_c, int64_t B, int64_t L, int64_t d, double* y,
                     int nthreads) {
  const int64_t G = d / 16;
  if (!h) h = x;
#pragma omp parallel for schedule(static) num_threads(threads_for(nthreads))
  for (int64_t m = 0; m < B * L; ++m) {
    const int64_t b = m / L, t = m % L;
    std::vector<double> c(static_cast<size_t>(2 * G));
    for (int64_t n = 0; n < 2 * G; ++n) {
      double acc = b_c ? static_cast<double>(b_c[n]) : 0.0;
      for (int64_t kk = 0; kk < d; ++kk) acc += widen_bf16(W_c[n * d + kk]) * widen_bf16(h[m * d + kk]);
      c[n] = acc;
    }
    const uint16_t* xp = (t > 0) ? x + (m - 1) * d : x_prev + b * d;
    for (int64_t ch = 0; ch < d; ++ch) {
      const int64_t g = ch / 16;
      y[m * d + ch] = (widen_bf16(k0[ch]) + c[g]) * widen_bf16(x[m * d + ch]) +
                      (widen_bf16(k1[ch]) + c[G + g]) * widen_bf16(xp[ch]);
    }
  }
}

// ---------------------------------------------------------------------------
// Stage 4, fused into the producing GEMM (reading R20): the conv's input is the
// output of the sublayer's projection, x = A W^T, taken exactly:
//   x[m, ch] = sum_k A[m, k] W[ch, k]
//   c[m, n]  = sum_k W_c[n, k] h[m, k] (+ b_c[n])
//   y[m, ch] = (k0[ch] + c[m, g]) x[m, ch] + (k1[ch] + c[m, G + g]) xp[ch]
// with xp = x[m - 1] for t > 0 and x_prev[b] (bf16) at t = 0.
// A: [B, L, K] bf16; W: [d, K] bf16; h: [B, L, d] bf16; the rest as
// oracle_conv2tap; y: [B, L, d] double.
// ---------------------------------------------------------------------------
void oracle_gemm_conv2tap(const uint16_t* A, const uint16_t* W, const uint16_t* x_prev, const uint16_t* h,
                          const uint16_t* k0, const uint16_t* k1, const uint16_t* W_c, const float* b_c, int64_t B,
                          int64_t L, int64_t K, int64_t d, double* y, int nthreads) {
  const int64_t G = d / 16;
#pragma omp parallel for schedule(static) num_threads(threads_for(nthreads))
  for (int64_t b = 0; b < B; ++b) {
    std::vector<double> x(static_cast<size_t>(L * d)), c(static_cast<size_t>(2 * G));
    for (int64_t t = 0; t < L; ++t)
      for (int64_t ch = 0; ch < d; ++ch) {
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) acc += widen_bf16(A[((b * L + t) * K) + k]) * widen_bf16(W[ch * K + k]);
        x[t * d + ch] = acc;
      }
    for (int64_t t = 0; t < L; ++t) {
      const int64_t m = b * L + t;
      for (int64_t n = 0; n < 2 * G; ++n) {
        double acc = b_c ? static_cast<double>(b_c[n]) : 0.0;
        for (int64_t k = 0; k < d; ++k) acc += widen_bf16(W_c[n * d + k]) * widen_bf16(h[m * d + k]);
        c[n] = acc;
      }
      for (int64_t ch = 0; ch < d; ++ch) {
        const int64_t g = ch / 16;
        const double xp = (t > 0) ? x[(t - 1) * d + ch] : widen_bf16(x_prev[b * d + ch]);
        y[m * d + ch] = (widen_bf16(k0[ch]) + c[g]) * x[t * d + ch] + (widen_bf16(k1[ch]) + c[G + g]) * xp;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Stage 5: block verification against the target's logits.  "A Lightweight
// Path Selector" (rejection sampling restores the exact target distribution),
// Table 1's note (the acceptance length includes the verifier's next token),
// and the post's opening (the target verifies the whole block in one pass).
//
// temperature <= 0 (greedy): a_t = lowest id maximising target[b, t, :]
//   (values compared exactly); n = first t < L with draft_tok[b, t] != a_t,
//   else L; out = draft[0..n-1], a_n; accept_len = n + 1.
// temperature > 0 (readings R7 and R21): for t = 0..L-1 with p_t(v) = W_v / Z
//   (the fixed-point weights of row t), x = draft_tok[t] (W_x = 0 outside
//   [0, V)), q = draft_q[t, draft_slot[t]] (slot clamped to [0, 16)),
//   u1 = uniform24(seed, b, t, 1, offset): accept iff (u1 * q) * Z < W_x.
//   On the first rejection at t: draw from the residual R_v = max(0, W_v -
//   sum_{j: cand_idx[t, j] = v} Q_j), Q_j = floor(min(q_j, 1) * Z) (q_j = draft_q[t, j],
//   NaN or negative read as 0), by inverse CDF in id order with the target
//   floor(U2 * R / 2^24), U2 the 24-bit integer of (b, t, stream 2);
//   accept_len = t + 1.  If all L are accepted: draw the bonus token from W of
//   row L the same way with the integer of (b, L, stream 2); accept_len = L + 1.
// target: [B, L + 1, ld] bf16 (row (b, t) starts at (b * (L + 1) + t) * ld);
// out_tok: [B, L + 1], -1 after the last emitted token.
// margin: [B, 2] or null -- T > 0 only (+inf at T = 0, whose decisions are
// exact): [0] the smallest |u1 q Z - W_x| / W_x over the accept tests on the
// path, [1] the smallest distance of a draw's target to the bounds of the
// drawn token's interval, relative to the total.  They say how close a
// decision came to flipping, for comparisons with a floating-point restatement.
// ---------------------------------------------------------------------------
void oracle_verify(const uint16_t* target, int64_t ld, const int32_t* draft_tok,
                   const int32_t* draft_slot, const float* draft_q, const int32_t* cand_idx,
                   int64_t B, int64_t L, int64_t K, int64_t V, double temperature,
                   uint64_t seed, uint64_t offset, int32_t* accept_len, int32_t* out_tok,
                   double* margin, int nthreads) {
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads_for(nthreads))
  for (int64_t b = 0; b < B; ++b) {
    int32_t* out = out_tok + b * (L + 1);
    for (int64_t t = 0; t <= L; ++t) out[t] = -1;
    double accept_margin = std::numeric_limits<double>::infinity();
    double draw_margin = std::numeric_limits<double>::infinity();
    int64_t n = L;
    int32_t last = -1;
    if (temperature <= 0.0) {
      for (int64_t t = 0; t <= L; ++t) {
        const uint16_t* row = target + (b * (L + 1) + t) * ld;
        int64_t a = 0;
        for (int64_t v = 1; v < V; ++v)
          if (ranks_before(widen_bf16(row[v]), v, widen_bf16(row[a]), a)) a = v;
        if (t == L || draft_tok[b * L + t] != a) {
          n = t;
          last = static_cast<int32_t>(a);
          break;
        }
      }
    } else {
      const float c = 1.44269504f / static_cast<float>(temperature);
      std::vector<uint64_t> W(static_cast<size_t>(V)), R(static_cast<size_t>(V)), Qs(static_cast<size_t>(V));
      std::vector<char> is_cand(static_cast<size_t>(V));
      auto row_of = [&](int64_t t) { return target + (b * (L + 1) + t) * ld; };
      // the row's arg-max in R1's order (the token when no weight is positive)
      auto argmax_row = [&](int64_t t) -> int32_t {
        const uint16_t* row = row_of(t);
        int64_t a = 0;
        for (int64_t v = 1; v < V; ++v)
          if (ranks_before(widen_bf16(row[v]), v, widen_bf16(row[a]), a)) a = v;
        return static_cast<int32_t>(a);
      };
      // inverse CDF over integer weights w in id order (total > 0); records the margin
      auto draw = [&](const std::vector<uint64_t>& w, uint64_t total, uint64_t U) -> int32_t {
        const uint64_t tgt = scaled_target(U, total);
        uint64_t run = 0;
        for (int64_t v = 0; v < V; ++v) {
          const uint64_t prev = run;
          run += w[v];
          if (tgt < run) {
            const double gap = static_cast<double>(std::min(run - tgt, tgt - prev + 1));
            draw_margin = std::min(draw_margin, gap / static_cast<double>(total));
            return static_cast<int32_t>(v);
          }
        }
        return static_cast<int32_t>(V - 1);   // not reached: tgt < total
      };
      n = L;
      for (int64_t t = 0; t < L; ++t) {
        const uint64_t Z = fixed_row_weights(row_of(t), V, c, W.data());
        const int32_t x = draft_tok[b * L + t];
        int64_t slot = draft_slot[b * L + t];
        slot = slot < 0 ? 0 : (slot >= K ? K - 1 : slot);
        const double qx = static_cast<double>(draft_q[(b * L + t) * K + slot]);
        const uint64_t Wx = (x >= 0 && x < V) ? W[x] : 0;
        const double u1 = uniform24(seed, static_cast<uint64_t>(b), static_cast<uint64_t>(t), 1, offset);
        const double lhs = (u1 * qx) * static_cast<double>(Z);
        const double rhs = static_cast<double>(Wx);
        accept_margin = std::min(accept_margin, std::fabs(lhs - rhs) / std::max(rhs, 1e-300));
        if (lhs < rhs) continue;
        n = t;
        const uint64_t U2 = uniform24_bits(seed, static_cast<uint64_t>(b), static_cast<uint64_t>(t), 2, offset);
        if (Z == 0) {
          last = argmax_row(t);
          break;
        }
        // residual: each candidate slot takes Q_j off its (clamped) id
        std::fill(Qs.begin(), Qs.end(), 0);
        std::fill(is_cand.begin(), is_cand.end(), 0);
        for (int64_t j = 0; j < K; ++j) {
          const int64_t v = clamp_id(cand_idx[(b * L + t) * K + j], V, nullptr);
          const float qj = draft_q[(b * L + t) * K + j];
          const double qc = qj > 0.0f ? std::min(static_cast<double>(qj), 1.0) : 0.0;
          Qs[v] += static_cast<uint64_t>(qc * static_cast<double>(Z));
          is_cand[v] = 1;
        }
        uint64_t Rtot = 0;
        for (int64_t v = 0; v < V; ++v) {
          R[v] = is_cand[v] ? (W[v] > Qs[v] ? W[v] - Qs[v] : 0) : W[v];
          Rtot += R[v];
        }
        last = Rtot > 0 ? draw(R, Rtot, U2) : draw(W, Z, U2);
        break;
      }
      if (n == L) {
        const uint64_t Z = fixed_row_weights(row_of(L), V, c, W.data());
        const uint64_t U2 = uniform24_bits(seed, static_cast<uint64_t>(b), static_cast<uint64_t>(L), 2, offset);
        last = Z > 0 ? draw(W, Z, U2) : argmax_row(L);
      }
    }
    for (int64_t t = 0; t < n; ++t) out[t] = draft_tok[b * L + t];
    out[n] = last;
    accept_len[b] = static_cast<int32_t>(n + 1);
    if (margin) {
      margin[2 * b] = accept_margin;
      margin[2 * b + 1] = draw_margin;
    }
  }
}

// ---------------------------------------------------------------------------
// Fused LM head + top-k, restated unfused: logits[m, v] = sum_k hidden[m, k] W[v, k]
// in double for the requested rows only, then the top-k of each row by
// reading R1 (the head produces U_t, "DFlash's own logit", "A Lightweight Path
// Selector").  hidden: [M, d] bf16; W: [V, d] bf16; rows: [n_rows] row ids;
// vals (double) / idx: [n_rows, k].
// ---------------------------------------------------------------------------
void oracle_lmhead_topk(const uint16_t* hidden, const uint16_t* W, int64_t V, int64_t d,
                        const int64_t* rows, int64_t n_rows, int k, double* vals,
                        int32_t* idx, int nthreads) {
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads_for(nthreads))
  for (int64_t i = 0; i < n_rows; ++i) {
    const uint16_t* hrow = hidden + rows[i] * d;
    std::vector<double> logit(static_cast<size_t>(V));
    for (int64_t v = 0; v < V; ++v) {
      double acc = 0.0;
      for (int64_t kk = 0; kk < d; ++kk) acc += widen_bf16(hrow[kk]) * widen_bf16(W[v * d + kk]);
      logit[v] = acc;
    }
    std::vector<int64_t> order(static_cast<size_t>(V));
    for (int64_t v = 0; v < V; ++v) order[v] = v;
    std::partial_sort(order.begin(), order.begin() + k, order.end(),
                      [&logit](int64_t a, int64_t b) { return ranks_before(logit[a], a, logit[b], b); });
    for (int j = 0; j < k; ++j) {
      vals[i * k + j] = logit[order[j]];
      idx[i * k + j] = static_cast<int32_t>(order[j]);
    }
  }
}

// ---------------------------------------------------------------------------
// Exact best-path walk over the pair scores (reading R17).  The
// max-sum (Viterbi) recurrence over the 16 slots of each position:
//   V_0[j] = S[b][0][0][j]
//   V_t[j] = max_i (V_{t-1}[i] + S[b][t][i][j]),  P_t[j] = the first i attaining it
// then j_{L-1} = the first slot attaining max_j V_{L-1}[j] and j_{t-1} = P_t[j_t].
// Every V is an fp32 sum formed left to right, as written.
// S: [B, L, K, K] fp32; outputs draft_tok, draft_slot: [B, L]; score: [B] (the
// best path's V) or null.
// ---------------------------------------------------------------------------
void oracle_walk_viterbi(const float* S, const int32_t* cand_idx, int64_t B, int64_t L, int64_t K,
                         int32_t* draft_tok, int32_t* draft_slot, float* score, int nthreads) {
#pragma omp parallel for schedule(static) num_threads(threads_for(nthreads))
  for (int64_t b = 0; b < B; ++b) {
    std::vector<float> Vp(static_cast<size_t>(K)), Vn(static_cast<size_t>(K));
    std::vector<int32_t> back(static_cast<size_t>(L * K), 0);
    for (int64_t j = 0; j < K; ++j) Vp[j] = S[((b * L + 0) * K + 0) * K + j];
    for (int64_t t = 1; t < L; ++t) {
      for (int64_t j = 0; j < K; ++j) {
        int64_t arg = 0;
        float best = Vp[0] + S[((b * L + t) * K + 0) * K + j];
        for (int64_t i = 1; i < K; ++i) {
          const float v = Vp[i] + S[((b * L + t) * K + i) * K + j];
          if (v > best) {
            best = v;
            arg = i;
          }
        }
        Vn[j] = best;
        back[t * K + j] = static_cast<int32_t>(arg);
      }
      Vp.swap(Vn);
    }
    int64_t j = 0;
    for (int64_t k = 1; k < K; ++k)
      if (Vp[k] > Vp[j]) j = k;
    if (score) score[b] = Vp[j];
    for (int64_t t = L - 1; t >= 0; --t) {
      draft_slot[b * L + t] = static_cast<int32_t>(j);
      draft_tok[b * L + t] = cand_idx[(b * L + t) * K + j];
      if (t > 0) j = back[t * K + j];
    }
  }
}

// ---------------------------------------------------------------------------
// Selector evaluation, Table 1 ("The Right Tokens Are Already There"; reading
// R18).  For sequence b with true tokens gt[b][0..L) and candidates
// cand_idx[b][t][0..16) (value-descending, so slot 0 is the top-1):
//   hit1[t]  = cand_idx[b][t][0] == gt[b][t]
//   hit16[t] = gt[b][t] is one of cand_idx[b][t][0..16)
// accept1[b]  = 1 + the number of leading t with hit1,
// accept16[b] = 1 + the number of leading t with hit16 (an oracle selector
// that always picks the right candidate when it is there).
// counts [L, 4] (int64, accumulated over b): at position t, the number of
// sequences whose positions before t all hit under the top-1 rule, how many of
// those hit at t, and the same two for the top-16 rule; Recall@1[t] and
// Recall@16[t] are the ratios.
// ---------------------------------------------------------------------------
void oracle_selector_eval(const int32_t* gt, const int32_t* cand_idx, int64_t B, int64_t L, int64_t K,
                          int32_t* accept1, int32_t* accept16, int64_t* counts) {
  for (int64_t i = 0; i < L * 4; ++i) counts[i] = 0;
  for (int64_t b = 0; b < B; ++b) {
    bool alive1 = true, alive16 = true;
    int32_t n1 = 0, n16 = 0;
    for (int64_t t = 0; t < L; ++t) {
      const int32_t* c = cand_idx + (b * L + t) * K;
      const int32_t g = gt[b * L + t];
      const bool h1 = c[0] == g;
      bool h16 = false;
      for (int64_t j = 0; j < K; ++j)
        if (c[j] == g) h16 = true;
      if (alive1) {
        counts[t * 4 + 0] += 1;
        if (h1) {
          counts[t * 4 + 1] += 1;
          ++n1;
        } else {
          alive1 = false;
        }
      }
      if (alive16) {
        counts[t * 4 + 2] += 1;
        if (h16) {
          counts[t * 4 + 3] += 1;
          ++n16;
        } else {
          alive16 = false;
        }
      }
    }
    accept1[b] = 1 + n1;
    accept16[b] = 1 + n16;
  }
}

// The thread count an OpenMP region would use for `nthreads` (reported as the
// CPU baseline's core count).
int oracle_threads(int nthreads) {
#ifdef _OPENMP
  int used = 1;
#pragma omp parallel num_threads(threads_for(nthreads))
  {
#pragma omp single
    used = omp_get_num_threads();
  }
  return used;
#else
  (void)nthreads;
  return 1;
#endif
}

}  // extern "C"
