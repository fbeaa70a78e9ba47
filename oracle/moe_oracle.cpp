// moe_oracle.cpp -- plain, slow CPU oracle for the MoE layer hot path.
//
// TEST INFRASTRUCTURE ONLY.  Nothing on the product path may load, link or call
// this file.  Only tests/, __graft_entry__.smoke() and the CPU-baseline leg of
// bench.py use it, to check the CUDA library and to time a CPU baseline.  It
// shares no code, header, table or constant generator with the CUDA sources.
//
// What it computes (the pages' MoE layer, one process, no device):
//   1. router logits      logits[t,e] = sum_i x[t,i] W[e,i] + b[e]          (fp64 accumulate, one fp32 rounding)
//   2. routing            score, optional group limit, top-k, combine weights
//   3. counting           per-expert and per-rank assignment counts
//   4. capacity           C = ceil(cf * N * k / E); overflow dropped in token order
//   5. dispatch order     rank ascending, expert ascending, token order; slot_of / perm_src
//   6. expert FFN         SwiGLU, fp64, no intermediate rounding
//   7. combine            out[t] = x[t] + shared(x[t]) + sum_j w[t,j] y_j, fp64
//   8. bias update        sign rule, fp32
//   9. INT8 payload       per-row symmetric quantisation of the rows an all-to-all
//                         sends, and the receiver's dequantisation and combine
//  10. backward           gradients of the layer output with respect to the hidden
//                         states, the expert and shared-expert weights and the router
//                         weight and bias (the selection itself is piecewise constant)
//
// Sources ("the pages"):
//   [UG] Ultralytics glossary "Expert Parallelism" (Chinese, German and Japanese
//        editions carry the same text); sections "How tokens move between GPUs"
//        (de: "Wie Tokens zwischen GPUs uebertragen werden") and "Load balancing
//        and capacity" (de: "Lastausgleich und Kapazitaet").
//   [BZ] bowenzhou.top knowledge planet, "专家并行" (expert parallelism); sections
//        "机制：all-to-all 两轮" and the worked answer to exercise 2 (capacity factor).
//   [FD] fudan-mlsys-cn chapter 10, section 10.5 (expert parallelism, shared experts).
//   [BZ-D] the same bowenzhou.top note, section "深入推导：all-to-all 通信模型与
//        DeepSeek-V3 的 EP 配置", paragraph on DeepSeek-V3's two-level EP (INT8
//        quantised communication halves the traffic again).
//
// Readings where the pages are silent (each one is a choice, listed in the design notes):
//   * ties in every ordering break toward the lower expert (or group) index;
//   * softmax top-k selects on the logits themselves (softmax is monotone);
//   * the sigmoid used for selection is the fp32 function S() below, fully specified
//     from correctly rounded operations, so that two independent implementations
//     reach identical selections;
//   * group score = sum of the two largest selection scores in the group (the one
//     largest if the group has a single expert);
//   * capacity counts assignments, C = ceil(cf*N*k/E), drop priority is token order
//     (then choice order j within a token), a dropped term is omitted with no
//     re-normalisation of the remaining weights;
//   * the layer output includes the residual, so a token whose every choice was
//     dropped leaves the layer unchanged;
//   * bias update compares the routed count with the mean load N*k/E.
//
// Build: g++ -O2 -fopenmp -ffp-contract=off -std=c++17 -shared -fPIC (see build.py).
// -ffp-contract=off matters: the fp32 steps of S() must round exactly as written.

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

// ---------------------------------------------------------------- element access

// bf16 is the upper half of an IEEE binary32; widening is exact.
inline double bf16_bits_to_double(uint16_t v) {
  uint32_t u = static_cast<uint32_t>(v) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return static_cast<double>(f);
}

// act_dtype: 0 = fp32, 1 = bf16 (stored as raw 16-bit patterns).
inline double load_act(const void* base, int act_dtype, int64_t i) {
  if (act_dtype == 0) return static_cast<double>(static_cast<const float*>(base)[i]);
  return bf16_bits_to_double(static_cast<const uint16_t*>(base)[i]);
}

// fp32 -> bf16, round to nearest, ties to even, from the definition: of the two bf16
// values that bracket f (f with its low 16 bits cleared, and the next bf16 away from
// zero), take the nearer; on a tie take the one whose last kept bit is 0.  Finite
// inputs only; a value that rounds past the largest bf16 becomes infinity.
inline uint16_t float_to_bf16_rne(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  const uint32_t lo_bits = u & 0xffff0000u;
  const uint32_t hi_bits = lo_bits + 0x10000u;  // next magnitude up, same sign
  float lo, hi;
  std::memcpy(&lo, &lo_bits, 4);
  std::memcpy(&hi, &hi_bits, 4);
  // past the largest finite bf16 the next value up is infinity, which the rounding
  // rule places at 2^128 (an unbounded exponent's next power of two)
  const double hi_d = ((hi_bits & 0x7f800000u) == 0x7f800000u)
                          ? std::copysign(std::ldexp(1.0, 128), static_cast<double>(f))
                          : static_cast<double>(hi);
  const double dl = std::fabs(static_cast<double>(f) - lo);
  const double dh = std::fabs(hi_d - f);
  uint32_t pick;
  if (dl < dh) {
    pick = lo_bits;
  } else if (dh < dl) {
    pick = hi_bits;
  } else {
    pick = ((lo_bits >> 16) & 1u) ? hi_bits : lo_bits;
  }
  return static_cast<uint16_t>(pick >> 16);
}

// ---------------------------------------------------------------- fp32 sigmoid spec
//
// S(l) = 1 / (1 + exp(-l)) evaluated in fp32 with a fixed sequence of correctly
// rounded operations, so that any implementation that follows the same steps gets
// the same bits:
//   z  = clamp(-l, -20, 86)      (below -20 the fp32 result is exactly 1; above 86
//                                 the result would leave the normal range)
//   n  = rint(z * log2e)         fp32 multiply, round-half-even to integer
//   r  = z - n*ln2_hi - n*ln2_lo two fused multiply-adds (Cody & Waite 1980 reduction:
//                                 ln2_hi keeps 16 significant bits, ln2_lo the rest)
//   p  = sum_{j=0..7} r^j / j!   degree-7 Taylor polynomial in Horner form, one fma
//                                 per degree (|r| <= ln2/2, truncation < 4e-9 relative)
//   e  = p * 2^n                 exact (power-of-two scale, n in [-29, 125])
//   S  = 1 / (1 + e)             fp32 add, fp32 divide
const float kLog2e = 0x1.715476p+0f;       // fp32 nearest to 1/ln 2
const float kLn2Hi = 0x1.62e4p-1f;         // 45426 / 65536
const float kLn2Lo = 0x1.7f7d1cp-20f;      // fp32 nearest to ln 2 - kLn2Hi
const float kInvFact[8] = {1.0f, 1.0f, 0x1p-1f, 0x1.555556p-3f, 0x1.555556p-5f,
                           0x1.111112p-7f, 0x1.6c16c2p-10f, 0x1.a01a02p-13f};

float sigmoid_spec(float l) {
  float z = -l;
  z = std::fmax(z, -20.0f);
  z = std::fmin(z, 86.0f);
  float t = z * kLog2e;
  float n = std::rint(t);
  float r = std::fma(-n, kLn2Hi, z);
  r = std::fma(-n, kLn2Lo, r);
  float p = kInvFact[7];
  for (int j = 6; j >= 0; --j) p = std::fma(p, r, kInvFact[j]);
  int ni = static_cast<int>(n);
  uint32_t sbits = static_cast<uint32_t>(ni + 127) << 23;
  float scale;
  std::memcpy(&scale, &sbits, 4);
  float e = p * scale;
  float den = 1.0f + e;
  return 1.0f / den;
}

// ---------------------------------------------------------------- ordering

struct Cand {
  float key;
  int idx;
};
// "a ranks before b": larger key first, lower index on equal keys.
inline bool ranks_before(const Cand& a, const Cand& b) {
  if (a.key != b.key) return a.key > b.key;
  return a.idx < b.idx;
}

// Expert -> logical EP rank.  [UG] "How tokens move between GPUs": with E experts
// on R devices, experts 0..E/R-1 live on device 0, the next E/R on device 1, and so
// on (contiguous, rank = e / (E/R)).  Round-robin (rank = e mod R) is the decode
// placement of the DeepSeek-V3-shaped workload.
inline int rank_of(int e, int E, int R, int rank_map) {
  if (rank_map == 1) return e % R;
  return e / (E / R);
}

// SwiGLU expert FFN on one row, fp64 throughout.
//   h_f = silu(x . Wgu[f]) * (x . Wgu[F + f]),  silu(z) = z / (1 + exp(-z))
//   y_o = h . Wd[o]
// Weight layout: Wgu [2F, d] (rows 0..F-1 gate, F..2F-1 up), Wd [d, F].
// [UG] step 3: each device runs its local experts on the tokens it received; an
// expert is a feed-forward block ([UG] intro); SwiGLU is the workloads' choice.
void ffn_row(const double* x, int d, int F, int act_dtype, const void* wgu, int64_t wgu_off,
             const void* wd, int64_t wd_off, double* y, std::vector<double>& h) {
  h.assign(F, 0.0);
  for (int f = 0; f < F; ++f) {
    double g = 0.0, u = 0.0;
    const int64_t rg = wgu_off + static_cast<int64_t>(f) * d;
    const int64_t ru = wgu_off + static_cast<int64_t>(F + f) * d;
    for (int i = 0; i < d; ++i) {
      g += x[i] * load_act(wgu, act_dtype, rg + i);
      u += x[i] * load_act(wgu, act_dtype, ru + i);
    }
    h[f] = g / (1.0 + std::exp(-g)) * u;
  }
  for (int o = 0; o < d; ++o) {
    double acc = 0.0;
    const int64_t ro = wd_off + static_cast<int64_t>(o) * F;
    for (int f = 0; f < F; ++f) acc += h[f] * load_act(wd, act_dtype, ro + f);
    y[o] = acc;
  }
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------- 0. helpers

float oracle_sigmoid_spec(float l) { return sigmoid_spec(l); }

void oracle_sigmoid_spec_many(int64_t n, const float* l, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = sigmoid_spec(l[i]);
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

int oracle_rank_of(int e, int E, int R, int rank_map) { return rank_of(e, E, R, rank_map); }

// Capacity: [UG] "Load balancing and capacity": each expert takes at most a fixed
// number per batch, e.g. 1.25 times its even share; [BZ] exercise 2: each expert's
// buffer is reserved at the mean times 1.25.  The even share of N*k assignments over
// E experts is N*k/E, so C = ceil(cf * N * k / E).  cf <= 0 means no cap (INT_MAX).
int oracle_capacity(int N, int k, int E, float cf) {
  if (!(cf > 0.0f)) return INT_MAX;
  double c = std::ceil(static_cast<double>(cf) * static_cast<double>(N) * static_cast<double>(k) /
                       static_cast<double>(E));
  if (c > static_cast<double>(INT_MAX)) return INT_MAX;
  return static_cast<int>(c);
}

// ---------------------------------------------------------------- 1. router logits
//
// [UG] step 1: the router scores every token against every expert; in the page's
// example the router is a linear layer (hidden -> num_experts, with bias).
// logits[t,e] = sum_i x[t,i] * W[e,i] + b[e], accumulated in fp64 and rounded once.
// x: [N, d] in act_dtype; W: [E, d] fp32; b: [E] fp32 or null.
int oracle_router_logits(int N, int d, int E, int act_dtype, const void* x, const float* W,
                         const float* b, float* logits) {
#pragma omp parallel
  {
    std::vector<double> xr(d);
#pragma omp for schedule(static)
    for (int t = 0; t < N; ++t) {
      for (int i = 0; i < d; ++i) xr[i] = load_act(x, act_dtype, static_cast<int64_t>(t) * d + i);
      for (int e = 0; e < E; ++e) {
        double acc = 0.0;
        const float* w = W + static_cast<int64_t>(e) * d;
        for (int i = 0; i < d; ++i) acc += xr[i] * static_cast<double>(w[i]);
        if (b) acc += static_cast<double>(b[e]);
        logits[static_cast<int64_t>(t) * E + e] = static_cast<float>(acc);
      }
    }
  }
  return 0;
}

// ---------------------------------------------------------------- 2. routing
//
// [UG] step 1: keep the k highest-scoring experts per token (k is typically 1, 2
// or 8).  [UG] step 4: outputs are weighted by the router scores.
// [UG] "Load balancing and capacity", bias-based balancing: a per-expert bias is
// added to the router scores and affects only which experts are selected.
// [UG] same section: each token is sent to experts on at most 4 of the 8 nodes
// (group-limited routing; one group per node).
//
// score_fn 0 (softmax): selection key = logit; weight_j = softmax(logits)_j over all E
//   experts, fp64; with normalize, weight_j / sum over the k selected.
// score_fn 1 (sigmoid): s_e = S(l_e) (fp32 spec above); key_e = s_e + bias_e (one fp32
//   add; bias may be null = 0); weight_j = s_j (no bias), with normalize divided by the
//   sum of s over the k selected, fp64.
// Group limit (num_groups > 1): groups are num_groups runs of E/num_groups contiguous
//   experts; group score = fp32 sum of the two largest keys in the group; the
//   topk_groups best groups (ties: lower group index) stay eligible.
// Outputs: idx [N, k] int32 in selection order (best first); w64 [N, k] fp64.
int oracle_route(int N, int E, int k, int score_fn, int normalize, int num_groups,
                 int topk_groups, const float* logits, const float* sel_bias, int32_t* idx,
                 double* w64) {
  if (k < 1 || k > E) return -1;
  if (num_groups < 1 || E % num_groups != 0) return -1;
  if (topk_groups < 1 || topk_groups > num_groups) return -1;
  const int gs = E / num_groups;
  if (topk_groups * gs < k) return -1;
#pragma omp parallel
  {
    std::vector<float> sig(E), key(E);
    std::vector<Cand> cands, groups;
    std::vector<char> allowed(E);
#pragma omp for schedule(static)
    for (int t = 0; t < N; ++t) {
      const float* l = logits + static_cast<int64_t>(t) * E;
      for (int e = 0; e < E; ++e) {
        if (score_fn == 1) {
          sig[e] = sigmoid_spec(l[e]);
          key[e] = sel_bias ? sig[e] + sel_bias[e] : sig[e];
        } else {
          key[e] = l[e];
        }
        allowed[e] = 1;
      }
      if (num_groups > 1) {
        groups.clear();
        for (int g = 0; g < num_groups; ++g) {
          std::vector<float> gk(key.begin() + g * gs, key.begin() + (g + 1) * gs);
          std::sort(gk.begin(), gk.end(), [](float a, float b) { return a > b; });
          float score = gs >= 2 ? gk[0] + gk[1] : gk[0];
          groups.push_back({score, g});
        }
        std::sort(groups.begin(), groups.end(), ranks_before);
        std::vector<char> gkeep(num_groups, 0);
        for (int i = 0; i < topk_groups; ++i) gkeep[groups[i].idx] = 1;
        for (int e = 0; e < E; ++e) allowed[e] = gkeep[e / gs];
      }
      cands.clear();
      for (int e = 0; e < E; ++e)
        if (allowed[e]) cands.push_back({key[e], e});
      std::sort(cands.begin(), cands.end(), ranks_before);
      int32_t* out_i = idx + static_cast<int64_t>(t) * k;
      double* out_w = w64 + static_cast<int64_t>(t) * k;
      for (int j = 0; j < k; ++j) out_i[j] = cands[j].idx;
      if (score_fn == 1) {
        double s = 0.0;
        for (int j = 0; j < k; ++j) s += static_cast<double>(sig[out_i[j]]);
        for (int j = 0; j < k; ++j) {
          double v = static_cast<double>(sig[out_i[j]]);
          out_w[j] = normalize ? v / s : v;
        }
      } else {
        double m = -INFINITY;
        for (int e = 0; e < E; ++e) m = std::max(m, static_cast<double>(l[e]));
        double z = 0.0;
        for (int e = 0; e < E; ++e) z += std::exp(static_cast<double>(l[e]) - m);
        double zs = 0.0;
        for (int j = 0; j < k; ++j) zs += std::exp(static_cast<double>(l[out_i[j]]) - m);
        for (int j = 0; j < k; ++j) {
          double p = std::exp(static_cast<double>(l[out_i[j]]) - m);
          out_w[j] = normalize ? p / zs : p / z;
        }
      }
    }
  }
  return 0;
}

// ---------------------------------------------------------------- 3-5. count, cap, dispatch order
//
// [UG] "How tokens move between GPUs", step 2 and the example: count the
// token-expert assignments per expert and per device (bincount of the chosen experts
// and of their devices).  [UG] "Load balancing and capacity": over capacity, a token
// skips that expert.  Dispatch (step 2) sends each token's hidden state to the device
// holding its expert; the single-device equivalent is the permuted buffer an
// all-to-all would send: rank-major, then expert, then token order.
//
// Inputs: idx [N, k].  Outputs:
//   expert_counts [E]  routed assignments (before the cap)
//   kept_counts   [E]  min(count, C)
//   expert_start  [E]  first slot of each expert in the send buffer
//   rank_counts   [R]  kept assignments per rank
//   rank_offsets  [R+1] exclusive prefix of rank_counts
//   slot_of       [N*k] slot of assignment a = t*k + j, or -1 if dropped
//   perm_src      [N*k] perm_src[slot] = a for slot < num_kept, -1 beyond
//   num_kept      [1]
//
// mode 0 (packed): assignments compete for capacity in token order (t, then j), and
//   the send buffer is packed: expert segments follow each other with no gaps.
// mode 1 (capacity-padded, choice-major): the buffer reserves C rows per expert, as
//   [BZ] exercise 2 describes ("each expert's buffer is reserved at the mean times
//   1.25"), so expert e's rows start at (its send position) * C; capacity goes to all
//   first choices in token order, then all second choices, and so on (the priority
//   GShard uses).  Padding rows carry perm_src = -1.  Requires cf > 0.  perm_src then
//   spans E*C rows; rank_offsets are the padded rank starts.
int oracle_dispatch_mode(int N, int E, int k, int R, int rank_map, float cf, int mode,
                         const int32_t* idx, int32_t* expert_counts, int32_t* kept_counts,
                         int32_t* expert_start, int32_t* rank_counts, int32_t* rank_offsets,
                         int32_t* slot_of, int32_t* perm_src, int32_t* num_kept) {
  if (R < 1 || R > E) return -1;
  if (rank_map == 0 && E % R != 0) return -1;
  if (mode != 0 && mode != 1) return -1;
  if (mode == 1 && !(cf > 0.0f)) return -1;
  const int64_t A = static_cast<int64_t>(N) * k;
  const int C = oracle_capacity(N, k, E, cf);
  std::vector<int64_t> seen(E, 0);
  std::vector<int64_t> pos(A);
  for (int e = 0; e < E; ++e) expert_counts[e] = 0;
  for (int64_t p = 0; p < A; ++p) {  // priority order
    const int64_t a = (mode == 0) ? p : (p % N) * k + p / N;  // mode 1: j major, t minor
    const int e = idx[a];
    if (e < 0 || e >= E) return -2;
    pos[a] = seen[e]++;
    expert_counts[e] += 1;
  }
  for (int e = 0; e < E; ++e) kept_counts[e] = std::min<int64_t>(expert_counts[e], C);
  // send order: rank ascending, expert ascending inside a rank
  std::vector<int> order(E);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
    return rank_of(a, E, R, rank_map) < rank_of(b, E, R, rank_map);
  });
  int64_t run = 0, kept_total = 0;
  for (int r = 0; r < R; ++r) rank_counts[r] = 0;
  for (int r = 0; r <= R; ++r) rank_offsets[r] = -1;
  for (int i = 0; i < E; ++i) {
    const int e = order[i];
    const int r = rank_of(e, E, R, rank_map);
    if (rank_offsets[r] < 0) rank_offsets[r] = static_cast<int32_t>(run);
    expert_start[e] = static_cast<int32_t>(run);
    run += (mode == 0) ? kept_counts[e] : C;
    kept_total += kept_counts[e];
    rank_counts[r] += kept_counts[e];
  }
  rank_offsets[R] = static_cast<int32_t>(run);
  *num_kept = static_cast<int32_t>(kept_total);
  const int64_t rows = (mode == 0) ? A : static_cast<int64_t>(E) * C;
  for (int64_t s = 0; s < rows; ++s) perm_src[s] = -1;
  for (int64_t a = 0; a < A; ++a) {
    const int e = idx[a];
    if (pos[a] < C) {
      const int64_t s = expert_start[e] + pos[a];
      slot_of[a] = static_cast<int32_t>(s);
      perm_src[s] = static_cast<int32_t>(a);
    } else {
      slot_of[a] = -1;
    }
  }
  return 0;
}

int oracle_dispatch(int N, int E, int k, int R, int rank_map, float cf, const int32_t* idx,
                    int32_t* expert_counts, int32_t* kept_counts, int32_t* expert_start,
                    int32_t* rank_counts, int32_t* rank_offsets, int32_t* slot_of,
                    int32_t* perm_src, int32_t* num_kept) {
  return oracle_dispatch_mode(N, E, k, R, rank_map, cf, 0, idx, expert_counts, kept_counts,
                              expert_start, rank_counts, rank_offsets, slot_of, perm_src,
                              num_kept);
}

// ---------------------------------------------------------------- 6. expert FFN
//
// y[i] = FFN_{expert[i]}(x[i]) for a list of rows (fp64 result).
// xrows [n, d] act_dtype; expert ids [n] (an id equal to E selects the shared
// expert, whose weights are passed separately); w_gate_up [E, 2F, d]; w_down [E, d, F];
// shared weights [2Fs, d], [d, Fs] (null if Fs == 0).
// [FD] 10.5: a shared expert processes every token and absorbs common patterns.
int oracle_expert_rows(int n, int d, int E, int F, int Fs, int act_dtype, const void* xrows,
                       const int32_t* expert, const void* w_gate_up, const void* w_down,
                       const void* shared_gate_up, const void* shared_down, double* y) {
#pragma omp parallel
  {
    std::vector<double> xr(d), h;
#pragma omp for schedule(dynamic, 1)
    for (int i = 0; i < n; ++i) {
      for (int c = 0; c < d; ++c) xr[c] = load_act(xrows, act_dtype, static_cast<int64_t>(i) * d + c);
      const int e = expert[i];
      double* yr = y + static_cast<int64_t>(i) * d;
      if (e == E) {
        ffn_row(xr.data(), d, Fs, act_dtype, shared_gate_up, 0, shared_down, 0, yr, h);
      } else {
        ffn_row(xr.data(), d, F, act_dtype, w_gate_up, static_cast<int64_t>(e) * 2 * F * d, w_down,
                static_cast<int64_t>(e) * d * F, yr, h);
      }
    }
  }
  return 0;
}

// ---------------------------------------------------------------- 7. combine
//
// [UG] step 4: expert outputs return to each token's home and are summed after
// weighting by the router scores.  [UG] "Load balancing and capacity": a skipped
// token passes through the layer unchanged via the residual connection.
// out[t] = x[t] + ys[t] + sum_{j kept} w[t,j] * yperm[slot_of[t,j]], fp64, j ascending.
// yperm: [*, d] in act_dtype (the values under test); ys: [N, d] act_dtype or null.
// tokens: the list of token ids to produce (out is [ntok, d]).
int oracle_combine(int ntok, const int32_t* tokens, int d, int k, int act_dtype, const void* x,
                   const void* yperm, const void* ys, const int32_t* slot_of, const double* w,
                   double* out) {
#pragma omp parallel for schedule(static)
  for (int i = 0; i < ntok; ++i) {
    const int64_t t = tokens[i];
    double* o = out + static_cast<int64_t>(i) * d;
    for (int c = 0; c < d; ++c) {
      double acc = load_act(x, act_dtype, t * d + c);
      if (ys) acc += load_act(ys, act_dtype, t * d + c);
      for (int j = 0; j < k; ++j) {
        const int32_t s = slot_of[t * k + j];
        if (s < 0) continue;
        acc += w[t * k + j] * load_act(yperm, act_dtype, static_cast<int64_t>(s) * d + c);
      }
      o[c] = acc;
    }
  }
  return 0;
}

// Whole layer for a list of tokens, from the hidden states and weights: the same
// sum as oracle_combine, with every expert output computed here in fp64 (no
// intermediate rounding).  Routing (idx, w, slot_of) is passed in.
int oracle_layer_tokens(int ntok, const int32_t* tokens, int d, int E, int k, int F, int Fs,
                        int act_dtype, const void* x, const int32_t* idx, const double* w,
                        const int32_t* slot_of, const void* w_gate_up, const void* w_down,
                        const void* shared_gate_up, const void* shared_down, double* out) {
#pragma omp parallel
  {
    std::vector<double> xr(d), yr(d), h;
#pragma omp for schedule(dynamic, 1)
    for (int i = 0; i < ntok; ++i) {
      const int64_t t = tokens[i];
      for (int c = 0; c < d; ++c) xr[c] = load_act(x, act_dtype, t * d + c);
      double* o = out + static_cast<int64_t>(i) * d;
      for (int c = 0; c < d; ++c) o[c] = xr[c];
      if (Fs > 0) {
        ffn_row(xr.data(), d, Fs, act_dtype, shared_gate_up, 0, shared_down, 0, yr.data(), h);
        for (int c = 0; c < d; ++c) o[c] += yr[c];
      }
      for (int j = 0; j < k; ++j) {
        if (slot_of[t * k + j] < 0) continue;
        const int e = idx[t * k + j];
        ffn_row(xr.data(), d, F, act_dtype, w_gate_up, static_cast<int64_t>(e) * 2 * F * d, w_down,
                static_cast<int64_t>(e) * d * F, yr.data(), h);
        const double wj = w[t * k + j];
        for (int c = 0; c < d; ++c) o[c] += wj * yr[c];
      }
    }
  }
  return 0;
}

// ---------------------------------------------------------------- 8. bias update
//
// [UG] "Load balancing and capacity", bias-based balancing: after each step the
// bias of overloaded experts is lowered and the bias of underloaded experts raised.
// Overloaded means more routed assignments than the mean load N*k/E (compared
// exactly in integers as c*E vs N*k); equal load leaves the bias unchanged.
// b_e <- b_e - step (fp32) if overloaded, b_e + step if underloaded.
int oracle_bias_update(int E, int N, int k, const int32_t* counts, float step, float* bias) {
  const int64_t mean_num = static_cast<int64_t>(N) * k;
  for (int e = 0; e < E; ++e) {
    const int64_t lhs = static_cast<int64_t>(counts[e]) * E;
    if (lhs > mean_num) {
      bias[e] = bias[e] - step;
    } else if (lhs < mean_num) {
      bias[e] = bias[e] + step;
    }
  }
  return 0;
}

// ---------------------------------------------------------------- 9. INT8 payload
//
// [BZ-D]: quantising the all-to-all payload to INT8 halves its traffic again.  The
// pages fix no format; the reading taken (symmetric, one fp32 scale per row):
//   s   = max_i |v_i| / 127                  fp32 divide
//   r   = 1 / s                              fp32 divide, once per row
//   q_i = rint(v_i * r), clamped to +-127     fp32 multiply, round half to even
//   a row of zeros has s = 0 and q = 0
// The receiver's value is (float)q_i * s, one fp32 multiply, rounded once to the
// activation type.  A code is an integer decided in floating point, so it is decided
// in fp32 (v is widened exactly from bf16).  Rows with valid[r] < 0 are skipped
// (left untouched); valid may be null (every row).
int oracle_quant_rows(int rows, int d, int act_dtype, const void* in, const int32_t* valid,
                      int8_t* q, float* scale) {
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; ++r) {
    if (valid && valid[r] < 0) continue;
    const int64_t base = static_cast<int64_t>(r) * d;
    float amax = 0.0f;
    for (int i = 0; i < d; ++i) {
      const float v = static_cast<float>(load_act(in, act_dtype, base + i));
      amax = std::max(amax, std::fabs(v));
    }
    const float s = amax / 127.0f;
    scale[r] = s;
    const float inv = s > 0.0f ? 1.0f / s : 0.0f;
    for (int i = 0; i < d; ++i) {
      int c = 0;
      if (s > 0.0f) {
        const float v = static_cast<float>(load_act(in, act_dtype, base + i));
        const float ratio = v * inv;
        c = static_cast<int>(std::nearbyint(ratio));  // default mode: nearest, ties even
        c = std::min(127, std::max(-127, c));
      }
      q[base + i] = static_cast<int8_t>(c);
    }
  }
  return 0;
}

// out[r, i] = (float)q[r, i] * scale[r] in fp32, stored in act_dtype (bf16: one
// round-to-nearest-even).  Rows with valid[r] < 0 are left untouched.
int oracle_dequant_rows(int rows, int d, int act_dtype, const int8_t* q, const float* scale,
                        const int32_t* valid, void* out) {
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; ++r) {
    if (valid && valid[r] < 0) continue;
    const int64_t base = static_cast<int64_t>(r) * d;
    for (int i = 0; i < d; ++i) {
      const float v = static_cast<float>(q[base + i]) * scale[r];
      if (act_dtype == 0) {
        static_cast<float*>(out)[base + i] = v;
      } else {
        static_cast<uint16_t*>(out)[base + i] = float_to_bf16_rne(v);
      }
    }
  }
  return 0;
}

// Combine from an INT8 return payload: as oracle_combine, with each expert output
// element taken as (float)yq * yscale (fp32 multiply), then summed in fp64:
// out[t] = x[t] + ys[t] + sum_{j kept} w[t,j] * ((float)yq[s,c] * yscale[s]), s = slot_of[t,j].
int oracle_combine_q8(int ntok, const int32_t* tokens, int d, int k, int act_dtype,
                      const void* x, const int8_t* yq, const float* yscale, const void* ys,
                      const int32_t* slot_of, const double* w, double* out) {
#pragma omp parallel for schedule(static)
  for (int i = 0; i < ntok; ++i) {
    const int64_t t = tokens[i];
    double* o = out + static_cast<int64_t>(i) * d;
    for (int c = 0; c < d; ++c) {
      double acc = load_act(x, act_dtype, t * d + c);
      if (ys) acc += load_act(ys, act_dtype, t * d + c);
      for (int j = 0; j < k; ++j) {
        const int32_t s = slot_of[t * k + j];
        if (s < 0) continue;
        const float v = static_cast<float>(yq[static_cast<int64_t>(s) * d + c]) * yscale[s];
        acc += w[t * k + j] * static_cast<double>(v);
      }
      o[c] = acc;
    }
  }
  return 0;
}

// fp32 -> bf16 bits (round to nearest even), exposed for its own pin.
int oracle_float_to_bf16(int64_t n, const float* in, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = float_to_bf16_rne(in[i]);
  return 0;
}

// ---------------------------------------------------------------- 10. backward
//
// The layer of sections 1-7 for a fixed selection (the top-k choice, the capacity
// drops and the group limit are piecewise constant in the inputs, so they pass no
// gradient; the selection-only bias has none and is moved by the sign rule of
// section 8 instead).  With dout = dL/dout:
//   combine      dy_j = w_j * dout (kept j);  dw_j = dout . y_j (kept j), 0 if dropped
//   residual     dout flows to x unchanged;  shared expert: its dy is dout itself
//   expert FFN   g = Wg x, u = Wu x, h = silu(g) * u, y = Wd h:
//                dh = Wd^T dy;  dg = dh * u * silu'(g);  du = dh * silu(g)
//                dx = Wg^T dg + Wu^T du;  dWd += dy h^T;  dWg += dg x^T;  dWu += du x^T
//                silu'(z) = s(z) (1 + z (1 - s(z))), s = the logistic function
//   router       weights from logits l (section 2):
//                softmax, normalised:   w_j = exp(l_j) / sum_sel exp  ->
//                                       dl_j = w_j (dw_j - sum_i w_i dw_i), 0 off the selection
//                softmax, unnormalised: w_j = p_j, p = softmax over all E ->
//                                       dl_e = p_e (dw_e - sum_j w_j dw_j), dw_e = 0 off the selection
//                sigmoid, normalised:   w_j = s_j / sum_sel s ->
//                                       dl_j = s_j (1 - s_j) (dw_j - sum_i w_i dw_i) / sum_sel s
//                sigmoid, unnormalised: dl_j = s_j (1 - s_j) dw_j
//                (s_j = S(l_j), the fp32 function of section 2, as in the forward;
//                its derivative is that of the logistic function)
//                dx += Wr^T dl;  dWr += dl x^T;  db += dl
//   dispatch     dx[t] = dout[t] + dx_shared[t] + dx_router[t] + sum_{j kept} dx_j
// All in fp64.

// Combine backward.  dout [N, d] act; yperm [*, d] act (the forward's expert rows);
// slot_of [N*k]; w [N*k] fp64.  dy [*, d] fp64 written at the kept slots only;
// dw [N*k] fp64 (0 for dropped choices).
int oracle_combine_backward(int N, int d, int k, int act_dtype, const void* dout,
                            const void* yperm, const int32_t* slot_of, const double* w,
                            double* dy, double* dw) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < N; ++t) {
    for (int j = 0; j < k; ++j) {
      const int64_t a = static_cast<int64_t>(t) * k + j;
      const int32_t s = slot_of[a];
      if (s < 0) {
        dw[a] = 0.0;
        continue;
      }
      double dot = 0.0;
      for (int c = 0; c < d; ++c) {
        const double g = load_act(dout, act_dtype, static_cast<int64_t>(t) * d + c);
        dot += g * load_act(yperm, act_dtype, static_cast<int64_t>(s) * d + c);
        dy[static_cast<int64_t>(s) * d + c] = w[a] * g;
      }
      dw[a] = dot;
    }
  }
  return 0;
}

namespace {
inline double logistic(double z) { return 1.0 / (1.0 + std::exp(-z)); }

// g, u of one row for the gate/up rows f (fp64).
inline void gate_up_at(const double* x, int d, int F, int act_dtype, const void* wgu,
                       int64_t wgu_off, int f, double* g, double* u) {
  double a = 0.0, b = 0.0;
  const int64_t rg = wgu_off + static_cast<int64_t>(f) * d;
  const int64_t ru = wgu_off + static_cast<int64_t>(F + f) * d;
  for (int i = 0; i < d; ++i) {
    a += x[i] * load_act(wgu, act_dtype, rg + i);
    b += x[i] * load_act(wgu, act_dtype, ru + i);
  }
  *g = a;
  *u = b;
}

// dh_f = sum_o dy_o Wd[o][f]
inline double dh_at(const double* dy, int d, int F, int act_dtype, const void* wd, int64_t wd_off,
                    int f) {
  double acc = 0.0;
  for (int o = 0; o < d; ++o)
    acc += dy[o] * load_act(wd, act_dtype, wd_off + static_cast<int64_t>(o) * F + f);
  return acc;
}
}  // namespace

// Expert FFN backward, input gradient of each row.  Row r belongs to expert
// expert[r] (E = the shared expert); x rows and dy rows in act_dtype.
// dx [n, d] fp64.
int oracle_ffn_backward_rows(int n, int d, int E, int F, int Fs, int act_dtype, const void* xrows,
                             const void* dyrows, const int32_t* expert, const void* w_gate_up,
                             const void* w_down, const void* shared_gate_up,
                             const void* shared_down, double* dx) {
#pragma omp parallel
  {
    std::vector<double> xr(d), dyr(d), dg, du;
#pragma omp for schedule(dynamic, 1)
    for (int r = 0; r < n; ++r) {
      for (int c = 0; c < d; ++c) {
        xr[c] = load_act(xrows, act_dtype, static_cast<int64_t>(r) * d + c);
        dyr[c] = load_act(dyrows, act_dtype, static_cast<int64_t>(r) * d + c);
      }
      const int e = expert[r];
      const bool sh = e >= E;
      const int Fx = sh ? Fs : F;
      const void* wgu = sh ? shared_gate_up : w_gate_up;
      const void* wd = sh ? shared_down : w_down;
      const int64_t gu_off = sh ? 0 : static_cast<int64_t>(e) * 2 * F * d;
      const int64_t d_off = sh ? 0 : static_cast<int64_t>(e) * d * F;
      dg.assign(Fx, 0.0);
      du.assign(Fx, 0.0);
      for (int f = 0; f < Fx; ++f) {
        double g, u;
        gate_up_at(xr.data(), d, Fx, act_dtype, wgu, gu_off, f, &g, &u);
        const double dh = dh_at(dyr.data(), d, Fx, act_dtype, wd, d_off, f);
        const double sg = logistic(g);
        dg[f] = dh * u * sg * (1.0 + g * (1.0 - sg));
        du[f] = dh * g * sg;
      }
      double* o = dx + static_cast<int64_t>(r) * d;
      for (int i = 0; i < d; ++i) {
        double acc = 0.0;
        for (int f = 0; f < Fx; ++f) {
          acc += dg[f] * load_act(wgu, act_dtype, gu_off + static_cast<int64_t>(f) * d + i);
          acc += du[f] * load_act(wgu, act_dtype, gu_off + static_cast<int64_t>(Fx + f) * d + i);
        }
        o[i] = acc;
      }
    }
  }
  return 0;
}

// Weight gradients of one expert (or the shared expert) from its n rows, for the
// listed hidden units f (nf of them; pass all 0..Fx-1 for the full gradients):
//   dWd[:, f]   = sum_r dy_r h_r[f]        -> dwd_cols [nf, d]  (column f of dWd, as a row)
//   dWg[f, :]   = sum_r dg_r[f] x_r        -> dwg_rows [nf, d]
//   dWu[f, :]   = sum_r du_r[f] x_r        -> dwu_rows [nf, d]
// wgu / wd point at this expert's [2Fx, d] and [d, Fx] weights.
int oracle_ffn_wgrad(int n, int d, int Fx, int act_dtype, const void* xrows, const void* dyrows,
                     const void* wgu, const void* wd, int nf, const int32_t* fs,
                     double* dwd_cols, double* dwg_rows, double* dwu_rows) {
#pragma omp parallel
  {
    std::vector<double> xr(d), dyr(d);
#pragma omp for schedule(dynamic, 1)
    for (int q = 0; q < nf; ++q) {
      const int f = fs[q];
      double* cd = dwd_cols + static_cast<int64_t>(q) * d;
      double* rg = dwg_rows + static_cast<int64_t>(q) * d;
      double* ru = dwu_rows + static_cast<int64_t>(q) * d;
      for (int i = 0; i < d; ++i) cd[i] = rg[i] = ru[i] = 0.0;
      for (int r = 0; r < n; ++r) {
        for (int c = 0; c < d; ++c) {
          xr[c] = load_act(xrows, act_dtype, static_cast<int64_t>(r) * d + c);
          dyr[c] = load_act(dyrows, act_dtype, static_cast<int64_t>(r) * d + c);
        }
        double g, u;
        gate_up_at(xr.data(), d, Fx, act_dtype, wgu, 0, f, &g, &u);
        const double sg = logistic(g);
        const double h = g * sg * u;
        const double dh = dh_at(dyr.data(), d, Fx, act_dtype, wd, 0, f);
        const double dgv = dh * u * sg * (1.0 + g * (1.0 - sg));
        const double duv = dh * g * sg;
        for (int i = 0; i < d; ++i) {
          cd[i] += dyr[i] * h;
          rg[i] += dgv * xr[i];
          ru[i] += duv * xr[i];
        }
      }
    }
  }
  return 0;
}

// Router backward, logits gradient.  logits [N, E] fp32 (the forward's), idx [N, k],
// dw [N, k] fp64 (from the combine backward; 0 for dropped choices).  dl [N, E] fp64.
int oracle_route_backward(int N, int E, int k, int score_fn, int normalize, const float* logits,
                          const int32_t* idx, const double* dw, double* dl) {
#pragma omp parallel
  {
    std::vector<double> w(k), sv(k);
#pragma omp for schedule(static)
    for (int t = 0; t < N; ++t) {
      const float* l = logits + static_cast<int64_t>(t) * E;
      const int32_t* id = idx + static_cast<int64_t>(t) * k;
      const double* g = dw + static_cast<int64_t>(t) * k;
      double* o = dl + static_cast<int64_t>(t) * E;
      for (int e = 0; e < E; ++e) o[e] = 0.0;
      if (score_fn == 1) {
        double ssum = 0.0;
        for (int j = 0; j < k; ++j) {
          sv[j] = static_cast<double>(sigmoid_spec(l[id[j]]));
          ssum += sv[j];
        }
        if (normalize) {
          double wdw = 0.0;
          for (int j = 0; j < k; ++j) wdw += sv[j] / ssum * g[j];
          for (int j = 0; j < k; ++j)
            o[id[j]] = sv[j] * (1.0 - sv[j]) * (g[j] - wdw) / ssum;
        } else {
          for (int j = 0; j < k; ++j) o[id[j]] = sv[j] * (1.0 - sv[j]) * g[j];
        }
      } else {
        double m = -INFINITY;
        for (int e = 0; e < E; ++e) m = std::max(m, static_cast<double>(l[e]));
        if (normalize) {
          double zs = 0.0;
          for (int j = 0; j < k; ++j) zs += std::exp(static_cast<double>(l[id[j]]) - m);
          double wdw = 0.0;
          for (int j = 0; j < k; ++j) {
            w[j] = std::exp(static_cast<double>(l[id[j]]) - m) / zs;
            wdw += w[j] * g[j];
          }
          for (int j = 0; j < k; ++j) o[id[j]] = w[j] * (g[j] - wdw);
        } else {
          double z = 0.0;
          for (int e = 0; e < E; ++e) z += std::exp(static_cast<double>(l[e]) - m);
          double wdw = 0.0;
          for (int j = 0; j < k; ++j) wdw += std::exp(static_cast<double>(l[id[j]]) - m) / z * g[j];
          for (int e = 0; e < E; ++e) o[e] = -std::exp(static_cast<double>(l[e]) - m) / z * wdw;
          for (int j = 0; j < k; ++j)
            o[id[j]] += std::exp(static_cast<double>(l[id[j]]) - m) / z * g[j];
        }
      }
    }
  }
  return 0;
}

// Router parameter and input gradients from dl [N, E] (fp64):
//   dx_router [ntok, d] for the listed tokens: dl[t] . Wr  (Wr [E, d] fp32)
//   dWr [E, d] = sum_t dl[t, e] x[t]  and db [E] = sum_t dl[t, e]   (all N tokens;
//   dwr / db may be null to skip them)
int oracle_router_grads(int N, int d, int E, int act_dtype, const void* x, const float* Wr,
                        const double* dl, int ntok, const int32_t* tokens, double* dx_router,
                        double* dwr, double* db) {
#pragma omp parallel for schedule(static)
  for (int i = 0; i < ntok; ++i) {
    const int64_t t = tokens[i];
    for (int c = 0; c < d; ++c) {
      double acc = 0.0;
      for (int e = 0; e < E; ++e) acc += dl[t * E + e] * static_cast<double>(Wr[static_cast<int64_t>(e) * d + c]);
      dx_router[static_cast<int64_t>(i) * d + c] = acc;
    }
  }
  if (dwr) {
#pragma omp parallel for schedule(static)
    for (int e = 0; e < E; ++e) {
      double* o = dwr + static_cast<int64_t>(e) * d;
      for (int c = 0; c < d; ++c) o[c] = 0.0;
      double bsum = 0.0;
      for (int t = 0; t < N; ++t) {
        const double v = dl[static_cast<int64_t>(t) * E + e];
        if (v == 0.0) continue;
        bsum += v;
        for (int c = 0; c < d; ++c) o[c] += v * load_act(x, act_dtype, static_cast<int64_t>(t) * d + c);
      }
      if (db) db[e] = bsum;
    }
  }
  return 0;
}

// Dispatch backward for the listed tokens: dx[t] = dout[t] + dxs[t] + dxr[t] +
// sum_{j kept} dxperm[slot_of[t, j]].  dout, dxs, dxperm act_dtype (dxs may be null);
// dxr fp32 [N, d] or null.  out [ntok, d] fp64.
int oracle_dispatch_backward(int ntok, const int32_t* tokens, int d, int k, int act_dtype,
                             const void* dout, const void* dxs, const float* dxr,
                             const void* dxperm, const int32_t* slot_of, double* out) {
#pragma omp parallel for schedule(static)
  for (int i = 0; i < ntok; ++i) {
    const int64_t t = tokens[i];
    for (int c = 0; c < d; ++c) {
      double acc = load_act(dout, act_dtype, t * d + c);
      if (dxs) acc += load_act(dxs, act_dtype, t * d + c);
      if (dxr) acc += static_cast<double>(dxr[t * d + c]);
      for (int j = 0; j < k; ++j) {
        const int32_t s = slot_of[t * k + j];
        if (s >= 0) acc += load_act(dxperm, act_dtype, static_cast<int64_t>(s) * d + c);
      }
      out[static_cast<int64_t>(i) * d + c] = acc;
    }
  }
  return 0;
}

}  // extern "C"
