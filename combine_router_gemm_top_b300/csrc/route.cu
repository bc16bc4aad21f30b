// moe_route kernels: router GEMM (tcgen05 split-K for bf16, fp32 FMA for
// fp32), then per-token scoring, group-limited top-k and gates; for up to
// 32 experts, both in one kernel (bf16: 16 tokens a block on the warp-level
// MMA; fp32 with a small W_r: one warp per token on the FMA pipes)
// ("Expert Parallelism in LLMs", The Execution Pipeline, step 1 "Router
// Gating and Softmax Selection": g_t = Softmax(TopK(W_g x_t, k))).
#include <cuda.h>
#include <float.h>

#include "common.cuh"
#include "internal.h"
#include "umma_gemm.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// Sigmoid score of the sigmoid router: s = fp32(1 / (1 + e^-l)), evaluated in
// float64 and rounded once to fp32 (round to nearest even).  The selection key
// is then s + b_e, added in fp32.  A float64 evaluation carries a few float64
// ulp of error, so s is the correctly rounded sigmoid except where the exact
// value lies within that distance of the midpoint between two fp32 values.
// For l >= 18 the exact sigmoid is above 1 - 2^-25 and rounds to 1.0, so no
// exponential is evaluated there.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float sigmoid_score(float l) {
  if (l >= 18.0f) return 1.0f;
  const double e = exp(-static_cast<double>(l));
  return __double2float_rn(1.0 / (1.0 + e));
}

// Order-preserving code of an fp32 selection key: for keys a, b (+0 and -0
// equal), a > b exactly when key_code(a) > key_code(b).  Every key, even
// -inf, codes above 0, and 0 marks an expert that is not (or no longer)
// eligible.
__device__ __forceinline__ uint32_t key_code(float f) {
  const uint32_t u = f == 0.0f ? 0u : __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1)
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, d));
  return v;
}

// The winner among the warp's candidates: lane l holds expert l + 32*i in
// code[i].  Largest code first, the lower expert index on equal codes; -1
// when no candidate is eligible.  Two warp reductions (redux.sync) per call.
template <int NI>
__device__ __forceinline__ int warp_argmax(const uint32_t (&code)[NI],
                                           int lane) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < NI; ++i) m = max(m, code[i]);
  const uint32_t top = __reduce_max_sync(0xffffffffu, m);
  if (top == 0) return -1;
  uint32_t first = 0xffffffffu;
#pragma unroll
  for (int i = NI - 1; i >= 0; --i)
    if (code[i] == top) first = static_cast<uint32_t>(lane + 32 * i);
  return static_cast<int>(__reduce_min_sync(0xffffffffu, first));
}

// group of expert e (< 256) for group size gs: e / gs through one fp32
// multiply.  (e + 0.5) / gs lies at least 1/512 away from an integer and the
// product's error is below 2^-15, so truncation gives the exact quotient.
__device__ __forceinline__ int group_of(int e, float inv_gs) {
  return static_cast<int>((static_cast<float>(e) + 0.5f) * inv_gs);
}

constexpr int kSelWarps = 8;
constexpr int kSelGroupTop = 8;   // per-lane scan handles group_score_topk <= 8

// Lane g < n_groups: the fp32 sum of the m largest keys of group g (added
// largest first) and the m-th largest key; keys of experts e = lane + 32 i
// in key[] (-inf for none).  Lane g scans its group's keys from the warp's
// shared scratch keeping the MT largest in a sorted list (m <= MT <= 8;
// equal keys are interchangeable for the sum).
template <int NI, int MT>
__device__ __forceinline__ void group_top_mt(const float (&key)[NI], int lane,
                                             int E, int n_groups, int gs,
                                             int m, float* sk, float& sum,
                                             float& mth) {
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int e = lane + 32 * i;
    if (e < E) sk[e + (e >> 5)] = key[i];
  }
  __syncwarp();
  sum = 0.0f;
  mth = -INFINITY;
  if (lane < n_groups) {
    float v[MT];
#pragma unroll
    for (int j = 0; j < MT; ++j) v[j] = -INFINITY;
    for (int e = lane * gs; e < (lane + 1) * gs; ++e) {
      float x = sk[e + (e >> 5)];
#pragma unroll
      for (int j = 0; j < MT; ++j) {
        const float hi = fmaxf(v[j], x);
        x = fminf(v[j], x);
        v[j] = hi;
      }
    }
#pragma unroll
    for (int j = 0; j < MT; ++j) {
      if (j < m) sum = __fadd_rn(sum, v[j]);
      if (j == m - 1) mth = v[j];
    }
  }
  __syncwarp();
}
// the sorted list as short as m allows (the common m = 2 keeps two)
template <int NI>
__device__ __forceinline__ void group_top(const float (&key)[NI], int lane,
                                          int E, int n_groups, int gs, int m,
                                          float* sk, float& sum, float& mth) {
  if (m <= 2)
    group_top_mt<NI, 2>(key, lane, E, n_groups, gs, m, sk, sum, mth);
  else
    group_top_mt<NI, kSelGroupTop>(key, lane, E, n_groups, gs, m, sk, sum, mth);
}

// Lane g < n_groups: the fp32 sum of the m largest keys of group g by m
// warp-wide arg-max rounds per group (any m).
template <int NI>
__device__ __forceinline__ float group_sum_rounds(const float (&key)[NI],
                                                  const uint32_t (&code)[NI],
                                                  int lane, int n_groups,
                                                  float inv_gs, int m) {
  float gscore = 0.0f;
  for (int g = 0; g < n_groups; ++g) {
    uint32_t c[NI];
#pragma unroll
    for (int i = 0; i < NI; ++i)
      c[i] = group_of(lane + 32 * i, inv_gs) == g ? code[i] : 0u;
    float acc = 0.0f;   // the same on every lane, largest key first
    for (int j = 0; j < m; ++j) {
      const int w = warp_argmax<NI>(c, lane);
      float mine = 0.0f;
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        if (lane + 32 * i == w) {
          mine = key[i];
          c[i] = 0u;
        }
      }
      acc = __fadd_rn(acc, __shfl_sync(0xffffffffu, mine, w & 31));
    }
    if (lane == g) gscore = acc;
  }
  return gscore;
}

// The topk_groups best groups by score (lower group index on equal scores)
// as a bit mask, from lane g's score of group g.
__device__ __forceinline__ uint32_t choose_groups(float gscore, int lane,
                                                  int n_groups,
                                                  int topk_groups) {
  uint32_t gc[1] = {lane < n_groups ? key_code(gscore) : 0u};
  uint32_t chosen = 0;
  for (int j = 0; j < topk_groups; ++j) {
    const int w = warp_argmax<1>(gc, lane);
    if (w < 0) break;
    chosen |= 1u << w;
    if (lane == w) gc[0] = 0u;
  }
  return chosen;
}

// top-k by repeated warp arg-max over code[]: lane j < k receives slot j's
// expert and its logit.
template <int NI>
__device__ __forceinline__ void topk_rounds(uint32_t (&code)[NI],
                                            const float (&lg)[NI], int k,
                                            int lane, int& my_idx,
                                            float& my_logit) {
  my_idx = -1;
  my_logit = 0.0f;
  for (int j = 0; j < k; ++j) {
    const int w = warp_argmax<NI>(code, lane);
    float mine = 0.0f;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      if (lane + 32 * i == w) {
        mine = lg[i];
        code[i] = 0u;
      }
    }
    const float wl = __shfl_sync(0xffffffffu, mine, w & 31);
    if (lane == j) {
      my_idx = w;
      my_logit = wl;
    }
  }
}

// The same top-k as topk_rounds with each lane's NI candidates sorted
// first (key code descending, the lower expert first on equal codes), so a
// round compares one head per lane: the largest head code, the lowest
// expert holding it, and the winner's lane drops its head.  The lowest
// expert with the top code is always a head (a lane's own equal codes are
// ordered by expert), so the rounds pick what topk_rounds picks.
template <int NI>
__device__ __forceinline__ void topk_presorted(uint32_t (&code)[NI],
                                               const float (&lg)[NI], int k,
                                               int lane, int& my_idx,
                                               float& my_logit) {
  int ex[NI];
  float lv[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    ex[i] = lane + 32 * i;
    lv[i] = lg[i];
  }
  // odd-even transposition sort, descending by (code, -expert)
#pragma unroll
  for (int pass = 0; pass < NI; ++pass) {
#pragma unroll
    for (int i = pass & 1; i + 1 < NI; i += 2) {
      const bool sw = code[i + 1] > code[i] ||
                      (code[i + 1] == code[i] && ex[i + 1] < ex[i]);
      if (sw) {
        const uint32_t tc = code[i];
        code[i] = code[i + 1];
        code[i + 1] = tc;
        const int te = ex[i];
        ex[i] = ex[i + 1];
        ex[i + 1] = te;
        const float tl = lv[i];
        lv[i] = lv[i + 1];
        lv[i + 1] = tl;
      }
    }
  }
  my_idx = -1;
  my_logit = 0.0f;
  for (int j = 0; j < k; ++j) {
    const uint32_t top = __reduce_max_sync(0xffffffffu, code[0]);
    if (top == 0) break;   // no eligible expert left
    const uint32_t cand = code[0] == top ? static_cast<uint32_t>(ex[0])
                                         : 0xffffffffu;
    const int w = static_cast<int>(__reduce_min_sync(0xffffffffu, cand));
    const float wl = __shfl_sync(0xffffffffu, lv[0], w & 31);
    if (lane == j) {
      my_idx = w;
      my_logit = wl;
    }
    if ((w & 31) == lane) {
#pragma unroll
      for (int i = 0; i + 1 < NI; ++i) {
        code[i] = code[i + 1];
        ex[i] = ex[i + 1];
        lv[i] = lv[i + 1];
      }
      code[NI - 1] = 0u;
    }
  }
}

// Softmax modes: the key is the logit itself.
template <int NI>
__device__ __forceinline__ void select_by_logit(const RouteSelectArgs& a,
                                                int lane, const float (&lg)[NI],
                                                float* sk, int& my_idx,
                                                float& my_logit) {
  const int E = a.E;
  float key[NI];
  uint32_t code[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const bool in = lane + 32 * i < E;
    key[i] = in ? lg[i] : -INFINITY;
    code[i] = in ? key_code(lg[i]) : 0u;
  }
  if (a.n_groups > 1) {
    const int gs = E / a.n_groups;
    const float inv_gs = 1.0f / static_cast<float>(gs);
    const int m = a.group_score_topk;
    float gscore, mth;
    if (m <= kSelGroupTop)
      group_top<NI>(key, lane, E, a.n_groups, gs, m, sk, gscore, mth);
    else
      gscore = group_sum_rounds<NI>(key, code, lane, a.n_groups, inv_gs, m);
    const uint32_t chosen = choose_groups(gscore, lane, a.n_groups,
                                          a.topk_groups);
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((chosen >> group_of(e, inv_gs)) & 1u)) code[i] = 0u;
    }
  }
  topk_presorted<NI>(code, lg, a.k, lane, my_idx, my_logit);
}

// fp32 approximation of the sigmoid score: expf (within 2 ulp), one add and
// one division, so it lies within 3.5 * 2^-24 of fp32(sigmoid(l)), and an
// approximate key fp32(approx + b) within 2^-21.5 (1 + |b|) of the exact
// key.  The selection trusts it only where keys lie more than twice that
// bound, taken four times over, apart; the gates use it as it is.
__device__ __forceinline__ float sigmoid_approx(float l) {
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-l)));
}
constexpr float kSigmoidKeySlack = 1.0f / 524288.0f;   // 2^-19

// Exact keys fp32(sigmoid_score(l) + b_e) of the experts flagged in need[]
// (this lane's slots), spread over the warp: the flagged experts are
// numbered slot by slot, lane by lane, and candidate c is evaluated by lane
// c mod 32 in round c / 32, so the float64 work is not left to the lanes
// that happen to own the candidates.
template <int NI>
__device__ __forceinline__ void exact_sigmoid_keys(const RouteSelectArgs& a,
                                                   int lane,
                                                   const float (&lg)[NI],
                                                   const bool (&need)[NI],
                                                   float (&key)[NI]) {
  uint32_t mask[NI];
  int base[NI];
  int total = 0;
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    mask[i] = __ballot_sync(0xffffffffu, need[i]);
    base[i] = total;
    total += __popc(mask[i]);
  }
  const uint32_t below = (1u << lane) - 1u;
  for (int r0 = 0; r0 < total; r0 += 32) {
    const int c = r0 + lane;   // the candidate this lane evaluates
    float l = 0.0f;
    int e = -1;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int n = c - base[i];
      const bool mine = n >= 0 && n < __popc(mask[i]);
      int owner = 0;
      if (mine) {
        uint32_t mm = mask[i];
        for (int q = 0; q < n; ++q) mm &= mm - 1u;   // drop the n lowest
        owner = __ffs(mm) - 1;
      }
      const float v = __shfl_sync(0xffffffffu, lg[i], owner);
      if (mine) {
        l = v;
        e = owner + 32 * i;
      }
    }
    float kx = 0.0f;
    if (e >= 0) {
      kx = sigmoid_score(l);
      if (a.sel_bias != nullptr) kx = __fadd_rn(kx, a.sel_bias[e]);
    }
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int cc = base[i] + __popc(mask[i] & below);   // (lane, i)'s number
      const bool here = need[i] && cc >= r0 && cc < r0 + 32;
      const float v = __shfl_sync(0xffffffffu, kx, here ? cc - r0 : 0);
      if (here) key[i] = v;
    }
  }
}

// Sigmoid mode: key = fp32(fp32(sigmoid(l)) + b_e), the sigmoid in float64.
// Float64 runs at a small fraction of the fp32 rate on this part, so every
// expert gets the cheap approximate key, within delta = 2^-19 (1 + max|b|)
// of its exact key, and exact keys are evaluated only where the approximate
// ones cannot decide.  Two approximate keys more than 2 delta ("slack")
// apart are ordered as their exact keys are, and an expert whose approximate
// key is more than slack from every other candidate's compares correctly
// with exact keys too, so only candidates within slack of another one need
// their exact key.
//   Groups: a group score (sum of the m largest keys) from approximate keys
//   lies within eps_g of the exact one; when the weakest chosen group leads
//   the strongest other group by more than 2 eps_g the chosen set is
//   certain, otherwise the exact scores are formed from exact keys of each
//   group's candidates (those within slack of its m-th approximate key).
//   Top-k: the eligible experts are taken in approximate-key order down to
//   slack below the k-th (the candidates; an expert further below lies under
//   k others whatever the exact keys are), and the candidates within slack
//   of a neighbour in that order get exact keys before the final rounds.
__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1)
    v = fminf(v, __shfl_xor_sync(0xffffffffu, v, d));
  return v;
}

template <int NI>
__device__ __forceinline__ void select_by_sigmoid(const RouteSelectArgs& a,
                                                  int lane,
                                                  const float (&lg)[NI],
                                                  float* sk, int& my_idx,
                                                  float& my_logit) {
  const int E = a.E;
  float ka[NI], key[NI];
  bool elig[NI], exact[NI], need[NI];
  float bmax = 0.0f;
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int e = lane + 32 * i;
    elig[i] = e < E;
    exact[i] = false;
    float b = 0.0f;
    if (elig[i] && a.sel_bias != nullptr) b = a.sel_bias[e];
    ka[i] = elig[i] ? __fadd_rn(sigmoid_approx(lg[i]), b) : -INFINITY;
    key[i] = ka[i];
    bmax = fmaxf(bmax, fabsf(b));
  }
  bmax = warp_max(bmax);
  const float delta = kSigmoidKeySlack * (1.0f + bmax);
  const float slack = 2.0f * delta;

  if (a.n_groups > 1) {
    const int gs = E / a.n_groups;
    const float inv_gs = 1.0f / static_cast<float>(gs);
    const int m = a.group_score_topk;
    float gscore, mth;
    uint32_t chosen;
    if (m <= kSelGroupTop) {
      group_top<NI>(ka, lane, E, a.n_groups, gs, m, sk, gscore, mth);
      chosen = choose_groups(gscore, lane, a.n_groups, a.topk_groups);
      // m keys off by delta each, and the m - 1 fp32 additions of either
      // sum rounding by at most 2^-24 of a partial sum below m (1 + max|b|)
      const float eps_g = static_cast<float>(m) * delta +
                          2.0f * static_cast<float>((m - 1) * m) *
                              5.9604645e-8f * (1.0f + bmax);
      const bool grp = lane < a.n_groups;
      const bool in = grp && ((chosen >> lane) & 1u);
      const float lo_in = warp_min(in ? gscore : INFINITY);
      const float hi_out = warp_max(grp && !in ? gscore : -INFINITY);
      if (!(lo_in - hi_out > 2.0f * eps_g)) {
        // exact keys for each group's candidates, then the exact group
        // scores from those alone
        const float thr_own = mth - slack;
#pragma unroll
        for (int i = 0; i < NI; ++i) {
          const int g = group_of(lane + 32 * i, inv_gs);
          const float thr = __shfl_sync(0xffffffffu, thr_own, g & 31);
          need[i] = elig[i] && ka[i] >= thr;
        }
        exact_sigmoid_keys<NI>(a, lane, lg, need, key);
        float kc[NI];
#pragma unroll
        for (int i = 0; i < NI; ++i) {
          exact[i] = need[i];
          kc[i] = exact[i] ? key[i] : -INFINITY;
        }
        group_top<NI>(kc, lane, E, a.n_groups, gs, m, sk, gscore, mth);
        chosen = choose_groups(gscore, lane, a.n_groups, a.topk_groups);
      }
    } else {
      // wider group scores: exact keys for every expert
#pragma unroll
      for (int i = 0; i < NI; ++i) need[i] = elig[i];
      exact_sigmoid_keys<NI>(a, lane, lg, need, key);
      uint32_t code[NI];
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        exact[i] = elig[i];
        code[i] = elig[i] ? key_code(key[i]) : 0u;
      }
      gscore = group_sum_rounds<NI>(key, code, lane, a.n_groups, inv_gs, m);
      chosen = choose_groups(gscore, lane, a.n_groups, a.topk_groups);
    }
#pragma unroll
    for (int i = 0; i < NI; ++i)
      if (elig[i] && !((chosen >> group_of(lane + 32 * i, inv_gs)) & 1u))
        elig[i] = false;
  }

  // the eligible experts in approximate-key order down to slack below the
  // k-th: lane r holds the r-th (up to 32)
  uint32_t ca[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) ca[i] = elig[i] ? key_code(ka[i]) : 0u;
  float tk = -INFINITY;
  int n_ord = 0;
  bool many = false;   // more than 32 candidates
  int ord_e = -1;
  float ord_k = -INFINITY, ord_l = 0.0f;
  for (int r = 0;; ++r) {
    const int w = warp_argmax<NI>(ca, lane);
    if (w < 0) break;   // every eligible expert taken
    float mine = 0.0f, mine_l = 0.0f;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      if (lane + 32 * i == w) {
        mine = ka[i];
        mine_l = lg[i];
        ca[i] = 0u;
      }
    }
    const float kw = __shfl_sync(0xffffffffu, mine, w & 31);
    const float lw = __shfl_sync(0xffffffffu, mine_l, w & 31);
    if (r >= a.k && kw < tk - slack) break;
    if (r == a.k - 1) tk = kw;
    if (r == 32) {
      many = true;
      break;
    }
    if (lane == r) {
      ord_e = w;
      ord_k = kw;
      ord_l = lw;
    }
    n_ord = r + 1;
  }
  const float thr = tk - slack;
  if (many) {
    // exact keys for every candidate
#pragma unroll
    for (int i = 0; i < NI; ++i) need[i] = elig[i] && ka[i] >= thr && !exact[i];
  } else {
    const float up = __shfl_up_sync(0xffffffffu, ord_k, 1);
    const float down = __shfl_down_sync(0xffffffffu, ord_k, 1);
    const bool amb = lane < n_ord && ((lane > 0 && up - ord_k <= slack) ||
                                      (lane + 1 < n_ord && ord_k - down <= slack));
    if (!__any_sync(0xffffffffu, amb)) {
      // no near-tie among the candidates: the approximate order is the
      // exact order, and its first k are the selection
      my_idx = lane < a.k ? ord_e : -1;
      my_logit = lane < a.k ? ord_l : 0.0f;
      return;
    }
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const uint32_t bits = __reduce_or_sync(
          0xffffffffu,
          amb && (ord_e >> 5) == i ? (1u << (ord_e & 31)) : 0u);
      need[i] = ((bits >> lane) & 1u) && !exact[i];
    }
  }
  exact_sigmoid_keys<NI>(a, lane, lg, need, key);
  uint32_t code[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const bool cand = elig[i] && ka[i] >= thr;
    code[i] = cand ? key_code(key[i]) : 0u;
  }
  topk_rounds<NI>(code, lg, a.k, lane, my_idx, my_logit);
}

// Selection for one token, one warp: lane l holds the logits of experts
// e = l + 32*i, i < NI, in lg; sk is the warp's shared scratch for the
// group scan.  Writes the token's ids and gates (and logits when asked).
template <int NI>
__device__ __forceinline__ void select_token(const RouteSelectArgs& a,
                                             int64_t t, int lane,
                                             float (&lg)[NI], float* sk) {
  const int E = a.E;
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      if (a.logit_offset != nullptr) lg[i] = __fadd_rn(lg[i], a.logit_offset[e]);
      if (a.logits_out != nullptr) a.logits_out[t * E + e] = lg[i];
    }
  }
  int my_idx;
  float my_logit;
  if (a.score == MOE_SCORE_SIGMOID_BIAS)
    select_by_sigmoid<NI>(a, lane, lg, sk, my_idx, my_logit);
  else
    select_by_logit<NI>(a, lane, lg, sk, my_idx, my_logit);

  // gates
  const bool slot = lane < a.k;
  float g = 0.0f;
  if (a.score == MOE_SCORE_SOFTMAX_TOPK) {
    const float mx = __shfl_sync(0xffffffffu, my_logit, 0);   // slot 0 = max
    const float ex = slot ? expf(my_logit - mx) : 0.0f;
    g = ex / warp_sum(ex);
  } else if (a.score == MOE_SCORE_SOFTMAX_FULL) {
    float mx = -FLT_MAX;
#pragma unroll
    for (int i = 0; i < NI; ++i)
      if (lane + 32 * i < E) mx = fmaxf(mx, lg[i]);
    mx = warp_max(mx);
    float z = 0.0f;
#pragma unroll
    for (int i = 0; i < NI; ++i)
      if (lane + 32 * i < E) z += expf(lg[i] - mx);
    z = warp_sum(z);
    g = slot ? expf(my_logit - mx) / z : 0.0f;
  } else {
    // gates from the fp32 sigmoid (within 3.5 * 2^-24 of the exact score):
    // they are compared within a tolerance, unlike the selection keys
    const float sg = slot ? sigmoid_approx(my_logit) : 0.0f;
    g = sg / warp_sum(sg);
  }
  if (slot) {
    a.topk_idx[t * a.k + lane] = my_idx;
    a.topk_gate[t * a.k + lane] = g;
  }
}

// One warp per token: the split-K partial sums, added in split order (the
// loads of one split are independent of each other), then the selection.
template <int NI>
__global__ void __launch_bounds__(kSelWarps * 32, 4)
    route_select_kernel(RouteSelectArgs a) {
  // keys of each warp's token for the group scan, one pad word per 32 so
  // that lanes reading along different groups hit different banks
  __shared__ float skey[kSelWarps][256 + 8];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kSelWarps + warp;
  if (t >= a.T) return;
  const int E = a.E;
  float lg[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int e = lane + 32 * i;
    lg[i] = e < E ? a.partial[t * E + e] : 0.0f;
  }
#pragma unroll 2
  for (int s = 1; s < a.splits; ++s) {
    const float* ps = a.partial + (static_cast<int64_t>(s) * a.T + t) * E;
    float p[NI];
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int e = lane + 32 * i;
      p[i] = e < E ? ps[e] : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < NI; ++i) lg[i] = __fadd_rn(lg[i], p[i]);
  }
  select_token<NI>(a, t, lane, lg, skey[warp]);
}

// The whole fp32 router for small E x D in one kernel, one warp per token.
// One thread copies W_r (E x D) into shared memory with a single bulk copy
// while the warps' first x vectors are in flight; rows E..EP-1 are zero so
// that the expert loop has no branch.  Lane l owns the token's 16-byte
// vectors l, l + 32, ..., accumulates the EP dot products in fp32 on the FMA
// pipes, a shuffle tree adds the lanes' parts, and lane e keeps expert e's
// logit for the selection.  For few experts this replaces a router GEMM plus
// a separate select launch.
template <typename T, int EP>
__global__ void __launch_bounds__(kSelWarps * 32)
    route_warp_kernel(RouteSelectArgs a, const T* __restrict__ x,
                      const T* __restrict__ w, int D) {
  extern __shared__ __align__(16) uint4 wsm[];  // [EP][D / N] 16-byte vectors
  __shared__ float skey[kSelWarps][256 + 8];
  __shared__ uint64_t wbar;
  __shared__ int abort_flag;
  constexpr int N = Vec16<T>::N;
  constexpr int U = EP <= 8 ? 8 : 4;  // vectors a lane loads per batch; two batches in flight
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kSelWarps + warp;
  const bool active = t < a.T;
  const int E = a.E;
  const int nvec = D / N;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&wbar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t bytes = static_cast<uint32_t>(E) * nvec * 16u;
    mbar_arrive_expect_tx(&wbar, bytes);
    bulk_load_g2s(wsm, w, bytes, &wbar);
  }
  const uint4* xr = reinterpret_cast<const uint4*>(x + (active ? t : 0) * D);
  uint4 xv[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int v = lane + 32 * u;
    xv[u] = active && v < nvec ? ld_nc_v4(xr + v) : make_uint4(0u, 0u, 0u, 0u);
  }
  for (int i = E * nvec + threadIdx.x; i < EP * nvec; i += kSelWarps * 32)
    wsm[i] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  if (!mbar_wait(&wbar, 0, &abort_flag, kWaitLimitNs)) {
    if (threadIdx.x == 0) set_status(a.status, MOE_ERR_TIMEOUT);
    return;
  }
  if (!active) return;
  float acc[EP];
#pragma unroll
  for (int e = 0; e < EP; ++e) acc[e] = 0.0f;
  for (int v0 = lane; v0 < nvec; v0 += 32 * U) {
    uint4 cur[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      cur[u] = xv[u];
      const int v = v0 + 32 * (U + u);
      xv[u] = v < nvec ? ld_nc_v4(xr + v) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + 32 * u;
      if (v < nvec) {
        float xf[N];
        Vec16<T>::to_f32(cur[u], xf);
#pragma unroll
        for (int e = 0; e < EP; ++e) {
          float wf[N];
          Vec16<T>::to_f32(wsm[e * nvec + v], wf);
#pragma unroll
          for (int i = 0; i < N; ++i) acc[e] = fmaf(xf[i], wf[i], acc[e]);
        }
      }
    }
  }
  float lg[1] = {0.0f};
#pragma unroll
  for (int e = 0; e < EP; ++e) {
    float s = acc[e];
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) s += __shfl_xor_sync(0xffffffffu, s, d);
    if (lane == e) lg[0] = s;
  }
  select_token<1>(a, t, lane, lg, skey[warp]);
}

// The bf16 router for up to 32 experts in one kernel, on the warp-level MMA.
// A block takes tb tokens (16, or fewer when 16 would leave SMs without a
// block; the MMA tile's other rows load nothing) and its 16 warps split D
// between them; each warp accumulates a 16-token x EP-expert tile with
// m16n8k16 MMAs in two chains (even and odd chunks), operands straight from
// global memory into registers, one batch of loads per warp at D = 4096.  A dot product may take
// its D terms in any order, so lane (g, t) loads the 16 bytes at elements
// 8t..8t+7 of each 32-element chunk of token rows g and g + 8 and of expert
// row g, and hands elements 8t..8t+3 to one MMA and 8t+4..8t+7 to a second
// as their K pairs (2t, 2t+1) and (2t+8, 2t+9).  A and B see the same
// permutation of K, every load is 16 bytes, and the four lanes of a row read
// 64 contiguous bytes.  W_r is read once per block (from L2) instead of once
// per token from shared memory.  The warps' partial tiles are added in warp
// order, so a token's logits do not depend on the batch it is in; warp w then
// runs the selection for token w.
constexpr int kMmaRouteTok = 16;
constexpr int kMmaRouteWarps = 16;
constexpr int kMmaRouteKey = 64;   // per-warp selection scratch (E <= 32)
static_assert(kMmaRouteTok == kMmaRouteWarps, "warp w selects token w");

template <int EP>
__global__ void __launch_bounds__(kMmaRouteWarps * 32, 1)
    route_mma_kernel(RouteSelectArgs a, const __nv_bfloat16* __restrict__ x,
                     const __nv_bfloat16* __restrict__ w, int D, int tb) {
  constexpr int NB = EP / 8;            // n tiles of 8 experts
  constexpr int U = 24 / (2 + NB);      // chunks in flight: 96 registers of loads
  __shared__ float part[kMmaRouteWarps][kMmaRouteTok][EP];
  __shared__ float skey[kMmaRouteWarps][kMmaRouteKey];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int q = lane & 3;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * tb;
  const int E = a.E;
  const int nch = (D + 31) / 32;
  const int per = (nch + kMmaRouteWarps - 1) / kMmaRouteWarps;
  const int c_begin = warp * per;
  const int c_end = min(nch, c_begin + per);
  const bool lo_ok = g < tb && t0 + g < a.T;
  const bool hi_ok = g + 8 < tb && t0 + g + 8 < a.T;
  const __nv_bfloat16* xlo = x + (lo_ok ? t0 + g : 0) * D + 8 * q;
  const __nv_bfloat16* xhi = x + (hi_ok ? t0 + g + 8 : 0) * D + 8 * q;
  const __nv_bfloat16* wr[NB];
  bool w_ok[NB];
#pragma unroll
  for (int j = 0; j < NB; ++j) {
    w_ok[j] = 8 * j + g < E;
    wr[j] = w + static_cast<int64_t>(w_ok[j] ? 8 * j + g : 0) * D + 8 * q;
  }
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  float acc[2][NB][4];   // even and odd chunks: two MMA chains
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int j = 0; j < NB; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[h][j][i] = 0.0f;

  for (int c0 = c_begin; c0 < c_end; c0 += U) {
    uint4 ra[U][2], rb[U][NB];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u;
      const bool ok = c < c_end && 32 * c + 8 * q < D;
      ra[u][0] = ok && lo_ok ? ld_nc_v4(xlo + 32 * c) : zero;
      ra[u][1] = ok && hi_ok ? ld_nc_v4(xhi + 32 * c) : zero;
#pragma unroll
      for (int j = 0; j < NB; ++j)
        rb[u][j] = ok && w_ok[j]
                       ? __ldg(reinterpret_cast<const uint4*>(wr[j] + 32 * c))
                       : zero;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (c0 + u < c_end) {   // warp-uniform
#pragma unroll
        for (int j = 0; j < NB; ++j) {
          mma_m16n8k16_bf16(acc[u & 1][j], ra[u][0].x, ra[u][1].x,
                            ra[u][0].y, ra[u][1].y, rb[u][j].x, rb[u][j].y);
          mma_m16n8k16_bf16(acc[u & 1][j], ra[u][0].z, ra[u][1].z,
                            ra[u][0].w, ra[u][1].w, rb[u][j].z, rb[u][j].w);
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < NB; ++j) {
    const int e = 8 * j + 2 * q;
    part[warp][g][e] = __fadd_rn(acc[0][j][0], acc[1][j][0]);
    part[warp][g][e + 1] = __fadd_rn(acc[0][j][1], acc[1][j][1]);
    part[warp][g + 8][e] = __fadd_rn(acc[0][j][2], acc[1][j][2]);
    part[warp][g + 8][e + 1] = __fadd_rn(acc[0][j][3], acc[1][j][3]);
  }
  __syncthreads();
  const int64_t t = t0 + warp;
  if (warp >= tb || t >= a.T) return;
  float lg[1] = {0.0f};
  if (lane < EP) {
#pragma unroll
    for (int v = 0; v < kMmaRouteWarps; ++v)
      lg[0] = __fadd_rn(lg[0], part[v][warp][lane]);
  }
  select_token<1>(a, t, lane, lg, skey[warp]);
}

// fp32 router GEMM on the FMA pipes: one thread per (token, expert).
__global__ void route_gemm_f32_kernel(int T, int D, int E, const float* x,
                                      const float* w, float* logits) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<int64_t>(T) * E) return;
  const int64_t t = i / E;
  const int e = static_cast<int>(i - t * E);
  const float* xr = x + t * D;
  const float* wr = w + static_cast<int64_t>(e) * D;
  float acc = 0.0f;
  for (int d = 0; d < D; ++d) acc = fmaf(xr[d], wr[d], acc);
  logits[i] = acc;
}

__global__ void sigmoid_key_kernel(const float* l, float* out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = sigmoid_score(l[i]);
}

moe_status launch_sigmoid_key(const float* l, float* out, int n,
                              cudaStream_t stream) {
  if (n == 0) return MOE_OK;
  sigmoid_key_kernel<<<static_cast<unsigned>(ceil_div(n, 256)), 256, 0,
                       stream>>>(l, out, n);
  return launch_status();
}

// ------------------------------------------------------------------ host
RoutePlan plan_route(const moe_route_cfg& c, int num_sms) {
  RoutePlan p{};
  p.Npad = ((c.E + 15) / 16) * 16;
  p.k_blocks = static_cast<int>(ceil_div(c.D, kBK));
  const int m_tiles = static_cast<int>(ceil_div(c.T, kBM));
  int splits = 1;
  if (c.dtype == MOE_BF16) {
    // enough (m block, K split) tiles to cover the SMs, >= 4 K blocks each
    splits = num_sms / (m_tiles > 0 ? m_tiles : 1);
    splits = splits < 1 ? 1 : splits;
    // with more row blocks than SMs, two K halves when they even out the
    // last round by at least half a tile (512 blocks on 148 SMs: 3.5
    // tile-times instead of 4)
    if (m_tiles >= num_sms) {
      const int64_t whole = ceil_div(m_tiles, num_sms);
      const int64_t halves = ceil_div(2 * static_cast<int64_t>(m_tiles), num_sms);
      if (halves <= 2 * whole - 1) splits = 2;
    }
    const int max_splits = p.k_blocks / 4 > 0 ? p.k_blocks / 4 : 1;
    splits = splits > max_splits ? max_splits : splits;
  }
  p.kb_per_split = static_cast<int>(ceil_div(p.k_blocks, splits));
  p.splits = static_cast<int>(ceil_div(p.k_blocks, p.kb_per_split));
  if (c.dtype != MOE_BF16) p.splits = 1;
  p.ws_bytes = static_cast<size_t>(p.splits) * c.T * c.E * sizeof(float);
  return p;
}

// Up to 32 experts the router can be one kernel.  In bf16 that is the MMA
// kernel, which reads its operands straight from global memory: every block
// reads all of W_r (EP/16 times its tile's x bytes, from L2), so it is taken
// for up to 8 experts, for W_r of at most 96 KiB, or while the tokens fill at
// most one 16-token tile per SM; beyond that the split-K GEMM, which reads
// W_r once per 128-token tile, is faster (T = 16384, 32 experts, D = 4096:
// 47 against 57 us).  In fp32 it is the warp-per-token kernel on the FMA
// pipes when W_r fits in shared memory.  Otherwise the router GEMM (tensor
// cores in bf16), then the select kernel.
constexpr int kWarpRouteSmem = 96 * 1024;
static int route_ep(int E) { return E <= 8 ? 8 : E <= 16 ? 16 : 32; }
// The router GEMM selects in its epilogue (no partial logits, no select
// launch) when one thread can do a token's whole selection from registers:
// bf16, one K split, a softmax score without groups, k <= 2 and E <= 64.
bool route_fused_gemm(const moe_route_cfg& c, int num_sms) {
  if (route_single_kernel(c, num_sms) || c.dtype != MOE_BF16) return false;
  if (c.score == MOE_SCORE_SIGMOID_BIAS || c.n_groups != 1 || c.k > 2 ||
      c.E > kRouteSelMaxE)
    return false;
  return plan_route(c, num_sms).splits == 1;
}

bool route_single_kernel(const moe_route_cfg& c, int num_sms) {
  if (c.E > 32) return false;
  const bool small_w = static_cast<int64_t>(route_ep(c.E)) * c.D *
                           dtype_bytes(c.dtype) <= kWarpRouteSmem;
  if (c.dtype != MOE_BF16) return small_w;
  return c.E <= 8 || small_w ||
         static_cast<int64_t>(c.T) <= static_cast<int64_t>(kMmaRouteTok) * num_sms;
}

template <typename T, int EP>
static bool launch_route_warp_ep(const RouteSelectArgs& s, const T* x,
                                 const T* w, int D, cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done{0};
  if (!set_smem_limit_once(
          reinterpret_cast<const void*>(route_warp_kernel<T, EP>),
          kWarpRouteSmem, &attr_done))
    return false;
  const unsigned grid = static_cast<unsigned>(ceil_div(s.T, kSelWarps));
  const size_t smem = static_cast<size_t>(EP) * D * sizeof(T);
  route_warp_kernel<T, EP><<<grid, kSelWarps * 32, smem, stream>>>(s, x, w, D);
  return true;
}

// Tokens per block: 16, or fewer when that leaves SMs without a block (the
// MMA tile's remaining rows load nothing).
static int route_mma_tokens(int T, int num_sms) {
  const int64_t per = ceil_div(T, num_sms > 0 ? num_sms : 1);
  return per >= kMmaRouteTok ? kMmaRouteTok : per < 1 ? 1 : static_cast<int>(per);
}

template <int EP>
static void launch_route_mma_ep(const RouteSelectArgs& s,
                                const __nv_bfloat16* x,
                                const __nv_bfloat16* w, int D, int num_sms,
                                cudaStream_t stream) {
  const int tb = route_mma_tokens(s.T, num_sms);
  const unsigned grid = static_cast<unsigned>(ceil_div(s.T, tb));
  route_mma_kernel<EP><<<grid, kMmaRouteWarps * 32, 0, stream>>>(s, x, w, D, tb);
}

static bool launch_route_warp(const RouteSelectArgs& s, int32_t dtype,
                              const void* x, const void* w_r, int D,
                              int num_sms, cudaStream_t stream) {
  if (dtype == MOE_BF16) {
    const auto* xx = static_cast<const __nv_bfloat16*>(x);
    const auto* ww = static_cast<const __nv_bfloat16*>(w_r);
    if (s.E <= 8) launch_route_mma_ep<8>(s, xx, ww, D, num_sms, stream);
    else if (s.E <= 16) launch_route_mma_ep<16>(s, xx, ww, D, num_sms, stream);
    else launch_route_mma_ep<32>(s, xx, ww, D, num_sms, stream);
    return true;
  }
  const auto* xx = static_cast<const float*>(x);
  const auto* ww = static_cast<const float*>(w_r);
  if (s.E <= 8) return launch_route_warp_ep<float, 8>(s, xx, ww, D, stream);
  if (s.E <= 16) return launch_route_warp_ep<float, 16>(s, xx, ww, D, stream);
  return launch_route_warp_ep<float, 32>(s, xx, ww, D, stream);
}

moe_status launch_route(const moe_route_cfg& c, const void* x, const void* w_r,
                        const float* logit_offset, const float* sel_bias,
                        int32_t* topk_idx, float* topk_gate, float* logits_out,
                        void* ws, int32_t* status, cudaStream_t stream,
                        int num_sms) {
  if (route_single_kernel(c, num_sms)) {
    RouteSelectArgs s{};
    s.T = c.T;
    s.E = c.E;
    s.k = c.k;
    s.score = c.score;
    s.n_groups = c.n_groups;
    s.topk_groups = c.topk_groups;
    s.group_score_topk = c.group_score_topk;
    s.splits = 1;
    s.logit_offset = logit_offset;
    s.sel_bias = sel_bias;
    s.topk_idx = topk_idx;
    s.topk_gate = topk_gate;
    s.logits_out = logits_out;
    s.status = status;
    if (!launch_route_warp(s, c.dtype, x, w_r, c.D, num_sms, stream))
      return MOE_ERR_CUDA;
    return launch_status();
  }
  const RoutePlan p = plan_route(c, num_sms);
  float* partial = static_cast<float*>(ws);
  if (c.dtype == MOE_BF16) {
    CUtensorMap tmA, tmB;
    if (!make_tmap_bf16_2d(&tmA, x, c.D, c.T, kBM) ||
        !make_tmap_bf16_2d(&tmB, w_r, c.D, c.E, p.Npad))
      return MOE_ERR_CUDA;
    GemmArgs g{};
    g.M = c.T;
    g.k_blocks = p.k_blocks;
    g.BN = p.Npad;
    const size_t stage_bytes = kATileBytes + static_cast<size_t>(p.Npad) * kBK * 2;
    int stages = static_cast<int>((200 * 1024) / stage_bytes);
    g.stages = stages > kMaxStages ? kMaxStages : stages;
    int cols = 32;
    while (cols < 2 * p.Npad) cols <<= 1;
    g.tmem_cols = cols;
    g.splits = p.splits;
    g.kb_per_split = p.kb_per_split;
    g.E = c.E;
    g.out = partial;
    g.out_ld = c.E;
    g.out_cols = c.E;
    g.status = status;
    g.wait_limit_ns = kWaitLimitNs;
    const bool fused = route_fused_gemm(c, num_sms);
    if (fused) {
      g.sel_idx = topk_idx;
      g.sel_gate = topk_gate;
      g.sel_logits = logits_out;
      g.sel_offset = logit_offset;
      g.sel_k = c.k;
      g.sel_full = c.score == MOE_SCORE_SOFTMAX_FULL ? 1 : 0;
    }
    const size_t smem = umma_gemm_smem_bytes(g.BN, g.stages);
    // the kernel's static shared memory (the epilogue selection's exchange
    // slots, 6 KB) comes out of the same 227 KB as the dynamic part
    static std::atomic<uint64_t> attr_done{0};
    if (!set_smem_limit_once(
            reinterpret_cast<const void*>(umma_gemm_kernel<kRoute>),
            (227 - 8) * 1024, &attr_done))
      return MOE_ERR_CUDA;
    const int tiles = static_cast<int>(ceil_div(c.T, kBM)) * p.splits;
    const int grid = tiles < num_sms ? tiles : num_sms;
    umma_gemm_kernel<kRoute><<<grid, kGemmThreads, smem, stream>>>(tmA, tmB, g);
    if (fused) return launch_status();
  } else {
    const int64_t n = static_cast<int64_t>(c.T) * c.E;
    route_gemm_f32_kernel<<<static_cast<unsigned>(ceil_div(n, 256)), 256, 0,
                            stream>>>(c.T, c.D, c.E,
                                      static_cast<const float*>(x),
                                      static_cast<const float*>(w_r), partial);
  }
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;

  RouteSelectArgs s{};
  s.T = c.T;
  s.E = c.E;
  s.k = c.k;
  s.score = c.score;
  s.n_groups = c.n_groups;
  s.topk_groups = c.topk_groups;
  s.group_score_topk = c.group_score_topk;
  s.splits = p.splits;
  s.partial = partial;
  s.logit_offset = logit_offset;
  s.sel_bias = sel_bias;
  s.topk_idx = topk_idx;
  s.topk_gate = topk_gate;
  s.logits_out = logits_out;
  const int warps = kSelWarps;
  // four blocks per SM stay resident; past that the warps stride
  const unsigned grid = static_cast<unsigned>(ceil_div(c.T, warps));
  const int ni = static_cast<int>(ceil_div(c.E, 32));
  if (ni <= 1)
    route_select_kernel<1><<<grid, warps * 32, 0, stream>>>(s);
  else if (ni <= 2)
    route_select_kernel<2><<<grid, warps * 32, 0, stream>>>(s);
  else if (ni <= 4)
    route_select_kernel<4><<<grid, warps * 32, 0, stream>>>(s);
  else
    route_select_kernel<8><<<grid, warps * 32, 0, stream>>>(s);
  return launch_status();
}

}  // namespace moe
