// Sampling arithmetic of spec_verify: the weight of one vocabulary element
// at the sampled position, as the tile sweep and the locate step of the
// draw kernel (sv_draw.cuh) both compute it, and the fold of tile
// partials into a row's argmax that the tree verification uses.
//
// The rule is the exact rejection rule of the lesson "Decodificação
// Especulativa e EAGLE" (ai-engineering.academy, phase 10 lesson 25),
// sections "A Regra de Exatidão" and "Caso ganancioso"; the residual
// (p - q)+ / ||(p - q)+||_1 is taken over the full vocabulary as the same
// section states it.
#pragma once

#include "sv_plug.cuh"
#include "sv_stream.cuh"

namespace sv {

// A term whose probability exceeds about this is evaluated in
// double-float during sampling; smaller terms use the float32 path.  The
// test is made on the logit itself (x >= a per-row threshold), so the
// sweep and the locate step classify every element alike.
constexpr float kBigProb = 1.0e-4f;

// device flags (mirrors of the public SV_DEV_* values)
constexpr unsigned kDevBadTemperature = 1u;
constexpr unsigned kDevBadToken = 2u;
constexpr unsigned kDevNonFinite = 4u;
constexpr unsigned kDevBadK = 8u;

// Everything the weighing of the sampled position needs.
struct SampleCtx {
  const char* rowP;       // target row at the sampled position
  const char* rowQ;       // draft row there (nullptr for a bonus draw)
  int V;
  float MCp, MCq;         // shifts (c-scaled) of the two rows
  float c_hi, c_lo;       // log2(e)/T as hi + lo
  float cw;               // c_used = S_p / S_q at the streaming pass's shifts
  float tp, tq;           // large-term thresholds on the logits xp, xq
  DF L;                   // log2(e)/T as a double-float (= c_hi + c_lo)
};

// e = 2^(x * L - MC) for the float32 path: the product and the shift are
// formed exactly by the FMA and rounded once, plus the low part of L.
// c_lo > 0 (see SampleCtx), so x = -inf gives -inf, not inf - inf.
__device__ __forceinline__ float small_exp(float x, float MC, const SampleCtx& s) {
  return ex2_approx(__fmaf_rn(x, s.c_lo, __fmaf_rn(x, s.c_hi, -MC)));
}
// the same value in double-float: 2^(x*L - MC) with x*L exact (two-product)
__device__ __forceinline__ DF big_exp(float x, float MC, const SampleCtx& s, const float2* tab) {
  const float ph = __fmul_rn(x, s.L.hi);
  float pl = __fmaf_rn(x, s.L.hi, -ph);
  pl = __fmaf_rn(x, s.L.lo, pl);
  const DF y = df_add(DF{ph, pl}, DF{-MC, 0.f});
  return exp2_df(y.hi, y.lo, tab);
}

// Weight of element xp (and xq) as the sweep counts it.  kResidual:
// w = max(e^p - cw e^q, 0) with the e^q that goes with a positive w;
// otherwise w = e^p.  Large terms in double-float, the rest in float32.
template <bool kResidual>
__device__ __forceinline__ void eval_pair(float xp, float xq, const SampleCtx& s, const float2* tab,
                                          DF& w, DF& q) {
  const float ep = small_exp(xp, s.MCp, s);
  if (kResidual) {
    const float eq = small_exp(xq, s.MCq, s);
    if (xp >= s.tp || xq >= s.tq) {
      const DF epd = big_exp(xp, s.MCp, s, tab);
      const DF eqd = big_exp(xq, s.MCq, s, tab);
      const DF d = df_sub(epd, df_mul_f(eqd, s.cw));
      w = df_pos(d) ? d : DF{0.f, 0.f};
      q = df_pos(d) ? eqd : DF{0.f, 0.f};
    } else {
      const float d = __fmaf_rn(-s.cw, eq, ep);
      w = DF{d > 0.f ? d : 0.f, 0.f};
      q = DF{d > 0.f ? eq : 0.f, 0.f};
    }
  } else {
    w = (xp >= s.tp) ? big_exp(xp, s.MCp, s, tab) : DF{ep, 0.f};
    q = DF{0.f, 0.f};
  }
}

// Double-float weight of one large term with logits xp (and xq): w (and
// the q that goes with a positive w), plus e^p and e^q for the row totals.
template <bool kResidual>
__device__ __forceinline__ void big_term(const SampleCtx& x, const float2* tab, float xp, float xq,
                                         DF& w, DF& q, DF& ep, DF& eq) {
  ep = big_exp(xp, x.MCp, x, tab);
  w = ep;
  q = DF{0.f, 0.f};
  eq = DF{0.f, 0.f};
  if (kResidual) {
    eq = big_exp(xq, x.MCq, x, tab);
    const DF d = df_sub(ep, df_mul_f(eq, x.cw));
    w = df_pos(d) ? d : DF{0.f, 0.f};
    q = df_pos(d) ? eq : DF{0.f, 0.f};
  }
}

// Reductions over aligned groups of kLanes lanes (kLanes = 16 or 32); every
// lane of the warp takes part, each group reduces on its own.
template <int kLanes>
__device__ __forceinline__ float grp_max(float v) {
#pragma unroll
  for (int o = kLanes / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
template <int kLanes>
__device__ __forceinline__ float grp_sum(float v) {
#pragma unroll
  for (int o = kLanes / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
template <int kLanes>
__device__ __forceinline__ int grp_min_int(int v) {
#pragma unroll
  for (int o = kLanes / 2; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// A group of kLanes lanes (lane = index in the group) folds the tpr tile
// partials of one row: (MC, S) for a tempered row, (max logit, lowest index
// holding it as int bits) for a greedy row (whose partials hold the
// complemented index).  Every lane of the group returns the result.  With
// pp == nullptr the group folds nothing and returns the neutral values (it
// still takes part in the shuffles).
template <int kLanes>
__device__ __forceinline__ float2 fold_partials(const float2* pp, int tpr, bool greedy, int lane) {
  constexpr int kPer = 8;   // partials in flight per lane
  const int n = pp ? tpr : 0;
  if (greedy) {
    float best = SV_NEG_INF;
    int bi = 0x7fffffff;
    for (int base = 0; base < n; base += kLanes * kPer) {
      float2 v[kPer];
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int i = base + lane + kLanes * j;
        v[j] = i < n ? __ldcg(pp + i) : make_float2(SV_NEG_INF, __int_as_float(~0x7fffffff));
      }
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int idx = ~__float_as_int(v[j].y);
        if (v[j].x > best || (v[j].x == best && idx < bi)) {
          best = v[j].x;
          bi = idx;
        }
      }
    }
    const float m = grp_max<kLanes>(best);
    const int idx = grp_min_int<kLanes>(best == m ? bi : 0x7fffffff);
    return make_float2(m, __int_as_float(idx));
  }
  // loads first (independent), then the online fold
  float mc = SV_NEG_INF, s = 0.f;
  for (int base = 0; base < n; base += kLanes * kPer) {
    float2 v[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int i = base + lane + kLanes * j;
      v[j] = i < n ? __ldcg(pp + i) : make_float2(SV_NEG_INF, 0.f);
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      if (v[j].x == SV_NEG_INF) continue;
      if (v[j].x > mc) {
        s = s * ex2_approx(__fsub_rn(mc, v[j].x)) + v[j].y;
        mc = v[j].x;
      } else {
        s += v[j].y * ex2_approx(__fsub_rn(v[j].x, mc));
      }
    }
  }
  const float M = grp_max<kLanes>(mc);
  float sv = (mc == SV_NEG_INF) ? 0.f : s * ex2_approx(__fsub_rn(mc, M));
  sv = grp_sum<kLanes>(sv);
  return make_float2(M, sv);
}

}  // namespace sv
