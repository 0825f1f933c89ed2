// The acceptance and draw kernel of spec_verify (the launch after the
// streaming pass).
//
// The rule is the exact rejection rule of the lesson "Decodificação
// Especulativa e EAGLE" (ai-engineering.academy, phase 10 lesson 25),
// sections "A Regra de Exatidão" (test r q < p; replacement from the
// residual (p - q)+ / ||(p - q)+||_1 over the full vocabulary; bonus token
// from p_K) and "Caso ganancioso" (T = 0: argmax).
//
// G CTAs serve each batch row b (G = parts, chosen by the host so the grid
// fills the GPU).  Every one of them
//   1. reads the row's caller inputs -- drafted tokens, draws, the logits at
//      the drafted tokens -- before it waits for the streaming pass;
//   2. folds the streaming pass's tile partials of the row's positions into
//      (shift, sum) or (max, lowest argmax), one half-warp per position;
//   3. runs the left-to-right acceptance scan (one lane per position) --
//      all G CTAs reach the same n, and part 0 writes the outputs;
//   4. weighs its part of the sampled position's tiles -- w = max(p - q, 0)
//      at a rejection, w = p for the bonus -- one warp per tile, writing
//      one record per tile (totals of w, of the e^q under positive w, of
//      e^p and of e^q, as double-floats);
//   5. takes a ticket on the row; the CTA holding the last one locates the
//      token: the tile by a warp scan over the row's tile records (staged
//      in shared memory), the element by a block-wide scan of that tile,
//      re-read.
// Greedy rows (T = 0) and error rows are finished by part 0 in step 3.
// No CTA waits on another: the ticket is one atomic per CTA.
//
// Small terms are weighed in float32, terms whose probability exceeds
// kBigProb in double-float; the exact c = S_p / S_q (from the double-float
// totals) corrects the residual weights to first order from the c of the
// streaming pass's float32 sums.  The locate step weighs elements with the
// same rule as the sweep, so its sums agree with the records up to
// rounding; where rounding leaves u*W at or past a total, the last
// positive element is taken.
#pragma once

#include "sv_sample.cuh"

namespace sv {

constexpr int kDThreads = 256;
constexpr int kDWarps = kDThreads / 32;
constexpr int kMaxParts = 64;
constexpr int kDBigCap = 64;   // large terms listed per warp per tile (more: evaluated by their own lane)

struct DrawArgs {
  const void* target;
  const void* draft;
  const int32_t* tokens;
  const float* uniforms;
  const float* temperature;
  const int32_t* k_per_row;   // [B] or nullptr (every row verifies K)
  int B, K, V;
  int tpr;                    // 2 KB tiles per row
  int n_target_rows;          // B*(K+1)
  int parts;                  // G: CTAs per batch row, 1..kMaxParts
  const float2* partials;     // [B*(K+1) + B*K][tpr] from the streaming pass
  unsigned* err;
  unsigned* tickets;          // [B], zero on entry (the streaming pass clears them)
  float4* tile_recs;          // [B][tpr][2]: (W, Q), (P, S) as double-floats
  int32_t* accepted_len;
  int32_t* out_tokens;
  float* logp_out;
  float* logq_out;
  int32_t* plug_tokens;       // plug step fused in (nullptr: none)
  int32_t* plug_seq_len;
  int32_t* plug_last;
  int plug_max_len;
};

struct DrawSmem {
  float2 tab[256];
  uint32_t bigpos[kDWarps][kDBigCap];
  uint4 stage[kDWarps][2][kTileVecs];   // a warp's tile of each row, for its large terms
  float rowMC[2 * kMaxK + 1];
  float rowS[2 * kMaxK + 1];
  int rowArg[kMaxK + 1];
  int tok[kMaxK];
  float r[kMaxK + 1];
  float xp[kMaxK];
  float xq[kMaxK];
  int bad, n, kb, last;
  DF wsum[kDWarps];
  struct {
    int jstar, mode, last_mode, pick, lastpos, token;
    unsigned long long best;
    DF tg, dc;
  } loc;
};

__device__ __forceinline__ void dflag(const DrawArgs& a, unsigned f) { atomicOr(a.err, f); }

// Checked build: an index test guarding one access (always true, and
// compiled away, in the plain build).
__device__ __forceinline__ bool in_bounds(const DrawArgs& a, bool ok) {
  if (kChecked && !ok) {
    dflag(a, kDevOutOfBounds);
    return false;
  }
  return true;
}

// ---------------------------------------------------------------- steps 1-3
// Caller inputs of batch row b (warp 0): tokens, draws, the 2 K_b logits at
// the drafted tokens, and the row's validity.
template <typename E>
__device__ void draw_inputs(const DrawArgs& a, int b, float T, DrawSmem& sm) {
  const int K = a.K, lane = threadIdx.x & 31;
  const bool greedy = (T == 0.f);
  const long long ob = (long long)b * (K + 1);
  if ((threadIdx.x >> 5) == 0) {
    const int kb_in = a.k_per_row ? __ldg(a.k_per_row + b) : K;
    const bool k_ok = kb_in >= 0 && kb_in <= K;
    const int kb = k_ok ? kb_in : 0;
    int x = 0;
    bool tok_ok = true;
    if (lane < kb) {
      x = __ldg(a.tokens + (long long)b * K + lane);
      tok_ok = x >= 0 && x < a.V;
      sm.tok[lane] = x;
    }
    // r_0..r_{kb-1}, then u in column kb
    if (lane <= kb && !greedy) sm.r[lane] = __ldg(a.uniforms + ob + lane);
    const bool all_ok = __all_sync(0xffffffffu, tok_ok);
    if (lane == 0) {
      sm.kb = kb;
      sm.bad = !valid_temperature(T) ? (int)kDevBadTemperature
               : !k_ok                ? (int)kDevBadK
               : all_ok               ? 0
                                      : (int)kDevBadToken;
    }
    if (all_ok && k_ok && !greedy && valid_temperature(T) && lane < kb) {
      sm.xp[lane] = E::load_scalar(a.target, (ob + lane) * (long long)a.V + x);
      sm.xq[lane] = E::load_scalar(a.draft, ((long long)b * K + lane) * (long long)a.V + x);
    }
  }
  for (int i = threadIdx.x; i < 256; i += kDThreads) sm.tab[i] = kExp2Table256[i];
}

// Fold the tile partials of the row's positions, one half-warp per position
// (16 per round): target rows 0..K_b, draft rows 0..K_b-1 of tempered rows.
__device__ void fold_stats(const DrawArgs& a, int b, bool greedy, DrawSmem& sm) {
  constexpr int kHalves = kDThreads / 16;
  const int K = a.K, kb = sm.kb, hl = threadIdx.x & 15, hw = threadIdx.x >> 4;
  const long long tb = (long long)b * (K + 1);
  const long long db = a.n_target_rows + (long long)b * K;
  const int nrows = greedy ? K + 1 : 2 * K + 1;
  for (int base = 0; base < nrows; base += kHalves) {   // the same trip count in every warp
    const int rr = base + hw;
    const float2* pp = nullptr;
    if (rr < nrows && (rr <= K ? rr <= kb : rr - K - 1 < kb)) {
      const long long prow = (rr <= K) ? tb + rr : db + (rr - K - 1);
      if (in_bounds(a, prow < a.n_target_rows + (long long)a.B * K)) pp = a.partials + prow * a.tpr;
    }
    const float2 st = fold_partials<16>(pp, a.tpr, greedy, hl);
    if (pp && hl == 0) {
      sm.rowMC[rr] = st.x;
      if (greedy) sm.rowArg[rr] = __float_as_int(st.y);
      else sm.rowS[rr] = st.y;
    }
  }
}

// Acceptance scan (warp 0): one lane per drafted position; sets sm.n and
// sm.bad.  With `write` (part 0), also writes accepted_len, the
// log-probabilities and every out_tokens slot except the one a tempered row
// still has to draw.
template <bool kPlug>
__device__ void draw_scan(const DrawArgs& a, int b, float T, bool write, DrawSmem& sm) {
  const int K = a.K, lane = threadIdx.x & 31;
  if ((threadIdx.x >> 5) != 0) return;
  const bool greedy = (T == 0.f);
  const long long ob = (long long)b * (K + 1);
  const int nrows = greedy ? K + 1 : 2 * K + 1;
  const int kb = sm.kb;
  const float c = greedy ? 0.f : log2e_over_f(T);
  int bad = sm.bad;
  bool row_ok = true;
  for (int rr = lane; !bad && rr < nrows; rr += 32) {
    if (rr <= K ? rr > kb : rr - K - 1 >= kb) continue;   // a row this K_b does not verify
    const float M = sm.rowMC[rr];
    row_ok = row_ok && isfinite(M) && (greedy || (isfinite(sm.rowS[rr]) && sm.rowS[rr] > 0.f));
  }
  if (!bad && !__all_sync(0xffffffffu, row_ok)) bad = (int)kDevNonFinite;
  int n = kb;
  float lp = __int_as_float(0x7fffffff), lq = lp;
  if (!bad) {
    bool reject = false;
    if (greedy) {
      reject = lane < kb && sm.rowArg[lane] != sm.tok[lane];
    } else if (lane < kb) {
      // log p_t(x_t) = (x c - MC) ln 2 - ln S, with x c - MC formed exactly by the FMA
      constexpr float kLn2 = 0.693147180559945309f;
      lp = __fmaf_rn(sm.xp[lane], c, -sm.rowMC[lane]) * kLn2 - logf(sm.rowS[lane]);
      lq = __fmaf_rn(sm.xq[lane], c, -sm.rowMC[K + 1 + lane]) * kLn2 - logf(sm.rowS[K + 1 + lane]);
      // r q < p  <=>  r < p / q = exp(log p - log q)
      reject = !(sm.r[lane] < expf(lp - lq));
    }
    const unsigned rej = __ballot_sync(0xffffffffu, reject);
    n = rej ? __ffs(rej) - 1 : kb;
  }
  if (write) {
    if (lane < K) {
      if (a.logp_out) a.logp_out[(long long)b * K + lane] = bad || greedy ? __int_as_float(0x7fffffff) : lp;
      if (a.logq_out) a.logq_out[(long long)b * K + lane] = bad || greedy ? __int_as_float(0x7fffffff) : lq;
    }
    int v = -1;
    if (!bad && lane <= K) {
      if (lane < n) v = sm.tok[lane];
      else if (lane == n && greedy) v = sm.rowArg[n];
    }
    if (lane <= K && !(lane == n && !greedy && !bad)) a.out_tokens[ob + lane] = v;
    if (lane == 0) {
      a.accepted_len[b] = bad ? -1 : n;
      if (bad) dflag(a, (unsigned)bad);
    }
    // a greedy row's tokens are all known here (an error row is never plugged)
    if (kPlug && greedy && !bad)
      plug_row(lane, n, v, a.plug_tokens + (long long)b * a.plug_max_len, a.plug_seq_len + b,
               a.plug_max_len, a.plug_last ? a.plug_last + b : nullptr, a.err);
  }
  if (lane == 0) {
    sm.n = n;
    sm.bad = bad;
  }
}

// What weighing position n of batch row b needs (residual: n < K_b).
template <typename E>
__device__ __forceinline__ SampleCtx make_ctx(const DrawArgs& a, int b, int n, bool residual,
                                              float MCp, float Sp32, float MCq, float Sq32, float T) {
  const int K = a.K;
  const long long rowbytes = (long long)a.V * E::kBytes;
  SampleCtx x;
  x.rowP = (const char*)a.target + ((long long)b * (K + 1) + n) * rowbytes;
  x.rowQ = residual ? (const char*)a.draft + ((long long)b * K + n) * rowbytes : nullptr;
  x.V = a.V;
  x.MCp = MCp;
  x.MCq = residual ? MCq : 0.f;
  if (!residual) Sq32 = 1.f;
  x.L = log2e_over(T);
  x.c_hi = x.L.hi;
  x.c_lo = x.L.lo;
  if (!(x.c_lo > 0.f)) {   // a strictly positive low part (see small_exp)
    x.c_hi = __uint_as_float(__float_as_uint(x.L.hi) - 1u);
    x.c_lo = __fadd_rn(__fsub_rn(x.L.hi, x.c_hi), x.L.lo);
  }
  x.cw = __fdiv_rn(Sp32, Sq32);
  // large terms: e^p above about kBigProb S_p, i.e. x c - MC > log2(kBigProb S),
  // tested on the logit (rounded to the storage type, so that a packed
  // bf16 compare gives the same answer as a float32 one)
  const float c = log2e_over_f(T);
  x.tp = E::round_logit(__fdiv_rn(__fadd_rn(MCp, __log2f(kBigProb * Sp32)), c));
  x.tq = residual ? E::round_logit(__fdiv_rn(__fadd_rn(MCq, __log2f(kBigProb * Sq32)), c))
                  : __int_as_float(0x7f800000);
  return x;
}

// ---------------------------------------------------------------- step 4
// Element (vector j, element k) of lane `lane` as a tile offset.
template <typename E>
__device__ __forceinline__ int tile_elem(int lane, int j, int k) {
  return (32 * j + lane) * E::kVec + k;
}

// Element `pos` (a tile offset) of a tile staged in shared memory.
template <typename E>
__device__ __forceinline__ float staged(const uint4* st, uint32_t pos) {
  const uint4 v = st[pos / E::kVec];
  const int k = (int)(pos % E::kVec);
  if constexpr (E::kBytes == 2) {
    const uint32_t word = (k & 4) ? ((k & 2) ? v.w : v.z) : ((k & 2) ? v.y : v.x);
    return __uint_as_float((k & 1) ? (word & 0xffff0000u) : (word << 16));
  } else {
    return __uint_as_float((k & 2) ? ((k & 1) ? v.w : v.z) : ((k & 1) ? v.y : v.x));
  }
}

// Lane bit `bit` of a tile's large-term mask as a tile offset.  bf16: bit
// w < 16 is the low element of the lane's word w (vector w / 4, word w % 4),
// bit 16 + w its high element; float32: bit w is the lane's word w.
template <typename E>
__device__ __forceinline__ uint32_t big_pos(int lane, int bit) {
  if constexpr (E::kBytes == 2) {
    const int w = bit & 15;
    return (uint32_t)tile_elem<E>(lane, w >> 2, 2 * (w & 3) + (bit >> 4));
  } else {
    return (uint32_t)tile_elem<E>(lane, bit >> 2, bit & 3);
  }
}

__device__ __forceinline__ uint32_t ge_bf16x2(uint32_t a, uint32_t b) {
  uint32_t m;
  asm("set.ge.u32.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(a), "r"(b));
  return m;
}

// Weigh tile `tile` of the sampled row(s) (one warp) and write its record:
// W (weights at cw), Q (e^q where the weight is positive), P and S (all e^p
// and e^q).  Large terms (logit at or above the row's threshold) are listed
// and weighed in double-float, one per lane, from the tile staged in shared
// memory; in the float32 pass their logits read as -inf, so they add +0.
template <typename E, bool kAligned, bool kResidual>
__device__ void weigh_tile(const DrawArgs& a, DrawSmem& sm, const SampleCtx& x, int b, int tile,
                           int lane, int warp, int full_end) {
  constexpr int kTileElems = kTileVecs * E::kVec;
  uint32_t wp[kTileVecsPerLane][4], wq[kTileVecsPerLane][4];
  const bool ok = in_bounds(a, tile >= 0 && tile < a.tpr);
  load_tile<E, kAligned>(wp, x.rowP, tile, lane, a.V, tile < full_end, ok);
  if (kResidual) load_tile<E, kAligned>(wq, x.rowQ, tile, lane, a.V, tile < full_end, ok);
  // stage the logits as loaded, for the large terms
  uint4* stp = sm.stage[warp][0];
  uint4* stq = sm.stage[warp][1];
  __syncwarp();   // the previous tile's large terms are weighed
#pragma unroll
  for (int j = 0; j < kTileVecsPerLane; ++j) {
    stp[32 * j + lane] = make_uint4(wp[j][0], wp[j][1], wp[j][2], wp[j][3]);
    if (kResidual) stq[32 * j + lane] = make_uint4(wq[j][0], wq[j][1], wq[j][2], wq[j][3]);
  }
  // large-term mask; their logits become -inf for the float32 pass
  uint32_t big = 0u;
  if constexpr (E::kBytes == 2) {
    const uint32_t tp2 = (__float_as_uint(x.tp) >> 16) * 0x10001u;
    const uint32_t tq2 = (__float_as_uint(x.tq) >> 16) * 0x10001u;
#pragma unroll
    for (int j = 0; j < kTileVecsPerLane; ++j) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t m = ge_bf16x2(wp[j][i], tp2);
        if (kResidual) m |= ge_bf16x2(wq[j][i], tq2);
        big |= (m & 0x10001u) << (4 * j + i);
        wp[j][i] = (wp[j][i] & ~m) | (0xff80ff80u & m);
        if (kResidual) wq[j][i] = (wq[j][i] & ~m) | (0xff80ff80u & m);
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < kTileVecsPerLane; ++j) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const bool bb = __uint_as_float(wp[j][i]) >= x.tp ||
                        (kResidual && __uint_as_float(wq[j][i]) >= x.tq);
        big |= (uint32_t)bb << (4 * j + i);
        wp[j][i] = bb ? 0xff800000u : wp[j][i];
        if (kResidual) wq[j][i] = bb ? 0xff800000u : wq[j][i];
      }
    }
  }
  const unsigned long long chi2 = f2_pack(x.c_hi, x.c_hi), clo2 = f2_pack(x.c_lo, x.c_lo);
  const unsigned long long nmcp2 = f2_pack(-x.MCp, -x.MCp), nmcq2 = f2_pack(-x.MCq, -x.MCq);
  const unsigned long long ncw2 = f2_pack(-x.cw, -x.cw);
  unsigned long long sw2 = 0ull, sq2 = 0ull, sp2 = 0ull, sQ2 = 0ull;
#pragma unroll
  for (int j = 0; j < kTileVecsPerLane; ++j) {
#pragma unroll
    for (int k = 0; k < E::kVec; k += 2) {
      const unsigned long long xp2 = f2_pack(E::elem(wp[j], k), E::elem(wp[j], k + 1));
      float ep0, ep1;
      f2_unpack(f2_fma(xp2, clo2, f2_fma(xp2, chi2, nmcp2)), ep0, ep1);
      const unsigned long long ep2 = f2_pack(ex2_approx(ep0), ex2_approx(ep1));
      if (kResidual) {
        const unsigned long long xq2 = f2_pack(E::elem(wq[j], k), E::elem(wq[j], k + 1));
        float eq0, eq1;
        f2_unpack(f2_fma(xq2, clo2, f2_fma(xq2, chi2, nmcq2)), eq0, eq1);
        eq0 = ex2_approx(eq0);
        eq1 = ex2_approx(eq1);
        const unsigned long long eq2 = f2_pack(eq0, eq1);
        float d0, d1;
        f2_unpack(f2_fma(ncw2, eq2, ep2), d0, d1);
        sw2 = f2_add(sw2, f2_pack(fmaxf(d0, 0.f), fmaxf(d1, 0.f)));
        sq2 = f2_add(sq2, f2_pack(d0 > 0.f ? eq0 : 0.f, d1 > 0.f ? eq1 : 0.f));
        sp2 = f2_add(sp2, ep2);
        sQ2 = f2_add(sQ2, eq2);
      } else {
        sw2 = f2_add(sw2, ep2);
      }
    }
  }
  float a0, a1;
  f2_unpack(sw2, a0, a1);
  DF W{a0 + a1, 0.f};
  DF Q{0.f, 0.f}, P{0.f, 0.f}, S{0.f, 0.f};
  if (kResidual) {
    f2_unpack(sq2, a0, a1);
    Q = DF{a0 + a1, 0.f};
    f2_unpack(sp2, a0, a1);
    P = DF{a0 + a1, 0.f};
    f2_unpack(sQ2, a0, a1);
    S = DF{a0 + a1, 0.f};
  }
  // the large terms: listed in the warp's region and weighed one per lane
  const long long base = (long long)tile * kTileElems;
  const int cnt = __popc(big);
  int inc = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  const int total = __shfl_sync(0xffffffffu, inc, 31);
  if (total > 0) {
    DF w, q, ep, eq;
    if (total <= kDBigCap) {
      int o = inc - cnt;
      for (unsigned m = big; m; m &= m - 1u) sm.bigpos[warp][o++] = big_pos<E>(lane, __ffs(m) - 1);
      __syncwarp();
      for (int e = lane; e < total; e += 32) {
        const uint32_t pos = sm.bigpos[warp][e];
        if (!in_bounds(a, base + pos < a.V)) continue;
        big_term<kResidual>(x, sm.tab, staged<E>(stp, pos), kResidual ? staged<E>(stq, pos) : 0.f,
                            w, q, ep, eq);
        W = df_add(W, w);
        if (kResidual) {
          Q = df_add(Q, q);
          P = df_add(P, ep);
          S = df_add(S, eq);
        }
      }
    } else {
      __syncwarp();
      for (unsigned m = big; m; m &= m - 1u) {
        const uint32_t pos = big_pos<E>(lane, __ffs(m) - 1);
        if (!in_bounds(a, base + pos < a.V)) continue;
        big_term<kResidual>(x, sm.tab, staged<E>(stp, pos), kResidual ? staged<E>(stq, pos) : 0.f,
                            w, q, ep, eq);
        W = df_add(W, w);
        if (kResidual) {
          Q = df_add(Q, q);
          P = df_add(P, ep);
          S = df_add(S, eq);
        }
      }
    }
  }
  // the record: (W, Q), (P, S) as double-floats, one 8-byte store per total
  float2* rec = reinterpret_cast<float2*>(a.tile_recs + 2 * ((long long)b * a.tpr + tile));
  if (kResidual) {
    const DF tot = warp_sum4_df(W, Q, P, S);   // lanes 0, 8, 16, 24 hold W, Q, P, S
    if ((lane & 7) == 0 && ok) rec[lane >> 3] = make_float2(tot.hi, tot.lo);
  } else {
    W = warp_sum_df(W);   // P = W, no Q or S
    if (lane < 4 && ok)
      rec[lane] = (lane & 1) ? make_float2(0.f, 0.f) : make_float2(W.hi, W.lo);
  }
}

// ---------------------------------------------------------------- step 5
// Weight of a tile record (staged in shared memory) for the locate step:
// mode 0 the residual corrected to the exact c, mode 1 the bonus weights,
// mode 2 p (the residual was zero).
__device__ __forceinline__ DF rec_weight(const float4* recs, int j, int mode, DF dc) {
  const float4 r0 = recs[2 * j];
  if (mode == 0) return df_sub(DF{r0.x, r0.y}, df_mul(dc, DF{r0.z, r0.w}));
  if (mode == 1) return DF{r0.x, r0.y};
  const float4 r1 = recs[2 * j + 1];
  return DF{r1.x, r1.y};
}

// Among n records (one per lane, lanes >= n hold zero weight) choose the
// first whose inclusive prefix exceeds tau.  Returns its index and tau
// minus the prefix before it; at or past the total (rounding) the last
// record with positive weight, with `last` set.  Every lane gets the result.
__device__ __forceinline__ int pick_lane(DF w, DF tau, int lane, DF& tl, int& last) {
  DF inc = w;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const DF up = df_shfl_up(inc, o);
    if (lane >= o) inc = df_add(inc, up);
  }
  DF exc = df_shfl_up(inc, 1);
  if (lane == 0) exc = DF{0.f, 0.f};
  const bool pos = df_pos(w);
  const unsigned hit = __ballot_sync(0xffffffffu, pos && df_lt(tau, inc));
  const unsigned posm = __ballot_sync(0xffffffffu, pos);
  int h;
  if (hit) {
    h = __ffs(hit) - 1;
    last = 0;
  } else {
    h = posm ? 31 - __clz(posm) : 0;
    last = 1;
  }
  const DF t = df_sub(tau, exc);
  tl = DF{__shfl_sync(0xffffffffu, t.hi, h), __shfl_sync(0xffffffffu, t.lo, h)};
  return h;
}

// Warp 0 of the locating CTA: from the row's tile records (staged in
// shared memory) the exact c = S_p / S_q, the corrected total, u*W, and the
// tile holding it; lane l takes the records [l*per, (l+1)*per).  Leaves in
// sm.loc the tile, the mass left inside it, the weight mode, the
// correction dc, and whether rounding pushed u*W to the top (then the last
// positive element is taken).
__device__ void choose_tile(const DrawArgs& a, DrawSmem& sm, const SampleCtx& x, float u,
                            bool residual) {
  const int lane = threadIdx.x & 31;
  const int tpr = a.tpr;
  const float4* recs = reinterpret_cast<const float4*>(&sm.stage[0][0][0]);
  const int per = (tpr + 31) / 32;
  const int j0 = min(tpr, lane * per), j1 = min(tpr, j0 + per);
  DF v0{0.f, 0.f}, v1{0.f, 0.f}, v2{0.f, 0.f}, v3{0.f, 0.f};
  for (int j = j0; j < j1; ++j) {
    const float4 r0 = recs[2 * j], r1 = recs[2 * j + 1];
    v0 = df_add(v0, DF{r0.x, r0.y});
    v1 = df_add(v1, DF{r0.z, r0.w});
    v2 = df_add(v2, DF{r1.x, r1.y});
    v3 = df_add(v3, DF{r1.z, r1.w});
  }
  const DF t4 = warp_sum4_df(v0, v1, v2, v3);   // W, Q, P, S over the row at lanes 0, 8, 16, 24
  const DF Wt{__shfl_sync(0xffffffffu, t4.hi, 0), __shfl_sync(0xffffffffu, t4.lo, 0)};
  DF dc{0.f, 0.f};
  int mode = residual ? 0 : 1;
  DF tot = Wt;
  if (residual) {
    const DF Qt{__shfl_sync(0xffffffffu, t4.hi, 8), __shfl_sync(0xffffffffu, t4.lo, 8)};
    const DF Pt{__shfl_sync(0xffffffffu, t4.hi, 16), __shfl_sync(0xffffffffu, t4.lo, 16)};
    const DF St{__shfl_sync(0xffffffffu, t4.hi, 24), __shfl_sync(0xffffffffu, t4.lo, 24)};
    dc = df_sub(df_div(Pt, St), DF{x.cw, 0.f});
    tot = df_sub(Wt, df_mul(dc, Qt));
    if (!df_pos(tot)) {   // the residual is zero everywhere: draw from p_n
      mode = 2;
      tot = Pt;
    }
  }
  const DF tau = df_mul_f(tot, u);
  DF own{0.f, 0.f};
  int lastj = -1;
  for (int j = j0; j < j1; ++j) {
    const DF wj = rec_weight(recs, j, mode, dc);
    if (df_pos(wj)) {
      own = df_add(own, wj);
      lastj = j;
    }
  }
  DF tl;
  int past;
  const int h = pick_lane(own, tau, lane, tl, past);
  if (!past && lane == h) {
    DF run{0.f, 0.f};
    int js = -1, jl = -1;
    DF tg{0.f, 0.f};
    for (int j = j0; j < j1 && js < 0; ++j) {
      const DF wj = rec_weight(recs, j, mode, dc);
      if (!df_pos(wj)) continue;
      jl = j;
      const DF nxt = df_add(run, wj);
      if (df_lt(tl, nxt)) {
        js = j;
        tg = df_sub(tl, run);
      }
      run = nxt;
    }
    sm.loc.jstar = js >= 0 ? js : jl;   // rounding inside the lane: its last positive tile
    sm.loc.last_mode = js >= 0 ? 0 : 1;
    sm.loc.tg = tg;
  }
  if (past) {   // u*W at or past the total by rounding: the last tile with positive weight
    int lj = lastj;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lj = max(lj, __shfl_xor_sync(0xffffffffu, lj, o));
    if (lane == 0) {
      sm.loc.jstar = lj >= 0 ? lj : 0;
      sm.loc.last_mode = 1;
      sm.loc.tg = DF{0.f, 0.f};
    }
  }
  if (lane == 0) {
    sm.loc.mode = mode;
    sm.loc.dc = dc;
    sm.loc.pick = 0x7fffffff;
    sm.loc.lastpos = -1;
    sm.loc.best = 0ull;
  }
}

// Order-preserving bits of a float (larger float, larger key).
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// All threads of the CTA: the element of tile sm.loc.jstar.  Thread t
// weighs elements [t*kEpt, (t+1)*kEpt) of the tile with the rule the sweep
// used; a block-wide double-float scan finds the thread whose elements
// hold the remaining mass, and it walks them.  Returns the token (thread 0).
template <typename E>
__device__ int locate_element(const DrawArgs& a, DrawSmem& sm, const SampleCtx& x) {
  constexpr int kTileElems = kTileVecs * E::kVec;
  constexpr int kEpt = kTileElems / kDThreads;   // 4 (bf16) or 2 (f32)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int mode = sm.loc.mode;
  const DF dc = sm.loc.dc, tg = sm.loc.tg;
  const bool last_mode = sm.loc.last_mode != 0;
  const long long tbase = (long long)sm.loc.jstar * kTileElems;
  const long long e0 = tbase + (long long)tid * kEpt;
  DF w[kEpt];
  DF s{0.f, 0.f};
  int lpos = -1;
  unsigned long long best = 0ull;
#pragma unroll
  for (int k = 0; k < kEpt; ++k) {
    const long long e = e0 + k;
    DF q{0.f, 0.f};
    w[k] = DF{0.f, 0.f};
    if (e < a.V && in_bounds(a, sm.loc.jstar >= 0 && sm.loc.jstar < a.tpr)) {
      const float xp = E::load_scalar(x.rowP, e);
      if (mode == 0) {
        eval_pair<true>(xp, E::load_scalar(x.rowQ, e), x, sm.tab, w[k], q);
        w[k] = df_sub(w[k], df_mul(dc, q));
      } else {
        eval_pair<false>(xp, 0.f, x, sm.tab, w[k], q);
      }
      const unsigned long long key =
          ((unsigned long long)order_key(w[k].hi) << 32) | (0xffffffffu - (uint32_t)(e - tbase));
      best = key > best ? key : best;
    }
    if (df_pos(w[k])) {
      s = df_add(s, w[k]);
      lpos = (int)(e - tbase);
    }
  }
  // block-wide inclusive / exclusive prefix of the threads' sums
  DF inc = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const DF up = df_shfl_up(inc, o);
    if (lane >= o) inc = df_add(inc, up);
  }
  if (lane == 31) sm.wsum[warp] = inc;
  if (lpos >= 0) atomicMax(&sm.loc.lastpos, lpos);
  atomicMax(&sm.loc.best, best);
  __syncthreads();
  DF pre{0.f, 0.f};
  for (int w2 = 0; w2 < warp; ++w2) pre = df_add(pre, sm.wsum[w2]);
  const DF exc = df_add(pre, df_sub(inc, s));
  inc = df_add(pre, inc);
  if (!last_mode && df_pos(s) && df_lt(tg, inc)) atomicMin(&sm.loc.pick, tid);
  __syncthreads();
  if (tid == sm.loc.pick) {
    DF run = exc;
    int tk = -1;
#pragma unroll
    for (int k = 0; k < kEpt; ++k) {
      if (tk >= 0 || !df_pos(w[k])) continue;
      run = df_add(run, w[k]);
      if (df_lt(tg, run)) tk = tid * kEpt + k;
    }
    sm.loc.token = tk >= 0 ? tk : lpos;   // rounding inside the thread: its last positive element
  }
  __syncthreads();
  int token;
  if (sm.loc.pick != 0x7fffffff) {
    token = sm.loc.token;
  } else if (sm.loc.lastpos >= 0) {   // rounding or the last-record fallback
    token = sm.loc.lastpos;
  } else {                            // nothing positive: the largest weight, lowest index
    token = sm.loc.best ? (int)(0xffffffffu - (uint32_t)(sm.loc.best & 0xffffffffull)) : 0;
  }
  return (int)(tbase + token);
}

// ---------------------------------------------------------------- the kernel
template <typename E, bool kAligned, bool kPlug>
__global__ void __launch_bounds__(kDThreads, 4) sv_draw_kernel(DrawArgs a) {
  __shared__ DrawSmem sm;
  const int G = a.parts;
  const int b = blockIdx.x / G, g = blockIdx.x - b * G;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // inputs only: may run while the streaming pass drains
  const float T = __ldg(a.temperature + b);
  const bool greedy = (T == 0.f);
  if (g != 0 && (greedy || !valid_temperature(T))) return;   // part 0 finishes these rows alone
  draw_inputs<E>(a, b, T, sm);
  __syncthreads();
  if (sm.bad && g != 0) return;   // row-wide, so the same in every part

  // the streaming pass's partials are complete and visible after this
  wait_for_preceding_grid();
  if (!sm.bad) fold_stats(a, b, greedy, sm);
  __syncthreads();
  draw_scan<kPlug>(a, b, T, g == 0, sm);
  __syncthreads();
  if (sm.bad || greedy) return;   // the same in every part

  // step 4: this part's tiles of position n
  const int n = sm.n;
  const bool residual = n < sm.kb;
  const SampleCtx x = make_ctx<E>(a, b, n, residual, sm.rowMC[n], sm.rowS[n],
                                  residual ? sm.rowMC[a.K + 1 + n] : 0.f,
                                  residual ? sm.rowS[a.K + 1 + n] : 1.f, T);
  const int full_end = ((long long)a.tpr * kTileVecs * E::kVec == a.V) ? a.tpr : a.tpr - 1;
  const int t0 = g * a.tpr / G, t1 = (g + 1) * a.tpr / G;
  for (int t = t0 + warp; t < t1; t += kDWarps) {
    if (residual) weigh_tile<E, kAligned, true>(a, sm, x, b, t, lane, warp, full_end);
    else weigh_tile<E, kAligned, false>(a, sm, x, b, t, lane, warp, full_end);
  }
  __syncthreads();
  if (tid == 0) {
    // release: this part's tile records (written before the barrier) before
    // its ticket; acquire: the last part sees every part's records
    unsigned prev;
    asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;" : "=r"(prev) : "l"(a.tickets + b) : "memory");
    sm.last = prev + 1u == (unsigned)G;
  }
  __syncthreads();
  if (!sm.last) return;

  // step 5: every part's tile records are written; stage them so the tile
  // choice reads shared memory (the sweep's stage is free)
  {
    float4* st = reinterpret_cast<float4*>(&sm.stage[0][0][0]);
    const float4* trecs = a.tile_recs + 2 * (long long)b * a.tpr;
    for (int k = tid; k < 2 * a.tpr; k += kDThreads)
      st[k] = in_bounds(a, a.tpr <= 1024) ? __ldcg(trecs + k) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  __syncthreads();
  if (warp == 0) choose_tile(a, sm, x, sm.r[sm.kb], residual);
  __syncthreads();
  const int token = locate_element<E>(a, sm, x);
  if (warp == 0) {
    if (lane == 0) a.out_tokens[(long long)b * (a.K + 1) + n] = token;
    if (kPlug)
      plug_row(lane, n, lane < n ? sm.tok[lane] : token,
               a.plug_tokens + (long long)b * a.plug_max_len, a.plug_seq_len + b,
               a.plug_max_len, a.plug_last ? a.plug_last + b : nullptr, a.err);
  }
}

}  // namespace sv
