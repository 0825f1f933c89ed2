// The acceptance and sampling kernel of spec_verify.
//
//   Accept + sample (one thread-block cluster per batch row) folds the
//   streaming kernel's partials into row statistics, runs the
//   left-to-right acceptance test, and draws the replacement or bonus token
//   by inverse CDF over the one position that needs it, re-reading only
//   that position's rows.  The kPlug instantiation also appends each row's
//   emitted tokens to its sequence (the plug step, sv_plug.cuh).
//
// The rule is the exact rejection rule of the lesson "Decodificação
// Especulativa e EAGLE" (ai-engineering.academy, phase 10 lesson 25),
// sections "A Regra de Exatidão" and "Caso ganancioso"; the residual
// (p - q)+ / ||(p - q)+||_1 is taken over the full vocabulary as the same
// section states it.
#pragma once

#include <cooperative_groups.h>

#include "sv_plug.cuh"
#include "sv_stream.cuh"

namespace sv {

namespace cg = cooperative_groups;

constexpr int kP2Threads = 256;
constexpr int kP2Warps = kP2Threads / 32;
constexpr int kGroupVecs = 4;                     // a sampling group: 64 B of each row
constexpr int kMaxGroupsPerThread = 8;
constexpr int kMaxClusterSize = 16;
constexpr int kBigCap = 1024;                     // large terms listed per sweep (more: evaluated inline)
constexpr int kBigCapWarp = kBigCap / kP2Warps;   // each warp lists its own

// A term whose probability exceeds this is evaluated in double-float
// during sampling; smaller terms use the float32 path.
constexpr float kBigProb = 1.0e-4f;

// device flags (mirrors of the public SV_DEV_* values)
constexpr unsigned kDevBadTemperature = 1u;
constexpr unsigned kDevBadToken = 2u;
constexpr unsigned kDevNonFinite = 4u;
constexpr unsigned kDevBadK = 8u;

// ============================================================== sampling group
// The accept/sample code runs on a group of kP2Threads threads that starts
// at a warp boundary and ends the CTA (the whole CTA in
// sv_accept_sample_kernel).  gtid() is the thread's index in the group;
// gsync() is a barrier over the group only (named barrier 1), so a kernel
// may give its other warps other work.
__device__ __forceinline__ int gtid() { return (int)threadIdx.x - (int)blockDim.x + kP2Threads; }
__device__ __forceinline__ void gsync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kP2Threads) : "memory");
}

// ============================================================== accept + sample
struct AcceptArgs {
  const void* target;
  const void* draft;
  const int32_t* tokens;
  const float* uniforms;
  const float* temperature;
  int B, K, V;
  int tiles_per_row;
  int n_target_rows;
  int ngroups;                // sampling groups per logit row
  int groups_per_cta;         // groups of one row owned by one CTA of the cluster
  const float2* partials;
  const int32_t* k_per_row;   // [B] or nullptr (every row verifies K)
  unsigned* err;
  int32_t* accepted_len;
  int32_t* out_tokens;
  float* logp_out;
  float* logq_out;
  // plug step fused into the last writes (plug_tokens == nullptr: none)
  int32_t* plug_tokens;       // [B, plug_max_len]
  int32_t* plug_seq_len;      // [B]
  int32_t* plug_last;         // [B] or nullptr
  int plug_max_len;
};

// What each CTA of a cluster publishes after its sweep.
struct CtaRecord {
  DF W;            // sum of residual weights at c_used over the slice
  DF Q;            // sum of e^q over elements with positive weight
  DF Sp;           // sum of e^p over the slice
  DF Sq;           // sum of e^q over the slice
  int last_group;  // last group (row-global index) with positive weight, -1 if none
  int pad;
};

// The sampling decision the whole cluster agrees on.
struct Decision {
  int need_p_fallback;   // residual was zero everywhere: redo the sweep on p
  int rstar;             // CTA rank that locates the token
  int fallback_last;     // u*W fell beyond the total: take the last positive element
  int last_group;
  DF tau_local;          // target mass inside CTA rstar
  DF dc;                 // c_true - c_used
};

struct AcceptSmem {
  float2 tab[256];
  float rowMC[2 * kMaxK + 1];
  float rowS[2 * kMaxK + 1];
  int rowArg[kMaxK + 1];
  int tok[kMaxK];
  float r[kMaxK + 1];
  float xp[kMaxK];
  float xq[kMaxK];
  int bad;
  int n;
  int kb;   // drafted tokens this row verifies (K unless ragged)
  int redi[kP2Warps];
  CtaRecord rec;
  CtaRecord recs[2][kMaxClusterSize];   // every CTA's record, pushed here (per attempt)
  Decision dec;
  int pick_thread;
  int pick_last;
  int group_pick;
  DF tau_group;
  DF warp_tot[kP2Warps];
  // large terms of the current sweep, one list region per warp: their
  // positions ((local group << 5) | element), their double-float results
  // (w, q), and for every (step, thread) the slice of its warp's region its
  // group owns ((offset << 8) | count)
  uint32_t bigpos[kBigCap];
  float4 bigres[kBigCap];
  uint32_t bigref[kMaxGroupsPerThread][kP2Threads];
  DF red1[4];
};

// Everything the sampling sweep needs about the sampled position.
struct SampleCtx {
  const char* rowP;
  const char* rowQ;
  int V, g0, ng;          // CTA groups [g0, g0 + ng)
  float MCp, MCq;         // shifts (c-scaled) of the two rows
  float c_hi, c_lo;       // log2(e)/T as hi + lo
  float cw;               // c_used = S_p / S_q at the pass-1 shifts
  float thp, thq;         // big-term thresholds on 2^(x c - MC)
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
    if (ep > s.thp || eq > s.thq) {
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
    w = (ep > s.thp) ? big_exp(xp, s.MCp, s, tab) : DF{ep, 0.f};
    q = DF{0.f, 0.f};
  }
}

// Block-wide sum of four double-floats; every thread gets the totals.
// Block totals of four double-floats and the block maximum of an int (at
// least -1); every thread gets them.  Each thread leaves its values in the
// large-term lists (free once a sweep has folded them back), warps 0..3 sum
// one column each and warp 4 takes the maximum.
__device__ __forceinline__ void block_totals(DF (&v)[4], int& imax, AcceptSmem& sm) {
  static_assert(4 * kP2Threads * sizeof(DF) <= sizeof(sm.bigres), "scratch for the columns");
  static_assert(kP2Threads * sizeof(int) <= sizeof(sm.bigpos), "scratch for the maxima");
  static_assert(kP2Warps >= 5, "five reducing warps");
  const int tid = gtid(), lane = tid & 31, warp = tid >> 5;
  DF* col = reinterpret_cast<DF*>(sm.bigres);
  int* icol = reinterpret_cast<int*>(sm.bigpos);
#pragma unroll
  for (int i = 0; i < 4; ++i) col[i * kP2Threads + tid] = v[i];
  icol[tid] = imax;
  gsync();
  if (warp < 4) {
    DF t{0.f, 0.f};
    for (int k = lane; k < kP2Threads; k += 32) t = df_add(t, col[warp * kP2Threads + k]);
    t = warp_sum_df(t);
    if (lane == 0) sm.red1[warp] = t;
  } else if (warp == 4) {
    int m = -1;
    for (int k = lane; k < kP2Threads; k += 32) m = max(m, icol[k]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) sm.redi[0] = m;
  }
  gsync();
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = sm.red1[i];
  imax = sm.redi[0];
}

// Load group g (kGroupVecs vectors) of a row.
template <typename E, bool kAligned>
__device__ __forceinline__ void load_group(const char* row, int g, int V, uint32_t (&w)[kGroupVecs][4]) {
#pragma unroll
  for (int j = 0; j < kGroupVecs; ++j) load_vec<E, kAligned>(row, (long long)g * kGroupVecs + j, V, w[j]);
}

// Double-float weight of one large term at row position idx: w (and the
// q that goes with a positive w), plus e^p and e^q for the row totals.
template <typename E, bool kResidual>
__device__ __forceinline__ void big_term(const SampleCtx& x, const float2* tab, long long idx, DF& w,
                                         DF& q, DF& ep, DF& eq) {
  ep = big_exp(E::load_scalar(x.rowP, idx), x.MCp, x, tab);
  w = ep;
  q = DF{0.f, 0.f};
  eq = DF{0.f, 0.f};
  if (kResidual) {
    eq = big_exp(E::load_scalar(x.rowQ, idx), x.MCq, x, tab);
    const DF d = df_sub(ep, df_mul_f(eq, x.cw));
    w = df_pos(d) ? d : DF{0.f, 0.f};
    q = df_pos(d) ? eq : DF{0.f, 0.f};
  }
}

// Per-thread sums over a contiguous run of `ng` group weights: the prefix
// structure the locate step scans.  Thread t owns groups [t*cpt, (t+1)*cpt).
__device__ __forceinline__ void chunk_sums(const float4* part, int ng, DF& Wt, DF& Qt) {
  const int cpt = (ng + kP2Threads - 1) / kP2Threads;
  const int a0 = min(ng, (int)gtid() * cpt), a1 = min(ng, a0 + cpt);
  DF W{0.f, 0.f}, Q{0.f, 0.f};
  for (int gl = a0; gl < a1; ++gl) {
    const float4 p4 = part[gl];
    W = df_add(W, DF{p4.x, p4.y});
    Q = df_add(Q, DF{p4.z, p4.w});
  }
  Wt = W;
  Qt = Q;
}

// One sweep of this group of threads over its groups of the sampled row(s).
// Per-group weights go to part[] (w.hi, w.lo, q.hi, q.lo); the record to
// sm.rec.  The per-thread sums of part[] over the thread's contiguous run of
// groups come back in Wt, Qt (the locate step scans them).
//
// Small terms are summed in float32 as they stream by, two elements at a
// time (paired float32 arithmetic, each lane of a pair rounded as the
// scalar operation would be).  A large term only leaves its position in its
// warp's list; after the float32 pass each warp evaluates its own list in
// double-float (one term per lane) and every lane adds the results of its
// own groups' terms back into their weights.  Terms that find the list full
// are evaluated where they are found.
template <typename E, bool kAligned, bool kResidual>
__device__ void sweep_slice(const SampleCtx& x, AcceptSmem& sm, float4* part, DF& Wt, DF& Qt) {
  constexpr int kGroupElems = kGroupVecs * E::kVec;
  const int tid = gtid();
  const int lane = tid & 31, warp = tid >> 5;
  uint32_t* const wpos = sm.bigpos + warp * kBigCapWarp;
  float4* const wres = sm.bigres + warp * kBigCapWarp;
  DF accP{0.f, 0.f}, accQ{0.f, 0.f};
  int lastg = -1;
  int wcount = 0;   // entries of this warp's list (the same in every lane)
  const unsigned long long chi2 = f2_pack(x.c_hi, x.c_hi), clo2 = f2_pack(x.c_lo, x.c_lo);
  const unsigned long long nmcp2 = f2_pack(-x.MCp, -x.MCp), nmcq2 = f2_pack(-x.MCq, -x.MCq);
  const unsigned long long ncw2 = f2_pack(-x.cw, -x.cw);
  const int iters = (x.ng + kP2Threads - 1) / kP2Threads;   // the same for every thread
  for (int it = 0; it < iters; ++it) {
    const int gl = it * kP2Threads + tid;
    const bool valid = gl < x.ng;
    const int g = x.g0 + gl;
    uint32_t wp[kGroupVecs][4], wq[kGroupVecs][4];
#pragma unroll
    for (int j = 0; j < kGroupVecs; ++j) {
      wp[j][0] = wp[j][1] = wp[j][2] = wp[j][3] = E::kFillWord;
      wq[j][0] = wq[j][1] = wq[j][2] = wq[j][3] = E::kFillWord;
    }
    if (valid) {
      load_group<E, kAligned>(x.rowP, g, x.V, wp);
      if (kResidual) load_group<E, kAligned>(x.rowQ, g, x.V, wq);
    }
    // float32 pass; large terms only leave a bit in `big`
    unsigned long long sw2 = 0ull, sq2 = 0ull, sp2 = 0ull, sQ2 = 0ull;
    unsigned big = 0u;
#pragma unroll
    for (int j = 0; j < kGroupVecs; ++j) {
#pragma unroll
      for (int k = 0; k < E::kVec; k += 2) {
        const unsigned long long xp2 = f2_pack(E::elem(wp[j], k), E::elem(wp[j], k + 1));
        float ep0, ep1;
        f2_unpack(f2_fma(xp2, clo2, f2_fma(xp2, chi2, nmcp2)), ep0, ep1);
        ep0 = ex2_approx(ep0);
        ep1 = ex2_approx(ep1);
        const int bit = j * E::kVec + k;
        if (kResidual) {
          const unsigned long long xq2 = f2_pack(E::elem(wq[j], k), E::elem(wq[j], k + 1));
          float eq0, eq1;
          f2_unpack(f2_fma(xq2, clo2, f2_fma(xq2, chi2, nmcq2)), eq0, eq1);
          eq0 = ex2_approx(eq0);
          eq1 = ex2_approx(eq1);
          const bool b0 = ep0 > x.thp || eq0 > x.thq;
          const bool b1 = ep1 > x.thp || eq1 > x.thq;
          big |= ((unsigned)b0 << bit) | ((unsigned)b1 << (bit + 1));
          // a large term leaves the float32 sums: zero its e^p and e^q once
          // (then d = 0 - cw*0 = +0 and it adds +0 everywhere, as a skip would)
          ep0 = b0 ? 0.f : ep0;
          ep1 = b1 ? 0.f : ep1;
          eq0 = b0 ? 0.f : eq0;
          eq1 = b1 ? 0.f : eq1;
          const unsigned long long ep2 = f2_pack(ep0, ep1), eq2 = f2_pack(eq0, eq1);
          float d0, d1;
          f2_unpack(f2_fma(ncw2, eq2, ep2), d0, d1);
          sw2 = f2_add(sw2, f2_pack(fmaxf(d0, 0.f), fmaxf(d1, 0.f)));
          sq2 = f2_add(sq2, f2_pack(d0 > 0.f ? eq0 : 0.f, d1 > 0.f ? eq1 : 0.f));
          sp2 = f2_add(sp2, ep2);
          sQ2 = f2_add(sQ2, eq2);
        } else {
          const bool b0 = ep0 > x.thp, b1 = ep1 > x.thp;
          big |= ((unsigned)b0 << bit) | ((unsigned)b1 << (bit + 1));
          sw2 = f2_add(sw2, f2_pack(b0 ? 0.f : ep0, b1 ? 0.f : ep1));
        }
      }
    }
    float a0, a1;
    f2_unpack(sw2, a0, a1);
    const float sw = a0 + a1;
    f2_unpack(sq2, a0, a1);
    const float sq = a0 + a1;
    f2_unpack(sp2, a0, a1);
    const float sp = kResidual ? a0 + a1 : sw;
    f2_unpack(sQ2, a0, a1);
    const float sQ = a0 + a1;
    DF wg{sw, 0.f}, qg{sq, 0.f};
    // list this step's large terms in the warp's region
    uint32_t ref = 0;
    if (__any_sync(0xffffffffu, big != 0u)) {
      const int cnt = __popc(big);
      int inc = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += v;
      }
      const int total = __shfl_sync(0xffffffffu, inc, 31);
      if (wcount + total <= kBigCapWarp) {
        int o = wcount + inc - cnt;
        ref = ((uint32_t)o << 8) | (uint32_t)cnt;
        unsigned m = big;
        while (m) {
          const int e = __ffs(m) - 1;
          m &= m - 1u;
          wpos[o++] = ((uint32_t)gl << 5) | (uint32_t)e;
        }
        wcount += total;
      } else {
        // the list is full: evaluate the terms here
        unsigned m = big;
        while (m) {
          const int e = __ffs(m) - 1;
          m &= m - 1u;
          DF w, q, ep, eq;
          big_term<E, kResidual>(x, sm.tab, (long long)g * kGroupElems + e, w, q, ep, eq);
          wg = df_add(wg, w);
          qg = df_add(qg, q);
          accP = df_add(accP, ep);
          accQ = df_add(accQ, eq);
        }
      }
    }
    sm.bigref[it][tid] = ref;
    if (valid) {
      part[gl] = make_float4(wg.hi, wg.lo, qg.hi, qg.lo);
      if (df_pos(wg)) lastg = g;
    }
    accP = df_add_f(accP, sp);
    accQ = df_add_f(accQ, sQ);
  }
  __syncwarp();   // this warp's list is complete

  // this warp's listed large terms, one per lane
  for (int e = lane; e < wcount; e += 32) {
    const uint32_t pos = wpos[e];
    DF w, q, ep, eq;
    big_term<E, kResidual>(x, sm.tab, ((long long)x.g0 + (pos >> 5)) * kGroupElems + (pos & 31u), w,
                           q, ep, eq);
    wres[e] = make_float4(w.hi, w.lo, q.hi, q.lo);
    accP = df_add(accP, ep);   // the totals do not care which lane adds them
    accQ = df_add(accQ, eq);
  }
  __syncwarp();

  // fold the results back into the groups that own them
  for (int it = 0; it < iters; ++it) {
    const uint32_t ref = sm.bigref[it][tid];
    const int cnt = (int)(ref & 0xffu);
    if (cnt == 0) continue;
    const int gl = it * kP2Threads + tid;
    float4 p4 = part[gl];
    DF wg{p4.x, p4.y}, qg{p4.z, p4.w};
    for (int o = (int)(ref >> 8); o < (int)(ref >> 8) + cnt; ++o) {
      const float4 r = wres[o];
      wg = df_add(wg, DF{r.x, r.y});
      qg = df_add(qg, DF{r.z, r.w});
    }
    part[gl] = make_float4(wg.hi, wg.lo, qg.hi, qg.lo);
    if (df_pos(wg)) lastg = max(lastg, x.g0 + gl);
  }
  gsync();   // part[] complete

  chunk_sums(part, x.ng, Wt, Qt);
  DF tot[4] = {Wt, Qt, accP, accQ};
  int last = lastg;
  block_totals(tot, last, sm);
  if (tid == 0) {
    sm.rec.W = tot[0];
    sm.rec.Q = tot[1];
    sm.rec.Sp = tot[2];
    sm.rec.Sq = tot[3];
    sm.rec.last_group = last;
    sm.rec.pad = 0;
  }
}

// Warp 0 of every CTA: combine the cluster's records into the decision.
// Lane r holds record r (lanes from cs on hold nothing).  Every CTA runs the
// same lanes on the same records, so all agree.
__device__ void decide(const CtaRecord& rec, int cs, bool residual, float cw, float u,
                       int groups_per_cta, AcceptSmem& sm) {
  const int lane = gtid() & 31;
  const bool have = lane < cs;
  const DF zero{0.f, 0.f};
  const DF Sp = warp_sum_df(have ? rec.Sp : zero);
  const DF Sq = warp_sum_df(have ? rec.Sq : zero);
  int last_group = have ? rec.last_group : -1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) last_group = max(last_group, __shfl_xor_sync(0xffffffffu, last_group, o));
  DF dc = zero;
  if (residual) dc = df_sub(df_div(Sp, Sq), DF{cw, 0.f});
  const DF wr = !have ? zero : (residual ? df_sub(rec.W, df_mul(dc, rec.Q)) : rec.W);
  // inclusive and exclusive prefix sums of the corrected CTA weights
  DF inc = wr;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const DF up = df_shfl_up(inc, o);
    if (lane >= o) inc = df_add(inc, up);
  }
  DF exc = df_shfl_up(inc, 1);
  if (lane == 0) exc = zero;
  const DF tot{__shfl_sync(0xffffffffu, inc.hi, 31), __shfl_sync(0xffffffffu, inc.lo, 31)};
  Decision d;
  d.dc = dc;
  d.last_group = last_group;
  d.need_p_fallback = residual && !df_pos(tot);
  d.fallback_last = 0;
  d.rstar = -1;
  d.tau_local = zero;
  // tau = u * W: the token is the smallest index whose prefix exceeds tau
  const DF tau = df_mul_f(tot, u);
  const unsigned hit = __ballot_sync(0xffffffffu, have && df_pos(wr) && df_lt(tau, inc));
  const DF tl = df_sub(tau, exc);
  if (hit) {
    d.rstar = __ffs(hit) - 1;
    d.tau_local = DF{__shfl_sync(0xffffffffu, tl.hi, d.rstar), __shfl_sync(0xffffffffu, tl.lo, d.rstar)};
  }
  if (!d.need_p_fallback && d.rstar < 0) {
    d.fallback_last = 1;
    d.rstar = last_group >= 0 ? last_group / groups_per_cta : 0;
  }
  if (lane == 0) sm.dec = d;
}

// Find the token inside CTA rstar (all threads of that CTA).
template <typename E, bool kResidual>
__device__ int locate(const SampleCtx& x, AcceptSmem& sm, const float4* part, DF Wt, DF Qt) {
  const int tid = gtid(), lane = tid & 31, warp = tid >> 5;
  const DF dc = sm.dec.dc;
  const DF huge{3.0e38f, 0.f};
  const int cpt = (x.ng + kP2Threads - 1) / kP2Threads;
  if (tid == 0) {
    sm.pick_thread = 0x7fffffff;
    sm.pick_last = -1;
  }
  bool last_mode = sm.dec.fallback_last != 0;
  int gstar;
  DF tau_g = huge;
  if (last_mode) {
    gstar = sm.dec.last_group - x.g0;
  } else {
    // exclusive / inclusive prefix of the corrected per-thread sums
    const DF own = kResidual ? df_sub(Wt, df_mul(dc, Qt)) : Wt;
    DF inc = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const DF up = df_shfl_up(inc, o);
      if (lane >= o) inc = df_add(inc, up);
    }
    if (lane == 31) sm.warp_tot[warp] = inc;
    gsync();
    DF wpre{0.f, 0.f};
    for (int w = 0; w < warp; ++w) wpre = df_add(wpre, sm.warp_tot[w]);
    DF exc = df_shfl_up(inc, 1);
    if (lane == 0) exc = DF{0.f, 0.f};
    exc = df_add(wpre, exc);
    inc = df_add(wpre, inc);
    const DF tau = sm.dec.tau_local;
    if (df_pos(own)) {
      if (df_lt(tau, inc)) atomicMin(&sm.pick_thread, tid);
      atomicMax(&sm.pick_last, tid);
    }
    gsync();
    int ts = sm.pick_thread;
    bool at_top = false;
    if (ts == 0x7fffffff) {   // rounding pushed tau past this CTA's mass
      ts = max(sm.pick_last, 0);
      at_top = true;
    }
    if (tid == ts) {
      DF run = exc;
      int gs = -1, glast = -1;
      DF tg = huge;
      const int a0 = min(x.ng, tid * cpt), a1 = min(x.ng, a0 + cpt);
      for (int gl = a0; gl < a1; ++gl) {
        const float4 p4 = part[gl];
        DF wc{p4.x, p4.y};
        if (kResidual) wc = df_sub(wc, df_mul(dc, DF{p4.z, p4.w}));
        const DF nxt = df_add(run, wc);
        if (df_pos(wc)) {
          glast = gl;
          if (!at_top && gs < 0 && df_lt(tau, nxt)) {
            gs = gl;
            tg = df_sub(tau, run);
          }
        }
        run = nxt;
      }
      if (gs < 0) {   // fell off the end by rounding: top of the last positive group
        gs = glast >= 0 ? glast : a0;
        tg = huge;
      }
      sm.group_pick = gs;
      sm.tau_group = tg;
    }
    gsync();
    gstar = sm.group_pick;
    tau_g = sm.tau_group;
    if (tau_g.hi >= huge.hi) last_mode = true;
  }
  // the element inside group gstar: one lane per element, double-float scan
  int token = -1;
  if (warp == 0) {
    constexpr int kGroupElems = kGroupVecs * E::kVec;   // 32 (bf16) or 16 (f32)
    const long long e = ((long long)x.g0 + max(gstar, 0)) * kGroupElems + lane;
    const bool in = lane < kGroupElems && e < x.V;
    DF w{0.f, 0.f}, q{0.f, 0.f};
    if (in) {
      const float xp = E::load_scalar(x.rowP, e);
      const float xq = kResidual ? E::load_scalar(x.rowQ, e) : 0.f;
      eval_pair<kResidual>(xp, xq, x, sm.tab, w, q);
      if (kResidual) w = df_sub(w, df_mul(dc, q));
    }
    const bool pos = in && df_pos(w);
    DF inc = pos ? w : DF{0.f, 0.f};
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const DF up = df_shfl_up(inc, o);
      if (lane >= o) inc = df_add(inc, up);
    }
    const unsigned hit = __ballot_sync(0xffffffffu, pos && !last_mode && df_lt(tau_g, inc));
    const unsigned posm = __ballot_sync(0xffffffffu, pos);
    int k;
    if (hit) {
      k = __ffs(hit) - 1;
    } else if (posm) {
      k = 31 - __clz(posm);
    } else {
      // nothing positive here (rounding): the largest weight of the group
      float bw = in ? w.hi : -3.0e38f;
      int bk = lane;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ow = __shfl_xor_sync(0xffffffffu, bw, o);
        const int ok = __shfl_xor_sync(0xffffffffu, bk, o);
        if (ow > bw || (ow == bw && ok < bk)) {
          bw = ow;
          bk = ok;
        }
      }
      k = bk < kGroupElems ? bk : 0;
    }
    token = (int)(((long long)x.g0 + max(gstar, 0)) * kGroupElems + k);
  }
  return token;
}

// ---------------------------------------------------------------- accept stages
// Inputs of batch row b (warp 0): tokens, uniforms, the 2K gathered logits
// at the drafted tokens, and the row's validity (sm.bad).  Reads inputs
// only, so it may run before the statistics exist.
template <typename E>
__device__ void accept_inputs(const AcceptArgs& a, int b, float T, AcceptSmem& sm) {
  const int K = a.K, lane = gtid() & 31;
  const bool greedy = (T == 0.f);
  const long long ob = (long long)b * (K + 1);
  if ((gtid() >> 5) == 0) {
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
  if (!greedy)
    for (int i = gtid(); i < 256; i += kP2Threads) sm.tab[i] = kExp2Table256[i];
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

// Fold the tile partials of batch row b into row statistics, one half-warp
// per row (16 rows per round): (MC, S) for tempered rows, (max, lowest
// argmax) for greedy rows.
__device__ void fold_row_stats(const AcceptArgs& a, int b, bool greedy, AcceptSmem& sm) {
  constexpr int kHalves = kP2Threads / 16;
  const int K = a.K, kb = sm.kb, hl = gtid() & 15, hw = gtid() >> 4;
  const long long tb = (long long)b * (K + 1);
  const long long db = a.n_target_rows + (long long)b * K;
  const int nrows = greedy ? K + 1 : 2 * K + 1;
  for (int base = 0; base < nrows; base += kHalves) {   // the same trip count in every warp
    const int rr = base + hw;
    const float2* pp = nullptr;
    // only the rows the row's K_b verifies: target 0..kb, draft 0..kb-1
    if (rr < nrows && (rr <= K ? rr <= kb : rr - K - 1 < kb)) {
      const long long prow = (rr <= K) ? tb + rr : db + (rr - K - 1);
      pp = a.partials + prow * a.tiles_per_row;
    }
    const float2 st = fold_partials<16>(pp, a.tiles_per_row, greedy, hl);
    if (pp && hl == 0) {
      sm.rowMC[rr] = st.x;
      if (greedy) sm.rowArg[rr] = __float_as_int(st.y);
      else sm.rowS[rr] = st.y;
    }
  }
}

// The plug step for batch row b, by one warp: lane i <= n holds emitted
// token i.
__device__ __forceinline__ void plug_row_into(const AcceptArgs& a, int b, int lane, int n,
                                              int32_t tok) {
  plug_row(lane, n, tok, a.plug_tokens + (long long)b * a.plug_max_len, a.plug_seq_len + b,
           a.plug_max_len, a.plug_last ? a.plug_last + b : nullptr, a.err);
}

// Acceptance scan (warp 0): one lane per drafted position; sets sm.n and
// sm.bad.  With `write`, also writes accepted_len, the log-probabilities and
// every out_tokens slot except the one a tempered row still has to sample.
template <bool kPlug = false>
__device__ void accept_scan(const AcceptArgs& a, int b, float T, bool write, AcceptSmem& sm) {
  const int K = a.K, lane = gtid() & 31;
  if ((gtid() >> 5) != 0) return;
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
      if (bad) atomicOr(a.err, (unsigned)bad);
    }
    // a greedy row's tokens are all known here (a tempered row plugs after
    // its draw; an error row is never plugged)
    if (kPlug && greedy && !bad) plug_row_into(a, b, lane, n, v);
  }
  if (lane == 0) {
    sm.n = n;
    sm.bad = bad;
  }
}

// What the sampling sweep needs about position n of batch row b, for the
// groups [g0, g0 + ng) of the sampled row(s).
template <typename E>
__device__ SampleCtx sample_ctx(const AcceptArgs& a, int b, float T, int g0, int ng,
                                const AcceptSmem& sm) {
  const int K = a.K, n = sm.n;
  const long long rowbytes = (long long)a.V * E::kBytes;
  SampleCtx x;
  x.rowP = (const char*)a.target + ((long long)b * (K + 1) + n) * rowbytes;
  x.rowQ = (n < sm.kb) ? (const char*)a.draft + ((long long)b * K + n) * rowbytes : nullptr;
  x.V = a.V;
  x.g0 = g0;
  x.ng = ng;
  x.MCp = sm.rowMC[n];
  x.MCq = (n < sm.kb) ? sm.rowMC[K + 1 + n] : 0.f;
  const float Sp32 = sm.rowS[n];
  const float Sq32 = (n < sm.kb) ? sm.rowS[K + 1 + n] : 1.f;
  x.L = log2e_over(T);
  // float32 path split of L with a strictly positive low part
  x.c_hi = x.L.hi;
  x.c_lo = x.L.lo;
  if (!(x.c_lo > 0.f)) {
    x.c_hi = __uint_as_float(__float_as_uint(x.L.hi) - 1u);   // one ulp below (L > 0)
    x.c_lo = __fadd_rn(__fsub_rn(x.L.hi, x.c_hi), x.L.lo);
  }
  x.cw = __fdiv_rn(Sp32, Sq32);
  x.thp = kBigProb * Sp32;
  x.thq = kBigProb * Sq32;
  return x;
}

// ---------------------------------------------------------------- the cluster kernel
// kPlug: the plug step is fused in (a.plug_tokens != nullptr).
template <typename E, bool kAligned, bool kPlug>
__global__ void __launch_bounds__(kP2Threads, 4) sv_accept_sample_kernel(AcceptArgs a) {
  extern __shared__ __align__(16) float4 s_part[];
  __shared__ AcceptSmem sm;
  cg::cluster_group cluster = cg::this_cluster();
  const int cs = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int b = blockIdx.x / cs;
  const int tid = gtid();

  // inputs only
  const float T = __ldg(a.temperature + b);
  const bool greedy = (T == 0.f);
  if (rank != 0 && (greedy || !valid_temperature(T))) return;   // rank 0 alone handles these
  accept_inputs<E>(a, b, T, sm);
  gsync();
  if (sm.bad && rank != 0) return;   // row-wide, so the same in every CTA of the cluster

  // Everything above reads only the caller's inputs.  Launched as a
  // programmatic dependent of the streaming kernel, the grid may start as
  // that kernel's CTAs exit; this waits until its partials are complete and
  // visible (without that launch attribute it returns at once).
  wait_for_preceding_grid();
  if (!sm.bad) fold_row_stats(a, b, greedy, sm);
  gsync();
  accept_scan<kPlug>(a, b, T, rank == 0, sm);
  gsync();
  if (sm.bad || greedy) return;   // the same in every CTA of the cluster

  // sampling at position n
  const int g0 = rank * a.groups_per_cta;
  SampleCtx x = sample_ctx<E>(a, b, T, g0, max(0, min(a.ngroups - g0, a.groups_per_cta)), sm);
  const float u = sm.r[sm.kb];
  bool residual = sm.n < sm.kb;
  for (int attempt = 0; attempt < 2; ++attempt) {
    DF Wt, Qt;
    if (residual) sweep_slice<E, kAligned, true>(x, sm, s_part, Wt, Qt);
    else sweep_slice<E, kAligned, false>(x, sm, s_part, Wt, Qt);
    // push this CTA's record into every CTA of the cluster; after the
    // barrier each CTA reads only its own copies, so none waits for the
    // others to finish reading before it goes on (or exits)
    if (tid == 0)
      for (int r = 0; r < cs; ++r) *cluster.map_shared_rank(&sm.recs[attempt][rank], r) = sm.rec;
    cluster.sync();
    if (tid < 32) {   // warp 0: one record per lane, then the decision
      CtaRecord rec{};
      if (tid < cs) rec = sm.recs[attempt][tid];
      decide(rec, cs, residual, x.cw, u, a.groups_per_cta, sm);
    }
    gsync();
    if (sm.dec.need_p_fallback) {
      residual = false;   // the residual is zero everywhere: draw from p_t instead
      x.rowQ = nullptr;
      continue;
    }
    if (rank == sm.dec.rstar) {
      const int token = residual ? locate<E, true>(x, sm, s_part, Wt, Qt)
                                 : locate<E, false>(x, sm, s_part, Wt, Qt);
      if (tid == 0) a.out_tokens[(long long)b * (a.K + 1) + sm.n] = token;
      if (kPlug && tid < 32)   // warp 0 holds the token
        plug_row_into(a, b, tid, sm.n, tid < sm.n ? sm.tok[tid] : token);
    }
    break;
  }
}

}  // namespace sv
