// The two kernels of spec_verify.
//
//   sv_row_stats_kernel  (the streaming pass) reads every logit row once,
//     16 bytes per lane per load, and writes one partial per 4 KB tile:
//     (tile max m, sum of e^((x - m)/T)) for rows of tempered rows, or
//     (max logit, lowest index of it) for target rows of greedy rows.
//     Draft rows of greedy rows are not read at all.
//
//   sv_accept_sample_kernel  (one thread-block cluster per batch row)
//     folds the tile partials into row statistics, runs the left-to-right
//     acceptance test, and draws the replacement or bonus token by inverse
//     CDF over the one position that needs it, re-reading only that
//     position's target (and draft) row.
//
// The rule is the exact rejection rule of the lesson "Decodificação
// Especulativa e EAGLE" (ai-engineering.academy, phase 10 lesson 25),
// sections "A Regra de Exatidão" and "Caso ganancioso"; the residual
// (p - q)+ / ||(p - q)+||_1 is taken over the full vocabulary as the same
// section states it.
#pragma once

#include <cooperative_groups.h>

#include "sv_common.cuh"

namespace sv {

namespace cg = cooperative_groups;

constexpr int kMaxK = 16;
constexpr int kP1Threads = 256;
constexpr int kTileVecsPerLane = 8;             // 8 x 16 B = 128 B per lane
constexpr int kTileVecs = 32 * kTileVecsPerLane; // 4 KB of one row per tile
constexpr int kP2Threads = 512;
constexpr int kP2Warps = kP2Threads / 32;
constexpr int kMaxClusterSize = 8;
constexpr int kMaxVecsPerCta = 8192;            // 16 B of smem per vector -> 128 KB
// A term whose probability exceeds this is evaluated in double-float
// during sampling; smaller terms use the float32 path.
constexpr float kBigProb = 1.0e-4f;

// device flags (mirrors of the public SV_DEV_* values)
constexpr unsigned kDevBadTemperature = 1u;
constexpr unsigned kDevBadToken = 2u;
constexpr unsigned kDevNonFinite = 4u;

struct RowStatsArgs {
  const void* target;
  const void* draft;
  const float* temperature;
  int B, K, V;
  int tiles_per_row;
  long long n_tiles;          // (B*(K+1) + B*K) * tiles_per_row
  long long n_target_rows;    // B*(K+1)
  float2* partials;           // [n_target_rows + B*K][tiles_per_row]
  unsigned* err;
};

// ============================================================== streaming pass
template <typename E, bool kAligned>
__global__ void __launch_bounds__(kP1Threads) sv_row_stats_kernel(RowStatsArgs a) {
  if (blockIdx.x == 0 && threadIdx.x == 0) *a.err = 0u;
  // let the dependent accept/sample grid get scheduled early
  asm volatile("griddepcontrol.launch_dependents;");

  const int lane = threadIdx.x & 31;
  const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
  const long long t0 = gw * a.n_tiles / nw;
  const long long t1 = (gw + 1) * a.n_tiles / nw;
  if (t0 >= t1) return;
  long long row = t0 / a.tiles_per_row;
  int ti = (int)(t0 - row * a.tiles_per_row);

  for (long long tile = t0; tile < t1; ++tile) {
    const bool is_draft = row >= a.n_target_rows;
    const long long r = is_draft ? row - a.n_target_rows : row;
    const int b = (int)(r / (is_draft ? a.K : a.K + 1));
    const float T = __ldg(a.temperature + b);
    const bool greedy = (T == 0.f);
    if (valid_temperature(T) && !(is_draft && greedy)) {
      const char* rowp =
          (const char*)(is_draft ? a.draft : a.target) + r * (long long)a.V * E::kBytes;
      const long long v0 = (long long)ti * kTileVecs + lane;
      uint32_t w[kTileVecsPerLane][4];
#pragma unroll
      for (int j = 0; j < kTileVecsPerLane; ++j) load_vec<E, kAligned>(rowp, v0 + 32 * j, a.V, w[j]);

      float2 part;
      if (greedy) {
        // max logit and the lowest index holding it
        float best = SV_NEG_INF;
        int bi = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < kTileVecsPerLane; ++j) {
#pragma unroll
          for (int k = 0; k < E::kVec; ++k) {
            const float x = E::elem(w[j], k);
            if (x > best) {
              best = x;
              bi = (int)((v0 + 32 * j) * E::kVec + k);
            }
          }
        }
        const float m = warp_max(best);
        const int idx = warp_min_int(best == m ? bi : 0x7fffffff);
        part = make_float2(m, __int_as_float(idx));
      } else {
        float m = SV_NEG_INF;
#pragma unroll
        for (int j = 0; j < kTileVecsPerLane; ++j)
#pragma unroll
          for (int k = 0; k < E::kVec; ++k) m = fmaxf(m, E::elem(w[j], k));
        m = warp_max(m);
        float s = 0.f;
        if (m != SV_NEG_INF) {
          const float c = __fdiv_rn(kLog2eHi, T);
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int j = 0; j < kTileVecsPerLane; ++j)
#pragma unroll
            for (int k = 0; k < E::kVec; ++k)
              acc[k & 3] += ex2_approx(__fmul_rn(__fsub_rn(E::elem(w[j], k), m), c));
          s = warp_sum((acc[0] + acc[1]) + (acc[2] + acc[3]));
        }
        part = make_float2(m, s);
      }
      if (lane == 0) a.partials[row * a.tiles_per_row + ti] = part;
    }
    if (++ti == a.tiles_per_row) {
      ti = 0;
      ++row;
    }
  }
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
  long long n_target_rows;
  int nvec;                   // vectors per logit row
  int vecs_per_cta;           // vectors of one row owned by one CTA of the cluster
  const float2* partials;
  unsigned* err;
  int32_t* accepted_len;
  int32_t* out_tokens;
  float* logp_out;
  float* logq_out;
};

// What each CTA of a cluster publishes after its sweep.
struct CtaRecord {
  DF W;            // sum of residual weights at c_used over the slice
  DF Q;            // sum of e^q over elements with positive weight
  DF Sp;           // sum of e^p over the slice
  DF Sq;           // sum of e^q over the slice
  int last_vec;    // last vector (row-global index) with positive weight, -1 if none
  int pad;
};

// The sampling decision the whole cluster agrees on.
struct Decision {
  int need_p_fallback;   // residual was zero everywhere: redo the sweep on p
  int rstar;             // CTA rank that locates the token
  int fallback_last;     // u*W fell beyond the total: take the last positive element
  int last_vec;
  DF tau_local;          // target mass inside CTA rstar
  DF dc;                 // c_true - c_used
};

struct SampleSmem {
  float2 tab[256];
  DF warpW[kP2Warps], warpQ[kP2Warps], warpP[kP2Warps], warpSq[kP2Warps];
  int warpLast[kP2Warps];
  CtaRecord rec;
  Decision dec;
  float rowM[2 * kMaxK + 1];
  float rowS[2 * kMaxK + 1];
  int rowArg[kMaxK + 1];
  int n;
  int bad;
  int lane_pick;
  int vec_pick;
  DF tau_vec;
};

// Weight of element k of a loaded vector pair, exactly as the sweep counts it.
// kResidual: w = max(e^p - c e^q, 0) and the e^q that goes with it when w > 0;
// otherwise w = e^p.  Elements whose probability is above kBigProb are
// evaluated in double-float, the rest in float32.
template <typename E, bool kResidual>
__device__ __forceinline__ void eval_elem(const uint32_t (&wp)[4], const uint32_t (&wq)[4], int k,
                                          float Mp, float Mq, DF L, float c, float thp,
                                          float thq, const float2* tab, DF& w, DF& q) {
  const float xp = E::elem(wp, k);
  const float ep = ex2_approx(__fmul_rn(__fsub_rn(xp, Mp), L.hi));
  if (kResidual) {
    const float xq = E::elem(wq, k);
    const float eq = ex2_approx(__fmul_rn(__fsub_rn(xq, Mq), L.hi));
    if (ep > thp || eq > thq) {
      const DF epd = exp_df(xp, Mp, L, tab);
      const DF eqd = exp_df(xq, Mq, L, tab);
      const DF d = df_sub(epd, df_mul_f(eqd, c));
      if (df_pos(d)) {
        w = d;
        q = eqd;
      } else {
        w = DF{0.f, 0.f};
        q = DF{0.f, 0.f};
      }
    } else {
      const float d = __fmaf_rn(-c, eq, ep);
      w = DF{d > 0.f ? d : 0.f, 0.f};
      q = DF{d > 0.f ? eq : 0.f, 0.f};
    }
  } else {
    if (ep > thp) {
      w = exp_df(xp, Mp, L, tab);
    } else {
      w = DF{ep, 0.f};
    }
    q = DF{0.f, 0.f};
  }
}

// Sweep of one CTA over its slice of the row(s): per-vector weight sums go
// to s_vec, per-warp totals to sm.warp*, the CTA total to sm.rec.
template <typename E, bool kAligned, bool kResidual>
__device__ void sweep_slice(const char* rowP, const char* rowQ, int V, int cv0, int ncv, float Mp,
                            float Mq, DF L, float c, float thp, float thq, SampleSmem& sm,
                            float4* s_vec) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwr = (ncv + 31) >> 5;
  const int wr0 = warp * nwr / kP2Warps, wr1 = (warp + 1) * nwr / kP2Warps;
  DF accW{0.f, 0.f}, accQ{0.f, 0.f}, accP{0.f, 0.f}, accSq{0.f, 0.f};
  int last = -1;
  for (int wr = wr0; wr < wr1; ++wr) {
    const int vl = wr * 32 + lane;
    const bool valid = vl < ncv;
    const long long v = (long long)cv0 + vl;
    uint32_t wp[4], wq[4];
    if (valid) {
      load_vec<E, kAligned>(rowP, v, V, wp);
      if (kResidual) load_vec<E, kAligned>(rowQ, v, V, wq);
    } else {
      wp[0] = wp[1] = wp[2] = wp[3] = E::kFillWord;
    }
    if (!kResidual || !valid) wq[0] = wq[1] = wq[2] = wq[3] = E::kFillWord;
    float sw = 0.f, sq = 0.f, sp = 0.f, sQ = 0.f;
    unsigned big = 0u;
#pragma unroll
    for (int k = 0; k < E::kVec; ++k) {
      const float ep = ex2_approx(__fmul_rn(__fsub_rn(E::elem(wp, k), Mp), L.hi));
      if (kResidual) {
        const float eq = ex2_approx(__fmul_rn(__fsub_rn(E::elem(wq, k), Mq), L.hi));
        if (ep > thp || eq > thq) {
          big |= 1u << k;
        } else {
          const float d = __fmaf_rn(-c, eq, ep);
          sw += d > 0.f ? d : 0.f;
          sq += d > 0.f ? eq : 0.f;
          sp += ep;
          sQ += eq;
        }
      } else {
        if (ep > thp) {
          big |= 1u << k;
        } else {
          sw += ep;
          sp += ep;
        }
      }
    }
    DF wb{0.f, 0.f}, qb{0.f, 0.f}, pb{0.f, 0.f}, Qb{0.f, 0.f};
    // the rare large terms, in double-float; every lane with one pending
    // works on it in the same pass
    while (__any_sync(0xffffffffu, big != 0u)) {
      if (big) {
        const int k = __ffs(big) - 1;
        big &= big - 1u;
        const float xp = E::elem(wp, k);
        const DF epd = exp_df(xp, Mp, L, sm.tab);
        pb = df_add(pb, epd);
        if (kResidual) {
          const DF eqd = exp_df(E::elem(wq, k), Mq, L, sm.tab);
          Qb = df_add(Qb, eqd);
          const DF d = df_sub(epd, df_mul_f(eqd, c));
          if (df_pos(d)) {
            wb = df_add(wb, d);
            qb = df_add(qb, eqd);
          }
        } else {
          wb = df_add(wb, epd);
        }
      }
    }
    const DF wv = df_add_f(wb, sw);
    const DF qv = df_add_f(qb, sq);
    if (valid) {
      s_vec[vl] = make_float4(wv.hi, wv.lo, qv.hi, qv.lo);
      if (df_pos(wv)) last = (int)v;
    }
    accW = df_add(accW, wv);
    accQ = df_add(accQ, qv);
    accP = df_add(accP, df_add_f(pb, sp));
    accSq = df_add(accSq, df_add_f(Qb, sQ));
  }
  accW = warp_sum_df(accW);
  accQ = warp_sum_df(accQ);
  accP = warp_sum_df(accP);
  accSq = warp_sum_df(accSq);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
  if (lane == 0) {
    sm.warpW[warp] = accW;
    sm.warpQ[warp] = accQ;
    sm.warpP[warp] = accP;
    sm.warpSq[warp] = accSq;
    sm.warpLast[warp] = last;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    CtaRecord rec;
    rec.W = rec.Q = rec.Sp = rec.Sq = DF{0.f, 0.f};
    rec.last_vec = -1;
    rec.pad = 0;
    for (int i = 0; i < kP2Warps; ++i) {
      rec.W = df_add(rec.W, sm.warpW[i]);
      rec.Q = df_add(rec.Q, sm.warpQ[i]);
      rec.Sp = df_add(rec.Sp, sm.warpP[i]);
      rec.Sq = df_add(rec.Sq, sm.warpSq[i]);
      rec.last_vec = max(rec.last_vec, sm.warpLast[i]);
    }
    sm.rec = rec;
  }
}

// Thread 0 of every CTA: combine the cluster's records into the decision.
// Every CTA reads the same records in the same order, so all agree.
__device__ void decide(cg::cluster_group& cluster, int cs, bool residual, float c_used, float u,
                       int vecs_per_cta, SampleSmem& sm) {
  DF Sp{0.f, 0.f}, Sq{0.f, 0.f};
  CtaRecord recs[kMaxClusterSize];
  for (int r = 0; r < cs; ++r) {
    const CtaRecord* rp = cluster.map_shared_rank(&sm.rec, r);
    recs[r] = *rp;
    Sp = df_add(Sp, recs[r].Sp);
    Sq = df_add(Sq, recs[r].Sq);
  }
  DF dc{0.f, 0.f};
  if (residual) dc = df_sub(df_div(Sp, Sq), DF{c_used, 0.f});
  DF Wc[kMaxClusterSize];
  DF tot{0.f, 0.f};
  int last_vec = -1;
  for (int r = 0; r < cs; ++r) {
    Wc[r] = residual ? df_sub(recs[r].W, df_mul(dc, recs[r].Q)) : recs[r].W;
    tot = df_add(tot, Wc[r]);
    last_vec = max(last_vec, recs[r].last_vec);
  }
  Decision d;
  d.dc = dc;
  d.last_vec = last_vec;
  d.need_p_fallback = residual && !df_pos(tot);
  d.fallback_last = 0;
  d.rstar = -1;
  d.tau_local = DF{0.f, 0.f};
  if (!d.need_p_fallback) {
    // tau = u * W: the token is the smallest index whose prefix exceeds tau
    const DF tau = df_mul_f(tot, u);
    DF pre{0.f, 0.f};
    for (int r = 0; r < cs; ++r) {
      const DF nxt = df_add(pre, Wc[r]);
      if (df_pos(Wc[r]) && df_lt(tau, nxt)) {
        d.rstar = r;
        d.tau_local = df_sub(tau, pre);
        break;
      }
      pre = nxt;
    }
    if (d.rstar < 0) {
      d.fallback_last = 1;
      d.rstar = last_vec >= 0 ? last_vec / vecs_per_cta : 0;
    }
  }
  sm.dec = d;
}

// Find the token inside CTA rstar.  Runs on all threads of that CTA.
template <typename E, bool kAligned, bool kResidual>
__device__ int locate(const char* rowP, const char* rowQ, int V, int cv0, int ncv, float Mp,
                      float Mq, DF L, float c, float thp, float thq, SampleSmem& sm,
                      const float4* s_vec) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const DF dc = sm.dec.dc;
  const int nwr = (ncv + 31) >> 5;
  int vstar = -1;            // CTA-local vector that holds the token
  DF tau_v{0.f, 0.f};
  bool last_mode = sm.dec.fallback_last != 0;
  if (last_mode) {
    vstar = sm.dec.last_vec - cv0;
  } else {
    // the warp, then the lane chunk, then the vector whose prefix passes tau
    __shared__ int s_wstar;
    __shared__ DF s_tauw;
    if (threadIdx.x == 0) {
      DF pre{0.f, 0.f};
      int ws = -1, wlast = -1;
      DF tw{0.f, 0.f};
      for (int i = 0; i < kP2Warps; ++i) {
        const DF wc = kResidual ? df_sub(sm.warpW[i], df_mul(dc, sm.warpQ[i])) : sm.warpW[i];
        const DF nxt = df_add(pre, wc);
        if (df_pos(wc)) {
          wlast = i;
          if (ws < 0 && df_lt(sm.dec.tau_local, nxt)) {
            ws = i;
            tw = df_sub(sm.dec.tau_local, pre);
          }
        }
        pre = nxt;
      }
      if (ws < 0) {   // rounding pushed tau past this CTA's mass: last positive warp, top end
        ws = wlast < 0 ? 0 : wlast;
        tw = DF{3.4e38f, 0.f};
      }
      s_wstar = ws;
      s_tauw = tw;
    }
    __syncthreads();
    if (warp == s_wstar) {
      const int vs = (warp * nwr / kP2Warps) * 32;
      const int ve = min(ncv, ((warp + 1) * nwr / kP2Warps) * 32);
      const int nv = max(0, ve - vs);
      const int chunk = (nv + 31) >> 5;
      const int a0 = vs + lane * chunk;
      const int a1 = min(ve, a0 + chunk);
      DF own{0.f, 0.f};
      for (int i = a0; i < a1; ++i) {
        const float4 s = s_vec[i];
        DF wc{s.x, s.y};
        if (kResidual) wc = df_sub(wc, df_mul(dc, DF{s.z, s.w}));
        own = df_add(own, wc);
      }
      // inclusive scan over lanes
      DF inc = own;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const DF up = df_shfl_up(inc, o);
        if (lane >= o) inc = df_add(inc, up);
      }
      const DF exc = df_sub(inc, own);
      const DF tw = s_tauw;
      const bool hit = df_pos(own) && df_lt(tw, inc);
      const unsigned hits = __ballot_sync(0xffffffffu, hit);
      const unsigned posl = __ballot_sync(0xffffffffu, df_pos(own));
      int lstar;
      bool at_top = false;
      if (hits) {
        lstar = __ffs(hits) - 1;
      } else {
        lstar = posl ? 31 - __clz(posl) : 0;
        at_top = true;
      }
      if (lane == lstar) {
        DF run = exc;
        int vs2 = -1, vlastpos = -1;
        DF tv{0.f, 0.f};
        for (int i = a0; i < a1; ++i) {
          const float4 s = s_vec[i];
          DF wc{s.x, s.y};
          if (kResidual) wc = df_sub(wc, df_mul(dc, DF{s.z, s.w}));
          const DF nxt = df_add(run, wc);
          if (df_pos(wc)) {
            vlastpos = i;
            if (!at_top && vs2 < 0 && df_lt(tw, nxt)) {
              vs2 = i;
              tv = df_sub(tw, run);
            }
          }
          run = nxt;
        }
        if (vs2 < 0) {   // fell off the end by rounding: top of the last positive vector
          vs2 = vlastpos < 0 ? max(a0, 0) : vlastpos;
          tv = DF{3.4e38f, 0.f};
        }
        sm.vec_pick = vs2;
        sm.tau_vec = tv;
      }
      __syncwarp();
    }
    __syncthreads();
    vstar = sm.vec_pick;
    tau_v = sm.tau_vec;
    if (tau_v.hi >= 3.4e38f) last_mode = true;
  }
  // walk the elements of vector vstar
  int token = -1;
  if (threadIdx.x == 0) {
    const long long v = (long long)cv0 + max(vstar, 0);
    uint32_t wp[4], wq[4];
    load_vec<E, kAligned>(rowP, v, V, wp);
    if (kResidual) {
      load_vec<E, kAligned>(rowQ, v, V, wq);
    } else {
      wq[0] = wq[1] = wq[2] = wq[3] = E::kFillWord;
    }
    DF run{0.f, 0.f};
    int lastpos = -1, best = -1;
    float bestw = -1.f;
    for (int k = 0; k < E::kVec; ++k) {
      if (v * E::kVec + k >= V) break;
      DF w, q;
      eval_elem<E, kResidual>(wp, wq, k, Mp, Mq, L, c, thp, thq, sm.tab, w, q);
      if (kResidual) w = df_sub(w, df_mul(dc, q));
      if (w.hi > bestw) {
        bestw = w.hi;
        best = k;
      }
      if (!df_pos(w)) continue;
      lastpos = k;
      run = df_add(run, w);
      if (!last_mode && df_lt(tau_v, run)) {
        token = (int)(v * E::kVec + k);
        break;
      }
    }
    if (token < 0) token = (int)(v * E::kVec + (lastpos >= 0 ? lastpos : max(best, 0)));
  }
  return token;
}

template <typename E, bool kAligned>
__global__ void __launch_bounds__(kP2Threads) sv_accept_sample_kernel(AcceptArgs a) {
  extern __shared__ float4 s_vec[];
  __shared__ SampleSmem sm;
  cg::cluster_group cluster = cg::this_cluster();
  const int cs = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int b = blockIdx.x / cs;
  const int K = a.K;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;

  // wait for the streaming pass (and the visibility of its writes)
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const float T = __ldg(a.temperature + b);
  const bool greedy = (T == 0.f);
  if (threadIdx.x == 0) {
    int bad = valid_temperature(T) ? 0 : (int)kDevBadTemperature;
    for (int t = 0; t < K && !bad; ++t) {
      const int x = __ldg(a.tokens + (long long)b * K + t);
      if (x < 0 || x >= a.V) bad = (int)kDevBadToken;
    }
    sm.bad = bad;
  }
  __syncthreads();

  const long long tb = (long long)b * (K + 1);   // first target row of b
  const long long db = a.n_target_rows + (long long)b * K;  // first draft row of b (partials index)

  // fold the tile partials into row statistics; one warp per row
  const int nrows = greedy ? K + 1 : 2 * K + 1;
  const float c32 = greedy ? 0.f : __fdiv_rn(kLog2eHi, T);
  if (!sm.bad && (!greedy || rank == 0)) {
    for (int r = warp; r < nrows; r += kP2Warps) {
      const long long prow = (r <= K) ? tb + r : db + (r - K - 1);
      const float2* pp = a.partials + prow * a.tiles_per_row;
      if (greedy) {
        float best = SV_NEG_INF;
        int bi = 0x7fffffff;
        for (int i = lane; i < a.tiles_per_row; i += 32) {
          const float2 v = pp[i];
          const int idx = __float_as_int(v.y);
          if (v.x > best || (v.x == best && idx < bi)) {
            best = v.x;
            bi = idx;
          }
        }
        const float m = warp_max(best);
        const int idx = warp_min_int(best == m ? bi : 0x7fffffff);
        if (lane == 0) {
          sm.rowM[r] = m;
          sm.rowArg[r] = idx;
        }
      } else {
        float m = SV_NEG_INF;
        for (int i = lane; i < a.tiles_per_row; i += 32) m = fmaxf(m, pp[i].x);
        m = warp_max(m);
        float s = 0.f;
        for (int i = lane; i < a.tiles_per_row; i += 32) {
          const float2 v = pp[i];
          if (v.x != SV_NEG_INF) s += v.y * ex2_approx(__fmul_rn(__fsub_rn(v.x, m), c32));
        }
        s = warp_sum(s);
        if (lane == 0) {
          sm.rowM[r] = m;
          sm.rowS[r] = s;
        }
      }
    }
  }
  __syncthreads();

  // ---------------------------------------------------------------- accept scan
  const long long ob = (long long)b * (K + 1);
  if (threadIdx.x == 0) {
    int bad = sm.bad;
    int n = K;
    if (!bad) {
      for (int r = 0; r < nrows; ++r) {
        const bool ok = isfinite(sm.rowM[r]) && (greedy || (isfinite(sm.rowS[r]) && sm.rowS[r] > 0.f));
        if (!ok) bad = (int)kDevNonFinite;
      }
    }
    if (!bad && greedy && rank == 0) {
      // "Caso ganancioso": accept while argmax(p_t) == x_t
      for (int t = 0; t < K; ++t) {
        if (sm.rowArg[t] != __ldg(a.tokens + (long long)b * K + t)) {
          n = t;
          break;
        }
      }
    } else if (!bad && !greedy) {
      const char* tgt = (const char*)a.target;
      const char* drf = (const char*)a.draft;
      n = -1;
      for (int t = 0; t < K; ++t) {
        const int x = __ldg(a.tokens + (long long)b * K + t);
        const float xp = E::load_scalar(tgt, (tb + t) * (long long)a.V + x);
        const float xq = E::load_scalar(drf, ((long long)b * K + t) * (long long)a.V + x);
        // log p_t(x_t) = (z_x - m)/T - ln S
        const float lp = __fdiv_rn(__fsub_rn(xp, sm.rowM[t]), T) - logf(sm.rowS[t]);
        const float lq = __fdiv_rn(__fsub_rn(xq, sm.rowM[K + 1 + t]), T) - logf(sm.rowS[K + 1 + t]);
        if (rank == 0) {
          if (a.logp_out) a.logp_out[(long long)b * K + t] = lp;
          if (a.logq_out) a.logq_out[(long long)b * K + t] = lq;
        }
        if (n < 0) {
          const float r = __ldg(a.uniforms + ob + t);
          // r q < p  <=>  r < p / q = exp(log p - log q)
          if (!(r < expf(lp - lq))) n = t;
        }
      }
      if (n < 0) n = K;
    }
    if (bad && rank == 0) {
      atomicOr(a.err, (unsigned)bad);
      a.accepted_len[b] = -1;
      for (int t = 0; t <= K; ++t) a.out_tokens[ob + t] = -1;
    }
    if (rank == 0 && (bad || greedy)) {
      for (int t = 0; t < K; ++t) {
        if (a.logp_out) a.logp_out[(long long)b * K + t] = __int_as_float(0x7fffffff);
        if (a.logq_out) a.logq_out[(long long)b * K + t] = __int_as_float(0x7fffffff);
      }
    }
    if (!bad && rank == 0) {
      a.accepted_len[b] = n;
      for (int t = 0; t <= K; ++t) {
        int v = -1;
        if (t < n) v = __ldg(a.tokens + (long long)b * K + t);
        else if (t == n && greedy) v = sm.rowArg[n];
        a.out_tokens[ob + t] = v;
      }
    }
    sm.n = n;
    sm.bad = bad;
  }
  __syncthreads();
  if (sm.bad || greedy) return;   // uniform across the cluster; no shared memory was shared

  // ---------------------------------------------------------------- sampling
  const int n = sm.n;
  for (int i = threadIdx.x; i < 256; i += kP2Threads) sm.tab[i] = kExp2Table256[i];
  const long long rowbytes = (long long)a.V * E::kBytes;
  const char* rowP = (const char*)a.target + (tb + n) * rowbytes;
  const char* rowQ = (n < K) ? (const char*)a.draft + ((long long)b * K + n) * rowbytes : nullptr;
  const float Mp = sm.rowM[n];
  const float Sp32 = sm.rowS[n];
  const float Mq = (n < K) ? sm.rowM[K + 1 + n] : 0.f;
  const float Sq32 = (n < K) ? sm.rowS[K + 1 + n] : 1.f;
  const float c_used = __fdiv_rn(Sp32, Sq32);
  const float thp = kBigProb * Sp32;
  const float thq = kBigProb * Sq32;
  const DF L = log2e_over(T);
  const float u = __ldg(a.uniforms + ob + K);
  const int cv0 = rank * a.vecs_per_cta;
  const int ncv = max(0, min(a.nvec - cv0, a.vecs_per_cta));
  __syncthreads();

  bool residual = n < K;
  int token = -1;
  for (int attempt = 0; attempt < 2; ++attempt) {
    if (residual) {
      sweep_slice<E, kAligned, true>(rowP, rowQ, a.V, cv0, ncv, Mp, Mq, L, c_used, thp, thq, sm, s_vec);
    } else {
      sweep_slice<E, kAligned, false>(rowP, rowQ, a.V, cv0, ncv, Mp, Mq, L, c_used, thp, thq, sm, s_vec);
    }
    cluster.sync();
    if (threadIdx.x == 0) decide(cluster, cs, residual, c_used, u, a.vecs_per_cta, sm);
    cluster.sync();   // every record has been read; the smem may be reused
    if (sm.dec.need_p_fallback) {
      residual = false;   // "residual" identically zero: draw from p_t instead
      continue;
    }
    if (rank == sm.dec.rstar) {
      if (residual) {
        token = locate<E, kAligned, true>(rowP, rowQ, a.V, cv0, ncv, Mp, Mq, L, c_used, thp, thq, sm, s_vec);
      } else {
        token = locate<E, kAligned, false>(rowP, rowQ, a.V, cv0, ncv, Mp, Mq, L, c_used, thp, thq, sm, s_vec);
      }
      if (threadIdx.x == 0) a.out_tokens[ob + n] = token;
    }
    break;
  }
}

}  // namespace sv
