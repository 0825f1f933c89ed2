// The streaming kernel of spec_verify (row statistics).
//
//   Row statistics (the streaming pass) reads every logit row once.  Each
//   warp streams a contiguous range of 2 KB row tiles (16 bytes per lane per
//   load, the next tile in flight while the current one is reduced) and
//   writes one partial per tile:
//     tempered rows:  (MC, S) with S = sum of 2^(x*c - MC), c = log2(e)/T
//                     rounded to float32 and MC a float32 shift >= max x*c;
//     greedy rows:    (max logit, ~(lowest index holding it)), the index
//                     stored complemented (no written partial is all-zero
//                     bits).
//   A lane folds its tiles into running values and the warp reduces them
//   only where its range leaves a row; the other tiles of that stretch get
//   the neutral partial (-inf, 0).  Draft rows of greedy rows are not read.
//
// The softmax normalisers are those of the rule's p_t = softmax(target / T)
// and q_t = softmax(draft / T) in the lesson "Decodificação Especulativa e
// EAGLE" (ai-engineering.academy, phase 10 lesson 25), section "A Regra de
// Exatidão"; the greedy maxima are those of its section "Caso ganancioso".
#pragma once

#include "sv_common.cuh"

namespace sv {

constexpr int kMaxK = 16;
constexpr int kTileVecsPerLane = 4;               // 4 x 16 B per lane
constexpr int kTileVecs = 32 * kTileVecsPerLane;  // one 2 KB tile of one row
constexpr int kP1Threads = 256;


struct RowStatsArgs {
  const void* target;
  const void* draft;
  const float* temperature;
  int B, K, V;
  int tiles_per_row;
  long long n_tiles;          // (B*(K+1) + B*K) * tiles_per_row
  int n_target_rows;          // B*(K+1)
  float2* partials;           // [n_target_rows + B*K][tiles_per_row]
  unsigned* err;
};

// float32 c = log2(e)/T, the same in both kernels
__device__ __forceinline__ float log2e_over_f(float T) { return __fdiv_rn(kLog2eHi, T); }

// Row `row` of the stacked [target rows; draft rows] and its batch row.
__device__ __forceinline__ void row_info(const RowStatsArgs& a, int row, int& b, bool& is_draft,
                                         int& r) {
  is_draft = row >= a.n_target_rows;
  r = is_draft ? row - a.n_target_rows : row;
  b = is_draft ? r / a.K : r / (a.K + 1);
}

// ============================================================== streaming pass
// One tile of one lane: kTileVecsPerLane 16-byte vectors, 512 bytes apart.
template <typename E, bool kAligned>
__device__ __forceinline__ void load_tile(uint32_t (&w)[kTileVecsPerLane][4], const char* rowp,
                                          int ti, int lane, int V, bool full, bool act) {
  if (!act) {
#pragma unroll
    for (int j = 0; j < kTileVecsPerLane; ++j) w[j][0] = w[j][1] = w[j][2] = w[j][3] = E::kFillWord;
    return;
  }
  if (kAligned && full) {
    // a whole tile inside the row: one base pointer, immediate offsets
    const uint4* p = reinterpret_cast<const uint4*>(rowp) + (long long)ti * kTileVecs + lane;
#pragma unroll
    for (int j = 0; j < kTileVecsPerLane; ++j) ldg_stream16(p + 32 * j, w[j]);
  } else {
    const long long v0 = (long long)ti * kTileVecs + lane;
#pragma unroll
    for (int j = 0; j < kTileVecsPerLane; ++j) load_vec<E, kAligned>(rowp, v0 + 32 * j, V, w[j]);
  }
}

// Running per-lane values of a row stretch.
struct LaneStats {
  float mc, s;       // tempered rows: shift (c-scaled) and sum of 2^(x c - mc)
  float best;        // greedy rows: max logit ...
  int bi;            // ... and its lowest index
  __device__ __forceinline__ void reset() {
    mc = SV_NEG_INF;
    s = 0.f;
    best = SV_NEG_INF;
    bi = 0x7fffffff;
  }
};

template <typename E>
__device__ __forceinline__ void fold_tile(const uint32_t (&w)[kTileVecsPerLane][4], long long v0,
                                          bool greedy, float c, LaneStats& st) {
  if (greedy) {
#pragma unroll
    for (int j = 0; j < kTileVecsPerLane; ++j) {
#pragma unroll
      for (int k = 0; k < E::kVec; ++k) {
        const float x = E::elem(w[j], k);
        if (x > st.best) {
          st.best = x;
          st.bi = (int)((v0 + 32 * j) * E::kVec + k);
        }
      }
    }
    return;
  }
  // lane max of the tile, then one FFMA + ex2 + add per element
  float m;
  if constexpr (E::kBytes == 2) {
    uint32_t mm = 0xff80ff80u;
#pragma unroll
    for (int j = 0; j < kTileVecsPerLane; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) mm = bf2_max(mm, w[j][i]);
    m = fmaxf(__uint_as_float(mm << 16), __uint_as_float(mm & 0xffff0000u));
  } else {
    m = SV_NEG_INF;
#pragma unroll
    for (int j = 0; j < kTileVecsPerLane; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) m = fmaxf(m, __uint_as_float(w[j][i]));
  }
  if (m == SV_NEG_INF) return;
  const float tmc = __fmul_rn(m, c);
  if (tmc > st.mc) {   // new lane shift: rescale what was summed so far
    st.s *= ex2_approx(__fsub_rn(st.mc, tmc));
    st.mc = tmc;
  }
  const float nmc = -st.mc;
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
  for (int j = 0; j < kTileVecsPerLane; ++j) {
#pragma unroll
    for (int k = 0; k < E::kVec; k += 4) {
      a0 += ex2_approx(__fmaf_rn(E::elem(w[j], k + 0), c, nmc));
      a1 += ex2_approx(__fmaf_rn(E::elem(w[j], k + 1), c, nmc));
      a2 += ex2_approx(__fmaf_rn(E::elem(w[j], k + 2), c, nmc));
      a3 += ex2_approx(__fmaf_rn(E::elem(w[j], k + 3), c, nmc));
    }
  }
  st.s += (a0 + a1) + (a2 + a3);
}

// Warp-combine the lane values of a finished row stretch [first, last] and
// write its partials: the combined one at `last`, neutral ones before it.
__device__ __forceinline__ void flush_stretch(float2* pp, int first, int last, bool greedy,
                                              int lane, const LaneStats& st) {
  float2 part;
  if (greedy) {
    const float m = warp_max(st.best);
    const int idx = warp_min_int(st.best == m ? st.bi : 0x7fffffff);
    part = make_float2(m, __int_as_float(~idx));
  } else {
    const float M = warp_max(st.mc);
    float sv = (st.mc == SV_NEG_INF) ? 0.f : st.s * ex2_approx(__fsub_rn(st.mc, M));
    sv = warp_sum(sv);
    part = make_float2(M, sv);
  }
  const float2 neutral = make_float2(SV_NEG_INF, greedy ? __int_as_float(~0x7fffffff) : 0.f);
  for (int k = first + lane; k <= last; k += 32) pp[k] = (k == last) ? part : neutral;
}

// Parameters of one row of the stacked [target rows; draft rows].
struct RowParams {
  bool active, greedy;
  float c;
  const char* rowp;
  RowParams() = default;
  __device__ __forceinline__ RowParams(const RowStatsArgs& a, int row, int elem_bytes) {
    int b, r;
    bool is_draft;
    row_info(a, row, b, is_draft, r);
    const float T = __ldg(a.temperature + b);
    greedy = (T == 0.f);
    active = valid_temperature(T) && !(is_draft && greedy);
    c = greedy ? 0.f : log2e_over_f(T);
    rowp = (const char*)(is_draft ? a.draft : a.target) + (long long)r * a.V * elem_bytes;
  }
};

// Fold tiles [ti0, ti1) of one row into `st`, two tiles per trip with the
// next tile's loads in flight while the current one is folded.
template <typename E, bool kAligned, bool kGreedy>
__device__ __forceinline__ void fold_stretch(const RowParams& rp, int ti0, int ti1, int lane, int V,
                                             int full_end, LaneStats& st) {
  uint32_t wa[kTileVecsPerLane][4], wb[kTileVecsPerLane][4];
  load_tile<E, kAligned>(wa, rp.rowp, ti0, lane, V, ti0 < full_end, true);
  for (int ti = ti0; ti < ti1; ti += 2) {
    const bool has1 = ti + 1 < ti1;
    if (has1) load_tile<E, kAligned>(wb, rp.rowp, ti + 1, lane, V, ti + 1 < full_end, true);
    fold_tile<E>(wa, (long long)ti * kTileVecs + lane, kGreedy, rp.c, st);
    if (!has1) break;
    if (ti + 2 < ti1) load_tile<E, kAligned>(wa, rp.rowp, ti + 2, lane, V, ti + 2 < full_end, true);
    fold_tile<E>(wb, (long long)(ti + 1) * kTileVecs + lane, kGreedy, rp.c, st);
  }
}

template <typename E, bool kAligned>
__global__ void __launch_bounds__(kP1Threads, 4) sv_row_stats_kernel(RowStatsArgs a) {
  if (blockIdx.x == 0 && threadIdx.x == 0) *a.err = 0u;

  const int lane = threadIdx.x & 31;
  const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
  const long long t0 = gw * a.n_tiles / nw;
  const long long t1 = (gw + 1) * a.n_tiles / nw;
  const int tpr = a.tiles_per_row;
  // tiles below full_end lie wholly inside the row (the last one may be ragged)
  const int full_end = ((long long)tpr * kTileVecs * E::kVec == a.V) ? tpr : tpr - 1;

  // the warp's range crosses a few rows: one stretch per row
  for (long long tile = t0; tile < t1;) {
    const int row = (int)(tile / tpr);
    const int ti0 = (int)(tile - (long long)row * tpr);
    const int ti1 = (int)min((long long)tpr, ti0 + (t1 - tile));
    const RowParams rp(a, row, E::kBytes);
    if (rp.active) {
      LaneStats st;
      st.reset();
      if (rp.greedy) fold_stretch<E, kAligned, true>(rp, ti0, ti1, lane, a.V, full_end, st);
      else fold_stretch<E, kAligned, false>(rp, ti0, ti1, lane, a.V, full_end, st);
      flush_stretch(a.partials + (long long)row * tpr, ti0, ti1 - 1, rp.greedy, lane, st);
    }
    tile += ti1 - ti0;
  }
}

}  // namespace sv
