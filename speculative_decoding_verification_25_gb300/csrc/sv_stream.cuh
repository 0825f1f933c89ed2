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
//   With verified lengths per row (and B <= kCompactMaxB) many rows are not
//   read, and which ones lives on the device.  sv_row_stats_compact_kernel
//   then first counts, in every CTA, the rows read per segment (segment
//   b < B: target rows of batch row b; segment B + b: its draft rows), and
//   the warps split the tiles of those rows alone, in stacked order.
//   Without lengths (sv_row_stats_kernel) every warp takes a fixed share of
//   all tiles and skips the rows it need not read.
//
//   Both kernels may be launched before the preceding kernel on the stream
//   has finished; they wait for it before their first memory access.  Right
//   after that wait every CTA lets the next grid on the stream (the draw
//   launch of the same call) be scheduled, and block 0 clears the flag word
//   and the draw tickets.
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
// batches up to this size split only the rows that are read (compact order)
constexpr int kCompactMaxB = 2048;

struct RowStatsArgs {
  const void* target;
  const void* draft;
  const float* temperature;   // [B], or nullptr: every row greedy (T = 0)
  int B, K, V;
  int tiles_per_row;
  long long n_tiles;          // (B*(K+1) + B*K) * tiles_per_row
  int n_target_rows;          // B*(K+1)
  const int32_t* k_per_row;   // [B] drafted tokens each row verifies, or nullptr (all K)
  float2* partials;           // [n_target_rows + B*K][tiles_per_row]
  unsigned* err;
  unsigned* tickets;          // [n_tickets] cleared for the draw launch that follows, or nullptr
  int n_tickets;
};

// Clear the device flag word and the draw launch's tickets (block 0).  The
// preceding kernel has completed (the caller waited for it), and the draw
// launch that reads them runs after this grid.
__device__ __forceinline__ void clear_control(const RowStatsArgs& a) {
  if (blockIdx.x != 0) return;
  if (threadIdx.x == 0) *a.err = 0u;
  for (int i = threadIdx.x; i < a.n_tickets; i += blockDim.x) a.tickets[i] = 0u;
}

// Checked build: an index test guarding one access (always true, and
// compiled away, in the plain build).
__device__ __forceinline__ bool rs_in_bounds(const RowStatsArgs& a, bool ok) {
  if (kChecked && !ok) {
    atomicOr(a.err, kDevOutOfBounds);
    return false;
  }
  return true;
}
__device__ __forceinline__ int rs_rows(const RowStatsArgs& a) {
  return a.n_target_rows + (a.draft ? a.B * a.K : 0);
}

// float32 c = log2(e)/T, the same in both kernels
__device__ __forceinline__ float log2e_over_f(float T) { return __fdiv_rn(kLog2eHi, T); }


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
  // new lane shift (no branches): a tile whose max is not above the shift
  // leaves it and the sum as they are; an all -inf tile adds zeros
  const float tmc = __fmul_rn(m, c);
  const float mc1 = fmaxf(st.mc, tmc);
  st.s *= (mc1 == st.mc) ? 1.f : ex2_approx(__fsub_rn(st.mc, mc1));
  st.mc = mc1;
  const float nmc = (mc1 == SV_NEG_INF) ? 0.f : -mc1;
  // four running sums (elements k mod 4), two per paired instruction; each
  // half rounds as the scalar FFMA / FADD would
  const unsigned long long c2 = f2_pack(c, c), nmc2 = f2_pack(nmc, nmc);
  unsigned long long s01 = 0ull, s23 = 0ull;
#pragma unroll
  for (int j = 0; j < kTileVecsPerLane; ++j) {
#pragma unroll
    for (int k = 0; k < E::kVec; k += 4) {
      float y0, y1, y2, y3;
      f2_unpack(f2_fma(f2_pack(E::elem(w[j], k + 0), E::elem(w[j], k + 1)), c2, nmc2), y0, y1);
      f2_unpack(f2_fma(f2_pack(E::elem(w[j], k + 2), E::elem(w[j], k + 3)), c2, nmc2), y2, y3);
      s01 = f2_add(s01, f2_pack(ex2_approx(y0), ex2_approx(y1)));
      s23 = f2_add(s23, f2_pack(ex2_approx(y2), ex2_approx(y3)));
    }
  }
  float a0, a1, a2, a3;
  f2_unpack(s01, a0, a1);
  f2_unpack(s23, a2, a3);
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

// Everything a warp needs about the rows its range touches.  Lane i holds
// the temperature (and verified length) of the range's i-th row's batch
// row; later rows (ranges over 32 rows long, tiny vocabularies only) read
// theirs when they are reached.
struct WarpRows {
  const RowStatsArgs* a;
  long long t1;        // end of the range (stacked tile index)
  int row0;            // first row of the range
  float T_lane;
  int kb_lane;
  unsigned act_mask;   // bit i: row row0 + i is read (i < 32)

  __device__ __forceinline__ int batch_of(int row) const {
    return row < a->n_target_rows ? row / (a->K + 1) : (row - a->n_target_rows) / a->K;
  }
  __device__ __forceinline__ int kb_of_batch(int b) const {
    return a->k_per_row ? __ldg(a->k_per_row + b) : a->K;
  }
  __device__ __forceinline__ float T_of(int row) const {   // warp-uniform call
    const int d = row - row0;
    const float t = __shfl_sync(0xffffffffu, T_lane, d & 31);
    return d < 32 ? t : (a->temperature ? __ldg(a->temperature + batch_of(row)) : 0.f);
  }
  // Is the row read?  Target rows 0..K_b and, for T > 0, draft rows
  // 0..K_b-1 of a batch row with a valid temperature and 0 <= K_b <= K.
  __device__ __forceinline__ bool row_read(int row, float T, int kb) const {
    const bool draft = row >= a->n_target_rows;
    const int b = batch_of(row);
    const int pos = draft ? row - a->n_target_rows - b * a->K : row - b * (a->K + 1);
    return valid_temperature(T) && !(draft && T == 0.f) && kb >= 0 && kb <= a->K &&
           (draft ? pos < kb : pos <= kb);
  }
  __device__ __forceinline__ bool active(int row) const {   // warp-uniform call
    const int d = row - row0;
    if (d < 32) return ((act_mask >> d) & 1u) != 0u;
    return row_read(row, T_of(row), kb_of_batch(batch_of(row)));
  }
  __device__ __forceinline__ const char* rowp(int row, int elem_bytes) const {
    const bool d = row >= a->n_target_rows;
    const long long r = d ? row - a->n_target_rows : row;
    return (const char*)(d ? a->draft : a->target) + r * a->V * elem_bytes;
  }
};

// A position in a warp's range: stacked tile index t, its row and its tile
// within the row (kept in step without divisions).
struct TilePos {
  long long t;
  int row, ti;
  // move forward to the first tile of an active row at or after this one
  // (t = t1 if there is none)
  __device__ __forceinline__ void settle(const WarpRows& wr) {
    const int tpr = wr.a->tiles_per_row;
    while (t < wr.t1 && !wr.active(row)) {
      t += tpr - ti;
      ti = 0;
      ++row;
    }
    if (t > wr.t1) t = wr.t1;
  }
  __device__ __forceinline__ TilePos next(const WarpRows& wr) const {
    TilePos p = *this;
    ++p.t;
    if (++p.ti == wr.a->tiles_per_row) {
      p.ti = 0;
      ++p.row;
    }
    p.settle(wr);
    return p;
  }
};

// The open row stretch of a warp: which row, its first tile, its parameters.
struct Stretch {
  int row, first;
  bool greedy;
  float c;
  LaneStats st;
  __device__ __forceinline__ void open(const WarpRows& wr, int r, int ti) {
    row = r;
    first = ti;
    const float T = wr.T_of(r);
    greedy = (T == 0.f);
    c = greedy ? 0.f : log2e_over_f(T);
    st.reset();
  }
};

template <typename E, bool kAligned>
__device__ __forceinline__ void load_at(uint32_t (&w)[kTileVecsPerLane][4], const WarpRows& wr,
                                        const TilePos& p, int lane, int full_end) {
  const bool ok = rs_in_bounds(*wr.a, p.row >= 0 && p.row < rs_rows(*wr.a) && p.ti >= 0 &&
                                          p.ti < wr.a->tiles_per_row);
  load_tile<E, kAligned>(w, wr.rowp(p.row, E::kBytes), p.ti, lane, wr.a->V, p.ti < full_end, ok);
}

// Fold the tile at t (its data in w) into the open stretch; if the next tile
// `nt` of the sequence is in another row (or past the end), write the
// stretch's partials and open the next one.
template <typename E>
__device__ __forceinline__ void fold_at(const uint32_t (&w)[kTileVecsPerLane][4], const WarpRows& wr,
                                        const TilePos& p, const TilePos& np, int lane, Stretch& sr) {
  fold_tile<E>(w, (long long)p.ti * kTileVecs + lane, sr.greedy, sr.c, sr.st);
  const bool more = np.t < wr.t1;
  if (!more || np.row != p.row) {
    if (rs_in_bounds(*wr.a, p.row >= 0 && p.row < rs_rows(*wr.a) && sr.first >= 0 &&
                                p.ti < wr.a->tiles_per_row))
      flush_stretch(wr.a->partials + (long long)p.row * wr.a->tiles_per_row, sr.first, p.ti,
                    sr.greedy, lane, sr.st);
    if (more) sr.open(wr, np.row, np.ti);
  }
}

// ------------------------------------------------------- compact order
// Rows read in segment s: s < B target rows 0..K_b of batch row s; s >= B
// draft rows 0..K_b-1 of batch row s - B (tempered rows only).  A batch row
// with an invalid temperature or K_b outside [0, K] reads nothing.
__device__ __forceinline__ int segment_rows(const RowStatsArgs& a, int s) {
  const bool draft = s >= a.B;
  const int b = draft ? s - a.B : s;
  const float T = a.temperature ? __ldg(a.temperature + b) : 0.f;
  const int kb = a.k_per_row ? __ldg(a.k_per_row + b) : a.K;
  if (!valid_temperature(T) || kb < 0 || kb > a.K) return 0;
  if (draft) return T == 0.f ? 0 : kb;
  return kb + 1;
}
__device__ __forceinline__ int segment_row(const RowStatsArgs& a, int s, int r) {
  return s < a.B ? s * (a.K + 1) + r : a.n_target_rows + (s - a.B) * a.K + r;
}

// pref[s] = rows read in segments before s, pref[2B] = all of them (every
// thread of the CTA calls this)
__device__ __forceinline__ void segment_prefix(const RowStatsArgs& a, int* pref, int* wsum) {
  const int nseg = 2 * a.B;
  const int per = (nseg + (int)blockDim.x - 1) / (int)blockDim.x;
  const int s0 = min((int)threadIdx.x * per, nseg), s1 = min(s0 + per, nseg);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int sum = 0;
  for (int s = s0; s < s1; ++s) sum += segment_rows(a, s);
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int run = incl - sum;
  for (int w = 0; w < warp; ++w) run += wsum[w];
  for (int s = s0; s < s1; ++s) {
    pref[s] = run;
    run += segment_rows(a, s);
  }
  if (threadIdx.x == blockDim.x - 1) pref[nseg] = run;
  __syncthreads();
}

// A position in a warp's range of the compact order: tile index t among the
// tiles read, its segment, row within the segment, tile within the row.
struct CompactPos {
  long long t;
  int seg, r, ti, row;
  __device__ __forceinline__ CompactPos next(const RowStatsArgs& a, const int* pref) const {
    CompactPos p = *this;
    ++p.t;
    if (++p.ti == a.tiles_per_row) {
      p.ti = 0;
      ++p.r;
      const int nseg = 2 * a.B;
      while (p.seg < nseg && p.r == pref[p.seg + 1] - pref[p.seg]) {
        ++p.seg;
        p.r = 0;
      }
      p.row = p.seg < nseg ? segment_row(a, p.seg, p.r) : -1;
    }
    return p;
  }
};

__device__ __forceinline__ const char* stacked_rowp(const RowStatsArgs& a, int row, int elem_bytes) {
  const bool d = row >= a.n_target_rows;
  const long long r = d ? row - a.n_target_rows : row;
  return (const char*)(d ? a.draft : a.target) + r * a.V * elem_bytes;
}

__device__ __forceinline__ void open_compact(const RowStatsArgs& a, const CompactPos& p, Stretch& sr) {
  sr.row = p.row;
  sr.first = p.ti;
  const int b = p.seg < a.B ? p.seg : p.seg - a.B;
  const float T = a.temperature ? __ldg(a.temperature + b) : 0.f;
  sr.greedy = (T == 0.f);
  sr.c = sr.greedy ? 0.f : log2e_over_f(T);
  sr.st.reset();
}

template <typename E>
__device__ __forceinline__ void fold_compact(const uint32_t (&w)[kTileVecsPerLane][4],
                                             const RowStatsArgs& a, const CompactPos& p,
                                             const CompactPos& np, long long t1, int lane,
                                             Stretch& sr) {
  fold_tile<E>(w, (long long)p.ti * kTileVecs + lane, sr.greedy, sr.c, sr.st);
  const bool more = np.t < t1;
  if (!more || np.row != p.row) {
    if (rs_in_bounds(a, p.row >= 0 && p.row < rs_rows(a) && sr.first >= 0 && p.ti < a.tiles_per_row))
      flush_stretch(a.partials + (long long)p.row * a.tiles_per_row, sr.first, p.ti, sr.greedy,
                    lane, sr.st);
    if (more) open_compact(a, np, sr);
  }
}

// The tiles of one warp in the compact order (n_read rows are read).
template <typename E, bool kAligned>
__device__ __forceinline__ void stream_compact(const RowStatsArgs& a, const int* pref, int n_read, long long gw,
                               long long nw, int lane, int full_end) {
  const int tpr = a.tiles_per_row;
  const long long total = (long long)n_read * tpr;
  const long long t0 = gw * total / nw, t1 = (gw + 1) * total / nw;
  if (t0 >= t1) return;
  const int cr = (int)(t0 / tpr);
  // the segment holding compact row cr: the last s with pref[s] <= cr
  int lo = 0, hi = 2 * a.B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pref[mid] <= cr) lo = mid;
    else hi = mid;
  }
  CompactPos pa;
  pa.t = t0;
  pa.seg = lo;
  pa.r = cr - pref[lo];
  pa.ti = (int)(t0 - (long long)cr * tpr);
  pa.row = segment_row(a, pa.seg, pa.r);
  uint32_t wa[kTileVecsPerLane][4], wb[kTileVecsPerLane][4];
  load_tile<E, kAligned>(wa, stacked_rowp(a, pa.row, E::kBytes), pa.ti, lane, a.V, pa.ti < full_end,
                         rs_in_bounds(a, pa.row >= 0 && pa.row < rs_rows(a) && pa.ti < a.tiles_per_row));
  Stretch sr;
  open_compact(a, pa, sr);
  for (;;) {
    const CompactPos pb = pa.next(a, pref);
    if (pb.t < t1)
      load_tile<E, kAligned>(wb, stacked_rowp(a, pb.row, E::kBytes), pb.ti, lane, a.V, pb.ti < full_end,
                             rs_in_bounds(a, pb.row >= 0 && pb.row < rs_rows(a) && pb.ti < a.tiles_per_row));
    fold_compact<E>(wa, a, pa, pb, t1, lane, sr);
    if (pb.t >= t1) break;
    pa = pb.next(a, pref);
    if (pa.t < t1)
      load_tile<E, kAligned>(wa, stacked_rowp(a, pa.row, E::kBytes), pa.ti, lane, a.V, pa.ti < full_end,
                         rs_in_bounds(a, pa.row >= 0 && pa.row < rs_rows(a) && pa.ti < a.tiles_per_row));
    fold_compact<E>(wb, a, pb, pa, t1, lane, sr);
    if (pa.t >= t1) break;
  }
}

template <typename E, bool kAligned>
__global__ void __launch_bounds__(kP1Threads, 4) sv_row_stats_compact_kernel(RowStatsArgs a) {
  wait_for_preceding_grid();   // before any access: the previous step may still read the workspace
  allow_dependent_launch();
  clear_control(a);
  __shared__ int s_pref[2 * kCompactMaxB + 1];
  __shared__ int s_wsum[kP1Threads / 32];
  segment_prefix(a, s_pref, s_wsum);
  const int tpr = a.tiles_per_row;
  const int full_end = ((long long)tpr * kTileVecs * E::kVec == a.V) ? tpr : tpr - 1;
  stream_compact<E, kAligned>(a, s_pref, s_pref[2 * a.B],
                              ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5,
                              ((long long)gridDim.x * blockDim.x) >> 5, threadIdx.x & 31, full_end);
}

template <typename E, bool kAligned>
__global__ void __launch_bounds__(kP1Threads, 4) sv_row_stats_kernel(RowStatsArgs a) {
  wait_for_preceding_grid();   // before any access: the previous step may still read the workspace
  allow_dependent_launch();
  clear_control(a);

  const int lane = threadIdx.x & 31;
  const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
  const long long t0 = gw * a.n_tiles / nw;
  const long long t1 = (gw + 1) * a.n_tiles / nw;
  if (t0 >= t1) return;
  const int tpr = a.tiles_per_row;
  // tiles below full_end lie wholly inside the row (the last one may be ragged)
  const int full_end = ((long long)tpr * kTileVecs * E::kVec == a.V) ? tpr : tpr - 1;

  WarpRows wr;
  wr.a = &a;
  wr.t1 = t1;
  wr.row0 = (int)(t0 / tpr);
  TilePos pa;
  pa.t = t0;
  pa.row = wr.row0;
  pa.ti = (int)(t0 - (long long)wr.row0 * tpr);
  // the first tile's loads go out before the row's temperature is known
  // (they are repeated elsewhere in the rare case its row is not read)
  uint32_t wa[kTileVecsPerLane][4], wb[kTileVecsPerLane][4];
  load_at<E, kAligned>(wa, wr, pa, lane, full_end);
  const int row_last = (int)((t1 - 1) / tpr);
  const bool lane_row = wr.row0 + lane <= row_last;
  const int lane_b = lane_row ? wr.batch_of(wr.row0 + lane) : 0;
  wr.T_lane = (lane_row && a.temperature) ? __ldg(a.temperature + lane_b) : 0.f;
  wr.kb_lane = lane_row ? wr.kb_of_batch(lane_b) : 0;
  wr.act_mask = __ballot_sync(0xffffffffu,
                              lane_row && wr.row_read(wr.row0 + lane, wr.T_lane, wr.kb_lane));

  // one register ping-pong over the warp's active tiles, across row
  // boundaries: the next tile's loads are always in flight while the
  // current one is folded
  pa.settle(wr);
  if (pa.t >= t1) return;
  if (pa.t != t0) load_at<E, kAligned>(wa, wr, pa, lane, full_end);
  Stretch sr;
  sr.open(wr, pa.row, pa.ti);
  for (;;) {
    const TilePos pb = pa.next(wr);
    if (pb.t < t1) load_at<E, kAligned>(wb, wr, pb, lane, full_end);
    fold_at<E>(wa, wr, pa, pb, lane, sr);
    if (pb.t >= t1) break;
    pa = pb.next(wr);
    if (pa.t < t1) load_at<E, kAligned>(wa, wr, pa, lane, full_end);
    fold_at<E>(wb, wr, pb, pa, lane, sr);
    if (pa.t >= t1) break;
  }
}

}  // namespace sv
