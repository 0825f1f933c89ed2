// The verify-and-accept step as one persistent kernel.
//
// The rule is the exact rejection rule of the lesson "Decodificação
// Especulativa e EAGLE" (ai-engineering.academy, phase 10 lesson 25),
// sections "A Regra de Exatidão" (test r q < p, residual (p - q)+ over the
// full vocabulary, bonus token from p_K) and "Caso ganancioso" (T = 0:
// argmax).  Every warp of the grid runs two phases.
//
//   Phase 1, streaming.  The logit rows are taken in batch-major order
//   (batch row b: its target rows 0..K, then its draft rows 0..K-1) and cut
//   into chunks of kChunkTiles 2 KB tiles; chunk c goes to warp c mod W.  All
//   warps therefore work on a narrow window of batch rows at any moment, and
//   the rows of batch row b are complete soon after the window passes it.
//   A warp reduces its chunk to one partial -- (shift MC, sum of
//   2^(x c - MC)) for a tempered row, (max, ~lowest argmax) for a greedy one
//   -- and takes a ticket on the row.  The warp holding the row's last
//   ticket folds the row's partials into its statistics and gathers the
//   logit at the drafted token; the warp that folds the last row of a batch
//   row runs the acceptance scan for it (one lane per drafted position),
//   writes its outputs, and for a tempered row publishes what the sampling
//   needs.
//
//   Phase 2, sampling.  Warps claim items (batch row b, tile j) in order.
//   For a tempered row the item waits until the row is published, then
//   weighs the tile of the sampled position -- residual w = max(p - q, 0) at
//   a rejection, w = p for the bonus -- and writes the tile's totals.  The
//   warp that completes a row's last item locates the token: tile by the
//   prefix of the tile totals, element by a scan inside that tile (re-read
//   once more).
//
// Hand-offs between warps carry no fences in phase 1: every partial and
// every row record is a 64-bit word that is never all-zero once written,
// the slots are zero between calls, and the reader re-reads a zero slot
// until the writer's store lands.  Phase 2 records are ordered by a fence
// before each ticket.  Every wait is bounded: past kSpinLimit polls the
// kernel sets kDevTimeout and carries on.  A warp waits only once every CTA
// of the grid has started, so no wait can hold a slot that an unstarted
// CTA with streaming work needs.
//
// Every counter, flag and slot of the workspace is returned to zero by its
// last user, and the last warp to finish resets the grid counters: a zeroed
// workspace stays zeroed between calls (the flag word at offset 0 then holds
// the call's device flags).
#pragma once

#include "sv_sample.cuh"

#ifndef SV_CHUNK_TILES
#define SV_CHUNK_TILES 4
#endif

namespace sv {

constexpr int kFThreads = 256;
constexpr int kFWarps = kFThreads / 32;
constexpr int kChunkTiles = SV_CHUNK_TILES;
constexpr int kFBigCap = 64;                 // large terms listed per warp per tile
constexpr unsigned kDevTimeout = 128u;
constexpr unsigned kSpinLimit = 1u << 20;    // polls (each sleeping ~0.1 us) before a wait gives up

// Grid control words at workspace offset 0.
struct FusedHeader {
  unsigned err;         // device flags of the last completed call
  unsigned err_accum;   // flags OR-ed during a call
  unsigned claim;       // next phase-2 item
  unsigned exited;      // warps that have finished
  unsigned arrived;     // CTAs that have started
};

// What the acceptance scan publishes for a tempered row that needs a draw.
struct RowState {
  int n;        // sampled position
  int kind;     // 1 residual (n < K_b), 2 bonus (n == K_b)
  float MCp, Sp, MCq, Sq, u, T;
};

struct FusedArgs {
  const void* target;
  const void* draft;
  const int32_t* tokens;
  const float* uniforms;
  const float* temperature;
  const int32_t* k_per_row;       // [B] or nullptr (every row verifies K)
  int B, K, V;
  int tpr;                        // 2 KB tiles per row
  int cpr;                        // chunks per row
  int n_target_rows;              // B*(K+1)
  long long n_chunks;             // B*(2K+1)*cpr
  long long n_items;              // B*tpr
  FusedHeader* hdr;
  unsigned* fold_ticket;          // [B*(2K+1)] per stacked row: chunks done
  unsigned* scan_ticket;          // [B] rows folded
  unsigned* samp_ticket;          // [B] phase-2 items done
  unsigned* ready;                // [B] 0, or 1/2 (RowState.kind), or 3 (no draw)
  RowState* rowstate;             // [B]
  unsigned long long* rowstat;    // [B*(2K+1)][2]: statistics word, token word
  unsigned long long* partials;   // [B*(2K+1)][cpr]
  float4* recs;                   // [B][tpr][2]: (W, Q), (Sp, Sq) as double-floats
  int32_t* accepted_len;
  int32_t* out_tokens;
  float* logp_out;
  float* logq_out;
  int32_t* plug_tokens;           // plug step fused in (nullptr: none)
  int32_t* plug_seq_len;
  int32_t* plug_last;
  int plug_max_len;
};

struct FusedSmem {
  float2 tab[256];
  uint32_t bigpos[kFWarps][kFBigCap];
};

// ---------------------------------------------------------------- memory ops
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned atom_add_u32(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.relaxed.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
  return (unsigned long long)__float_as_uint(lo) | ((unsigned long long)__float_as_uint(hi) << 32);
}
__device__ __forceinline__ float2 unpack2(unsigned long long v) {
  return make_float2(__uint_as_float((unsigned)v), __uint_as_float((unsigned)(v >> 32)));
}

__device__ __forceinline__ void flag(const FusedArgs& a, unsigned f) { atomicOr(&a.hdr->err_accum, f); }

// Has any wait of this call given up?  Then every other wait gives up at
// once too, so a call never spends more than about one wait limit.
__device__ __forceinline__ bool gave_up(const FusedArgs& a) {
  return (ld_relaxed_u32(&a.hdr->err_accum) & kDevTimeout) != 0u;
}
__device__ __forceinline__ bool stop_waiting(const FusedArgs& a, unsigned spins) {
  return spins >= kSpinLimit || ((spins & 255u) == 255u && gave_up(a));
}

// Re-read a 64-bit slot until its writer's store has landed (non-zero).
__device__ __forceinline__ unsigned long long wait_word(const FusedArgs& a, const unsigned long long* p,
                                                        bool& timeout) {
  unsigned long long v = ld_relaxed_u64(p);
  for (unsigned spins = 0; v == 0ull; ++spins) {
    if (stop_waiting(a, spins)) {
      timeout = true;
      flag(a, kDevTimeout);
      break;
    }
    __nanosleep(64);
    v = ld_relaxed_u64(p);
  }
  return v;
}

// ---------------------------------------------------------------- rows
// A logit row in batch-major order R = b*(2K+1) + k: target position k for
// k <= K, draft position k-K-1 after that.  Its stacked index srow (target
// rows b*(K+1)+pos first, then draft rows B*(K+1) + b*K + pos) addresses the
// partials and the statistics.

__device__ __forceinline__ int kb_of(const FusedArgs& a, int b) {
  return a.k_per_row ? __ldg(a.k_per_row + b) : a.K;
}

// Rows a valid batch row reads: target 0..K_b, and draft 0..K_b-1 if tempered.
__device__ __forceinline__ int rows_read(int kb, bool greedy) { return kb + 1 + (greedy ? 0 : kb); }

template <typename E>
__device__ __forceinline__ const char* srow_ptr(const FusedArgs& a, int srow) {
  const bool d = srow >= a.n_target_rows;
  const long long r = d ? srow - a.n_target_rows : srow;
  return (const char*)(d ? a.draft : a.target) + r * (long long)a.V * E::kBytes;
}

// batch row and position of a stacked row
__device__ __forceinline__ void srow_split(const FusedArgs& a, int srow, int& b, int& pos, bool& draft) {
  draft = srow >= a.n_target_rows;
  if (draft) {
    const int r = srow - a.n_target_rows;
    b = r / a.K;
    pos = r - b * a.K;
  } else {
    b = srow / (a.K + 1);
    pos = srow - b * (a.K + 1);
  }
}

// A warp's place in phase 1: chunk c (c >= n_chunks: none), tile t of the
// stacked row srow, and the row's c = log2(e)/T (0 for a greedy row).
struct FPos {
  long long c;
  int t, srow;
  float cs;
};

// The first chunk at or after c (step W) whose row is read.
__device__ __forceinline__ FPos first_read_chunk(const FusedArgs& a, long long c, long long W) {
  FPos p;
  p.t = 0;
  p.srow = 0;
  p.cs = 0.f;
  const int per = 2 * a.K + 1;
  for (; c < a.n_chunks; c += W) {
    const int R = (int)(c / a.cpr);
    const int b = R / per;
    const int k = R - b * per;
    const bool draft = k > a.K;
    const int pos = draft ? k - a.K - 1 : k;
    const float T = __ldg(a.temperature + b);
    const int kb = kb_of(a, b);
    const bool greedy = (T == 0.f);
    if (valid_temperature(T) && kb >= 0 && kb <= a.K &&
        (draft ? (!greedy && pos < kb) : pos <= kb)) {
      p.t = (int)(c - (long long)R * a.cpr) * kChunkTiles;
      p.srow = draft ? a.n_target_rows + b * a.K + pos : b * (a.K + 1) + pos;
      p.cs = greedy ? 0.f : log2e_over_f(T);
      break;
    }
  }
  p.c = c;
  return p;
}

// the end tile of the chunk holding tile t
__device__ __forceinline__ int chunk_end(const FusedArgs& a, int t) {
  return min(a.tpr, (t / kChunkTiles + 1) * kChunkTiles);
}

__device__ __forceinline__ FPos next_pos(const FusedArgs& a, const FPos& p, long long W) {
  if (p.t + 1 < chunk_end(a, p.t)) {
    FPos q = p;
    ++q.t;
    return q;
  }
  return first_read_chunk(a, p.c + W, W);
}

// ---------------------------------------------------------------- acceptance scan
// The warp that folded the last row of batch row b.  Lane t holds position
// t: the target row's statistics (t <= K_b), the draft row's (t < K_b,
// tempered rows), token x_t and draw r_t (u for t = K_b).
template <bool kPlug>
__device__ void scan_row(const FusedArgs& a, int b, int lane) {
  const int K = a.K;
  const float T = __ldg(a.temperature + b);
  const bool greedy = (T == 0.f);
  const int kb = kb_of(a, b);
  bool timeout = false;
  unsigned long long tstat = 0, ttok = 0, dstat = 0, dtok = 0;
  if (lane <= kb) {
    unsigned long long* p = a.rowstat + 2 * ((long long)b * (K + 1) + lane);
    tstat = wait_word(a, p, timeout);
    ttok = wait_word(a, p + 1, timeout);
    st_relaxed_u64(p, 0ull);
    st_relaxed_u64(p + 1, 0ull);
  }
  if (!greedy && lane < kb) {
    unsigned long long* p = a.rowstat + 2 * ((long long)a.n_target_rows + (long long)b * K + lane);
    dstat = wait_word(a, p, timeout);
    dtok = wait_word(a, p + 1, timeout);
    st_relaxed_u64(p, 0ull);
    st_relaxed_u64(p + 1, 0ull);
  }
  if (lane == 0) a.scan_ticket[b] = 0u;
  if (__any_sync(0xffffffffu, timeout) && lane == 0) flag(a, kDevTimeout);

  int x = 0;
  bool tok_ok = true;
  if (lane < kb) {
    x = __ldg(a.tokens + (long long)b * K + lane);
    tok_ok = x >= 0 && x < a.V;
  }
  const float r = (!greedy && lane <= kb) ? __ldg(a.uniforms + (long long)b * (K + 1) + lane) : 0.f;
  const float2 ts = unpack2(tstat), ds = unpack2(dstat);
  int bad = __all_sync(0xffffffffu, tok_ok) ? 0 : (int)kDevBadToken;
  bool row_ok = true;
  if (lane <= kb) row_ok = isfinite(ts.x) && (greedy || (isfinite(ts.y) && ts.y > 0.f));
  if (!greedy && lane < kb) row_ok = row_ok && isfinite(ds.x) && isfinite(ds.y) && ds.y > 0.f;
  if (!bad && !__all_sync(0xffffffffu, row_ok)) bad = (int)kDevNonFinite;

  int n = kb;
  float lp = __int_as_float(0x7fffffff), lq = lp;
  const int amax = ~__float_as_int(ts.y);   // greedy rows: the lowest argmax
  if (!bad) {
    bool reject = false;
    if (greedy) {
      reject = lane < kb && amax != x;
    } else if (lane < kb) {
      // log p_t(x_t) = (x c - MC) ln 2 - ln S, with x c - MC formed exactly by the FMA
      constexpr float kLn2 = 0.693147180559945309f;
      const float c = log2e_over_f(T);
      const float xp = unpack2(ttok).x, xq = unpack2(dtok).x;
      lp = __fmaf_rn(xp, c, -ts.x) * kLn2 - logf(ts.y);
      lq = __fmaf_rn(xq, c, -ds.x) * kLn2 - logf(ds.y);
      // r q < p  <=>  r < p / q = exp(log p - log q)
      reject = !(r < expf(lp - lq));
    }
    const unsigned rej = __ballot_sync(0xffffffffu, reject);
    n = rej ? __ffs(rej) - 1 : kb;
  }
  if (lane < K) {
    const float nanv = __int_as_float(0x7fffffff);
    if (a.logp_out) a.logp_out[(long long)b * K + lane] = bad || greedy ? nanv : lp;
    if (a.logq_out) a.logq_out[(long long)b * K + lane] = bad || greedy ? nanv : lq;
  }
  int v = -1;
  if (!bad && lane <= K) {
    if (lane < n) v = x;
    else if (lane == n && greedy) v = amax;
  }
  const long long ob = (long long)b * (K + 1);
  if (lane <= K && !(lane == n && !greedy && !bad)) a.out_tokens[ob + lane] = v;
  if (lane == 0) {
    a.accepted_len[b] = bad ? -1 : n;
    if (bad) flag(a, (unsigned)bad);
  }
  if (kPlug && greedy && !bad)
    plug_row(lane, n, v, a.plug_tokens + (long long)b * a.plug_max_len, a.plug_seq_len + b,
             a.plug_max_len, a.plug_last ? a.plug_last + b : nullptr, &a.hdr->err_accum);
  if (!greedy) {
    // publish the draw's parameters (lane n holds position n)
    const int kind = bad ? 3 : (n < kb ? 1 : 2);
    const float MCp = __shfl_sync(0xffffffffu, ts.x, n), Sp = __shfl_sync(0xffffffffu, ts.y, n);
    const float MCq = __shfl_sync(0xffffffffu, ds.x, n), Sq = __shfl_sync(0xffffffffu, ds.y, n);
    const float u = __shfl_sync(0xffffffffu, r, kb);
    if (lane == 0) {
      if (kind != 3) {
        RowState rs;
        rs.n = n;
        rs.kind = kind;
        rs.MCp = MCp;
        rs.Sp = Sp;
        rs.MCq = kind == 1 ? MCq : 0.f;
        rs.Sq = kind == 1 ? Sq : 1.f;
        rs.u = u;
        rs.T = T;
        a.rowstate[b] = rs;
        __threadfence();
      }
      asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(a.ready + b), "r"((unsigned)kind) : "memory");
    }
  }
}

// The warp holding the last chunk ticket of row r: fold the row's partials
// into its statistics, gather the logit at the drafted token, and take the
// batch row's scan ticket.
template <typename E, bool kPlug>
__device__ __noinline__ void fold_row(const FusedArgs& a, int srow, bool greedy, int lane) {
  int rb, rpos;
  bool rdraft;
  srow_split(a, srow, rb, rpos, rdraft);
  unsigned long long* pp = a.partials + (long long)srow * a.cpr;
  bool timeout = false;
  float mc = SV_NEG_INF, s = 0.f, best = SV_NEG_INF;
  int bi = 0x7fffffff;
  for (int base = 0; base < a.cpr; base += 64) {
    const int i0 = base + lane, i1 = base + 32 + lane;
    unsigned long long v0 = i0 < a.cpr ? ld_relaxed_u64(pp + i0) : 0ull;
    unsigned long long v1 = i1 < a.cpr ? ld_relaxed_u64(pp + i1) : 0ull;
    if (i0 < a.cpr && v0 == 0ull) v0 = wait_word(a, pp + i0, timeout);
    if (i1 < a.cpr && v1 == 0ull) v1 = wait_word(a, pp + i1, timeout);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = h ? i1 : i0;
      if (i >= a.cpr) continue;
      const float2 f = unpack2(h ? v1 : v0);
      st_relaxed_u64(pp + i, 0ull);
      if (greedy) {
        const int idx = ~__float_as_int(f.y);
        if (f.x > best || (f.x == best && idx < bi)) {
          best = f.x;
          bi = idx;
        }
      } else if (f.x != SV_NEG_INF) {
        if (f.x > mc) {
          s = s * ex2_approx(__fsub_rn(mc, f.x)) + f.y;
          mc = f.x;
        } else {
          s += f.y * ex2_approx(__fsub_rn(f.x, mc));
        }
      }
    }
  }
  float2 stat;
  if (greedy) {
    const float m = warp_max(best);
    const int idx = warp_min_int(best == m ? bi : 0x7fffffff);
    stat = make_float2(m, __int_as_float(~idx));
  } else {
    const float M = warp_max(mc);
    float sv = (mc == SV_NEG_INF) ? 0.f : s * ex2_approx(__fsub_rn(mc, M));
    stat = make_float2(M, warp_sum(sv));
  }
  if (__any_sync(0xffffffffu, timeout) && lane == 0) flag(a, kDevTimeout);
  const int kb = kb_of(a, rb);
  unsigned old = 0;
  if (lane == 0) {
    a.fold_ticket[srow] = 0u;
    // token word: (logit at the drafted token, tag): 1 gathered, 2 token out of range, 3 none
    float xt = 0.f;
    int tag = 3;
    if (!greedy && rpos < kb) {
      const int x = __ldg(a.tokens + (long long)rb * a.K + rpos);
      tag = 2;
      if (x >= 0 && x < a.V) {
        xt = E::load_scalar(srow_ptr<E>(a, srow), x);
        tag = 1;
      }
    }
    unsigned long long* rs = a.rowstat + 2 * (long long)srow;
    st_relaxed_u64(rs, pack2(stat.x, stat.y));
    st_relaxed_u64(rs + 1, pack2(xt, __int_as_float(tag)));
    old = atom_add_u32(a.scan_ticket + rb, 1u);
  }
  old = __shfl_sync(0xffffffffu, old, 0);
  if (old + 1 == (unsigned)rows_read(kb, greedy)) scan_row<kPlug>(a, rb, lane);
}

// Reduce the lane values of a finished chunk, write its partial and take the
// row's chunk ticket; the last one folds the row.
template <typename E, bool kPlug>
__device__ __forceinline__ void flush_chunk(const FusedArgs& a, const FPos& p, int lane,
                                            const LaneStats& st) {
  const bool greedy = (p.cs == 0.f);
  float2 part;
  if (greedy) {
    const float m = warp_max(st.best);
    const int idx = warp_min_int(st.best == m ? st.bi : 0x7fffffff);
    part = make_float2(m, __int_as_float(~idx));
  } else {
    const float M = warp_max(st.mc);
    const float sv = (st.mc == SV_NEG_INF) ? 0.f : st.s * ex2_approx(__fsub_rn(st.mc, M));
    part = make_float2(M, warp_sum(sv));
  }
  unsigned old = 0;
  if (lane == 0) {
    st_relaxed_u64(a.partials + (long long)p.srow * a.cpr + p.t / kChunkTiles, pack2(part.x, part.y));
    old = atom_add_u32(a.fold_ticket + p.srow, 1u);
  }
  old = __shfl_sync(0xffffffffu, old, 0);
  if (old + 1 == (unsigned)a.cpr) fold_row<E, kPlug>(a, p.srow, greedy, lane);
}

template <typename E, bool kAligned>
__device__ __forceinline__ void load_pos(uint32_t (&w)[kTileVecsPerLane][4], const FusedArgs& a,
                                         const FPos& p, int lane, int full_end) {
  load_tile<E, kAligned>(w, srow_ptr<E>(a, p.srow), p.t, lane, a.V, p.t < full_end, true);
}

template <typename E, bool kAligned, bool kPlug>
__device__ void stream_phase(const FusedArgs& a, long long gw, long long W, int lane) {
  const int full_end = ((long long)a.tpr * kTileVecs * E::kVec == a.V) ? a.tpr : a.tpr - 1;
  FPos pa = first_read_chunk(a, gw, W);
  if (pa.c >= a.n_chunks) return;
  // register ping-pong: the next tile's loads are in flight while the
  // current one is folded, across chunk boundaries
  uint32_t wa[kTileVecsPerLane][4], wb[kTileVecsPerLane][4];
  load_pos<E, kAligned>(wa, a, pa, lane, full_end);
  LaneStats st;
  st.reset();
  for (;;) {
    const FPos pb = next_pos(a, pa, W);
    if (pb.c < a.n_chunks) load_pos<E, kAligned>(wb, a, pb, lane, full_end);
    fold_tile<E>(wa, (long long)pa.t * kTileVecs + lane, pa.cs == 0.f, pa.cs, st);
    if (pa.t + 1 == chunk_end(a, pa.t)) {
      flush_chunk<E, kPlug>(a, pa, lane, st);
      st.reset();
    }
    if (pb.c >= a.n_chunks) break;
    pa = next_pos(a, pb, W);
    if (pa.c < a.n_chunks) load_pos<E, kAligned>(wa, a, pa, lane, full_end);
    fold_tile<E>(wb, (long long)pb.t * kTileVecs + lane, pb.cs == 0.f, pb.cs, st);
    if (pb.t + 1 == chunk_end(a, pb.t)) {
      flush_chunk<E, kPlug>(a, pb, lane, st);
      st.reset();
    }
    if (pa.c >= a.n_chunks) break;
  }
}

// ---------------------------------------------------------------- phase 2
// The sampling context of a published row (the same derivation the weights
// of every tile and the locate step use).
template <typename E>
__device__ __forceinline__ SampleCtx ctx_of(const FusedArgs& a, int b, const RowState& rs) {
  const long long rowbytes = (long long)a.V * E::kBytes;
  SampleCtx x;
  x.rowP = (const char*)a.target + ((long long)b * (a.K + 1) + rs.n) * rowbytes;
  x.rowQ = rs.kind == 1 ? (const char*)a.draft + ((long long)b * a.K + rs.n) * rowbytes : nullptr;
  x.V = a.V;
  x.MCp = rs.MCp;
  x.MCq = rs.MCq;
  x.L = log2e_over(rs.T);
  x.c_hi = x.L.hi;
  x.c_lo = x.L.lo;
  if (!(x.c_lo > 0.f)) {   // a strictly positive low part (see small_exp)
    x.c_hi = __uint_as_float(__float_as_uint(x.L.hi) - 1u);
    x.c_lo = __fadd_rn(__fsub_rn(x.L.hi, x.c_hi), x.L.lo);
  }
  x.cw = __fdiv_rn(rs.Sp, rs.Sq);
  x.thp = kBigProb * rs.Sp;
  x.thq = kBigProb * rs.Sq;
  return x;
}

// Element (vector j, element k) of lane `lane` in a tile, as a tile offset.
template <typename E>
__device__ __forceinline__ int tile_elem(int lane, int j, int k) {
  return (32 * j + lane) * E::kVec + k;
}

// Weigh tile `tile` of the sampled row(s): the tile totals W (of the
// weights at cw), Q (e^q where the weight is positive), Sp and Sq (all e^p,
// e^q), as double-floats, written to the tile's record.  Small terms are
// summed in float32 pairs, large terms listed and weighed in double-float
// one per lane -- the same per-element rule the locate step applies.
template <typename E, bool kAligned, bool kResidual>
__device__ void weigh_tile(const FusedArgs& a, FusedSmem& sm, const SampleCtx& x, int b, int tile,
                           int lane, int warp, int full_end) {
  constexpr int kTileElems = kTileVecs * E::kVec;
  uint32_t wp[kTileVecsPerLane][4], wq[kTileVecsPerLane][4];
  load_tile<E, kAligned>(wp, x.rowP, tile, lane, a.V, tile < full_end, true);
  if (kResidual) load_tile<E, kAligned>(wq, x.rowQ, tile, lane, a.V, tile < full_end, true);
  const unsigned long long chi2 = f2_pack(x.c_hi, x.c_hi), clo2 = f2_pack(x.c_lo, x.c_lo);
  const unsigned long long nmcp2 = f2_pack(-x.MCp, -x.MCp), nmcq2 = f2_pack(-x.MCq, -x.MCq);
  const unsigned long long ncw2 = f2_pack(-x.cw, -x.cw);
  unsigned long long sw2 = 0ull, sq2 = 0ull, sp2 = 0ull, sQ2 = 0ull;
  unsigned big = 0u;
#pragma unroll
  for (int j = 0; j < kTileVecsPerLane; ++j) {
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
        // a large term leaves the float32 sums (it adds +0 everywhere)
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
  // the large terms: listed in the warp's region, one per lane
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
    if (total <= kFBigCap) {
      int o = inc - cnt;
      for (unsigned m = big; m; m &= m - 1u) {
        const int bit = __ffs(m) - 1;
        sm.bigpos[warp][o++] = (uint32_t)tile_elem<E>(lane, bit / E::kVec, bit % E::kVec);
      }
      __syncwarp();
      for (int e = lane; e < total; e += 32) {
        big_term<E, kResidual>(x, sm.tab, base + sm.bigpos[warp][e], w, q, ep, eq);
        W = df_add(W, w);
        if (kResidual) {
          Q = df_add(Q, q);
          P = df_add(P, ep);
          S = df_add(S, eq);
        }
      }
      __syncwarp();
    } else {
      for (unsigned m = big; m; m &= m - 1u) {
        const int bit = __ffs(m) - 1;
        big_term<E, kResidual>(x, sm.tab, base + tile_elem<E>(lane, bit / E::kVec, bit % E::kVec), w,
                               q, ep, eq);
        W = df_add(W, w);
        if (kResidual) {
          Q = df_add(Q, q);
          P = df_add(P, ep);
          S = df_add(S, eq);
        }
      }
    }
  }
  W = warp_sum_df(W);
  if (kResidual) {
    Q = warp_sum_df(Q);
    P = warp_sum_df(P);
    S = warp_sum_df(S);
  } else {
    P = W;
  }
  if (lane == 0) {
    float4* rec = a.recs + 2 * ((long long)b * a.tpr + tile);
    rec[0] = make_float4(W.hi, W.lo, Q.hi, Q.lo);
    rec[1] = make_float4(P.hi, P.lo, S.hi, S.lo);
  }
}

// Weight of tile j for the locate step: mode 0 the residual corrected to
// the exact c, mode 1 the bonus weights, mode 2 p (the residual was zero).
__device__ __forceinline__ DF rec_weight(const float4* recs, long long j, int mode, DF dc) {
  const float4 r0 = __ldcg(recs + 2 * j);
  if (mode == 0) return df_sub(DF{r0.x, r0.y}, df_mul(dc, DF{r0.z, r0.w}));
  if (mode == 1) return DF{r0.x, r0.y};
  const float4 r1 = __ldcg(recs + 2 * j + 1);
  return DF{r1.x, r1.y};
}

// Element weights of one 16-byte vector of the chosen tile, as the tiles
// were weighed (mode as in rec_weight).
template <typename E>
__device__ __forceinline__ void vec_weights(const uint32_t (&wp)[4], const uint32_t (&wq)[4],
                                            long long e0, int V, const SampleCtx& x,
                                            const float2* tab, int mode, DF dc, DF (&w)[E::kVec]) {
#pragma unroll
  for (int k = 0; k < E::kVec; ++k) {
    DF q{0.f, 0.f};
    if (e0 + k >= V) {
      w[k] = DF{0.f, 0.f};
    } else if (mode == 0) {
      eval_pair<true>(E::elem(wp, k), E::elem(wq, k), x, tab, w[k], q);
      w[k] = df_sub(w[k], df_mul(dc, q));
    } else {
      eval_pair<false>(E::elem(wp, k), 0.f, x, tab, w[k], q);
    }
  }
}

// The warp that completed row b's last item: choose the tile by the prefix
// of the tile totals, then the element inside it.  Returns the token (every
// lane).
template <typename E, bool kAligned>
__device__ __noinline__ int locate_row(const FusedArgs& a, FusedSmem& sm, const SampleCtx& x, const RowState& rs,
                          int b, int lane, int full_end) {
  constexpr int kTileElems = kTileVecs * E::kVec;
  const float4* recs = a.recs + 2 * (long long)b * a.tpr;
  const int tpr = a.tpr;
  const int per = (tpr + 31) / 32;                  // tiles per lane, contiguous
  const int j0 = min(tpr, lane * per), j1 = min(tpr, j0 + per);
  const bool residual = rs.kind == 1;
  // row totals of e^p and e^q, hence the exact c = S_p / S_q
  DF P{0.f, 0.f}, S{0.f, 0.f}, Wl{0.f, 0.f}, Ql{0.f, 0.f};
  for (int j = j0; j < j1; ++j) {
    const float4 r0 = __ldcg(recs + 2 * j), r1 = __ldcg(recs + 2 * j + 1);
    Wl = df_add(Wl, DF{r0.x, r0.y});
    Ql = df_add(Ql, DF{r0.z, r0.w});
    P = df_add(P, DF{r1.x, r1.y});
    S = df_add(S, DF{r1.z, r1.w});
  }
  DF dc{0.f, 0.f};
  int mode = residual ? 0 : 1;
  DF own = Wl;
  if (residual) {
    const DF Sp = warp_sum_df(P), Sq = warp_sum_df(S);
    dc = df_sub(df_div(Sp, Sq), DF{x.cw, 0.f});
    own = df_sub(Wl, df_mul(dc, Ql));
  }
  DF tot = warp_sum_df(own);
  if (residual && !df_pos(tot)) {   // the residual is zero everywhere: draw from p_n
    mode = 2;
    own = P;
    tot = warp_sum_df(own);
  }
  const DF tau = df_mul_f(tot, rs.u);
  // inclusive / exclusive prefix of the lanes' sums
  DF inc = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const DF up = df_shfl_up(inc, o);
    if (lane >= o) inc = df_add(inc, up);
  }
  DF exc = df_shfl_up(inc, 1);
  if (lane == 0) exc = DF{0.f, 0.f};
  const unsigned hit = __ballot_sync(0xffffffffu, df_pos(own) && df_lt(tau, inc));
  int jstar = -1, last_mode = 0;
  DF tl{0.f, 0.f};
  if (hit) {
    const int h = __ffs(hit) - 1;
    int gs = -1, glast = -1;
    if (lane == h) {
      DF run = exc;
      for (int j = j0; j < j1; ++j) {
        const DF wj = rec_weight(recs, j, mode, dc);
        const DF nxt = df_add(run, wj);
        if (df_pos(wj)) {
          glast = j;
          if (gs < 0 && df_lt(tau, nxt)) {
            gs = j;
            tl = df_sub(tau, run);
          }
        }
        run = nxt;
      }
      if (gs < 0) {   // fell off the end by rounding: the top of the last positive tile
        gs = glast >= 0 ? glast : j0;
        last_mode = 1;
      }
    }
    jstar = __shfl_sync(0xffffffffu, gs, h);
    last_mode = __shfl_sync(0xffffffffu, last_mode, h);
    tl = DF{__shfl_sync(0xffffffffu, tl.hi, h), __shfl_sync(0xffffffffu, tl.lo, h)};
  } else {
    // u*W at or past the total by rounding: the last tile with positive weight
    int gl = -1;
    for (int j = j0; j < j1; ++j)
      if (df_pos(rec_weight(recs, j, mode, dc))) gl = j;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) gl = max(gl, __shfl_xor_sync(0xffffffffu, gl, o));
    jstar = gl >= 0 ? gl : 0;
    last_mode = 1;
  }

  // the element inside tile jstar, in index order: vector j of every lane
  // covers elements [32 j kVec, 32 (j+1) kVec) of the tile
  uint32_t wp[kTileVecsPerLane][4], wq[kTileVecsPerLane][4];
  load_tile<E, kAligned>(wp, x.rowP, jstar, lane, a.V, jstar < full_end, true);
  if (mode == 0) load_tile<E, kAligned>(wq, x.rowQ, jstar, lane, a.V, jstar < full_end, true);
  const long long tbase = (long long)jstar * kTileElems;
  DF base{0.f, 0.f};
  int token = -1, lastpos = -1;
  float bestw = -3.0e38f;
  int bestk = 0x7fffffff;
#pragma unroll 1
  for (int j = 0; j < kTileVecsPerLane; ++j) {
    DF w[E::kVec];
    const long long e0 = tbase + tile_elem<E>(lane, j, 0);
    vec_weights<E>(wp[j], wq[j], e0, a.V, x, sm.tab, mode, dc, w);
    DF ls{0.f, 0.f};
    int lpos = -1;
#pragma unroll
    for (int k = 0; k < E::kVec; ++k) {
      if (df_pos(w[k])) {
        ls = df_add(ls, w[k]);
        lpos = tile_elem<E>(lane, j, k);
      }
      if (e0 + k < a.V && (w[k].hi > bestw)) {
        bestw = w[k].hi;
        bestk = tile_elem<E>(lane, j, k);
      }
    }
    lastpos = max(lastpos, lpos);
    DF li = ls;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const DF up = df_shfl_up(li, o);
      if (lane >= o) li = df_add(li, up);
    }
    DF le = df_shfl_up(li, 1);
    if (lane == 0) le = DF{0.f, 0.f};
    const DF vt{__shfl_sync(0xffffffffu, li.hi, 31), __shfl_sync(0xffffffffu, li.lo, 31)};
    if (!last_mode && token < 0) {
      const unsigned h2 = __ballot_sync(0xffffffffu, df_pos(ls) && df_lt(tl, df_add(base, li)));
      if (h2) {
        const int h = __ffs(h2) - 1;
        int tk = -1;
        if (lane == h) {
          DF run = df_add(base, le);
          for (int k = 0; k < E::kVec && tk < 0; ++k) {
            if (!df_pos(w[k])) continue;
            run = df_add(run, w[k]);
            if (df_lt(tl, run)) tk = tile_elem<E>(lane, j, k);
          }
          if (tk < 0) tk = lpos;   // rounding inside the lane: its last positive element
        }
        token = __shfl_sync(0xffffffffu, tk, h);
      }
    }
    base = df_add(base, vt);
  }
  if (token < 0) {
    // rounding or the last-mode fallback: the last positive element of the
    // tile, else (nothing positive) its largest weight, lowest index on ties
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lastpos = max(lastpos, __shfl_xor_sync(0xffffffffu, lastpos, o));
    if (lastpos >= 0) {
      token = lastpos;
    } else {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ow = __shfl_xor_sync(0xffffffffu, bestw, o);
        const int ok = __shfl_xor_sync(0xffffffffu, bestk, o);
        if (ow > bestw || (ow == bestw && ok < bestk)) {
          bestw = ow;
          bestk = ok;
        }
      }
      token = bestk == 0x7fffffff ? 0 : bestk;
    }
  }
  return (int)(tbase + token);
}

// The RowState of batch row b, read by lane 0 after its acquire and
// broadcast.
__device__ __forceinline__ RowState load_rowstate(const FusedArgs& a, int b, int lane) {
  int4 v0 = make_int4(0, 0, 0, 0), v1 = v0;
  if (lane == 0) {
    const int4* p = reinterpret_cast<const int4*>(a.rowstate + b);
    v0 = __ldcg(p);
    v1 = __ldcg(p + 1);
  }
  RowState rs;
  rs.n = __shfl_sync(0xffffffffu, v0.x, 0);
  rs.kind = __shfl_sync(0xffffffffu, v0.y, 0);
  rs.MCp = __int_as_float(__shfl_sync(0xffffffffu, v0.z, 0));
  rs.Sp = __int_as_float(__shfl_sync(0xffffffffu, v0.w, 0));
  rs.MCq = __int_as_float(__shfl_sync(0xffffffffu, v1.x, 0));
  rs.Sq = __int_as_float(__shfl_sync(0xffffffffu, v1.y, 0));
  rs.u = __int_as_float(__shfl_sync(0xffffffffu, v1.z, 0));
  rs.T = __int_as_float(__shfl_sync(0xffffffffu, v1.w, 0));
  return rs;
}

// A batch row whose temperature or verified length is invalid (found from
// the inputs alone): error row.
__device__ void error_row(const FusedArgs& a, int b, unsigned f, int lane) {
  const int K = a.K;
  if (lane <= K) a.out_tokens[(long long)b * (K + 1) + lane] = -1;
  if (lane < K) {
    if (a.logp_out) a.logp_out[(long long)b * K + lane] = __int_as_float(0x7fffffff);
    if (a.logq_out) a.logq_out[(long long)b * K + lane] = __int_as_float(0x7fffffff);
  }
  if (lane == 0) {
    a.accepted_len[b] = -1;
    flag(a, f);
  }
}

template <typename E, bool kAligned, bool kPlug>
__device__ void sample_phase(const FusedArgs& a, FusedSmem& sm, int lane, int warp) {
  // wait for other warps' work only once every CTA has started
  unsigned go = 0;
  if (lane == 0) go = ld_relaxed_u32(&a.hdr->arrived) >= gridDim.x;
  if (!__shfl_sync(0xffffffffu, go, 0)) return;
  const int full_end = ((long long)a.tpr * kTileVecs * E::kVec == a.V) ? a.tpr : a.tpr - 1;
  for (;;) {
    unsigned k = 0;
    if (lane == 0) k = atom_add_u32(&a.hdr->claim, 1u);
    k = __shfl_sync(0xffffffffu, k, 0);
    if ((long long)k >= a.n_items) break;
    const int b = (int)(k / (unsigned)a.tpr);
    const int j = (int)(k - (unsigned)b * (unsigned)a.tpr);
    const float T = __ldg(a.temperature + b);
    const int kb = kb_of(a, b);
    if (!valid_temperature(T) || kb < 0 || kb > a.K) {
      if (j == 0) error_row(a, b, !valid_temperature(T) ? kDevBadTemperature : kDevBadK, lane);
      continue;
    }
    if (T == 0.f) continue;   // greedy rows were finished by their scan
    unsigned rdy = 0;
    if (lane == 0) {
      rdy = ld_acquire_u32(a.ready + b);
      for (unsigned spins = 0; rdy == 0u; ++spins) {
        if (stop_waiting(a, spins)) {
          flag(a, kDevTimeout);
          rdy = 3u;
          break;
        }
        __nanosleep(128);
        rdy = ld_acquire_u32(a.ready + b);
      }
    }
    rdy = __shfl_sync(0xffffffffu, rdy, 0);
    RowState rs;
    SampleCtx x;
    if (rdy == 1u || rdy == 2u) {
      rs = load_rowstate(a, b, lane);
      x = ctx_of<E>(a, b, rs);
      if (rdy == 1u) weigh_tile<E, kAligned, true>(a, sm, x, b, j, lane, warp, full_end);
      else weigh_tile<E, kAligned, false>(a, sm, x, b, j, lane, warp, full_end);
    }
    unsigned old = 0;
    __syncwarp();
    if (lane == 0) {
      __threadfence();   // this tile's record before the ticket
      old = atom_add_u32(a.samp_ticket + b, 1u);
    }
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old + 1 != (unsigned)a.tpr) continue;
    // every tile of row b is weighed: locate the token, then return the
    // row's slots to zero
    __threadfence();
    if (rdy == 1u || rdy == 2u) {
      const int token = locate_row<E, kAligned>(a, sm, x, rs, b, lane, full_end);
      const long long ob = (long long)b * (a.K + 1);
      if (lane == 0) a.out_tokens[ob + rs.n] = token;
      if (kPlug) {
        const int32_t tok = lane < rs.n ? __ldg(a.tokens + (long long)b * a.K + lane) : token;
        plug_row(lane, rs.n, tok, a.plug_tokens + (long long)b * a.plug_max_len, a.plug_seq_len + b,
                 a.plug_max_len, a.plug_last ? a.plug_last + b : nullptr, &a.hdr->err_accum);
      }
      float4* rr = a.recs + 2 * (long long)b * a.tpr;
      for (int i = lane; i < 2 * a.tpr; i += 32) rr[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (lane < 2) reinterpret_cast<int4*>(a.rowstate + b)[lane] = make_int4(0, 0, 0, 0);
    }
    if (lane == 0) {
      a.ready[b] = 0u;
      a.samp_ticket[b] = 0u;
    }
  }
}

template <typename E, bool kAligned, bool kPlug>
__global__ void __launch_bounds__(kFThreads, 4) sv_fused_kernel(FusedArgs a) {
  __shared__ FusedSmem sm;
  // the preceding kernel on the stream may still be draining (programmatic
  // dependent launch): wait for it before touching any memory
  wait_for_preceding_grid();
  if (threadIdx.x == 0) atom_add_u32(&a.hdr->arrived, 1u);
  for (int i = threadIdx.x; i < 256; i += kFThreads) sm.tab[i] = kExp2Table256[i];
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long gw = (long long)blockIdx.x * kFWarps + warp;
  const long long W = (long long)gridDim.x * kFWarps;
  stream_phase<E, kAligned, kPlug>(a, gw, W, lane);
  sample_phase<E, kAligned, kPlug>(a, sm, lane, warp);
  // the last warp to finish hands the call's flags to the public word and
  // resets the grid counters
  __syncwarp();
  if (lane == 0) {
    __threadfence();
    const unsigned total = gridDim.x * (unsigned)kFWarps;
    if (atom_add_u32(&a.hdr->exited, 1u) + 1u == total) {
      __threadfence();
      a.hdr->err = atomicExch(&a.hdr->err_accum, 0u);
      a.hdr->claim = 0u;
      a.hdr->arrived = 0u;
      a.hdr->exited = 0u;
    }
  }
}

}  // namespace sv
