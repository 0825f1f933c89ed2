// Greedy verification of a draft tree (the lesson "Decodificação
// Especulativa e EAGLE", section "Verificação de Atenção em Árvore": every
// node of the tree is checked in one target pass and the longest prefix
// along an accepted path is kept; the page "Accelerating Sonar through
// speculation", section EAGLE: the longest acceptable sequence continues,
// plus one token from the target).
//
// The streaming kernel runs first with every row greedy over the N+1
// target slots of each tree (slot 0 after the context, slot i+1 after node
// i) and leaves (max, lowest argmax) partials per tile.  This kernel, one
// CTA per tree, folds them into the argmax of every slot and walks the
// tree: node i is accepted iff its parent is the root or accepted and its
// token equals the argmax at the parent's slot; the deepest accepted node
// (lowest index on ties) gives the path, followed by the argmax at its slot.
#pragma once

#include "sv_sample.cuh"

namespace sv {

constexpr int kMaxTreeNodes = 128;
constexpr unsigned kDevBadTree = 64u;
// 32 half-warps: trees of up to 31 nodes fold every slot in one round
constexpr int kTreeThreads = 512;

struct TreeArgs {
  const int32_t* node_tokens;    // [B, N]
  const int32_t* parents;        // [B, N]
  int B, N, V;
  int tiles_per_row;
  const float2* partials;        // [B * (N+1)][tiles_per_row]
  unsigned* err;
  int32_t* accepted_len;         // [B]
  int32_t* out_tokens;           // [B, N+1]
  int32_t* accepted_nodes;       // [B, N] or nullptr
};

struct TreeSmem {
  int am[kMaxTreeNodes + 1];     // argmax of every slot
  float mx[kMaxTreeNodes + 1];   // max of every slot
  int tok[kMaxTreeNodes];
  int par[kMaxTreeNodes];
  int depth[kMaxTreeNodes];      // 0 = not accepted, else depth of the accepted node
  int path[kMaxTreeNodes];
  int bad;
};

__global__ void __launch_bounds__(kTreeThreads) sv_tree_kernel(TreeArgs a) {
  wait_for_preceding_grid();   // the streaming pass's partials, before any access
  __shared__ TreeSmem sm;
  const int b = blockIdx.x, tid = threadIdx.x;
  const int N = a.N;
  if (tid == 0) sm.bad = 0;
  __syncthreads();
  for (int i = tid; i < N; i += blockDim.x) {
    const int t = __ldg(a.node_tokens + (long long)b * N + i);
    const int p = __ldg(a.parents + (long long)b * N + i);
    sm.tok[i] = t;
    sm.par[i] = p;
    if (t < 0 || t >= a.V || p < -1 || p >= i) atomicOr(&sm.bad, (int)kDevBadTree);
  }
  // argmax of every slot: one half-warp per slot, 32 slots per round
  constexpr int kHalves = kTreeThreads / 16;
  const int hl = tid & 15, hw = tid >> 4;
  for (int base = 0; base <= N; base += kHalves) {   // the same trip count in every warp
    const int s = base + hw;
    const float2* pp = s <= N ? a.partials + ((long long)b * (N + 1) + s) * a.tiles_per_row : nullptr;
    const float2 st = fold_partials<16>(pp, a.tiles_per_row, true, hl);
    if (pp && hl == 0) {
      sm.mx[s] = st.x;
      sm.am[s] = __float_as_int(st.y);
    }
  }
  __syncthreads();
  if (tid != 0) return;
  int bad = sm.bad;
  for (int s = 0; !bad && s <= N; ++s)
    if (!isfinite(sm.mx[s])) bad = (int)kDevNonFinite;
  int32_t* out = a.out_tokens + (long long)b * (N + 1);
  int32_t* nodes = a.accepted_nodes ? a.accepted_nodes + (long long)b * N : nullptr;
  if (bad) {
    a.accepted_len[b] = -1;
    for (int i = 0; i <= N; ++i) out[i] = -1;
    if (nodes)
      for (int i = 0; i < N; ++i) nodes[i] = -1;
    atomicOr(a.err, (unsigned)bad);
    return;
  }
  // parents precede their children: one pass in node order
  int best = -1;
  for (int i = 0; i < N; ++i) {
    const int p = sm.par[i];
    const int pd = p < 0 ? 0 : sm.depth[p];
    const bool ok = (p < 0 || pd > 0) && sm.tok[i] == sm.am[p < 0 ? 0 : p + 1];
    sm.depth[i] = ok ? pd + 1 : 0;
    if (ok && (best < 0 || sm.depth[i] > sm.depth[best])) best = i;
  }
  const int d = best < 0 ? 0 : sm.depth[best];
  for (int i = best, k = d - 1; i >= 0; i = sm.par[i], --k) sm.path[k] = i;
  for (int k = 0; k < d; ++k) out[k] = sm.tok[sm.path[k]];
  out[d] = sm.am[best < 0 ? 0 : best + 1];
  for (int k = d + 1; k <= N; ++k) out[k] = -1;
  if (nodes)
    for (int k = 0; k < N; ++k) nodes[k] = k < d ? sm.path[k] : -1;
  a.accepted_len[b] = d;
}

}  // namespace sv
