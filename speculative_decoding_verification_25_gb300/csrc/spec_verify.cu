// Host side of spec_verify: argument checks, workspace layout, launch
// geometry and the C ABI declared in include/spec_verify.h.
//
// spec_verify, spec_verify_ragged, spec_verify_and_plug and
// spec_verify_static are two launches each on the caller's stream:
//   1. sv_row_stats_kernel (sv_stream.cuh), a persistent grid (SM count x
//      resident CTAs) whose warps stream contiguous ranges of 2 KB row
//      tiles and leave one partial per tile; with verified lengths per row
//      (B <= kCompactMaxB) its compact instantiation, whose warps split only
//      the rows read;
//   2. sv_draw_kernel (sv_draw.cuh), G CTAs per batch row: statistics fold,
//      acceptance scan, and the draw over the sampled position's tiles.
// spec_verify_row_stats is the first launch alone.  spec_verify_tree runs
// the first kernel over the target slots and then sv_tree_kernel;
// spec_verify_plug is one small launch of its own.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "spec_verify.h"
#include "sv_draw.cuh"
#include "sv_plug.cuh"
#include "sv_tree.cuh"

namespace {

constexpr size_t kHeaderBytes = 256;   // device flag word at offset 0
constexpr int kMaxDevices = 64;

struct DeviceCache {
  std::once_flag once;
  int sm_count = 0;
  int row_stats_blocks_per_sm[2][2][2] = {};  // [dtype][aligned][compact]
  int draw_blocks_per_sm = 1;
  cudaError_t init_error = cudaSuccess;
  // device address of g_static_scratch, looked up by the first
  // spec_verify_static call on this device
  std::once_flag static_once;
  void* static_scratch = nullptr;
  cudaError_t static_error = cudaSuccess;
};

DeviceCache g_devices[kMaxDevices];

// Scratch of spec_verify_static: one array per device, loaded with the module.
__device__ __align__(256) unsigned char g_static_scratch[SV_STATIC_SCRATCH_BYTES];

int vec_of(int dtype) { return dtype == SV_BF16 ? 8 : 4; }
int elt_of(int dtype) { return dtype == SV_BF16 ? 2 : 4; }

bool shape_ok(int B, int K, int V, int dtype) {
  if (dtype != SV_F32 && dtype != SV_BF16) return false;
  if (B < 0 || K < 1 || K > SV_MAX_K || V < 1) return false;
  return V <= spec_verify_max_vocab(dtype);
}

long long tiles_per_row(int V, int dtype) {
  const long long tile_elems = (long long)sv::kTileVecs * vec_of(dtype);
  return (V + tile_elems - 1) / tile_elems;
}

template <typename E, bool kAligned>
void* row_stats_fn(bool compact) {
  return compact ? (void*)sv::sv_row_stats_compact_kernel<E, kAligned>
                 : (void*)sv::sv_row_stats_kernel<E, kAligned>;
}
// compact: the kernel that splits only the rows read (verified lengths given,
// B <= kCompactMaxB)
void* pick_row_stats(int dtype, bool aligned, bool compact) {
  if (dtype == SV_BF16)
    return aligned ? row_stats_fn<sv::Bf16, true>(compact) : row_stats_fn<sv::Bf16, false>(compact);
  return aligned ? row_stats_fn<sv::F32, true>(compact) : row_stats_fn<sv::F32, false>(compact);
}
bool use_compact(const int32_t* k_per_row, int B) {
  return k_per_row != nullptr && B <= sv::kCompactMaxB;
}
template <typename E, bool kAligned>
void* draw_fn(bool plug) {
  return plug ? (void*)sv::sv_draw_kernel<E, kAligned, true>
              : (void*)sv::sv_draw_kernel<E, kAligned, false>;
}
void* pick_draw(int dtype, bool aligned, bool plug) {
  if (dtype == SV_BF16)
    return aligned ? draw_fn<sv::Bf16, true>(plug) : draw_fn<sv::Bf16, false>(plug);
  return aligned ? draw_fn<sv::F32, true>(plug) : draw_fn<sv::F32, false>(plug);
}

// SM count and occupancy of the kernels; once per device.
DeviceCache* device_cache(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceCache& dc = g_devices[dev];
  std::call_once(dc.once, [&dc, dev]() {
    cudaError_t e = cudaDeviceGetAttribute(&dc.sm_count, cudaDevAttrMultiProcessorCount, dev);
    for (int dt = 0; dt < 2 && e == cudaSuccess; ++dt) {
      for (int al = 0; al < 2 && e == cudaSuccess; ++al) {
        for (int cp = 0; cp < 2 && e == cudaSuccess; ++cp) {
          int nb = 0;
          e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, pick_row_stats(dt, al != 0, cp != 0),
                                                            sv::kP1Threads, 0);
          dc.row_stats_blocks_per_sm[dt][al][cp] = nb > 0 ? nb : 1;
        }
      }
    }
    int nb = 0;
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, pick_draw(SV_BF16, true, false),
                                                        sv::kDThreads, 0);
    dc.draw_blocks_per_sm = nb > 0 ? nb : 1;
    dc.init_error = e;
  });
  return &dc;
}

bool aligned_to(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace of the verify calls, in 256-byte aligned regions after the
// header (device flag word at offset 0): one float2 partial per 2 KB tile of
// every target and draft row; a draw ticket per batch row; one 32-byte
// record per tile of every batch row's sampled row.  The streaming launch
// clears the flag word and the tickets and writes every partial the draw
// launch reads, so nothing needs initialising.
struct Layout {
  size_t partials, counters, tile_recs, total;
};
Layout layout(int B, int K, int V, int dtype) {
  const long long rows = (long long)B * (2 * K + 1);
  const long long tpr = tiles_per_row(V, dtype);
  Layout L;
  size_t off = kHeaderBytes;
  L.partials = off;
  off = align_up(off + (size_t)(rows * tpr) * sizeof(float2), 256);
  L.counters = off;
  off = align_up(off + (size_t)B * 4, 256);
  L.tile_recs = off;
  off = align_up(off + (size_t)((long long)B * tpr) * 32, 256);
  L.total = off;
  return L;
}

// CTAs per batch row for the draw launch: enough to fill the GPU once, and
// at least one per 64 tiles of a row (more waves for large batches), at most
// kMaxParts and one per tile.
int draw_parts(int B, long long tpr, const DeviceCache* dc) {
  const long long fill = (long long)dc->sm_count * dc->draw_blocks_per_sm / (B > 0 ? B : 1);
  long long g = fill > (tpr + 63) / 64 ? fill : (tpr + 63) / 64;
  if (g > sv::kMaxParts) g = sv::kMaxParts;
  if (g > tpr) g = tpr;
  return g < 1 ? 1 : (int)g;
}

}  // namespace

namespace {

// Checks shared by the verify entry points; SV_OK means the arguments are
// usable (B may be 0).
int validate(const void* target_logits, const void* draft_logits, int dtype,
             const int32_t* draft_tokens, const float* uniforms, const float* temperature,
             int B, int K, int V, const int32_t* accepted_len, const int32_t* out_tokens,
             const float* logp_out, const float* logq_out, const void* workspace,
             size_t workspace_bytes) {
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_DTYPE;
  if (!shape_ok(B, K, V, dtype)) return SV_ERR_SHAPE;
  if (B == 0) return SV_OK;
  if (!target_logits || !draft_logits || !temperature || !workspace || !draft_tokens ||
      !uniforms || !accepted_len || !out_tokens)
    return SV_ERR_NULL;
  const size_t elt = (size_t)elt_of(dtype);
  if (!aligned_to(target_logits, elt) || !aligned_to(draft_logits, elt) ||
      !aligned_to(temperature, 4) || !aligned_to(workspace, 16) || !aligned_to(draft_tokens, 4) ||
      !aligned_to(uniforms, 4) || !aligned_to(accepted_len, 4) || !aligned_to(out_tokens, 4) ||
      (logp_out && !aligned_to(logp_out, 4)) || (logq_out && !aligned_to(logq_out, 4)))
    return SV_ERR_ALIGN;
  if (workspace_bytes < spec_verify_workspace_bytes(B, K, V, dtype)) return SV_ERR_WORKSPACE;
  return SV_OK;
}

bool vector_path(const void* target_logits, const void* draft_logits, int V, int dtype) {
  return aligned_to(target_logits, 16) && aligned_to(draft_logits, 16) &&
         ((size_t)V * (size_t)elt_of(dtype)) % 16 == 0;
}

// A plain launch that may start while the preceding kernel on the stream
// drains (programmatic dependent launch).  Only for kernels that call
// wait_for_preceding_grid() before their first memory access; without the
// attribute (refused) it falls back to plain stream order.
cudaError_t launch_early(const void* fn, dim3 grid, dim3 block, void** args, cudaStream_t st) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    e = cudaLaunchKernel(fn, grid, block, args, 0, st);
  }
  return e;
}

// Where the fused plug step writes (tokens == nullptr: no plug).
struct PlugTarget {
  int32_t* tokens = nullptr;
  int32_t* seq_len = nullptr;
  int32_t* last_token = nullptr;
  int max_len = 0;
};

// The streaming launch (partials of every row read, flag word and the draw
// launch's counters cleared); counters == nullptr for the tree's use.
int launch_row_stats(const void* target_logits, const void* draft_logits, int dtype,
                     const float* temperature, const int32_t* k_per_row, int B, int K, int V,
                     void* workspace, unsigned* counters, DeviceCache* dc, cudaStream_t st) {
  const bool aligned = vector_path(target_logits, draft_logits, V, dtype);
  const long long tpr = tiles_per_row(V, dtype);
  const long long n_target_rows = (long long)B * (K + 1);
  sv::RowStatsArgs ra;
  memset(&ra, 0, sizeof(ra));
  ra.target = target_logits;
  ra.draft = draft_logits;
  ra.temperature = temperature;
  ra.B = B;
  ra.K = K;
  ra.V = V;
  ra.tiles_per_row = (int)tpr;
  ra.n_tiles = (n_target_rows + (long long)B * K) * tpr;
  ra.n_target_rows = (int)n_target_rows;
  ra.k_per_row = k_per_row;
  ra.partials = (float2*)((char*)workspace + kHeaderBytes);
  ra.err = (unsigned*)workspace;
  ra.tickets = counters;
  ra.n_tickets = counters ? B : 0;
  // persistent grid: every SM filled once; every warp a contiguous tile range
  const int warps_per_block = sv::kP1Threads / 32;
  const bool compact = use_compact(k_per_row, B);
  long long blocks =
      (long long)dc->sm_count * dc->row_stats_blocks_per_sm[dtype][aligned ? 1 : 0][compact ? 1 : 0];
  const long long need = (ra.n_tiles + warps_per_block - 1) / warps_per_block;
  if (blocks > need) blocks = need;
  if (blocks < 1) blocks = 1;
  void* args[] = {&ra};
  return launch_early(pick_row_stats(dtype, aligned, compact), dim3((unsigned)blocks),
                      dim3(sv::kP1Threads), args, st) == cudaSuccess
             ? SV_OK
             : SV_ERR_CUDA;
}

// The whole step: the streaming launch, then the draw launch.  The draw
// grid may start as the streaming kernel's CTAs exit (programmatic
// dependent launch): it reads only caller inputs before it waits for the
// partials.
int launch_verify(const void* target_logits, const void* draft_logits, int dtype,
                  const int32_t* draft_tokens, const float* uniforms, const float* temperature,
                  const int32_t* k_per_row, int B, int K, int V, int32_t* accepted_len,
                  int32_t* out_tokens, float* logp_out, float* logq_out, void* workspace,
                  DeviceCache* dc, cudaStream_t st, const PlugTarget& plug = PlugTarget()) {
  const Layout L = layout(B, K, V, dtype);
  char* ws = (char*)workspace;
  unsigned* counters = (unsigned*)(ws + L.counters);
  const int r = launch_row_stats(target_logits, draft_logits, dtype, temperature, k_per_row, B, K,
                                 V, workspace, counters, dc, st);
  if (r != SV_OK) return r;
  const bool aligned = vector_path(target_logits, draft_logits, V, dtype);
  const long long tpr = tiles_per_row(V, dtype);
  sv::DrawArgs a;
  memset(&a, 0, sizeof(a));
  a.target = target_logits;
  a.draft = draft_logits;
  a.tokens = draft_tokens;
  a.uniforms = uniforms;
  a.temperature = temperature;
  a.k_per_row = k_per_row;
  a.B = B;
  a.K = K;
  a.V = V;
  a.tpr = (int)tpr;
  a.n_target_rows = B * (K + 1);
  a.parts = draw_parts(B, tpr, dc);
  a.partials = (const float2*)(ws + L.partials);
  a.err = (unsigned*)ws;
  a.tickets = counters;
  a.tile_recs = (float4*)(ws + L.tile_recs);
  a.accepted_len = accepted_len;
  a.out_tokens = out_tokens;
  a.logp_out = logp_out;
  a.logq_out = logq_out;
  a.plug_tokens = plug.tokens;
  a.plug_seq_len = plug.seq_len;
  a.plug_last = plug.last_token;
  a.plug_max_len = plug.max_len;
  void* args[] = {&a};
  const long long blocks = (long long)B * a.parts;
  return launch_early(pick_draw(dtype, aligned, plug.tokens != nullptr), dim3((unsigned)blocks),
                      dim3(sv::kDThreads), args, st) == cudaSuccess
             ? SV_OK
             : SV_ERR_CUDA;
}

DeviceCache* current_device_cache() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  DeviceCache* dc = device_cache(dev);
  if (!dc || dc->init_error != cudaSuccess) return nullptr;
  return dc;
}

// Device address of this device's g_static_scratch (nullptr if the lookup
// failed); the lookup runs once per device.
void* static_scratch(DeviceCache* dc) {
  std::call_once(dc->static_once, [dc]() {
    void* p = nullptr;
    dc->static_error = cudaGetSymbolAddress(&p, g_static_scratch);
    dc->static_scratch = (dc->static_error == cudaSuccess) ? p : nullptr;
  });
  return dc->static_scratch;
}

// Partials of the tree's streaming pass: one float2 per tile of every slot.
size_t tree_partials_offset() { return kHeaderBytes; }

}  // namespace

extern "C" {

int spec_verify_max_vocab(int dtype) {
  if (dtype != SV_F32 && dtype != SV_BF16) return 0;
  // 2^20 bf16 or 2^19 float32 elements (1024 tiles of 2 KB per row)
  return (1 << 19) * (dtype == SV_BF16 ? 2 : 1);
}

size_t spec_verify_workspace_bytes(int B, int K, int V, int dtype) {
  if (!shape_ok(B, K, V, dtype)) return 0;
  return layout(B, K, V, dtype).total;
}

const char* spec_verify_status_string(int status) {
  switch (status) {
    case SV_OK: return "ok";
    case SV_ERR_NULL: return "a required pointer is NULL";
    case SV_ERR_SHAPE: return "B, K or V out of range";
    case SV_ERR_DTYPE: return "unknown logit dtype";
    case SV_ERR_ALIGN: return "a pointer is not aligned to its element size (workspace: 16 bytes)";
    case SV_ERR_WORKSPACE: return "workspace smaller than spec_verify_workspace_bytes()";
    case SV_ERR_CUDA: return "a CUDA runtime call failed";
    case SV_ERR_TOO_LARGE:
      return "shape needs more scratch than spec_verify_static holds (SV_STATIC_SCRATCH_BYTES)";
    default: return "unknown status";
  }
}

int spec_verify(const void* target_logits, const void* draft_logits, int dtype,
                const int32_t* draft_tokens, const float* uniforms, const float* temperature,
                int B, int K, int V, int32_t* accepted_len, int32_t* out_tokens,
                float* logp_out, float* logq_out, void* workspace, size_t workspace_bytes,
                void* stream) {
  const int st = validate(target_logits, draft_logits, dtype, draft_tokens, uniforms, temperature,
                          B, K, V, accepted_len, out_tokens, logp_out, logq_out, workspace,
                          workspace_bytes);
  if (st != SV_OK || B == 0) return st;
  DeviceCache* dc = current_device_cache();
  if (!dc) return SV_ERR_CUDA;
  return launch_verify(target_logits, draft_logits, dtype, draft_tokens, uniforms, temperature,
                       nullptr, B, K, V, accepted_len, out_tokens, logp_out, logq_out, workspace, dc,
                       (cudaStream_t)stream);
}

int spec_verify_and_plug(const void* target_logits, const void* draft_logits, int dtype,
                         const int32_t* draft_tokens, const float* uniforms,
                         const float* temperature, const int32_t* k_per_row, int B, int K, int V,
                         int32_t* accepted_len, int32_t* out_tokens, float* logp_out,
                         float* logq_out, int32_t* tokens, int32_t* seq_len, int max_len,
                         int32_t* last_token, void* workspace, size_t workspace_bytes,
                         void* stream) {
  const int st = validate(target_logits, draft_logits, dtype, draft_tokens, uniforms, temperature,
                          B, K, V, accepted_len, out_tokens, logp_out, logq_out, workspace,
                          workspace_bytes);
  if (st != SV_OK) return st;
  if (max_len < 1) return SV_ERR_SHAPE;
  if (B == 0) return SV_OK;
  if (!tokens || !seq_len) return SV_ERR_NULL;
  if (!aligned_to(tokens, 4) || !aligned_to(seq_len, 4) || !aligned_to(last_token, 4) ||
      !aligned_to(k_per_row, 4))
    return SV_ERR_ALIGN;
  DeviceCache* dc = current_device_cache();
  if (!dc) return SV_ERR_CUDA;
  PlugTarget plug;
  plug.tokens = tokens;
  plug.seq_len = seq_len;
  plug.last_token = last_token;
  plug.max_len = max_len;
  return launch_verify(target_logits, draft_logits, dtype, draft_tokens, uniforms, temperature,
                       k_per_row, B, K, V, accepted_len, out_tokens, logp_out, logq_out, workspace,
                       dc, (cudaStream_t)stream, plug);
}

int spec_verify_row_stats(const void* target_logits, const void* draft_logits, int dtype,
                          const float* temperature, const int32_t* k_per_row, int B, int K, int V,
                          void* workspace, size_t workspace_bytes, void* stream) {
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_DTYPE;
  if (!shape_ok(B, K, V, dtype)) return SV_ERR_SHAPE;
  if (B == 0) return SV_OK;
  if (!target_logits || !draft_logits || !temperature || !workspace) return SV_ERR_NULL;
  const size_t elt = (size_t)elt_of(dtype);
  if (!aligned_to(target_logits, elt) || !aligned_to(draft_logits, elt) ||
      !aligned_to(temperature, 4) || !aligned_to(workspace, 16) || !aligned_to(k_per_row, 4))
    return SV_ERR_ALIGN;
  if (workspace_bytes < spec_verify_workspace_bytes(B, K, V, dtype)) return SV_ERR_WORKSPACE;
  DeviceCache* dc = current_device_cache();
  if (!dc) return SV_ERR_CUDA;
  const Layout L = layout(B, K, V, dtype);
  return launch_row_stats(target_logits, draft_logits, dtype, temperature, k_per_row, B, K, V,
                          workspace, (unsigned*)((char*)workspace + L.counters), dc,
                          (cudaStream_t)stream);
}

int spec_verify_ragged(const void* target_logits, const void* draft_logits, int dtype,
                       const int32_t* draft_tokens, const float* uniforms, const float* temperature,
                       const int32_t* k_per_row, int B, int K, int V, int32_t* accepted_len,
                       int32_t* out_tokens, float* logp_out, float* logq_out, void* workspace,
                       size_t workspace_bytes, void* stream) {
  const int st = validate(target_logits, draft_logits, dtype, draft_tokens, uniforms, temperature,
                          B, K, V, accepted_len, out_tokens, logp_out, logq_out, workspace,
                          workspace_bytes);
  if (st != SV_OK || B == 0) return st;
  if (!k_per_row) return SV_ERR_NULL;
  if (!aligned_to(k_per_row, 4)) return SV_ERR_ALIGN;
  DeviceCache* dc = current_device_cache();
  if (!dc) return SV_ERR_CUDA;
  return launch_verify(target_logits, draft_logits, dtype, draft_tokens, uniforms, temperature,
                       k_per_row, B, K, V, accepted_len, out_tokens, logp_out, logq_out, workspace,
                       dc, (cudaStream_t)stream);
}

int spec_verify_static(const void* target_logits, const void* draft_logits, int dtype,
                       const int32_t* draft_tokens, const float* uniforms,
                       const float* temperature, int B, int K, int V, int32_t* accepted_len,
                       int32_t* out_tokens, float* logp_out, float* logq_out, void* stream) {
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_DTYPE;
  if (!shape_ok(B, K, V, dtype)) return SV_ERR_SHAPE;
  if (B == 0) return SV_OK;
  if (spec_verify_workspace_bytes(B, K, V, dtype) > (size_t)SV_STATIC_SCRATCH_BYTES)
    return SV_ERR_TOO_LARGE;
  DeviceCache* dc = current_device_cache();
  if (!dc) return SV_ERR_CUDA;
  void* scratch = static_scratch(dc);
  if (!scratch) return SV_ERR_CUDA;
  const int st = validate(target_logits, draft_logits, dtype, draft_tokens, uniforms, temperature,
                          B, K, V, accepted_len, out_tokens, logp_out, logq_out, scratch,
                          (size_t)SV_STATIC_SCRATCH_BYTES);
  if (st != SV_OK) return st;
  return launch_verify(target_logits, draft_logits, dtype, draft_tokens, uniforms, temperature,
                       nullptr, B, K, V, accepted_len, out_tokens, logp_out, logq_out, scratch, dc,
                       (cudaStream_t)stream);
}

int spec_verify_static_device_errors(void* stream, uint32_t* flags) {
  if (!flags) return SV_ERR_NULL;
  DeviceCache* dc = current_device_cache();
  if (!dc) return SV_ERR_CUDA;
  void* scratch = static_scratch(dc);
  if (!scratch) return SV_ERR_CUDA;
  return spec_verify_device_errors(scratch, stream, flags);
}

size_t spec_verify_tree_workspace_bytes(int B, int N, int V, int dtype) {
  if (dtype != SV_F32 && dtype != SV_BF16) return 0;
  if (B < 0 || N < 1 || N > SV_MAX_TREE_NODES || V < 1 || V > spec_verify_max_vocab(dtype)) return 0;
  return tree_partials_offset() +
         (size_t)((long long)B * (N + 1) * tiles_per_row(V, dtype)) * sizeof(float2);
}

int spec_verify_tree(const void* target_logits, int dtype, const int32_t* node_tokens,
                     const int32_t* parents, int B, int N, int V, int32_t* accepted_len,
                     int32_t* out_tokens, int32_t* accepted_nodes, void* workspace,
                     size_t workspace_bytes, void* stream) {
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_DTYPE;
  const size_t need = spec_verify_tree_workspace_bytes(B, N, V, dtype);
  if (need == 0) return SV_ERR_SHAPE;
  if (B == 0) return SV_OK;
  if (!target_logits || !node_tokens || !parents || !accepted_len || !out_tokens || !workspace)
    return SV_ERR_NULL;
  if (!aligned_to(target_logits, (size_t)elt_of(dtype)) || !aligned_to(node_tokens, 4) ||
      !aligned_to(parents, 4) || !aligned_to(accepted_len, 4) || !aligned_to(out_tokens, 4) ||
      (accepted_nodes && !aligned_to(accepted_nodes, 4)) || !aligned_to(workspace, 16))
    return SV_ERR_ALIGN;
  if (workspace_bytes < need) return SV_ERR_WORKSPACE;
  DeviceCache* dc = current_device_cache();
  if (!dc) return SV_ERR_CUDA;
  cudaStream_t st = (cudaStream_t)stream;
  // 1. argmax partials of every target slot (every row greedy, no draft rows)
  const bool aligned = vector_path(target_logits, target_logits, V, dtype);
  const long long tpr = tiles_per_row(V, dtype);
  sv::RowStatsArgs ra;
  memset(&ra, 0, sizeof(ra));
  ra.target = target_logits;
  ra.draft = nullptr;
  ra.temperature = nullptr;
  ra.B = B;
  ra.K = N;
  ra.V = V;
  ra.tiles_per_row = (int)tpr;
  ra.n_target_rows = B * (N + 1);
  ra.n_tiles = (long long)B * (N + 1) * tpr;   // target slots only
  ra.k_per_row = nullptr;
  ra.partials = (float2*)((char*)workspace + tree_partials_offset());
  ra.err = (unsigned*)workspace;
  long long blocks = (long long)dc->sm_count * dc->row_stats_blocks_per_sm[dtype][aligned ? 1 : 0][0];
  const long long need_blocks = (ra.n_tiles + sv::kP1Threads / 32 - 1) / (sv::kP1Threads / 32);
  if (blocks > need_blocks) blocks = need_blocks;
  if (blocks < 1) blocks = 1;
  void* args1[] = {&ra};
  if (launch_early(pick_row_stats(dtype, aligned, false), dim3((unsigned)blocks),
                   dim3(sv::kP1Threads), args1, st) != cudaSuccess)
    return SV_ERR_CUDA;
  // 2. one CTA per tree
  sv::TreeArgs ta;
  ta.node_tokens = node_tokens;
  ta.parents = parents;
  ta.B = B;
  ta.N = N;
  ta.V = V;
  ta.tiles_per_row = (int)tpr;
  ta.partials = ra.partials;
  ta.err = (unsigned*)workspace;
  ta.accepted_len = accepted_len;
  ta.out_tokens = out_tokens;
  ta.accepted_nodes = accepted_nodes;
  void* args2[] = {&ta};
  return launch_early((void*)sv::sv_tree_kernel, dim3((unsigned)B), dim3(sv::kTreeThreads), args2,
                      st) == cudaSuccess
             ? SV_OK
             : SV_ERR_CUDA;
}

int spec_verify_plug(const int32_t* accepted_len, const int32_t* out_tokens, int B, int K,
                     int32_t* tokens, int32_t* seq_len, int max_len, int32_t* last_token,
                     uint32_t* flags, void* stream) {
  if (B < 0 || K < 1 || K > SV_MAX_K || max_len < 1) return SV_ERR_SHAPE;
  if (B == 0) return SV_OK;
  if (!accepted_len || !out_tokens || !tokens || !seq_len) return SV_ERR_NULL;
  if (!aligned_to(accepted_len, 4) || !aligned_to(out_tokens, 4) || !aligned_to(tokens, 4) ||
      !aligned_to(seq_len, 4) || (last_token && !aligned_to(last_token, 4)) ||
      (flags && !aligned_to(flags, 4)))
    return SV_ERR_ALIGN;
  sv::PlugArgs pa;
  pa.accepted_len = accepted_len;
  pa.out_tokens = out_tokens;
  pa.B = B;
  pa.K = K;
  pa.max_len = max_len;
  pa.tokens = tokens;
  pa.seq_len = seq_len;
  pa.last_token = last_token;
  pa.flags = flags;
  const long long threads = (long long)B * 32;
  const unsigned blocks = (unsigned)((threads + 255) / 256);
  void* args[] = {&pa};
  return launch_early((void*)sv::sv_plug_kernel, dim3(blocks), dim3(256), args,
                      (cudaStream_t)stream) == cudaSuccess
             ? SV_OK
             : SV_ERR_CUDA;
}

int spec_verify_device_errors(const void* workspace, void* stream, uint32_t* flags) {
  if (!workspace || !flags) return SV_ERR_NULL;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(flags, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return SV_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SV_ERR_CUDA;
  return SV_OK;
}

}  // extern "C"
