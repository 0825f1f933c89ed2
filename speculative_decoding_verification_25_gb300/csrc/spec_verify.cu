// Host side of spec_verify: argument checks, launch geometry and the C ABI
// declared in include/spec_verify.h.
//
// One call (spec_verify, spec_verify_ragged, spec_verify_static, or their
// two stage entry points) = two launches on the caller's stream:
//   1. sv_row_stats_kernel, a persistent grid (SM count x resident CTAs)
//      whose warps stream contiguous ranges of 2 KB row tiles; with
//      verified lengths per row (B <= kCompactMaxB) its compact
//      instantiation, whose warps split only the rows read;
//   2. sv_accept_sample_kernel, one thread-block cluster per batch row.
// spec_verify_tree runs the first kernel (target rows only) and then
// sv_tree_kernel; spec_verify_plug is one small launch of its own.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "spec_verify.h"
#include "sv_plug.cuh"
#include "sv_sample.cuh"
#include "sv_tree.cuh"

namespace {

constexpr size_t kHeaderBytes = 256;   // device error word lives at offset 0
constexpr int kMaxDevices = 64;

struct DeviceCache {
  std::once_flag once;
  int sm_count = 0;
  int row_stats_blocks_per_sm[2][2][2] = {};  // [dtype][aligned][compact]
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
template <typename E, bool kAligned>
void* accept_fn(bool plug) {
  return plug ? (void*)sv::sv_accept_sample_kernel<E, kAligned, true>
              : (void*)sv::sv_accept_sample_kernel<E, kAligned, false>;
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
// plug: the instantiation with the plug step fused in
void* pick_accept(int dtype, bool aligned, bool plug) {
  if (dtype == SV_BF16)
    return aligned ? accept_fn<sv::Bf16, true>(plug) : accept_fn<sv::Bf16, false>(plug);
  return aligned ? accept_fn<sv::F32, true>(plug) : accept_fn<sv::F32, false>(plug);
}

// dynamic shared memory of the accept/sample kernel: 16 B of per-group
// weights for every group of the sampled row the CTA owns
size_t accept_smem_bytes(int groups_per_cta) { return (size_t)groups_per_cta * 16; }

constexpr int kMaxGroupsPerCta = sv::kMaxGroupsPerThread * sv::kP2Threads;

// SM count, occupancy of the streaming kernel, and the shared-memory limit
// of the sampling kernel; once per device.
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
        for (int pl = 0; pl < 2 && e == cudaSuccess; ++pl) {
          void* ac = pick_accept(dt, al != 0, pl != 0);
          e = cudaFuncSetAttribute(ac, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)accept_smem_bytes(kMaxGroupsPerCta));
          if (e == cudaSuccess)
            e = cudaFuncSetAttribute(ac, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        }
      }
    }
    dc.init_error = e;
  });
  return &dc;
}

// Cluster size for the sampling step: the smallest power of two for which
// every CTA owns at most two groups per thread, at most 16 (16 needs the
// non-portable cluster size, allowed at initialisation).  Only about 33
// clusters of 16 fit on the GPU at once, against 74 of 8, so batches of
// more than 32 rows use clusters of 8 when a CTA can hold the larger slice
// (at most kMaxGroupsPerCta groups): fewer waves, each paying the fixed
// per-row chain once.  Likewise clusters of 8 become clusters of 4 when B
// clusters of 8 would not all be resident at once (SMs x 4 CTAs).  A small
// batch leaves SMs idle instead: the cluster doubles while every CTA still
// gets an SM of its own and keeps at least 64 groups, since a smaller slice
// shortens the row's chain.
void cluster_geometry(int V, int dtype, int B, int sm_count, int* cs, int* ngroups, int* gpc) {
  const int gelems = sv::kGroupVecs * vec_of(dtype);
  *ngroups = (V + gelems - 1) / gelems;
  int c = 1;
  while (c < sv::kMaxClusterSize && (*ngroups + c - 1) / c > 2 * sv::kP2Threads) c *= 2;
  if (B > 32 && c > 8 && (*ngroups + 7) / 8 <= kMaxGroupsPerCta) c = 8;
  if (c == 8 && (long long)B * 8 > 4LL * sm_count && (*ngroups + 3) / 4 <= kMaxGroupsPerCta) c = 4;
  while (c < sv::kMaxClusterSize && (long long)B * 2 * c <= sm_count &&
         (*ngroups + 2 * c - 1) / (2 * c) >= 64)
    c *= 2;
  *cs = c;
  *gpc = (*ngroups + c - 1) / c;
}

bool aligned_to(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace: a 256-byte header (the row-flag word at offset 0), then one
// float2 partial per tile of every target and draft row.  The streaming
// launch clears the flag word and writes every partial the accept launch
// reads, so no part of the workspace needs initialising.
size_t partials_offset() { return align_up(kHeaderBytes, 256); }
size_t workspace_total(int B, int K, int V, int dtype) {
  const long long rows = (long long)B * (K + 1) + (long long)B * K;
  return partials_offset() + (size_t)(rows * tiles_per_row(V, dtype)) * sizeof(float2);
}

}  // namespace

namespace {

// Checks shared by every launching entry point; SV_OK means the arguments
// are usable (B may be 0).
int validate(const void* target_logits, const void* draft_logits, int dtype,
             const int32_t* draft_tokens, const float* uniforms, const float* temperature,
             int B, int K, int V, const int32_t* accepted_len, const int32_t* out_tokens,
             const float* logp_out, const float* logq_out, const void* workspace,
             size_t workspace_bytes, bool need_outputs) {
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_DTYPE;
  if (!shape_ok(B, K, V, dtype)) return SV_ERR_SHAPE;
  if (B == 0) return SV_OK;
  if (!target_logits || !draft_logits || !temperature || !workspace) return SV_ERR_NULL;
  if (need_outputs && (!draft_tokens || !uniforms || !accepted_len || !out_tokens))
    return SV_ERR_NULL;
  const size_t elt = (size_t)elt_of(dtype);
  if (!aligned_to(target_logits, elt) || !aligned_to(draft_logits, elt) ||
      !aligned_to(temperature, 4) || !aligned_to(workspace, 16))
    return SV_ERR_ALIGN;
  if (need_outputs &&
      (!aligned_to(draft_tokens, 4) || !aligned_to(uniforms, 4) || !aligned_to(accepted_len, 4) ||
       !aligned_to(out_tokens, 4) || (logp_out && !aligned_to(logp_out, 4)) ||
       (logq_out && !aligned_to(logq_out, 4))))
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

int launch_row_stats(const void* target_logits, const void* draft_logits, int dtype,
                     const float* temperature, const int32_t* k_per_row, int B, int K, int V,
                     void* workspace, DeviceCache* dc, cudaStream_t st) {
  const bool aligned = vector_path(target_logits, draft_logits, V, dtype);
  const long long tpr = tiles_per_row(V, dtype);
  const long long n_target_rows = (long long)B * (K + 1);
  sv::RowStatsArgs ra;
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
  ra.partials = (float2*)((char*)workspace + partials_offset());
  ra.err = (unsigned*)workspace;
  // persistent grid: every SM filled once; every warp a contiguous tile range
  const int threads = sv::kP1Threads;
  const int warps_per_block = threads / 32;
  const bool compact = use_compact(k_per_row, B);
  long long blocks =
      (long long)dc->sm_count * dc->row_stats_blocks_per_sm[dtype][aligned ? 1 : 0][compact ? 1 : 0];
  const long long need = (ra.n_tiles + warps_per_block - 1) / warps_per_block;
  if (blocks > need) blocks = need;
  if (blocks < 1) blocks = 1;
  void* args[] = {&ra};
  return launch_early(pick_row_stats(dtype, aligned, compact), dim3((unsigned)blocks),
                      dim3(threads), args, st) == cudaSuccess
             ? SV_OK
             : SV_ERR_CUDA;
}

DeviceCache* current_device_cache();

// Where the fused plug step writes (tokens == nullptr: no plug).
struct PlugTarget {
  int32_t* tokens = nullptr;
  int32_t* seq_len = nullptr;
  int32_t* last_token = nullptr;
  int max_len = 0;
};

int launch_accept_sample(const void* target_logits, const void* draft_logits, int dtype,
                         const int32_t* draft_tokens, const float* uniforms,
                         const float* temperature, const int32_t* k_per_row, int B, int K, int V,
                         int32_t* accepted_len, int32_t* out_tokens, float* logp_out,
                         float* logq_out, void* workspace, cudaStream_t st,
                         const PlugTarget& plug = PlugTarget(), bool early = false) {
  const bool aligned = vector_path(target_logits, draft_logits, V, dtype);
  int cs, ngroups, gpc;
  const DeviceCache* dc = current_device_cache();
  cluster_geometry(V, dtype, B, dc && dc->sm_count > 0 ? dc->sm_count : 148, &cs, &ngroups, &gpc);
  sv::AcceptArgs aa;
  aa.target = target_logits;
  aa.draft = draft_logits;
  aa.tokens = draft_tokens;
  aa.uniforms = uniforms;
  aa.temperature = temperature;
  aa.B = B;
  aa.K = K;
  aa.V = V;
  aa.tiles_per_row = (int)tiles_per_row(V, dtype);
  aa.n_target_rows = B * (K + 1);
  aa.ngroups = ngroups;
  aa.groups_per_cta = gpc;
  aa.partials = (const float2*)((const char*)workspace + partials_offset());
  aa.k_per_row = k_per_row;
  aa.err = (unsigned*)workspace;
  aa.accepted_len = accepted_len;
  aa.out_tokens = out_tokens;
  aa.logp_out = logp_out;
  aa.logq_out = logq_out;
  aa.plug_tokens = plug.tokens;
  aa.plug_seq_len = plug.seq_len;
  aa.plug_last = plug.last_token;
  aa.plug_max_len = plug.max_len;
  void* args[] = {&aa};

  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)B * (unsigned)cs);
  cfg.blockDim = dim3(sv::kP2Threads);
  cfg.dynamicSmemBytes = accept_smem_bytes(gpc);
  cfg.stream = st;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = (unsigned)cs;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  // early: the grid may start as the streaming kernel's CTAs exit
  // (programmatic dependent launch; every CTA exit is its trigger).  Only
  // for a launch that directly follows this call's own streaming launch:
  // the kernel reads caller inputs before it waits for the partials.
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = early ? 2 : 1;
  void* fn = pick_accept(dtype, aligned, plug.tokens != nullptr);
  cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e != cudaSuccess && early) {
    // without the early start the dependency is plain stream order
    (void)cudaGetLastError();
    cfg.numAttrs = 1;
    e = cudaLaunchKernelExC(&cfg, fn, args);
  }
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

// The whole step: the streaming launch, then the accept/sample launch.
int launch_both(const void* target_logits, const void* draft_logits, int dtype,
                const int32_t* draft_tokens, const float* uniforms, const float* temperature,
                const int32_t* k_per_row, int B, int K, int V, int32_t* accepted_len,
                int32_t* out_tokens, float* logp_out, float* logq_out, void* workspace,
                DeviceCache* dc, cudaStream_t st, const PlugTarget& plug = PlugTarget()) {
  const int r = launch_row_stats(target_logits, draft_logits, dtype, temperature, k_per_row, B, K,
                                 V, workspace, dc, st);
  if (r != SV_OK) return r;
  return launch_accept_sample(target_logits, draft_logits, dtype, draft_tokens, uniforms,
                              temperature, k_per_row, B, K, V, accepted_len, out_tokens, logp_out,
                              logq_out, workspace, st, plug, /*early=*/true);
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

}  // namespace

extern "C" {

int spec_verify_max_vocab(int dtype) {
  if (dtype != SV_F32 && dtype != SV_BF16) return 0;
  // every CTA of a 16-CTA cluster owns at most kMaxGroupsPerCta groups
  return sv::kMaxClusterSize * kMaxGroupsPerCta * sv::kGroupVecs * vec_of(dtype);
}

size_t spec_verify_workspace_bytes(int B, int K, int V, int dtype) {
  if (!shape_ok(B, K, V, dtype)) return 0;
  return workspace_total(B, K, V, dtype);
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

int spec_verify_row_stats(const void* target_logits, const void* draft_logits, int dtype,
                          const float* temperature, int B, int K, int V, void* workspace,
                          size_t workspace_bytes, void* stream) {
  const int st = validate(target_logits, draft_logits, dtype, nullptr, nullptr, temperature, B, K,
                          V, nullptr, nullptr, nullptr, nullptr, workspace, workspace_bytes, false);
  if (st != SV_OK || B == 0) return st;
  DeviceCache* dc = current_device_cache();
  if (!dc) return SV_ERR_CUDA;
  return launch_row_stats(target_logits, draft_logits, dtype, temperature, nullptr, B, K, V,
                          workspace, dc, (cudaStream_t)stream);
}

int spec_verify_accept_sample(const void* target_logits, const void* draft_logits, int dtype,
                              const int32_t* draft_tokens, const float* uniforms,
                              const float* temperature, int B, int K, int V,
                              int32_t* accepted_len, int32_t* out_tokens, float* logp_out,
                              float* logq_out, void* workspace, size_t workspace_bytes,
                              void* stream) {
  const int st = validate(target_logits, draft_logits, dtype, draft_tokens, uniforms, temperature,
                          B, K, V, accepted_len, out_tokens, logp_out, logq_out, workspace,
                          workspace_bytes, true);
  if (st != SV_OK || B == 0) return st;
  if (!current_device_cache()) return SV_ERR_CUDA;
  return launch_accept_sample(target_logits, draft_logits, dtype, draft_tokens, uniforms,
                              temperature, nullptr, B, K, V, accepted_len, out_tokens, logp_out,
                              logq_out, workspace, (cudaStream_t)stream);
}

int spec_verify_ragged_row_stats(const void* target_logits, const void* draft_logits, int dtype,
                                 const float* temperature, const int32_t* k_per_row, int B, int K,
                                 int V, void* workspace, size_t workspace_bytes, void* stream) {
  const int st = validate(target_logits, draft_logits, dtype, nullptr, nullptr, temperature, B, K,
                          V, nullptr, nullptr, nullptr, nullptr, workspace, workspace_bytes, false);
  if (st != SV_OK || B == 0) return st;
  if (!k_per_row) return SV_ERR_NULL;
  if (!aligned_to(k_per_row, 4)) return SV_ERR_ALIGN;
  DeviceCache* dc = current_device_cache();
  if (!dc) return SV_ERR_CUDA;
  return launch_row_stats(target_logits, draft_logits, dtype, temperature, k_per_row, B, K, V,
                          workspace, dc, (cudaStream_t)stream);
}

int spec_verify_ragged_accept_sample(const void* target_logits, const void* draft_logits,
                                     int dtype, const int32_t* draft_tokens,
                                     const float* uniforms, const float* temperature,
                                     const int32_t* k_per_row, int B, int K, int V,
                                     int32_t* accepted_len, int32_t* out_tokens, float* logp_out,
                                     float* logq_out, void* workspace, size_t workspace_bytes,
                                     void* stream) {
  const int st = validate(target_logits, draft_logits, dtype, draft_tokens, uniforms, temperature,
                          B, K, V, accepted_len, out_tokens, logp_out, logq_out, workspace,
                          workspace_bytes, true);
  if (st != SV_OK || B == 0) return st;
  if (!k_per_row) return SV_ERR_NULL;
  if (!aligned_to(k_per_row, 4)) return SV_ERR_ALIGN;
  if (!current_device_cache()) return SV_ERR_CUDA;
  return launch_accept_sample(target_logits, draft_logits, dtype, draft_tokens, uniforms,
                              temperature, k_per_row, B, K, V, accepted_len, out_tokens, logp_out,
                              logq_out, workspace, (cudaStream_t)stream);
}

int spec_verify(const void* target_logits, const void* draft_logits, int dtype,
                const int32_t* draft_tokens, const float* uniforms, const float* temperature,
                int B, int K, int V, int32_t* accepted_len, int32_t* out_tokens,
                float* logp_out, float* logq_out, void* workspace, size_t workspace_bytes,
                void* stream) {
  const int st = validate(target_logits, draft_logits, dtype, draft_tokens, uniforms, temperature,
                          B, K, V, accepted_len, out_tokens, logp_out, logq_out, workspace,
                          workspace_bytes, true);
  if (st != SV_OK || B == 0) return st;
  DeviceCache* dc = current_device_cache();
  if (!dc) return SV_ERR_CUDA;
  return launch_both(target_logits, draft_logits, dtype, draft_tokens, uniforms, temperature,
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
                          workspace_bytes, true);
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
  return launch_both(target_logits, draft_logits, dtype, draft_tokens, uniforms, temperature,
                     k_per_row, B, K, V, accepted_len, out_tokens, logp_out, logq_out, workspace,
                     dc, (cudaStream_t)stream, plug);
}

int spec_verify_ragged(const void* target_logits, const void* draft_logits, int dtype,
                       const int32_t* draft_tokens, const float* uniforms, const float* temperature,
                       const int32_t* k_per_row, int B, int K, int V, int32_t* accepted_len,
                       int32_t* out_tokens, float* logp_out, float* logq_out, void* workspace,
                       size_t workspace_bytes, void* stream) {
  const int st = validate(target_logits, draft_logits, dtype, draft_tokens, uniforms, temperature,
                          B, K, V, accepted_len, out_tokens, logp_out, logq_out, workspace,
                          workspace_bytes, true);
  if (st != SV_OK || B == 0) return st;
  if (!k_per_row) return SV_ERR_NULL;
  if (!aligned_to(k_per_row, 4)) return SV_ERR_ALIGN;
  DeviceCache* dc = current_device_cache();
  if (!dc) return SV_ERR_CUDA;
  return launch_both(target_logits, draft_logits, dtype, draft_tokens, uniforms, temperature,
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
                          (size_t)SV_STATIC_SCRATCH_BYTES, true);
  if (st != SV_OK) return st;
  return launch_both(target_logits, draft_logits, dtype, draft_tokens, uniforms, temperature,
                     nullptr, B, K, V, accepted_len, out_tokens, logp_out, logq_out, scratch, dc,
                     (cudaStream_t)stream);
}

size_t spec_verify_tree_workspace_bytes(int B, int N, int V, int dtype) {
  if (dtype != SV_F32 && dtype != SV_BF16) return 0;
  if (B < 0 || N < 1 || N > SV_MAX_TREE_NODES || V < 1 || V > spec_verify_max_vocab(dtype)) return 0;
  return partials_offset() + (size_t)((long long)B * (N + 1) * tiles_per_row(V, dtype)) * sizeof(float2);
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
  ra.partials = (float2*)((char*)workspace + partials_offset());
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
