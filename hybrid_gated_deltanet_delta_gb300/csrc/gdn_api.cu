// The C ABI (include/gdn.h): argument checks, tile choice and launches.
// Nothing here allocates, synchronises or keeps state between calls.
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>
#include <stdlib.h>

#include "gdn_common.cuh"
#include "gdn_launch.h"

namespace {

// NVTX range around one entry point, pushed only when GDN_NVTX is set (to
// anything but "0") at the first call; the header-only NVTX calls are no-ops
// unless a profiler injects itself.
bool nvtx_on() {
  static const bool on = [] {
    const char* e = getenv("GDN_NVTX");
    return e != nullptr && e[0] != '\0' && !(e[0] == '0' && e[1] == '\0');
  }();
  return on;
}

struct Range {
  const bool on;
  explicit Range(const char* name) : on(nvtx_on()) {
    if (on) nvtxRangePushA(name);
  }
  ~Range() {
    if (on) nvtxRangePop();
  }
};
#define GDN_RANGE() Range gdn_range_(__func__)

bool ok_ptr16(const void* p) { return p != nullptr && gdn::aligned16(p); }
bool ok_ptr4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Default slab shape for the verify and replay kernels: 16 columns per block
// and one warp per block for a chain: its node loop overlaps each node's
// update with the shuffle tree of the look-ahead sums, which a cross-warp
// exchange would interrupt (measured on the 16-node chain: one warp 13.1 us,
// two row warps 13.4 us per launch).  Tree blocks take whole nodes per warp,
// so the row-warp count applies to chains and replays only.  A replay takes
// the chain's shape, so that a chain committed by replay repeats the verify
// arithmetic bit for bit.
void auto_tile(int* wc, int* nw) {
  *wc = 16;
  *nw = 1;
}

int verify_common(const gdn_verify_args* a, const int32_t* parent, int32_t* depth_out, bool tree,
                  void* stream, void* snap16 = nullptr, bool prep = false) {
  if (a == nullptr) return GDN_ERR_INVALID_ARG;
  if (a->B < 0 || a->N < 1 || a->Hk < 1 || a->Hv < 1 || a->Hv % a->Hk != 0)
    return GDN_ERR_INVALID_ARG;
  if (a->in_dtype != GDN_F32 && a->in_dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (a->N > 64 || a->B > 65535 || a->Hv > 65535) return GDN_ERR_UNSUPPORTED;
  if (a->dk != 16 && a->dk != 32 && a->dk != 64 && a->dk != 128) return GDN_ERR_UNSUPPORTED;
  if (a->dv < 16 || a->dv > 1024 || a->dv % 16 != 0) return GDN_ERR_UNSUPPORTED;
  if (a->B == 0) return GDN_OK;
  if (a->n_slots < 1) return GDN_ERR_INVALID_ARG;
  const int64_t head_set = (int64_t)a->Hv * a->dk * a->dv;
  if (a->cache_slot_stride < head_set) return GDN_ERR_INVALID_ARG;
  if (a->cache_slot_stride % 4 != 0) return GDN_ERR_MISALIGNED;
  const void* need16[] = {a->q, a->k, a->v, a->state_cache, a->o};
  for (const void* p : need16) {
    if (p == nullptr) return GDN_ERR_INVALID_ARG;
    if (!gdn::aligned16(p)) return GDN_ERR_MISALIGNED;
  }
  // snapshots may be NULL: nothing is persisted and the accepted state is
  // committed by replay
  if (snap16 == nullptr && a->snapshots != nullptr && !gdn::aligned16(a->snapshots))
    return GDN_ERR_MISALIGNED;
  if (snap16 != nullptr && !gdn::aligned16(snap16)) return GDN_ERR_MISALIGNED;
  if (a->alpha == nullptr || a->beta == nullptr) return GDN_ERR_INVALID_ARG;
  if (tree && parent == nullptr) return GDN_ERR_INVALID_ARG;
  if (tree && a->max_depth < 0) return GDN_ERR_INVALID_ARG;
  const void* need4[] = {a->alpha, a->beta, a->slot, a->status, parent, depth_out};
  for (const void* p : need4)
    if (!ok_ptr4(p)) return GDN_ERR_MISALIGNED;

  int wc = 0, nw = 0;
  auto_tile(&wc, &nw);
  if (a->tile_cols != 0) wc = a->tile_cols;
  if (a->row_warps != 0) nw = a->row_warps;
  else if (!gdn::verify_tile_supported(a->dk, wc, nw)) nw = 1;  // automatic, for a forced width
  if (!gdn::verify_tile_supported(a->dk, wc, nw) || a->dv % wc != 0) return GDN_ERR_UNSUPPORTED;
  return gdn::launch_verify(a, tree ? parent : nullptr, tree ? depth_out : nullptr, wc, nw,
                            static_cast<cudaStream_t>(stream), snap16, prep);
}

int commit_common(const void* snapshots, bool src16, int64_t snap_layer_stride,
                  const int32_t* accept_idx, float* state_cache, int64_t cache_slot_stride,
                  int64_t cache_layer_stride, const int32_t* slot, int32_t n_slots, int32_t B,
                  int32_t N, int32_t Hv, int32_t dk, int32_t dv, int32_t n_layers,
                  int32_t* status, void* stream) {
  if (B < 0 || n_layers < 0 || N < 1 || Hv < 1 || dk < 1 || dv < 1) return GDN_ERR_INVALID_ARG;
  if (snap_layer_stride < 0 || cache_slot_stride < 0 || cache_layer_stride < 0)
    return GDN_ERR_INVALID_ARG;
  if (B > 65535 || n_layers > 65535) return GDN_ERR_UNSUPPORTED;
  if (B == 0 || n_layers == 0) return GDN_OK;
  const int64_t head_set = (int64_t)Hv * dk * dv;
  if (n_slots < 1 || cache_slot_stride < head_set) return GDN_ERR_INVALID_ARG;
  if (head_set % 4 != 0 || snap_layer_stride % 4 != 0 || cache_slot_stride % 4 != 0 ||
      cache_layer_stride % 4 != 0)
    return GDN_ERR_MISALIGNED;
  if (snapshots == nullptr || accept_idx == nullptr || state_cache == nullptr)
    return GDN_ERR_INVALID_ARG;
  if (!ok_ptr16(snapshots) || !ok_ptr16(state_cache)) return GDN_ERR_MISALIGNED;
  if (!ok_ptr4(accept_idx) || !ok_ptr4(slot) || !ok_ptr4(status)) return GDN_ERR_MISALIGNED;
  return gdn::launch_commit(snapshots, src16, snap_layer_stride, accept_idx, state_cache,
                            cache_slot_stride, cache_layer_stride, slot, n_slots, B, N, Hv, dk,
                            dv, n_layers, status, static_cast<cudaStream_t>(stream));
}

int replay_common(const gdn_verify_args* a, const int32_t* parent, const int32_t* accept,
                  void* stream, bool prep = false) {
  if (a == nullptr) return GDN_ERR_INVALID_ARG;
  if (a->B < 0 || a->N < 1 || a->Hk < 1 || a->Hv < 1 || a->Hv % a->Hk != 0)
    return GDN_ERR_INVALID_ARG;
  if (a->in_dtype != GDN_F32 && a->in_dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (a->N > 64 || a->B > 65535 || a->Hv > 65535) return GDN_ERR_UNSUPPORTED;
  if (a->dk != 16 && a->dk != 32 && a->dk != 64 && a->dk != 128) return GDN_ERR_UNSUPPORTED;
  if (a->dv < 16 || a->dv > 1024 || a->dv % 16 != 0) return GDN_ERR_UNSUPPORTED;
  if (a->B == 0) return GDN_OK;
  if (a->n_slots < 1) return GDN_ERR_INVALID_ARG;
  const int64_t head_set = (int64_t)a->Hv * a->dk * a->dv;
  if (a->cache_slot_stride < head_set) return GDN_ERR_INVALID_ARG;
  if (a->cache_slot_stride % 4 != 0) return GDN_ERR_MISALIGNED;
  const void* need16[] = {a->k, a->v, a->state_cache};
  for (const void* p : need16) {
    if (p == nullptr) return GDN_ERR_INVALID_ARG;
    if (!gdn::aligned16(p)) return GDN_ERR_MISALIGNED;
  }
  if (a->alpha == nullptr || a->beta == nullptr || accept == nullptr) return GDN_ERR_INVALID_ARG;
  const void* need4[] = {a->alpha, a->beta, a->slot, a->status, parent, accept};
  for (const void* p : need4)
    if (!ok_ptr4(p)) return GDN_ERR_MISALIGNED;
  int wc = 0, nw = 0;
  auto_tile(&wc, &nw);
  if (a->tile_cols != 0) wc = a->tile_cols;
  if (a->row_warps != 0) nw = a->row_warps;
  else if (!gdn::verify_tile_supported(a->dk, wc, nw)) nw = 1;  // automatic, for a forced width
  if (!gdn::verify_tile_supported(a->dk, wc, nw) || a->dv % wc != 0) return GDN_ERR_UNSUPPORTED;
  return gdn::launch_replay(a, parent, accept, wc, nw, static_cast<cudaStream_t>(stream), prep);
}

// Host checks shared by the two prefill entry points.
int prefill_checks(const void* q, const void* k, const void* v, int32_t in_dtype,
                   const float* alpha, const float* beta, int32_t T, int32_t Hk, int32_t Hv,
                   int32_t dk, int32_t dv, int32_t chunk, const float* state, const float* o,
                   const int32_t* status) {
  if (T < 0 || Hk < 1 || Hv < 1 || Hv % Hk != 0) return GDN_ERR_INVALID_ARG;
  if (in_dtype != GDN_F32 && in_dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  // the tensor-core form takes bf16 inputs at d_k = d_v = 128, chunk 64 only
  if (dk != 128 || dv != 128 || chunk != 64 || in_dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
  if (Hv > 65535) return GDN_ERR_UNSUPPORTED;
  if (state == nullptr) return GDN_ERR_INVALID_ARG;
  if (!gdn::aligned16(state)) return GDN_ERR_MISALIGNED;
  if (!ok_ptr4(status)) return GDN_ERR_MISALIGNED;
  if (T == 0) return GDN_OK;
  const void* need16[] = {q, k, v, o};
  for (const void* p : need16) {
    if (p == nullptr) return GDN_ERR_INVALID_ARG;
    if (!gdn::aligned16(p)) return GDN_ERR_MISALIGNED;
  }
  if (alpha == nullptr || beta == nullptr) return GDN_ERR_INVALID_ARG;
  if (!ok_ptr4(alpha) || !ok_ptr4(beta)) return GDN_ERR_MISALIGNED;
  return GDN_OK;
}

}  // namespace

extern "C" {

int gdn_replay_accepted(const gdn_verify_args* args, const int32_t* parent,
                        const int32_t* accept_idx, void* stream) {
  GDN_RANGE();
  return replay_common(args, parent, accept_idx, stream);
}

int gdn_verify_chain_prep(const gdn_verify_args* args, void* stream) {
  GDN_RANGE();
  return verify_common(args, nullptr, nullptr, false, stream, nullptr, true);
}

int gdn_verify_tree_prep(const gdn_verify_args* args, const int32_t* parent, int32_t* depth_out,
                         void* stream) {
  GDN_RANGE();
  return verify_common(args, parent, depth_out, true, stream, nullptr, true);
}

int gdn_replay_accepted_prep(const gdn_verify_args* args, const int32_t* parent,
                             const int32_t* accept_idx, void* stream) {
  GDN_RANGE();
  return replay_common(args, parent, accept_idx, stream, true);
}

int gdn_verify_chain(const gdn_verify_args* args, void* stream) {
  GDN_RANGE();
  return verify_common(args, nullptr, nullptr, false, stream);
}

int gdn_verify_tree(const gdn_verify_args* args, const int32_t* parent, int32_t* depth_out,
                    void* stream) {
  GDN_RANGE();
  return verify_common(args, parent, depth_out, true, stream);
}

int gdn_verify_chain_f16(const gdn_verify_args* args, void* snapshots_f16, void* stream) {
  GDN_RANGE();
  if (snapshots_f16 == nullptr) return GDN_ERR_INVALID_ARG;
  return verify_common(args, nullptr, nullptr, false, stream, snapshots_f16);
}

int gdn_verify_tree_f16(const gdn_verify_args* args, const int32_t* parent, int32_t* depth_out,
                        void* snapshots_f16, void* stream) {
  GDN_RANGE();
  if (snapshots_f16 == nullptr) return GDN_ERR_INVALID_ARG;
  return verify_common(args, parent, depth_out, true, stream, snapshots_f16);
}

int gdn_commit_accepted(const float* snapshots, int64_t snap_layer_stride,
                        const int32_t* accept_idx, float* state_cache, int64_t cache_slot_stride,
                        int64_t cache_layer_stride, const int32_t* slot, int32_t n_slots,
                        int32_t B, int32_t N, int32_t Hv, int32_t dk, int32_t dv,
                        int32_t n_layers, int32_t* status, void* stream) {
  GDN_RANGE();
  return commit_common(snapshots, false, snap_layer_stride, accept_idx, state_cache,
                       cache_slot_stride, cache_layer_stride, slot, n_slots, B, N, Hv, dk, dv,
                       n_layers, status, stream);
}

int gdn_commit_accepted_f16(const void* snapshots_f16, int64_t snap_layer_stride,
                            const int32_t* accept_idx, float* state_cache,
                            int64_t cache_slot_stride, int64_t cache_layer_stride,
                            const int32_t* slot, int32_t n_slots, int32_t B, int32_t N,
                            int32_t Hv, int32_t dk, int32_t dv, int32_t n_layers,
                            int32_t* status, void* stream) {
  GDN_RANGE();
  return commit_common(snapshots_f16, true, snap_layer_stride, accept_idx, state_cache,
                       cache_slot_stride, cache_layer_stride, slot, n_slots, B, N, Hv, dk, dv,
                       n_layers, status, stream);
}

int gdn_conv_commit(const void* x, int32_t in_dtype, void* conv_state,
                    int64_t state_slot_stride, const int32_t* slot, int32_t n_slots,
                    const int32_t* parent, const int32_t* accept_idx, int32_t B, int32_t N,
                    int32_t C, int32_t W, int32_t* status, void* stream) {
  GDN_RANGE();
  if (in_dtype != GDN_F32 && in_dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (B < 0 || N < 1 || C < 1 || W < 1 || n_slots < 1) return GDN_ERR_INVALID_ARG;
  if (W > 8 || B > 65535) return GDN_ERR_UNSUPPORTED;
  if (state_slot_stride < (int64_t)C * W) return GDN_ERR_INVALID_ARG;
  if (B == 0) return GDN_OK;
  if (x == nullptr || conv_state == nullptr || accept_idx == nullptr) return GDN_ERR_INVALID_ARG;
  const uintptr_t esz = in_dtype == GDN_BF16 ? 2 : 4;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(conv_state)) % esz != 0)
    return GDN_ERR_MISALIGNED;
  if (!ok_ptr4(accept_idx) || !ok_ptr4(slot) || !ok_ptr4(parent) || !ok_ptr4(status))
    return GDN_ERR_MISALIGNED;
  return gdn::launch_conv_commit(x, in_dtype == GDN_BF16, conv_state, state_slot_stride, slot,
                                 n_slots, parent, accept_idx, B, N, C, W, status,
                                 static_cast<cudaStream_t>(stream));
}

int gdn_commit_index(const int32_t* accept_idx, int32_t B, int32_t N, int32_t base_slot,
                     int32_t* slot, int32_t* status, void* stream) {
  GDN_RANGE();
  if (B < 0 || N < 1 || base_slot < 0) return GDN_ERR_INVALID_ARG;
  if ((int64_t)base_slot + (int64_t)B * N > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
  if (B == 0) return GDN_OK;
  if (accept_idx == nullptr || slot == nullptr) return GDN_ERR_INVALID_ARG;
  if (!ok_ptr4(accept_idx) || !ok_ptr4(slot) || !ok_ptr4(status)) return GDN_ERR_MISALIGNED;
  return gdn::launch_commit_index(accept_idx, B, N, base_slot, slot, status,
                                  static_cast<cudaStream_t>(stream));
}

size_t gdn_prefill_workspace_bytes(int32_t T, int32_t Hk, int32_t Hv, int32_t dk, int32_t dv,
                                   int32_t chunk) {
  if (T < 0 || Hk < 1 || Hv < 1 || dk < 1 || dv < 1 || chunk < 1) return 0;
  return gdn::prefill_workspace_bytes(T, Hk, Hv, dk, dv, chunk);
}

int gdn_prefill_chunked(const void* q, const void* k, const void* v, int32_t in_dtype,
                        const float* alpha, const float* beta, int32_t T, int32_t Hk, int32_t Hv,
                        int32_t dk, int32_t dv, int32_t chunk, float* state, float* o,
                        void* workspace, size_t workspace_bytes, int32_t* status, void* stream) {
  GDN_RANGE();
  const int st = prefill_checks(q, k, v, in_dtype, alpha, beta, T, Hk, Hv, dk, dv, chunk, state,
                                o, status);
  if (st != GDN_OK || T == 0) return st;
  const size_t need = gdn::prefill_workspace_bytes(T, Hk, Hv, dk, dv, chunk);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return GDN_ERR_WORKSPACE;
  if (need > 0 && !gdn::aligned16(workspace)) return GDN_ERR_MISALIGNED;
  return gdn::launch_prefill(q, k, v, true, alpha, beta, T, Hk, Hv, dk, dv, chunk, state, o,
                             workspace, status, static_cast<cudaStream_t>(stream));
}

int gdn_prefill_chunked_noalloc(const void* q, const void* k, const void* v, int32_t in_dtype,
                                const float* alpha, const float* beta, int32_t T, int32_t Hk,
                                int32_t Hv, int32_t dk, int32_t dv, int32_t chunk, float* state,
                                float* o, int32_t* status, void* stream) {
  GDN_RANGE();
  const int st = prefill_checks(q, k, v, in_dtype, alpha, beta, T, Hk, Hv, dk, dv, chunk, state,
                                o, status);
  if (st != GDN_OK || T == 0) return st;
  return gdn::launch_prefill_noalloc(q, k, v, true, alpha, beta, T, Hk, Hv, dk, dv, chunk, state,
                                     o, status, static_cast<cudaStream_t>(stream));
}

const char* gdn_status_string(int status) {
  switch (status) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
    case GDN_ERR_MISALIGNED: return "GDN_ERR_MISALIGNED";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
    case GDN_ERR_BAD_TREE: return "GDN_ERR_BAD_TREE";
    case GDN_ERR_ACCEPT_RANGE: return "GDN_ERR_ACCEPT_RANGE";
    case GDN_ERR_SLOT_RANGE: return "GDN_ERR_SLOT_RANGE";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE";
    case GDN_ERR_SCRATCH_LIMIT: return "GDN_ERR_SCRATCH_LIMIT";
    case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT";
    default: return "GDN_ERR_UNKNOWN";
  }
}

int gdn_version(void) { return GDN_VERSION; }

}  // extern "C"
