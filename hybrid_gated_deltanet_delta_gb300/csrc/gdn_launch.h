// Internal launchers (one per kernel family); the C ABI in gdn_api.cu checks
// every argument before calling them.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

bool verify_tile_supported(int dk, int wc, int nw);
// snap16 != NULL: chain with binary16 snapshots there (a->snapshots unused).
// prep: q, k are raw projections (L2-normalised here) and alpha, beta hold the
// gate pre-activations (alpha = exp(-softplus(a)), beta = sigmoid(b) here).
int launch_verify(const gdn_verify_args* a, const int32_t* parent, int32_t* depth_out, int wc,
                  int nw, cudaStream_t stream, void* snap16 = nullptr, bool prep = false);

// Tree verify without snapshots by one solve per block (gdn_solve.cu): the
// outputs (and depths) only, for a block committed by replay.
int launch_verify_tree_solve(const gdn_verify_args* a, const int32_t* parent, int32_t* depth_out,
                             int wc, cudaStream_t stream, bool prep);

// Replay of the accepted path from the cached state, written back in place.
int launch_replay(const gdn_verify_args* a, const int32_t* parent, const int32_t* accept, int wc,
                  int nw, cudaStream_t stream, bool prep = false);

// src16: the snapshots are binary16 (widened exactly into the fp32 cache).
int launch_commit(const void* snap, bool src16, int64_t snap_layer_stride, const int32_t* accept,
                  float* cache, int64_t cache_slot_stride, int64_t cache_layer_stride,
                  const int32_t* slot, int n_slots, int B, int N, int Hv, int dk, int dv,
                  int n_layers, int32_t* status, cudaStream_t stream);

// slot[b] = base_slot + b*N + accept[b] (accept checked).
int launch_commit_index(const int32_t* accept, int B, int N, int base_slot, int32_t* slot,
                        int32_t* status, cudaStream_t stream);

// Convolution history: the last W elements of [history, x of the accepted path].
int launch_conv_commit(const void* x, bool bf16, void* state, int64_t slot_stride,
                       const int32_t* slot, int n_slots, const int32_t* parent,
                       const int32_t* accept, int B, int N, int C, int W, int32_t* status,
                       cudaStream_t stream);

size_t prefill_workspace_bytes(int T, int Hk, int Hv, int dk, int dv, int chunk);
int launch_prefill(const void* q, const void* k, const void* v, bool bf16, const float* alpha,
                   const float* beta, int T, int Hk, int Hv, int dk, int dv, int chunk,
                   float* state, float* o, void* workspace, int32_t* status, cudaStream_t stream);

// gdn_prefill_chunked on the library's built-in scratch (no allocation).
int launch_prefill_noalloc(const void* q, const void* k, const void* v, bool bf16,
                           const float* alpha, const float* beta, int T, int Hk, int Hv, int dk,
                           int dv, int chunk, float* state, float* o, int32_t* status,
                           cudaStream_t stream);

}  // namespace gdn
