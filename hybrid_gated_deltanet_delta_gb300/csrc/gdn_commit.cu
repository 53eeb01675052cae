// Commit kernel: copy the accepted node's persisted state into the
// recurrent-state cache, for every sequence and every layer in one launch
// ("Photon 2.6", section "Handling recurrent state": the state at the accepted
// boundary becomes the request's state; when the whole block is accepted it is
// the last node's state).
//
// For one (layer, sequence) the source, snapshots[l][b][accept[b]][0..Hv), and
// the destination, cache[l][slot[b]][0..Hv), are each one contiguous run of
// Hv*dk*dv floats, so the kernel is a batched, bit-exact 16-byte-vector copy:
// grid = (pieces of the run, B, n_layers); each thread issues all its loads
// before its stores.  The snapshots are read with an evict-first hint since
// nothing reads them again.
#include <cuda_fp16.h>

#include "gdn_common.cuh"
#include "gdn_launch.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

// Four consecutive snapshot elements as fp32: a float4, or four binary16
// values (8 bytes) widened exactly.
template <bool SRC16>
__device__ __forceinline__ float4 load4(const void* base, int64_t i) {
  if constexpr (SRC16) {
    const uint2 u = __ldcs(reinterpret_cast<const uint2*>(base) + i);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
  } else {
    return __ldcs(reinterpret_cast<const float4*>(base) + i);
  }
}

template <bool SRC16>
__global__ void __launch_bounds__(kThreads)
commit_kernel(const void* __restrict__ snap, int64_t snap_layer4, const int32_t* accept,
              float4* __restrict__ cache, int64_t slot4, int64_t layer4, const int32_t* slot,
              int n_slots, int N, int64_t run4, int32_t* status) {
  pdl_enter();
  const int b = blockIdx.y, l = blockIdx.z;
  const int a = __ldg(accept + b);
  const int s = slot != nullptr ? __ldg(slot + b) : b;
  if (a < 0 || a >= N || s < 0 || s >= n_slots) {
    if (blockIdx.x == 0 && l == 0 && threadIdx.x == 0)
      report(status, (a < 0 || a >= N) ? GDN_ERR_ACCEPT_RANGE : GDN_ERR_SLOT_RANGE);
    return;
  }
  const int64_t src = l * snap_layer4 + ((int64_t)b * N + a) * run4;  // in groups of 4
  float4* dst = cache + l * layer4 + (int64_t)s * slot4;
  const int64_t base = (int64_t)blockIdx.x * kThreads * kUnroll + threadIdx.x;
  float4 t[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int64_t i = base + (int64_t)u * kThreads;
    if (i < run4) t[u] = load4<SRC16>(snap, src + i);
  }
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int64_t i = base + (int64_t)u * kThreads;
    if (i < run4) dst[i] = t[u];
  }
}

// Index-table commit: point each sequence's slot at its accepted node in the
// block's snapshot region ("TokenSpeed hits 580 tok/s", section "How they
// actually got there": move pointers, not data).  One thread per sequence.
__global__ void commit_index_kernel(const int32_t* accept, int B, int N, int base_slot,
                                    int32_t* slot, int32_t* status) {
  pdl_enter();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int a = __ldg(accept + b);
  if (a < 0 || a >= N) {
    report(status, GDN_ERR_ACCEPT_RANGE);
    return;
  }
  slot[b] = base_slot + b * N + a;
}

// Convolution-history commit ("Photon 2.6", section "Handling recurrent
// state": the convolution history is committed to the same boundary as the
// state).  Block (channel range, sequence b), one thread per channel: the new
// window is the last W elements of [old history, x of the accepted path],
// written in place after all old values are read.  Every thread checks the
// sequence and loads its old window first; a chain's path tail is
// acc-P+1 .. acc, a tree's is collected by thread 0 walking the parents.  E is
// the element type moved bit for bit.
constexpr int kMaxConvW = 8;

template <typename E>
__global__ void __launch_bounds__(256)
conv_commit_kernel(const E* __restrict__ x, E* __restrict__ state, int64_t slot_stride,
                   const int32_t* slot, int n_slots, const int32_t* parent,
                   const int32_t* accept, int N, int C, int W, int32_t* status) {
  pdl_enter();
  __shared__ int s_tail[kMaxConvW];
  __shared__ int s_count;
  const int b = blockIdx.y;
  const int64_t node0 = (int64_t)b * N;
  const int a = __ldg(accept + b);
  const int sl = slot != nullptr ? __ldg(slot + b) : b;
  const bool ok = a >= 0 && a < N && sl >= 0 && sl < n_slots;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  const bool mine = ok && c < C;
  E* h = state + (int64_t)(ok ? sl : 0) * slot_stride + (int64_t)c * W;
  E old[kMaxConvW];
#pragma unroll
  for (int w = 0; w < kMaxConvW; ++w)
    if (mine && w < W) old[w] = h[w];
  if (!ok) {
    if (blockIdx.x == 0 && threadIdx.x == 0)
      report(status, (a < 0 || a >= N) ? GDN_ERR_ACCEPT_RANGE : GDN_ERR_SLOT_RANGE);
    return;
  }
  int P;  // min(path length, W); the path tail, oldest first, in s_tail (tree)
  if (parent == nullptr) {
    P = min(a + 1, W);
  } else {
    if (threadIdx.x == 0) {
      int count = 0;
      bool valid = true;
      for (int n = 0; n < N && valid; ++n) {
        const int pp = __ldg(parent + node0 + n);
        valid = n == 0 ? pp == -1 : (pp >= 0 && pp < n);
      }
      if (valid) {
        int rev[kMaxConvW];
        for (int m = a; m >= 0 && count < W; m = __ldg(parent + node0 + m)) rev[count++] = m;
        for (int i = 0; i < count; ++i) s_tail[i] = rev[count - 1 - i];
      } else if (blockIdx.x == 0) {
        report(status, GDN_ERR_BAD_TREE);
      }
      s_count = valid ? count : -1;
    }
    __syncthreads();
    P = s_count;
    if (P < 0) return;
  }
  if (!mine) return;
  const int keep = W - P;  // old entries that stay: the newest `keep`
#pragma unroll
  for (int w = 0; w < kMaxConvW; ++w) {
    if (w < keep) {
      h[w] = old[w + P];
    } else if (w < W) {
      const int i = w - keep;  // 0 .. P-1: the path tail, oldest first
      const int node = parent == nullptr ? a - P + 1 + i : s_tail[i];
      h[w] = x[(node0 + node) * C + c];
    }
  }
}

}  // namespace

int launch_conv_commit(const void* x, bool bf16, void* state, int64_t slot_stride,
                       const int32_t* slot, int n_slots, const int32_t* parent,
                       const int32_t* accept, int B, int N, int C, int W, int32_t* status,
                       cudaStream_t stream) {
  const dim3 grid((unsigned)((C + 255) / 256), B);
  if (bf16)
    return launch_pdl(conv_commit_kernel<uint16_t>, grid, dim3(256), 0, stream,
                      static_cast<const uint16_t*>(x), static_cast<uint16_t*>(state),
                      slot_stride, slot, n_slots, parent, accept, N, C, W, status);
  return launch_pdl(conv_commit_kernel<uint32_t>, grid, dim3(256), 0, stream,
                    static_cast<const uint32_t*>(x), static_cast<uint32_t*>(state), slot_stride,
                    slot, n_slots, parent, accept, N, C, W, status);
}

int launch_commit_index(const int32_t* accept, int B, int N, int base_slot, int32_t* slot,
                        int32_t* status, cudaStream_t stream) {
  const int threads = 128;
  return launch_pdl(commit_index_kernel, dim3((B + threads - 1) / threads), dim3(threads), 0,
                    stream, accept, B, N, base_slot, slot, status);
}

int launch_commit(const void* snap, bool src16, int64_t snap_layer_stride, const int32_t* accept,
                  float* cache, int64_t cache_slot_stride, int64_t cache_layer_stride,
                  const int32_t* slot, int n_slots, int B, int N, int Hv, int dk, int dv,
                  int n_layers, int32_t* status, cudaStream_t stream) {
  const int64_t run4 = (int64_t)Hv * dk * dv / 4;
  const int64_t per_block = (int64_t)kThreads * kUnroll;
  const int64_t gx = (run4 + per_block - 1) / per_block;
  if (gx > 0x7fffffff) return GDN_ERR_UNSUPPORTED;
  const dim3 grid((unsigned)gx, B, n_layers);
  if (src16)
    return launch_pdl(commit_kernel<true>, grid, dim3(kThreads), 0, stream, snap,
                      snap_layer_stride / 4, accept, reinterpret_cast<float4*>(cache),
                      cache_slot_stride / 4, cache_layer_stride / 4, slot, n_slots, N, run4,
                      status);
  return launch_pdl(commit_kernel<false>, grid, dim3(kThreads), 0, stream, snap,
                    snap_layer_stride / 4, accept, reinterpret_cast<float4*>(cache),
                    cache_slot_stride / 4, cache_layer_stride / 4, slot, n_slots, N, run4,
                    status);
}

}  // namespace gdn
