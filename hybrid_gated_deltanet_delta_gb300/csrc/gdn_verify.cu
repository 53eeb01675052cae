// Verify kernels: the gated delta rule over a causal chain or a draft tree,
// every node's state persisted ("We got 207 tok/s with Qwen3.5-27B on an RTX
// 3090", list "Key wins": per-node states written inside the recurrence
// kernel instead of by a separate copy; "Photon 2.6", section "Handling
// recurrent state": the working state stays in registers across the block).
//
// Recurrence
// ----------
// The state of one value head is H = S^T (d_k x d_v, fp32, row-major).  With
// src(n) = n - 1 for a chain and the parent for a tree,
//     u_n = H_src(n)^T k_n,   delta_n = beta_n (v_n - alpha_n u_n),
//     H_n = alpha_n H_src(n) + k_n delta_n^T,   o_n = H_n^T q_n,
// which is S_n = alpha_n S_src(n) (I - beta_n k_n k_n^T) + beta_n v_n k_n^T,
// o_n = S_n q_n with the product distributed.  Column j of every H_n depends
// only on column j of the cached state, so a head splits into independent
// column slabs.
//
// Work decomposition
// ------------------
// A thread block owns a slab of WC columns of one (sequence, value head):
// grid = (dv / WC, Hv, B).  In a warp, lane = cg + CG*rl: cg picks 4 adjacent
// columns (a 16-byte vector), rl one of RL = 32/CG row lanes, and each lane
// keeps R consecutive rows x 4 columns of the state in registers (as float2
// pairs for the paired fp32 FMA).  Column sums reduce over the row lanes with
// warp shuffles.
//
// Chain (verify_kernel): the slab's d_k rows are split over NW row warps (one,
// or two when there are too few blocks to give every SM sub-partition a warp);
// the warps add their column sums through shared memory.  The node loop is
// built so that snapshot stores never wait on a reduction: the reduction that
// feeds node n+1 runs while node n updates and stores, since
//     u_{n+1} = H_n^T k_{n+1} = alpha_n (H_{n-1}^T k_{n+1}) + delta_n (k_n . k_{n+1}),
// and both sums on the right come from the registers BEFORE node n's update.
// Tree (tree_kernel, below): the block's warps take the nodes of each depth
// level in turn; a warp reduces its previous node's output sums in the same
// shuffle tree as its next node's u.
// q, k, v and the gates are staged with cp.async while the cached state
// loads.  Snapshots leave as 16-byte stores; a warp-wide store covers RL rows
// x WC*4 contiguous bytes.
//
// Variants (template flags): SNAP16 persists binary16 snapshots (RNE from
// the fp32 state; in a tree, a parent that is neither in the warp's registers
// nor stashed is continued from its binary16 snapshot); PREP takes raw q/k
// projections and gate pre-activations (the per-node inverse norms scale the
// reduced sums and delta instead of every element).  A chain may persist
// nothing at all and commit by replay, for which replay_kernel below re-runs
// the accepted path from the cached state; a tree that persists nothing is
// verified by the per-block solve in gdn_solve.cu.
#include <cuda_fp16.h>

#include "gdn_common.cuh"
#include "gdn_launch.h"

namespace gdn {
namespace {

constexpr unsigned FULL = 0xffffffffu;

template <int DK, int WC, int NW = 1>
struct Shape {
  static constexpr int CG = WC / 4;        // 16-byte column groups per row of the slab
  static constexpr int RL = 32 / CG;       // row lanes per warp
  static constexpr int R = DK / (RL * NW); // rows per lane (NW warps split the rows)
  static_assert(WC % 4 == 0 && 32 % CG == 0 && RL >= 2, "slab width");
  static_assert(R >= 1 && R * RL * NW == DK, "row split");
};

// Exchange slots for the cross-warp column sums: [2 buffers][NW][CG][XS]
constexpr int XS = 12;

__host__ __device__ constexpr int xchg_bytes(int nw, int WC) {
  return nw > 1 ? 2 * nw * (WC / 4) * XS * 4 : 0;
}

// Barrier over the NW warps of a block.
template <int NW>
__device__ __forceinline__ void block_sync() {
  if constexpr (NW == 1) __syncwarp();
  else __syncthreads();
}

template <int NW>
__device__ __forceinline__ bool block_all(bool x) {
  if constexpr (NW == 1) return __all_sync(0xffffffffu, x);
  else return __syncthreads_and(x) != 0;
}

// x[e] <- the sum of x[e] over the NW row warps of the block, added in warp
// order so that every warp gets the same bits.  Each warp's value must already
// be its full warp sum (all row lanes agree).  Exchanges alternate between two
// buffers, so one barrier per exchange suffices: a warp can only refill a
// buffer after the barrier of the next exchange, which every warp reaches
// after reading that buffer.
template <int NW, int CG, int NV>
__device__ __forceinline__ void warps_sum(float (&x)[NV], float* sx, int& xc, int wi, int cg,
                                          int rl) {
  if constexpr (NW > 1) {
    static_assert(NV <= XS, "exchange slot");
    float* buf = sx + (xc & 1) * (NW * CG * XS);
    ++xc;
    if (rl == 0) {
#pragma unroll
      for (int e = 0; e < NV; ++e) buf[(wi * CG + cg) * XS + e] = x[e];
    }
    __syncthreads();
    float acc[NV];
#pragma unroll
    for (int e = 0; e < NV; ++e) acc[e] = buf[cg * XS + e];
#pragma unroll
    for (int w = 1; w < NW; ++w)
#pragma unroll
      for (int e = 0; e < NV; ++e) acc[e] += buf[(w * CG + cg) * XS + e];
#pragma unroll
    for (int e = 0; e < NV; ++e) x[e] = acc[e];
  }
}

__host__ __device__ constexpr int round16(int x) { return (x + 15) & ~15; }

// Shared-memory plan of a chain block in bytes; every array starts on a
// 16-byte boundary.
struct SmemPlan {
  int q, k, v, a, b, inv, x, total;
};

__host__ __device__ inline SmemPlan smem_plan(int N, int DK, int WC, int esz, int nw = 1) {
  SmemPlan s{};
  s.q = 0;
  s.k = s.q + round16(N * DK * esz);
  s.v = s.k + round16(N * DK * esz);
  s.a = s.v + round16(N * WC * esz);
  s.b = s.a + round16(N * 4);
  s.inv = s.b + round16(N * 4);       // 1/|q_n|, 1/|k_n| (input preparation)
  s.x = s.inv + 2 * round16(N * 4);   // cross-warp sums (NW > 1)
  s.total = s.x + xchg_bytes(nw, WC);
  return s;
}

struct VerifyParams {
  const void* q;
  const void* k;
  const void* v;
  const float* alpha;
  const float* beta;
  const float* cache;
  const int32_t* slot;
  float* snap;
  __half* snap16;  // binary16 snapshots instead of snap (chain only)
  float* o;
  int32_t* status;
  const int32_t* parent;
  int32_t* depth_out;
  int64_t cache_slot_stride;
  int n_slots, N, Hk, Hv, dv, bf16;
  int hint;       // issue the pre-wait L2 hints
  int max_depth;  // tree: deepest node allowed (root = 1), 0 = no cap
};

// Launches of up to this many blocks (4 per SM on 152 SMs, one wave) issue
// the pre-wait L2 hints.  A larger launch runs in several waves behind a
// stream of snapshot writes that evicts the hinted lines before they are
// used (measured on 3072-block launches: 2 us slower per launch with hints).
constexpr int kHintBlocks = 608;

__device__ __forceinline__ void prefetch_l2(const void* a) {
  asm volatile("prefetch.global.L2 [%0];\n" ::"l"(a));
}

// Before the programmatic wait (which orders this kernel after the previous
// one on the stream): hint L2 with the lines the block is about to read, so
// that their DRAM latency overlaps the previous kernel's tail.  The slot table
// and the inputs may still be being written by that kernel: a stale or
// out-of-range slot only wastes (or skips) the hint, a prefetch never changes
// memory, and every load that feeds a result is issued after the wait (L2 is
// the point of coherence, and the hint bypasses L1).  Thread t of nt; the
// state rows are those of thread t's own layout (row0, R rows, 16-byte column
// group col), hinted once per 64-byte row segment.
template <int DK, int R>
__device__ __forceinline__ void prefetch_block(const VerifyParams& p, int b, int h, int hk, int j0,
                                               bool state, int row0, int col, int t, int nt) {
  const int N = p.N, dv = p.dv, esz = p.bf16 ? 2 : 4;
  if (state) {
    const int s0 = p.slot != nullptr ? __ldcg(p.slot + b) : b;
    if (s0 >= 0 && s0 < p.n_slots) {
      const float* c0 = p.cache + (int64_t)s0 * p.cache_slot_stride + (int64_t)h * DK * dv +
                        (int64_t)row0 * dv + col;
#pragma unroll
      for (int m = 0; m < R; ++m) prefetch_l2(c0 + (int64_t)m * dv);
    }
  }
  // q and k rows of the block's q/k head (128-byte lines), v segments
  const int per = (DK * esz + 127) / 128;
  const int qk_lines = N * per;
  const int64_t node0 = (int64_t)b * N;
  for (int i = t; i < 2 * qk_lines + N; i += nt) {
    if (i < 2 * qk_lines) {
      const int which = i / qk_lines, r = i - which * qk_lines;
      const int n = r / per, part = r - n * per;
      const char* base = static_cast<const char*>(which ? p.q : p.k);
      prefetch_l2(base + ((node0 + n) * p.Hk + hk) * DK * esz + part * 128);
    } else {
      const int n = i - 2 * qk_lines;
      prefetch_l2(static_cast<const char*>(p.v) + ((node0 + n) * p.Hv + h) * dv * esz +
                  (int64_t)j0 * esz);
    }
  }
}

// Start copying n_rows rows of row_bytes bytes (row r at src + r*src_stride)
// to dst + r*row_bytes with 16-byte cp.async, thread t of nt.
__device__ __forceinline__ void stage_rows(char* dst, const char* src, int64_t src_stride,
                                           int n_rows, int row_bytes, int t, int nt) {
  const int per_row = row_bytes / 16;
  for (int idx = t; idx < n_rows * per_row; idx += nt) {
    const int r = idx / per_row, c = idx - r * per_row;
    cp_async16(dst + r * row_bytes + c * 16, src + r * src_stride + c * 16);
  }
}

// x[0..R) = R consecutive values of a staged row (bf16 or fp32), as fp32.
template <int R>
__device__ __forceinline__ void load_rows(float (&x)[R], const char* row, int first, bool bf16) {
  if (bf16) {
    const uint16_t* s = reinterpret_cast<const uint16_t*>(row) + first;
    if constexpr (R % 8 == 0) {
#pragma unroll
      for (int m = 0; m < R; m += 8) {
        const uint4 t = *reinterpret_cast<const uint4*>(s + m);
        const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          x[m + 2 * e] = __uint_as_float(w[e] << 16);
          x[m + 2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
        }
      }
    } else {
#pragma unroll
      for (int m = 0; m < R; ++m) x[m] = bf16_to_f32(s[m]);
    }
  } else {
    const float* s = reinterpret_cast<const float*>(row) + first;
    if constexpr (R % 4 == 0) {
#pragma unroll
      for (int m = 0; m < R; m += 4) {
        const float4 t = *reinterpret_cast<const float4*>(s + m);
        x[m] = t.x; x[m + 1] = t.y; x[m + 2] = t.z; x[m + 3] = t.w;
      }
    } else {
#pragma unroll
      for (int m = 0; m < R; ++m) x[m] = s[m];
    }
  }
}

__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }

// Input preparation from raw projections: 1/|x| of `rows` staged rows of DK
// elements (bf16 or fp32) into inv[] (0 for a zero row, which then stays
// zero), one row per thread; and the gates alpha = exp(-softplus(a)) =
// 1/(1 + e^a), beta = sigmoid(b) = 1/(1 + e^-b) in place.
template <int DK>
__device__ __forceinline__ void prep_rows(const char* rows_base, int rows, bool bf16, float* inv,
                                          int t, int nt) {
  for (int r = t; r < rows; r += nt) {
    float ss = 0.f;
    if (bf16) {
      const uint4* s = reinterpret_cast<const uint4*>(rows_base + (size_t)r * DK * 2);
#pragma unroll 4
      for (int c = 0; c < DK / 8; ++c) {
        const uint4 t = s[c];
        const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xffff0000u);
          ss = fmaf(lo, lo, fmaf(hi, hi, ss));
        }
      }
    } else {
      const float4* s = reinterpret_cast<const float4*>(rows_base + (size_t)r * DK * 4);
#pragma unroll 4
      for (int c = 0; c < DK / 4; ++c) {
        const float4 t = s[c];
        ss = fmaf(t.x, t.x, fmaf(t.y, t.y, fmaf(t.z, t.z, fmaf(t.w, t.w, ss))));
      }
    }
    inv[r] = ss > 0.f ? rsqrtf(ss) : 0.f;
  }
}

__device__ __forceinline__ void prep_gates(float* a, float* b, int n_rows, int t, int nt) {
  for (int r = t; r < n_rows; r += nt) {
    a[r] = 1.f / (1.f + __expf(a[r]));
    b[r] = 1.f / (1.f + __expf(-b[r]));
  }
}

template <int DK, int WC, int NW, bool SNAP16, bool PREP>
__global__ void __launch_bounds__(32 * NW) verify_kernel(const VerifyParams p) {
  using S = Shape<DK, WC, NW>;
  constexpr int R = S::R;
  constexpr int NT = 32 * NW;
  if (p.hint) {
    const int t = threadIdx.x, ln = t & 31;
    prefetch_block<DK, R>(p, blockIdx.z, blockIdx.y, blockIdx.y / (p.Hv / p.Hk),
                          blockIdx.x * WC, ln % S::CG == 0,
                          (t >> 5) * (DK / NW) + (ln / S::CG) * R, blockIdx.x * WC, t, NT);
  }
  pdl_enter();
  extern __shared__ __align__(16) char smem[];
  const int N = p.N;
  const bool bf16 = p.bf16 != 0;
  const int esz = bf16 ? 2 : 4;
  const SmemPlan pl = smem_plan(N, DK, WC, esz, NW);
  char* sq = smem + pl.q;
  char* sk = smem + pl.k;
  char* sv = smem + pl.v;
  float* sa = reinterpret_cast<float*>(smem + pl.a);
  float* sb = reinterpret_cast<float*>(smem + pl.b);
  float* sinvq = reinterpret_cast<float*>(smem + pl.inv);
  float* sinvk = sinvq + round16(N * 4) / 4;
  float* sx = reinterpret_cast<float*>(smem + pl.x);
  int xc = 0;  // cross-warp exchanges so far

  const int tid = threadIdx.x, lane = tid & 31, wi = tid >> 5;
  const int cg = lane % S::CG, rl = lane / S::CG;
  const int j0 = blockIdx.x * WC, h = blockIdx.y, b = blockIdx.z;
  const int hk = h / (p.Hv / p.Hk);
  const bool lead = blockIdx.x == 0 && blockIdx.y == 0;  // per-sequence reporting
  const int dv = p.dv;
  const int row0 = wi * (DK / NW) + rl * R;

  // ---- stage q, k, v, gates (independent of the slot: issued first)
  {
    const int64_t node0 = (int64_t)b * N;
    const char* qb = static_cast<const char*>(p.q) + ((node0 * p.Hk + hk) * DK) * esz;
    const char* kb = static_cast<const char*>(p.k) + ((node0 * p.Hk + hk) * DK) * esz;
    const char* vb = static_cast<const char*>(p.v) + ((node0 * p.Hv + h) * dv + j0) * esz;
    stage_rows(sk, kb, (int64_t)p.Hk * DK * esz, N, DK * esz, tid, NT);
    stage_rows(sq, qb, (int64_t)p.Hk * DK * esz, N, DK * esz, tid, NT);
    stage_rows(sv, vb, (int64_t)p.Hv * dv * esz, N, WC * esz, tid, NT);
    for (int n = tid; n < N; n += NT) {
      cp_async4(sa + n, p.alpha + (node0 + n) * p.Hv + h);
      cp_async4(sb + n, p.beta + (node0 + n) * p.Hv + h);
    }
  }

  const int sl = p.slot != nullptr ? __ldg(p.slot + b) : b;
  if (sl < 0 || sl >= p.n_slots) {
    cp_async_wait_all();
    if (lead && tid == 0) report(p.status, GDN_ERR_SLOT_RANGE);
    return;
  }

  // ---- the cached state -> registers (an L2 load: with an index-table
  //      commit the cache is this block's snapshot region, written below)
  float2 H[R][2];
  {
    const float* c0 = p.cache + (int64_t)sl * p.cache_slot_stride + (int64_t)h * DK * dv +
                      (int64_t)row0 * dv + j0 + cg * 4;
#pragma unroll
    for (int m = 0; m < R; ++m) {
      const float4 t = ld_cg_f4(c0 + (int64_t)m * dv);
      H[m][0] = make_float2(t.x, t.y);
      H[m][1] = make_float2(t.z, t.w);
    }
  }
  cp_async_wait_all();
  block_sync<NW>();

  if constexpr (PREP) {
    // raw projections: norms of q and k, gates from their pre-activations
    prep_rows<DK>(sq, N, bf16, sinvq, tid, NT);
    prep_rows<DK>(sk, N, bf16, sinvk, tid, NT);
    prep_gates(sa, sb, N, tid, NT);
    block_sync<NW>();
  }

  // ---- u_0 = H0^T k_0
  float kn[R];  // k of the current node
  load_rows<R>(kn, sk, row0, bf16);
  float u[4];
  {
    float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
#pragma unroll
    for (int m = 0; m < R; ++m) {
      a01 = __ffma2_rn(H[m][0], f2(kn[m]), a01);
      a23 = __ffma2_rn(H[m][1], f2(kn[m]), a23);
    }
    u[0] = a01.x; u[1] = a01.y; u[2] = a23.x; u[3] = a23.y;
#pragma unroll
    for (int off = S::CG; off < 32; off <<= 1)
#pragma unroll
      for (int c = 0; c < 4; ++c) u[c] += __shfl_xor_sync(FULL, u[c], off);
    warps_sum<NW, S::CG>(u, sx, xc, wi, cg, rl);
    if constexpr (PREP) {
#pragma unroll
      for (int c = 0; c < 4; ++c) u[c] *= sinvk[0];
    }
  }

  const int64_t node_stride = (int64_t)p.Hv * DK * dv;
  const int64_t lane_off = ((int64_t)b * N * p.Hv + h) * DK * dv + (int64_t)row0 * dv + j0 + cg * 4;
  float* snap_h = p.snap == nullptr ? nullptr : p.snap + lane_off;
  __half* snap16_h = SNAP16 ? p.snap16 + lane_off : nullptr;
  float* o_h = p.o + ((int64_t)b * N * p.Hv + h) * dv + j0 + cg * 4;

  // The shuffle tree of node n reduces the look-ahead sums for u_{n+1} (from
  // the state before node n's update) together with the output sums of node
  // n-1, so that it does not wait for node n's update: the update, its
  // output partials and the snapshot stores overlap the tree's latency, and
  // o_{n-1} is stored one node late (o_{N-1} after the loop).
  float po[4] = {0.f, 0.f, 0.f, 0.f};  // output partials of the previous node
  float iq_prev = 1.f;
  for (int n = 0; n < N; ++n) {
    const bool has_next = n + 1 < N;
    float knx[R];  // k of node n+1
    if (has_next) {
      load_rows<R>(knx, sk + (n + 1) * DK * esz, row0, bf16);
    } else {
#pragma unroll
      for (int m = 0; m < R; ++m) knx[m] = 0.f;
    }
    float qr[R];
    load_rows<R>(qr, sq + n * DK * esz, row0, bf16);
    float vj[4];
    load_rows<4>(vj, sv + n * WC * esz, cg * 4, bf16);
    const float al = sa[n], be = sb[n];
    // 1/|k_n|, 1/|k_{n+1}|, 1/|q_n| when the inputs are raw projections
    const float ik = PREP ? sinvk[n] : 1.f;
    const float ikx = PREP && has_next ? sinvk[n + 1] : 1.f;
    const float iq = PREP ? sinvq[n] : 1.f;

    // (c) partial sums for u_{n+1}: from the registers before node n's update
    float2 w01 = make_float2(0.f, 0.f), w23 = make_float2(0.f, 0.f);
    float kk = 0.f;
#pragma unroll
    for (int m = 0; m < R; ++m) {
      w01 = __ffma2_rn(H[m][0], f2(knx[m]), w01);
      w23 = __ffma2_rn(H[m][1], f2(knx[m]), w23);
      kk = fmaf(kn[m], knx[m], kk);
    }
    // (e) one shuffle tree for those 4 + 1 sums and the previous node's 4
    float red[9] = {w01.x, w01.y, w23.x, w23.y, kk, po[0], po[1], po[2], po[3]};
#pragma unroll
    for (int off = S::CG; off < 32; off <<= 1)
#pragma unroll
      for (int i = 0; i < 9; ++i) red[i] += __shfl_xor_sync(FULL, red[i], off);

    // (d) delta_n, update, output partial (independent of the tree above)
    float d[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) d[c] = be * (vj[c] - al * u[c]);
    const float2 d01 = make_float2(d[0] * ik, d[1] * ik), d23 = make_float2(d[2] * ik, d[3] * ik);
    const float2 al2 = f2(al);
    float2 o01 = make_float2(0.f, 0.f), o23 = make_float2(0.f, 0.f);
#pragma unroll
    for (int m = 0; m < R; ++m) {
      H[m][0] = __ffma2_rn(f2(kn[m]), d01, __fmul2_rn(al2, H[m][0]));
      H[m][1] = __ffma2_rn(f2(kn[m]), d23, __fmul2_rn(al2, H[m][1]));
      o01 = __ffma2_rn(H[m][0], f2(qr[m]), o01);
      o23 = __ffma2_rn(H[m][1], f2(qr[m]), o23);
    }
    // (f) persist (a chain verified for a replay commit keeps no snapshots)
    if constexpr (SNAP16) {
      // binary16, round to nearest even: 8 bytes per lane and row
      __half* dst = snap16_h + (int64_t)n * node_stride;
#pragma unroll
      for (int m = 0; m < R; ++m) {
        const __half2 lo = __floats2half2_rn(H[m][0].x, H[m][0].y);
        const __half2 hi = __floats2half2_rn(H[m][1].x, H[m][1].y);
        *reinterpret_cast<uint2*>(dst + (int64_t)m * dv) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&lo),
                       *reinterpret_cast<const uint32_t*>(&hi));
      }
    } else if (p.snap != nullptr) {
      float* dst = snap_h + (int64_t)n * node_stride;
#pragma unroll
      for (int m = 0; m < R; ++m)
        st_f4(dst + (int64_t)m * dv, H[m][0].x, H[m][0].y, H[m][1].x, H[m][1].y);
    }
    // cross-warp sums, u_{n+1}, and the previous node's output
    warps_sum<NW, S::CG>(red, sx, xc, wi, cg, rl);
#pragma unroll
    for (int c = 0; c < 4; ++c) u[c] = fmaf(al, red[c] * ikx, d[c] * (red[4] * (ik * ikx)));
    if (n > 0 && rl == 0 && wi == 0)
      st_f4(o_h + (int64_t)(n - 1) * p.Hv * dv, red[5] * iq_prev, red[6] * iq_prev,
            red[7] * iq_prev, red[8] * iq_prev);
    po[0] = o01.x; po[1] = o01.y; po[2] = o23.x; po[3] = o23.y;
    iq_prev = iq;
#pragma unroll
    for (int m = 0; m < R; ++m) kn[m] = knx[m];
  }
  // the last node's output
#pragma unroll
  for (int off = S::CG; off < 32; off <<= 1)
#pragma unroll
    for (int c = 0; c < 4; ++c) po[c] += __shfl_xor_sync(FULL, po[c], off);
  warps_sum<NW, S::CG>(po, sx, xc, wi, cg, rl);
  if (rl == 0 && wi == 0)
    st_f4(o_h + (int64_t)(N - 1) * p.Hv * dv, po[0] * iq_prev, po[1] * iq_prev, po[2] * iq_prev,
          po[3] * iq_prev);
}

// ------------------------------------------------------------------ tree
// Tree verification, level by level.  Nodes of equal depth depend on nodes of
// smaller depth only, so the TW warps of a block (one column slab of one
// (sequence, value head)) take the nodes of each depth level in turn, all
// rows of the slab per warp (the verify lane layout with one row warp).  A
// node starts from its parent's state: still in the registers of the warp
// that computed it when that warp takes the child, otherwise read back from
// the parent's snapshot, which a warp of this block stored one level earlier
// (the barrier between levels makes it visible; it is read through L2).  Each
// node reduces u = H^T k before its update and o = H'^T q after it.
// Tree state stash: the states of up to kTreeSlots nodes of a level that have
// children stay in shared memory for the next level (two level buffers), so
// their children read them from shared memory instead of L2.  The tree's
// shape (depths, walk order, level starts, stash slots) is worked out by one
// warp with shuffles while the block's inputs and the cached state load.
constexpr int kTreeSlots = 3;

struct TreePlan {
  int q, k, v, a, b, par, dep, ord, lev, slot, inv, stash, total;
};

__host__ __device__ inline TreePlan tree_plan(int N, int DK, int WC, int esz) {
  TreePlan s{};
  s.q = 0;
  s.k = s.q + round16(N * DK * esz);
  s.v = s.k + round16(N * DK * esz);
  s.a = s.v + round16(N * WC * esz);
  s.b = s.a + round16(N * 4);
  s.par = s.b + round16(N * 4);
  s.dep = s.par + round16(N * 4);        // depth of each node (root = 1)
  s.ord = s.dep + round16(N * 4);        // nodes by depth, then index
  s.lev = s.ord + round16(N * 4);        // lev[L] = first position of depth L
  s.slot = s.lev + round16((N + 2) * 4); // stash slot of each node, -1 = none
  s.inv = s.slot + round16(N * 4);       // 1/|q_n|, 1/|k_n| (input preparation)
  s.stash = s.inv + 2 * round16(N * 4);  // [2 levels][kTreeSlots][DK * WC] fp32
  s.total = s.stash + 2 * kTreeSlots * DK * WC * 4;
  return s;
}

// The value of node m (0 <= m < 64) from the two per-lane registers that
// hold nodes lane and lane + 32 (every lane of the warp must call).
__device__ __forceinline__ int node_val(int v0, int v1, int m) {
  const int a = __shfl_sync(FULL, v0, m & 31), b = __shfl_sync(FULL, v1, m & 31);
  return m < 32 ? a : b;
}

// The parents of nodes lane and lane + 32 of a tree of N <= 64 nodes (-2
// past the end), read through L2.
__device__ __forceinline__ void load_parents(const int32_t* parent, int N, int& p0, int& p1) {
  const int lane = threadIdx.x & 31;
  p0 = lane < N ? __ldcg(parent + lane) : -2;
  p1 = lane + 32 < N ? __ldcg(parent + lane + 32) : -2;
}

// The shape of a tree of N <= 64 nodes, by one warp: lane l takes nodes l
// and l + 32, whose parents p0 and p1 it holds (load_parents).  Writes
// par[], dep[] (root = 1), ord[] (the walk order: by depth, then index),
// lev[L] (first position of depth L, L = 1 .. N + 1) and slot[] (the stash
// slot: the rank of the node among the nodes of its depth that have
// children, when below kTreeSlots; otherwise -1).  Returns 0, 1 for a
// malformed parent array, 2 for a tree deeper than max_depth (depths
// written); the same value in every lane.  A pure function of the parents,
// N and max_depth: any values, valid or not, give a result in bounded time.
__device__ int tree_shape(int p0, int p1, int N, int max_depth, int* spar, int* sdep, int* sord,
                          int* slev, int* sslot) {
  const int lane = threadIdx.x & 31;
  const int n0 = lane, n1 = lane + 32;
  const bool ok0 = n0 >= N || (n0 == 0 ? p0 == -1 : (p0 >= 0 && p0 < n0));
  const bool ok1 = n1 >= N || (p1 >= 0 && p1 < n1);
  if (!__all_sync(FULL, ok0 && ok1)) return 1;
  // depths by pointer jumping: d counts the nodes from n up to (not
  // including) the ancestor a; six rounds cover 64 levels
  int d0 = n0 < N ? 1 : 0, d1 = n1 < N ? 1 : 0, a0 = p0, a1 = p1;
#pragma unroll
  for (int r = 0; r < 6; ++r) {
    const int x0 = node_val(d0, d1, a0 < 0 ? 0 : a0), y0 = node_val(a0, a1, a0 < 0 ? 0 : a0);
    const int x1 = node_val(d0, d1, a1 < 0 ? 0 : a1), y1 = node_val(a0, a1, a1 < 0 ? 0 : a1);
    if (a0 >= 0) { d0 += x0; a0 = y0; }
    if (a1 >= 0) { d1 += x1; a1 = y1; }
  }
  if (n0 < N) { spar[n0] = p0; sdep[n0] = d0; }
  if (n1 < N) { spar[n1] = p1; sdep[n1] = d1; }
  const bool shallow = max_depth <= 0 || ((n0 >= N || d0 <= max_depth) && (n1 >= N || d1 <= max_depth));
  if (!__all_sync(FULL, shallow)) return 2;
  // walk positions, level starts (lane l: depths l + 1 and l + 33) and which
  // nodes have children, in one pass over the nodes
  int pos0 = 0, pos1 = 0, lv0 = 0, lv1 = 0;
  bool ch0 = false, ch1 = false;
  for (int m = 0; m < N; ++m) {
    const int dm = node_val(d0, d1, m), pm = node_val(p0, p1, m);
    pos0 += (dm < d0 || (dm == d0 && m < n0)) ? 1 : 0;
    pos1 += (dm < d1 || (dm == d1 && m < n1)) ? 1 : 0;
    lv0 += dm < lane + 1 ? 1 : 0;
    lv1 += dm < lane + 33 ? 1 : 0;
    ch0 = ch0 || pm == n0;
    ch1 = ch1 || pm == n1;
  }
  if (n0 < N) sord[pos0] = n0;
  if (n1 < N) sord[pos1] = n1;
  if (lane + 1 <= N) slev[lane + 1] = lv0;
  if (lane + 33 <= N) slev[lane + 33] = lv1;
  if (lane == 0) slev[N + 1] = N;  // past the deepest level
  // stash slots: rank among the nodes of the same depth that have children
  int r0 = 0, r1 = 0;
  const int c0 = ch0 ? 1 : 0, c1 = ch1 ? 1 : 0;
  for (int m = 0; m < N; ++m) {
    const int dm = node_val(d0, d1, m), cm = node_val(c0, c1, m);
    r0 += (cm != 0 && dm == d0 && m < n0) ? 1 : 0;
    r1 += (cm != 0 && dm == d1 && m < n1) ? 1 : 0;
  }
  if (n0 < N) sslot[n0] = ch0 && r0 < kTreeSlots ? r0 : -1;
  if (n1 < N) sslot[n1] = ch1 && r1 < kTreeSlots ? r1 : -1;
  return 0;
}

// Three blocks per SM keep a single-wave launch of 384 slab blocks resident.
template <int DK, int WC, int TW, bool PREP, bool SNAP16>
__global__ void __launch_bounds__(32 * TW, 3) tree_kernel(const VerifyParams p) {
  using S = Shape<DK, WC, 1>;
  constexpr int R = S::R;
  constexpr int NT = 32 * TW;
  if (p.hint) {
    const int t = threadIdx.x, ln = t & 31;
    prefetch_block<DK, R>(p, blockIdx.z, blockIdx.y, blockIdx.y / (p.Hv / p.Hk),
                          blockIdx.x * WC, t < 32 && ln % S::CG == 0, (ln / S::CG) * R,
                          blockIdx.x * WC, t, NT);
  }
  extern __shared__ __align__(16) char smem[];
  const int N = p.N;
  const bool bf16 = p.bf16 != 0;
  const int esz = bf16 ? 2 : 4;
  const TreePlan pl = tree_plan(N, DK, WC, esz);
  char* sq = smem + pl.q;
  char* sk = smem + pl.k;
  char* sv = smem + pl.v;
  float* sa = reinterpret_cast<float*>(smem + pl.a);
  float* sb = reinterpret_cast<float*>(smem + pl.b);
  int* spar = reinterpret_cast<int*>(smem + pl.par);
  int* sdep = reinterpret_cast<int*>(smem + pl.dep);
  int* sord = reinterpret_cast<int*>(smem + pl.ord);
  int* slev = reinterpret_cast<int*>(smem + pl.lev);
  int* sslot = reinterpret_cast<int*>(smem + pl.slot);
  float* sinvq = reinterpret_cast<float*>(smem + pl.inv);
  float* sinvk = sinvq + round16(N * 4) / 4;
  float* stash = reinterpret_cast<float*>(smem + pl.stash);

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int cg = lane % S::CG, rl = lane / S::CG;
  const int j0 = blockIdx.x * WC, h = blockIdx.y, b = blockIdx.z;
  const int hk = h / (p.Hv / p.Hk);
  const bool lead = blockIdx.x == 0 && blockIdx.y == 0;  // per-sequence reporting
  const int dv = p.dv;
  const int row0 = rl * R;
  const int64_t node0 = (int64_t)b * N;

  // ---- the tree's shape, by the last warp, from the parent array as it
  //      reads before the programmatic wait; after the wait the warp reads
  //      the array again and works the shape out anew only if a value
  //      changed, so the analysis is off the block's critical path whenever
  //      the parents were in place before this kernel started (shared memory
  //      is the block's own, so writing it before the wait is safe).  Only
  //      in a launch whose blocks are all resident while the previous kernel
  //      runs (the one that takes the L2 hints): a block of a later wave
  //      finds the wait already passed and works the shape out after its
  //      copies have left, as they land
  const bool early = p.hint != 0;
  int gp0 = -2, gp1 = -2, shape = 0;
  if (early && w == TW - 1) {
    load_parents(p.parent + node0, N, gp0, gp1);
    shape = tree_shape(gp0, gp1, N, p.max_depth, spar, sdep, sord, slev, sslot);
  }
  pdl_enter();

  // ---- stage q, k, v, gates
  {
    const char* qb = static_cast<const char*>(p.q) + ((node0 * p.Hk + hk) * DK) * esz;
    const char* kb = static_cast<const char*>(p.k) + ((node0 * p.Hk + hk) * DK) * esz;
    const char* vb = static_cast<const char*>(p.v) + ((node0 * p.Hv + h) * dv + j0) * esz;
    stage_rows(sk, kb, (int64_t)p.Hk * DK * esz, N, DK * esz, tid, NT);
    stage_rows(sq, qb, (int64_t)p.Hk * DK * esz, N, DK * esz, tid, NT);
    stage_rows(sv, vb, (int64_t)p.Hv * dv * esz, N, WC * esz, tid, NT);
    for (int n = tid; n < N; n += NT) {
      cp_async4(sa + n, p.alpha + (node0 + n) * p.Hv + h);
      cp_async4(sb + n, p.beta + (node0 + n) * p.Hv + h);
    }
  }
  // the last warp reads the parents again; the root's warp starts the
  // cached state on its way
  float2 H[R][2];
  const int64_t state_off = (int64_t)h * DK * dv + (int64_t)row0 * dv + j0 + cg * 4;
  auto load_state = [&](int s) {
    const float* c0 = p.cache + (int64_t)s * p.cache_slot_stride + state_off;
#pragma unroll
    for (int m = 0; m < R; ++m) {
      const float4 t = ld_cg_f4(c0 + (int64_t)m * dv);
      H[m][0] = make_float2(t.x, t.y);
      H[m][1] = make_float2(t.z, t.w);
    }
  };
  int np0 = -2, np1 = -2;
  if (w == TW - 1) load_parents(p.parent + node0, N, np0, np1);
  const int sl = p.slot != nullptr ? __ldg(p.slot + b) : b;
  if (sl < 0 || sl >= p.n_slots) {
    cp_async_wait_all();
    if (lead && tid == 0) report(p.status, GDN_ERR_SLOT_RANGE);
    return;
  }
  if (w == 0) load_state(sl);
  const float* cache_h = p.cache + (int64_t)sl * p.cache_slot_stride + state_off;
  int held = w == 0 ? -1 : -2;  // node whose state this warp holds (-1: the cache)
  // the shape's verdict (0 ok, 1 malformed parent array, 2 deeper than the
  // caller's cap) in lev[0], which the walk does not use
  if (w == TW - 1) {
    if (!early || __any_sync(FULL, np0 != gp0 || np1 != gp1))
      shape = tree_shape(np0, np1, N, p.max_depth, spar, sdep, sord, slev, sslot);
    if (lane == 0) slev[0] = shape;
  }
  cp_async_wait_all();
  __syncthreads();
  const int bad = slev[0];

  if (bad != 0) {
    if (lead && tid == 0) report(p.status, GDN_ERR_BAD_TREE);
    if (bad == 2 && lead && p.depth_out != nullptr)  // skipped; depths reported
      for (int n = tid; n < N; n += NT) p.depth_out[(int64_t)b * N + n] = sdep[n];
    return;
  }
  if constexpr (PREP) {
    prep_rows<DK>(sq, N, bf16, sinvq, tid, NT);
    prep_rows<DK>(sk, N, bf16, sinvk, tid, NT);
    prep_gates(sa, sb, N, tid, NT);
    __syncthreads();
  }
  // a stash slot holds each lane's R x 4 block lane-major: row m of lane l at
  // float offset (m*32 + l)*4, so every slot access is bank-conflict free
  constexpr int kSlot = DK * WC;

  const int64_t node_stride = (int64_t)p.Hv * DK * dv;
  const int64_t lane_off = ((int64_t)b * N * p.Hv + h) * DK * dv + (int64_t)row0 * dv + j0 + cg * 4;
  float* snap_h = SNAP16 ? nullptr : p.snap + lane_off;
  __half* snap16_h = SNAP16 ? p.snap16 + lane_off : nullptr;
  float* o_h = p.o + ((int64_t)b * N * p.Hv + h) * dv + j0 + cg * 4;

  // A warp's pending output: the output sums of the last node it formed are
  // reduced in the shuffle tree of its next node's u (or after the walk), so
  // that each node takes one tree, not two.
  float po[4] = {0.f, 0.f, 0.f, 0.f};
  int pn = -1;
  float piq = 1.f;
  for (int L = 1; L <= N && slev[L] < N; ++L) {
    for (int i = slev[L] + w; i < slev[L + 1]; i += TW) {
      const int n = sord[i], par = spar[n];
      if (par != held) {
        const int pslot = par < 0 ? -1 : sslot[par];
        if (pslot >= 0) {
          const float* rs = stash + (((L - 1) & 1) * kTreeSlots + pslot) * kSlot + lane * 4;
#pragma unroll
          for (int m = 0; m < R; ++m) {
            const float4 t = *reinterpret_cast<const float4*>(rs + m * 128);
            H[m][0] = make_float2(t.x, t.y);
            H[m][1] = make_float2(t.z, t.w);
          }
        } else if (SNAP16 && par >= 0) {
          // binary16 snapshots: the parent continues from its rounded state
          const __half* from = snap16_h + (int64_t)par * node_stride;
#pragma unroll
          for (int m = 0; m < R; ++m) {
            const uint2 t = __ldcg(reinterpret_cast<const uint2*>(from + (int64_t)m * dv));
            H[m][0] = __half22float2(*reinterpret_cast<const __half2*>(&t.x));
            H[m][1] = __half22float2(*reinterpret_cast<const __half2*>(&t.y));
          }
        } else {
          const float* from = par < 0 ? cache_h : snap_h + (int64_t)par * node_stride;
#pragma unroll
          for (int m = 0; m < R; ++m) {
            const float4 t = ld_cg_f4(from + (int64_t)m * dv);
            H[m][0] = make_float2(t.x, t.y);
            H[m][1] = make_float2(t.z, t.w);
          }
        }
      }
      float kn[R], qr[R], vj[4];
      load_rows<R>(kn, sk + n * DK * esz, row0, bf16);
      load_rows<R>(qr, sq + n * DK * esz, row0, bf16);
      load_rows<4>(vj, sv + n * WC * esz, cg * 4, bf16);
      const float al = sa[n], be = sb[n];
      const float ik = PREP ? sinvk[n] : 1.f;
      const float iq = PREP ? sinvq[n] : 1.f;

      // u_n = H_par^T k_n, reduced together with the pending output sums
      float red[8];
      {
        float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
#pragma unroll
        for (int m = 0; m < R; ++m) {
          a01 = __ffma2_rn(H[m][0], f2(kn[m]), a01);
          a23 = __ffma2_rn(H[m][1], f2(kn[m]), a23);
        }
        red[0] = a01.x; red[1] = a01.y; red[2] = a23.x; red[3] = a23.y;
        red[4] = po[0]; red[5] = po[1]; red[6] = po[2]; red[7] = po[3];
#pragma unroll
        for (int off = S::CG; off < 32; off <<= 1)
#pragma unroll
          for (int c = 0; c < 8; ++c) red[c] += __shfl_xor_sync(FULL, red[c], off);
      }
      if (pn >= 0 && rl == 0)
        st_f4(o_h + (int64_t)pn * p.Hv * dv, red[4] * piq, red[5] * piq, red[6] * piq,
              red[7] * piq);
      // delta_n, update, o_n partials
      float d[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) d[c] = be * (vj[c] - al * (red[c] * ik));
      const float2 d01 = make_float2(d[0] * ik, d[1] * ik), d23 = make_float2(d[2] * ik, d[3] * ik);
      const float2 al2 = f2(al);
      float2 o01 = make_float2(0.f, 0.f), o23 = make_float2(0.f, 0.f);
#pragma unroll
      for (int m = 0; m < R; ++m) {
        H[m][0] = __ffma2_rn(f2(kn[m]), d01, __fmul2_rn(al2, H[m][0]));
        H[m][1] = __ffma2_rn(f2(kn[m]), d23, __fmul2_rn(al2, H[m][1]));
        o01 = __ffma2_rn(H[m][0], f2(qr[m]), o01);
        o23 = __ffma2_rn(H[m][1], f2(qr[m]), o23);
      }
      if constexpr (SNAP16) {
        // binary16, round to nearest even: 8 bytes per lane and row
        __half* dst = snap16_h + (int64_t)n * node_stride;
#pragma unroll
        for (int m = 0; m < R; ++m) {
          const __half2 lo = __floats2half2_rn(H[m][0].x, H[m][0].y);
          const __half2 hi = __floats2half2_rn(H[m][1].x, H[m][1].y);
          *reinterpret_cast<uint2*>(dst + (int64_t)m * dv) =
              make_uint2(*reinterpret_cast<const uint32_t*>(&lo),
                         *reinterpret_cast<const uint32_t*>(&hi));
        }
      } else {
        // streaming stores (evict first in L2): measured 4 % faster per
        // verify + commit step of a 22-node tree than plain stores
        float* dst = snap_h + (int64_t)n * node_stride;
#pragma unroll
        for (int m = 0; m < R; ++m)
          __stcs(reinterpret_cast<float4*>(dst + (int64_t)m * dv),
                 make_float4(H[m][0].x, H[m][0].y, H[m][1].x, H[m][1].y));
      }
      const int myslot = sslot[n];
      if (myslot >= 0) {
        float* to = stash + ((L & 1) * kTreeSlots + myslot) * kSlot + lane * 4;
#pragma unroll
        for (int m = 0; m < R; ++m)
          *reinterpret_cast<float4*>(to + m * 128) =
              make_float4(H[m][0].x, H[m][0].y, H[m][1].x, H[m][1].y);
      }
      po[0] = o01.x; po[1] = o01.y; po[2] = o23.x; po[3] = o23.y;
      pn = n;
      piq = iq;
      held = n;
    }
    __syncthreads();  // this level's snapshots are visible to the next level
  }
  if (pn >= 0) {  // the last node this warp formed
#pragma unroll
    for (int off = S::CG; off < 32; off <<= 1)
#pragma unroll
      for (int c = 0; c < 4; ++c) po[c] += __shfl_xor_sync(FULL, po[c], off);
    if (rl == 0)
      st_f4(o_h + (int64_t)pn * p.Hv * dv, po[0] * piq, po[1] * piq, po[2] * piq, po[3] * piq);
  }

  // node depths (root = 1), written once per sequence
  if (lead && p.depth_out != nullptr)
    for (int n = tid; n < N; n += NT) p.depth_out[(int64_t)b * N + n] = sdep[n];
}

// ---------------------------------------------------------------- replay
// Checkpoint-and-replay commit: the recurrence again over the accepted path
// (chain: nodes 0 .. acc; tree: the ancestors of acc from the root), from the
// cached state, written back into the same cache slot.  Same slab
// decomposition as verify; along a path every node continues from the
// previous one, so u always comes from the look-ahead
//     u_{i+1} = alpha_i (H_{i-1}^T k_{i+1}) + delta_i (k_i . k_{i+1}),
// which also makes a chain replay repeat the verify kernel's arithmetic.
struct ReplayParams {
  const void* k;
  const void* v;
  const float* alpha;
  const float* beta;
  float* cache;
  const int32_t* slot;
  const int32_t* parent;
  const int32_t* accept;
  int32_t* status;
  int64_t cache_slot_stride;
  int n_slots, N, Hk, Hv, dv, bf16;
};

struct ReplayPlan {
  int path, par, k, v, a, b, inv, len, x, total;
};

__host__ __device__ inline ReplayPlan replay_plan(int N, int DK, int WC, int esz, int nw = 1) {
  ReplayPlan s{};
  s.path = 0;
  s.par = s.path + round16(N * 4);
  s.k = s.par + round16(N * 4);
  s.v = s.k + round16(N * DK * esz);
  s.a = s.v + round16(N * WC * esz);
  s.b = s.a + round16(N * 4);
  s.inv = s.b + round16(N * 4);  // 1/|k| of the path nodes (input preparation)
  s.len = s.inv + round16(N * 4);  // path length
  s.x = s.len + 16;               // cross-warp sums (NW > 1)
  s.total = s.x + xchg_bytes(nw, WC);
  return s;
}

template <int DK, int WC, int NW, bool PREP>
__global__ void __launch_bounds__(32 * NW) replay_kernel(const ReplayParams p) {
  pdl_enter();
  using S = Shape<DK, WC, NW>;
  constexpr int R = S::R;
  constexpr int NT = 32 * NW;
  extern __shared__ __align__(16) char smem[];
  const int N = p.N;
  const bool bf16 = p.bf16 != 0;
  const int esz = bf16 ? 2 : 4;
  const ReplayPlan pl = replay_plan(N, DK, WC, esz, NW);
  int* spath = reinterpret_cast<int*>(smem + pl.path);
  int* spar = reinterpret_cast<int*>(smem + pl.par);
  char* sk = smem + pl.k;
  char* sv = smem + pl.v;
  float* sa = reinterpret_cast<float*>(smem + pl.a);
  float* sb = reinterpret_cast<float*>(smem + pl.b);
  float* sinvk = reinterpret_cast<float*>(smem + pl.inv);
  int* slen = reinterpret_cast<int*>(smem + pl.len);
  float* sx = reinterpret_cast<float*>(smem + pl.x);
  int xc = 0;  // cross-warp exchanges so far

  const int tid = threadIdx.x, lane = tid & 31, wi = tid >> 5;
  const int cg = lane % S::CG, rl = lane / S::CG;
  const int j0 = blockIdx.x * WC, h = blockIdx.y, b = blockIdx.z;
  const int hk = h / (p.Hv / p.Hk);
  const bool lead = blockIdx.x == 0 && blockIdx.y == 0;
  const int dv = p.dv;
  const int row0 = wi * (DK / NW) + rl * R;
  const int64_t node0 = (int64_t)b * N;

  const int acc = __ldg(p.accept + b);
  const int sl = p.slot != nullptr ? __ldg(p.slot + b) : b;
  if (acc < 0 || acc >= N) {
    if (lead && tid == 0) report(p.status, GDN_ERR_ACCEPT_RANGE);
    return;
  }
  if (sl < 0 || sl >= p.n_slots) {
    if (lead && tid == 0) report(p.status, GDN_ERR_SLOT_RANGE);
    return;
  }

  // ---- the cached state -> registers, in flight while the path is found
  //      and its inputs are staged
  float* c0 = p.cache + (int64_t)sl * p.cache_slot_stride + (int64_t)h * DK * dv +
              (int64_t)row0 * dv + j0 + cg * 4;
  float2 H[R][2];
#pragma unroll
  for (int m = 0; m < R; ++m) {
    const float4 t = *reinterpret_cast<const float4*>(c0 + (int64_t)m * dv);
    H[m][0] = make_float2(t.x, t.y);
    H[m][1] = make_float2(t.z, t.w);
  }

  // ---- the accepted path, root first
  int L = acc + 1;
  if (p.parent == nullptr) {
    for (int n = tid; n < L; n += NT) spath[n] = n;
  } else {
    bool ok = true;
    for (int n = tid; n < N; n += NT) {
      const int pp = __ldg(p.parent + node0 + n);
      spar[n] = pp;
      ok = ok && (n == 0 ? pp == -1 : (pp >= 0 && pp < n));
    }
    if (!block_all<NW>(ok)) {
      if (lead && tid == 0) report(p.status, GDN_ERR_BAD_TREE);
      return;
    }
    block_sync<NW>();
    if (tid == 0) {
      int len = 0;
      for (int m = acc; m >= 0; m = spar[m]) ++len;
      int i = len;
      for (int m = acc; m >= 0; m = spar[m]) spath[--i] = m;
      *slen = len;
    }
    block_sync<NW>();
    L = *slen;
  }
  block_sync<NW>();

  // ---- stage k, v, gates of the path nodes
  {
    const char* kb = static_cast<const char*>(p.k) + ((node0 * p.Hk + hk) * DK) * esz;
    const char* vb = static_cast<const char*>(p.v) + ((node0 * p.Hv + h) * dv + j0) * esz;
    const int64_t kstride = (int64_t)p.Hk * DK * esz, vstride = (int64_t)p.Hv * dv * esz;
    const int kper = DK * esz / 16, vper = WC * esz / 16;
    for (int idx = tid; idx < L * kper; idx += NT) {
      const int r = idx / kper, c = idx - r * kper;
      cp_async16(sk + r * DK * esz + c * 16, kb + spath[r] * kstride + c * 16);
    }
    for (int idx = tid; idx < L * vper; idx += NT) {
      const int r = idx / vper, c = idx - r * vper;
      cp_async16(sv + r * WC * esz + c * 16, vb + spath[r] * vstride + c * 16);
    }
    for (int r = tid; r < L; r += NT) {
      cp_async4(sa + r, p.alpha + (node0 + spath[r]) * p.Hv + h);
      cp_async4(sb + r, p.beta + (node0 + spath[r]) * p.Hv + h);
    }
  }

  cp_async_wait_all();
  block_sync<NW>();
  if constexpr (PREP) {
    prep_rows<DK>(sk, L, bf16, sinvk, tid, NT);
    prep_gates(sa, sb, L, tid, NT);
    block_sync<NW>();
  }

  float kn[R];
  load_rows<R>(kn, sk, row0, bf16);
  float u[4];
  {
    float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
#pragma unroll
    for (int m = 0; m < R; ++m) {
      a01 = __ffma2_rn(H[m][0], f2(kn[m]), a01);
      a23 = __ffma2_rn(H[m][1], f2(kn[m]), a23);
    }
    u[0] = a01.x; u[1] = a01.y; u[2] = a23.x; u[3] = a23.y;
#pragma unroll
    for (int off = S::CG; off < 32; off <<= 1)
#pragma unroll
      for (int c = 0; c < 4; ++c) u[c] += __shfl_xor_sync(FULL, u[c], off);
    warps_sum<NW, S::CG>(u, sx, xc, wi, cg, rl);
    if constexpr (PREP) {
#pragma unroll
      for (int c = 0; c < 4; ++c) u[c] *= sinvk[0];
    }
  }
  for (int i = 0; i < L; ++i) {
    float knx[R];
    if (i + 1 < L) {
      load_rows<R>(knx, sk + (i + 1) * DK * esz, row0, bf16);
    } else {
#pragma unroll
      for (int m = 0; m < R; ++m) knx[m] = 0.f;
    }
    float vj[4];
    load_rows<4>(vj, sv + i * WC * esz, cg * 4, bf16);
    const float al = sa[i], be = sb[i];
    const float ik = PREP ? sinvk[i] : 1.f;
    const float ikx = PREP && i + 1 < L ? sinvk[i + 1] : 1.f;
    float2 w01 = make_float2(0.f, 0.f), w23 = make_float2(0.f, 0.f);
    float kk = 0.f;
#pragma unroll
    for (int m = 0; m < R; ++m) {
      w01 = __ffma2_rn(H[m][0], f2(knx[m]), w01);
      w23 = __ffma2_rn(H[m][1], f2(knx[m]), w23);
      kk = fmaf(kn[m], knx[m], kk);
    }
    float d[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) d[c] = be * (vj[c] - al * u[c]);
    const float2 d01 = make_float2(d[0] * ik, d[1] * ik), d23 = make_float2(d[2] * ik, d[3] * ik);
    const float2 al2 = f2(al);
#pragma unroll
    for (int m = 0; m < R; ++m) {
      H[m][0] = __ffma2_rn(f2(kn[m]), d01, __fmul2_rn(al2, H[m][0]));
      H[m][1] = __ffma2_rn(f2(kn[m]), d23, __fmul2_rn(al2, H[m][1]));
    }
    float red[5] = {w01.x, w01.y, w23.x, w23.y, kk};
#pragma unroll
    for (int off = S::CG; off < 32; off <<= 1)
#pragma unroll
      for (int e = 0; e < 5; ++e) red[e] += __shfl_xor_sync(FULL, red[e], off);
    warps_sum<NW, S::CG>(red, sx, xc, wi, cg, rl);
#pragma unroll
    for (int c = 0; c < 4; ++c) u[c] = fmaf(al, red[c] * ikx, d[c] * (red[4] * (ik * ikx)));
#pragma unroll
    for (int m = 0; m < R; ++m) kn[m] = knx[m];
  }

  // ---- back into the cache slot (each thread is the only reader and writer
  //      of its rows)
#pragma unroll
  for (int m = 0; m < R; ++m)
    st_f4(c0 + (int64_t)m * dv, H[m][0].x, H[m][0].y, H[m][1].x, H[m][1].y);
}

template <int DK, int WC, int NW>
int launch_replay_t(const ReplayParams& p, int B, bool prep, cudaStream_t stream) {
  const ReplayPlan pl = replay_plan(p.N, DK, WC, p.bf16 ? 2 : 4, NW);
  const dim3 grid(p.dv / WC, p.Hv, B);
  if (prep)
    return launch_pdl(replay_kernel<DK, WC, NW, true>, grid, dim3(32 * NW), pl.total, stream, p);
  return launch_pdl(replay_kernel<DK, WC, NW, false>, grid, dim3(32 * NW), pl.total, stream, p);
}

template <int DK, int WC, int NW, bool SNAP16, bool PREP>
int launch(const VerifyParams& p, int B, cudaStream_t stream) {
  const SmemPlan pl = smem_plan(p.N, DK, WC, p.bf16 ? 2 : 4, NW);
  const size_t smem = (size_t)pl.total;
  if (smem > 227 * 1024) return GDN_ERR_UNSUPPORTED;
  auto kern = verify_kernel<DK, WC, NW, SNAP16, PREP>;
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return GDN_ERR_CUDA;
  }
  const dim3 grid(p.dv / WC, p.Hv, B);
  return launch_pdl(kern, grid, dim3(32 * NW), smem, stream, p);
}

// Warps per tree block: each takes whole nodes of a depth level (measured on
// a 22-node draft tree: 4 warps 20.7 us, 8 warps 33.5 us per launch).
constexpr int kTreeWarps = 4;

template <int DK, int WC, int TW, bool PREP, bool SNAP16>
int launch_tree(const VerifyParams& p, int B, cudaStream_t stream) {
  const TreePlan pl = tree_plan(p.N, DK, WC, p.bf16 ? 2 : 4);
  const size_t smem = (size_t)pl.total;
  if (smem > 227 * 1024) return GDN_ERR_UNSUPPORTED;
  auto kern = tree_kernel<DK, WC, TW, PREP, SNAP16>;
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return GDN_ERR_CUDA;
  }
  const dim3 grid(p.dv / WC, p.Hv, B);
  return launch_pdl(kern, grid, dim3(32 * TW), smem, stream, p);
}

template <bool PREP, bool SNAP16>
int dispatch_tree(const VerifyParams& p, int B, int dk, int wc, cudaStream_t s) {
#define GDN_CASE(DK_, WC_) \
  if (dk == DK_ && wc == WC_) return launch_tree<DK_, WC_, kTreeWarps, PREP, SNAP16>(p, B, s);
  GDN_CASE(128, 16)
  GDN_CASE(128, 8)
  GDN_CASE(64, 16)
  GDN_CASE(64, 8)
  GDN_CASE(32, 16)
  GDN_CASE(32, 8)
  GDN_CASE(16, 16)
  GDN_CASE(16, 8)
#undef GDN_CASE
  return GDN_ERR_UNSUPPORTED;
}

template <bool SNAP16, bool PREP>
int dispatch(const VerifyParams& p, int B, int dk, int wc, int nw, cudaStream_t s) {
#define GDN_CASE(DK_, WC_, NW_) \
  if (dk == DK_ && wc == WC_ && nw == NW_) return launch<DK_, WC_, NW_, SNAP16, PREP>(p, B, s);
  GDN_CASE(128, 16, 1)
  GDN_CASE(128, 16, 2)
  GDN_CASE(128, 8, 1)
  GDN_CASE(64, 16, 1)
  GDN_CASE(64, 16, 2)
  GDN_CASE(64, 8, 1)
  GDN_CASE(32, 16, 1)
  GDN_CASE(32, 8, 1)
  GDN_CASE(16, 16, 1)
  GDN_CASE(16, 8, 1)
#undef GDN_CASE
  return GDN_ERR_UNSUPPORTED;
}

}  // namespace

bool verify_tile_supported(int dk, int wc, int nw) {
  if (!(dk == 128 || dk == 64 || dk == 32 || dk == 16) || !(wc == 16 || wc == 8)) return false;
  // two row warps: 16-column slabs of d_k = 64 or 128
  return nw == 1 || (nw == 2 && wc == 16 && (dk == 128 || dk == 64));
}

int launch_verify(const gdn_verify_args* a, const int32_t* parent, int32_t* depth_out, int wc,
                  int nw, cudaStream_t stream, void* snap16, bool prep) {
  VerifyParams p{};
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  p.alpha = a->alpha;
  p.beta = a->beta;
  p.cache = a->state_cache;
  p.slot = a->slot;
  p.snap = a->snapshots;
  p.o = a->o;
  p.status = a->status;
  p.parent = parent;
  p.depth_out = depth_out;
  p.cache_slot_stride = a->cache_slot_stride;
  p.n_slots = a->n_slots;
  p.N = a->N;
  p.Hk = a->Hk;
  p.Hv = a->Hv;
  p.dv = a->dv;
  p.bf16 = a->in_dtype == GDN_BF16;
  p.snap16 = static_cast<__half*>(snap16);
  p.hint = (int64_t)(p.dv / wc) * a->Hv * a->B <= kHintBlocks;
  p.max_depth = parent != nullptr ? a->max_depth : 0;
  // a tree that keeps no snapshots cannot re-read a parent's state from
  // them: it is solved per block instead (gdn_solve.cu)
  if (parent != nullptr && (a->snapshots == nullptr && snap16 == nullptr))
    return launch_verify_tree_solve(a, parent, depth_out, wc, stream, prep);
  if (parent != nullptr && snap16 != nullptr)
    return prep ? GDN_ERR_UNSUPPORTED : dispatch_tree<false, true>(p, a->B, a->dk, wc, stream);
  if (parent != nullptr)  // row warps do not apply: a tree block's warps take whole nodes
    return prep ? dispatch_tree<true, false>(p, a->B, a->dk, wc, stream)
                : dispatch_tree<false, false>(p, a->B, a->dk, wc, stream);
  if (snap16 != nullptr) {
    if (prep) return GDN_ERR_UNSUPPORTED;
    return dispatch<true, false>(p, a->B, a->dk, wc, nw, stream);
  }
  return prep ? dispatch<false, true>(p, a->B, a->dk, wc, nw, stream)
              : dispatch<false, false>(p, a->B, a->dk, wc, nw, stream);
}

int launch_replay(const gdn_verify_args* a, const int32_t* parent, const int32_t* accept, int wc,
                  int nw, cudaStream_t stream, bool prep) {
  ReplayParams p{};
  p.k = a->k;
  p.v = a->v;
  p.alpha = a->alpha;
  p.beta = a->beta;
  p.cache = const_cast<float*>(a->state_cache);
  p.slot = a->slot;
  p.parent = parent;
  p.accept = accept;
  p.status = a->status;
  p.cache_slot_stride = a->cache_slot_stride;
  p.n_slots = a->n_slots;
  p.N = a->N;
  p.Hk = a->Hk;
  p.Hv = a->Hv;
  p.dv = a->dv;
  p.bf16 = a->in_dtype == GDN_BF16;
#define GDN_CASE(DK_, WC_, NW_) \
  if (a->dk == DK_ && wc == WC_ && nw == NW_) \
    return launch_replay_t<DK_, WC_, NW_>(p, a->B, prep, stream);
  GDN_CASE(128, 16, 1)
  GDN_CASE(128, 16, 2)
  GDN_CASE(128, 8, 1)
  GDN_CASE(64, 16, 1)
  GDN_CASE(64, 16, 2)
  GDN_CASE(64, 8, 1)
  GDN_CASE(32, 16, 1)
  GDN_CASE(32, 8, 1)
  GDN_CASE(16, 16, 1)
  GDN_CASE(16, 8, 1)
#undef GDN_CASE
  return GDN_ERR_UNSUPPORTED;
}

}  // namespace gdn
