// Tree verification without persisted states, by one solve per block: the
// gated delta rule over a draft tree verified under its ancestor mask ("Qwen3.6
// 27B: From 20 t/s to 184 t/s", DFlash section, steps 3-4) for a block that
// keeps no snapshots and is committed by replay ("Photon 2.6", section
// "Handling recurrent state").  The level-by-level tree walk in gdn_verify.cu
// continues a node from its parent's snapshot when the parent is neither in a
// warp's registers nor in its shared-memory stash; without snapshots there is
// nothing to continue from, so this kernel forms every node's delta and output
// from the cached state directly and writes only the outputs.
//
// Recurrence
// ----------
// The state of one value head is H = S^T (d_k x d_v, fp32, row-major).  With
// src(n) the parent of node n (the cached state H0 for the root),
//     delta_n = beta_n (v_n - alpha_n H_src(n)^T k_n),
//     H_n = alpha_n H_src(n) + k_n delta_n^T,   o_n = H_n^T q_n,
// which is S_n = alpha_n S_src(n) (I - beta_n k_n k_n^T) + beta_n v_n k_n^T,
// o_n = S_n q_n with the product distributed.
//
// The block solved at once
// ------------------------
// Unrolling the recurrence along the path from H0 to node n, with r(n, m) the
// product of alpha over the path nodes after m up to n (r(n, n) = 1; g_n =
// r(n, -1), the product over the whole path),
//     H_n = g_n H0 + sum_{m in path(n)} r(n, m) k_m delta_m^T.
// Putting that into delta_n gives one lower-triangular system for all nodes
// of the block,
//     (I + A) Delta = X,   A[n][m] = beta_n r(n, m) (k_n . k_m)   (m a strict ancestor of n),
//                          X[n]    = beta_n (v_n - g_n H0^T k_n),
// and the outputs
//     o_n = g_n H0^T q_n + sum_{m in path(n)} r(n, m) (q_n . k_m) delta_m.
// With T = (I + A)^-1 and P[n][m] = r(n, m) (q_n . k_m) on the path,
//     Delta = T X,   O = diag(g) Q H0 + (P T) X,
// and T, P T depend on the block's inputs only, not on the cached state.  T
// inherits the ancestor mask (T[n][m] = 0 unless m is on n's path), and a row
// of T needs only the rows of the node's ancestors, so it is formed depth
// level by depth level.  The decay products come from the log decay along
// the path, r(n, m) = e^(L_n - L_m) with L_n the sum of log alpha over
// path(n).  A block is verified in two phases:
//   1. while the cached state's slab loads: K K^T and Q K^T on tensor cores
//      (mma.sync; exact for bf16 inputs), r, A and P under the ancestor mask,
//      T by depth levels and P T;
//   2. once it has landed: K H0 and Q H0 on tensor cores (the fp32 state
//      split into bf16 hi + lo) with X formed in the epilogue, then Delta and
//      the outputs in one pass, every entry on its own (a sum over the node's
//      path).
//
// Work decomposition
// ------------------
// A thread block of four warps owns a slab of WC columns of one (sequence,
// value head): grid = (dv / WC, Hv, B); both phases spread over all threads.
//
// Variants (template flags): PREP takes raw q/k projections and gate
// pre-activations (1/|q|, 1/|k| scale the products, alpha = 1/(1 + e^a),
// beta = sigmoid(b)); SPLIT takes fp32 q/k/v, whose tensor-core operands are
// split into bf16 hi + lo.
#include "gdn_common.cuh"
#include "gdn_launch.h"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int kWarps = 4;
constexpr int NT = 32 * kWarps;

__host__ __device__ constexpr int round16(int x) { return (x + 15) & ~15; }

// Shared-memory plan in bytes (every array on a 16-byte boundary).  NP = N
// rounded up to the 16 rows of a tensor-core tile.
//   ks, qs   [NP][lds]  bf16  k and q rows (with SPLIT a lo plane follows)
//   kf       [N][DK]    fp32  SPLIT only: the fp32 k rows as staged (the fp32
//                             q rows are staged over kk.., dead until K K^T)
//   h0       [DK][ldh]  fp32  the cached state's slab
//   v        [N][WC]    input the v slab
//   a, b, la [N]        fp32  alpha, beta, log alpha
//   g, L     [N]        fp32  g_n = e^(L_n), L_n = log decay along path(n)
//   iq, ik   [NP]       fp32  1/|q_n|, 1/|k_n| (PREP; zero past N)
//   par, dep [N]        int   parent, depth (root = 1)
//   ord      [N]        int   the nodes by depth, then index
//   lev      [N + 2]    int   lev[L] = first position of depth L in ord
//   anc      [N]        u64   strict ancestors as a bit set
//   kk       [NP][ldm]  fp32  K K^T -> A -> P T
//   qk       [NP][ldm]  fp32  Q K^T -> P
//   rr, tt   [NP][ldm]  fp32  r(n, m); T = (I + A)^-1
//   x, qh, d [NP][WC]   fp32  X, Q H0, Delta
struct Plan {
  int ks, qs, kf, h0, v, a, b, la, g, L, iq, ik, par, dep, ord, lev, anc, kk, qk, rr, tt, x, qh, d;
  int total, NP, lds, ldh, ldm;
};

__host__ __device__ inline Plan make_plan(int N, int DK, int WC, bool split) {
  Plan s{};
  s.NP = round16(N);
  s.lds = DK + 8;
  s.ldh = WC + 4;
  s.ldm = s.NP + 4;
  const int esz = split ? 4 : 2;
  const int planes = split ? 2 : 1;
  int o = 0;
  s.ks = o; o += round16(planes * s.NP * s.lds * 2);
  s.qs = o; o += round16(planes * s.NP * s.lds * 2);
  s.kf = o; o += split ? round16(N * DK * 4) : 0;
  s.h0 = o; o += round16(DK * s.ldh * 4);
  s.v = o; o += round16(N * WC * esz);
  s.a = o; o += round16(N * 4);
  s.b = o; o += round16(N * 4);
  s.la = o; o += round16(N * 4);
  s.g = o; o += round16(N * 4);
  s.L = o; o += round16(N * 4);
  s.iq = o; o += round16(s.NP * 4);
  s.ik = o; o += round16(s.NP * 4);
  s.par = o; o += round16(N * 4);
  s.dep = o; o += round16(N * 4);
  s.ord = o; o += round16(N * 4);
  s.lev = o; o += round16((N + 2) * 4);
  s.anc = o; o += round16(N * 8);
  const int mat = round16(s.NP * s.ldm * 4);
  s.kk = o; o += mat;
  s.qk = o; o += mat;
  s.rr = o; o += mat;
  s.tt = o; o += mat;
  const int slab = round16(s.NP * WC * 4);
  s.x = o; o += slab;
  s.qh = o; o += slab;
  s.d = o; o += slab;
  s.total = o;
  if (split && s.total < s.kk + N * DK * 4) s.total = s.kk + round16(N * DK * 4);
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
  float* o;
  int32_t* status;
  const int32_t* parent;
  int32_t* depth_out;
  int64_t cache_slot_stride;
  int n_slots, N, Hk, Hv, dv, bf16;
  int hint;       // issue the pre-wait L2 hints
  int max_depth;  // deepest node allowed (root = 1), 0 = no cap
};

// Launches of up to this many blocks (four per SM on 152 SMs) issue the
// pre-wait L2 hints.  A larger launch runs in several waves behind a stream
// of snapshot writes that evicts the hinted lines before they are used.
constexpr int kHintBlocks = 608;

__device__ __forceinline__ void prefetch_l2(const void* a) {
  asm volatile("prefetch.global.L2 [%0];\n" ::"l"(a));
}

// Before the programmatic wait (which orders this kernel after the previous
// one on the stream): hint L2 with the lines the block is about to read, so
// that their DRAM latency overlaps the previous kernel's tail.  The slot table
// and the inputs may still be being written by that kernel: a stale or
// out-of-range slot only wastes (or skips) the hint, a prefetch never changes
// memory, and every load that feeds a result is issued after the wait.
template <int DK>
__device__ __forceinline__ void prefetch_block(const VerifyParams& p, int b, int h, int hk, int j0,
                                               int WC, int t) {
  const int N = p.N, dv = p.dv, esz = p.bf16 ? 2 : 4;
  const int s0 = p.slot != nullptr ? __ldcg(p.slot + b) : b;
  const int seg = (WC * 4 + 127) / 128;  // 128-byte lines per state row of the slab
  if (s0 >= 0 && s0 < p.n_slots) {
    const char* c0 = reinterpret_cast<const char*>(p.cache + (int64_t)s0 * p.cache_slot_stride +
                                                   (int64_t)h * DK * dv + j0);
    for (int i = t; i < DK * seg; i += NT)
      prefetch_l2(c0 + (int64_t)(i / seg) * dv * 4 + (i % seg) * 128);
  }
  const int per = (DK * esz + 127) / 128;
  const int qk_lines = N * per;
  const int64_t node0 = (int64_t)b * N;
  for (int i = t; i < 2 * qk_lines + N; i += NT) {
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

// Start copying n_rows rows of row_bytes bytes each (row r at src +
// r*src_stride) to dst + r*dst_stride with 16-byte cp.async, thread t.
__device__ __forceinline__ void stage_rows(char* dst, int dst_stride, const char* src,
                                           int64_t src_stride, int n_rows, int row_bytes, int t) {
  const int per_row = row_bytes / 16;
  for (int idx = t; idx < n_rows * per_row; idx += NT) {
    const int r = idx / per_row, c = idx - r * per_row;
    cp_async16(dst + r * dst_stride + c * 16, src + r * src_stride + c * 16);
  }
}

__device__ __forceinline__ uint32_t lds32(const uint16_t* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}

// Next member of a bit set (lowest first), removed from it.
__device__ __forceinline__ int pop_low(uint64_t& set) {
  const int m = __ffsll(static_cast<long long>(set)) - 1;
  set &= set - 1;
  return m;
}

// ---------------------------------------------------------- phases 1 and 2
// Tile fragments for mma.sync m16n8k16 (bf16 operands, fp32 accumulate):
//   frag_a:  rows r0..r0+15, columns k0..k0+15 of a bf16 matrix [row][ld]
//   frag_bt: B[k][n] = M[n][k] for n0..n0+7 (a bf16 matrix stored [n][ld])
//   frag_bs: B[k][n] = M[k][n] of an fp32 matrix [k][ld], split into hi + lo
__device__ __forceinline__ void frag_a(const uint16_t* A, int ld, int r0, int k0, int g8, int t4,
                                       uint32_t (&a)[4]) {
  const uint16_t* p = A + (r0 + g8) * ld + k0 + 2 * t4;
  a[0] = lds32(p);
  a[1] = lds32(p + 8 * ld);
  a[2] = lds32(p + 8);
  a[3] = lds32(p + 8 * ld + 8);
}

__device__ __forceinline__ void frag_bt(const uint16_t* M, int ld, int n0, int k0, int g8, int t4,
                                        uint32_t& b0, uint32_t& b1) {
  const uint16_t* p = M + (n0 + g8) * ld + k0 + 2 * t4;
  b0 = lds32(p);
  b1 = lds32(p + 8);
}

__device__ __forceinline__ void frag_bs(const float* M, int ld, int k0, int n0, int g8, int t4,
                                        uint32_t (&hi)[2], uint32_t (&lo)[2]) {
  const float* p = M + (k0 + 2 * t4) * ld + n0 + g8;
  tc::split_bf16x2(p[0], p[ld], hi[0], lo[0]);
  tc::split_bf16x2(p[8 * ld], p[9 * ld], hi[1], lo[1]);
}

// One 16 x 8 tile of A B over DK into acc: rows r0 + g8 (acc[0], acc[1]) and
// r0 + g8 + 8 (acc[2], acc[3]), columns n0 + 2 t4, +1.
//   BT: B[k][n] = Bm[n][k] (bf16, exact); otherwise B is the fp32 state slab
//   [k][ldb] split into hi + lo.  SPLIT: A (and a bf16 B) carry a lo plane
//   `plane` elements after the hi plane.
template <int DK, bool BT, bool SPLIT>
__device__ __forceinline__ void tile_mma(const uint16_t* A, int lda, int plane, const void* Bm,
                                         int ldb, int r0, int n0, int g8, int t4,
                                         float (&acc)[4]) {
  // two accumulators (even and odd k-steps) halve the chain of dependent MMAs
  float accs[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
  for (int k0 = 0; k0 < DK; k0 += 16) {
    float (&c)[4] = accs[(k0 >> 4) & 1];
    uint32_t ah[4];
    frag_a(A, lda, r0, k0, g8, t4, ah);
    if constexpr (BT) {
      const uint16_t* B = static_cast<const uint16_t*>(Bm);
      uint32_t b0, b1;
      frag_bt(B, ldb, n0, k0, g8, t4, b0, b1);
      mma_bf16_16816(c, ah, b0, b1);
      if constexpr (SPLIT) {
        uint32_t al[4], c0, c1;
        frag_a(A + plane, lda, r0, k0, g8, t4, al);
        frag_bt(B + plane, ldb, n0, k0, g8, t4, c0, c1);
        mma_bf16_16816(c, ah, c0, c1);
        mma_bf16_16816(c, al, b0, b1);
      }
    } else {
      uint32_t bh[2], bl[2];
      frag_bs(static_cast<const float*>(Bm), ldb, k0, n0, g8, t4, bh, bl);
      mma_bf16_16816(c, ah, bh[0], bh[1]);
      mma_bf16_16816(c, ah, bl[0], bl[1]);
      if constexpr (SPLIT) {
        uint32_t al[4];
        frag_a(A + plane, lda, r0, k0, g8, t4, al);
        mma_bf16_16816(c, al, bh[0], bh[1]);
      }
    }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) acc[e] = accs[0][e] + accs[1][e];
}

// Phase 1 for N nodes whose k and q rows, gates and parents are staged: the
// working forms of the inputs, the tree's depths, ancestor sets and log decay,
// K K^T and Q K^T, r, A and P, then T = (I + A)^-1 by depth levels and P T.
// Returns 0, or 1 if the parent array is malformed, 2 if the tree is deeper
// than max_depth (depths filled in); every thread returns the same value.
template <int DK, bool SPLIT, bool PREP>
__device__ int solve_prepare(const Plan& pl, char* smem, int N, int max_depth) {
  const int tid = threadIdx.x, lane = tid & 31, wi = tid >> 5;
  const int g8 = lane >> 2, t4 = lane & 3;
  uint16_t* ks = reinterpret_cast<uint16_t*>(smem + pl.ks);
  uint16_t* qs = reinterpret_cast<uint16_t*>(smem + pl.qs);
  // fp32 inputs (SPLIT): k staged in kf, q over the matrices
  const float* rawk = reinterpret_cast<const float*>(smem + pl.kf);
  const float* rawq = reinterpret_cast<const float*>(smem + pl.kk);
  float* sa = reinterpret_cast<float*>(smem + pl.a);
  float* sb = reinterpret_cast<float*>(smem + pl.b);
  float* sla = reinterpret_cast<float*>(smem + pl.la);
  float* sg = reinterpret_cast<float*>(smem + pl.g);
  float* sL = reinterpret_cast<float*>(smem + pl.L);
  float* siq = reinterpret_cast<float*>(smem + pl.iq);
  float* sik = reinterpret_cast<float*>(smem + pl.ik);
  const int* spar = reinterpret_cast<const int*>(smem + pl.par);
  int* sdep = reinterpret_cast<int*>(smem + pl.dep);
  uint64_t* sanc = reinterpret_cast<uint64_t*>(smem + pl.anc);
  int* sord = reinterpret_cast<int*>(smem + pl.ord);
  int* slev = reinterpret_cast<int*>(smem + pl.lev);
  float* kk = reinterpret_cast<float*>(smem + pl.kk);
  float* qk = reinterpret_cast<float*>(smem + pl.qk);
  float* rr = reinterpret_cast<float*>(smem + pl.rr);
  float* tt = reinterpret_cast<float*>(smem + pl.tt);
  const int NP = pl.NP, lds = pl.lds, ldm = pl.ldm;
  const int plane = NP * lds;

  // ---- fp32 rows split into bf16 planes (SPLIT), norms and gate maps (PREP)
  if constexpr (SPLIT) {
    const int half = N * DK / 2;
    for (int i = tid; i < 2 * half; i += NT) {
      const int which = i / half, e = 2 * (i - which * half);
      const int n = e / DK, c = e - n * DK;
      const float2 x = *reinterpret_cast<const float2*>((which ? rawq : rawk) + e);
      uint32_t hi, lo;
      tc::split_bf16x2(x.x, x.y, hi, lo);
      uint16_t* dst = (which ? qs : ks) + n * lds + c;
      *reinterpret_cast<uint32_t*>(dst) = hi;
      *reinterpret_cast<uint32_t*>(dst + plane) = lo;
    }
  }
  if constexpr (PREP) {
    for (int r = tid; r < 2 * NP; r += NT) {
      const int which = r / NP, n = r - which * NP;
      float ss = 0.f;
      if (n < N) {
        if constexpr (SPLIT) {
          const float* x = (which ? rawq : rawk) + n * DK;
          for (int c = 0; c < DK; ++c) ss = fmaf(x[c], x[c], ss);
        } else {
          const uint16_t* x = (which ? qs : ks) + n * lds;
          for (int c = 0; c < DK; c += 2) {
            const uint32_t w = lds32(x + c);
            const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xffff0000u);
            ss = fmaf(lo, lo, fmaf(hi, hi, ss));
          }
        }
      }
      (which ? siq : sik)[n] = ss > 0.f ? rsqrtf(ss) : 0.f;
    }
    for (int n = tid; n < N; n += NT) {
      sa[n] = 1.f / (1.f + __expf(sa[n]));
      sb[n] = 1.f / (1.f + __expf(-sb[n]));
    }
  }
  __syncthreads();
  // log alpha (clamped below at 1e-30, where its log is finite); a malformed
  // parent array stops the block
  bool ok = true;
  for (int n = tid; n < N; n += NT) {
    sla[n] = logf(fmaxf(sa[n], 1e-30f));
    const int pp = spar[n];
    ok = ok && (n == 0 ? pp == -1 : (pp >= 0 && pp < n));
  }
  if (__syncthreads_and(ok) == 0) return 1;

  // ---- depths, strict ancestors, L_n and g_n (one node per thread, walking
  //      up to the root); K K^T and Q K^T, the tiles on and below the
  //      diagonal (PREP: scaled by 1/|q_n| or 1/|k_n| and 1/|k_m|)
  bool shallow = true;
  for (int n = tid; n < N; n += NT) {
    int d = 1;
    uint64_t anc = 0;
    float l = sla[n];
    for (int m = spar[n]; m >= 0; m = spar[m]) {
      ++d;
      anc |= 1ull << m;
      l += sla[m];
    }
    sdep[n] = d;
    sanc[n] = anc;
    sL[n] = l;
    sg[n] = expf(l);
    shallow = shallow && (max_depth <= 0 || d <= max_depth);
  }
  {
    const int mt_n = NP / 16, nt_n = NP / 8, n_tiles = mt_n * nt_n;
    for (int task = wi; task < 2 * n_tiles; task += kWarps) {
      const int which = task / n_tiles, tl = task - which * n_tiles;
      const int mt = tl / nt_n, nt = tl - mt * nt_n;
      if (nt * 8 > mt * 16 + 15) continue;
      float acc[4];
      tile_mma<DK, true, SPLIT>(which ? qs : ks, lds, plane, ks, lds, mt * 16, nt * 8, g8, t4,
                                acc);
      const int r = mt * 16 + g8, c = nt * 8 + 2 * t4;
      float s0 = 1.f, s1 = 1.f, c0 = 1.f, c1 = 1.f;
      if constexpr (PREP) {
        const float* rs = which ? siq : sik;
        s0 = rs[r];
        s1 = rs[r + 8];
        c0 = sik[c];
        c1 = sik[c + 1];
      }
      float* C = which ? qk : kk;
      *reinterpret_cast<float2*>(C + r * ldm + c) = make_float2(acc[0] * s0 * c0, acc[1] * s0 * c1);
      *reinterpret_cast<float2*>(C + (r + 8) * ldm + c) =
          make_float2(acc[2] * s1 * c0, acc[3] * s1 * c1);
    }
  }
  if (__syncthreads_and(shallow) == 0) return 2;

  // ---- r(n, m) = e^(L_n - L_m) on n's path (1 at m = n), A = beta r (K K^T)
  //      for the strict ancestors, P = r (Q K^T) on the path (entries off the
  //      path are never read): one warp per node, lanes over m (N <= 64).
  //      Meanwhile the walk order (by depth, then index) and the level starts.
  for (int n = wi; n < N; n += kWarps) {
    const uint64_t path = sanc[n] | (1ull << n);
    const float Ln = sL[n], bn = sb[n];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int m = lane + 32 * h;
      if (m >= N || ((path >> m) & 1ull) == 0) continue;
      const float r = m == n ? 1.f : expf(Ln - sL[m]);
      rr[n * ldm + m] = r;
      if (m < n) kk[n * ldm + m] = bn * r * kk[n * ldm + m];
      qk[n * ldm + m] = r * qk[n * ldm + m];
    }
  }
  for (int n = tid; n < N; n += NT) {
    const int dn = sdep[n];
    int pos = 0;
    for (int m = 0; m < N; ++m) {
      const int dm = sdep[m];
      pos += (dm < dn || (dm == dn && m < n)) ? 1 : 0;
    }
    sord[pos] = n;
  }
  for (int L = tid; L < N + 2; L += NT) {
    int c = 0;
    for (int m = 0; m < N; ++m) c += sdep[m] < L ? 1 : 0;
    slev[L] = c;
  }
  __syncthreads();

  // ---- T = (I + A)^-1, depth level by depth level, one warp per node of the
  //      level and lanes over m:
  //      T[n][m] = [n = m] - sum over the strict ancestors s >= m of n of
  //      A[n][s] T[s][m], zero unless m is on n's path (then m is on the path
  //      of every such s, whose row an earlier level formed)
  for (int L = 1; L <= N && slev[L] < N; ++L) {
    for (int i = slev[L] + wi; i < slev[L + 1]; i += kWarps) {
      const int n = sord[i];
      const uint64_t anc = sanc[n];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int m = lane + 32 * h;
        if (m > n || (m < n && ((anc >> m) & 1ull) == 0)) continue;
        float t = m == n ? 1.f : 0.f;
        uint64_t s_set = anc & ~((1ull << m) - 1ull);  // strict ancestors s >= m
        while (s_set != 0) {
          const int s2 = pop_low(s_set);
          t = fmaf(-kk[n * ldm + s2], tt[s2 * ldm + m], t);
        }
        tt[n * ldm + m] = t;
      }
    }
    __syncthreads();
  }

  // ---- P T over A (A is dead), one warp per node, lanes over m:
  //      (P T)[n][m] = sum over the path nodes s >= m of P[n][s] T[s][m]
  for (int n = wi; n < N; n += kWarps) {
    const uint64_t path = sanc[n] | (1ull << n);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int m = lane + 32 * h;
      if (m >= N || ((path >> m) & 1ull) == 0) continue;
      float acc = 0.f;
      uint64_t s_set = path & ~((1ull << m) - 1ull);
      while (s_set != 0) {
        const int s2 = pop_low(s_set);
        acc = fmaf(qk[n * ldm + s2], tt[s2 * ldm + m], acc);
      }
      kk[n * ldm + m] = acc;
    }
  }
  return 0;
}

// Phase 2, once the state slab is in h0 (and phase 1's results are visible):
// K H0 and Q H0 on tensor cores, X = diag(beta)(V - diag(g) K H0) formed in
// the epilogue, then every entry of Delta = T X and of the outputs
// O = diag(g) Q H0 + (P T) X on its own, a sum over the node's path; row n of
// O to o_out + n*o_stride (WC columns).
template <int DK, int WC, bool SPLIT, bool PREP>
__device__ void solve_finish(const Plan& pl, char* smem, int N, float* o_out, int64_t o_stride) {
  const int tid = threadIdx.x, lane = tid & 31, wi = tid >> 5;
  const int g8 = lane >> 2, t4 = lane & 3;
  const uint16_t* ks = reinterpret_cast<const uint16_t*>(smem + pl.ks);
  const uint16_t* qs = reinterpret_cast<const uint16_t*>(smem + pl.qs);
  const float* h0 = reinterpret_cast<const float*>(smem + pl.h0);
  const float* sb = reinterpret_cast<const float*>(smem + pl.b);
  const float* sg = reinterpret_cast<const float*>(smem + pl.g);
  const float* siq = reinterpret_cast<const float*>(smem + pl.iq);
  const float* sik = reinterpret_cast<const float*>(smem + pl.ik);
  const uint64_t* sanc = reinterpret_cast<const uint64_t*>(smem + pl.anc);
  const float* pt = reinterpret_cast<const float*>(smem + pl.kk);
  const float* tt = reinterpret_cast<const float*>(smem + pl.tt);
  float* sx = reinterpret_cast<float*>(smem + pl.x);
  float* sqh = reinterpret_cast<float*>(smem + pl.qh);
  float* sd = reinterpret_cast<float*>(smem + pl.d);
  const int NP = pl.NP, lds = pl.lds, ldm = pl.ldm, ldh = pl.ldh;
  const int plane = NP * lds;

  {
    const int mt_n = NP / 16, nt_n = WC / 8, n_tiles = mt_n * nt_n;
    for (int task = wi; task < 2 * n_tiles; task += kWarps) {
      const int which = task / n_tiles, tl = task - which * n_tiles;
      const int mt = tl / nt_n, nt = tl - mt * nt_n;
      float acc[4];
      tile_mma<DK, false, SPLIT>(which ? qs : ks, lds, plane, h0, ldh, mt * 16, nt * 8, g8, t4,
                                 acc);
      const int c = nt * 8 + 2 * t4;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = mt * 16 + g8 + 8 * hh;
        if (r >= N) continue;
        float e0 = acc[2 * hh], e1 = acc[2 * hh + 1];
        if constexpr (PREP) {
          const float sc = which ? siq[r] : sik[r];
          e0 *= sc;
          e1 *= sc;
        }
        if (which) {
          *reinterpret_cast<float2*>(sqh + r * WC + c) = make_float2(e0, e1);
        } else {
          // X = beta (v - g K H0); the v slab is staged in the input dtype
          float v0, v1;
          if constexpr (SPLIT) {
            const float2 vv = *reinterpret_cast<const float2*>(
                reinterpret_cast<const float*>(smem + pl.v) + r * WC + c);
            v0 = vv.x;
            v1 = vv.y;
          } else {
            const uint32_t w =
                lds32(reinterpret_cast<const uint16_t*>(smem + pl.v) + r * WC + c);
            v0 = __uint_as_float(w << 16);
            v1 = __uint_as_float(w & 0xffff0000u);
          }
          const float be = sb[r], gr = sg[r];
          *reinterpret_cast<float2*>(sx + r * WC + c) =
              make_float2(be * (v0 - gr * e0), be * (v1 - gr * e1));
        }
      }
    }
  }
  __syncthreads();
  for (int idx = tid; idx < 2 * N * WC; idx += NT) {
    const int which = idx >= N * WC;
    const int e = idx - (which ? N * WC : 0);
    const int n = e / WC, c = e - n * WC;
    const float* M = which ? pt : tt;
    float a0 = which ? sg[n] * sqh[e] : 0.f, a1 = 0.f;
    uint64_t path = sanc[n] | (1ull << n);
    while (path != 0) {
      const int m = pop_low(path);
      a0 = fmaf(M[n * ldm + m], sx[m * WC + c], a0);
      if (path == 0) break;
      const int m2 = pop_low(path);
      a1 = fmaf(M[n * ldm + m2], sx[m2 * WC + c], a1);
    }
    if (which) o_out[n * o_stride + c] = a0 + a1;
    else sd[e] = a0 + a1;
  }
}

// Zero the padding rows N .. NP-1 of the bf16 k and q tiles.
__device__ __forceinline__ void zero_padding(const Plan& pl, char* smem, int N, bool split, int t) {
  uint16_t* ks = reinterpret_cast<uint16_t*>(smem + pl.ks);
  uint16_t* qs = reinterpret_cast<uint16_t*>(smem + pl.qs);
  const int per_plane = (pl.NP - N) * pl.lds;
  const int planes = split ? 2 : 1;
  for (int i = t; i < planes * per_plane; i += NT) {
    const int pi = i / per_plane, e = i - pi * per_plane;
    ks[pi * pl.NP * pl.lds + N * pl.lds + e] = 0;
    qs[pi * pl.NP * pl.lds + N * pl.lds + e] = 0;
  }
}

// ---------------------------------------------------------------- verify
template <int DK, int WC, bool PREP, bool SPLIT>
__global__ void __launch_bounds__(NT) tree_solve_kernel(const VerifyParams p) {
  const int tid = threadIdx.x;
  const int j0 = blockIdx.x * WC, h = blockIdx.y, b = blockIdx.z;
  const int hk = h / (p.Hv / p.Hk);
  if (p.hint) prefetch_block<DK>(p, b, h, hk, j0, WC, tid);
  pdl_enter();
  extern __shared__ __align__(16) char smem[];
  const int N = p.N, dv = p.dv;
  const Plan pl = make_plan(N, DK, WC, SPLIT);
  const bool lead = blockIdx.x == 0 && blockIdx.y == 0;  // per-sequence reporting
  const int64_t node0 = (int64_t)b * N;
  constexpr int esz = SPLIT ? 4 : 2;
  int* spar = reinterpret_cast<int*>(smem + pl.par);
  const int* sdep = reinterpret_cast<const int*>(smem + pl.dep);

  // ---- stage k, q, v, gates and parents (cp.async group 0), then the
  //      cached state's slab (group 1, waited for only in phase 2)
  {
    const char* kb = static_cast<const char*>(p.k) + ((node0 * p.Hk + hk) * DK) * esz;
    const char* qb = static_cast<const char*>(p.q) + ((node0 * p.Hk + hk) * DK) * esz;
    const char* vb = static_cast<const char*>(p.v) + ((node0 * p.Hv + h) * dv + j0) * esz;
    const int64_t qk_stride = (int64_t)p.Hk * DK * esz;
    if constexpr (SPLIT) {
      stage_rows(smem + pl.kf, DK * 4, kb, qk_stride, N, DK * 4, tid);
      stage_rows(smem + pl.kk, DK * 4, qb, qk_stride, N, DK * 4, tid);
    } else {
      stage_rows(smem + pl.ks, pl.lds * 2, kb, qk_stride, N, DK * 2, tid);
      stage_rows(smem + pl.qs, pl.lds * 2, qb, qk_stride, N, DK * 2, tid);
    }
    stage_rows(smem + pl.v, WC * esz, vb, (int64_t)p.Hv * dv * esz, N, WC * esz, tid);
    for (int n = tid; n < N; n += NT) {
      cp_async4(reinterpret_cast<float*>(smem + pl.a) + n, p.alpha + (node0 + n) * p.Hv + h);
      cp_async4(reinterpret_cast<float*>(smem + pl.b) + n, p.beta + (node0 + n) * p.Hv + h);
      cp_async4(spar + n, p.parent + node0 + n);
    }
    zero_padding(pl, smem, N, SPLIT, tid);
    cp_async_commit();
  }
  const int sl = p.slot != nullptr ? __ldg(p.slot + b) : b;
  const bool slot_ok = sl >= 0 && sl < p.n_slots;
  if (slot_ok) {
    const char* c0 = reinterpret_cast<const char*>(p.cache + (int64_t)sl * p.cache_slot_stride +
                                                   (int64_t)h * DK * dv + j0);
    stage_rows(smem + pl.h0, pl.ldh * 4, c0, (int64_t)dv * 4, DK, WC * 4, tid);
  }
  cp_async_commit();
  if (!slot_ok) {
    cp_async_wait<0>();
    if (lead && tid == 0) report(p.status, GDN_ERR_SLOT_RANGE);
    return;
  }
  cp_async_wait<1>();
  __syncthreads();

  const int bad = solve_prepare<DK, SPLIT, PREP>(pl, smem, N, p.max_depth);
  if (bad != 0) {  // a malformed tree, or one deeper than the cap (depths reported)
    cp_async_wait<0>();
    if (lead && tid == 0) report(p.status, GDN_ERR_BAD_TREE);
    if (bad == 2 && lead && p.depth_out != nullptr)
      for (int n = tid; n < N; n += NT) p.depth_out[node0 + n] = sdep[n];
    return;
  }
  cp_async_wait<0>();
  __syncthreads();
  solve_finish<DK, WC, SPLIT, PREP>(pl, smem, N, p.o + (node0 * p.Hv + h) * dv + j0,
                                    (int64_t)p.Hv * dv);
  if (lead && p.depth_out != nullptr)
    for (int n = tid; n < N; n += NT) p.depth_out[node0 + n] = sdep[n];
}

template <int DK, int WC, bool PREP>
int launch_solve_t(const VerifyParams& p, int B, cudaStream_t stream) {
  const dim3 grid(p.dv / WC, p.Hv, B);
  const bool split = !p.bf16;
  const size_t smem = (size_t)make_plan(p.N, DK, WC, split).total;
  if (smem > 227 * 1024) return GDN_ERR_UNSUPPORTED;
  auto kern = split ? tree_solve_kernel<DK, WC, PREP, true>
                    : tree_solve_kernel<DK, WC, PREP, false>;
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return GDN_ERR_CUDA;
  }
  return launch_pdl(kern, grid, dim3(NT), smem, stream, p);
}

template <bool PREP>
int dispatch_solve(const VerifyParams& p, int B, int dk, int wc, cudaStream_t s) {
#define GDN_CASE(DK_, WC_) \
  if (dk == DK_ && wc == WC_) return launch_solve_t<DK_, WC_, PREP>(p, B, s);
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

}  // namespace

int launch_verify_tree_solve(const gdn_verify_args* a, const int32_t* parent, int32_t* depth_out,
                             int wc, cudaStream_t stream, bool prep) {
  VerifyParams p{};
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  p.alpha = a->alpha;
  p.beta = a->beta;
  p.cache = a->state_cache;
  p.slot = a->slot;
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
  p.hint = (int64_t)(p.dv / wc) * a->Hv * a->B <= kHintBlocks;
  p.max_depth = a->max_depth;
  return prep ? dispatch_solve<true>(p, a->B, a->dk, wc, stream)
              : dispatch_solve<false>(p, a->B, a->dk, wc, stream);
}

}  // namespace gdn
