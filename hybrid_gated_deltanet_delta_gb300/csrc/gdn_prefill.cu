// Chunked prefill: the gated delta rule over T tokens, evaluated 64 tokens at
// a time in the WY / UT-transform form on tensor cores.
//
// Chunk form (one value head; rows t, s index the chunk; H = S^T is d_k x d_v)
// ----------------------------------------------------------------------------
// With g_t = prod_{s<=t} alpha_s inside the chunk and
// delta_t = beta_t (v_t - alpha_t H_{t-1}^T k_t), the deltas of a chunk solve
//     (I + A) Delta = X,   A[t][s] = beta_t (g_t/g_s) (k_t . k_s)  (s < t),
//                          X = diag(beta) (V - diag(g) K H),
// and then
//     O = diag(g) Q H + P Delta,   P[t][s] = (g_t/g_s) (q_t . k_s)  (s <= t),
//     H <- g_C H + K^T D',         D' = diag(g_C/g) Delta.
// (The unrolled step recurrence; the same algebra is checked against the step
// oracle in the test suite.)  The prefill splits the work in two launches:
//
//   prep  (grid: chunk x q/k head, fully parallel): K K^T and Q K^T on tensor
//         cores, the log-space cumulative decay, A, T = (I + A)^-1 by forward
//         substitution, P; T and P are written to the caller's workspace as
//         bf16 hi/lo pairs, with g and beta.
//   scan  (grid: value head x 3 column slabs of the state, sequential over
//         chunks): per chunk K H and Q H, X, Delta = T X, O = g Q H + P Delta,
//         H <- g_C H + K^T D'.  The state stays in fp32 mma accumulator
//         fragments for the whole sequence; the next chunk's inputs are staged
//         with cp.async while the current one is processed.
//
// Precision: every tensor-core operand that is not exactly a bf16 input (the
// state, X, Delta, D', T, P) is carried as a bf16 pair hi + lo and multiplied
// as hi*hi + hi*lo + lo*hi (or hi + lo against an exact bf16 K / Q), which
// keeps ~16 significant bits per operand; a single bf16 rounding of any of
// them costs ~1% of the output RMS at this size.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "gdn_common.cuh"
#include "gdn_launch.h"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int C = 64;         // chunk length
constexpr int DK = 128;       // key / query width
constexpr int DV = 128;       // value width
constexpr int KS = DK * 2 + 16;  // staged bf16 row of K / Q, padded (bytes)

// workspace block of one (chunk, value head): A = [T; P T] (128 x 64) as bf16
// hi then lo, in 128-byte rows whose 16-byte chunks are XOR-swizzled by row
// (chunk ch of row r at chunk ch ^ (r & 7): the tensor cores' 128-byte
// swizzle), then the log decay G_t = sum_{s<=t} log alpha_s (g_t = exp G_t) and
// beta.  The scan copies the block into shared memory as is and hands A to the
// tensor cores without further staging.
constexpr int WS_AH = 0;      // rows 0-63: T, rows 64-127: P T
constexpr int WS_AL = 16384;
constexpr int WS_G = 32768;
constexpr int WS_B = 33024;
constexpr int WS_STRIDE = 33280;

__device__ __forceinline__ uint32_t ld32(const char* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}

// ------------------------------------------------------------------- prep
constexpr int PREP_THREADS = 256;
constexpr int TS = 65;  // fp32 row stride of the 64 x 64 work matrices (bank spread)
constexpr int PREP_K = 0;
constexpr int PREP_Q = PREP_K + C * KS;
constexpr int PREP_KK = PREP_Q + C * KS;
constexpr int PREP_QK = PREP_KK + C * C * 4;
constexpr int PREP_A = PREP_QK + C * C * 4;
// T and the product scratch reuse the K / Q staging area, dead once K K^T and
// Q K^T are formed
constexpr int PREP_T = PREP_K;
constexpr int PREP_S = PREP_T + C * TS * 4;
static_assert(PREP_S + C * TS * 4 <= PREP_KK, "T and S must fit in the K/Q staging area");
constexpr int PREP_GATE = PREP_A + C * TS * 4;  // [2 buffers][alpha 64, beta 64]
constexpr int PREP_LG = PREP_GATE + 2 * 2 * C * 4;
constexpr int PREP_G = PREP_LG + C * 4;
constexpr int PREP_B = PREP_G + C * 4;
constexpr int PREP_SMEM = PREP_B + C * 4;

// C = sign * X Y for M x N outputs over K terms (all three row stride TS);
// `nthreads` threads starting at `tid` = 0 share the 2 x 2 output tiles.
__device__ __forceinline__ void mm_tiles(float* Cm, const float* X, const float* Y, int M, int N,
                                         int K, float sign, int tid, int nthreads) {
  const int tn = N / 2;
  for (int tile = tid; tile < (M / 2) * tn; tile += nthreads) {
    const int r = 2 * (tile / tn), c = 2 * (tile % tn);
    float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;
    for (int k = 0; k < K; ++k) {
      const float x0 = X[r * TS + k], x1 = X[(r + 1) * TS + k];
      const float y0 = Y[k * TS + c], y1 = Y[k * TS + c + 1];
      a00 = fmaf(x0, y0, a00); a01 = fmaf(x0, y1, a01);
      a10 = fmaf(x1, y0, a10); a11 = fmaf(x1, y1, a11);
    }
    Cm[r * TS + c] = sign * a00;
    Cm[r * TS + c + 1] = sign * a01;
    Cm[(r + 1) * TS + c] = sign * a10;
    Cm[(r + 1) * TS + c + 1] = sign * a11;
  }
}

// R = X Y for lower-triangular 64 x 64 X and Y (row stride TS): only the
// terms k in [s, t] of R[t][s] are nonzero.  All PREP_THREADS threads share
// the 2 x 2 output tiles; tiles above the diagonal are written as zero.
__device__ __forceinline__ void mm_lower(float* R, const float* X, const float* Y, int tid) {
  for (int tile = tid; tile < (C / 2) * (C / 2); tile += PREP_THREADS) {
    const int r = 2 * (tile >> 5), c = 2 * (tile & 31);
    float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;
    for (int k = c; k <= r + 1; ++k) {
      const float x0 = X[r * TS + k], x1 = X[(r + 1) * TS + k];
      const float y0 = Y[k * TS + c], y1 = Y[k * TS + c + 1];
      a00 = fmaf(x0, y0, a00); a01 = fmaf(x0, y1, a01);
      a10 = fmaf(x1, y0, a10); a11 = fmaf(x1, y1, a11);
    }
    R[r * TS + c] = a00;
    R[r * TS + c + 1] = a01;
    R[(r + 1) * TS + c] = a10;
    R[(r + 1) * TS + c + 1] = a11;
  }
}

// T = (I + A)^-1 for a strictly lower-triangular 64 x 64 A (row stride TS) by
// recursive doubling of the block inverse
//     [[L11, 0], [L21, L22]]^-1 = [[L11^-1, 0], [-L22^-1 L21 L11^-1, L22^-1]]:
// the four 16 x 16 diagonal blocks by forward substitution held in registers
// (one column per lane), then the 16 -> 32 and 32 -> 64 merges as two products
// each.  S is 64 x 64 scratch.
__device__ void invert_unit_lower(const float* A, float* T, float* S, int tid) {
  const int w = tid >> 5, lane = tid & 31;
  if (w < 2) {
    const int b0 = 16 * (2 * w + (lane >> 4)), j = lane & 15;
    float tc[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      float acc = 0.f;
#pragma unroll
      for (int r = 0; r < t; ++r) acc = fmaf(A[(b0 + t) * TS + b0 + r], tc[r], acc);
      tc[t] = t < j ? 0.f : (t == j ? 1.f : -acc);
    }
#pragma unroll
    for (int t = 0; t < 16; ++t) T[(b0 + t) * TS + b0 + j] = tc[t];
  }
  // blocks above the diagonal are zero
  for (int idx = tid; idx < C * C; idx += PREP_THREADS) {
    const int t = idx >> 6, s = idx & 63;
    if ((s >> 4) > (t >> 4)) T[t * TS + s] = 0.f;
  }
  __syncthreads();
  // 16 -> 32: T[b+16.., b..] = -T[b+16.., b+16..] (A[b+16.., b..] T[b.., b..]), b = 0, 32
  {
    const int half = tid >> 7, ht = tid & 127, b = 32 * half;
    mm_tiles(S + (b + 16) * TS + b, A + (b + 16) * TS + b, T + b * TS + b, 16, 16, 16, 1.f, ht,
             128);
    __syncthreads();
    mm_tiles(T + (b + 16) * TS + b, T + (b + 16) * TS + b + 16, S + (b + 16) * TS + b, 16, 16,
             16, -1.f, ht, 128);
    __syncthreads();
  }
  // 32 -> 64: T[32.., 0..] = -T[32.., 32..] (A[32.., 0..] T[0.., 0..])
  mm_tiles(S + 32 * TS, A + 32 * TS, T, 32, 32, 32, 1.f, tid, PREP_THREADS);
  __syncthreads();
  mm_tiles(T + 32 * TS, T + 32 * TS + 32, S + 32 * TS, 32, 32, 32, -1.f, tid, PREP_THREADS);
  __syncthreads();
}

__device__ __forceinline__ void cp_async4_zfill(void* smem, const void* gmem, bool valid) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  const int n = valid ? 4 : 0;
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(s), "l"(gmem), "r"(n)
               : "memory");
}

__global__ void __launch_bounds__(PREP_THREADS)
prep_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
            const float* __restrict__ alpha, const float* __restrict__ beta, int T, int Hk,
            int Hv, char* __restrict__ ws) {
  extern __shared__ __align__(16) char smem[];
  char* sk = smem + PREP_K;
  char* sq = smem + PREP_Q;
  float* skk = reinterpret_cast<float*>(smem + PREP_KK);
  float* sqk = reinterpret_cast<float*>(smem + PREP_QK);
  float* sa = reinterpret_cast<float*>(smem + PREP_A);
  float* st = reinterpret_cast<float*>(smem + PREP_T);
  float* ss = reinterpret_cast<float*>(smem + PREP_S);
  float* sgate = reinterpret_cast<float*>(smem + PREP_GATE);
  float* slg = reinterpret_cast<float*>(smem + PREP_LG);
  float* sg = reinterpret_cast<float*>(smem + PREP_G);
  float* sb = reinterpret_cast<float*>(smem + PREP_B);

  const int c = blockIdx.x, hk = blockIdx.y, G = Hv / Hk;
  const int t0 = c * C, nv = min(C, T - t0);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int g8 = lane >> 2, t4 = lane & 3;

  // gates of value head hk*G + j into gate buffer j & 1 (rows past the end read as 0)
  auto stage_gates = [&](int j) {
    float* dst = sgate + (j & 1) * 2 * C;
    const int h = hk * G + j;
    if (tid < 2 * C) {
      const int t = tid & 63;
      const bool valid = t < nv;
      const float* src = (tid < C ? alpha : beta) + (size_t)(t0 + (valid ? t : 0)) * Hv + h;
      cp_async4_zfill(dst + tid, src, valid);
    }
  };

  // K and Q rows of the chunk (rows past the end of the sequence read as zero)
  for (int idx = tid; idx < C * 16; idx += PREP_THREADS) {
    const int r = idx >> 4, ch = idx & 15;
    const bool valid = r < nv;
    const size_t src = ((size_t)(t0 + (valid ? r : 0)) * Hk + hk) * DK + ch * 8;
    cp_async16_zfill(sk + r * KS + ch * 16, k + src, valid);
    cp_async16_zfill(sq + r * KS + ch * 16, q + src, valid);
  }
  stage_gates(0);
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();

  // K K^T (warps 0-3) and Q K^T (warps 4-7): 16 rows each, 64 columns
  {
    float acc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
    const int mt = w & 3;
    const char* a0 = (w < 4 ? sk : sq) + (16 * mt + g8) * KS;
#pragma unroll
    for (int kc = 0; kc < DK / 16; ++kc) {
      const int off = (kc * 16 + t4 * 2) * 2;
      const uint32_t a[4] = {ld32(a0 + off), ld32(a0 + 8 * KS + off), ld32(a0 + off + 16),
                             ld32(a0 + 8 * KS + off + 16)};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const char* rb = sk + (nt * 8 + g8) * KS + off;
        mma_bf16_16816(acc[nt], a, ld32(rb), ld32(rb + 16));
      }
    }
    float* dst = w < 4 ? skk : sqk;
    const int r0 = 16 * mt + g8;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int c0 = nt * 8 + t4 * 2;
      dst[r0 * C + c0] = acc[nt][0];
      dst[r0 * C + c0 + 1] = acc[nt][1];
      dst[(r0 + 8) * C + c0] = acc[nt][2];
      dst[(r0 + 8) * C + c0 + 1] = acc[nt][3];
    }
  }
  __syncthreads();

  for (int j = 0; j < G; ++j) {
    const int h = hk * G + j;
    if (j + 1 < G) {
      stage_gates(j + 1);
      cp_async_commit();
    }
    // log-space cumulative decay G_t = sum_{s<=t} log alpha_s (gates of head j landed)
    if (tid < C) {
      const int t = tid;
      const float* gate = sgate + (j & 1) * 2 * C;
      const float a = gate[t], b = gate[C + t];
      float lg = t < nv ? __logf(fmaxf(a, 1e-30f)) : 0.f;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, lg, off);
        if (lane >= off) lg += y;
      }
      slg[t] = lg;
      sb[t] = b;
    }
    __syncthreads();
    if (tid < C) sg[tid] = slg[tid] + (tid >= 32 ? slg[31] : 0.f);
    __syncthreads();
    // A (strictly lower)
    for (int idx = tid; idx < C * C; idx += PREP_THREADS) {
      const int t = idx >> 6, s = idx & 63;
      sa[t * TS + s] = s < t ? sb[t] * __expf(sg[t] - sg[s]) * skk[t * C + s] : 0.f;
    }
    __syncthreads();
    invert_unit_lower(sa, st, ss, tid);
    // P (lower triangular with the diagonal) into S, then P T into the A buffer
    for (int idx = tid; idx < C * C; idx += PREP_THREADS) {
      const int t = idx >> 6, s = idx & 63;
      ss[t * TS + s] = s <= t ? __expf(sg[t] - sg[s]) * sqk[t * C + s] : 0.f;
    }
    __syncthreads();
    mm_lower(sa, ss, st, tid);
    __syncthreads();
    // A = [T; P T] as bf16 hi/lo pairs, g and beta
    char* wsb = ws + ((size_t)c * Hv + h) * WS_STRIDE;
    for (int idx = tid; idx < 2 * C * 8; idx += PREP_THREADS) {
      const int r = idx >> 3, e8 = (idx & 7) * 8;
      const float* src = r < C ? st + r * TS : sa + (r - C) * TS;
      uint32_t hv[4], lv[4];
#pragma unroll
      for (int qd = 0; qd < 4; ++qd) {
        uint32_t h0, l0, h1, l1;
        split_bf16(src[e8 + 2 * qd], h0, l0);
        split_bf16(src[e8 + 2 * qd + 1], h1, l1);
        hv[qd] = h0 | (h1 << 16);
        lv[qd] = l0 | (l1 << 16);
      }
      // 128-byte rows, 16-byte chunk ch of row r stored at chunk ch ^ (r & 7)
      const int off = r * 128 + (((e8 >> 3) ^ (r & 7)) << 4);
      *reinterpret_cast<uint4*>(wsb + WS_AH + off) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
      *reinterpret_cast<uint4*>(wsb + WS_AL + off) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
    }
    if (tid < C) {
      reinterpret_cast<float*>(wsb + WS_G)[tid] = sg[tid];
      reinterpret_cast<float*>(wsb + WS_B)[tid] = sb[tid];
    }
    // the next head's gates have landed and every thread is done with this head
    cp_async_wait<0>();
    __syncthreads();
  }
}

// ------------------------------------------------------------------- scan
// One CTA of 8 warps per (value head, column slab of the state), sequential
// over the chunks.  Every product is a tcgen05 MMA with M = 128 and the slab
// width n as N, accumulating in TMEM:
//
//   D1 = [K; Q] H            rows 0-63: K H,      rows 64-127: Q H
//   D2 = [T; P T] X          rows 0-63: Delta,    rows 64-127: P Delta
//   D3 = K^T D'              rows = the d_k rows of the state update
//
// TMEM lane i is row i of each product.  Warp w reads lanes 32*(w%4) .. +31
// and the columns of its half of the slab (w / 4), so each thread owns one
// row and n/2 columns of D1, D2 and D3 and of the fp32 state.  The "chunk"
// warps (lanes 0-63) turn K H into X and Delta into D' and carry the
// recurrence; the "output" warps (lanes 64-127) keep Q H and finish
// O = g Q H + P Delta while the next MMA runs, joining only for the state
// update.  The B operands (H, X, D' as bf16 hi/lo pairs) are written by their
// owners straight into the 128-byte-swizzle layout.  Thread 0 issues the MMAs;
// thread 64 issues, one chunk ahead, the TMA loads of K, Q and the V slab and
// the bulk copy of the chunk's workspace block (all completing on one mbarrier
// per buffer), and the TMA store of each chunk's output tile.
constexpr int SCAN_THREADS = 256;
constexpr int NMAX = 48;                     // widest column slab
constexpr int NH = NMAX / 2;                 // columns per thread
constexpr int TMEM_COLS = 512;               // D1 at column 0, D2 at 128, D3 at 256
// one staging buffer: K and Q in two d_k halves of 128 rows x 128 bytes (K
// rows 0-63, Q rows 64-127), the workspace block as copied, the V slab [64][n]
constexpr int SB_KQ = 0;
constexpr int SB_KQ_HALF = 16384;
constexpr int SB_W = 32768;
constexpr int SB_V = 66560;                  // SB_W + WS_STRIDE, rounded up to 1 KB
constexpr int SB_SIZE = SB_V + C * NMAX * 2;
static_assert(SB_W + WS_STRIDE <= SB_V && SB_SIZE % 1024 == 0, "staging buffer layout");
// B operands [hi | lo] side by side (2n columns, MN-major): columns 0-63 in
// the first block of 128-byte rows, 64-127 in the second
constexpr int SCAN_HB = 2 * SB_SIZE;         // H: 2 blocks of [128 d_k rows][128 B]
constexpr int SCAN_XB = SCAN_HB + 2 * 16384;  // X: 2 blocks of [64 chunk rows][128 B]
constexpr int SCAN_DB = SCAN_XB + 2 * 8192;   // D'
constexpr int SCAN_O = SCAN_DB + 2 * 8192;    // O tile [64][n] fp32, stored by TMA
constexpr int SCAN_BAR = SCAN_O + C * NMAX * 4;  // mbarriers; TMEM address
constexpr int SCAN_SMEM = SCAN_BAR + 64 + 1024;  // + room to align the base to 1 KB

// polls of an mbarrier before a block gives up
constexpr long long kWaitPolls = 1ll << 22;

// the three column slabs of a 128-wide state: 48 + 48 + 32 columns
__device__ __forceinline__ int slab_width(int s) { return s == 2 ? 32 : 48; }

// nh (16 or 24) fp32 columns of TMEM lane (warp quarter base + lane) starting
// at `taddr`; columns past nh read as zero.
__device__ __forceinline__ void tmem_cols(uint32_t taddr, int nh, float (&x)[NH]) {
  uint32_t r0[8], r1[8], r2[8];
  tc::tmem_ld8(taddr, r0);
  tc::tmem_ld8(taddr + 8, r1);
  if (nh > 16) tc::tmem_ld8(taddr + 16, r2);
  tc::tmem_wait_ld(r0);
  tc::tmem_wait_ld(r1);
  if (nh > 16) {
    tc::tmem_wait_ld(r2);
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) r2[e] = 0u;
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    x[e] = __uint_as_float(r0[e]);
    x[8 + e] = __uint_as_float(r1[e]);
    x[16 + e] = __uint_as_float(r2[e]);
  }
}

// An accumulator of the [hi | lo] products: columns c .. c+nh-1 (at `taddr`)
// plus columns n+c .. n+c+nh-1.
__device__ __forceinline__ void tmem_cols_sum(uint32_t taddr, int n, int nh, float (&x)[NH]) {
  float y[NH];
  tmem_cols(taddr, nh, x);
  tmem_cols(taddr + n, nh, y);
#pragma unroll
  for (int e = 0; e < NH; ++e) x[e] += y[e];
}

// Row `row`, columns c0 .. c0+nh-1 of an fp32 matrix as bf16 hi (columns c0..)
// and lo (columns n+c0..) of a [hi | lo] operand: MN-major, 128-byte swizzle,
// 64 columns per block of rows, blocks `blk` bytes apart (c0, n, nh multiples
// of 8).
__device__ __forceinline__ void put_split(char* base, int blk, int row, int c0, int n,
                                          const float (&x)[NH], int nh) {
#pragma unroll
  for (int cc = 0; cc < NH / 8; ++cc) {
    if (cc * 8 < nh) {
      uint32_t hv[4], lv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        tc::split_bf16x2(x[cc * 8 + 2 * e], x[cc * 8 + 2 * e + 1], hv[e], lv[e]);
      const int ch = c0 + cc * 8, cl = n + ch;
      const int oh = (ch >> 6) * blk + row * 128 + ((((ch & 63) >> 3) ^ (row & 7)) << 4);
      const int ol = (cl >> 6) * blk + row * 128 + ((((cl & 63) >> 3) ^ (row & 7)) << 4);
      *reinterpret_cast<uint4*>(base + oh) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
      *reinterpret_cast<uint4*>(base + ol) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
    }
  }
}

// Barrier over the whole CTA that also orders tcgen05 operations and generic
// shared-memory writes (made visible to the tensor cores) across it; returns
// the AND of `ok` over the CTA.
__device__ __forceinline__ bool tc_barrier(bool ok) {
  fence_proxy_async_smem();
  tc::fence_before_sync();
  const bool all = __syncthreads_and(ok) != 0;
  tc::fence_after_sync();
  return all;
}

// The same over the chunk warps only (warps 0, 1, 4, 5; barrier 1).
__device__ __forceinline__ void chunk_barrier() {
  fence_proxy_async_smem();
  tc::fence_before_sync();
  tc::named_barrier(1, SCAN_THREADS / 2);
  tc::fence_after_sync();
}

__global__ void __launch_bounds__(SCAN_THREADS, 1)
scan_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
            const __grid_constant__ CUtensorMap tm_v48, const __grid_constant__ CUtensorMap tm_v32,
            const __grid_constant__ CUtensorMap tm_o48, const __grid_constant__ CUtensorMap tm_o32,
            float* __restrict__ state, const char* __restrict__ ws, int T, int Hk, int Hv) {
  extern __shared__ __align__(1024) char smem_raw[];
  char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int sl = blockIdx.x, h = blockIdx.y, hk = h / (Hv / Hk);
  const int j0 = 48 * sl, n = slab_width(sl), nh = n / 2;
  const int n_chunks = (T + C - 1) / C;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int qd = w & 3, c0 = (w >> 2) * nh;  // lane quarter; first slab column of this thread
  const int r = 32 * qd + lane;              // TMEM lane: row of D1 / D2 / D3
  const bool chunk_warp = qd < 2;            // rows 0-63: K H, Delta
  const int row = r & (C - 1);               // chunk row (D1 / D2)
  constexpr int kIssuer = 0;                 // issues the MMAs (a chunk warp)
  constexpr int kCopier = 64;                // issues staging and output copies (an output warp)
  const CUtensorMap* tm_v = n == 48 ? &tm_v48 : &tm_v32;
  const CUtensorMap* tm_o = n == 48 ? &tm_o48 : &tm_o32;
  const unsigned stage_bytes = 4 * 8192 + WS_STRIDE + C * n * 2;
  char* hb = smem + SCAN_HB;
  char* xb = smem + SCAN_XB;
  char* db = smem + SCAN_DB;
  float* otile = reinterpret_cast<float*>(smem + SCAN_O);
  // mbarriers: [0], [1] staging buffers; [2], [3], [4] completion of the
  // chunk's first, second and third MMA group (one phase per chunk each)
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + SCAN_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + SCAN_BAR + 40);

  if (tid == 0) {
    for (int i = 0; i < 5; ++i) mbar_init(&bar[i], 1);
    mbar_init_fence();
  }
  if (w == 0) {
    tc::tmem_alloc(tslot, TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc_barrier(true);
  const uint32_t tmem = *tslot;
  const uint32_t t_mine = tmem + ((uint32_t)(32 * qd) << 16) + c0;

  // Staging of chunk c into buffer buf (thread kCopier): K and Q as four TMA
  // tiles of 64 rows x 64 columns in the 128-byte swizzle, the V slab as one
  // tile (rows past the end of the sequence arrive as zero), the workspace
  // block by one bulk copy, all completing on bar[buf].
  auto stage = [&](int c, int buf) {
    char* B = smem + buf * SB_SIZE;
    const int t0 = c * C;
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(&bar[buf], stage_bytes);
    tc::tma_load_2d(B + SB_KQ, &tm_k, hk * DK, t0, &bar[buf]);
    tc::tma_load_2d(B + SB_KQ + SB_KQ_HALF, &tm_k, hk * DK + 64, t0, &bar[buf]);
    tc::tma_load_2d(B + SB_KQ + C * 128, &tm_q, hk * DK, t0, &bar[buf]);
    tc::tma_load_2d(B + SB_KQ + SB_KQ_HALF + C * 128, &tm_q, hk * DK + 64, t0, &bar[buf]);
    tc::tma_load_2d(B + SB_V, tm_v, h * DV + j0, t0, &bar[buf]);
    bulk_g2s(B + SB_W, ws + ((size_t)c * Hv + h) * WS_STRIDE, WS_STRIDE, &bar[buf]);
  };

  // this thread's part of the state: d_k row r, slab columns c0 .. c0+nh-1
  float Hr[NH];
  float* srow = state + ((size_t)h * DK + r) * DV + j0 + c0;
#pragma unroll
  for (int e = 0; e < NH; e += 4) {
    const float4 x = e < nh ? *reinterpret_cast<const float4*>(srow + e)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
    Hr[e] = x.x; Hr[e + 1] = x.y; Hr[e + 2] = x.z; Hr[e + 3] = x.w;
  }
  put_split(hb, 16384, r, c0, n, Hr, nh);
  if (tid == kCopier) stage(0, 0);
  int inflight = 0;  // chunk whose staging is in flight, or -1

  // A K-major or MN-major (K^T); B MN-major with 2n ([hi | lo]) or n (hi) columns
  const uint32_t id_cat = tc::idesc_bf16_f32(128, 2 * n, false, true);
  const uint32_t id_hi = tc::idesc_bf16_f32(128, n, false, true);
  const uint32_t id_kt = tc::idesc_bf16_f32(128, 2 * n, true, true);
  const uint32_t s_hb = smem_addr(hb), s_xb = smem_addr(xb), s_db = smem_addr(db);
  bool ok = true;
  for (int c = 0; c < n_chunks; ++c) {
    const int buf = c & 1, t0 = c * C;
    const unsigned par = c & 1;
    char* B = smem + buf * SB_SIZE;
    ok = tc_barrier(ok && mbar_wait_bounded(&bar[buf], (c >> 1) & 1, kWaitPolls));
    if (!ok) break;
    const uint32_t s_kq = smem_addr(B + SB_KQ);
    const uint32_t s_ah = smem_addr(B + SB_W + WS_AH), s_al = smem_addr(B + SB_W + WS_AL);
    const float* bG = reinterpret_cast<const float*>(B + SB_W + WS_G);
    const float* bb = reinterpret_cast<const float*>(B + SB_W + WS_B);

    // ---- D1 = [K; Q] [H_hi | H_lo]
    if (tid == kIssuer) {
#pragma unroll
      for (int s = 0; s < DK / 16; ++s) {
        const uint64_t a = tc::sdesc_sw128(s_kq + (s >> 2) * SB_KQ_HALF + (s & 3) * 32, 16, 1024);
        tc::mma_bf16(tmem, a, tc::sdesc_sw128(s_hb + s * 2048, 16384, 1024), id_cat, s > 0);
      }
      tc::mma_commit(&bar[2]);
    }
    // the next chunk's staging (its buffer was last read by the previous chunk)
    inflight = -1;
    if (c + 1 < n_chunks) {
      if (tid == kCopier) stage(c + 1, buf ^ 1);
      inflight = c + 1;
    }
    const float G_r = bG[row], GC = bG[C - 1];
    const float g_r = __expf(G_r), b_r = bb[row], gC = __expf(GC);
    uint4 vr[NH / 8];
    if (chunk_warp) {
      const uint4* vsrc = reinterpret_cast<const uint4*>(B + SB_V + (row * n + c0) * 2);
#pragma unroll
      for (int e = 0; e < NH / 8; ++e) vr[e] = e * 8 < nh ? vsrc[e] : make_uint4(0u, 0u, 0u, 0u);
    }
    ok = mbar_wait_bounded(&bar[2], par, kWaitPolls) && ok;
    tc::fence_after_sync();
    float qh[NH];
    {
      float x[NH];
      tmem_cols_sum(t_mine, n, nh, x);
      if (chunk_warp) {
        // X = beta (V - g K H)
#pragma unroll
        for (int e = 0; e < NH / 8; ++e) {
          const uint32_t p[4] = {vr[e].x, vr[e].y, vr[e].z, vr[e].w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = e * 8 + 2 * u;
            x[j] = b_r * (__uint_as_float(p[u] << 16) - g_r * x[j]);
            x[j + 1] = b_r * (__uint_as_float(p[u] & 0xffff0000u) - g_r * x[j + 1]);
          }
        }
        put_split(xb, 8192, row, c0, n, x, nh);
        chunk_barrier();
        // ---- D2 = A_hi [X_hi | X_lo] + A_lo X_hi,  A = [T; P T]
        if (tid == kIssuer) {
#pragma unroll
          for (int s = 0; s < C / 16; ++s) {
            const uint64_t xd = tc::sdesc_sw128(s_xb + s * 2048, 8192, 1024);
            tc::mma_bf16(tmem + 128, tc::sdesc_sw128(s_ah + s * 32, 16, 1024), xd, id_cat, s > 0);
            tc::mma_bf16(tmem + 128, tc::sdesc_sw128(s_al + s * 32, 16, 1024), xd, id_hi, 1);
          }
          tc::mma_commit(&bar[3]);
        }
      } else {
#pragma unroll
        for (int e = 0; e < NH; ++e) qh[e] = g_r * x[e];
      }
    }
    ok = mbar_wait_bounded(&bar[3], par, kWaitPolls) && ok;
    tc::fence_after_sync();
    {
      float x[NH];
      tmem_cols_sum(t_mine + 128, n, nh, x);
      if (chunk_warp) {
        // D' = (g_C / g) Delta
        const float rg = __expf(GC - G_r);
#pragma unroll
        for (int e = 0; e < NH; ++e) x[e] *= rg;
        put_split(db, 8192, row, c0, n, x, nh);
        chunk_barrier();
        // ---- D3 = K^T [D'_hi | D'_lo]
        if (tid == kIssuer) {
#pragma unroll
          for (int s = 0; s < C / 16; ++s)
            tc::mma_bf16(tmem + 256, tc::sdesc_sw128(s_kq + s * 2048, SB_KQ_HALF, 1024),
                         tc::sdesc_sw128(s_db + s * 2048, 8192, 1024), id_kt, s > 0);
          tc::mma_commit(&bar[4]);
        }
      } else {
        // O = g Q H + P Delta into the output tile, stored by one TMA copy
        float* orow = otile + row * n + c0;
#pragma unroll
        for (int e = 0; e < NH; e += 4)
          if (e < nh)
            *reinterpret_cast<float4*>(orow + e) =
                make_float4(qh[e] + x[e], qh[e + 1] + x[e + 1], qh[e + 2] + x[e + 2],
                            qh[e + 3] + x[e + 3]);
        fence_proxy_async_smem();
        tc::named_barrier(2, SCAN_THREADS / 2);
        if (tid == kCopier) {
          tc::tma_store_2d(tm_o, h * DV + j0, t0, otile);
          tc::bulk_commit();
        }
      }
    }
    // ---- H <- g_C H + D3
    ok = mbar_wait_bounded(&bar[4], par, kWaitPolls) && ok;
    tc::fence_after_sync();
    {
      float x[NH];
      tmem_cols_sum(t_mine + 256, n, nh, x);
#pragma unroll
      for (int e = 0; e < NH; ++e) Hr[e] = fmaf(gC, Hr[e], x[e]);
      put_split(hb, 16384, r, c0, n, Hr, nh);
    }
    // the output tile is rewritten next chunk: its store must have read it
    if (tid == kCopier) tc::bulk_wait_read_all();
  }

  ok = tc_barrier(ok);
  if (tid == kCopier) {
    // a staged chunk or an MMA never completed: give the staging still in
    // flight a last bounded chance to land; the output stores complete here
    if (!ok && inflight >= 0)
      mbar_wait_bounded(&bar[inflight & 1], (inflight >> 1) & 1, kWaitPolls);
    tc::bulk_wait_all();
  }
  if (!ok) {
#pragma unroll
    for (int e = 0; e < NH; ++e) Hr[e] = __int_as_float(0x7fc00000);  // the slab failed
  }
#pragma unroll
  for (int e = 0; e < NH; e += 4)
    if (e < nh)
      *reinterpret_cast<float4*>(srow + e) = make_float4(Hr[e], Hr[e + 1], Hr[e + 2], Hr[e + 3]);
  tc_barrier(true);
  if (w == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

// ---------------------------------------------------------------------------
// Built-in scratch for gdn_prefill_chunked_noalloc: a file-scope device array,
// so that callers who cannot allocate device memory still get the chunked
// prefill.  Every GPU that loads the library holds it until the process exits.
// Host code must not hand the symbol itself to a kernel (on the host it names
// a stand-in, not device memory): its device address is looked up once per
// device with cudaGetSymbolAddress and cached.
static __device__ __align__(256) char g_prefill_scratch[GDN_PREFILL_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 256;

// Device address of g_prefill_scratch on the current device (set up on the
// first call for that device).  Returns GDN_OK or GDN_ERR_CUDA.
int scratch_on_current_device(void** ptr) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_prefill_scratch) != cudaSuccess || p == nullptr)
      return GDN_ERR_CUDA;
    addr[dev] = p;
  }
  *ptr = addr[dev];
  return GDN_OK;
}

}  // namespace

int launch_prefill_noalloc(const void* q, const void* k, const void* v, bool bf16,
                           const float* alpha, const float* beta, int T, int Hk, int Hv, int dk,
                           int dv, int chunk, float* state, float* o, cudaStream_t stream) {
  if (!bf16 || dk != DK || dv != DV || chunk != C) return GDN_ERR_UNSUPPORTED;
  const size_t need = prefill_workspace_bytes(T, Hk, Hv, dk, dv, chunk);
  if (need > (size_t)GDN_PREFILL_NOALLOC_SCRATCH_BYTES) return GDN_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  const int st = scratch_on_current_device(&scratch);
  if (st != GDN_OK) return st;
  return launch_prefill(q, k, v, bf16, alpha, beta, T, Hk, Hv, dk, dv, chunk, state, o, scratch,
                        stream);
}

size_t prefill_workspace_bytes(int T, int Hk, int Hv, int dk, int dv, int chunk) {
  (void)Hk;
  if (dk != DK || dv != DV || chunk != C) return 0;
  const size_t n_chunks = ((size_t)T + C - 1) / C;
  return n_chunks * (size_t)Hv * WS_STRIDE;
}

namespace {

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library); null if the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult res;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &res) != cudaSuccess ||
        res != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// A [T][heads][128] tensor (bf16 or fp32) as a 2-D tensor of T rows and
// heads*128 columns, moved in tiles of `box_cols` x 64 rows (rows past T read
// as zero and are not written).
int rows_tensor_map(CUtensorMap* m, const void* base, CUtensorMapDataType type, int elem_bytes,
                    int T, int heads, int box_cols, CUtensorMapSwizzle swizzle) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return GDN_ERR_CUDA;
  const cuuint64_t dims[2] = {(cuuint64_t)heads * DK, (cuuint64_t)T};
  const cuuint64_t strides[1] = {(cuuint64_t)heads * DK * elem_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, 64};
  const cuuint32_t elem[2] = {1, 1};
  const CUresult r = enc(m, type, 2, const_cast<void*>(base), dims, strides, box, elem,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

int launch_prefill(const void* q, const void* k, const void* v, bool bf16, const float* alpha,
                   const float* beta, int T, int Hk, int Hv, int dk, int dv, int chunk,
                   float* state, float* o, void* workspace, cudaStream_t stream) {
  if (!bf16 || dk != DK || dv != DV || chunk != C) return GDN_ERR_UNSUPPORTED;
  const int n_chunks = (T + C - 1) / C;
  // K and Q in 64 x 64 tiles, 128-byte swizzle; V and O in 64-row tiles of
  // one column slab (48 or 32 wide), unswizzled
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapDataType f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  CUtensorMap tm_k, tm_q, tm_v48, tm_v32, tm_o48, tm_o32;
  int st = rows_tensor_map(&tm_k, k, bf, 2, T, Hk, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st == GDN_OK) st = rows_tensor_map(&tm_q, q, bf, 2, T, Hk, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st == GDN_OK) st = rows_tensor_map(&tm_v48, v, bf, 2, T, Hv, 48, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st == GDN_OK) st = rows_tensor_map(&tm_v32, v, bf, 2, T, Hv, 32, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st == GDN_OK) st = rows_tensor_map(&tm_o48, o, f32, 4, T, Hv, 48, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st == GDN_OK) st = rows_tensor_map(&tm_o32, o, f32, 4, T, Hv, 32, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st != GDN_OK) return st;
  if (cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           PREP_SMEM) != cudaSuccess ||
      cudaFuncSetAttribute(scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           SCAN_SMEM) != cudaSuccess)
    return GDN_ERR_CUDA;
  prep_kernel<<<dim3(n_chunks, Hk), PREP_THREADS, PREP_SMEM, stream>>>(
      static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(k), alpha, beta, T, Hk, Hv,
      static_cast<char*>(workspace));
  st = launch_status();
  if (st != GDN_OK) return st;
  scan_kernel<<<dim3(3, Hv), SCAN_THREADS, SCAN_SMEM, stream>>>(
      tm_k, tm_q, tm_v48, tm_v32, tm_o48, tm_o32, state, static_cast<const char*>(workspace), T,
      Hk, Hv);
  return launch_status();
}

}  // namespace gdn
