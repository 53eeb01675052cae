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
//         cores (mma.sync), the log-space cumulative decay G, A and P, the
//         inverse T = (I + A)^-1 by 16 x 16 blocks and P T; [T; P T] goes to
//         the caller's workspace as bf16 hi/lo pairs in the tensor cores'
//         128-byte swizzle, with G and beta.
//   scan  (grid: value head x 3 column slabs of the state, sequential over
//         chunks): per chunk three tcgen05 MMA groups with M = 128 into
//         tensor memory, [K; Q] H, [T; P T] X and K^T D', with the
//         elementwise steps between them (X, D', O = g Q H + P Delta,
//         H <- g_C H + K^T D').  The fp32 state stays in registers for the
//         whole sequence; the next chunk's K, Q, V and workspace block are
//         staged by TMA while the current one is processed, and each chunk's
//         output tile leaves by one TMA store.
//
// Precision: every tensor-core operand that is not exactly a bf16 input (the
// state, X, D', T, P T and the fp32 operands of the prep's block products) is
// carried as a bf16 pair hi + lo and multiplied as hi*hi + hi*lo + lo*hi (or
// hi + lo against an exact bf16 K / Q), which keeps ~16 significant bits per
// operand; a single bf16 rounding of any of them costs ~1% of the output RMS
// at this size.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

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
// One CTA per (chunk, q/k head), 8 warps.  K K^T and Q K^T are formed once on
// tensor cores and stay in the warps' accumulator fragments; the value heads
// of the q/k head are then handled three at a time:
//   1. gates: warp j scans log alpha of head j (two rows per lane) into the
//      log decay G, and writes G and beta to the workspace;
//   2. A = beta_t e^{G_t - G_s} K K^T (s < t) and P = e^{G_t - G_s} Q K^T
//      (s <= t) straight from the accumulators into shared memory (fp32);
//   3. T = (I + A)^-1 by blocks of 16: the diagonal blocks by forward
//      substitution, then N = D A below the diagonal and T block row by block
//      row; P T block by block (the block products on tensor cores with the
//      fp32 operands split into bf16 hi/lo pairs);
//   4. [T; P T] as bf16 hi/lo pairs into the workspace block, 16 bytes a store.
constexpr int PREP_THREADS = 256;
constexpr int HG = 3;    // value heads per pass
constexpr int AS = 68;   // fp32 row stride of A and P (16-byte rows, spread banks)
// shared memory: the K / Q staging (dead once K K^T and Q K^T are formed) is
// reused by A and P of the pass's heads
constexpr int PREP_K = 0;
constexpr int PREP_Q = PREP_K + C * KS;
constexpr int PREP_AP = 0;                          // [head][A, P][64][AS] fp32
constexpr int PREP_AP_SIZE = HG * 2 * C * AS * 4;
static_assert(2 * C * KS <= PREP_AP_SIZE, "K and Q staging fits in the A / P area");
constexpr int PREP_GATE = PREP_AP_SIZE;              // [head][alpha 64, beta 64]
constexpr int PREP_G = PREP_GATE + HG * 2 * C * 4;   // [head][64] log decay
constexpr int PREP_B = PREP_G + HG * C * 4;          // [head][64] beta
constexpr int PREP_E = PREP_B + HG * C * 4;          // [head][64] exp(G_t - G_ref)
constexpr int PREP_F = PREP_E + HG * C * 4;          // [head][64] exp(G_ref - G_s)
constexpr int PREP_SEP = PREP_F + HG * C * 4;        // [head] the split above is safe
constexpr int PREP_SMEM = PREP_SEP + 16;
// with more than HG value heads per q/k head the accumulator fragments are
// parked in shared memory between passes (one float4 row per thread and tile)
constexpr int PREP_ACC = PREP_SMEM;
constexpr int PREP_SMEM_MULTIPASS = PREP_ACC + PREP_THREADS * 32 * 4;

__device__ __forceinline__ void cp_async4_zfill(void* smem, const void* gmem, bool valid) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  const int n = valid ? 4 : 0;
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(s), "l"(gmem), "r"(n)
               : "memory");
}

// Fragments of 16 x 16 fp32 blocks (row stride AS) for mma m16n8k16, as bf16
// hi/lo pairs: the A operand X (row-major) and the B operand Y (columns
// 8*nh .. 8*nh+7).
__device__ __forceinline__ void frag_a(const float* X, int g8, int t4, uint32_t (&hi)[4],
                                       uint32_t (&lo)[4]) {
  const float2 x0 = *reinterpret_cast<const float2*>(X + g8 * AS + 2 * t4);
  const float2 x1 = *reinterpret_cast<const float2*>(X + (g8 + 8) * AS + 2 * t4);
  const float2 x2 = *reinterpret_cast<const float2*>(X + g8 * AS + 2 * t4 + 8);
  const float2 x3 = *reinterpret_cast<const float2*>(X + (g8 + 8) * AS + 2 * t4 + 8);
  tc::split_bf16x2(x0.x, x0.y, hi[0], lo[0]);
  tc::split_bf16x2(x1.x, x1.y, hi[1], lo[1]);
  tc::split_bf16x2(x2.x, x2.y, hi[2], lo[2]);
  tc::split_bf16x2(x3.x, x3.y, hi[3], lo[3]);
}

__device__ __forceinline__ void frag_b(const float* Y, int nh, int g8, int t4, uint32_t (&hi)[2],
                                       uint32_t (&lo)[2]) {
  const int n = 8 * nh + g8;
  tc::split_bf16x2(Y[(2 * t4) * AS + n], Y[(2 * t4 + 1) * AS + n], hi[0], lo[0]);
  tc::split_bf16x2(Y[(2 * t4 + 8) * AS + n], Y[(2 * t4 + 9) * AS + n], hi[1], lo[1]);
}

// acc (16 x 16 as two 16 x 8 accumulator tiles) += X Y, with the three
// products hi*hi + hi*lo + lo*hi of the bf16 pairs.
__device__ __forceinline__ void block_mma(float (&acc)[2][4], const float* X, const float* Y,
                                          int g8, int t4) {
  uint32_t ah[4], al[4];
  frag_a(X, g8, t4, ah, al);
#pragma unroll
  for (int nh = 0; nh < 2; ++nh) {
    uint32_t bh[2], bl[2];
    frag_b(Y, nh, g8, t4, bh, bl);
    mma_bf16_16816(acc[nh], ah, bh[0], bh[1]);
    mma_bf16_16816(acc[nh], ah, bl[0], bl[1]);
    mma_bf16_16816(acc[nh], al, bh[0], bh[1]);
  }
}

// sign * acc into the 16 x 16 fp32 block at Z (row stride AS).
__device__ __forceinline__ void put_block(float* Z, const float (&acc)[2][4], float sign, int g8,
                                          int t4) {
#pragma unroll
  for (int nh = 0; nh < 2; ++nh) {
    const int col = 8 * nh + 2 * t4;
    *reinterpret_cast<float2*>(Z + g8 * AS + col) = make_float2(sign * acc[nh][0], sign * acc[nh][1]);
    *reinterpret_cast<float2*>(Z + (g8 + 8) * AS + col) =
        make_float2(sign * acc[nh][2], sign * acc[nh][3]);
  }
}

__global__ void __launch_bounds__(PREP_THREADS, 2)
prep_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
            const float* __restrict__ alpha, const float* __restrict__ beta, int T, int Hk,
            int Hv, char* __restrict__ ws) {
  pdl_enter();
  extern __shared__ __align__(16) char smem[];
  char* sk = smem + PREP_K;
  char* sq = smem + PREP_Q;
  float* sap = reinterpret_cast<float*>(smem + PREP_AP);
  float* sgate = reinterpret_cast<float*>(smem + PREP_GATE);
  float* sG = reinterpret_cast<float*>(smem + PREP_G);
  float* sB = reinterpret_cast<float*>(smem + PREP_B);
  float* sE = reinterpret_cast<float*>(smem + PREP_E);
  float* sF = reinterpret_cast<float*>(smem + PREP_F);
  int* ssep = reinterpret_cast<int*>(smem + PREP_SEP);

  const int c = blockIdx.x, hk = blockIdx.y, G = Hv / Hk;
  const int t0 = c * C, nv = min(C, T - t0);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int g8 = lane >> 2, t4 = lane & 3;

  // gates of the pass's value heads (rows past the end read as zero)
  auto stage_gates = [&](int h0, int ng) {
    for (int idx = tid; idx < ng * 2 * C; idx += PREP_THREADS) {
      const int j = idx / (2 * C), e = idx - j * 2 * C, t = e & (C - 1);
      const bool valid = t < nv;
      const float* src = (e < C ? alpha : beta) + (size_t)(t0 + (valid ? t : 0)) * Hv + h0 + j;
      cp_async4_zfill(sgate + idx, src, valid);
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
  stage_gates(hk * G, min(HG, G));
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();

  // K K^T (warps 0-3) and Q K^T (warps 4-7): rows 16*mt + g8 (+8), all 64 columns
  const int mt = w & 3;
  const bool is_kk = w < 4;
  float acc[8][4];
#pragma unroll
  for (int nt = 0; nt < 8; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
  {
    const char* a0 = (is_kk ? sk : sq) + (16 * mt + g8) * KS;
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
  }

  // Steps 1-3 for value heads h0 .. h0+ng-1 from the accumulators `a`.
  auto pass = [&](int h0, int ng, const float (&a)[8][4]) {
    __syncthreads();  // gates landed; K / Q (or the previous A / P) no longer read
    // ---- 1. log decay of head j by warp j: lane l holds rows 2l, 2l+1
    if (w < ng) {
      const float* ga = sgate + w * 2 * C;
      const int ta = 2 * lane, tb = ta + 1;
      const float la = ta < nv ? __logf(fmaxf(ga[ta], 1e-30f)) : 0.f;
      const float lb = tb < nv ? __logf(fmaxf(ga[tb], 1e-30f)) : 0.f;
      float sum = la + lb;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, sum, off);
        if (lane >= off) sum += y;
      }
      const float Ga = sum - lb, Gb = sum;
      sG[w * C + ta] = Ga;
      sG[w * C + tb] = Gb;
      sB[w * C + ta] = ga[C + ta];
      sB[w * C + tb] = ga[C + tb];
      char* wsb = ws + ((size_t)c * Hv + h0 + w) * WS_STRIDE;
      *reinterpret_cast<float2*>(wsb + WS_G + ta * 4) = make_float2(Ga, Gb);
      *reinterpret_cast<float2*>(wsb + WS_B + ta * 4) = make_float2(ga[C + ta], ga[C + tb]);
      // e^{G_t - G_s} = E_t F_s with E_t = e^{G_t - G_ref}, F_s = e^{G_ref - G_s}
      // around the middle row; used when no factor can overflow (the decay
      // across the chunk stays within e^{+-80}), else A and P take e^{G_t - G_s}
      const float Gref = __shfl_sync(0xffffffffu, Gb, 15);
      float span = fmaxf(fabsf(Ga - Gref), fabsf(Gb - Gref));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
        span = fmaxf(span, __shfl_xor_sync(0xffffffffu, span, off));
      sE[w * C + ta] = __expf(Ga - Gref);
      sE[w * C + tb] = __expf(Gb - Gref);
      sF[w * C + ta] = __expf(Gref - Ga);
      sF[w * C + tb] = __expf(Gref - Gb);
      if (lane == 0) ssep[w] = span <= 80.f;
    }
    __syncthreads();
    // ---- 2. A (warps 0-3) and P (warps 4-7) of each head from the accumulators
    //      (column tiles wholly above this warp's 16 rows are zero)
    for (int j = 0; j < ng; ++j) {
      float* dst = sap + (j * 2 + (is_kk ? 0 : 1)) * C * AS;
      const float* Gj = sG + j * C;
      const float* Ej = sE + j * C;
      const float* Fj = sF + j * C;
      const bool sep = ssep[j] != 0;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int t = 16 * mt + g8 + 8 * half;
        const float Gt = Gj[t], bt = is_kk ? sB[j * C + t] : 1.f, bE = bt * Ej[t];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          const int s = nt * 8 + 2 * t4;
          float v0 = 0.f, v1 = 0.f;
          if (nt * 8 <= 16 * mt + 15) {
            const bool m0 = is_kk ? s < t : s <= t, m1 = is_kk ? s + 1 < t : s + 1 <= t;
            if (sep) {
              const float2 f = *reinterpret_cast<const float2*>(Fj + s);
              v0 = m0 ? bE * f.x * a[nt][2 * half] : 0.f;
              v1 = m1 ? bE * f.y * a[nt][2 * half + 1] : 0.f;
            } else {
              v0 = m0 ? bt * __expf(Gt - Gj[s]) * a[nt][2 * half] : 0.f;
              v1 = m1 ? bt * __expf(Gt - Gj[s + 1]) * a[nt][2 * half + 1] : 0.f;
            }
          }
          *reinterpret_cast<float2*>(dst + t * AS + s) = make_float2(v0, v1);
        }
      }
    }
    __syncthreads();
    // ---- 3. T = (I + A)^-1 in 16 x 16 blocks, in place of A:
    //   D_b = (I + A_bb)^-1 (forward substitution, one column per thread),
    //   N_ik = D_i A_ik (i > k), then block row by block row
    //   T_ij = -sum_{k=j}^{i-1} N_ik T_kj  (T_jj = D_j),
    // and P T in place of P: (P T)_ij = sum_{k=j}^{i} P_ik T_kj.
    {
      const bool solver = tid < ng * C;
      const int j = tid >> 6, b = (tid >> 4) & 3, cl = tid & 15;
      float* Ab = sap + (j * 2) * C * AS + (16 * b) * AS + 16 * b;
      float x[16];
      if (solver) {
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
          for (int r = 0; r < t; ++r) {
            if (r & 1) acc1 = fmaf(Ab[t * AS + r], x[r], acc1);
            else acc0 = fmaf(Ab[t * AS + r], x[r], acc0);
          }
          x[t] = t == cl ? 1.f : (t < cl ? 0.f : -(acc0 + acc1));
        }
      }
      __syncthreads();  // every solver has read its diagonal block
      if (solver) {
#pragma unroll
        for (int t = 0; t < 16; ++t) Ab[t * AS + cl] = x[t];
      }
    }
    __syncthreads();
    // N_ik = D_i A_ik over the 6 blocks below the diagonal of each head
    for (int task = w; task < ng * 6; task += PREP_THREADS / 32) {
      const int j = task / 6, p = task - j * 6;
      const int i = p < 1 ? 1 : (p < 3 ? 2 : 3), k = p - (i * (i - 1)) / 2;
      float* Am = sap + (j * 2) * C * AS;
      float acc[2][4] = {};
      block_mma(acc, Am + 16 * i * AS + 16 * i, Am + 16 * i * AS + 16 * k, g8, t4);
      put_block(Am + 16 * i * AS + 16 * k, acc, 1.f, g8, t4);  // only this task reads A_ik
    }
    __syncthreads();
    // block rows 1, 2, 3 of T
    for (int i = 1; i < 4; ++i) {
      float res[2][2][4];
      int dst[2] = {-1, -1};
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int task = w + u * (PREP_THREADS / 32);
        if (task < ng * i) {
          const int j = task / i, jb = task - j * i;
          float* Am = sap + (j * 2) * C * AS;
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e) res[u][h][e] = 0.f;
          for (int k = jb; k < i; ++k)
            block_mma(res[u], Am + 16 * i * AS + 16 * k, Am + 16 * k * AS + 16 * jb, g8, t4);
          dst[u] = (j * 2) * C * AS + 16 * i * AS + 16 * jb;
        }
      }
      __syncthreads();  // the row's N blocks are read
#pragma unroll
      for (int u = 0; u < 2; ++u)
        if (dst[u] >= 0) put_block(sap + dst[u], res[u], -1.f, g8, t4);
      __syncthreads();
    }
    // P T over the 10 blocks on and below the diagonal of each head
    {
      float res[4][2][4];
      int dst[4] = {-1, -1, -1, -1};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int task = w + u * (PREP_THREADS / 32);
        if (task < ng * 10) {
          const int j = task / 10, p = task - j * 10;
          const int i = p < 1 ? 0 : (p < 3 ? 1 : (p < 6 ? 2 : 3)), jb = p - (i * (i + 1)) / 2;
          const float* Tm = sap + (j * 2) * C * AS;
          float* Pm = sap + (j * 2 + 1) * C * AS;
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e) res[u][h][e] = 0.f;
          for (int k = jb; k <= i; ++k)
            block_mma(res[u], Pm + 16 * i * AS + 16 * k, Tm + 16 * k * AS + 16 * jb, g8, t4);
          dst[u] = (j * 2 + 1) * C * AS + 16 * i * AS + 16 * jb;
        }
      }
      __syncthreads();  // P is read
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (dst[u] >= 0) put_block(sap + dst[u], res[u], 1.f, g8, t4);
      __syncthreads();
    }
    // ---- 4. [T; P T] as bf16 hi/lo into the workspace: 16 bytes per row chunk
    for (int idx = tid; idx < ng * 2 * C * 8; idx += PREP_THREADS) {
      const int j = idx / (2 * C * 8), rem = idx - j * 2 * C * 8;
      const int r = rem >> 3, e8 = (rem & 7) * 8;  // row of [T; P T], first column
      const float* src = sap + (j * 2 + (r >= C)) * C * AS + (r & (C - 1)) * AS + e8;
      const float4 x0 = *reinterpret_cast<const float4*>(src);
      const float4 x1 = *reinterpret_cast<const float4*>(src + 4);
      uint32_t hv[4], lv[4];
      tc::split_bf16x2(x0.x, x0.y, hv[0], lv[0]);
      tc::split_bf16x2(x0.z, x0.w, hv[1], lv[1]);
      tc::split_bf16x2(x1.x, x1.y, hv[2], lv[2]);
      tc::split_bf16x2(x1.z, x1.w, hv[3], lv[3]);
      char* wsb = ws + ((size_t)c * Hv + h0 + j) * WS_STRIDE;
      const int off = r * 128 + (((e8 >> 3) ^ (r & 7)) << 4);
      *reinterpret_cast<uint4*>(wsb + WS_AH + off) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
      *reinterpret_cast<uint4*>(wsb + WS_AL + off) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
    }
  };

  if (G > HG) {
    // park the accumulators for the later passes
    float4* park = reinterpret_cast<float4*>(smem + PREP_ACC) + tid;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
      park[nt * PREP_THREADS] = make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
  }
  pass(hk * G, min(HG, G), acc);
  for (int h0 = hk * G + HG; h0 < (hk + 1) * G; h0 += HG) {
    // the previous pass is done with the gate buffer once every thread is here
    __syncthreads();
    stage_gates(h0, min(HG, (hk + 1) * G - h0));
    cp_async_commit();
    cp_async_wait<0>();
    float a2[8][4];
    const float4* park = reinterpret_cast<const float4*>(smem + PREP_ACC) + tid;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const float4 x = park[nt * PREP_THREADS];
      a2[nt][0] = x.x; a2[nt][1] = x.y; a2[nt][2] = x.z; a2[nt][3] = x.w;
    }
    pass(h0, min(HG, (hk + 1) * G - h0), a2);
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
constexpr int SCAN_THREADS = 384;          // 12 warps: 4 lane quarters x 3 column groups
constexpr int NMAX = 48;                     // widest column slab
constexpr int NH = 16;                       // columns per thread
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

// An accumulator of the [hi | lo] products: the NH = 16 fp32 columns of this
// thread's TMEM lane at `taddr` plus the 16 at taddr + n, both loads in
// flight together (one wait).
__device__ __forceinline__ void tmem_cols_sum(uint32_t taddr, int n, float (&x)[NH]) {
  uint32_t r0[16], r1[16];
  tc::tmem_ld16(taddr, r0);
  tc::tmem_ld16(taddr + n, r1);
  tc::tmem_wait_ld(r0);
  tc::tmem_ready(r1);
#pragma unroll
  for (int e = 0; e < NH; ++e) x[e] = __uint_as_float(r0[e]) + __uint_as_float(r1[e]);
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

// The same over the chunk warps only (lane quarters 0 and 1; barrier 1).
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
            float* __restrict__ state, const char* __restrict__ ws, int T, int Hk, int Hv,
            int32_t* __restrict__ status) {
  pdl_enter();
  extern __shared__ __align__(1024) char smem_raw[];
  char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int sl = blockIdx.x, h = blockIdx.y, hk = h / (Hv / Hk);
  const int j0 = 48 * sl, n = slab_width(sl);
  const int n_chunks = (T + C - 1) / C;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int qd = w & 3, c0 = (w >> 2) * NH;  // lane quarter; first slab column of this thread
  const bool active = c0 < n;                // a 32-wide slab leaves the third group idle
  const int nh = active ? NH : 0;            // columns this thread owns
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
  // chunk's first, second and third MMA group (one phase per chunk each);
  // [5] all MMAs issued, on the failure path only
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + SCAN_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + SCAN_BAR + 48);

  if (tid == 0) {
    for (int i = 0; i < 6; ++i) mbar_init(&bar[i], 1);
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
      if (active) tmem_cols_sum(t_mine, n, x);
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
      if (active) tmem_cols_sum(t_mine + 128, n, x);
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
      if (active) tmem_cols_sum(t_mine + 256, n, x);
#pragma unroll
      for (int e = 0; e < NH; ++e) Hr[e] = fmaf(gC, Hr[e], x[e]);
      put_split(hb, 16384, r, c0, n, Hr, nh);
    }
    // the output tile is rewritten next chunk: its store must have read it
    if (tid == kCopier) tc::bulk_wait_read_all();
  }

  ok = tc_barrier(ok);
  if (!ok) {
    // A wait expired.  Before the tensor memory is released, every MMA this
    // CTA issued must have completed (one more commit tracks all of them) and
    // the staging still in flight must have landed; each wait is bounded.
    if (tid == kIssuer) {
      tc::mma_commit(&bar[5]);
      mbar_wait_bounded(&bar[5], 0, kWaitPolls);
      report(status, GDN_ERR_TIMEOUT);
    }
    if (tid == kCopier && inflight >= 0)
      mbar_wait_bounded(&bar[inflight & 1], (inflight >> 1) & 1, kWaitPolls);
  }
  if (tid == kCopier) tc::bulk_wait_all();  // the output stores complete here
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
// a stand-in, not device memory): its device address on the current device is
// looked up with cudaGetSymbolAddress on every call.  The lookup is a host-side
// query; repeating it means that a device reset or a new primary context,
// after which the module is loaded again (possibly elsewhere), never receives
// an address from before.
static __device__ __align__(256) char g_prefill_scratch[GDN_PREFILL_NOALLOC_SCRATCH_BYTES];

int launch_prefill_noalloc(const void* q, const void* k, const void* v, bool bf16,
                           const float* alpha, const float* beta, int T, int Hk, int Hv, int dk,
                           int dv, int chunk, float* state, float* o, int32_t* status,
                           cudaStream_t stream) {
  if (!bf16 || dk != DK || dv != DV || chunk != C) return GDN_ERR_UNSUPPORTED;
  const size_t need = prefill_workspace_bytes(T, Hk, Hv, dk, dv, chunk);
  if (need > (size_t)GDN_PREFILL_NOALLOC_SCRATCH_BYTES) return GDN_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  if (cudaGetSymbolAddress(&scratch, g_prefill_scratch) != cudaSuccess || scratch == nullptr) {
    (void)cudaGetLastError();
    return GDN_ERR_CUDA;
  }
  return launch_prefill(q, k, v, bf16, alpha, beta, T, Hk, Hv, dk, dv, chunk, state, o, scratch,
                        status, stream);
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
                   float* state, float* o, void* workspace, int32_t* status,
                   cudaStream_t stream) {
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
  const int prep_smem = Hv / Hk > HG ? PREP_SMEM_MULTIPASS : PREP_SMEM;
  if (cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           PREP_SMEM_MULTIPASS) != cudaSuccess ||
      cudaFuncSetAttribute(scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           SCAN_SMEM) != cudaSuccess)
    return GDN_ERR_CUDA;
  st = launch_pdl(prep_kernel, dim3(n_chunks, Hk), dim3(PREP_THREADS), prep_smem, stream,
                  static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(k), alpha, beta,
                  T, Hk, Hv, static_cast<char*>(workspace));
  if (st != GDN_OK) return st;
  return launch_pdl(scan_kernel, dim3(3, Hv), dim3(SCAN_THREADS), SCAN_SMEM, stream, tm_k, tm_q,
                    tm_v48, tm_v32, tm_o48, tm_o32, state, static_cast<const char*>(workspace),
                    T, Hk, Hv, status);
}

}  // namespace gdn
