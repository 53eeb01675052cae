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
#include <cuda_bf16.h>

#include <mutex>

#include "gdn_common.cuh"
#include "gdn_launch.h"

namespace gdn {
namespace {

constexpr int C = 64;         // chunk length
constexpr int DK = 128;       // key / query width
constexpr int DV = 128;       // value width
constexpr int KS = DK * 2 + 16;  // staged bf16 row of K / Q, padded (bytes)
constexpr int XS = C * 2 + 16;   // staged bf16 row of length C, padded (bytes)

// workspace block of one (chunk, value head)
constexpr int WS_T_HI = 0;
constexpr int WS_T_LO = 8192;
constexpr int WS_P_HI = 16384;
constexpr int WS_P_LO = 24576;
constexpr int WS_G = 32768;
constexpr int WS_B = 33024;
constexpr int WS_STRIDE = 33280;

__device__ __forceinline__ uint32_t ld32(const char* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}

// ------------------------------------------------------------------- prep
constexpr int PREP_K = 0;
constexpr int PREP_Q = PREP_K + C * KS;
constexpr int PREP_KK = PREP_Q + C * KS;
constexpr int PREP_QK = PREP_KK + C * C * 4;
constexpr int PREP_A = PREP_QK + C * C * 4;
constexpr int PREP_T = PREP_A + C * 65 * 4;
constexpr int PREP_LG = PREP_T + C * 65 * 4;
constexpr int PREP_G = PREP_LG + C * 4;
constexpr int PREP_B = PREP_G + C * 4;
constexpr int PREP_SMEM = PREP_B + C * 4;

__global__ void __launch_bounds__(128)
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
  float* slg = reinterpret_cast<float*>(smem + PREP_LG);
  float* sg = reinterpret_cast<float*>(smem + PREP_G);
  float* sb = reinterpret_cast<float*>(smem + PREP_B);

  const int c = blockIdx.x, hk = blockIdx.y, G = Hv / Hk;
  const int t0 = c * C, nv = min(C, T - t0);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int g8 = lane >> 2, t4 = lane & 3;

  // K and Q rows of the chunk (rows past the end of the sequence read as zero)
  for (int idx = tid; idx < C * 16; idx += 128) {
    const int r = idx >> 4, ch = idx & 15;
    const bool valid = r < nv;
    const size_t src = ((size_t)(t0 + (valid ? r : 0)) * Hk + hk) * DK + ch * 8;
    cp_async16_zfill(sk + r * KS + ch * 16, k + src, valid);
    cp_async16_zfill(sq + r * KS + ch * 16, q + src, valid);
  }
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();

  // K K^T and Q K^T (64 x 64, fp32 accumulate of exact bf16 products)
  {
    float ckk[8][4], cqk[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) ckk[nt][e] = cqk[nt][e] = 0.f;
    const char* ka0 = sk + (16 * w + g8) * KS;
    const char* qa0 = sq + (16 * w + g8) * KS;
#pragma unroll
    for (int kc = 0; kc < DK / 16; ++kc) {
      const int off = (kc * 16 + t4 * 2) * 2;
      const uint32_t ak[4] = {ld32(ka0 + off), ld32(ka0 + 8 * KS + off), ld32(ka0 + off + 16),
                              ld32(ka0 + 8 * KS + off + 16)};
      const uint32_t aq[4] = {ld32(qa0 + off), ld32(qa0 + 8 * KS + off), ld32(qa0 + off + 16),
                              ld32(qa0 + 8 * KS + off + 16)};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const char* rb = sk + (nt * 8 + g8) * KS + off;
        const uint32_t b0 = ld32(rb), b1 = ld32(rb + 16);
        mma_bf16_16816(ckk[nt], ak, b0, b1);
        mma_bf16_16816(cqk[nt], aq, b0, b1);
      }
    }
    const int r0 = 16 * w + g8;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int c0 = nt * 8 + t4 * 2;
      skk[r0 * C + c0] = ckk[nt][0];
      skk[r0 * C + c0 + 1] = ckk[nt][1];
      skk[(r0 + 8) * C + c0] = ckk[nt][2];
      skk[(r0 + 8) * C + c0 + 1] = ckk[nt][3];
      sqk[r0 * C + c0] = cqk[nt][0];
      sqk[r0 * C + c0 + 1] = cqk[nt][1];
      sqk[(r0 + 8) * C + c0] = cqk[nt][2];
      sqk[(r0 + 8) * C + c0 + 1] = cqk[nt][3];
    }
  }
  __syncthreads();

  for (int j = 0; j < G; ++j) {
    const int h = hk * G + j;
    // gates and the log-space cumulative decay G_t = sum_{s<=t} log alpha_s
    if (tid < C) {
      const int t = tid;
      const bool valid = t < nv;
      const float a = valid ? alpha[(size_t)(t0 + t) * Hv + h] : 1.f;
      const float b = valid ? beta[(size_t)(t0 + t) * Hv + h] : 0.f;
      float lg = valid ? logf(fmaxf(a, 1e-30f)) : 0.f;
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
    for (int idx = tid; idx < C * C; idx += 128) {
      const int t = idx >> 6, s = idx & 63;
      sa[t * 65 + s] = s < t ? sb[t] * expf(sg[t] - sg[s]) * skk[t * C + s] : 0.f;
    }
    __syncthreads();
    // T = (I + A)^-1, one column per thread, rows in order
    if (tid < C) {
      const int s = tid;
      for (int r = 0; r <= s; ++r) st[r * 65 + s] = r == s ? 1.f : 0.f;
      for (int t = s + 1; t < C; ++t) {
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
        int r = s;
        for (; r + 3 < t; r += 4) {
          a0 = fmaf(sa[t * 65 + r], st[r * 65 + s], a0);
          a1 = fmaf(sa[t * 65 + r + 1], st[(r + 1) * 65 + s], a1);
          a2 = fmaf(sa[t * 65 + r + 2], st[(r + 2) * 65 + s], a2);
          a3 = fmaf(sa[t * 65 + r + 3], st[(r + 3) * 65 + s], a3);
        }
        for (; r < t; ++r) a0 = fmaf(sa[t * 65 + r], st[r * 65 + s], a0);
        st[t * 65 + s] = -((a0 + a1) + (a2 + a3));
      }
    }
    __syncthreads();
    // T and P as bf16 hi/lo pairs, g and beta
    char* wsb = ws + ((size_t)c * Hv + h) * WS_STRIDE;
    for (int idx = tid; idx < C * 8; idx += 128) {
      const int t = idx >> 3, e8 = (idx & 7) * 8;
      uint32_t th[4], tl[4], ph[4], pl[4];
#pragma unroll
      for (int qd = 0; qd < 4; ++qd) {
        const int s = e8 + 2 * qd;
        uint32_t h0, l0, h1, l1;
        split_bf16(st[t * 65 + s], h0, l0);
        split_bf16(st[t * 65 + s + 1], h1, l1);
        th[qd] = h0 | (h1 << 16);
        tl[qd] = l0 | (l1 << 16);
        const float p0 = s <= t ? expf(sg[t] - sg[s]) * sqk[t * C + s] : 0.f;
        const float p1 = s + 1 <= t ? expf(sg[t] - sg[s + 1]) * sqk[t * C + s + 1] : 0.f;
        split_bf16(p0, h0, l0);
        split_bf16(p1, h1, l1);
        ph[qd] = h0 | (h1 << 16);
        pl[qd] = l0 | (l1 << 16);
      }
      const int off = (t * C + e8) * 2;
      *reinterpret_cast<uint4*>(wsb + WS_T_HI + off) = make_uint4(th[0], th[1], th[2], th[3]);
      *reinterpret_cast<uint4*>(wsb + WS_T_LO + off) = make_uint4(tl[0], tl[1], tl[2], tl[3]);
      *reinterpret_cast<uint4*>(wsb + WS_P_HI + off) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
      *reinterpret_cast<uint4*>(wsb + WS_P_LO + off) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
    }
    if (tid < C) {
      reinterpret_cast<float*>(wsb + WS_G)[tid] = expf(sg[tid]);
      reinterpret_cast<float*>(wsb + WS_B)[tid] = sb[tid];
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------- scan
constexpr int NTMAX = 6;         // 8-column tiles per state slab (<= 48 columns)
constexpr int VS = NTMAX * 16;   // staged V slab row (bytes)

// one staging buffer
constexpr int BUF_K = 0;
constexpr int BUF_Q = BUF_K + C * KS;
constexpr int BUF_V = BUF_Q + C * KS;
constexpr int BUF_TH = BUF_V + C * VS;
constexpr int BUF_TL = BUF_TH + C * XS;
constexpr int BUF_PH = BUF_TL + C * XS;
constexpr int BUF_PL = BUF_PH + C * XS;
constexpr int BUF_G = BUF_PL + C * XS;
constexpr int BUF_B = BUF_G + C * 4;
constexpr int BUF_SIZE = BUF_B + C * 4;

constexpr int SCAN_HTH = 2 * BUF_SIZE;          // H^T hi: [48][KS]
constexpr int SCAN_HTL = SCAN_HTH + 48 * KS;
constexpr int SCAN_XTH = SCAN_HTL + 48 * KS;    // X^T hi: [48][XS]
constexpr int SCAN_XTL = SCAN_XTH + 48 * XS;
constexpr int SCAN_DTH = SCAN_XTL + 48 * XS;    // Delta^T
constexpr int SCAN_DTL = SCAN_DTH + 48 * XS;
constexpr int SCAN_PTH = SCAN_DTL + 48 * XS;    // D'^T
constexpr int SCAN_PTL = SCAN_PTH + 48 * XS;
constexpr int SCAN_SMEM = SCAN_PTL + 48 * XS;

// the three column slabs of a 128-wide state: 48 + 40 + 40 columns
__device__ __forceinline__ int slab_j0(int s) { return s == 0 ? 0 : (s == 1 ? 48 : 88); }
__device__ __forceinline__ int slab_nt(int s) { return s == 0 ? 6 : 5; }

__device__ __forceinline__ void st16(char* base, int idx, uint32_t v) {
  reinterpret_cast<uint16_t*>(base)[idx] = static_cast<uint16_t>(v);
}

__global__ void __launch_bounds__(128, 1)
scan_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
            const uint16_t* __restrict__ v, float* __restrict__ state, float* __restrict__ o,
            const char* __restrict__ ws, int T, int Hk, int Hv) {
  extern __shared__ __align__(16) char smem[];
  const int sl = blockIdx.x, h = blockIdx.y, hk = h / (Hv / Hk);
  const int j0 = slab_j0(sl), NT = slab_nt(sl);
  const int n_chunks = (T + C - 1) / C;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int g8 = lane >> 2, t4 = lane & 3;
  char* hth = smem + SCAN_HTH;
  char* htl = smem + SCAN_HTL;
  char* xth = smem + SCAN_XTH;
  char* xtl = smem + SCAN_XTL;
  char* dth = smem + SCAN_DTH;
  char* dtl = smem + SCAN_DTL;
  char* pth = smem + SCAN_PTH;
  char* ptl = smem + SCAN_PTL;

  auto stage = [&](int c, int buf) {
    char* B = smem + buf * BUF_SIZE;
    const int t0 = c * C, nv = min(C, T - t0);
    for (int idx = tid; idx < C * 16; idx += 128) {
      const int r = idx >> 4, ch = idx & 15;
      const bool valid = r < nv;
      const size_t src = ((size_t)(t0 + (valid ? r : 0)) * Hk + hk) * DK + ch * 8;
      cp_async16_zfill(B + BUF_K + r * KS + ch * 16, k + src, valid);
      cp_async16_zfill(B + BUF_Q + r * KS + ch * 16, q + src, valid);
    }
    for (int idx = tid; idx < C * NT; idx += 128) {
      const int r = idx / NT, ch = idx - r * NT;
      const bool valid = r < nv;
      const size_t src = ((size_t)(t0 + (valid ? r : 0)) * Hv + h) * DV + j0 + ch * 8;
      cp_async16_zfill(B + BUF_V + r * VS + ch * 16, v + src, valid);
    }
    const char* wsb = ws + ((size_t)c * Hv + h) * WS_STRIDE;
    for (int idx = tid; idx < 4 * C * 8; idx += 128) {
      const int m = idx >> 9, r = (idx >> 3) & 63, ch = idx & 7;
      cp_async16(B + BUF_TH + m * C * XS + r * XS + ch * 16, wsb + m * 8192 + r * 128 + ch * 16);
    }
    for (int idx = tid; idx < 32; idx += 128)
      cp_async16(B + BUF_G + idx * 16, wsb + WS_G + idx * 16);
    cp_async_commit();
  };

  // ---- the state slab -> fp32 fragments (rows 32w + 16mi + g8 (+8), cols nt*8 + 2t4)
  float Hf[2][NTMAX][4];
  float* sth = state + (size_t)h * DK * DV + j0;
#pragma unroll
  for (int mi = 0; mi < 2; ++mi) {
    const int ia = 32 * w + 16 * mi + g8;
#pragma unroll
    for (int nt = 0; nt < NTMAX; ++nt) {
      if (nt < NT) {
        const int jj = nt * 8 + t4 * 2;
        const float2 x = *reinterpret_cast<const float2*>(sth + (size_t)ia * DV + jj);
        const float2 y = *reinterpret_cast<const float2*>(sth + (size_t)(ia + 8) * DV + jj);
        Hf[mi][nt][0] = x.x; Hf[mi][nt][1] = x.y; Hf[mi][nt][2] = y.x; Hf[mi][nt][3] = y.y;
      } else {
        Hf[mi][nt][0] = Hf[mi][nt][1] = Hf[mi][nt][2] = Hf[mi][nt][3] = 0.f;
      }
    }
  }
  // H^T as bf16 hi/lo: element (j, i) at j*KS/2 + i
  auto write_ht = [&]() {
#pragma unroll
    for (int mi = 0; mi < 2; ++mi) {
      const int ia = 32 * w + 16 * mi + g8;
#pragma unroll
      for (int nt = 0; nt < NTMAX; ++nt) {
        if (nt < NT) {
          const int jj = nt * 8 + t4 * 2;
          uint32_t hi, lo;
          split_bf16(Hf[mi][nt][0], hi, lo);
          st16(hth, jj * (KS / 2) + ia, hi); st16(htl, jj * (KS / 2) + ia, lo);
          split_bf16(Hf[mi][nt][1], hi, lo);
          st16(hth, (jj + 1) * (KS / 2) + ia, hi); st16(htl, (jj + 1) * (KS / 2) + ia, lo);
          split_bf16(Hf[mi][nt][2], hi, lo);
          st16(hth, jj * (KS / 2) + ia + 8, hi); st16(htl, jj * (KS / 2) + ia + 8, lo);
          split_bf16(Hf[mi][nt][3], hi, lo);
          st16(hth, (jj + 1) * (KS / 2) + ia + 8, hi); st16(htl, (jj + 1) * (KS / 2) + ia + 8, lo);
        }
      }
    }
  };
  write_ht();
  stage(0, 0);

  const int ta = 16 * w + g8, tb = ta + 8;  // this thread's chunk rows in C x slab tiles
  for (int c = 0; c < n_chunks; ++c) {
    const int buf = c & 1;
    const int nv = min(C, T - c * C);
    if (c + 1 < n_chunks) {
      stage(c + 1, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const char* B = smem + buf * BUF_SIZE;
    const float* bg = reinterpret_cast<const float*>(B + BUF_G);
    const float* bb = reinterpret_cast<const float*>(B + BUF_B);

    // ---- K H and Q H for rows ta, tb
    float kh[NTMAX][4], qh[NTMAX][4];
#pragma unroll
    for (int nt = 0; nt < NTMAX; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) kh[nt][e] = qh[nt][e] = 0.f;
    {
      const char* ka = B + BUF_K + ta * KS;
      const char* qa = B + BUF_Q + ta * KS;
#pragma unroll
      for (int kc = 0; kc < DK / 16; ++kc) {
        const int off = (kc * 16 + t4 * 2) * 2;
        const uint32_t ak[4] = {ld32(ka + off), ld32(ka + 8 * KS + off), ld32(ka + off + 16),
                                ld32(ka + 8 * KS + off + 16)};
        const uint32_t aq[4] = {ld32(qa + off), ld32(qa + 8 * KS + off), ld32(qa + off + 16),
                                ld32(qa + 8 * KS + off + 16)};
#pragma unroll
        for (int nt = 0; nt < NTMAX; ++nt) {
          if (nt < NT) {
            const int rb = (nt * 8 + g8) * KS + off;
            const uint32_t bh0 = ld32(hth + rb), bh1 = ld32(hth + rb + 16);
            const uint32_t bl0 = ld32(htl + rb), bl1 = ld32(htl + rb + 16);
            mma_bf16_16816(kh[nt], ak, bh0, bh1);
            mma_bf16_16816(kh[nt], ak, bl0, bl1);
            mma_bf16_16816(qh[nt], aq, bh0, bh1);
            mma_bf16_16816(qh[nt], aq, bl0, bl1);
          }
        }
      }
    }
    // ---- X = beta (V - g K H), stored transposed as bf16 hi/lo
    {
      const float ga = bg[ta], gb = bg[tb], ba = bb[ta], bbv = bb[tb];
      const char* va = B + BUF_V + ta * VS;
      const char* vb = B + BUF_V + tb * VS;
#pragma unroll
      for (int nt = 0; nt < NTMAX; ++nt) {
        if (nt < NT) {
          const int jj = nt * 8 + t4 * 2;
          const uint32_t pa = ld32(va + jj * 2), pb = ld32(vb + jj * 2);
          const float x0 = ba * (__uint_as_float(pa << 16) - ga * kh[nt][0]);
          const float x1 = ba * (__uint_as_float(pa & 0xffff0000u) - ga * kh[nt][1]);
          const float x2 = bbv * (__uint_as_float(pb << 16) - gb * kh[nt][2]);
          const float x3 = bbv * (__uint_as_float(pb & 0xffff0000u) - gb * kh[nt][3]);
          uint32_t hi, lo;
          split_bf16(x0, hi, lo); st16(xth, jj * (XS / 2) + ta, hi); st16(xtl, jj * (XS / 2) + ta, lo);
          split_bf16(x1, hi, lo); st16(xth, (jj + 1) * (XS / 2) + ta, hi); st16(xtl, (jj + 1) * (XS / 2) + ta, lo);
          split_bf16(x2, hi, lo); st16(xth, jj * (XS / 2) + tb, hi); st16(xtl, jj * (XS / 2) + tb, lo);
          split_bf16(x3, hi, lo); st16(xth, (jj + 1) * (XS / 2) + tb, hi); st16(xtl, (jj + 1) * (XS / 2) + tb, lo);
        }
      }
    }
    __syncthreads();

    // ---- Delta = T X (T lower triangular: k-blocks 0..w)
    float dl[NTMAX][4];
#pragma unroll
    for (int nt = 0; nt < NTMAX; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) dl[nt][e] = 0.f;
    for (int kc = 0; kc <= w; ++kc) {
      const int off = (kc * 16 + t4 * 2) * 2;
      const char* th = B + BUF_TH + ta * XS + off;
      const char* tl = B + BUF_TL + ta * XS + off;
      const uint32_t ah[4] = {ld32(th), ld32(th + 8 * XS), ld32(th + 16), ld32(th + 8 * XS + 16)};
      const uint32_t al[4] = {ld32(tl), ld32(tl + 8 * XS), ld32(tl + 16), ld32(tl + 8 * XS + 16)};
#pragma unroll
      for (int nt = 0; nt < NTMAX; ++nt) {
        if (nt < NT) {
          const int rb = (nt * 8 + g8) * XS + off;
          const uint32_t bh0 = ld32(xth + rb), bh1 = ld32(xth + rb + 16);
          const uint32_t bl0 = ld32(xtl + rb), bl1 = ld32(xtl + rb + 16);
          mma_bf16_16816(dl[nt], ah, bh0, bh1);
          mma_bf16_16816(dl[nt], ah, bl0, bl1);
          mma_bf16_16816(dl[nt], al, bh0, bh1);
        }
      }
    }
    const float gC = bg[C - 1];
    {
      const float ra = gC / bg[ta], rbv = gC / bg[tb];
#pragma unroll
      for (int nt = 0; nt < NTMAX; ++nt) {
        if (nt < NT) {
          const int jj = nt * 8 + t4 * 2;
          const int idx[4] = {jj * (XS / 2) + ta, (jj + 1) * (XS / 2) + ta, jj * (XS / 2) + tb,
                              (jj + 1) * (XS / 2) + tb};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint32_t hi, lo;
            split_bf16(dl[nt][e], hi, lo);
            st16(dth, idx[e], hi); st16(dtl, idx[e], lo);
            split_bf16((e < 2 ? ra : rbv) * dl[nt][e], hi, lo);
            st16(pth, idx[e], hi); st16(ptl, idx[e], lo);
          }
        }
      }
    }
    __syncthreads();

    // ---- O = g Q H + P Delta (P lower triangular incl. the diagonal)
    {
      const float ga = bg[ta], gb = bg[tb];
#pragma unroll
      for (int nt = 0; nt < NTMAX; ++nt) {
        qh[nt][0] *= ga; qh[nt][1] *= ga; qh[nt][2] *= gb; qh[nt][3] *= gb;
      }
      for (int kc = 0; kc <= w; ++kc) {
        const int off = (kc * 16 + t4 * 2) * 2;
        const char* ph = B + BUF_PH + ta * XS + off;
        const char* pl = B + BUF_PL + ta * XS + off;
        const uint32_t ah[4] = {ld32(ph), ld32(ph + 8 * XS), ld32(ph + 16), ld32(ph + 8 * XS + 16)};
        const uint32_t al[4] = {ld32(pl), ld32(pl + 8 * XS), ld32(pl + 16), ld32(pl + 8 * XS + 16)};
#pragma unroll
        for (int nt = 0; nt < NTMAX; ++nt) {
          if (nt < NT) {
            const int rb = (nt * 8 + g8) * XS + off;
            const uint32_t bh0 = ld32(dth + rb), bh1 = ld32(dth + rb + 16);
            const uint32_t bl0 = ld32(dtl + rb), bl1 = ld32(dtl + rb + 16);
            mma_bf16_16816(qh[nt], ah, bh0, bh1);
            mma_bf16_16816(qh[nt], ah, bl0, bl1);
            mma_bf16_16816(qh[nt], al, bh0, bh1);
          }
        }
      }
      float* oa = o + ((size_t)(c * C + ta) * Hv + h) * DV + j0;
      float* ob = o + ((size_t)(c * C + tb) * Hv + h) * DV + j0;
#pragma unroll
      for (int nt = 0; nt < NTMAX; ++nt) {
        if (nt < NT) {
          const int jj = nt * 8 + t4 * 2;
          if (ta < nv) *reinterpret_cast<float2*>(oa + jj) = make_float2(qh[nt][0], qh[nt][1]);
          if (tb < nv) *reinterpret_cast<float2*>(ob + jj) = make_float2(qh[nt][2], qh[nt][3]);
        }
      }
    }

    // ---- H <- g_C H + K^T D'  (A = K^T tiles through ldmatrix.trans)
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
      for (int nt = 0; nt < NTMAX; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) Hf[mi][nt][e] *= gC;
    {
      const int q4 = lane >> 3, r8 = lane & 7;
#pragma unroll
      for (int kc = 0; kc < C / 16; ++kc) {
        const int off = (kc * 16 + t4 * 2) * 2;
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) {
          const int i0 = 32 * w + 16 * mi;
          const int row = kc * 16 + ((q4 & 2) ? 8 : 0) + r8;
          const int col = i0 + ((q4 & 1) ? 8 : 0);
          uint32_t a[4];
          ldmatrix_x4_trans(a, B + BUF_K + row * KS + col * 2);
#pragma unroll
          for (int nt = 0; nt < NTMAX; ++nt) {
            if (nt < NT) {
              const int rb = (nt * 8 + g8) * XS + off;
              mma_bf16_16816(Hf[mi][nt], a, ld32(pth + rb), ld32(pth + rb + 16));
              mma_bf16_16816(Hf[mi][nt], a, ld32(ptl + rb), ld32(ptl + rb + 16));
            }
          }
        }
      }
    }
    write_ht();
    __syncthreads();
  }

#pragma unroll
  for (int mi = 0; mi < 2; ++mi) {
    const int ia = 32 * w + 16 * mi + g8;
#pragma unroll
    for (int nt = 0; nt < NTMAX; ++nt) {
      if (nt < NT) {
        const int jj = nt * 8 + t4 * 2;
        *reinterpret_cast<float2*>(sth + (size_t)ia * DV + jj) = make_float2(Hf[mi][nt][0], Hf[mi][nt][1]);
        *reinterpret_cast<float2*>(sth + (size_t)(ia + 8) * DV + jj) = make_float2(Hf[mi][nt][2], Hf[mi][nt][3]);
      }
    }
  }
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

int launch_prefill(const void* q, const void* k, const void* v, bool bf16, const float* alpha,
                   const float* beta, int T, int Hk, int Hv, int dk, int dv, int chunk,
                   float* state, float* o, void* workspace, cudaStream_t stream) {
  if (!bf16 || dk != DK || dv != DV || chunk != C) return GDN_ERR_UNSUPPORTED;
  const int n_chunks = (T + C - 1) / C;
  if (cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           PREP_SMEM) != cudaSuccess ||
      cudaFuncSetAttribute(scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           SCAN_SMEM) != cudaSuccess)
    return GDN_ERR_CUDA;
  prep_kernel<<<dim3(n_chunks, Hk), 128, PREP_SMEM, stream>>>(
      static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(k), alpha, beta, T, Hk, Hv,
      static_cast<char*>(workspace));
  int st = launch_status();
  if (st != GDN_OK) return st;
  scan_kernel<<<dim3(3, Hv), 128, SCAN_SMEM, stream>>>(
      static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(k),
      static_cast<const uint16_t*>(v), state, o, static_cast<const char*>(workspace), T, Hk, Hv);
  return launch_status();
}

}  // namespace gdn
