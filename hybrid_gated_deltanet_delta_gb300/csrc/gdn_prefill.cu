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

// workspace block of one (chunk, value head): T and P as bf16 hi/lo, 64 x 64
// each in 128-byte rows whose 16-byte chunks are XOR-swizzled by row (chunk ch
// of row t at chunk ch ^ (t & 7)), then g and beta.  The scan copies the block
// into shared memory as is; the swizzle keeps its fragment loads free of bank
// conflicts.
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
    // T and P as bf16 hi/lo pairs, g and beta
    char* wsb = ws + ((size_t)c * Hv + h) * WS_STRIDE;
    for (int idx = tid; idx < C * 8; idx += PREP_THREADS) {
      const int t = idx >> 3, e8 = (idx & 7) * 8;
      uint32_t th[4], tl[4], ph[4], pl[4];
#pragma unroll
      for (int qd = 0; qd < 4; ++qd) {
        const int s = e8 + 2 * qd;
        uint32_t h0, l0, h1, l1;
        split_bf16(st[t * TS + s], h0, l0);
        split_bf16(st[t * TS + s + 1], h1, l1);
        th[qd] = h0 | (h1 << 16);
        tl[qd] = l0 | (l1 << 16);
        const float p0 = s <= t ? __expf(sg[t] - sg[s]) * sqk[t * C + s] : 0.f;
        const float p1 = s + 1 <= t ? __expf(sg[t] - sg[s + 1]) * sqk[t * C + s + 1] : 0.f;
        split_bf16(p0, h0, l0);
        split_bf16(p1, h1, l1);
        ph[qd] = h0 | (h1 << 16);
        pl[qd] = l0 | (l1 << 16);
      }
      // 128-byte rows, 16-byte chunk ch of row t stored at chunk ch ^ (t & 7)
      const int off = t * 128 + (((e8 >> 3) ^ (t & 7)) << 4);
      *reinterpret_cast<uint4*>(wsb + WS_T_HI + off) = make_uint4(th[0], th[1], th[2], th[3]);
      *reinterpret_cast<uint4*>(wsb + WS_T_LO + off) = make_uint4(tl[0], tl[1], tl[2], tl[3]);
      *reinterpret_cast<uint4*>(wsb + WS_P_HI + off) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
      *reinterpret_cast<uint4*>(wsb + WS_P_LO + off) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
    }
    if (tid < C) {
      reinterpret_cast<float*>(wsb + WS_G)[tid] = __expf(sg[tid]);
      reinterpret_cast<float*>(wsb + WS_B)[tid] = sb[tid];
    }
    // the next head's gates have landed and every thread is done with this head
    cp_async_wait<0>();
    __syncthreads();
  }
}

// ------------------------------------------------------------------- scan
constexpr int SCAN_THREADS = 256;  // 8 warps
constexpr int NTMAX = 6;           // 8-column tiles per state slab (<= 48 columns)
constexpr int NTW = 3;             // tiles per warp in the chunk x slab products
constexpr int VS = NTMAX * 16;     // staged V slab row (bytes)

// one staging buffer: K and Q rows (padded), the V slab, then the chunk's
// workspace block copied as is (T hi/lo, P hi/lo in swizzled 128-byte rows, g, beta)
constexpr int BUF_K = 0;
constexpr int BUF_Q = BUF_K + C * KS;
constexpr int BUF_V = BUF_Q + C * KS;
constexpr int BUF_W = BUF_V + C * VS;
constexpr int BUF_TH = BUF_W + WS_T_HI;
constexpr int BUF_TL = BUF_W + WS_T_LO;
constexpr int BUF_PH = BUF_W + WS_P_HI;
constexpr int BUF_PL = BUF_W + WS_P_LO;
constexpr int BUF_G = BUF_W + WS_G;
constexpr int BUF_B = BUF_W + WS_B;
constexpr int BUF_SIZE = BUF_W + WS_STRIDE;
static_assert(BUF_W % 16 == 0 && BUF_SIZE % 16 == 0, "bulk copy destinations are 16-byte aligned");

constexpr int SCAN_HTH = 2 * BUF_SIZE;          // H^T hi: [48][KS]
constexpr int SCAN_HTL = SCAN_HTH + 48 * KS;
constexpr int SCAN_XTH = SCAN_HTL + 48 * KS;    // X^T hi: [48][XS]
constexpr int SCAN_XTL = SCAN_XTH + 48 * XS;
constexpr int SCAN_DTH = SCAN_XTL + 48 * XS;    // Delta^T
constexpr int SCAN_DTL = SCAN_DTH + 48 * XS;
constexpr int SCAN_PTH = SCAN_DTL + 48 * XS;    // D'^T
constexpr int SCAN_PTL = SCAN_PTH + 48 * XS;
constexpr int SCAN_BAR = SCAN_PTL + 48 * XS;    // two mbarriers, one per buffer
constexpr int SCAN_SMEM = SCAN_BAR + 16;

// polls of an mbarrier before a block gives up on its staged chunk
constexpr long long kWaitPolls = 1ll << 22;

// the three column slabs of a 128-wide state: 48 + 40 + 40 columns
__device__ __forceinline__ int slab_j0(int s) { return s == 0 ? 0 : (s == 1 ? 48 : 88); }
__device__ __forceinline__ int slab_nt(int s) { return s == 0 ? 6 : 5; }

__device__ __forceinline__ void st16(char* base, int idx, uint32_t v) {
  reinterpret_cast<uint16_t*>(base)[idx] = static_cast<uint16_t>(v);
}

// A fragment (16 x 16 bf16, row-major, row stride `stride` bytes) at (m0, k0)
__device__ __forceinline__ void load_a(uint32_t (&a)[4], const char* base, int stride, int m0,
                                       int k0, int lane) {
  const int q = lane >> 3, r = lane & 7;
  ldmatrix_x4(a, base + (m0 + (q & 1) * 8 + r) * stride + (k0 + (q >> 1) * 8) * 2);
}

// A fragment (16 x 16) of a 64 x 64 bf16 matrix in swizzled 128-byte rows
// (16-byte chunk ch of row r stored at chunk ch ^ (r & 7)) at (m0, k0)
__device__ __forceinline__ void load_a_swz(uint32_t (&a)[4], const char* base, int m0, int k0,
                                           int lane) {
  const int q = lane >> 3, r = lane & 7;
  const int row = m0 + (q & 1) * 8 + r, ch = (k0 >> 3) + (q >> 1);
  ldmatrix_x4(a, base + row * 128 + ((ch ^ (row & 7)) << 4));
}

// B fragments of one 8-column tile for the hi and lo halves (stored [n][k],
// row stride `stride` bytes): b[0], b[1] = hi; b[2], b[3] = lo.
__device__ __forceinline__ void load_b_pair(uint32_t (&b)[4], const char* hi, const char* lo,
                                            int stride, int n0, int k0, int lane) {
  const int q = lane >> 3, r = lane & 7;
  ldmatrix_x4(b, (q < 2 ? hi : lo) + (n0 + r) * stride + (k0 + (q & 1) * 8) * 2);
}

__global__ void __launch_bounds__(SCAN_THREADS, 1)
scan_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
            const uint16_t* __restrict__ v, float* __restrict__ state, float* __restrict__ o,
            const char* __restrict__ ws, int T, int Hk, int Hv) {
  extern __shared__ __align__(16) char smem[];
  const int sl = blockIdx.x, h = blockIdx.y, hk = h / (Hv / Hk);
  const int j0 = slab_j0(sl), NT = slab_nt(sl);
  const int n_chunks = (T + C - 1) / C;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int g8 = lane >> 2, t4 = lane & 3;
  const int mt = w & 3, nt0 = (w >> 2) * NTW;  // this warp's chunk rows and column tiles
  char* hth = smem + SCAN_HTH;
  char* htl = smem + SCAN_HTL;
  char* xth = smem + SCAN_XTH;
  char* xtl = smem + SCAN_XTL;
  char* dth = smem + SCAN_DTH;
  char* dtl = smem + SCAN_DTL;
  char* pth = smem + SCAN_PTH;
  char* ptl = smem + SCAN_PTL;

  // Staging of one chunk: the chunk's workspace block (33 KB, contiguous) by a
  // single bulk (TMA) copy completing on the buffer's mbarrier; the K, Q and V
  // slab rows by 16-byte cp.async spread over all threads, whose (row, piece)
  // assignment is the same for every chunk, so the offsets are computed once.
  // Rows past the end of the sequence read as zero.  The buffer being filled
  // was last read before the previous iteration's closing barrier.
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + SCAN_BAR);
  if (tid == 0) {
    mbar_init(&mbar[0], 1);
    mbar_init(&mbar[1], 1);
    mbar_init_fence();
  }
  __syncthreads();
  constexpr int KQ_PER = C * 16 / SCAN_THREADS;
  int kq_row[KQ_PER], kq_dst[KQ_PER], kq_src[KQ_PER];
#pragma unroll
  for (int u = 0; u < KQ_PER; ++u) {
    const int idx = tid + u * SCAN_THREADS, r = idx >> 4, ch = idx & 15;
    kq_row[u] = r;
    kq_dst[u] = r * KS + ch * 16;
    kq_src[u] = (r * Hk + hk) * DK + ch * 8;  // elements, relative to the chunk's first row
  }
  int v_row[2], v_dst[2], v_src[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int idx = tid + u * SCAN_THREADS;
    const int r = idx < C * NT ? idx / NT : C, ch = idx < C * NT ? idx - (idx / NT) * NT : 0;
    v_row[u] = r;
    v_dst[u] = r * VS + ch * 16;
    v_src[u] = (r * Hv + h) * DV + j0 + ch * 8;
  }
  auto stage = [&](int c, int buf) {
    char* B = smem + buf * BUF_SIZE;
    const int t0 = c * C, nv = min(C, T - t0);
    if (tid == 0) {
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&mbar[buf], (unsigned)WS_STRIDE);
      bulk_g2s(B + BUF_W, ws + ((size_t)c * Hv + h) * WS_STRIDE, WS_STRIDE, &mbar[buf]);
    }
    const uint16_t* kb = k + (size_t)t0 * Hk * DK;
    const uint16_t* qb = q + (size_t)t0 * Hk * DK;
    const uint16_t* vbase = v + (size_t)t0 * Hv * DV;
#pragma unroll
    for (int u = 0; u < KQ_PER; ++u) {
      const bool valid = kq_row[u] < nv;
      const int src = valid ? kq_src[u] : 0;
      cp_async16_zfill(B + BUF_K + kq_dst[u], kb + src, valid);
      cp_async16_zfill(B + BUF_Q + kq_dst[u], qb + src, valid);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (v_row[u] < C) {
        const bool valid = v_row[u] < nv;
        cp_async16_zfill(B + BUF_V + v_dst[u], vbase + (valid ? v_src[u] : 0), valid);
      }
    }
    cp_async_commit();
  };

  // ---- this warp's 16 state rows (16w + g8 (+8)), all slab columns (nt*8 + 2t4)
  float Hf[NTMAX][4];
  float* sth = state + (size_t)h * DK * DV + j0;
  const int ia = 16 * w + g8;
#pragma unroll
  for (int nt = 0; nt < NTMAX; ++nt) {
    if (nt < NT) {
      const int jj = nt * 8 + t4 * 2;
      const float2 x = *reinterpret_cast<const float2*>(sth + (size_t)ia * DV + jj);
      const float2 y = *reinterpret_cast<const float2*>(sth + (size_t)(ia + 8) * DV + jj);
      Hf[nt][0] = x.x; Hf[nt][1] = x.y; Hf[nt][2] = y.x; Hf[nt][3] = y.y;
    } else {
      Hf[nt][0] = Hf[nt][1] = Hf[nt][2] = Hf[nt][3] = 0.f;
    }
  }
  // H^T as bf16 hi/lo: element (j, i) at j*KS/2 + i
  auto write_ht = [&]() {
#pragma unroll
    for (int nt = 0; nt < NTMAX; ++nt) {
      if (nt < NT) {
        const int jj = nt * 8 + t4 * 2;
        const int idx[4] = {jj * (KS / 2) + ia, (jj + 1) * (KS / 2) + ia, jj * (KS / 2) + ia + 8,
                            (jj + 1) * (KS / 2) + ia + 8};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          uint32_t hi, lo;
          split_bf16(Hf[nt][e], hi, lo);
          st16(hth, idx[e], hi);
          st16(htl, idx[e], lo);
        }
      }
    }
  };
  write_ht();
  stage(0, 0);

  const int ta = 16 * mt + g8, tb = ta + 8;  // this thread's chunk rows
  for (int c = 0; c < n_chunks; ++c) {
    const int buf = c & 1;
    const int nv = min(C, T - c * C);
    if (c + 1 < n_chunks) {
      stage(c + 1, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    // chunk c is the (c/2)-th use of its buffer: wait for that phase
    if (!__syncthreads_and(mbar_wait_bounded(&mbar[buf], (c >> 1) & 1, kWaitPolls))) {
      // a staged chunk never arrived: give the copies in flight a last bounded
      // chance to land, mark this block's state slab as failed (NaN), stop
      mbar_wait_bounded(&mbar[buf ^ 1], ((c + 1) >> 1) & 1, kWaitPolls);
      for (int idx = tid; idx < DK * 8 * NT; idx += SCAN_THREADS)
        sth[(size_t)(idx / (8 * NT)) * DV + idx % (8 * NT)] = __int_as_float(0x7fc00000);
      return;
    }
    const char* B = smem + buf * BUF_SIZE;
    const float* bg = reinterpret_cast<const float*>(B + BUF_G);
    const float* bb = reinterpret_cast<const float*>(B + BUF_B);

    // ---- K H and Q H: rows of m-tile mt, column tiles nt0 .. nt0+2
    float kh[NTW][4], qh[NTW][4];
#pragma unroll
    for (int i = 0; i < NTW; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) kh[i][e] = qh[i][e] = 0.f;
#pragma unroll
    for (int kc = 0; kc < DK / 16; ++kc) {
      uint32_t ak[4], aq[4];
      load_a(ak, B + BUF_K, KS, 16 * mt, kc * 16, lane);
      load_a(aq, B + BUF_Q, KS, 16 * mt, kc * 16, lane);
#pragma unroll
      for (int i = 0; i < NTW; ++i) {
        if (nt0 + i < NT) {
          uint32_t b[4];
          load_b_pair(b, hth, htl, KS, (nt0 + i) * 8, kc * 16, lane);
          mma_bf16_16816(kh[i], ak, b[0], b[1]);
          mma_bf16_16816(kh[i], ak, b[2], b[3]);
          mma_bf16_16816(qh[i], aq, b[0], b[1]);
          mma_bf16_16816(qh[i], aq, b[2], b[3]);
        }
      }
    }
    // ---- X = beta (V - g K H), stored transposed as bf16 hi/lo
    {
      const float ga = bg[ta], gb = bg[tb], ba = bb[ta], bbv = bb[tb];
      const char* va = B + BUF_V + ta * VS;
      const char* vb = B + BUF_V + tb * VS;
#pragma unroll
      for (int i = 0; i < NTW; ++i) {
        if (nt0 + i < NT) {
          const int jj = (nt0 + i) * 8 + t4 * 2;
          const uint32_t pa = ld32(va + jj * 2), pb = ld32(vb + jj * 2);
          const float x[4] = {ba * (__uint_as_float(pa << 16) - ga * kh[i][0]),
                              ba * (__uint_as_float(pa & 0xffff0000u) - ga * kh[i][1]),
                              bbv * (__uint_as_float(pb << 16) - gb * kh[i][2]),
                              bbv * (__uint_as_float(pb & 0xffff0000u) - gb * kh[i][3])};
          const int idx[4] = {jj * (XS / 2) + ta, (jj + 1) * (XS / 2) + ta, jj * (XS / 2) + tb,
                              (jj + 1) * (XS / 2) + tb};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint32_t hi, lo;
            split_bf16(x[e], hi, lo);
            st16(xth, idx[e], hi);
            st16(xtl, idx[e], lo);
          }
        }
      }
    }
    __syncthreads();

    // ---- Delta = T X (T lower triangular: k-blocks 0..mt)
    float dl[NTW][4];
#pragma unroll
    for (int i = 0; i < NTW; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) dl[i][e] = 0.f;
    for (int kc = 0; kc <= mt; ++kc) {
      uint32_t ah[4], al[4];
      load_a_swz(ah, B + BUF_TH, 16 * mt, kc * 16, lane);
      load_a_swz(al, B + BUF_TL, 16 * mt, kc * 16, lane);
#pragma unroll
      for (int i = 0; i < NTW; ++i) {
        if (nt0 + i < NT) {
          uint32_t b[4];
          load_b_pair(b, xth, xtl, XS, (nt0 + i) * 8, kc * 16, lane);
          mma_bf16_16816(dl[i], ah, b[0], b[1]);
          mma_bf16_16816(dl[i], ah, b[2], b[3]);
          mma_bf16_16816(dl[i], al, b[0], b[1]);
        }
      }
    }
    const float gC = bg[C - 1];
    {
      const float ra = gC / bg[ta], rbv = gC / bg[tb];
#pragma unroll
      for (int i = 0; i < NTW; ++i) {
        if (nt0 + i < NT) {
          const int jj = (nt0 + i) * 8 + t4 * 2;
          const int idx[4] = {jj * (XS / 2) + ta, (jj + 1) * (XS / 2) + ta, jj * (XS / 2) + tb,
                              (jj + 1) * (XS / 2) + tb};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint32_t hi, lo;
            split_bf16(dl[i][e], hi, lo);
            st16(dth, idx[e], hi);
            st16(dtl, idx[e], lo);
            split_bf16((e < 2 ? ra : rbv) * dl[i][e], hi, lo);
            st16(pth, idx[e], hi);
            st16(ptl, idx[e], lo);
          }
        }
      }
    }
    __syncthreads();

    // ---- O = g Q H + P Delta (P lower triangular incl. the diagonal)
    {
      const float ga = bg[ta], gb = bg[tb];
#pragma unroll
      for (int i = 0; i < NTW; ++i) {
        qh[i][0] *= ga; qh[i][1] *= ga; qh[i][2] *= gb; qh[i][3] *= gb;
      }
      for (int kc = 0; kc <= mt; ++kc) {
        uint32_t ah[4], al[4];
        load_a_swz(ah, B + BUF_PH, 16 * mt, kc * 16, lane);
        load_a_swz(al, B + BUF_PL, 16 * mt, kc * 16, lane);
#pragma unroll
        for (int i = 0; i < NTW; ++i) {
          if (nt0 + i < NT) {
            uint32_t b[4];
            load_b_pair(b, dth, dtl, XS, (nt0 + i) * 8, kc * 16, lane);
            mma_bf16_16816(qh[i], ah, b[0], b[1]);
            mma_bf16_16816(qh[i], ah, b[2], b[3]);
            mma_bf16_16816(qh[i], al, b[0], b[1]);
          }
        }
      }
      float* oa = o + ((size_t)(c * C + ta) * Hv + h) * DV + j0;
      float* ob = o + ((size_t)(c * C + tb) * Hv + h) * DV + j0;
#pragma unroll
      for (int i = 0; i < NTW; ++i) {
        if (nt0 + i < NT) {
          const int jj = (nt0 + i) * 8 + t4 * 2;
          if (ta < nv) *reinterpret_cast<float2*>(oa + jj) = make_float2(qh[i][0], qh[i][1]);
          if (tb < nv) *reinterpret_cast<float2*>(ob + jj) = make_float2(qh[i][2], qh[i][3]);
        }
      }
    }

    // ---- H <- g_C H + K^T D'  (A = K^T tiles through ldmatrix.trans)
#pragma unroll
    for (int nt = 0; nt < NTMAX; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) Hf[nt][e] *= gC;
    {
      const int q4 = lane >> 3, r8 = lane & 7;
#pragma unroll
      for (int kc = 0; kc < C / 16; ++kc) {
        const int row = kc * 16 + ((q4 & 2) ? 8 : 0) + r8;
        const int col = 16 * w + ((q4 & 1) ? 8 : 0);
        uint32_t a[4];
        ldmatrix_x4_trans(a, B + BUF_K + row * KS + col * 2);
#pragma unroll
        for (int nt = 0; nt < NTMAX; ++nt) {
          if (nt < NT) {
            uint32_t b[4];
            load_b_pair(b, pth, ptl, XS, nt * 8, kc * 16, lane);
            mma_bf16_16816(Hf[nt], a, b[0], b[1]);
            mma_bf16_16816(Hf[nt], a, b[2], b[3]);
          }
        }
      }
    }
    write_ht();
    __syncthreads();
  }

#pragma unroll
  for (int nt = 0; nt < NTMAX; ++nt) {
    if (nt < NT) {
      const int jj = nt * 8 + t4 * 2;
      *reinterpret_cast<float2*>(sth + (size_t)ia * DV + jj) = make_float2(Hf[nt][0], Hf[nt][1]);
      *reinterpret_cast<float2*>(sth + (size_t)(ia + 8) * DV + jj) = make_float2(Hf[nt][2], Hf[nt][3]);
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
  prep_kernel<<<dim3(n_chunks, Hk), PREP_THREADS, PREP_SMEM, stream>>>(
      static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(k), alpha, beta, T, Hk, Hv,
      static_cast<char*>(workspace));
  int st = launch_status();
  if (st != GDN_OK) return st;
  scan_kernel<<<dim3(3, Hv), SCAN_THREADS, SCAN_SMEM, stream>>>(
      static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(k),
      static_cast<const uint16_t*>(v), state, o, static_cast<const char*>(workspace), T, Hk, Hv);
  return launch_status();
}

}  // namespace gdn
